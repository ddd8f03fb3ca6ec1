"""The allocation-free backward entry point (ne_attn_bwd_noalloc).

Some callers cannot call cudaMalloc when they need the gradients: a stream being
captured into a CUDA graph, a runtime whose own allocator already owns the device's
free memory, a real-time loop that forbids allocation after start-up.  For them the
library offers a backward whose scratch lives in a fixed device array compiled into
the library.  These tests call it through the C ABI and check it against the regular
entry point (which takes a caller-allocated workspace), twice in a row, since the
second call finds the first call's leftovers in the shared scratch.

This file sorts last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import causal_gqa_flash_attention_gb300 as ne
from causal_gqa_flash_attention_gb300 import _build, synthetic

pytestmark = pytest.mark.gpu

GRAD_TOL = 1e-2     # the bf16 gradient bound the parity tests use


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return ne.load()


def rel(x, ref):
    x, ref = x.double().cpu().numpy(), ref.double().cpu().numpy()
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30))


def call_noalloc(lib, q, k, v, o, lse, dO, dq, dk, dv, theta=10000.0):
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ne_attn_bwd_noalloc(p(q), p(k), p(v), p(o), p(lse), p(dO), p(dq), p(dk), p(dv),
                                   B, T, Hq, Hkv, D, theta, st)


def noalloc_error(lib):
    return lib.ne_noalloc_get_device_error(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [(2, 300, 6, 2, 64), (1, 256, 4, 1, 128)])
def test_noalloc_backward_matches_workspace_backward_twice(lib, shape):
    import oracle
    B, T, Hq, Hkv, D = shape
    qc, kc, vc, dOc = synthetic.make_custom(B, T, Hq, Hkv, D, torch.bfloat16, seed=31 + D)
    q, k, v, dO = (t.cuda() for t in (qc, kc, vc, dOc))
    o, lse = ne.attn_fwd(q, k, v)
    dq_ref, dk_ref, dv_ref = ne.attn_bwd(q, k, v, o, lse, dO)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK
    # The fp64 oracle on the same inputs: a mistake shared by both GPU entry points
    # (the RoPE table, the preprocess pass) shows up here, not in the comparison above.
    f = lambda t: t.double().numpy()
    ora = dict(zip(("dq", "dk", "dv"), oracle.attn_bwd(f(qc), f(kc), f(vc), f(dOc))))
    for call in range(2):
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        alloc_before = torch.cuda.memory_allocated()
        assert call_noalloc(lib, q, k, v, o, lse, dO, dq, dk, dv) == ne.NE_OK, lib.ne_last_error()
        torch.cuda.synchronize()
        assert noalloc_error(lib) == ne.NE_OK, lib.ne_last_error()
        # Nothing may be allocated by the call (memory freed meanwhile by torch is fine).
        if call == 1:   # the first call may still load the module holding the scratch
            assert torch.cuda.mem_get_info()[0] >= free_before
        assert torch.cuda.memory_allocated() <= alloc_before
        for name, got, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
            assert torch.isfinite(got).all(), (call, name)
            e = rel(got, ref)
            assert e <= GRAD_TOL, (call, name, e)
            e = rel(got, torch.from_numpy(ora[name]))
            assert e <= GRAD_TOL, ("oracle", call, name, e)


def test_noalloc_backward_reports_fp16_overflow_in_its_own_error_word(lib):
    """An upstream gradient large enough to push dS past the fp16 range of its MMA
    operand is recorded in the allocation-free calls' own device word (the call has no
    allocated one) and read back, then cleared, by ne_noalloc_get_device_error."""
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(1, 96, 2, 1, 64, torch.bfloat16, seed=13))
    o, lse = ne.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK
    assert noalloc_error(lib) == ne.NE_OK
    big = (dO * 1.0e6).contiguous()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert call_noalloc(lib, q, k, v, o, lse, big, dq, dk, dv) == ne.NE_OK, lib.ne_last_error()
    assert noalloc_error(lib) == ne.NE_ERR_INVALID_ARG
    assert "fp16" in lib.ne_last_error().decode()
    assert noalloc_error(lib) == ne.NE_OK          # read and cleared
    assert ne.get_device_error() == ne.NE_OK       # the allocated word was not touched


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    B, T, Hq, Hkv, D = 64, 512, 12, 4, 64          # needs ~152 MB > 48 MiB
    need = (math.ceil(T * (D // 2) * 8 / 256) * 256 + math.ceil(B * Hq * T * 4 / 256) * 256
            + math.ceil(B * T * Hq * D * 4 / 256) * 256 + B * T * Hq * D * 2)
    assert need > 48 << 20
    q = torch.empty(16, dtype=torch.uint8, device="cuda")   # never touched: rejected first
    p = ctypes.c_void_p(q.data_ptr())
    st = lib.ne_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, T, Hq, Hkv, D, 10000.0, ctypes.c_void_p(0))
    assert st == ne.NE_ERR_INVALID_ARG
    assert "scratch" in lib.ne_last_error().decode()
