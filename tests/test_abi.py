"""C-ABI checks that need no GPU: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

import causal_gqa_flash_attention_gb300 as ne
from causal_gqa_flash_attention_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "neattn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ne.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ne_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_symbols() == sorted(ne.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    names = [lib.ne_status_string(i).decode() for i in range(6)]
    assert names == ["NE_OK", "NE_ERR_INVALID_ARG", "NE_ERR_UNSUPPORTED", "NE_ERR_CUDA",
                     "NE_ERR_DEVICE_TIMEOUT", "NE_ERR_NO_DEVICE"]


def test_workspace_size_formula(lib):
    B, T, Hq, Hkv, D = 16, 512, 12, 4, 64
    r256 = lambda x: (x + 255) // 256 * 256
    # Delta fp32 [B,Hq,T] | dQ accumulator fp32 [B,T,Hq,D] | rotated fp16 Q [B,T,Hq,D]
    want = r256(B * Hq * T * 4) + r256(B * T * Hq * D * 4) + B * T * Hq * D * 2
    assert lib.ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D) == want
    assert lib.ne_attn_bwd_workspace_size(1, 8, 3, 2, 64) == 0   # Hq % Hkv != 0


@pytest.mark.parametrize("args,expect", [
    ((1, 8, 3, 2, 64, 10000.0), ne.NE_ERR_INVALID_ARG),    # Hq % Hkv
    ((1, 8, 4, 2, 63, 10000.0), ne.NE_ERR_INVALID_ARG),    # odd D
    ((1, 8, 4, 2, 64, -1.0), ne.NE_ERR_INVALID_ARG),       # theta
    ((-1, 8, 4, 2, 64, 10000.0), ne.NE_ERR_INVALID_ARG),   # B
    ((1, 8, 4, 2, 96, 10000.0), ne.NE_ERR_UNSUPPORTED),    # head_dim
    ((1, 8, 4, 0, 64, 10000.0), ne.NE_ERR_INVALID_ARG),    # Hkv
])
def test_forward_rejects_bad_shapes_before_any_device_work(lib, args, expect):
    null = ctypes.c_void_p(0)
    B, T, Hq, Hkv, D, theta = args
    st = lib.ne_attn_fwd(null, null, null, null, null, B, T, Hq, Hkv, D, theta, null)
    assert st == expect
    assert lib.ne_last_error().decode() != ""


def test_empty_problem_is_a_no_op(lib):
    null = ctypes.c_void_p(0)
    assert lib.ne_attn_fwd(null, null, null, null, null, 0, 128, 4, 2, 64, 10000.0, null) == ne.NE_OK
    assert lib.ne_attn_fwd(null, null, null, null, null, 2, 0, 4, 2, 64, 10000.0, null) == ne.NE_OK


def test_backward_rejects_small_workspace_and_misalignment(lib):
    vp = ctypes.c_void_p
    p = vp(4096)   # never dereferenced: validation fails first
    st = lib.ne_attn_bwd(p, p, p, p, p, p, p, p, p, 1, 8, 4, 2, 64, 10000.0, vp(4096), 16, vp(0))
    assert st == ne.NE_ERR_INVALID_ARG and "workspace" in lib.ne_last_error().decode()
    q = vp(4096 + 8)
    st = lib.ne_attn_bwd(q, p, p, p, p, p, p, p, p, 1, 8, 4, 2, 64, 10000.0, vp(4096), 1 << 20, vp(0))
    assert st == ne.NE_ERR_INVALID_ARG and "aligned" in lib.ne_last_error().decode()


# ---------------------------------------------------------------- decode step

def test_decode_workspace_size(lib):
    r256 = lambda x: (x + 255) // 256 * 256
    # One (batch, kv head) and 512 positions: the positions are cut into 8 chunks of 64,
    # so the workspace holds 8 partial rows [D] fp32 and 8 (max, sum) pairs per query head.
    B, T, Hq, Hkv, D = 1, 512, 4, 1, 64
    assert lib.ne_attn_decode_workspace_size(B, T, Hq, Hkv, D) == r256(B * Hq * 8 * D * 4) + B * Hq * 8 * 8
    # 152 sequences x 4 kv heads already give 608 CTAs: one chunk, no workspace.
    assert lib.ne_attn_decode_workspace_size(152, 512, 12, 4, 64) == 0
    assert lib.ne_attn_decode_workspace_size(1, 8, 3, 2, 64) == 0   # Hq % Hkv != 0


@pytest.mark.parametrize("args,expect", [
    ((1, 8, 3, 2, 64), ne.NE_ERR_INVALID_ARG),     # Hq % Hkv
    ((1, 8, 4, 2, 96), ne.NE_ERR_UNSUPPORTED),     # head_dim
    ((1, 0, 4, 2, 64), ne.NE_ERR_INVALID_ARG),     # empty cache: the newest token must be in it
    ((1, (1 << 30) + 1, 4, 2, 64), ne.NE_ERR_INVALID_ARG),  # positions beyond 2^30
    ((70000, 8, 4, 2, 64), ne.NE_ERR_INVALID_ARG), # batch beyond the grid's z extent
])
def test_decode_rejects_bad_shapes_before_any_device_work(lib, args, expect):
    p = ctypes.c_void_p(4096)
    B, T, Hq, Hkv, D = args
    st = lib.ne_attn_decode(p, p, p, p, p, p, B, T, Hq, Hkv, D, 10000.0, p, 1 << 20, ctypes.c_void_p(0))
    assert st == expect and lib.ne_last_error().decode() != ""


def test_decode_rejects_bad_pointers_and_workspace(lib):
    vp = ctypes.c_void_p
    p, null = vp(4096), vp(0)
    assert lib.ne_attn_decode(null, null, null, null, null, null, 0, 8, 4, 2, 64, 10000.0, null, 0, null) == ne.NE_OK
    st = lib.ne_attn_decode(p, p, p, null, p, p, 1, 512, 4, 1, 64, 10000.0, p, 1 << 20, null)
    assert st == ne.NE_ERR_INVALID_ARG and "seq_lens" in lib.ne_last_error().decode()
    st = lib.ne_attn_decode(p, p, p, p, p, p, 1, 512, 4, 1, 64, 10000.0, p, 16, null)
    assert st == ne.NE_ERR_INVALID_ARG and "workspace" in lib.ne_last_error().decode()
    st = lib.ne_attn_decode(vp(4104), p, p, p, p, p, 1, 512, 4, 1, 64, 10000.0, p, 1 << 20, null)
    assert st == ne.NE_ERR_INVALID_ARG and "aligned" in lib.ne_last_error().decode()


# ---------------------------------------------------------------- binding checks (no device work)

def test_binding_rejects_host_tensors_and_bad_shapes(lib):
    import torch
    q = torch.zeros(1, 8, 4, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        ne.attn_fwd(q, k, k)                                   # host tensors never reach the library
    with pytest.raises(ValueError, match="Hkv"):
        ne.attn_fwd(q, torch.zeros(1, 9, 2, 64, dtype=torch.bfloat16), k)
    with pytest.raises(ValueError):
        ne.attn_fwd(q[0], k, k)                                # not [B, T, H, D]


def test_decode_binding_rejects_bad_inputs(lib):
    import torch
    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    kc = torch.zeros(2, 16, 2, 64, dtype=torch.bfloat16)
    lens = torch.tensor([16, 3], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        ne.attn_decode(q, kc, kc, lens)
    with pytest.raises(ValueError, match="T_max"):
        ne.attn_decode(q, kc[:1], kc[:1], lens)                # caches of another batch
    with pytest.raises(ValueError):
        ne.attn_decode(q.unsqueeze(1), kc, kc, lens)           # q must be [B, Hq, D]
