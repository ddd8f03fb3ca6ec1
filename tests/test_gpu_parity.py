"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Error metric (per whole output tensor): relative Frobenius error
||X - X_ref||_F / ||X_ref||_F.  Bounds: bf16 inputs O <= 5e-3, dQ/dK/dV <= 1e-2;
fp32 inputs on TF32 tensor cores O <= 1e-3, dQ/dK/dV <= 2e-3.  LSE (natural log,
values ~ ln(t+1) + O(1)) is checked with a max absolute error: 3e-2 for bf16 (the
logits carry the bf16 rounding of the rotated Q', K', ~2^-8 relative, times |logit|
of a few units) and 3e-3 for TF32 (~2^-11 relative).
"""
import math

import numpy as np
import pytest
import torch

import causal_gqa_flash_attention_gb300 as ne
from causal_gqa_flash_attention_gb300 import _build, synthetic

pytestmark = pytest.mark.gpu

TOL = {"bf16": {"o": 5e-3, "grad": 1e-2, "lse": 3e-2}, "f32": {"o": 1e-3, "grad": 2e-3, "lse": 3e-3}}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    ne.load()


def rel(x, ref):
    """Relative Frobenius error; where the reference is (numerically) zero -- e.g. dQ
    and dK at T = 1, a softmax over one key -- the RMS absolute error instead."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    n = max(ref.size, 1)
    den = np.linalg.norm(ref.ravel())
    if den <= 1e-6 * math.sqrt(n):
        return float(np.linalg.norm((x - ref).ravel()) / math.sqrt(n))
    return float(np.linalg.norm((x - ref).ravel()) / den)


def f64(t):
    return t.detach().double().cpu().numpy()


def run_gpu(q, k, v, dO, theta=10000.0, bwd=True):
    dev = "cuda"
    qd, kd, vd, dOd = (t.to(dev).contiguous() for t in (q, k, v, dO))
    o, lse = ne.attn_fwd(qd, kd, vd, theta)
    out = {"o": o, "lse": lse}
    if bwd:
        dq, dk, dv = ne.attn_bwd(qd, kd, vd, o, lse, dOd, theta)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()
    return {kk: f64(vv) for kk, vv in out.items()}


def check(q, k, v, dO, dtype, theta=10000.0, bwd=True):
    import oracle
    got = run_gpu(q, k, v, dO, theta, bwd)
    o_ref, lse_ref = oracle.attn_fwd(f64(q), f64(k), f64(v), theta)
    tol = TOL[dtype]
    errs = {"o": rel(got["o"], o_ref), "lse_abs": float(np.max(np.abs(got["lse"] - lse_ref)))}
    assert np.all(np.isfinite(got["o"])) and np.all(np.isfinite(got["lse"]))
    if bwd:
        dq, dk, dv = oracle.attn_bwd(f64(q), f64(k), f64(v), f64(dO), theta)
        errs.update(dq=rel(got["dq"], dq), dk=rel(got["dk"], dk), dv=rel(got["dv"], dv))
    print(errs)
    assert errs["o"] <= tol["o"], errs
    assert errs["lse_abs"] <= tol["lse"], errs
    if bwd:
        for name in ("dq", "dk", "dv"):
            assert errs[name] <= tol["grad"], errs
    return errs


# ---------------------------------------------------------------- bf16

@pytest.mark.parametrize("B,T,Hq,Hkv,D", [
    (2, 512, 12, 4, 64),     # the GPU-pipeline shape (two batch rows): 4 query tiles
    (1, 300, 4, 2, 64),      # ragged tail
    (2, 129, 4, 4, 64),      # MHA, one row into the second tile
    (1, 127, 6, 2, 64),
    (1, 5, 2, 1, 64),
    (3, 1, 4, 2, 64),        # T = 1: every row attends to itself only
    (1, 600, 4, 1, 64),      # last CTA: second subtile past T while the K/V ring wraps
    (1, 384, 8, 2, 128),     # head_dim 128
    (1, 200, 4, 1, 128),
])
def test_bf16_matches_oracle(B, T, Hq, Hkv, D):
    q, k, v, dO = synthetic.make_custom(B, T, Hq, Hkv, D, torch.bfloat16, seed=B * 1000 + T + D)
    check(q, k, v, dO, "bf16")


def test_bf16_peaky_logits_softmax_stress():
    """Q, K ~ N(0, 3^2) at D=128: logits of tens of units, the max moves often."""
    q, k, v, dO = synthetic.make_custom(1, 640, 4, 1, 128, torch.bfloat16, seed=77, qk_sigma=3.0)
    check(q, k, v, dO, "bf16")


def test_bf16_small_model_shape_workload_inputs():
    """First two batch rows of the GPU-pipeline workload's layer-0 inputs."""
    w = synthetic.WORKLOADS[2]
    q, k, v, dO = synthetic.make_inputs(w, layer=0, batch=slice(0, 2))
    check(q, k, v, dO, "bf16")


def test_bf16_row_zero_and_zero_queries():
    """Row 0 copies v_0 of its kv head; Q = 0 gives the causal running mean of V."""
    B, T, Hq, Hkv, D = 1, 260, 4, 2, 64
    q, k, v, dO = synthetic.make_custom(B, T, Hq, Hkv, D, torch.bfloat16, seed=5)
    got = run_gpu(q, k, v, dO, bwd=False)
    for h in range(Hq):
        np.testing.assert_allclose(got["o"][:, 0, h], f64(v)[:, 0, h // 2], rtol=0, atol=1e-2)
    q0 = torch.zeros_like(q)
    got = run_gpu(q0, k, v, dO, bwd=False)
    running = np.cumsum(f64(v), axis=1) / np.arange(1, T + 1)[None, :, None, None]
    for h in range(Hq):
        assert rel(got["o"][:, :, h], running[:, :, h // 2]) < 5e-3
        np.testing.assert_allclose(got["lse"][:, h], np.log(np.arange(1, T + 1))[None], atol=1e-4)


def test_bf16_deterministic_dk_dv():
    """dK and dV reduce over the group inside one CTA: bit-identical on a rerun."""
    q, k, v, dO = synthetic.make_custom(2, 512, 12, 4, 64, torch.bfloat16, seed=9)
    a = run_gpu(q, k, v, dO)
    b = run_gpu(q, k, v, dO)
    for name in ("o", "lse", "dk", "dv"):
        assert np.array_equal(a[name], b[name]), name


@pytest.mark.parametrize("B,T,Hq,Hkv,D,dtype", [
    (16, 512, 12, 4, 64, torch.bfloat16),
    (16, 512, 12, 4, 64, torch.float32),
    (8, 1024, 16, 4, 128, torch.bfloat16),   # head_dim 128: one Q/dO stage, dQ' staged in chunks
    (4, 2048, 12, 4, 64, torch.float32),     # TF32 backward: stages freed by the transposes' reads
])
def test_repeated_runs_identical(B, T, Hq, Hkv, D, dtype):
    """The GPU-pipeline batch (B16 T512 Hq12 Hkv4 D64) and longer or wider cases: the
    forward's CTAs walk several work units each and the backward's key loops run over
    every query tile of a head group.  O, LSE, dK and dV come out bit-identical over three runs (dQ is summed by
    reduce-adds in whatever order they land and is not compared); a difference between
    runs is a race, whatever its size."""
    q, k, v, dO = synthetic.make_custom(B, T, Hq, Hkv, D, dtype, seed=21)
    runs = [run_gpu(q, k, v, dO) for _ in range(3)]
    for r in runs[1:]:
        for name in ("o", "lse", "dk", "dv"):
            assert np.array_equal(runs[0][name], r[name]), (name, int((runs[0][name] != r[name]).sum()))


@pytest.mark.parametrize("B,T,Hq,Hkv,D,dtype", [
    (8, 64, 64, 8, 64, torch.bfloat16),     # 512 one-tile units: S runs across several units
    (4, 320, 48, 8, 64, torch.bfloat16),    # 384 units of 8 and 2 tiles, ragged second unit
    (6, 100, 64, 16, 32, torch.bfloat16),   # head_dim 32 (run zero-padded to 64)
    (8, 64, 64, 8, 64, torch.float32),
])
def test_many_units_per_cta(B, T, Hq, Hkv, D, dtype):
    """More work units than 2.5 per SM: every CTA of the persistent forward crosses unit
    boundaries several times (the small cases above give a CTA one unit at most), with
    subtiles of one key tile, where the S issue runs furthest ahead of the PV issue."""
    q, k, v, dO = synthetic.make_custom(B, T, Hq, Hkv, D, dtype, seed=B * 10 + T + D)
    check(q, k, v, dO, "bf16" if dtype == torch.bfloat16 else "f32")


# ---------------------------------------------------------------- f32 (TF32)

@pytest.mark.parametrize("B,T,Hq,Hkv,D", [
    (2, 512, 12, 4, 64),     # GPU-pipeline shape, two batch rows
    (1, 77, 4, 1, 64),       # ragged tail
    (1, 300, 6, 2, 32),
    (2, 1, 4, 2, 32),
])
def test_f32_matches_oracle(B, T, Hq, Hkv, D):
    q, k, v, dO = synthetic.make_custom(B, T, Hq, Hkv, D, torch.float32, seed=B * 100 + T + D)
    check(q, k, v, dO, "f32")


def test_f32_small_model_workload_full_size():
    """The small CPU-model workload (B4 T128 Hq4 Hkv2 D32, fp32 on TF32) at full size."""
    q, k, v, dO = synthetic.make_inputs(synthetic.WORKLOADS[1])
    check(q, k, v, dO, "f32")


# ---------------------------------------------------------------- RoPE table

def test_rope_table_matches_fp64():
    import oracle
    for T, D, theta in ((16384, 64, 10000.0), (300, 128, 10000.0), (5, 2, 10000.0), (1000, 64, 500.0)):
        c, s = ne.rope_table(T, D, theta)
        cr, sr = oracle.rope_table(T, D, theta)
        assert np.max(np.abs(f64(c) - cr)) < 1e-7
        assert np.max(np.abs(f64(s) - sr)) < 1e-7


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_other_rope_theta_matches_oracle(dtype):
    """theta is an argument of every call: at theta = 500 the forward and backward match
    the oracle at theta = 500 (and differ from theta = 10000 by far more than the bars)."""
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v, dO = synthetic.make_custom(2, 200, 6, 2, 64, dt, seed=37)
    check(q, k, v, dO, dtype, theta=500.0)


# ---------------------------------------------------------------- error paths

def test_bounded_wait_times_out_and_reports():
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()
    ne.selftest_wait_timeout(20)
    assert ne.get_device_error() == ne.NE_ERR_DEVICE_TIMEOUT
    assert "bounded wait" in ne.last_error()
    assert ne.get_device_error() == ne.NE_OK   # cleared
    # the context is still usable
    q, k, v, dO = synthetic.make_custom(1, 64, 2, 1, 64, torch.bfloat16, seed=3)
    check(q, k, v, dO, "bf16")


def test_rotated_values_beyond_fp16_range_are_reported():
    """The bf16 path rounds rotated q/k to fp16 for the logits; a value beyond 65504
    must not pass silently."""
    q, k, v, dO = synthetic.make_custom(1, 64, 2, 1, 64, torch.bfloat16, seed=4)
    q[0, 3, 1, 10] = 1.0e5
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ne.attn_fwd(qd, kd, vd)
    assert ne.get_device_error() == ne.NE_ERR_INVALID_ARG
    assert "fp16" in ne.last_error()
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()


def test_bad_arguments_raise():
    q = torch.zeros(1, 8, 3, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ne.NeError) as ei:
        ne.attn_fwd(q, k, k)
    assert ei.value.status == ne.NE_ERR_INVALID_ARG


# ---------------------------------------------------------------- bf16, head_dim 32
# The small model's head size (dim 128 with 4 query heads, "NanoEuler: C와 CUDA로 밑바닥부터
# 구축한 GPT-2 규모의 LLM", 모델 구성).  It runs on the head_dim-64 kernels with the upper
# 32 columns zero, so these cases also pin that the padding never reaches an output row.
@pytest.mark.parametrize("T", [1, 5, 128, 129, 300])
def test_bf16_d32_small_model_heads_ragged_T(T):
    q, k, v, dO = synthetic.make_custom(2, T, 4, 2, 32, torch.bfloat16, seed=41 + T)
    check(q, k, v, dO, "bf16")


def test_bf16_d32_theta_500_and_gqa_group_4():
    q, k, v, dO = synthetic.make_custom(1, 257, 8, 2, 32, torch.bfloat16, seed=43)
    check(q, k, v, dO, "bf16", theta=500.0)


def test_bf16_d32_does_not_write_past_its_rows():
    """Outputs are [.., 32] wide; a store of the 64-wide kernel's padded columns would
    overwrite the next head's row.  Surround the outputs with a canary and check it."""
    B, T, Hq, Hkv, D = 1, 130, 3, 1, 32
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(B, T, Hq, Hkv, D, torch.bfloat16, seed=44))
    canary = 7.0
    big = torch.full((B * T * Hq * D + 64,), canary, dtype=torch.bfloat16, device="cuda")
    o = big[:B * T * Hq * D].view(B, T, Hq, D)
    o2, lse = ne.attn_fwd(q, k, v, o=o)
    dq_buf = torch.full((B * T * Hq * D + 64,), canary, dtype=torch.bfloat16, device="cuda")
    dk_buf = torch.full((B * T * Hkv * D + 64,), canary, dtype=torch.bfloat16, device="cuda")
    dv_buf = torch.full((B * T * Hkv * D + 64,), canary, dtype=torch.bfloat16, device="cuda")
    ne.attn_bwd(q, k, v, o2, lse, dO, dq=dq_buf[:B * T * Hq * D].view(B, T, Hq, D),
                dk=dk_buf[:B * T * Hkv * D].view(B, T, Hkv, D), dv=dv_buf[:B * T * Hkv * D].view(B, T, Hkv, D))
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()
    for buf, n in ((big, B * T * Hq * D), (dq_buf, B * T * Hq * D), (dk_buf, B * T * Hkv * D),
                   (dv_buf, B * T * Hkv * D)):
        assert torch.all(buf[n:] == canary)
