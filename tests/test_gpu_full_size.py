"""GPU parity at the workloads' full sizes, on sampled outputs.

Every workload runs forward and backward on the GPU at its full size, through the same
calls and launch configuration the benchmark times.  The fp64 oracle cannot hold these
T x T matrices, so it computes sampled rows one by one from the same definitions
(oracle.attn_qrows / attn_krows, pinned against the full oracle in test_oracle.py):
  - query rows at tile boundaries, the first and the last positions, for the first and the
    last batch row and every query head: O, LSE, dQ;
  - key rows of the first key tiles (0, 1, 63, 64, 127, 128), the middle and the last
    tiles, for the same batch rows and every kv head: dK, dV.  The first key tile is the
    heaviest: its backward loops over every query tile of every head in the group (128
    tiles x 3 heads at T = 16384), so it carries the longest TMEM accumulation and the
    most barrier phases.  At T = 16384 the oracle's pass over every query row costs
    O(T^2 D G) per (batch row, kv head), so the heavy rows are checked for the first
    (batch, kv head) and the last one; the other kv heads keep the tail rows.
The bound is the tolerance of the whole-tensor parity tests applied to the sampled rows:
relative Frobenius error over all sampled rows of an output, bf16 O <= 5e-3 and
dQ/dK/dV <= 1e-2, fp32 (TF32) 1e-3 / 2e-3; LSE max absolute error 3e-2 / 3e-3.

Also here: the backward's fp16 range checks (rotated queries in the preprocess kernel,
dS in the head_dim-64 main kernel) report instead of saturating.
"""
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
    x = np.asarray(x, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30))


def query_rows(T):
    rows = {0, 1, 63, 64, 127, 128, T // 2, T - 129, T - 128, T - 65, T - 64, T - 1}
    return sorted(r for r in rows if 0 <= r < T)


def key_rows(T, heavy=True):
    rows = {T - 1, T - 2, T - 64, T - 65, T - 128, T - 129}
    if heavy:
        rows |= {0, 1, 63, 64, 127, 128, T // 2}
    return sorted(r for r in rows if 0 <= r < T)


def heavy_key_rows(T, B, Hkv, b, g):
    """Whether (b, g) gets the first key tiles: always up to T = 8192, else only the first
    and the last (batch row, kv head)."""
    return T <= 8192 or (b, g) in ((0, 0), (B - 1, Hkv - 1))


def check_workload(w):
    import oracle
    q, k, v, dO = synthetic.make_inputs(w, layer=0)
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    o, lse = ne.attn_fwd(qd, kd, vd, w.theta)
    dq, dk, dv = ne.attn_bwd(qd, kd, vd, o, lse, dOd, w.theta)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()
    B, T, Hq, Hkv, G = w.B, w.T, w.Hq, w.Hkv, w.Hq // w.Hkv
    qr = query_rows(T)
    got = {n: [] for n in ("o", "dq", "dk", "dv")}
    ref = {n: [] for n in ("o", "dq", "dk", "dv")}
    lse_err = 0.0
    for b in sorted({0, B - 1}):
        o_b, lse_b, dq_b = (x[b].double().cpu().numpy() for x in (o, lse, dq))
        dk_b, dv_b = dk[b].double().cpu().numpy(), dv[b].double().cpu().numpy()
        for h in range(Hq):
            o_r, l_r, dq_r, _ = oracle.attn_qrows(q, k, v, dO, b, h, qr, w.theta)
            got["o"].append(o_b[qr, h]); ref["o"].append(o_r)
            got["dq"].append(dq_b[qr, h]); ref["dq"].append(dq_r)
            lse_err = max(lse_err, float(np.max(np.abs(lse_b[h, qr] - l_r))))
        for g in range(Hkv):
            kr = key_rows(T, heavy_key_rows(T, B, Hkv, b, g))
            dk_r, dv_r = oracle.attn_krows(q, k, v, dO, b, g, kr, w.theta)
            got["dk"].append(dk_b[kr, g]); ref["dk"].append(dk_r)
            got["dv"].append(dv_b[kr, g]); ref["dv"].append(dv_r)
    errs = {n: rel(np.concatenate(got[n]), np.concatenate(ref[n])) for n in got}
    errs["lse_abs"] = lse_err
    print(w.name, errs)
    tol = TOL[w.dtype]
    assert errs["o"] <= tol["o"], errs
    assert errs["lse_abs"] <= tol["lse"], errs
    for n in ("dq", "dk", "dv"):
        assert errs[n] <= tol["grad"], errs
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t).all()


@pytest.mark.parametrize("wid", [2, 3, 4, 51, 52, 53, 54])
def test_full_size_workload_sampled_rows(wid):
    check_workload(synthetic.WORKLOADS[wid])


def test_bwd_rotated_query_beyond_fp16_range_is_reported():
    """The preprocess kernel rounds the rotated queries to fp16 for the head_dim-64
    backward; a value beyond 65504 is reported, not saturated."""
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(1, 96, 2, 1, 64, torch.bfloat16, seed=12))
    o, lse = ne.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK
    qbig = q.clone()
    qbig[0, 40, 1, 6] = 1.0e5
    ne.attn_bwd(qbig, k, v, o, lse, dO)
    assert ne.get_device_error() == ne.NE_ERR_INVALID_ARG
    assert "fp16" in ne.last_error()
    assert ne.get_device_error() == ne.NE_OK


def test_bwd_ds_beyond_fp16_range_is_reported():
    """dS = P o (dP - Delta) is an fp16 MMA operand in the head_dim-64 backward; an upstream
    gradient large enough to push it past 65504 is reported, not saturated."""
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(1, 96, 2, 1, 64, torch.bfloat16, seed=13))
    o, lse = ne.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK
    ne.attn_bwd(q, k, v, o, lse, dO * 1.0e6)
    assert ne.get_device_error() == ne.NE_ERR_INVALID_ARG
    assert "fp16" in ne.last_error()
    assert ne.get_device_error() == ne.NE_OK
