"""GPU parity of the training pair (ne_attn_fwd_train / ne_attn_bwd_train).

The training forward also leaves the backward's rotated fp16 queries and a zeroed dQ
accumulator in the layer's workspace (bf16, head_dim 32 and 64); the training backward
then skips that work.  The pair must compute what the regular pair computes:

- against the fp64 oracle with the bounds of test_gpu_parity.py (relative Frobenius
  error: bf16 O <= 5e-3, dQ/dK/dV <= 1e-2; TF32 1e-3 / 2e-3; LSE max abs 3e-2 / 3e-3),
  on a workspace filled with 0xFF bytes beforehand (NaN as fp32 and as fp16), so a
  region the forward failed to fill would poison the gradients;
- against the regular pair at the GPU-pipeline shape (B16 T512 Hq12 Hkv4 D64), where
  the two differ only in rounding (the forward is another instantiation; dQ partials
  are summed in a run-dependent order).
"""
import math

import numpy as np
import pytest
import torch

import causal_gqa_flash_attention_gb300 as ne
from causal_gqa_flash_attention_gb300 import _build, synthetic

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: {"o": 5e-3, "grad": 1e-2, "lse": 3e-2}, torch.float32: {"o": 1e-3, "grad": 2e-3, "lse": 3e-3}}


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


def f64(t):
    return t.detach().double().cpu().numpy()


def train_pair(q, k, v, dO, theta=10000.0, poison=True):
    B, T, Hq, Hkv, D = q.shape[0], q.shape[1], q.shape[2], k.shape[2], q.shape[3]
    ws = ne.alloc_workspace(B, T, Hq, Hkv, D, q.device)
    if poison:
        ws.fill_(0xFF)
    o, lse = ne.attn_fwd_train(q, k, v, ws, theta)
    dq, dk, dv = ne.attn_bwd_train(q, k, v, o, lse, dO, ws, theta)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("D,dtype,T", [(64, torch.bfloat16, 300), (32, torch.bfloat16, 200),
                                       (128, torch.bfloat16, 260), (64, torch.float32, 200)])
def test_train_pair_matches_oracle(D, dtype, T):
    import oracle
    B, Hq, Hkv = 2, 6, 2
    q, k, v, dO = synthetic.make_custom(B, T, Hq, Hkv, D, dtype, seed=31)
    o, lse, dq, dk, dv = train_pair(*(t.cuda() for t in (q, k, v, dO)))
    qd, kd, vd, dOd = (f64(t) for t in (q, k, v, dO))
    o_r, lse_r = oracle.attn_fwd(qd, kd, vd)
    dq_r, dk_r, dv_r = oracle.attn_bwd(qd, kd, vd, dOd)
    tol = TOL[dtype]
    errs = {"o": rel(f64(o), o_r), "dq": rel(f64(dq), dq_r), "dk": rel(f64(dk), dk_r), "dv": rel(f64(dv), dv_r),
            "lse": float(np.max(np.abs(f64(lse) - lse_r)))}
    print(D, dtype, T, errs)
    assert errs["o"] <= tol["o"] and errs["lse"] <= tol["lse"], errs
    for n in ("dq", "dk", "dv"):
        assert errs[n] <= tol["grad"], errs


def test_train_pair_many_units_per_cta():
    """384 units (8 and 2 key tiles): every CTA of the training forward stores R Q and
    zeroes dQ' for several units in turn."""
    import oracle
    B, T, Hq, Hkv, D = 4, 320, 48, 8, 64
    q, k, v, dO = synthetic.make_custom(B, T, Hq, Hkv, D, torch.bfloat16, seed=41)
    o, lse, dq, dk, dv = train_pair(*(t.cuda() for t in (q, k, v, dO)))
    qd, kd, vd, dOd = (f64(t) for t in (q, k, v, dO))
    o_r, lse_r = oracle.attn_fwd(qd, kd, vd)
    dq_r, dk_r, dv_r = oracle.attn_bwd(qd, kd, vd, dOd)
    tol = TOL[torch.bfloat16]
    assert rel(f64(o), o_r) <= tol["o"]
    assert float(np.max(np.abs(f64(lse) - lse_r))) <= tol["lse"]
    for a, b in ((dq, dq_r), (dk, dk_r), (dv, dv_r)):
        assert rel(f64(a), b) <= tol["grad"]


def test_train_pair_equals_regular_pair_at_the_gpu_pipeline_shape():
    w = synthetic.WORKLOADS[2]
    q, k, v, dO = (t.cuda() for t in synthetic.make_inputs(w, layer=0))
    o1, l1 = ne.attn_fwd(q, k, v)
    g1 = ne.attn_bwd(q, k, v, o1, l1, dO)
    o2, l2, *g2 = train_pair(q, k, v, dO)
    assert rel(f64(o2), f64(o1)) <= 5e-4
    assert float((l1 - l2).abs().max()) <= 1e-5
    for a, b in zip(g2, g1):
        assert rel(f64(a), f64(b)) <= 1e-3


def test_train_pair_repeated_runs_identical():
    """The bench's path at its shape (B16 T512 Hq12 Hkv4 D64 bf16): O, LSE, dK and dV are
    bit-identical over three runs of the training pair (dQ, summed by reduce-adds in
    whatever order they land, is not compared)."""
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(16, 512, 12, 4, 64, torch.bfloat16, seed=22))
    runs = [train_pair(q, k, v, dO, poison=False) for _ in range(3)]
    for r in runs[1:]:
        for i, name in ((0, "o"), (1, "lse"), (3, "dk"), (4, "dv")):
            assert torch.equal(runs[0][i], r[i]), (name, int((runs[0][i] != r[i]).sum()))


def test_train_forward_fills_the_workspace_for_the_backward():
    """The stored R Q equals the preprocess pass's, and the dQ accumulator is zero."""
    B, T, Hq, Hkv, D = 2, 300, 4, 2, 64
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(B, T, Hq, Hkv, D, torch.bfloat16, seed=5))
    n = ne.workspace_size(B, T, Hq, Hkv, D)
    acc_off = ((B * Hq * T * 4 + 255) // 256) * 256
    q16_off = acc_off + ((B * T * Hq * D * 4 + 255) // 256) * 256
    ws_train = ne.alloc_workspace(B, T, Hq, Hkv, D).fill_(0xFF)
    ne.attn_fwd_train(q, k, v, ws_train)
    ws_reg = ne.alloc_workspace(B, T, Hq, Hkv, D).fill_(0xFF)
    o, lse = ne.attn_fwd(q, k, v)
    ne.attn_bwd(q, k, v, o, lse, dO, workspace=ws_reg)      # its preprocess writes R Q
    torch.cuda.synchronize()
    acc = ws_train[acc_off:acc_off + B * T * Hq * D * 4].view(torch.float32)
    assert torch.count_nonzero(acc).item() == 0
    q16_t = ws_train[q16_off:q16_off + B * T * Hq * D * 2].view(torch.float16)
    q16_r = ws_reg[q16_off:q16_off + B * T * Hq * D * 2].view(torch.float16)
    assert torch.isfinite(q16_t).all()
    # Both round R Q to fp16; the rotations differ only in the order of their roundings.
    assert rel(f64(q16_t), f64(q16_r)) <= 1e-3
    assert n >= q16_off + B * T * Hq * D * 2


def test_train_pair_rejects_a_small_workspace():
    B, T, Hq, Hkv, D = 1, 64, 2, 1, 64
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(B, T, Hq, Hkv, D, torch.bfloat16, seed=2))
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ne.NeError) as e:
        ne.attn_fwd_train(q, k, v, small)
    assert e.value.status == ne.NE_ERR_INVALID_ARG
