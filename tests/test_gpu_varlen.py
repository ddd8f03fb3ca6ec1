"""GPU parity of the variable-length calls (ne_attn_fwd_varlen / ne_attn_bwd_varlen).

A padded batch holds sequences of different lengths; sequence b occupies positions
0 .. len_b - 1 of row b and the rest is padding (the SFT batches of "NanoEuler: C와
CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM", 2단계 학습 프로세스).  Each sequence's valid
outputs are checked against the fp64 oracle run on that sequence alone (T = len_b), with
the bounds of the other parity tests (relative Frobenius error over all valid rows of an
output: bf16 O <= 5e-3, dQ/dK/dV <= 1e-2; fp32 on TF32 1e-3 / 2e-3; LSE max abs error
3e-2 / 3e-3).  Padding outputs must be exactly zero (O, dQ, dK, dV) and LSE -inf.  The
padding of q and k holds large finite values and that of v and dO ordinary ones, so a
padding value that leaked into a valid output would show.
"""
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


def padded_inputs(B, T, Hq, Hkv, D, dtype, lens, seed):
    """Inputs whose padding holds values that must not matter: q and k padding is large
    (beyond the fp16 range once rotated, if it were used), v and dO padding is N(0, 1)."""
    q, k, v, dO = synthetic.make_custom(B, T, Hq, Hkv, D, dtype, seed=seed)
    for b, L in enumerate(lens):
        q[b, L:] = 1.0e5
        k[b, L:] = -1.0e5
    return q, k, v, dO


def check_varlen(B, T, Hq, Hkv, D, dtype, lens, seed=7):
    import oracle
    lens = list(lens)
    assert len(lens) == B
    q, k, v, dO = padded_inputs(B, T, Hq, Hkv, D, dtype, lens, seed)
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = ne.attn_fwd_varlen(qd, kd, vd, sl)
    dq, dk, dv = ne.attn_bwd_varlen(qd, kd, vd, o, lse, dOd, sl)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()
    f = lambda t: t.double().cpu().numpy()
    got = {n: [] for n in ("o", "dq", "dk", "dv")}
    ref = {n: [] for n in ("o", "dq", "dk", "dv")}
    lse_err = 0.0
    for b, L in enumerate(lens):
        # Padding: exact zeros and -inf.
        for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
            assert torch.count_nonzero(t[b, L:]).item() == 0, (name, b, L)
        assert torch.all(torch.isneginf(lse[b, :, L:])), (b, L)
        if L == 0:
            continue
        sq, sk, sv, sdo = (f(t[b:b + 1, :L]) for t in (q, k, v, dO))
        o_r, lse_r = oracle.attn_fwd(sq, sk, sv)
        dq_r, dk_r, dv_r = oracle.attn_bwd(sq, sk, sv, sdo)
        got["o"].append(f(o[b:b + 1, :L])); ref["o"].append(o_r)
        got["dq"].append(f(dq[b:b + 1, :L])); ref["dq"].append(dq_r)
        got["dk"].append(f(dk[b:b + 1, :L])); ref["dk"].append(dk_r)
        got["dv"].append(f(dv[b:b + 1, :L])); ref["dv"].append(dv_r)
        lse_err = max(lse_err, float(np.max(np.abs(f(lse[b:b + 1, :, :L]) - lse_r))))
    errs = {n: rel(np.concatenate([x.ravel() for x in got[n]]), np.concatenate([x.ravel() for x in ref[n]]))
            for n in got}
    errs["lse_abs"] = lse_err
    print(dtype, D, lens, errs)
    tol = TOL[dtype]
    assert errs["o"] <= tol["o"], errs
    assert errs["lse_abs"] <= tol["lse"], errs
    for n in ("dq", "dk", "dv"):
        assert errs[n] <= tol["grad"], errs


def test_varlen_bf16_d64_ragged_lengths():
    """Lengths 1, 5, 129, 300 and 512 in one batch of T = 512 (several tiles, ragged
    tails, a one-token sequence and a full one)."""
    check_varlen(5, 512, 6, 2, 64, torch.bfloat16, [1, 5, 129, 300, 512])


def test_varlen_bf16_d64_gpu_pipeline_heads_with_empty_sequence():
    check_varlen(4, 384, 12, 4, 64, torch.bfloat16, [0, 383, 64, 256])


def test_varlen_bf16_d64_many_units_per_cta():
    """Sixteen sequences of mixed lengths over 48 heads: 576 units, several per CTA,
    among them empty subtiles and one-tile subtiles, so the persistent forward's S issue
    crosses unit boundaries ahead of its PV issue many times."""
    lens = [1, 64, 65, 300, 320, 0, 129, 200, 17, 256, 257, 320, 64, 90, 310, 2]
    check_varlen(16, 320, 48, 8, 64, torch.bfloat16, lens)


def test_varlen_bf16_d128():
    check_varlen(4, 256, 8, 2, 128, torch.bfloat16, [1, 77, 200, 256])


def test_varlen_f32_d64_tf32():
    check_varlen(4, 200, 6, 3, 64, torch.float32, [3, 64, 130, 200])


def test_varlen_f32_d32_tf32():
    check_varlen(3, 128, 4, 2, 32, torch.float32, [1, 100, 128])


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.bfloat16, 128), (torch.float32, 64)])
def test_varlen_with_every_length_full_equals_the_regular_call(dtype, D):
    """With every length equal to T the variable-length calls compute what the regular
    calls compute, within rounding: they run another instantiation of the same kernels,
    whose instruction scheduling may round a product of the first (diagonal) tile
    differently (measured: O to one unit in the last place of its type, LSE to 1.3e-7);
    the backward's dQ partials are summed in an order that varies between runs."""
    B, T, Hq, Hkv = 2, 300, 4, 2
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(B, T, Hq, Hkv, D, dtype, seed=21))
    sl = torch.full((B,), T, dtype=torch.int32, device="cuda")
    o1, l1 = ne.attn_fwd(q, k, v)
    o2, l2 = ne.attn_fwd_varlen(q, k, v, sl)
    g1 = ne.attn_bwd(q, k, v, o1, l1, dO)
    g2 = ne.attn_bwd_varlen(q, k, v, o1, l1, dO, sl)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK
    assert rel(o2.double().cpu(), o1.double().cpu()) <= 5e-4
    assert float((l1 - l2).abs().max()) <= 1e-5
    for a, b in zip(g1, g2):
        assert rel(a.double().cpu(), b.double().cpu()) <= 1e-3


def test_varlen_bad_length_is_reported():
    B, T, Hq, Hkv, D = 2, 64, 2, 1, 64
    q, k, v, dO = (t.cuda() for t in synthetic.make_custom(B, T, Hq, Hkv, D, torch.bfloat16, seed=5))
    sl = torch.tensor([T + 5, 10], dtype=torch.int32, device="cuda")
    ne.attn_fwd_varlen(q, k, v, sl)
    assert ne.get_device_error() == ne.NE_ERR_INVALID_ARG
    assert "seq_lens" in ne.last_error()
    assert ne.get_device_error() == ne.NE_OK
