"""GPU parity of the decode step (ne_attn_decode) against the fp64 oracle.

A decode step for a sequence of length L is row L - 1 of the causal attention over its
first L positions, so the oracle is its row-sampled form (attn_qrows) on those
positions, with the new token's query at row L - 1.  Error metric as in the other
parity tests: relative Frobenius error of O over the whole call.  Bounds: O <= 5e-3 for
bf16 and 1e-3 for f32 (the same bars as the forward).  LSE <= 1e-3 absolute: the step
has no low-precision operand (q and the cache are widened to fp32, rotated and reduced
in fp32), so its LSE error is fp32 rounding of logits of a few units.
"""
import math

import numpy as np
import pytest
import torch

import causal_gqa_flash_attention_gb300 as ne
from causal_gqa_flash_attention_gb300 import _build, synthetic

pytestmark = pytest.mark.gpu

TOL_O = {torch.bfloat16: 5e-3, torch.float32: 1e-3}
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    ne.load()


def rel(x, ref):
    return float(np.linalg.norm((x - ref).ravel()) / np.linalg.norm(ref.ravel()))


def oracle_decode(q, k, v, lens, theta=10000.0):
    """Row L-1 of the causal attention over positions 0..L-1 of each sequence."""
    import oracle
    B, Hq, D = q.shape
    o = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    for b in range(B):
        L = int(lens[b])
        qf = torch.zeros((1, L, Hq, D), dtype=torch.float64)
        qf[0, L - 1] = q[b].double()
        kb, vb = k[b:b + 1, :L], v[b:b + 1, :L]
        for h in range(Hq):
            ob, lb, _, _ = oracle.attn_qrows(qf, kb, vb, None, 0, h, [L - 1], theta)
            o[b, h], lse[b, h] = ob[0], lb[0]
    return o, lse


def run_decode(q, k, v, lens, theta=10000.0):
    o, lse = ne.attn_decode(q.cuda(), k.cuda(), v.cuda(), lens.cuda(), theta)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def check(q, k, v, lens, dtype):
    o, lse = run_decode(q, k, v, lens)
    o_ref, lse_ref = oracle_decode(q, k, v, lens)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    err = {"o": rel(o, o_ref), "lse_abs": float(np.max(np.abs(lse - lse_ref)))}
    print(err)
    assert err["o"] <= TOL_O[dtype], err
    assert err["lse_abs"] <= TOL_LSE, err
    return err


@pytest.mark.parametrize("dtype,B,T,Hq,Hkv,D,lens", [
    (torch.bfloat16, 5, 300, 12, 4, 64, [1, 2, 150, 299, 300]),   # G=3, ragged, several chunks
    (torch.bfloat16, 3, 257, 8, 1, 128, [257, 64, 65]),           # G=8: two groups of four heads
    (torch.bfloat16, 2, 130, 6, 6, 64, [130, 1]),                 # G=1 (MHA)
    (torch.bfloat16, 2, 200, 10, 2, 64, [200, 77]),               # G=5: one head per CTA
    (torch.bfloat16, 2, 96, 12, 2, 128, [96, 33]),                # G=6: two groups of three
    (torch.float32, 4, 128, 4, 2, 32, [128, 1, 64, 100]),         # small-CPU-model shape
    (torch.float32, 3, 300, 12, 4, 64, [300, 299, 5]),
], ids=["bf16-g3-ragged", "bf16-d128-g8", "bf16-mha", "bf16-g5", "bf16-d128-g6", "f32-d32", "f32-d64"])
def test_decode_matches_oracle(dtype, B, T, Hq, Hkv, D, lens):
    q, k, v, ln = synthetic.make_decode(B, T, Hq, Hkv, D, dtype, seed=B + T, lens=lens)
    check(q, k, v, ln, dtype)


def test_decode_other_rope_theta():
    q, k, v, ln = synthetic.make_decode(3, 300, 12, 4, 64, torch.bfloat16, seed=41, lens=[300, 17, 1])
    o, lse = ne.attn_decode(q.cuda(), k.cuda(), v.cuda(), ln.cuda(), 500.0)
    torch.cuda.synchronize()
    assert ne.get_device_error() == ne.NE_OK, ne.last_error()
    o_ref, lse_ref = oracle_decode(q, k, v, ln, theta=500.0)
    o = o.double().cpu().numpy()
    assert rel(o, o_ref) <= TOL_O[torch.bfloat16]
    assert float(np.max(np.abs(lse.double().cpu().numpy() - lse_ref))) <= TOL_LSE


def test_decode_single_chunk_wide_batch():
    """152 sequences x 4 kv heads fill the GPU with one chunk each: no merge kernel."""
    assert ne.decode_workspace_size(152, 64, 12, 4, 64) == 0
    q, k, v, ln = synthetic.make_decode(152, 64, 12, 4, 64, torch.bfloat16, seed=7)
    check(q, k, v, ln, torch.bfloat16)


def test_decode_gpu_pipeline_shape_every_row():
    """The GPU-pipeline model (12/4 heads, D 64, context 512), 16 sequences of mixed
    lengths, every (sequence, head) row checked."""
    q, k, v, ln = synthetic.make_decode(16, 512, 12, 4, 64, torch.bfloat16, seed=11)
    check(q, k, v, ln, torch.bfloat16)


def test_decode_long_context():
    q, k, v, ln = synthetic.make_decode(2, 16384, 12, 4, 64, torch.bfloat16, seed=13, lens=[16384, 9001])
    check(q, k, v, ln, torch.bfloat16)


def test_decode_never_reads_past_the_length():
    """Cache rows at and past each length hold NaN; the outputs stay finite and exact."""
    q, k, v, ln = synthetic.make_decode(4, 200, 12, 4, 64, torch.bfloat16, seed=17, lens=[1, 63, 64, 199],
                                        tail=float("nan"))
    check(q, k, v, ln, torch.bfloat16)


def test_decode_is_deterministic():
    q, k, v, ln = synthetic.make_decode(3, 1000, 12, 4, 64, torch.bfloat16, seed=19)
    a = ne.attn_decode(q.cuda(), k.cuda(), v.cuda(), ln.cuda())
    b = ne.attn_decode(q.cuda(), k.cuda(), v.cuda(), ln.cuda())
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_bad_length_is_reported():
    """A length outside [1, T_max] is clamped on the device (no read leaves the cache)
    and reported as an argument error by the next device-error check."""
    q, k, v, _ = synthetic.make_decode(2, 64, 4, 2, 64, torch.bfloat16, seed=23)
    for bad in (0, 65):
        lens = torch.tensor([bad, 10], dtype=torch.int32)
        o, lse = ne.attn_decode(q.cuda(), k.cuda(), v.cuda(), lens.cuda())
        assert ne.get_device_error() == ne.NE_ERR_INVALID_ARG
        assert "seq_lens" in ne.last_error()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert ne.get_device_error() == ne.NE_OK


def test_decode_bad_arguments_raise():
    q, k, v, ln = synthetic.make_decode(2, 64, 4, 2, 64, torch.bfloat16, seed=29)
    with pytest.raises(ValueError):
        ne.attn_decode(q.cuda(), k.cuda(), v.cuda(), ln.long().cuda())
    with pytest.raises(ne.NeError):
        q2, k2, v2, _ = synthetic.make_decode(2, 64, 4, 2, 96, torch.bfloat16, seed=29)
        ne.attn_decode(q2.cuda(), k2.cuda(), v2.cuda(), ln.cuda())
