"""Pins for the fp64 oracle (CPU only).

Each test checks the oracle against something other than itself: central finite
differences (the pages' own validation method: "NanoEuler: C와 CUDA로 밑바닥부터
구축한 GPT-2 규모의 LLM", 검증 및 안정성), closed forms worked out by hand, invariants
of softmax and of rotations, and a library routine (PyTorch's fp64 scaled-dot-product
attention with autograd) on inputs rotated by an independent complex-number
formulation of RoPE.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from causal_gqa_flash_attention_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("shape", [(1, 5, 4, 2, 4), (2, 7, 3, 1, 6), (1, 1, 2, 1, 2), (1, 6, 2, 2, 2)])
def test_backward_matches_central_finite_differences(oracle_mod, shape):
    """Analytic dQ/dK/dV of L = <dO, O> against central differences in fp64, every
    input element perturbed (the pages' gradient-check method)."""
    B, T, Hq, Hkv, D = shape
    q = _rand((B, T, Hq, D), 1)
    k = _rand((B, T, Hkv, D), 2)
    v = _rand((B, T, Hkv, D), 3)
    dO = _rand((B, T, Hq, D), 4)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, dO)

    def loss(q_, k_, v_):
        o, _ = oracle_mod.attn_fwd(q_, k_, v_)
        return float(np.sum(o * dO))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp = x.copy(); xp[i] += h
            xm = x.copy(); xm[i] -= h
            args_p = {"q": q, "k": k, "v": v}; args_p[name] = xp
            args_m = {"q": q, "k": k, "v": v}; args_m[name] = xm
            fd[i] = (loss(**{k_ + "_": a for k_, a in args_p.items()})
                     - loss(**{k_ + "_": a for k_, a in args_m.items()})) / (2 * h)
        err = np.max(np.abs(fd - g)) / max(1.0, np.max(np.abs(g)))
        assert err <= 1e-7, (name, err)


# ---------------------------------------------------------------- softmax invariants

def test_probability_rows_sum_to_one_and_mask_is_exact_zero(oracle_mod):
    B, T, Hq, Hkv, D = 2, 37, 4, 2, 8
    q, k, v = _rand((B, T, Hq, D), 5), _rand((B, T, Hkv, D), 6), _rand((B, T, Hkv, D), 7)
    _, lse, P = oracle_mod.attn_fwd(q, k, v, return_probs=True)
    np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)
    upper = np.triu(np.ones((T, T), bool), k=1)
    assert np.all(P[..., upper] == 0.0)
    assert np.all(P[..., ~upper] > 0.0)
    # LSE is a log-partition: P_ij = exp(S_ij - LSE_i) implies LSE_i >= max_j S_ij.
    assert np.all(np.isfinite(lse))


def test_row_zero_attends_only_to_itself(oracle_mod):
    """Row 0 has a single key: O_0 = v_0 of its kv head, LSE_0 = s q_0.k_0 (R_0 = I),
    and dQ_0 = 0 (a softmax over one element has zero gradient)."""
    B, T, Hq, Hkv, D = 3, 9, 6, 2, 8
    G = Hq // Hkv
    q, k, v = _rand((B, T, Hq, D), 8), _rand((B, T, Hkv, D), 9), _rand((B, T, Hkv, D), 10)
    dO = _rand((B, T, Hq, D), 11)
    o, lse = oracle_mod.attn_fwd(q, k, v)
    dq, _, _ = oracle_mod.attn_bwd(q, k, v, dO)
    s = 1 / math.sqrt(D)
    for h in range(Hq):
        assert np.array_equal(o[:, 0, h], v[:, 0, h // G])
        np.testing.assert_allclose(lse[:, h, 0], s * np.sum(q[:, 0, h] * k[:, 0, h // G], -1),
                                   rtol=1e-14, atol=1e-14)
    assert np.max(np.abs(dq[:, 0])) <= 1e-15


def test_zero_queries_give_causal_running_mean(oracle_mod):
    """Q = 0 makes every logit 0: O_i = mean_{j<=i} V_j and LSE_i = ln(i+1)."""
    B, T, Hq, Hkv, D = 2, 23, 4, 1, 6
    q = np.zeros((B, T, Hq, D))
    k, v = _rand((B, T, Hkv, D), 12), _rand((B, T, Hkv, D), 13)
    o, lse = oracle_mod.attn_fwd(q, k, v)
    running = np.cumsum(v, axis=1) / np.arange(1, T + 1)[None, :, None, None]
    for h in range(Hq):
        np.testing.assert_allclose(o[:, :, h], running[:, :, 0], rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse[:, h], np.broadcast_to(np.log(np.arange(1, T + 1)), (B, T)), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- RoPE

def test_rope_table_hand_values(oracle_mod):
    """theta = 10000, D = 8: the pair frequencies are 1, 1/10, 1/100, 1/1000, so the
    angle is exactly 1 rad at (t=1, i=0), (t=10, i=1), (t=100, i=2), (t=1000, i=3)."""
    c, s = oracle_mod.rope_table(1001, 8, 10000.0)
    for t, i in ((1, 0), (10, 1), (100, 2), (1000, 3)):
        assert abs(c[t, i] - math.cos(1.0)) < 1e-13 and abs(s[t, i] - math.sin(1.0)) < 1e-13
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)


def test_rope_pairs_are_adjacent_and_rotate_counterclockwise(oracle_mod):
    """R_t e_{2i} = (cos, sin) on (2i, 2i+1); R_t e_{2i+1} = (-sin, cos)."""
    D, T = 8, 4
    c, s = oracle_mod.rope_table(T, D)
    for i in range(D // 2):
        for col, expect in ((2 * i, lambda t: (c[t, i], s[t, i])), (2 * i + 1, lambda t: (-s[t, i], c[t, i]))):
            x = np.zeros((1, T, 1, D)); x[..., col] = 1.0
            y = oracle_mod.rope_apply(x)
            for t in range(T):
                e0, e1 = expect(t)
                assert abs(y[0, t, 0, 2 * i] - e0) < 1e-15 and abs(y[0, t, 0, 2 * i + 1] - e1) < 1e-15
                others = np.delete(y[0, t, 0], [2 * i, 2 * i + 1])
                assert np.all(others == 0.0)


def test_rope_preserves_norms_and_depends_only_on_offset(oracle_mod):
    D, T = 16, 40
    x = _rand((2, T, 3, D), 14)
    y = oracle_mod.rope_apply(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-14)
    qv, kv = _rand(D, 15), _rand(D, 16)
    for (i, j, c) in ((3, 1, 5), (7, 7, 30), (20, 2, 11)):
        buf_q = np.zeros((1, T, 1, D)); buf_k = np.zeros((1, T, 1, D))
        buf_q[0, i, 0] = qv; buf_q[0, i + c, 0] = qv
        buf_k[0, j, 0] = kv; buf_k[0, j + c, 0] = kv
        rq, rk = oracle_mod.rope_apply(buf_q), oracle_mod.rope_apply(buf_k)
        a = rq[0, i, 0] @ rk[0, j, 0]
        b = rq[0, i + c, 0] @ rk[0, j + c, 0]
        assert abs(a - b) <= 1e-12 * max(1.0, abs(a))


# ---------------------------------------------------------------- hand case

def test_hand_case_two_positions_two_dims(oracle_mod):
    """T=2, D=2, one head; with D=2 the only pair frequency is 1, so R_1 rotates by
    1 rad.  q_1 = (1,0), k_0 = (1,0), k_1 = (0,1):
      a = s (R_1 q_1).(R_0 k_0) = s cos 1,  b = s (R_1 q_1).(R_1 k_1) = s q_1.k_1 = 0,
      O_1 = (e^a v_0 + e^b v_1) / (e^a + e^b),  LSE_1 = ln(e^a + e^b)."""
    s = 1 / math.sqrt(2)
    q = np.array([2.0, 3.0, 1.0, 0.0]).reshape(1, 2, 1, 2)
    k = np.array([1.0, 0.0, 0.0, 1.0]).reshape(1, 2, 1, 2)
    v = np.array([1.0, 2.0, 3.0, -1.0]).reshape(1, 2, 1, 2)
    o, lse = oracle_mod.attn_fwd(q, k, v)
    a, b = s * math.cos(1.0), 0.0
    o1 = (math.exp(a) * v[0, 0, 0] + math.exp(b) * v[0, 1, 0]) / (math.exp(a) + math.exp(b))
    np.testing.assert_allclose(o[0, 1, 0], o1, rtol=1e-14)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], rtol=0)
    assert abs(lse[0, 0, 1] - math.log(math.exp(a) + math.exp(b))) < 1e-14
    assert abs(lse[0, 0, 0] - s * 2.0) < 1e-15


# ---------------------------------------------------------------- GQA

def test_gqa_equals_mha_with_repeated_kv(oracle_mod):
    """Query head h reads kv head h // G: GQA equals MHA on K/V repeated G times along
    the head axis, and the GQA dK/dV are the group sums of the MHA ones."""
    B, T, Hq, Hkv, D = 2, 19, 6, 2, 8
    G = Hq // Hkv
    q, k, v = _rand((B, T, Hq, D), 17), _rand((B, T, Hkv, D), 18), _rand((B, T, Hkv, D), 19)
    dO = _rand((B, T, Hq, D), 20)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    o1, l1 = oracle_mod.attn_fwd(q, k, v)
    o2, l2 = oracle_mod.attn_fwd(q, kr, vr)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    dq1, dk1, dv1 = oracle_mod.attn_bwd(q, k, v, dO)
    dq2, dk2, dv2 = oracle_mod.attn_bwd(q, kr, vr, dO)
    np.testing.assert_allclose(dq1, dq2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dk1, dk2.reshape(B, T, Hkv, G, D).sum(3), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dv1, dv2.reshape(B, T, Hkv, G, D).sum(3), rtol=1e-12, atol=1e-12)


def test_delta_is_rowsum_of_dO_times_O(oracle_mod):
    """The oracle forms Delta_i = sum_j P_ij dP_ij; it must equal dO_i . O_i."""
    B, T, Hq, Hkv, D = 2, 21, 4, 2, 8
    q, k, v = _rand((B, T, Hq, D), 21), _rand((B, T, Hkv, D), 22), _rand((B, T, Hkv, D), 23)
    dO = _rand((B, T, Hq, D), 24)
    o, _ = oracle_mod.attn_fwd(q, k, v)
    *_, delta = oracle_mod.attn_bwd(q, k, v, dO, return_delta=True)
    np.testing.assert_allclose(delta, np.einsum("bthd,bthd->bht", dO, o), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- library cross-check

def _rope_complex(x: torch.Tensor, theta: float) -> torch.Tensor:
    """Independent RoPE: view adjacent pairs as complex numbers and multiply by
    exp(i t w_j), w_j = theta^(-2j/D)."""
    B, T, H, D = x.shape
    w = theta ** (-torch.arange(0, D, 2, dtype=torch.float64) / D)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * w[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[None, :, None, :]
    z = torch.view_as_complex(x.reshape(B, T, H, D // 2, 2).contiguous())
    return torch.view_as_real(z * rot).reshape(B, T, H, D)


def test_rope_theta_is_a_parameter(oracle_mod):
    """theta = 16, D = 4: the pair frequencies are 1 and 16^(-1/2) = 1/4, so the angle
    of pair 1 is exactly 1 rad at t = 4; and attention at theta = 500 matches PyTorch's
    fp64 attention on inputs rotated independently at theta = 500."""
    c, s = oracle_mod.rope_table(5, 4, 16.0)
    assert abs(c[4, 1] - math.cos(1.0)) < 1e-15 and abs(s[4, 1] - math.sin(1.0)) < 1e-15
    assert abs(c[3, 0] - math.cos(3.0)) < 1e-15
    B, T, Hq, Hkv, D = 1, 21, 4, 2, 8
    gen = torch.Generator().manual_seed(41)
    q = torch.randn(B, T, Hq, D, generator=gen, dtype=torch.float64)
    k = torch.randn(B, T, Hkv, D, generator=gen, dtype=torch.float64)
    v = torch.randn(B, T, Hkv, D, generator=gen, dtype=torch.float64)
    qr, kr = _rope_complex(q, 500.0), _rope_complex(k, 500.0)
    to_bhtd = lambda t: t.permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(
        to_bhtd(qr), to_bhtd(kr.repeat_interleave(2, 2)), to_bhtd(v.repeat_interleave(2, 2)),
        is_causal=True).permute(0, 2, 1, 3)
    o, _ = oracle_mod.attn_fwd(q.numpy(), k.numpy(), v.numpy(), 500.0)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-11, atol=1e-12)
    o_default, _ = oracle_mod.attn_fwd(q.numpy(), k.numpy(), v.numpy())
    assert np.max(np.abs(o_default - o)) > 1e-3      # theta changes the result


@pytest.mark.parametrize("shape", [(2, 33, 6, 2, 16), (1, 64, 4, 4, 32), (1, 17, 12, 4, 64)])
def test_matches_torch_sdpa_fp64_with_autograd(oracle_mod, shape):
    B, T, Hq, Hkv, D = shape
    G = Hq // Hkv
    gen = torch.Generator().manual_seed(sum(shape))
    q = torch.randn(B, T, Hq, D, generator=gen, dtype=torch.float64, requires_grad=True)
    k = torch.randn(B, T, Hkv, D, generator=gen, dtype=torch.float64, requires_grad=True)
    v = torch.randn(B, T, Hkv, D, generator=gen, dtype=torch.float64, requires_grad=True)
    dO = torch.randn(B, T, Hq, D, generator=gen, dtype=torch.float64)
    qr, kr = _rope_complex(q, 10000.0), _rope_complex(k, 10000.0)
    to_bhtd = lambda t: t.permute(0, 2, 1, 3)
    o = torch.nn.functional.scaled_dot_product_attention(
        to_bhtd(qr), to_bhtd(kr.repeat_interleave(G, 2)), to_bhtd(v.repeat_interleave(G, 2)),
        is_causal=True).permute(0, 2, 1, 3)
    (o * dO).sum().backward()
    o_ref, _ = oracle_mod.attn_fwd(q.detach().numpy(), k.detach().numpy(), v.detach().numpy())
    dq, dk, dv = oracle_mod.attn_bwd(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(),
                                     dO.numpy())
    np.testing.assert_allclose(o_ref, o.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-10, atol=1e-11)


# ---------------------------------------------------------------- stored fixture

def test_golden_fixture_unchanged(oracle_mod):
    """Regression pin: values written by tests/golden/make_golden.py (oracle only)."""
    with open(os.path.join(GOLDEN, "oracle_tiny_B1_T5_Hq4_Hkv2_D4.json")) as f:
        g = json.load(f)
    arr = {k: np.array(v, dtype=np.float64) for k, v in g["arrays"].items()}
    o, lse = oracle_mod.attn_fwd(arr["q"], arr["k"], arr["v"], g["theta"])
    dq, dk, dv = oracle_mod.attn_bwd(arr["q"], arr["k"], arr["v"], arr["dO"], g["theta"])
    for name, val in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(val, arr[name], rtol=1e-12, atol=1e-13, err_msg=name)


def test_empty_sequence_and_bad_shapes(oracle_mod):
    q = np.zeros((2, 0, 4, 8)); k = np.zeros((2, 0, 2, 8))
    o, lse = oracle_mod.attn_fwd(q, k, k)
    assert o.shape == (2, 0, 4, 8) and lse.shape == (2, 4, 0)
    with pytest.raises(ValueError):
        oracle_mod.attn_fwd(np.zeros((1, 3, 3, 8)), np.zeros((1, 3, 2, 8)), np.zeros((1, 3, 2, 8)))


def test_synthetic_inputs_are_seeded_and_rounded():
    w = synthetic.WORKLOADS[1]
    a = synthetic.make_inputs(w)
    b = synthetic.make_inputs(w)
    for x, y in zip(a, b):
        assert torch.equal(x, y) and x.dtype == torch.float32
    w4 = synthetic.WORKLOADS[4]
    small = synthetic.Workload(4, "t", 1, 8, 4, 2, 16, "bf16", qk_sigma=3.0)
    q, k, v, dO = synthetic.make_inputs(small)
    assert q.dtype == torch.bfloat16 and w4.qk_sigma == 3.0
    assert 2.0 < float(q.float().std()) < 4.0 and 0.5 < float(v.float().std()) < 1.5


@pytest.mark.parametrize("shape", [(2, 37, 6, 2, 8), (1, 70, 4, 4, 64), (1, 130, 3, 1, 32)])
def test_row_sampled_oracle_matches_full_oracle(oracle_mod, shape):
    """The row-by-row forms (used where the full matrices do not fit) give the full
    oracle's values: O, LSE, dQ, Delta for query rows, dK, dV for key rows."""
    B, T, Hq, Hkv, D = shape
    rng = np.random.default_rng(sum(shape))
    q, dO = rng.standard_normal((B, T, Hq, D)), rng.standard_normal((B, T, Hq, D))
    k, v = rng.standard_normal((B, T, Hkv, D)), rng.standard_normal((B, T, Hkv, D))
    o, lse = oracle_mod.attn_fwd(q, k, v)
    dq, dk, dv, delta = oracle_mod.attn_bwd(q, k, v, dO, return_delta=True)
    qrows = [0, T - 1, T // 2, 1]
    krows = [T - 1, 0, T // 3]
    for b in range(B):
        for h in range(Hq):
            o2, l2, dq2, d2 = oracle_mod.attn_qrows(q, k, v, dO, b, h, qrows)
            np.testing.assert_allclose(o2, o[b, qrows, h], rtol=0, atol=1e-12)
            np.testing.assert_allclose(l2, lse[b, h, qrows], rtol=0, atol=1e-12)
            np.testing.assert_allclose(dq2, dq[b, qrows, h], rtol=0, atol=1e-12)
            np.testing.assert_allclose(d2, delta[b, h, qrows], rtol=0, atol=1e-12)
            o3, l3, dq3, d3 = oracle_mod.attn_qrows(q, k, v, None, b, h, qrows)
            assert dq3 is None and d3 is None and np.array_equal(o3, o2)
        for g in range(Hkv):
            dk2, dv2 = oracle_mod.attn_krows(q, k, v, dO, b, g, krows)
            np.testing.assert_allclose(dk2, dk[b, krows, g], rtol=0, atol=1e-12)
            np.testing.assert_allclose(dv2, dv[b, krows, g], rtol=0, atol=1e-12)


def test_row_sampled_oracle_zero_queries_closed_form(oracle_mod):
    """With Q = 0 each query row averages the values at and before it: O_i is the causal
    running mean of V and LSE_i = ln(i + 1), independently of the full oracle."""
    T, D = 300, 16
    rng = np.random.default_rng(3)
    q = np.zeros((1, T, 2, D)); k = rng.standard_normal((1, T, 1, D)); v = rng.standard_normal((1, T, 1, D))
    rows = [0, 1, 149, 299]
    o, lse, _, _ = oracle_mod.attn_qrows(q, k, v, None, 0, 1, rows)
    running = np.cumsum(v[0, :, 0], axis=0) / np.arange(1, T + 1)[:, None]
    np.testing.assert_allclose(o, running[rows], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(np.asarray(rows) + 1.0), rtol=0, atol=1e-13)


def test_decode_reading_is_a_row_of_the_causal_attention(oracle_mod):
    """The decode step's reference: for a sequence of length L, the newest token's output
    is row L-1 of the causal attention.  The row-sampled oracle on the first L positions
    gives the full oracle's row L-1.  Positions after L-1 do not change that row, so a
    longer cache with arbitrary later rows gives the same result."""
    B, T, Hq, Hkv, D = 1, 50, 6, 2, 16
    rng = np.random.default_rng(31)
    q = rng.standard_normal((B, T, Hq, D))
    k, v = rng.standard_normal((B, T, Hkv, D)), rng.standard_normal((B, T, Hkv, D))
    o_full, lse_full = oracle_mod.attn_fwd(q, k, v)
    for L in (1, 2, 17, 50):
        o_pre, lse_pre = oracle_mod.attn_fwd(q[:, :L], k[:, :L], v[:, :L])
        for h in range(Hq):
            o_row, l_row, _, _ = oracle_mod.attn_qrows(q[:, :L], k[:, :L], v[:, :L], None, 0, h, [L - 1])
            np.testing.assert_allclose(o_row[0], o_pre[0, L - 1, h], rtol=0, atol=1e-13)
            np.testing.assert_allclose(o_row[0], o_full[0, L - 1, h], rtol=0, atol=1e-13)
            assert abs(l_row[0] - lse_full[0, h, L - 1]) < 1e-13 and abs(lse_pre[0, h, L - 1] - l_row[0]) < 1e-13


# ---------------------------------------------------------------- RMSNorm -> QKV -> RoPE prologue

def test_prologue_rows_have_unit_rms_and_ignore_the_row_scale(oracle_mod):
    """With a unit gain, an identity projection and eps = 0, q | k | v of a token row is
    x / rms(x): its root mean square is exactly 1, and scaling the row changes nothing."""
    Hq, Hkv, D = 2, 1, 4
    dim = (Hq + 2 * Hkv) * D
    x = _rand((2, 3, dim), 61) * 5.0
    gamma, w = np.ones(dim), np.eye(dim)
    q, k, v = oracle_mod.qkv_prologue(x, gamma, w, Hq, Hkv, D, eps=0.0, rotate=False)
    y = np.concatenate([q.reshape(2, 3, -1), k.reshape(2, 3, -1), v.reshape(2, 3, -1)], axis=-1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=0, atol=1e-14)
    q2, k2, v2 = oracle_mod.qkv_prologue(x * 7.25, gamma, w, Hq, Hkv, D, eps=0.0, rotate=False)
    for a, b in ((q, q2), (k, k2), (v, v2)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)


def test_prologue_matches_torch_rms_norm_matmul_and_rope(oracle_mod):
    """PyTorch's fp64 rms_norm (gain gamma, eps) and matmul, split into heads in the
    order q, k, v, then RoPE on q and k by the oracle's rotation (pinned above)."""
    B, T, Hq, Hkv, D, dim = 2, 9, 4, 2, 8, 24
    x = _rand((B, T, dim), 62)
    gamma = _rand((dim,), 63)
    w = _rand(((Hq + 2 * Hkv) * D, dim), 64)
    xt = torch.from_numpy(x)
    y = (torch.nn.functional.rms_norm(xt, (dim,), weight=torch.from_numpy(gamma), eps=1e-5)
         @ torch.from_numpy(w).T).numpy()
    qu = y[..., :Hq * D].reshape(B, T, Hq, D)
    ku = y[..., Hq * D:(Hq + Hkv) * D].reshape(B, T, Hkv, D)
    vu = y[..., (Hq + Hkv) * D:].reshape(B, T, Hkv, D)
    for theta in (10000.0, 500.0):
        q, k, v = oracle_mod.qkv_prologue(x, gamma, w, Hq, Hkv, D, eps=1e-5, theta=theta, rotate=True)
        np.testing.assert_allclose(q, oracle_mod.rope_apply(qu, theta), rtol=0, atol=1e-12)
        np.testing.assert_allclose(k, oracle_mod.rope_apply(ku, theta), rtol=0, atol=1e-12)
        np.testing.assert_allclose(v, vu, rtol=0, atol=1e-12)
    q, k, v = oracle_mod.qkv_prologue(x, gamma, w, Hq, Hkv, D, eps=1e-5, rotate=False)
    for a, b in ((q, qu), (k, ku), (v, vu)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
