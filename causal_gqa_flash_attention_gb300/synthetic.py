"""Seeded synthetic inputs and the named workloads.

This module draws random tensors and names shapes; it holds none of the attention
arithmetic.  Both the CUDA path's tests/benchmark and the fp64 oracle read the
tensors it returns, so the two sides always see identical input values.

Recipe: every tensor is i.i.d. N(0, sigma^2), drawn in fp32 from a CPU
``torch.Generator`` seeded with ``20261202 + 1000*workload_id + 10*layer + idx``
(idx: q=0, k=1, v=2, dO=3), then rounded to the workload's dtype.  The shapes are
the model-config table's ("NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM",
모델 구성: dim 128 with 4/2 heads and context 128; dim 768 with 12/4 heads, 16
layers and context 512) plus a longer-context, larger-head softmax-stress case and a
sequence-length sweep at a constant 65536 tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEED_BASE = 20261202
ROPE_THETA = 10000.0


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    D: int
    dtype: str            # "bf16" or "f32" (f32 runs on TF32 tensor cores)
    qk_sigma: float = 1.0
    layers: int = 1
    theta: float = ROPE_THETA

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def pairs(self) -> int:
        """Exact causal (query, key) pairs per (batch, query head): T(T+1)/2."""
        return self.T * (self.T + 1) // 2

    def flops_fwd(self) -> int:
        return 4 * self.D * self.pairs * self.B * self.Hq

    def flops_bwd(self) -> int:
        return 10 * self.D * self.pairs * self.B * self.Hq

    def flops(self) -> int:
        """fwd + bwd FLOPs of one layer (14 D per causal pair per query head)."""
        return self.flops_fwd() + self.flops_bwd()

    def compulsory_bytes(self) -> dict:
        """Compulsory HBM bytes per layer of each kernel step (inputs read once,
        outputs written once)."""
        e = 2 if self.dtype == "bf16" else 4
        q = self.B * self.T * self.Hq * self.D * e
        kv = self.B * self.T * self.Hkv * self.D * e
        row = self.B * self.Hq * self.T * 4
        return {
            "fwd": q + 2 * kv + q + row,                 # Q,K,V -> O, LSE
            "pre": 2 * q + row,                          # O, dO -> Delta
            "bwd": q + 2 * kv + q + 2 * row + q + 2 * kv,  # Q,K,V,dO,LSE,Delta -> dQ,dK,dV
        }


WORKLOADS = {
    1: Workload(1, "small-cpu-model B4 T128 Hq4 Hkv2 D32 f32", 4, 128, 4, 2, 32, "f32"),
    2: Workload(2, "gpu-pipeline B16 T512 Hq12 Hkv4 D64 bf16 x16 layers", 16, 512, 12, 4, 64, "bf16",
                layers=16),
    3: Workload(3, "gpu-pipeline B16 T512 Hq12 Hkv4 D64 f32 (TF32)", 16, 512, 12, 4, 64, "f32"),
    4: Workload(4, "softmax-stress B8 T2048 Hq16 Hkv4 D128 bf16 sigma_qk=3", 8, 2048, 16, 4, 128,
                "bf16", qk_sigma=3.0),
    51: Workload(51, "seq-sweep B128 T512 Hq12 Hkv4 D64 bf16", 128, 512, 12, 4, 64, "bf16"),
    52: Workload(52, "seq-sweep B32 T2048 Hq12 Hkv4 D64 bf16", 32, 2048, 12, 4, 64, "bf16"),
    53: Workload(53, "seq-sweep B8 T8192 Hq12 Hkv4 D64 bf16", 8, 8192, 12, 4, 64, "bf16"),
    54: Workload(54, "seq-sweep B4 T16384 Hq12 Hkv4 D64 bf16", 4, 16384, 12, 4, 64, "bf16"),
}


def _seed(wid: int, layer: int, idx: int) -> int:
    return SEED_BASE + 1000 * wid + 10 * layer + idx


def randn(shape, seed: int, sigma: float, dtype: torch.dtype) -> torch.Tensor:
    """i.i.d. N(0, sigma^2) drawn in fp32 on the CPU, rounded to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(dtype)


def make_inputs(w: Workload, layer: int = 0, batch: slice | None = None):
    """q [B,T,Hq,D], k, v [B,T,Hkv,D], dO [B,T,Hq,D] on the CPU in the workload dtype.

    ``batch`` selects a slice of the batch after drawing, so a sample keeps the
    values of the full workload."""
    dt = w.torch_dtype
    q = randn((w.B, w.T, w.Hq, w.D), _seed(w.wid, layer, 0), w.qk_sigma, dt)
    k = randn((w.B, w.T, w.Hkv, w.D), _seed(w.wid, layer, 1), w.qk_sigma, dt)
    v = randn((w.B, w.T, w.Hkv, w.D), _seed(w.wid, layer, 2), 1.0, dt)
    dO = randn((w.B, w.T, w.Hq, w.D), _seed(w.wid, layer, 3), 1.0, dt)
    if batch is not None:
        q, k, v, dO = (t[batch].contiguous() for t in (q, k, v, dO))
    return q, k, v, dO


def make_custom(B, T, Hq, Hkv, D, dtype=torch.bfloat16, seed=1, qk_sigma=1.0):
    """Inputs of an arbitrary shape (edge cases, ragged tails)."""
    q = randn((B, T, Hq, D), seed * 16 + 0, qk_sigma, dtype)
    k = randn((B, T, Hkv, D), seed * 16 + 1, qk_sigma, dtype)
    v = randn((B, T, Hkv, D), seed * 16 + 2, 1.0, dtype)
    dO = randn((B, T, Hq, D), seed * 16 + 3, 1.0, dtype)
    return q, k, v, dO


def make_decode(B, T_max, Hq, Hkv, D, dtype=torch.bfloat16, seed=1, lens=None, tail=None):
    """Inputs of one decode step: q [B, Hq, D] (each sequence's newest token), key and
    value caches [B, T_max, Hkv, D] and seq_lens int32 [B], all on the CPU.

    Lengths are ``lens`` when given, else drawn uniformly from [1, T_max] with the
    last sequence full.  Cache rows at or past a sequence's length hold N(0, 1) values
    like the rest (a reused cache), or ``tail`` (e.g. NaN) when given, so that a step
    which reads them shows it."""
    q = randn((B, Hq, D), seed * 16 + 0, 1.0, dtype)
    k = randn((B, T_max, Hkv, D), seed * 16 + 1, 1.0, dtype)
    v = randn((B, T_max, Hkv, D), seed * 16 + 2, 1.0, dtype)
    if lens is None:
        g = torch.Generator(device="cpu")
        g.manual_seed(seed * 16 + 3)
        lens = torch.randint(1, T_max + 1, (B,), generator=g, dtype=torch.int32)
        lens[-1] = T_max
    lens = torch.as_tensor(lens, dtype=torch.int32)
    if tail is not None:
        for b in range(B):
            k[b, int(lens[b]):] = tail
            v[b, int(lens[b]):] = tail
    return q, k, v, lens


def make_prologue(B, T, dim, Hq, Hkv, D, seed=1):
    """Inputs of the RMSNorm -> QKV -> RoPE prologue, bf16 on the CPU: x [B, T, dim]
    i.i.d. N(0, 1); gamma [dim] = 1 + N(0, 0.1^2) (a trained RMSNorm gain stays near 1);
    w [(Hq + 2 Hkv) D, dim] i.i.d. N(0, 1/dim) (unit-variance outputs)."""
    x = randn((B, T, dim), seed * 16 + 4, 1.0, torch.bfloat16)
    gamma = (1.0 + randn((dim,), seed * 16 + 5, 0.1, torch.float32)).to(torch.bfloat16)
    w = randn(((Hq + 2 * Hkv) * D, dim), seed * 16 + 6, dim ** -0.5, torch.bfloat16)
    return x, gamma, w
