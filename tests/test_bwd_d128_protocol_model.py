"""A model of the bf16 head_dim-128 backward kernel's barrier protocol (`attn_bwd_kernel`
in csrc/attn_bwd.cu), run on the CPU for every step count a CTA can get.

Roles: the TMA producer (warp 0), issuer A (S^T, dP^T; warp 1), issuer B (dV, dK';
warp 2), issuer C (dQ'; warp 3), the RoPE / dQ'-drain warps (4-7) and the two gradient
warp groups (8-11, 12-15, each on half of a step's query columns).  At head_dim 128 the
kernel has one Q/dO stage, P^T is written over S^T, dQ' over dP^T and dS^T over the
stage's fp16 Q'.  Each role is a coroutine running its waits and arrivals (a group of
threads arrives as one; MMAs and copies complete at once); a run fails on a deadlock,
on parity aliasing, or on an arrival that lands in another phase, as in the other
protocol models.  Kept in step with the kernel by hand.
"""
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arr, self.phase = name, count, 0, 0

    def arrive(self, phase):
        if phase != self.phase:
            raise ProtocolError(f"early arrival: {self.name} for phase {phase} in phase {self.phase}")
        self.arr += 1
        assert self.arr <= self.count, self.name
        if self.arr == self.count:
            self.arr = 0
            self.phase += 1


class ProtocolError(Exception):
    pass


def simulate(n_it, rng, producer_waits=True):
    bars = {}

    def bar(name, count):
        return bars.setdefault(name, Bar(name, count))

    kv_full, k_ready, dkv_full, final = bar("kv_full", 1), bar("k_ready", 1), bar("dkv_full", 1), bar("final", 3)
    qdo_full, q_ready, qdo_empty = bar("qdo_full", 1), bar("q_ready", 1), bar("qdo_empty", 2)   # issuers B, C
    s_full, dp_full, p_free = bar("s_full", 1), bar("dp_full", 1), bar("p_free", 1)
    ds_ready, ds_free = bar("ds_ready", 2), bar("ds_free", 2)   # both gradient groups; issuers B, C
    dq_full, dq_free = bar("dq_full", 1), bar("dq_free", 1)
    rows = [bar("rows0", 2), bar("rows1", 2)]

    def producer():
        kv_full.arrive(0)
        for it in range(n_it):
            if it >= 1 and producer_waits:
                yield qdo_empty, it - 1, f"producer: stage for step {it}"
            qdo_full.arrive(it)

    def issuer_a():
        yield k_ready, 0, "A: K'"
        for it in range(n_it):
            yield q_ready, it, f"A: Q' of step {it}"
            if it > 0:
                yield p_free, it - 1, f"A: P^T of step {it - 1} read"
            s_full.arrive(it)
            if it > 0:
                yield dq_free, it - 1, f"A: dQ' of step {it - 1} drained"
            dp_full.arrive(it)
        final.arrive(0)

    def issuer_b():
        for it in range(n_it):
            yield ds_ready, it, f"B: dS^T of step {it}"
            p_free.arrive(it)
            qdo_empty.arrive(it)
            ds_free.arrive(it)
        dkv_full.arrive(0)
        final.arrive(0)

    def issuer_c():
        for it in range(n_it):
            yield ds_ready, it, f"C: dS^T of step {it}"
            if it > 0:
                yield dq_free, it - 1, f"C: dQ' of step {it - 1} drained"
            yield dp_full, it, f"C: dP^T of step {it} done"
            dq_full.arrive(it)
            qdo_empty.arrive(it)
            ds_free.arrive(it)
        final.arrive(0)

    def rope():
        yield kv_full, 0, "rope: K"
        k_ready.arrive(0)
        for it in range(n_it + 1):
            if it < n_it:
                yield qdo_full, it, f"rope: tiles of step {it}"
                if it > 0:
                    yield ds_free, it - 1, f"rope: fp16 Q' buffer free after step {it - 1}"
                q_ready.arrive(it)
            if it > 0:
                yield dq_full, it - 1, f"drain: dQ' of step {it - 1}"
                dq_free.arrive(it - 1)

    def gradient(g):
        rows[0].arrive(0)
        for it in range(n_it):
            yield rows[it & 1], it >> 1, f"gradient {g}: LSE/Delta of step {it}"
            yield s_full, it, f"gradient {g}: S^T of step {it}"
            yield dp_full, it, f"gradient {g}: dP^T of step {it}"
            if it > 0:
                yield ds_free, it - 1, f"gradient {g}: dS^T buffer free after step {it - 1}"
            ds_ready.arrive(it)
            if it + 1 < n_it:
                rows[(it + 1) & 1].arrive((it + 1) >> 1)
        yield dkv_full, 0, f"gradient {g}: dK, dV"

    roles = {"producer": producer(), "A": issuer_a(), "B": issuer_b(), "C": issuer_c(), "rope": rope(),
             "grad0": gradient(0), "grad1": gradient(1)}
    pending = {}
    for name in list(roles):
        try:
            pending[name] = next(roles[name])
        except StopIteration:
            del roles[name]
    while roles:
        names = list(roles)
        rng.shuffle(names)
        for name in names:
            b, n, _ = pending[name]
            if b.phase not in (n, n + 1):
                raise ProtocolError(f"parity aliasing: {b.name} waited for phase {n} in phase {b.phase}")
            if b.phase == n + 1:
                try:
                    pending[name] = next(roles[name])
                except StopIteration:
                    del roles[name], pending[name]
                break
        else:
            raise ProtocolError("deadlock: " + "; ".join(pending[nm][2] for nm in roles))


@pytest.mark.parametrize("n_it", list(range(0, 9)) + [16, 64])
def test_d128_backward_protocol(n_it):
    for seed in range(30):
        simulate(n_it, random.Random(seed * 389 + n_it))


def test_the_model_finds_a_stage_refilled_too_early():
    """The model checks the barrier protocol, not the data it guards: a planted mistake
    it must catch is the producer refilling the single stage without waiting for it to
    be freed (the stage's full barrier then runs past the RoPE warps' wait)."""
    with pytest.raises(ProtocolError):
        for seed in range(200):
            simulate(5, random.Random(seed), producer_waits=False)
