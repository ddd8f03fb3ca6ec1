"""A model of the TF32 backward kernel's barrier protocol (csrc/attn_bwd_tf32.cu), run
on the CPU for every step count a CTA can get.

The four roles of a CTA -- the TMA producer, the UMMA issuer, the RoPE / rounding /
transpose / dQ-drain warps and the gradient warps -- are coroutines running the role's sequence of waits and arrivals (a group of threads
arrives as one); MMAs and copies complete at once.  As in the forward's model
(test_fwd_protocol_model.py), the check fails on a deadlock or on a wait evaluated while
its barrier is neither in the phase waited for nor the one after (mbarrier parity
aliasing); every arrival also names the phase it is meant for, and one that lands in
another phase (a role running a step ahead on a barrier that several roles complete)
fails too.  Two Q'/dO stages and two S^T/dP^T TMEM buffers: the next step's S^T and dP^T
go out before the current step's dV, dK and dQ.  Kept in step with the kernel by hand.
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


def simulate(n_it, rng, rope_waits_for_s=True):
    bars = {}

    def bar(name, count):
        return bars.setdefault(name, Bar(name, count))

    kv_full, k_ready = bar("kv_full", 1), bar("k_ready", 1)
    stage_full = [bar("stage_full0", 1), bar("stage_full1", 1)]
    stage_free = [bar("stage_free0", 2), bar("stage_free1", 2)]   # S/dP commit + the transposes
    s_full = [bar("s_full0", 1), bar("s_full1", 1)]
    q_rot, q_ready, qt_free = bar("q_rot", 1), bar("q_ready", 1), bar("qt_free", 1)
    ds_ready, dq_full, dq_free = bar("ds_ready", 1), bar("dq_full", 1), bar("dq_free", 1)
    dkv_full = bar("dkv_full", 1)
    rows = [bar("rows0", 1), bar("rows1", 1)]

    def producer():
        kv_full.arrive(0)
        for it in range(n_it):
            if it >= 2:
                yield stage_free[it & 1], (it >> 1) - 1, f"producer: stage for step {it}"
            stage_full[it & 1].arrive(it >> 1)

    def issuer():
        yield k_ready, 0, "issuer: K'"

        def sdp(it):
            yield q_rot, it, f"issuer: rotated tiles of step {it}"
            s_full[it & 1].arrive(it >> 1)
            stage_free[it & 1].arrive(it >> 1)

        if n_it:
            yield from sdp(0)
        for it in range(n_it):
            if it + 1 < n_it:
                yield from sdp(it + 1)
            yield ds_ready, it, f"issuer: dS of step {it}"
            yield q_ready, it, f"issuer: transposes of step {it}"
            qt_free.arrive(it)
            if it > 0:
                yield dq_free, it - 1, f"issuer: dQ' drained, step {it - 1}"
            dq_full.arrive(it)
        dkv_full.arrive(0)

    def rope():
        yield kv_full, 0, "rope: K, V"
        k_ready.arrive(0)

        def rotate(it):
            yield stage_full[it & 1], it >> 1, f"rope: tiles of step {it}"
            q_rot.arrive(it)

        def drain(it):
            yield dq_full, it, f"rope: dQ' of step {it}"
            dq_free.arrive(it)

        if n_it:
            yield from rotate(0)
        for it in range(n_it):
            yield q_rot, it, f"rope: rotation of step {it} (all threads)"
            if it > 0:
                yield qt_free, it - 1, f"rope: Q'^T free after step {it - 1}"
            q_ready.arrive(it)
            stage_free[it & 1].arrive(it >> 1)
            if it + 1 < n_it:
                if rope_waits_for_s:
                    yield s_full[it & 1], it >> 1, f"rope: S^T of step {it} issued"
                yield from rotate(it + 1)
            if it > 0:
                yield from drain(it - 1)
        if n_it:
            yield from drain(n_it - 1)

    def gradient():
        rows[0].arrive(0)
        for it in range(n_it):
            yield rows[it & 1], it >> 1, f"gradient: LSE/Delta of step {it}"
            yield s_full[it & 1], it >> 1, f"gradient: S^T of step {it}"
            if it > 0:
                yield dq_full, it - 1, f"gradient: dS buffer after step {it - 1}"
            ds_ready.arrive(it)
            if it + 1 < n_it:
                rows[(it + 1) & 1].arrive((it + 1) >> 1)
        yield dkv_full, 0, "gradient: dK, dV"

    roles = {"producer": producer(), "issuer": issuer(), "rope": rope(), "gradient": gradient()}
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


@pytest.mark.parametrize("n_it", list(range(0, 9)) + [24, 31, 96])
def test_tf32_backward_protocol(n_it):
    for seed in range(40):
        simulate(n_it, random.Random(seed * 131 + n_it))


def test_the_model_finds_the_first_step_race():
    """Without the RoPE warps' wait for step it's S^T before rotating step it + 1, the
    rotation barrier can complete two phases before the issuer looks at the first."""
    with pytest.raises(ProtocolError, match="aliasing"):
        for seed in range(200):
            simulate(3, random.Random(seed), rope_waits_for_s=False)
