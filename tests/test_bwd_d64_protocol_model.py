"""A model of the bf16 head_dim-64 backward kernel's barrier protocol
(csrc/attn_bwd_d64.cu), run on the CPU for every tile count a CTA can get.

The kernel's roles -- the TMA producer that also issues dQ' (warp 0), the S^T and dP^T
issuers (warps 1, 2), the dV/dK' issuer (warp 3), the RoPE / dQ'-drain warps (4-7) and
the two gradient warp groups (8-11 and 12-15, which take alternate 64-query half-steps)
-- are coroutines running the role's sequence of waits and arrivals; a group of threads
arrives as one, and MMAs and copies complete at once.  As in the forward's model
(test_fwd_protocol_model.py), a run fails on a deadlock, on a wait evaluated while its
barrier is neither in the phase waited for nor the one after (mbarrier parity aliasing),
or on an arrival that lands in a phase other than the one it names.  Kept in step with
the kernel by hand.
"""
import random

import pytest

NQS = 5   # Q'/dO half-step stages


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


def simulate(n_tiles, rng, s_waits_for_read=True):
    n_hs = 2 * n_tiles
    bars = {}

    def bar(name, count):
        return bars.setdefault(name, Bar(name, count))

    kv_full, k_ready, dkv_full = bar("kv_full", 1), bar("k_ready", 1), bar("dkv_full", 1)
    final = bar("final", 4)
    qdo_full = [bar(f"qdo_full{s}", 1) for s in range(NQS)]
    qdo_empty = [bar(f"qdo_empty{s}", 1) for s in range(NQS)]
    sdp_full = [bar(f"sdp_full{i}", 2) for i in range(2)]        # S^T and dP^T issuers
    sp_read = [bar(f"sp_read{i}", 1) for i in range(2)]          # the buffer's warp group
    ds_half = [bar(f"ds_half{i}", 1) for i in range(2)]          # the half's warp group
    ds_tile = [bar(f"ds_tile{i}", 2) for i in range(2)]          # both groups
    ds_free = [bar(f"ds_free{i}", 2) for i in range(2)]          # dK' issuer (odd half), dQ' issuer
    dq_full, dq_free = bar("dq_full", 1), bar("dq_free", 1)
    stage_free, staged = bar("stage_free", 1), bar("staged", 1)

    def producer():
        kv_full.arrive(0)

        def load(hs):
            s = hs % NQS
            if hs >= NQS:
                yield qdo_empty[s], hs // NQS - 1, f"producer: stage {s} for half-step {hs}"
            qdo_full[s].arrive(hs // NQS)

        for hs in range(min(NQS, n_hs)):
            yield from load(hs)
        yield k_ready, 0, "producer/dQ': K'"
        for tau in range(n_tiles):
            tb = tau & 1
            yield ds_tile[tb], tau >> 1, f"dQ' issuer: dS^T of tile {tau}"
            if tau >= 1:
                yield dq_free, tau - 1, f"dQ' issuer: drained tile {tau - 1}"
            dq_full.arrive(tau)
            ds_free[tb].arrive(tau >> 1)
            for hs in range(2 * tau + NQS, min(2 * tau + NQS + 2, n_hs)):
                yield from load(hs)
        final.arrive(0)

    def sdp_issuer(is_s):
        name = "S^T" if is_s else "dP^T"
        if is_s:
            yield k_ready, 0, "S^T issuer: K'"
        else:
            yield kv_full, 0, "dP^T issuer: V"
        for hs in range(n_hs):
            s, bf = hs % NQS, hs & 1
            yield qdo_full[s], hs // NQS, f"{name} issuer: tiles of half-step {hs}"
            if hs >= 2 and (s_waits_for_read or not is_s):
                yield sp_read[bf], (hs - 2) >> 1, f"{name} issuer: buffer {bf} read (half-step {hs - 2})"
            sdp_full[bf].arrive(hs >> 1)
        final.arrive(0)

    def dvdk_issuer():
        for hs in range(n_hs):
            s, half, tau = hs % NQS, hs & 1, hs >> 1
            yield ds_half[half], tau, f"dV/dK' issuer: dS^T of half-step {hs}"
            qdo_empty[s].arrive(hs // NQS)
            if half == 1:
                ds_free[tau & 1].arrive(tau >> 1)
        dkv_full.arrive(0)
        final.arrive(0)

    def drain():
        yield kv_full, 0, "rope: K"
        k_ready.arrive(0)
        for tau in range(n_tiles):
            yield dq_full, tau, f"drain: dQ' of tile {tau}"
            dq_free.arrive(tau)
            if tau > 0:
                stage_free.arrive(tau - 1)
                yield stage_free, tau - 1, f"drain: staging tile free (tile {tau - 1})"
            staged.arrive(tau)
            yield staged, tau, f"drain: tile {tau} staged"

    def gradient(g):
        for hs in range(g, n_hs, 2):
            tau, tb = hs >> 1, (hs >> 1) & 1
            yield sdp_full[g], hs >> 1, f"gradient {g}: S^T/dP^T of half-step {hs}"
            if hs >= 2:
                yield qdo_empty[(hs - 2) % NQS], (hs - 2) // NQS, f"gradient {g}: P^T free (half-step {hs - 2})"
            if tau >= 2:
                yield ds_free[tb], (tau - 2) >> 1, f"gradient {g}: dS^T tile free (tile {tau - 2})"
            sp_read[g].arrive(hs >> 1)
            ds_half[g].arrive(tau)
            ds_tile[tb].arrive(tau >> 1)
        yield dkv_full, 0, f"gradient {g}: dK, dV"

    roles = {"producer": producer(), "S": sdp_issuer(True), "dP": sdp_issuer(False), "dVdK": dvdk_issuer(),
             "drain": drain(), "grad0": gradient(0), "grad1": gradient(1)}
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


@pytest.mark.parametrize("n_tiles", list(range(0, 9)) + [12, 24, 48])
def test_d64_backward_protocol(n_tiles):
    for seed in range(30):
        simulate(n_tiles, random.Random(seed * 977 + n_tiles))


def test_the_model_finds_an_issuer_running_ahead():
    """Without the S^T issuer's wait for its buffer to be read, the S^T/dP^T barrier of a
    buffer can collect an arrival for a later half-step."""
    with pytest.raises(ProtocolError):
        for seed in range(200):
            simulate(6, random.Random(seed), s_waits_for_read=False)
