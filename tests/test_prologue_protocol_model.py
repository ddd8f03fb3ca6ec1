"""A model of the persistent RMSNorm -> QKV -> RoPE prologue kernel's barrier protocol
(csrc/qkv_prologue.cu), run on the CPU for every tile and chunk count a CTA can get.

Roles: the TMA producer (one ring over every chunk of every tile of the CTA), the UMMA
issuer (two TMEM accumulators, tile i in accumulator i % 2) and the epilogue warps (wait
for the accumulator, free it).  A stage is freed by the MMA commit alone; each row's
1/rms comes from a pass before the kernel.  Each role is a coroutine running its waits and arrivals
(a group of threads arrives as one; MMAs and copies complete at once); a run fails on a
deadlock, on parity aliasing, or on an arrival that lands in another phase, as in the
other protocol models.  Kept in step with the kernel by hand.
"""
import random

import pytest

NS = 4


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


def simulate(n_tiles, nk, rng, epilogue_frees_acc=True):
    bars = {}

    def bar(name, count):
        return bars.setdefault(name, Bar(name, count))

    full = [bar(f"full{s}", 1) for s in range(NS)]
    empty = [bar(f"empty{s}", 1) for s in range(NS)]             # the MMA commit
    acc_full = [bar(f"acc_full{i}", 1) for i in range(2)]
    acc_empty = [bar(f"acc_empty{i}", 1) for i in range(2)]

    def producer():
        for g in range(n_tiles * nk):
            s = g % NS
            if g >= NS:
                yield empty[s], g // NS - 1, f"producer: stage {s} for chunk {g}"
            full[s].arrive(g // NS)

    def issuer():
        g = 0
        for i in range(n_tiles):
            ab = i & 1
            if i >= 2:
                yield acc_empty[ab], (i >> 1) - 1, f"issuer: accumulator {ab} read (tile {i - 2})"
            for kc in range(nk):
                s = g % NS
                yield full[s], g // NS, f"issuer: chunk {g}"
                empty[s].arrive(g // NS)
                if kc == nk - 1:
                    acc_full[ab].arrive(i >> 1)
                g += 1

    def epilogue():
        for i in range(n_tiles):
            ab = i & 1
            yield acc_full[ab], i >> 1, f"epilogue: accumulator of tile {i}"
            if epilogue_frees_acc:
                acc_empty[ab].arrive(i >> 1)

    roles = {"producer": producer(), "issuer": issuer(), "epilogue": epilogue()}
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


@pytest.mark.parametrize("n_tiles", [0, 1, 2, 3, 5, 9])
@pytest.mark.parametrize("nk", [1, 2, 3, 4, 5, 12])
def test_prologue_protocol(n_tiles, nk):
    for seed in range(20):
        simulate(n_tiles, nk, random.Random(seed * 31 + n_tiles * 7 + nk))


def test_the_model_finds_an_accumulator_never_freed():
    with pytest.raises(ProtocolError, match="deadlock"):
        simulate(3, 4, random.Random(0), epilogue_frees_acc=False)
