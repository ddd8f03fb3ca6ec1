"""A model of the persistent forward kernel's barrier protocol (csrc/attn_fwd.cu), run
on the CPU over the unit schedules the kernel's CTAs get.

Each role of a CTA -- the TMA producer, the RoPE warps, the two UMMA issuers and the two
softmax warp groups -- is a coroutine that runs the role's sequence of waits and
arrivals; MMAs and copies complete at once (that adds no dependency).  A scheduler
advances, in random order, any role whose wait is satisfied.  Two failures are
reported:

- deadlock: no role can advance before all have finished;
- parity aliasing: a wait is evaluated while its barrier is not in the phase it waits
  for or the one after (an mbarrier parity wait then either passes on the wrong phase
  or never passes).

The model follows the kernel's rules step for step (the S look-ahead bounds, the fused
PV + S batch, the stage releases beyond the diagonal, the Q-buffer releases of subtiles
without rows, the O-rescale wait on the previous stage release, taken here on every
tile).  Kept in step with the kernel by hand: a change to the kernel's waits belongs
here too.  The previous rules are kept as switches, and the test checks that the model
finds the deadlock and the aliasing they had (several units per CTA where a subtile has
no rows).
"""
import random

import pytest

BM, BN = 128, 64
# (Q buffers, K/V stages) of the kernel's configurations: bf16 head_dim 32/64 and TF32
# head_dim 32; bf16 head_dim 128; TF32 head_dim 64.
CONFIGS = [(2, 6), (1, 4), (1, 3)]


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arr, self.phase = name, count, 0, 0

    def arrive(self):
        self.arr += 1
        assert self.arr <= self.count
        if self.arr == self.count:
            self.arr = 0
            self.phase += 1


class ProtocolError(Exception):
    pass


def cta_units(c, G, n_units, B, Hq, n_qt, lens, T):
    """Key tiles per subtile (n_u) and loaded K/V tiles (n_kv) of CTA c's units, in the
    kernel's order: heaviest first, dealt in snake order over G CTAs."""
    out = []
    k = 0
    while True:
        U = k * G + ((G - 1 - c) if (k & 1) else c)
        if U >= n_units:
            return out
        rank, rem = divmod(U, B * Hq)
        b = rem // Hq
        q0 = (n_qt - 1 - rank) * 2 * BM
        L = T if lens is None else lens[b]
        n_u = [min(q0 + u * BM + BM - 1, L - 1) // BN + 1 if q0 + u * BM < L else 0 for u in range(2)]
        out.append({"n_u": n_u, "n_kv": max(n_u)})
        k += 1


def simulate(units, NQB, NS, rng, old_lookahead=False, old_q_release=False):
    bars = {}

    def bar(name, i, count):
        return bars.setdefault((name, i), Bar((name, i), count))

    q_full = lambda qb: bar("q_full", qb, 1)
    q_empty = lambda qb: bar("q_empty", qb, 2)
    q_ready = lambda qb: bar("q_ready", qb, 1)
    kv_full = lambda s: bar("kv_full", s, 1)
    k_ready = lambda s: bar("k_ready", s, 1)
    kv_empty = lambda s: bar("kv_empty", s, 2)
    s_full = lambda u, b: bar("s_full", (u, b), 1)
    p_ready = lambda u, b: bar("p_ready", (u, b), 1)
    o_final = lambda u: bar("o_final", u, 1)
    K = len(units)

    def check(b, n):
        if b.phase not in (n, n + 1):
            raise ProtocolError(f"parity aliasing: {b.name} waited for phase {n} in phase {b.phase}")
        return b.phase == n + 1

    def producer():
        issued = 0
        for k, f in enumerate(units):
            if k >= NQB:
                yield q_empty(k % NQB), k // NQB - 1, f"producer: Q buffer for unit {k}"
            q_full(k % NQB).arrive()
            for _ in range(f["n_kv"]):
                g = issued
                if g >= NS:
                    yield kv_empty(g % NS), g // NS - 1, f"producer: stage for tile {g}"
                kv_full(g % NS).arrive()
                issued += 1

    def rope():
        g = 0
        for k, f in enumerate(units):
            yield q_full(k % NQB), k // NQB, f"rope: Q of unit {k}"
            q_ready(k % NQB).arrive()
            for _ in range(f["n_kv"]):
                yield kv_full(g % NS), g // NS, f"rope: K tile {g}"
                k_ready(g % NS).arrive()
                g += 1

    def issuer(u):
        sw = {"k": -1, "j": 0, "n": 0, "n_kv": 0, "kvb": 0}

        def load(kk):
            sw["k"] = kk if kk < K else -1
            if kk < K:
                sw["n"], sw["n_kv"] = units[kk]["n_u"][u], units[kk]["n_kv"]

        def skip_empty():
            while sw["k"] >= 0 and sw["n"] == 0:
                sw["kvb"] += sw["n_kv"]
                load(sw["k"] + 1)

        def advance():
            sw["j"] += 1
            if sw["j"] == sw["n"]:
                sw["j"] = 0
                sw["kvb"] += sw["n_kv"]
                load(sw["k"] + 1)
                skip_empty()

        load(0)
        skip_empty()
        st = {"t_s": 0, "qr": 0, "t": 0, "g": 0, "kp": 0, "jp": 0, "np": 0, "nkv": 0}

        def may_issue(k_cur, t_pv, g_rel):
            if sw["k"] < 0 or st["t_s"] >= t_pv + 2:
                return False
            if old_lookahead:
                return NQB == 2 or sw["k"] <= k_cur
            return sw["k"] <= k_cur + NQB - 1 and sw["kvb"] + sw["j"] < g_rel + NS

        def q_sync(upto):
            while st["qr"] <= min(upto, K - 1):
                q = st["qr"]
                yield q_ready(q % NQB), q // NQB, f"issuer {u}: Q of unit {q}"
                if not old_q_release and units[q]["n_u"][u] == 0:
                    q_empty(q % NQB).arrive()
                st["qr"] += 1

        def load_pv():
            while st["kp"] < K:
                f = units[st["kp"]]
                st["np"], st["nkv"] = f["n_u"][u], f["n_kv"]
                if st["nkv"] > 0:
                    return True
                st["kp"] += 1
            return False

        more = load_pv()
        if not old_q_release:
            yield from q_sync(st["kp"] if more else K)
        while True:
            if may_issue(st["kp"], st["t"], st["g"]):
                if sw["j"] == 0:
                    yield from q_sync(sw["k"])
                gs = sw["kvb"] + sw["j"]
                yield k_ready(gs % NS), gs // NS, f"issuer {u}: K tile {gs} for S"
                s_full(u, st["t_s"] & 1).arrive()
                st["t_s"] += 1
                advance()
                continue
            if not more:
                break
            g = st["g"]
            if st["jp"] < st["np"]:
                t = st["t"]
                yield p_ready(u, t & 1), t >> 1, f"issuer {u}: P of tile {t}"
                fuse = may_issue(st["kp"], t + 1, g + 1) and not (sw["j"] == 0 and st["qr"] <= sw["k"])
                if fuse:   # mbarrier.test_wait on the S tile's K: the state decides
                    gs = sw["kvb"] + sw["j"]
                    b = k_ready(gs % NS)
                    if b.phase not in (gs // NS, gs // NS + 1):
                        raise ProtocolError("parity aliasing in the fused-S test")
                    fuse = b.phase == gs // NS + 1
                if st["jp"] == st["np"] - 1:
                    o_final(u).arrive()
                kv_empty(g % NS).arrive()
                if fuse:
                    s_full(u, st["t_s"] & 1).arrive()
                    st["t_s"] += 1
                    advance()
                st["t"] += 1
            else:
                yield k_ready(g % NS), g // NS, f"issuer {u}: tile {g} beyond the diagonal"
                kv_empty(g % NS).arrive()
            st["g"] += 1
            st["jp"] += 1
            if st["jp"] == st["nkv"]:
                st["jp"] = 0
                st["kp"] += 1
                more = load_pv()
                if not old_q_release:
                    yield from q_sync(st["kp"] if more else K)
        if not old_q_release:
            yield from q_sync(K)

    def softmax(u):
        t = n_epi = kvb = 0
        for k, f in enumerate(units):
            n = f["n_u"][u]
            if n == 0:
                if old_q_release:
                    yield q_full(k % NQB), k // NQB, f"softmax {u}: Q of unit {k} (no rows)"
                    q_empty(k % NQB).arrive()
                kvb += f["n_kv"]
                continue
            for j in range(n):
                yield s_full(u, t & 1), t >> 1, f"softmax {u}: S of tile {t}"
                if j > 0:
                    g = kvb + j
                    yield kv_empty((g - 1) % NS), (g - 1) // NS, f"softmax {u}: O rescale at tile {g}"
                p_ready(u, t & 1).arrive()
                t += 1
            yield o_final(u), n_epi, f"softmax {u}: last PV of unit {k}"
            q_empty(k % NQB).arrive()
            n_epi += 1
            kvb += f["n_kv"]

    roles = {"producer": producer(), "rope": rope(), "issuer0": issuer(0), "issuer1": issuer(1),
             "softmax0": softmax(0), "softmax1": softmax(1)}
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
            if check(b, n):
                try:
                    pending[name] = next(roles[name])
                except StopIteration:
                    del roles[name], pending[name]
                break
        else:
            raise ProtocolError("deadlock: " + "; ".join(pending[nm][2] for nm in roles))


def failures(B, T, Hq, lens, NQB, NS, sms=152, trials=2, **old):
    n_qt = (T + 2 * BM - 1) // (2 * BM)
    n_units = n_qt * B * Hq
    G = min(n_units, sms)
    bad = []
    for c in range(G):
        units = cta_units(c, G, n_units, B, Hq, n_qt, lens, T)
        for tr in range(trials):
            try:
                simulate(units, NQB, NS, random.Random(tr * 7919 + c), **old)
            except ProtocolError as e:
                bad.append((c, str(e)))
                break
    return bad


CASES = [
    (16, 512, 12, None),                                    # the GPU-pipeline shape
    (4, 320, 48, None),                                     # second subtile past T in every other unit
    (8, 64, 64, None),                                      # one-tile units
    (8, 384, 16, None),
    (16, 320, 48, [1, 64, 65, 300, 320, 0, 129, 200, 17, 256, 257, 320, 64, 90, 310, 2]),
    (5, 512, 6, [1, 5, 129, 300, 512]),
]


@pytest.mark.parametrize("NQB,NS", CONFIGS)
@pytest.mark.parametrize("B,T,Hq,lens", CASES)
def test_forward_protocol_has_no_deadlock_or_aliasing(B, T, Hq, lens, NQB, NS):
    for sms in (152, 7):
        assert failures(B, T, Hq, lens, NQB, NS, sms=sms) == []


def test_random_schedules():
    rng = random.Random(2024)
    for it in range(24):
        NQB, NS = CONFIGS[it % 3]
        T = rng.choice([1, 5, 64, 65, 129, 192, 257, 320, 384, 600])
        B = rng.choice([1, 3, 8, 16])
        Hq = rng.choice([1, 6, 24, 64])
        lens = None
        if it % 2:
            lens = [min(T, rng.choice([0, 1, 63, 64, 65, 128, 129, 256, 257, T, rng.randint(0, T)])) for _ in range(B)]
        assert failures(B, T, Hq, lens, NQB, NS, sms=rng.choice([152, 7, 3]), trials=1) == [], (B, T, Hq, lens)


def test_the_model_finds_the_previous_rules_faults():
    """The S look-ahead without the unit and stage bounds deadlocks when a subtile has
    no rows in several units in a row; the Q buffer freed by a subtile's softmax warps
    after the Q landed lets a run of empty units lap the Q barriers."""
    bad = failures(4, 320, 48, None, 2, 6, old_lookahead=True)
    assert any("deadlock" in e for _, e in bad)
    lens = [1, 64, 65, 300, 320, 0, 129, 200, 17, 256, 257, 320, 64, 90, 310, 2]
    bad = failures(16, 320, 48, lens, 2, 6, old_q_release=True)
    assert any("aliasing" in e for _, e in bad)
