"""CPU model of the persistent sliding-window attention schedule (attn_fwd_tc_window.cu).

The kernel's CTAs each walk a list of 256-row units.  A TMA producer, an MMA
issuer and two softmax groups hand tiles to one another through mbarriers whose
phases run on across units.  This module restates, in Python, (a) which units
each CTA takes and which key tiles each unit's two query tiles see, and (b) the
order of every barrier wait, arrival and commit of the four roles.  It then
checks, for random interleavings, that every wait is satisfied by exactly the
completion it counts on.  An mbarrier wait names a phase only by its parity,
so a wait that starts two or more phases behind, or ahead, would pass on the
wrong phase or hang.  It also checks that every query tile with keys reaches
its epilogue.  The model mirrors the kernel's code and is kept beside it; the
GPU tests check the kernel's results.
"""
import random

import pytest

S = 3          # K/V ring stages
MAX_ITEMS = 1024


def cta_items(BH, nqt, Nk, window, G, b):
    """Units of CTA b in a grid of G: k*G + b in even rounds, k*G + G-1-b in odd ones."""
    out = []
    n_items = BH * nqt
    n_kv = -(-Nk // 128)
    for k in range(MAX_ITEMS):
        i = k * G + ((G - 1 - b) if k & 1 else b)
        if i >= n_items:
            break
        c = nqt - 1 - i // BH
        r0 = c * 256
        out.append(dict(unit=i, r0=r0, nt0=min(r0 // 128 + 1, n_kv), nt1=min(r0 // 128 + 2, n_kv),
                        lo0=max(0, r0 - window + 1) // 128, lo1=max(0, r0 + 128 - window + 1) // 128))
    return out


def grid_for(n_items, sms):
    g = min(n_items, sms)
    return max(g, -(-n_items // MAX_ITEMS))


class Barrier:
    def __init__(self):
        self.done = 0


class Model:
    def __init__(self, items):
        self.items = items
        self.bars = {}
        self.inflight = []   # commits and copies that complete later, in any order
        self.epilogues = []

    def bar(self, name):
        return self.bars.setdefault(name, Barrier())

    def wait(self, name, n):
        """Block until completion n (1-based) of the barrier, testing by parity as the hardware does."""
        b = self.bar(name)
        parity = (n - 1) & 1
        while True:
            assert b.done >= n - 1, f"{name}: wait for completion {n} would pass early (done {b.done})"
            assert b.done <= n, f"{name}: wait for completion {n} missed it (done {b.done})"
            if (b.done & 1) != parity:
                return
            yield

    def later(self, name):
        self.bar(name)
        self.inflight.append(name)

    def arrive(self, name):
        self.bar(name).done += 1

    def producer(self):
        nk = nv = 0
        for k, it in enumerate(self.items):
            qb = k & 1
            if k >= 2:
                yield from self.wait(f"q_empty0{qb}", k >> 1)
                yield from self.wait(f"q_empty1{qb}", k >> 1)
            self.later(f"q_full0{qb}")
            self.later(f"q_full1{qb}")
            for _ in range(it["lo0"], it["nt1"]):
                if nk >= S:
                    yield from self.wait(f"k_empty{nk % S}", nk // S)
                self.later(f"k_full{nk % S}")
                nk += 1
                if nv >= S:
                    yield from self.wait(f"v_empty{nv % S}", nv // S)
                self.later(f"v_full{nv % S}")
                nv += 1
            yield

    def issuer(self):
        items = self.items
        k = 0
        lo0, nt0, lo1, nt1 = (items[0][x] for x in ("lo0", "nt0", "lo1", "nt1"))
        ns, npv = [0, 0], [0, 0]
        uses = [0] * S   # ring-slot uses, to name the K/V completion each wait needs
        yield from self.wait("q_full00", 1)
        yield from self.wait("q_full10", 1)
        uses[0] = 1
        yield from self.wait("k_full0", 1)
        self.later("s_full0")
        ns[0] = 1
        if lo1 == lo0:
            self.later("s_full1")
            ns[1] = 1
        self.later("k_empty0")
        j, st = lo0, 0
        vuses = [0] * S
        while True:
            qb = k & 1
            last = j + 1 == nt1
            nxt, n_in0, n_in1, qbn, nx = True, j + 1 < nt0, j + 1 >= lo1, qb, None
            if last:
                nxt = k + 1 < len(items)
                qbn = (k + 1) & 1
                if nxt:
                    nx = items[k + 1]
                    yield from self.wait(f"q_full0{qbn}", ((k + 1) >> 1) + 1)
                    yield from self.wait(f"q_full1{qbn}", ((k + 1) >> 1) + 1)
                n_in0 = nxt
                n_in1 = nxt and nx["lo1"] == nx["lo0"]
            stn = (st + 1) % S
            k_ready = False
            if n_in0:
                if ns[0] > 0:
                    yield from self.wait("s_free0", ns[0])
                uses[stn] += 1
                yield from self.wait(f"k_full{stn}", uses[stn])
                k_ready = True
                self.later("s_full0")
                ns[0] += 1
            vuses[st] += 1
            yield from self.wait(f"v_full{st}", vuses[st])
            if j < nt0:
                yield from self.wait("p_ready0", npv[0] + 1)
                self.later("pv_done0")
                if j == nt0 - 1:
                    self.later("o_final0")
                npv[0] += 1
            if n_in1:
                if ns[1] > 0:
                    yield from self.wait("s_free1", ns[1])
                if not k_ready:
                    uses[stn] += 1
                    yield from self.wait(f"k_full{stn}", uses[stn])
                self.later("s_full1")
                ns[1] += 1
            if nxt:
                self.later(f"k_empty{stn}")
            if j >= lo1:
                yield from self.wait("p_ready1", npv[1] + 1)
                self.later("pv_done1")
                if j == nt1 - 1:
                    self.later("o_final1")
                npv[1] += 1
            self.later(f"v_empty{st}")
            st = stn
            if not last:
                j += 1
                yield
                continue
            self.later(f"q_empty0{qb}")
            self.later(f"q_empty1{qb}")
            if not nxt:
                break
            k += 1
            j = nx["lo0"]
            lo0, nt0, lo1, nt1 = nx["lo0"], nx["nt0"], nx["lo1"], nx["nt1"]
            yield
        self.later("drain")
        yield from self.wait("drain", 1)

    def softmax(self, t):
        cnt = nfin = 0
        for k, it in enumerate(self.items):
            jlo, jhi = (it["lo0"], it["nt0"]) if t == 0 else (it["lo1"], it["nt1"])
            for j in range(jlo, jhi):
                yield from self.wait(f"s_full{t}", cnt + 1)
                self.arrive(f"s_free{t}")
                yield
                if j > jlo:
                    yield from self.wait(f"pv_done{t}", cnt)
                self.arrive(f"p_ready{t}")
                cnt += 1
                yield
            if jhi <= jlo:
                continue
            yield from self.wait(f"o_final{t}", nfin + 1)
            nfin += 1
            self.epilogues.append((k, t))

    def run(self, seed):
        rng = random.Random(seed)
        live = {"producer": self.producer(), "issuer": self.issuer(), "softmax0": self.softmax(0),
                "softmax1": self.softmax(1)}
        steps = 0
        while live:
            steps += 1
            assert steps < 1_000_000, "no progress: a wait can never be satisfied"
            if self.inflight and rng.random() < 0.5:
                self.bar(self.inflight.pop(rng.randrange(len(self.inflight)))).done += 1
                continue
            name = rng.choice(sorted(live))
            try:
                next(live[name])
            except StopIteration:
                del live[name]


# (B*Hq, N, window, SM count): the bench shape, ragged N, a last unit whose second
# query tile sees no key tile, windows below and above a tile, few SMs (long lists)
SHAPES = [(48, 4096, 256, 152), (6, 513, 100, 4), (2, 600, 1, 3), (3, 1100, 300, 2), (1, 300, 129, 1),
          (4, 700, 64, 5), (1, 4096, 1024, 3), (80, 850, 1, 152)]


@pytest.mark.parametrize("BH,N,window,sms", SHAPES)
def test_every_unit_once(BH, N, window, sms):
    nqt = -(-N // 256)
    G = grid_for(BH * nqt, sms)
    seen = sorted(it["unit"] for b in range(G) for it in cta_items(BH, nqt, N, window, G, b))
    assert seen == list(range(BH * nqt))


@pytest.mark.parametrize("BH,N,window,sms", SHAPES)
def test_barrier_protocol(BH, N, window, sms):
    nqt = -(-N // 256)
    G = grid_for(BH * nqt, sms)
    rng = random.Random(N + window)
    for b in sorted(rng.sample(range(G), min(G, 4))):
        items = cta_items(BH, nqt, N, window, G, b)
        want = sorted((k, t) for k, it in enumerate(items) for t in (0, 1)
                      if (it["nt0"] > it["lo0"] if t == 0 else it["nt1"] > it["lo1"]))
        for seed in range(2):
            m = Model(items)
            m.run(seed * 7919 + b)
            assert sorted(m.epilogues) == want


def test_model_catches_a_wrong_phase():
    """The model must fail when a wait counts on the wrong completion (a softmax
    waiting for the current PV instead of the previous one deadlocks)."""
    items = cta_items(2, 1024, 1024, 256, 1, 0)

    class Broken(Model):
        def softmax(self, t):
            cnt = 0
            for it in self.items:
                jlo, jhi = (it["lo0"], it["nt0"]) if t == 0 else (it["lo1"], it["nt1"])
                for j in range(jlo, jhi):
                    yield from self.wait(f"s_full{t}", cnt + 1)
                    self.arrive(f"s_free{t}")
                    if j > jlo:
                        yield from self.wait(f"pv_done{t}", cnt + 1)  # wrong: PV of this tile is not issued yet
                    self.arrive(f"p_ready{t}")
                    cnt += 1
                    yield

    with pytest.raises(AssertionError):
        Broken(items).run(0)
