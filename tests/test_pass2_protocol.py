"""The barrier protocols of the pass-2 kernels (pass2_dual_kernel with two softmax
groups, pass2_kernel with one), run as models under random schedules on the CPU.

Actors: a TMA producer per ring, the S issuers, the PV issuer and the two softmax
groups, each a generator that waits on mbarriers by parity, arrives on them, and
issues asynchronous work.  TMA loads may complete in any order; the MMAs of one
issuing thread complete in issue order (tcgen05.commit tracks all of that thread's
earlier MMAs).  An mbarrier parity wait passes when the barrier's completed-phase
count has the other parity, exactly as in hardware, so a wait made a phase early
or two phases late passes on the wrong phase.  The checks:
  - every wait that passes lands on the phase it means (completed count = phase + 1);
  - every MMA reads the shared-memory stage, S slot or P buffer (or TMEM P slot)
    holding its entry, and no S is written over a P that its P.V has not read;
  - O is rescaled, or merged, only with none of its group's P.V in flight;
  - every schedule ends (no deadlock).
The layouts the kernel used (K ring of 6 stages owned by one S issuer per group, a V
ring of 4, P in shared memory) and uses (P written over its S slot in TMEM and read
from there by the P.V product, K ring of 8, V ring of 4) must pass every schedule.
A shared K/V ring of 5 stages with two S issuers must be caught: there consecutive
uses of a stage alternate between the issuers, and one of them can wait a phase
early while the stage's previous load is still landing.  Each run draws a speed per actor and a completion rate for copies
and for MMAs, so that lagging issuers and long-running MMAs occur."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.done = count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending, self.done = 0, self.done + 1


class Violation(Exception):
    pass


def run(n, nsk, nsv, s_issuers, split, seed, pbuf_wait=True, groups=2, np_=1, p_in_tmem=False):
    """One random schedule of one block with n hot-list entries.  split=False: one
    ring of nsk stages holding K and V (one producer); True: a K ring (nsk) and a V
    ring (nsv), a producer each.  pbuf_wait=False drops the groups' wait for the P
    buffer (a planted mistake).  groups=1 with one S issuer and one ring is the
    one-group kernel (pass2_kernel); np_ is the number of P buffers per group.
    p_in_tmem: the two-group kernel's form in which a group writes P (FP16) over the
    S slot it came from and the P.V product reads it from TMEM, so an S issuer waits
    for the P.V of the slot's previous entry instead of for its S to be read;
    pbuf_wait=False then drops that wait.  Raises Violation on a wrong phase or stage."""
    rng = random.Random(seed)
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(count)
        return bars[name]

    kst = {}    # K stage -> entry whose K has landed there (None while loading)
    vst = {}
    sslot = {}  # (group, slot) -> entry whose S is there
    pbuf = {}   # (group, buffer) -> entry whose P is there
    tslot = {}  # p_in_tmem: (group, slot) -> [entry whose P is there, read by its P.V]
    pv_inflight = [0, 0]
    inflight = []  # (order key or None, callback): None = may complete in any order

    def wait(name, phase, count=1):
        b = bar(name, count)
        while b.done % 2 == phase % 2:  # hardware parity test: passes once parity differs
            yield None
        if b.done != phase + 1:
            raise Violation(f"wait on {name} for phase {phase} passed at {b.done} completed phases")

    kring, vring = ("k", "v") if split else ("kv", "kv")
    nsv_ = nsv if split else nsk

    def producer(ring, ns, store):
        for i in range(n):
            st = i % ns
            if i >= ns:
                yield from wait((ring + "_empty", st), i // ns - 1, 1 if split else 2)
            store[st] = None

            def land(st=st, i=i):
                store[st] = i
                bar((ring + "_full", st)).arrive()
            inflight.append((None, land))
            yield None

    def s_issuer(x):
        for i in range(x, n, s_issuers):
            st, v, j = i % nsk, i % groups, i // groups
            b2 = j & 1
            yield from wait((kring + "_full", st), i // nsk)
            if kst.get(st) != i:
                raise Violation(f"S({i}) issued on K stage {st} holding {kst.get(st)}")
            if j >= 2:
                if not p_in_tmem:
                    yield from wait(("s_free", v, b2), (j >> 1) - 1, 1)
                elif pbuf_wait:  # the slot holds P of entry i - 2 groups until its P.V has read it
                    yield from wait(("pv_done", v, b2), (j >> 1) - 1)

            def done(i=i, st=st, v=v, b2=b2):
                if kst.get(st) != i:
                    raise Violation(f"S({i}) read K stage {st} holding {kst.get(st)}")
                if p_in_tmem and (v, b2) in tslot and not tslot[(v, b2)][1]:
                    raise Violation(f"S({i}) overwrote P of entry {tslot[(v, b2)][0]} before its P.V read it")
                sslot[(v, b2)] = i
                bar(("s_full", v, b2)).arrive()
                bar((kring + "_empty", st), 1 if split else 2).arrive()
            inflight.append((("s", x), done))
            yield None

    def pv_issuer():
        for i in range(n):
            st, v, j = i % nsv_, i % groups, i // groups
            b2, pb = j & 1, (i // groups) % np_
            yield from wait(("p_full", v, b2), j >> 1, 1)
            yield from wait((vring + "_full", st), i // nsv_)

            def p_of(v=v, b2=b2, pb=pb):
                return tslot.get((v, b2), [None])[0] if p_in_tmem else pbuf.get((v, pb))
            if vst.get(st) != i or p_of() != i:
                raise Violation(f"PV({i}) issued on V {vst.get(st)} / P {p_of()}")
            pv_inflight[v] += 1

            def done(i=i, st=st, v=v, b2=b2, p_of=p_of):
                if vst.get(st) != i or p_of() != i:
                    raise Violation(f"PV({i}) read V {vst.get(st)} / P {p_of()}")
                if p_in_tmem:
                    tslot[(v, b2)][1] = True
                pv_inflight[v] -= 1
                bar(("pv_done", v, b2)).arrive()
                bar((vring + "_empty", st), 1 if split else 2).arrive()
            inflight.append((("pv",), done))
            yield None

    def count(v):
        return (n - v + groups - 1) // groups

    def group(v):
        for j in range(count(v)):
            i = groups * j + v
            yield from wait(("s_full", v, j & 1), j >> 1)
            if sslot.get((v, j & 1)) != i:
                raise Violation(f"group {v} read S slot holding {sslot.get((v, j & 1))} for {i}")
            if not p_in_tmem:
                bar(("s_free", v, j & 1), 1).arrive()
            yield None
            if j >= np_ and pbuf_wait and not p_in_tmem:  # P buffer j % np_: P.V of entry j - np_ has read it
                yield from wait(("pv_done", v, (j - np_) & 1), (j - np_) >> 1)
            if j >= 1 and rng.random() < 0.3:  # the running maximum moved: rescale O
                yield from wait(("pv_done", v, (j - 1) & 1), (j - 1) >> 1)
                if pv_inflight[v]:
                    raise Violation(f"group {v} rescaled O with a P.V in flight at entry {i}")
            if p_in_tmem:  # P over the S it came from (tcgen05.st, waited for before the arrive)
                if sslot.get((v, j & 1)) != i:
                    raise Violation(f"group {v} wrote P of {i} over S slot holding {sslot.get((v, j & 1))}")
                tslot[(v, j & 1)] = [i, False]
            else:
                pbuf[(v, j % np_)] = i
            bar(("p_full", v, j & 1), 1).arrive()
            yield None
        if v == 0:  # the merge waits for every group's last P.V
            for u in range(groups):
                nl = count(u)
                if nl:
                    yield from wait(("pv_done", u, (nl - 1) & 1), (nl - 1) >> 1)
                    if pv_inflight[u]:
                        raise Violation(f"merge with a P.V of group {u} in flight")

    actors = [producer(kring, nsk, kst)]
    if split:
        actors.append(producer(vring, nsv, vst))
    actors += [s_issuer(x) for x in range(s_issuers)] + [pv_issuer()] + [group(v) for v in range(groups)]
    if not split:
        vst = kst  # one ring: V lands with K
    live = list(actors)
    # each run draws a speed per actor and a completion rate for copies and for MMAs,
    # over two decades, so that lagging issuers and long-running MMAs both occur
    speed = {id(a): 10 ** rng.uniform(-2, 0) for a in live}
    rate = {"copy": 10 ** rng.uniform(-2, 0), "mma": 10 ** rng.uniform(-2, 0)}
    for _ in range(400000):
        if not live and not inflight:
            return
        # in-order completion per issuing thread: only the oldest op of each key
        heads, seen = [], set()
        for k, (key, cb) in enumerate(inflight):
            if key is None or key not in seen:
                heads.append(k)
                if key is not None:
                    seen.add(key)
        choices = [("a", a) for a in live] + [("c", k) for k in heads]
        weights = [speed[id(a)] for a in live] + [rate["copy" if inflight[k][0] is None else "mma"] for k in heads]
        kind, what = rng.choices(choices, weights)[0]
        if kind == "c":
            inflight.pop(what)[1]()
            continue
        try:
            next(what)
        except StopIteration:
            live.remove(what)
    raise Violation("no progress: deadlock")


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 8, 13, 24])
def test_kept_layout_is_safe_under_random_schedules(n):
    # K ring of 6 (each S issuer owns three stages), V ring of 4
    for seed in range(60):
        run(n, nsk=6, nsv=4, s_issuers=2, split=True, seed=seed)


@pytest.mark.parametrize("nsk,nsv", [(2, 1), (4, 2), (8, 3)])
def test_other_even_k_rings_are_safe(nsk, nsv):
    for seed in range(40):
        run(17, nsk=nsk, nsv=nsv, s_issuers=2, split=True, seed=seed)


def test_first_form_one_ring_one_s_issuer_is_safe():
    for seed in range(60):
        run(17, nsk=5, nsv=5, s_issuers=1, split=False, seed=seed)


def test_two_s_issuers_over_an_odd_shared_ring_are_caught():
    """The layout whose timing was withdrawn: some schedule makes an issuer pass a
    wait on the phase before the one it means."""
    caught = 0
    for seed in range(400):
        try:
            run(24, nsk=5, nsv=5, s_issuers=2, split=False, seed=seed)
        except Violation:
            caught += 1
    assert caught > 0


def test_planted_mistake_is_caught():
    """The checker itself: a group that writes its next P without waiting for the
    P.V of its previous one overwrites a buffer still to be read."""
    caught = 0
    for seed in range(200):
        try:
            run(12, nsk=6, nsv=4, s_issuers=2, split=True, seed=seed, pbuf_wait=False)
        except Violation:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("ns,np_", [(4, 2), (3, 2), (2, 1), (4, 1)])
def test_one_group_kernel_is_safe(ns, np_):
    """pass2_kernel: one softmax group, one S issuer, one K/V ring (4 stages with
    two P buffers in APA mode at d = 128, 3 or 2 elsewhere)."""
    for n in (1, 2, 7, 15):
        for seed in range(25):
            run(n, nsk=ns, nsv=ns, s_issuers=1, split=False, seed=seed, groups=1, np_=np_)


def test_one_group_planted_mistake_is_caught():
    caught = 0
    for seed in range(200):
        try:
            run(12, nsk=4, nsv=4, s_issuers=1, split=False, seed=seed, groups=1, np_=2, pbuf_wait=False)
        except Violation:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("n", [0, 1, 2, 3, 5, 8, 13, 24])
def test_p_in_tmem_layout_is_safe_under_random_schedules(n):
    """The two-group kernel as it runs: P written over its S slot and read from TMEM
    by the P.V product, K ring of 8 (each S issuer owns four stages), V ring of 4."""
    for seed in range(60):
        run(n, nsk=8, nsv=4, s_issuers=2, split=True, seed=seed, p_in_tmem=True)


@pytest.mark.parametrize("nsk,nsv", [(6, 4), (8, 6), (4, 2)])
def test_p_in_tmem_other_rings_are_safe(nsk, nsv):
    for seed in range(40):
        run(17, nsk=nsk, nsv=nsv, s_issuers=2, split=True, seed=seed, p_in_tmem=True)


def test_p_in_tmem_planted_mistake_is_caught():
    """An S issuer that writes S over a slot without waiting for the P.V of the P in it."""
    caught = 0
    for seed in range(200):
        try:
            run(12, nsk=6, nsv=4, s_issuers=2, split=True, seed=seed, p_in_tmem=True, pbuf_wait=False)
        except Violation:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("ns", [2, 3, 4])
def test_one_group_p_in_tmem_is_safe(ns):
    """pass2_kernel with P over its S slot in TMEM (2 K/V stages at d = 256)."""
    for n in (1, 2, 7, 15):
        for seed in range(25):
            run(n, nsk=ns, nsv=ns, s_issuers=1, split=False, seed=seed, groups=1, p_in_tmem=True)


def test_one_group_p_in_tmem_planted_mistake_is_caught():
    """(With a 2-stage ring the load of entry i already waits for the P.V of entry
    i - 2, so the missing wait shows only with more stages.)"""
    caught = 0
    for seed in range(200):
        try:
            run(12, nsk=4, nsv=4, s_issuers=1, split=False, seed=seed, groups=1, p_in_tmem=True, pbuf_wait=False)
        except Violation:
            caught += 1
    assert caught > 0
