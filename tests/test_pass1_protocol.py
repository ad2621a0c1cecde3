"""The barrier protocol of the three-block pass-1 kernel (pass1_multi_kernel), run as
a model under random schedules on the CPU.

Actors: the bulk-copy producer, the S issuer, the PV issuer and the U units (the four
softmax warps of a 128-row block as one actor).  Asynchronous work:
  - bulk copies of the per-tile NVFP4 blobs land in any order;
  - each issuing thread's MMAs complete in issue order; a tcgen05.cp lands before
    any later op of its thread but not necessarily after that thread's earlier
    MMAs; a commit arrives once every earlier op of its thread has completed;
  - a unit writes P to shared memory and P's scales into TMEM itself (tcgen05.st,
    completed by tcgen05.wait::st before it hands P over).
mbarrier waits test parity as the hardware does.  The checks:
  - every wait that passes lands on the phase it means;
  - the one S buffer is never overwritten before its unit has read it, and a unit
    reads the S of its own (unit, tile);
  - every MMA reads the blob, the K or V scale columns, the P buffer and the P scale
    columns of its own tile;
  - O is rescaled or read out only with none of that unit's P.V in flight;
  - every schedule ends.
Each run draws a speed per actor and a completion rate per kind of op, so that
schedules with a lagging issuer or long-running MMAs occur.  Planted mistakes (a
missing wait) must be caught.

The unwind after a wait gives up is modelled too.  Some wait times out (at a random
moment), or the producer's wait for the in-launch quantizer's flag of some tile
does: the CTA's abort flag is set, and every wait that sees it returns false.  The
producer always ends by waiting (bounded, ignoring the flag) for its copies to land
(a consumer may give up after the producer's loop has ended);
each issuer commits a drain barrier and waits for it, so that all of its tcgen05
operations have completed; the units leave their loops.  When the CTA exits and
frees TMEM, no bulk copy, tcgen05 operation or commit may still be in flight."""
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


class Aborted(Exception):
    """A wait saw the CTA's abort flag (mbar_wait returning false)."""


def run(n, U, NS, seed, drop=None, abort_step=None, stuck_tile=None, drain=True):
    """One random schedule of one CTA walking n tiles with U units and an NS-stage
    blob ring.  drop names a wait to leave out (a planted mistake): "sfv" (the PV
    issuer's wait before copying tile i's V scales over those of tile i-2), "pbuf"
    (a unit's wait before writing P over the buffer of tile i-2), "s_free" (the S
    issuer's wait for the previous unit to read S).  abort_step: the scheduler step
    at which some wait times out and sets the abort flag; stuck_tile: the tile whose
    quantizer flag never comes (the producer's wait for it gives up); drain=False
    plants a missing unwind (no waits for copies and drain barriers)."""
    rng = random.Random(seed)
    bars = {}
    state = {"abort": False}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Bar(count)
        return bars[name]

    def wait(name, phase, count=1, abortable=True):
        b = bar(name, count)
        while b.done % 2 == phase % 2:
            if abortable and state["abort"]:
                raise Aborted
            yield None
        if b.done != phase + 1:
            raise Violation(f"wait on {name} for phase {phase} passed at {b.done} completed phases")

    blob, sfk, sfv, pbuf, sfp = {}, {}, {}, {}, {}
    sbuf = {"who": None, "read": True}
    pv_inflight = [0] * U
    ops = []  # [thread, seq, kind, callback]; thread None = a bulk copy (any order)
    seq = [0]

    def issue(thread, kind, cb):
        seq[0] += 1
        ops.append((thread, seq[0], kind, cb))

    def completable(op):
        thread, s, kind, _ = op
        if thread is None:
            return True
        earlier = [o for o in ops if o[0] == thread and o[1] < s]
        if kind == "cp":
            return not any(o[2] == "cp" for o in earlier)
        if kind == "mma":
            return not any(o[2] in ("cp", "mma") for o in earlier)
        return not earlier  # commit

    def producer():
        issued = 0
        try:
            for i in range(n):
                st = i % NS
                if i >= NS:
                    yield from wait(("blob_empty", st), i // NS - 1, 2)
                if i == stuck_tile:  # the quantizer's flag of this tile never comes
                    state["abort"] = True
                    raise Aborted
                blob[st] = None

                def land(st=st, i=i):
                    blob[st] = i
                    bar(("blob_full", st)).arrive()
                issue(None, "tma", land)
                issued = i + 1
                yield None
        except Aborted:
            pass
        if drain:  # every copy issued lands before the CTA exits (at once, normally)
            for i in range(max(0, issued - NS), issued):
                yield from wait(("blob_full", i % NS), i // NS, abortable=False)

    def drained(thread, name):
        if drain:
            issue(thread, "commit", lambda: bar(name).arrive())
            yield from wait(name, 0, abortable=False)

    def s_issuer():
        try:
            yield from s_loop()
        except Aborted:
            pass
        yield from drained("s", "drain_s")

    def s_loop():
        for i in range(n):
            st = i % NS
            for u in range(U):
                if u > 0:
                    if drop != "s_free":
                        yield from wait(("s_free", u - 1), i)
                else:
                    yield from wait(("blob_full", st), i // NS)
                    if blob.get(st) != i:
                        raise Violation(f"K scales of tile {i} copied from a stage holding {blob.get(st)}")

                    def cp(i=i, st=st):
                        if blob.get(st) != i:
                            raise Violation(f"K scales of tile {i} read from a stage holding {blob.get(st)}")
                        sfk[i & 1] = i
                    issue("s", "cp", cp)
                    if i > 0 and drop != "s_free":
                        yield from wait(("s_free", U - 1), i - 1)

                def mma(i=i, st=st, u=u):
                    if blob.get(st) != i or sfk.get(i & 1) != i:
                        raise Violation(f"S({u},{i}) read blob {blob.get(st)} / K scales {sfk.get(i & 1)}")
                    if not sbuf["read"]:
                        raise Violation(f"S({u},{i}) overwrote the unread S of {sbuf['who']}")
                    sbuf["who"], sbuf["read"] = (u, i), False
                issue("s", "mma", mma)
                issue("s", "commit", lambda u=u: bar(("s_full", u)).arrive())
                yield None
            issue("s", "commit", lambda st=st: bar(("blob_empty", st), 2).arrive())

    def pv_issuer():
        try:
            yield from pv_loop()
        except Aborted:
            pass
        yield from drained("pv", "drain_pv")

    def pv_loop():
        for i in range(n):
            st = i % NS
            for u in range(U):
                yield from wait(("p_full", u, i & 1), i >> 1)
                if u == 0:
                    yield from wait(("blob_full", st), i // NS)
                    if i >= 2 and drop != "sfv":
                        yield from wait(("pv_done", U - 1, i & 1), (i - 2) >> 1)

                    def cpv(i=i, st=st):
                        if blob.get(st) != i:
                            raise Violation(f"V scales of tile {i} read from a stage holding {blob.get(st)}")
                        sfv[i & 1] = i
                    issue("pv", "cp", cpv)
                if pbuf.get((u, i & 1)) != i:
                    raise Violation(f"PV issuer found P buffer ({u},{i & 1}) holding {pbuf.get((u, i & 1))}, not {i}")

                def mma(i=i, st=st, u=u):
                    got = (blob.get(st), sfv.get(i & 1), sfp.get((u, i & 1)), pbuf.get((u, i & 1)))
                    if got != (i, i, i, i):
                        raise Violation(f"PV({u},{i}) read blob/V scales/P scales/P {got}")
                    pv_inflight[u] -= 1
                pv_inflight[u] += 1
                issue("pv", "mma", mma)
                issue("pv", "commit", lambda u=u, i=i: bar(("pv_done", u, i & 1)).arrive())
                yield None
            issue("pv", "commit", lambda st=st: bar(("blob_empty", st), 2).arrive())

    def unit(u):
        try:
            yield from unit_loop(u)
        except Aborted:
            pass

    def unit_loop(u):
        for i in range(n):
            yield from wait(("s_full", u), i)
            if sbuf["who"] != (u, i):
                raise Violation(f"unit {u} read S of {sbuf['who']} at tile {i}")
            sbuf["read"] = True
            bar(("s_free", u)).arrive()
            yield None
            if i >= 1 and rng.random() < 0.3:  # the frame moved: rescale O
                yield from wait(("pv_done", u, (i - 1) & 1), (i - 1) >> 1)
                if pv_inflight[u]:
                    raise Violation(f"unit {u} rescaled O with a P.V in flight at tile {i}")
            if i >= 2 and drop != "pbuf":
                yield from wait(("pv_done", u, i & 1), (i - 2) >> 1)
            # P to shared memory, and its scales straight into TMEM by tcgen05.st, waited
            # for (tcgen05.wait::st) before the arrive
            pbuf[(u, i & 1)] = i
            sfp[(u, i & 1)] = i
            bar(("p_full", u, i & 1)).arrive()
            yield None
        if n:
            yield from wait(("pv_done", u, (n - 1) & 1), (n - 1) >> 1)
            if pv_inflight[u]:
                raise Violation(f"unit {u} read O out with a P.V in flight")

    live = [producer(), s_issuer(), pv_issuer()] + [unit(u) for u in range(U)]
    # each run draws a speed per actor and a completion rate per kind of op, over two
    # decades, so that slow issuers and long-running MMAs both occur
    speed = {id(a): 10 ** rng.uniform(-2, 0) for a in live}
    rate = {k: 10 ** rng.uniform(-2, 0) for k in ("tma", "cp", "mma", "commit")}
    for step in range(400000):
        if step == abort_step:
            state["abort"] = True  # some wait ran out of time
        if not live:
            # every warp is done: the CTA frees TMEM and exits
            if ops:
                raise Violation(f"CTA exits with {[o[2] for o in ops]} in flight")
            return
        ready = [k for k, op in enumerate(ops) if completable(op)]
        choices = [("a", a) for a in live] + [("c", k) for k in ready]
        weights = [speed[id(a)] for a in live] + [rate[ops[k][2]] for k in ready]
        kind, what = rng.choices(choices, weights)[0]
        if kind == "c":
            ops.pop(what)[3]()
            continue
        try:
            next(what)
        except StopIteration:
            live.remove(what)
    raise Violation("no progress: deadlock")


@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 5, 9, 16])
def test_three_units_four_stages_safe_under_random_schedules(n):
    for seed in range(40):
        run(n, U=3, NS=4, seed=seed)


@pytest.mark.parametrize("U,NS", [(1, 4), (2, 3), (3, 2)])
def test_other_shapes_safe(U, NS):
    for seed in range(30):
        run(11, U=U, NS=NS, seed=seed)


@pytest.mark.parametrize("drop", ["sfv", "pbuf", "s_free"])
def test_planted_missing_waits_are_caught(drop):
    caught = 0
    for seed in range(150):
        try:
            run(10, U=3, NS=4, seed=seed, drop=drop)
        except Violation:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("n", [1, 3, 9])
def test_unwind_after_a_timeout_ends_with_nothing_in_flight(n):
    """A wait that gives up at any moment: every actor stops and the CTA exits with
    no copy or tcgen05 operation in flight."""
    for seed in range(60):
        run(n, U=3, NS=4, seed=seed, abort_step=random.Random(seed).randrange(0, 60 * n + 1))


@pytest.mark.parametrize("stuck", [0, 1, 4, 7])
def test_unwind_when_the_quantizer_flag_never_comes(stuck):
    for seed in range(40):
        run(9, U=3, NS=4, seed=seed, stuck_tile=stuck)


def test_planted_missing_unwind_is_caught():
    # without the producer's wait for its copies and the issuers' drain barriers,
    # some schedules exit with work in flight
    caught = 0
    for seed in range(100):
        try:
            run(9, U=3, NS=4, seed=seed, stuck_tile=5, drain=False)
        except Violation:
            caught += 1
    assert caught > 0
