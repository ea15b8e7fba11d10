"""Model check of the expansion kernel's CTA-pair protocol (CPU only).

The expansion kernel (csrc/expand_kv.cu) runs as a pair of CTAs that share
every MMA (tcgen05 .cta_group::2): each CTA's TMA producer fills its own
shared memory, but every copy completes on a barrier of the even CTA, which
alone arms the phases and issues the MMAs; the MMA commits arrive on
barriers of both CTAs (multicast); each CTA's epilogue releases an
accumulator with arrivals on the even CTA's barrier.  After an abort the
even CTA's producer retires the last phase of each ring from both CTAs'
issue counts (a phase the odd CTA filled but the even CTA never armed, or
the reverse) and waits for it, so that no CTA exits with a copy in flight.

This file restates that protocol as a small Python model, runs it under
random interleavings of the five roles and of every asynchronous completion
(TMA copies landing, MMA work completing in issue order), over random unit
lists, with and without an abort raised at a random step, and checks:
  * no deadlock (without an abort every role finishes);
  * every parity wait passes only on its own phase;
  * the MMA reads a stage (and the resident rows) only when both CTAs'
    copies of the right use have landed;
  * a producer overwrites a stage (or its rows) only after the MMAs reading
    the previous use have completed;
  * the epilogues read an accumulator only after the unit's MMAs completed,
    and the MMA overwrites it only after both epilogues released it;
  * the teardown completes every phase either CTA fed, so every copy has
    landed before exit.
Negative controls plant one mistake each (the odd CTA arming phases too, an
accumulator released by one CTA's epilogue, a teardown without the retire
step, rows reloaded without waiting for the MMAs) and must be caught.  The
model computes none of the expansion's arithmetic.
"""
import random

import pytest

STAGES = 5
CHUNKS = 8          # W stages per unit (the latent's 512 columns in 64-wide chunks)
STAGE, ROWS = 16, 128   # bytes a CTA's copy counts on the even CTA's barrier (model units)


class ProtocolError(RuntimeError):
    pass


class Barrier:
    """mbarrier: arrival count and transaction count (the count may go below
    zero while copies land before their phase is armed); waits test parity."""

    def __init__(self, count):
        self.count, self.pending, self.phase, self.tx = count, count, 0, 0

    def arrive(self, expect_tx=0):
        self.tx += expect_tx
        self.pending -= 1
        if self.pending < 0:
            raise ProtocolError("more arrivals than the barrier's count")
        self._complete()

    def complete_tx(self, n):
        self.tx -= n
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def test(self, k):
        passed = self.phase >= 1 and ((self.phase - 1) & 1) == (k & 1)
        if passed and self.phase != k + 1:
            raise ProtocolError(f"parity wait for phase {k} passed at phase {self.phase}")
        return passed


def uses_of(issued, s):
    """How many of the first `issued` round-robin uses fell on stage s."""
    return (issued - 1 - s) // STAGES + 1 if issued > s else 0


def retire(bar, mine, peer, nbytes):
    """The even CTA's teardown step for one ring slot (its barrier's last phase)."""
    n = max(mine, peer)
    if n == 0:
        return 0
    if mine < n:
        bar.arrive(expect_tx=2 * nbytes)
        bar.complete_tx(nbytes)
    elif peer < n:
        bar.complete_tx(nbytes)
    return n


def run_model(units, seed, abort_at=None, odd_arms=False, single_release=False, no_retire=False,
              reload_unguarded=False, slow_mma=False):
    """units: the pair's (token block, head) list in order.
    abort_at: (cta, step) — that CTA's abort flag goes up after `step` model
    steps (a wait that timed out); its roles leave at their next wait."""
    rng = random.Random(seed)
    full = [Barrier(1) for _ in range(STAGES)]                        # even CTA
    empty = [[Barrier(1) for _ in range(STAGES)] for _ in range(2)]   # [cta][stage]
    a_full = Barrier(1)                                               # even CTA
    a_empty = [Barrier(1), Barrier(1)]
    acc_full = [[Barrier(1), Barrier(1)] for _ in range(2)]           # [cta][buffer]
    acc_empty = [Barrier(1 if single_release else 2) for _ in range(2)]  # even CTA
    abort = [False, False]
    stage_use = [[None] * STAGES for _ in range(2)]   # use landed in each CTA's stage
    rows_use = [None, None]
    in_flight = []                                    # (cta, kind, stage, use, barrier)
    mma_queue = []                                    # in issue order: ("read", stage, use) | ("acc", buf, unit) | ("arrive", [bars])
    acc_done = {0: None, 1: None}                     # buffer -> unit whose MMAs completed into it
    released = {0: set(), 1: set()}                   # buffer -> CTAs whose epilogue released it
    issued = {"w": [0, 0], "a": [0, 0]}

    def reads_pending(stage=None):
        return any(k == "read" and (stage is None or x == stage) for k, x, _ in mma_queue)

    def producer(cta):
        g, na, cur = 0, 0, None
        for tb, _h in units:
            if tb != cur:
                if na > 0 and not reload_unguarded:
                    while not a_empty[cta].test(na - 1):
                        if abort[cta]:
                            return
                        yield
                if reads_pending():
                    raise ProtocolError(f"CTA {cta} reloads its rows while MMAs still read them")
                if cta == 0 or odd_arms:
                    a_full.arrive(expect_tx=2 * ROWS)
                in_flight.append((cta, "rows", None, na, a_full))
                na += 1
                issued["a"][cta] = na
                cur = tb
                yield
            for _ in range(CHUNKS):
                s, use = g % STAGES, g // STAGES
                if use > 0:
                    while not empty[cta][s].test(use - 1):
                        if abort[cta]:
                            return
                        yield
                if reads_pending(s):
                    raise ProtocolError(f"CTA {cta} overwrites stage {s} while MMAs read it")
                if cta == 0 or odd_arms:
                    full[s].arrive(expect_tx=2 * STAGE)
                in_flight.append((cta, "w", s, use, full[s]))
                g += 1
                issued["w"][cta] = g
                yield

    def mma():
        g, na, cur = 0, 0, None
        for j, (tb, _h) in enumerate(units):
            if tb != cur:
                if na > 0:
                    mma_queue.append(("arrive", [a_empty[0], a_empty[1]], None))
                while not a_full.test(na):
                    if abort[0]:
                        return
                    yield
                if rows_use != [na, na]:
                    raise ProtocolError("MMA reads rows before both CTAs' copies landed")
                na += 1
                cur = tb
            buf, use = j & 1, j >> 1
            if use > 0:
                while not acc_empty[buf].test(use - 1):
                    if abort[0]:
                        return
                    yield
                if released[buf] != {0, 1}:
                    raise ProtocolError(f"accumulator {buf} reused before both epilogues released it")
            released[buf] = set()
            for _ in range(CHUNKS):
                s = g % STAGES
                while not full[s].test(g // STAGES):
                    if abort[0]:
                        return
                    yield
                if [stage_use[0][s], stage_use[1][s]] != [g // STAGES] * 2:
                    raise ProtocolError(f"MMA reads stage {s} before both CTAs' copies of use {g // STAGES} landed")
                mma_queue.append(("read", s, g // STAGES))
                mma_queue.append(("arrive", [empty[0][s], empty[1][s]], None))
                g += 1
                yield
            mma_queue.append(("acc", buf, j))
            mma_queue.append(("arrive", [acc_full[0][buf], acc_full[1][buf]], None))
            yield

    def epilogue(cta):
        for j in range(len(units)):
            buf = j & 1
            while not acc_full[cta][buf].test(j >> 1):
                if abort[cta]:
                    return
                yield
            if acc_done[buf] != j:
                raise ProtocolError(f"epilogue of CTA {cta} reads accumulator {buf} before unit {j} completed")
            yield   # TMEM loads, bf16 staging, TMA stores
            released[buf].add(cta)
            acc_empty[buf].arrive()

    def land(i):
        cta, kind, s, use, bar = in_flight.pop(i)
        if kind == "w":
            stage_use[cta][s] = use
            bar.complete_tx(STAGE)
        else:
            rows_use[cta] = use
            bar.complete_tx(ROWS)

    def complete_mma():
        kind, x, y = mma_queue.pop(0)
        if kind == "acc":
            acc_done[x] = y
        elif kind == "arrive":
            for b in x:
                b.arrive()

    live = {"p0": producer(0), "p1": producer(1), "mma": mma(), "e0": epilogue(0), "e1": epilogue(1)}
    steps = idle = 0
    while live:
        steps += 1
        if abort_at is not None and steps == abort_at[1]:
            abort[abort_at[0]] = True
        sig = (len(in_flight), len(mma_queue), len(live), tuple(issued["w"]), tuple(issued["a"]),
               sum(b.phase for b in full), a_full.phase, sum(b.phase for b in acc_empty),
               sum(b.phase for r in acc_full for b in r), len(released[0]) + len(released[1]))
        c = rng.choice(list(live) + ["copy lands"] * (len(in_flight) > 0) + ["MMA completes"] * (len(mma_queue) > 0))
        if c == "MMA completes" and slow_mma and rng.random() < 0.9:
            c = rng.choice(list(live))    # a slow tensor pipe: completions lag far behind issue
        if c == "copy lands":
            land(rng.randrange(len(in_flight)))
        elif c == "MMA completes":
            complete_mma()
        else:
            try:
                next(live[c])
            except StopIteration:
                del live[c]
        new = (len(in_flight), len(mma_queue), len(live), tuple(issued["w"]), tuple(issued["a"]),
               sum(b.phase for b in full), a_full.phase, sum(b.phase for b in acc_empty),
               sum(b.phase for r in acc_full for b in r), len(released[0]) + len(released[1]))
        idle = idle + 1 if new == sig else 0
        if idle > 5000:
            if not any(abort):
                raise ProtocolError("deadlock: no role or completion makes progress")
            abort[0] = abort[1] = True   # the other CTA's bounded waits expire too
            idle = 0

    # The MMAs in flight complete before TMEM is released (fin); some copies
    # may still be landing while the even CTA retires the rings' last phases.
    while mma_queue:
        complete_mma()
    rng.shuffle(in_flight)
    for _ in range(rng.randrange(len(in_flight) + 1)):
        land(0)
    counts = []
    for s in range(STAGES):
        mine, peer = uses_of(issued["w"][0], s), uses_of(issued["w"][1], s)
        if abs(mine - peer) > 1:
            raise ProtocolError("the CTAs' uses of a stage drifted more than one apart")
        counts.append((full[s], retire(full[s], mine, peer, STAGE) if not no_retire else max(mine, peer)))
    if abs(issued["a"][0] - issued["a"][1]) > 1:
        raise ProtocolError("the CTAs' row loads drifted more than one apart")
    counts.append((a_full, retire(a_full, issued["a"][0], issued["a"][1], ROWS) if not no_retire
                   else max(issued["a"])))
    while in_flight:
        land(0)
    for bar, n in counts:
        if bar.phase != n:
            raise ProtocolError(f"a ring phase ({bar.phase} of {n}) never completes: its drain would time out")
    if not any(abort) and (issued["w"] != [CHUNKS * len(units)] * 2 or released[(len(units) - 1) & 1] != {0, 1}):
        raise ProtocolError("the pair stopped early without an abort")
    return steps


def random_units(rng):
    """A pair's contiguous range of (256-token block, head) units, block-major."""
    n = rng.randint(1, 9)
    u0 = rng.randrange(0, 3 * 128)
    return [((u0 + i) >> 7, (u0 + i) & 127) for i in range(n)]


@pytest.mark.parametrize("seed", range(150))
def test_pair_protocol_random(seed):
    rng = random.Random(1000 + seed)
    run_model(random_units(rng), seed, slow_mma=seed % 2 == 1)


def test_pair_protocol_row_reloads():
    """Ranges that cross token blocks (the rows are reloaded) under many interleavings."""
    for seed in range(80):
        run_model([(0, 126), (0, 127), (1, 0), (1, 1), (1, 2)], seed)


@pytest.mark.parametrize("seed", range(120))
def test_pair_protocol_abort(seed):
    rng = random.Random(5000 + seed)
    units = random_units(rng)
    run_model(units, seed, abort_at=(rng.randrange(2), rng.randrange(1, 60 * len(units) + 2)))


def _caught(**kw):
    hits = 0
    for seed in range(60):
        try:
            run_model([(0, 125), (0, 126), (0, 127), (1, 0), (1, 1)], seed, **kw)
        except ProtocolError:
            hits += 1
    return hits


def test_control_odd_cta_arms():
    assert _caught(odd_arms=True) > 0


def test_control_single_release():
    assert _caught(single_release=True) > 0


def test_control_reload_unguarded():
    assert _caught(reload_unguarded=True) > 0


def test_control_teardown_without_retire():
    hits = 0
    for seed in range(200):
        rng = random.Random(7000 + seed)
        units = random_units(rng)
        try:
            run_model(units, seed, abort_at=(rng.randrange(2), rng.randrange(1, 60 * len(units) + 2)),
                      no_retire=True)
        except ProtocolError:
            hits += 1
    assert hits > 0
