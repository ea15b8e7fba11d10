"""Model check of the decode kernel's synchronisation protocol (CPU only).

The decode kernel (csrc/decode_paged.cu) coordinates seven roles per CTA and
two CTAs per cluster through mbarriers, a score-exchange ring in distributed
shared memory and tagged shared-memory slots.  Hardware mbarrier waits test
a phase *parity*, so a waiter that runs two phases ahead of the barrier
passes early; a buffer reused too soon is overwritten before it is read.
Neither shows up as a fault on the GPU: the first reads stale data, the
second corrupts it, and a wrong ordering hangs until the kernel's bounded
waits expire.

This file restates the protocol as a small Python model and runs it under
random interleavings of every role and every asynchronous completion (TMA
loads, MMA completions, copies landing in the peer CTA), over random segment
layouts.  It checks:
  * no deadlock (some role or completion can always make progress);
  * every parity wait passes only when its own phase has completed;
  * no exchange buffer region is overwritten while it holds unconsumed
    scores or while a copy out of it is still reading it;
  * no reference-max slot is overwritten before its reader has read it.
In the FP8 layout P·V of tile t also waits until QK^T of tile t+2 is
issued (the kernel orders the tensor pipe that way there).
Negative controls re-introduce, one at a time, a single shared score barrier,
two hand-off slots instead of four, and a staging offset of one or three
buffers; each must be caught.  The model is test infrastructure for the
kernel's control flow only: it computes none of the attention arithmetic.
"""
import random

import pytest

STAGES = 4      # page ring
XBUFS = 4       # exchange ring depth
WARPS = 2       # row blocks per warpgroup modelled (the kernel has 4)


class ProtocolError(RuntimeError):
    pass


class Barrier:
    """mbarrier with an arrival count and a transaction count; waits test parity."""

    def __init__(self, count):
        self.count, self.pending, self.phase, self.tx = count, count, 0, 0

    def arrive(self, n=1, expect_tx=0):
        self.tx += expect_tx
        self.pending -= n
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
        """Hardware semantics: true iff the last completed phase has k's parity."""
        passed = self.phase >= 1 and ((self.phase - 1) & 1) == (k & 1)
        if passed and self.phase != k + 1:
            raise ProtocolError(f"parity wait for phase {k} passed at phase {self.phase}")
        return passed


def run_model(segs, seed, shared_s_full=False, slots=4, xlead=2, fp8=False, conv_no_barrier=False,
              conv_skips_f8_full=False, abort_at=None, drain=True):
    """fp8: the FP8 layout — the producer's TMA fills stage t mod STAGES with
    codes, the converter warps read all of their codes, meet at a barrier and
    write the bf16 rows over them, and QK^T waits for all converter warps.
    Planted mistakes: converters without the barrier (a warp overwrites codes
    another warp has not read yet) and converters that do not wait for the
    codes to land.
    abort_at: (cta, step) — that CTA's abort flag goes up after `step` model
    steps (a wait that timed out); every role then leaves at its next wait.
    After the roles, each CTA tells the peer how many score copies each warp
    issued, both meet at the cluster barrier, a CTA that or whose peer aborted
    drains the copies still in flight into it (retiring by hand the bytes of
    copies never issued), and both meet again before they exit.  drain=False
    plants the mistake of exiting without the drain."""
    rnd = random.Random(seed)
    n_stages = STAGES
    tiles = []
    for si, n in enumerate(segs):
        for i in range(n):
            tiles.append((si, i == 0, i == n - 1))
    G = len(tiles)
    WG_THREADS = 128
    per_warp = WG_THREADS // WARPS
    ctas = []
    for _ in range(2):
        ctas.append(dict(
            kv_full=[Barrier(WARPS if fp8 else 1) for _ in range(n_stages)],
            kv_empty=[Barrier(1) for _ in range(n_stages)],
            f8_full=[Barrier(1) for _ in range(n_stages)],
            stage=[None] * n_stages,        # (tile, "codes" | "bf16") held by a stage
            codes_read=[set() for _ in range(n_stages)],   # converter warps that have read this tile's codes
            conv=Barrier(WARPS),            # converters' mbarrier: phase t = every warp holds tile t's codes
            s_full=[Barrier(1), Barrier(1)], s_free=Barrier(WG_THREADS), p_full=Barrier(WG_THREADS),
            o_done=[Barrier(1), Barrier(1)], q_ready=Barrier(WG_THREADS), o_free=Barrier(WG_THREADS),
            x_full=[Barrier(1) for _ in range(XBUFS)],
            xbuf=[[None] * WARPS for _ in range(XBUFS)],   # region state per (buffer, row block)
            reading=[[False] * WARPS for _ in range(XBUFS)],  # a copy out of this region is in flight
            slot=[[None] * WARPS for _ in range(slots)], slot_unread=[[False] * WARPS for _ in range(slots)],
            abort=False, pushes=[0] * (2 * WARPS), peer_pushes=None, peer_abort=None,
            armed=[-1] * XBUFS, exited=False, qk_issued=-1,
        ))
    events = []

    def wait(c, cond):
        """Yield until cond() holds; False if the CTA's abort flag went up
        first.  Once either CTA has aborted, a wait also gives up (and raises
        its own CTA's flag) after a while: the kernel's waits are bounded."""
        n = 0
        while not cond():
            if c["abort"]:
                return False
            n += 1
            if n > 200 and any(x["abort"] for x in ctas):
                c["abort"] = True
                return False
            yield
        return True

    def s_full_bar(c, t):
        return (c["s_full"][0], t) if shared_s_full else (c["s_full"][t & 1], t >> 1)

    def o_done_bar(c, t):
        return (c["o_done"][0], t) if shared_s_full else (c["o_done"][t & 1], t >> 1)

    def producer(ci):
        c = ctas[ci]
        for t in range(G):
            if t >= STAGES:
                if not (yield from wait(c, lambda: c["kv_empty"][t % STAGES].test(t // STAGES - 1))):
                    return
            events.append(("f8" if fp8 else "kv", ci, t))

    def converter(ci, w):
        c = ctas[ci]
        for t in range(G):
            st = t % n_stages
            if not conv_skips_f8_full:
                if not (yield from wait(c, lambda: c["f8_full"][st].test(t // n_stages))):
                    return
            if c["stage"][st] != (t, "codes"):
                raise ProtocolError(f"converter {w} reads tile {t}'s codes from a stage holding {c['stage'][st]}")
            c["codes_read"][st].add(w)
            yield
            if not conv_no_barrier:
                c["conv"].arrive()
                if not (yield from wait(c, lambda: c["conv"].test(t))):
                    return
            if c["codes_read"][st] != set(range(WARPS)):
                raise ProtocolError(f"converter {w} overwrites tile {t}'s codes before every warp read them")
            yield
            c["kv_full"][st].arrive()
            if c["kv_full"][st].pending == WARPS:    # the last converter warp of this tile
                c["stage"][st] = (t, "bf16")
                c["codes_read"][st] = set()

    def qk(ci):
        c = ctas[ci]
        for t in range(G):
            if not (yield from wait(c, lambda: c["kv_full"][t % n_stages].test(t // n_stages))):
                return
            if fp8:
                if not (yield from wait(c, lambda: c["f8_full"][t % n_stages].test(t // n_stages))):
                    return
                if c["stage"][t % n_stages] != (t, "bf16"):
                    raise ProtocolError(f"QK^T of tile {t} reads a stage holding {c['stage'][t % n_stages]}")
            if t > 0:
                if not (yield from wait(c, lambda: c["s_free"].test(t - 1))):
                    return
            seg, first, _ = tiles[t]
            if first:
                if not (yield from wait(c, lambda: c["q_ready"].test(seg))):
                    return
            events.append(("s", ci, t))
            c["qk_issued"] = t

    def pv(ci):
        c = ctas[ci]
        for t in range(G):
            if not (yield from wait(c, lambda: c["p_full"].test(t))):
                return
            seg, first, _ = tiles[t]
            if first:
                if not (yield from wait(c, lambda: c["o_free"].test(seg))):
                    return
            # FP8: P·V(t) only after QK^T(t+2) is issued (tensor-pipe order)
            if fp8 and t + 2 < G:
                if not (yield from wait(c, lambda: c["qk_issued"] >= t + 2)):
                    return
            if fp8 and c["stage"][t % n_stages] != (t, "bf16"):
                raise ProtocolError(f"P·V of tile {t} reads a stage holding {c['stage'][t % n_stages]}")
            events.append(("o", ci, t))

    def softmax_warp(ci, wg, w):
        c = ctas[ci]
        if wg == 0:
            c["o_free"].arrive(per_warp)
            c["q_ready"].arrive(per_warp)
            if w == 0:
                for t in range(min(G, XBUFS)):
                    c["x_full"][t].arrive(1, expect_tx=WARPS)
                    c["armed"][t] = t
        for t in range(wg, G, 2):
            seg, first, last = tiles[t]
            bar, k = s_full_bar(c, t)
            if not (yield from wait(c, lambda: bar.test(k))):
                return
            c["s_free"].arrive(per_warp)
            # stage this row block's scores and push them to the peer
            sb = (t + xlead) % XBUFS
            state = c["xbuf"][sb][w]
            if state is not None and state[0] == "data":
                raise ProtocolError(f"staging tile {t} over unconsumed scores of tile {state[1]}")
            if c["reading"][sb][w]:
                raise ProtocolError(f"staging tile {t} over a copy still in flight")
            c["xbuf"][sb][w] = ("stage", t)
            c["reading"][sb][w] = True
            events.append(("x", ci, (t, w, sb)))
            c["pushes"][wg * WARPS + w] += 1
            if last and seg + 1 < len(segs):
                c["q_ready"].arrive(per_warp)
            yield
            # the peer's half of tile t
            b = t % XBUFS
            if not (yield from wait(c, lambda: c["x_full"][b].test(t // XBUFS))):
                return
            if c["xbuf"][b][w] != ("data", t):
                raise ProtocolError(f"tile {t} reads {c['xbuf'][b][w]}")
            c["xbuf"][b][w] = None
            if w == 0 and t + XBUFS < G:
                c["x_full"][b].arrive(1, expect_tx=WARPS)
                c["armed"][b] = t + XBUFS
            # reference max from tile t-1
            if not first:
                sl = (t - 1) % slots
                if not (yield from wait(c, lambda: c["slot"][sl][w] == t - 1)):
                    return
                c["slot_unread"][sl][w] = False
            sl = t % slots
            if c["slot_unread"][sl][w]:
                raise ProtocolError(f"tile {t} overwrites tile {c['slot'][sl][w]}'s max before it was read")
            c["slot"][sl][w] = t
            c["slot_unread"][sl][w] = t + 1 < G and not tiles[t + 1][1]
            yield
            if t > 0:
                bar, k = o_done_bar(c, t - 1)
                if not (yield from wait(c, lambda: bar.test(k))):
                    return
            c["p_full"].arrive(per_warp)
            if last:
                bar, k = o_done_bar(c, t)
                if not (yield from wait(c, lambda: bar.test(k))):
                    return
                c["o_free"].arrive(per_warp)

    def exit_sequence(ci):
        """After the roles: counts to the peer, cluster barrier, drain, barrier."""
        c, p = ctas[ci], ctas[1 - ci]
        p["peer_pushes"] = list(c["pushes"])
        p["peer_abort"] = c["abort"]
        c["at_barrier"] = 1
        while p.get("at_barrier", 0) < 1:
            yield
        if drain and (c["abort"] or c["peer_abort"]):
            for b in range(XBUFS):
                t = c["armed"][b]
                if t < 0:
                    continue
                k = t // XBUFS
                xb = c["x_full"][b]
                if xb.phase >= k + 1:
                    continue
                idx, pg = t >> 1, t & 1
                issued = sum(1 for q in range(WARPS) if c["peer_pushes"][pg * WARPS + q] > idx)
                if issued < WARPS:
                    xb.complete_tx(WARPS - issued)
                while xb.phase < k + 1:
                    yield
            c["at_barrier"] = 2
            while p.get("at_barrier", 0) < 2 and not p["exited"]:
                yield
        c["exited"] = True
        for kind, cj, payload in events:
            if kind == "x":
                raise ProtocolError(f"CTA {ci} exits with a score copy of CTA {cj} in flight")

    roles = {}
    for ci in range(2):
        roles[("prod", ci)] = producer(ci)
        roles[("qk", ci)] = qk(ci)
        roles[("pv", ci)] = pv(ci)
        if fp8:
            for w in range(WARPS):
                roles[("conv", ci, w)] = converter(ci, w)
        for wg in range(2):
            for w in range(WARPS):
                roles[("sm", ci, wg, w)] = softmax_warp(ci, wg, w)
    idle = 0
    pending_exit = {0, 1}
    steps = 0
    while roles or events:
        steps += 1
        if abort_at is not None and steps == abort_at[1]:
            ctas[abort_at[0]]["abort"] = True
        for ci in list(pending_exit):
            if not any(key[1] == ci for key in roles):
                pending_exit.discard(ci)
                roles[("exit", ci)] = exit_sequence(ci)
        pick = rnd.randrange(len(roles) + len(events))
        if pick >= len(roles) and events[pick - len(roles)][0] == "x" and any(x["abort"] for x in ctas):
            # after an abort, copies in flight linger until every role has left
            working = [k for k in roles if k[0] != "exit"]
            if working:
                pick = list(roles).index(rnd.choice(working))
        if pick >= len(roles):
            kind, ci, t = events.pop(pick - len(roles))
            c = ctas[ci]
            if kind == "kv":
                c["kv_full"][t % STAGES].arrive()
            elif kind == "f8":
                st = t % n_stages
                held = c["stage"][st]
                if held is not None and held != (t - n_stages, "free"):
                    raise ProtocolError(f"tile {t}'s codes land over a stage holding {held}")
                c["stage"][st] = (t, "codes")
                c["f8_full"][st].arrive()
            elif kind == "s":
                bar, _ = s_full_bar(c, t)
                bar.arrive()
            elif kind == "o":
                if fp8:
                    c["stage"][t % n_stages] = (t, "free")
                c["kv_empty"][t % n_stages].arrive()
                bar, _ = o_done_bar(c, t)
                bar.arrive()
            else:  # a row block's copy lands in the peer's buffer t mod XBUFS
                tile, w, sb = t
                p = ctas[1 - ci]
                if p["exited"] or c["exited"]:
                    raise ProtocolError(f"a copy of tile {tile} lands after a CTA exited")
                b = tile % XBUFS
                state = p["xbuf"][b][w]
                if state is not None and state[0] == "data":
                    raise ProtocolError(f"tile {tile} lands over unconsumed tile {state[1]}")
                if p["reading"][b][w]:
                    raise ProtocolError(f"tile {tile} lands over staging still being copied")
                p["xbuf"][b][w] = ("data", tile)
                c["reading"][sb][w] = False
                p["x_full"][b].complete_tx(1)
            idle = 0
            continue
        key = list(roles)[pick]
        try:
            next(roles[key])
            idle += 1
        except StopIteration:
            del roles[key]
            idle = 0
        if idle > 50000:
            raise ProtocolError(f"deadlock; roles still running: {sorted(map(str, roles))}")
    if abort_at is None:
        for c in ctas:
            if not c["exited"]:
                raise ProtocolError("a CTA never reached its exit")


def _layouts(n, seed):
    rng = random.Random(seed)
    for _ in range(n):
        yield [rng.choice([1, 1, 2, 3, 5, 9]) for _ in range(rng.randint(1, 7))]


def test_protocol_holds_on_random_interleavings():
    for i, segs in enumerate(_layouts(150, 11)):
        run_model(segs, seed=i)


def test_protocol_holds_on_single_tile_segments():
    # the layout whose hazards were found on the GPU: many one-tile segments
    for seed in range(100):
        run_model([1, 1, 1, 1, 2, 2, 3, 3, 11], seed)


@pytest.mark.parametrize("mistake", [dict(shared_s_full=True), dict(slots=2), dict(xlead=1), dict(xlead=3)])
def test_planted_protocol_mistakes_are_caught(mistake):
    caught = 0
    for i, segs in enumerate(_layouts(60, 12)):
        try:
            run_model(segs + [1, 1, 3], seed=i, **mistake)
        except ProtocolError:
            caught += 1
    assert caught > 0, f"the model did not catch {mistake}"


def test_abort_drains_every_copy_before_exit():
    # either CTA's abort flag goes up at a random point; neither may exit
    # while a score copy into or out of its shared memory is in flight
    rng = random.Random(31)
    for i, segs in enumerate(_layouts(200, 32)):
        run_model(segs, seed=i, abort_at=(rng.randrange(2), rng.randrange(1, 3000)))
    for i, segs in enumerate(_layouts(60, 35)):
        run_model(segs, seed=i, fp8=True, abort_at=(rng.randrange(2), rng.randrange(1, 3000)))


def test_exit_without_drain_is_caught():
    rng = random.Random(33)
    caught = 0
    for i, segs in enumerate(_layouts(200, 34)):
        try:
            run_model(segs + [3, 5], seed=i, abort_at=(rng.randrange(2), rng.randrange(1, 3000)), drain=False)
        except ProtocolError:
            caught += 1
    assert caught > 0, "the model did not catch an exit with copies in flight"


def test_fp8_protocol_holds_on_random_interleavings():
    for i, segs in enumerate(_layouts(120, 21)):
        run_model(segs, seed=i, fp8=True)
    for seed in range(60):
        run_model([1, 1, 1, 1, 2, 2, 3, 3, 11], seed, fp8=True)


@pytest.mark.parametrize("mistake", [dict(conv_no_barrier=True), dict(conv_skips_f8_full=True)])
def test_planted_fp8_protocol_mistakes_are_caught(mistake):
    caught = 0
    for i, segs in enumerate(_layouts(60, 22)):
        try:
            run_model(segs + [1, 1, 3], seed=i, fp8=True, **mistake)
        except ProtocolError:
            caught += 1
    assert caught > 0, f"the model did not catch {mistake}"


def run_converter_abort_model(seed, tiles=6, warps=4, arrive_on_leave=True, check_flag=True):
    """The FP8 converters' exit protocol around their named barrier.  Each tile
    a warp passes its stage wait, or gives up (a timeout raises the CTA's abort
    flag; a wait that finds the flag up gives up too); it then checks the
    flag and syncs on the hardware barrier (which completes when `warps`
    arrivals are in, then starts its next generation).  A warp that leaves
    arrives first without waiting.  Returns once every warp has left or
    finished; a warp blocked for good in the barrier is a deadlock."""
    rnd = random.Random(seed)
    st = {"flag": False, "count": 0, "gen": 0}
    timeout_at = (rnd.randrange(warps), rnd.randrange(tiles))   # the warp and tile whose wait times out

    def arrive():
        st["count"] += 1
        if st["count"] == warps:
            st["count"] = 0
            st["gen"] += 1

    def warp(w):
        for t in range(tiles):
            yield
            gave_up = st["flag"] and rnd.random() < 0.5        # a wait that finds the flag up may give up
            if (w, t) == timeout_at:
                st["flag"] = True
                gave_up = True
            if gave_up:
                if arrive_on_leave:
                    arrive()
                return
            yield
            if check_flag and st["flag"]:
                if arrive_on_leave:
                    arrive()
                return
            g = st["gen"]
            arrive()
            while st["gen"] == g:
                yield

    roles = {w: warp(w) for w in range(warps)}
    idle = 0
    while roles:
        key = rnd.choice(list(roles))
        try:
            next(roles[key])
            idle += 1
        except StopIteration:
            del roles[key]
            idle = 0
        if idle > 5000:
            raise ProtocolError(f"converter warps {sorted(roles)} blocked in the barrier")


def test_converter_exit_never_blocks_a_warp():
    for seed in range(400):
        run_converter_abort_model(seed)


@pytest.mark.parametrize("mistake", [dict(arrive_on_leave=False), dict(check_flag=False)])
def test_converter_exit_mistakes_are_caught(mistake):
    caught = 0
    for seed in range(400):
        try:
            run_converter_abort_model(seed, **mistake)
        except ProtocolError:
            caught += 1
    assert caught > 0, f"the model did not catch {mistake}"
