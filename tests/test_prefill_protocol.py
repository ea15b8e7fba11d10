"""Model check of the decompress-branch attention kernel's synchronisation
(csrc/prefill_attn.cu), CPU only.

The kernel's roles — a TMA producer that issues K and V loads into two
2-deep rings as their stages free up, one thread that issues QK^T(j) into
one of two S buffers, another that issues P·V(j), and softmax warps
in pairs that swap row maxima through a tile-parity buffer — are restated
here with hardware parity semantics for every mbarrier wait and run under
random interleavings of the roles and of every asynchronous completion
(loads landing, MMAs completing).  Checks: no deadlock; every parity wait
passes only in its own phase; no K/V stage, S buffer, P buffer or max slot
is overwritten while its previous contents are still to be read.  Planted
mistakes (a softmax that writes P without waiting for P·V(j-1), one S
buffer, one max slot, a producer that ignores the V ring's release) are
each caught.
"""
import random

import pytest

STAGES = 2
SOFT = 4          # softmax warps modelled (two pairs)


class ProtocolError(RuntimeError):
    pass


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.phase, self.tx = count, count, 0, 0

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise ProtocolError("more arrivals than the barrier's count")
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def test(self, k):
        passed = self.phase >= 1 and ((self.phase - 1) & 1) == (k & 1)
        if passed and self.phase != k + 1:
            raise ProtocolError(f"parity wait for phase {k} passed at phase {self.phase}")
        return passed


def run_model(n_tiles, seed, wait_o_done=True, s_buffers=2, xmax_slots=2, wait_v_empty=True):
    rnd = random.Random(seed)
    B = dict(k_full=[Barrier(1) for _ in range(STAGES)], k_empty=[Barrier(1) for _ in range(STAGES)],
             v_full=[Barrier(1) for _ in range(STAGES)], v_empty=[Barrier(1) for _ in range(STAGES)],
             s_full=[Barrier(1) for _ in range(2)], s_free=[Barrier(SOFT) for _ in range(2)],
             p_full=Barrier(SOFT), o_done=Barrier(1), xmax=[Barrier(SOFT) for _ in range(2)])
    k_stage = [None] * STAGES      # tile held, or None
    k_reading = [None] * STAGES    # QK^T reading this stage (tile)
    v_stage = [None] * STAGES
    v_reading = [None] * STAGES
    s_buf = [None] * 2             # tile whose scores a buffer holds, still to be read by some warps
    s_unread = [set() for _ in range(2)]
    p_buf = {"tile": None, "reading": False}
    p_written = set()
    xslot = [dict() for _ in range(2)]   # warp -> tile of the value it wrote
    events = []

    def s_idx(j):
        return j % s_buffers

    def producer():
        nk = nv = 0
        while nv < n_tiles:
            progressed = False
            if nk < n_tiles and (nk < STAGES or B["k_empty"][nk % STAGES].test((nk - STAGES) // STAGES)):
                st = nk % STAGES
                if k_reading[st] is not None:
                    raise ProtocolError(f"K({nk}) lands over stage {st} while QK^T({k_reading[st]}) reads it")
                events.append(("k", nk))
                nk += 1
                progressed = True
            if nv < nk and (nv < STAGES or not wait_v_empty or B["v_empty"][nv % STAGES].test((nv - STAGES) // STAGES)):
                events.append(("v", nv))
                nv += 1
                progressed = True
            if not progressed:
                yield

    def qk():
        for nq in range(n_tiles):
            while not (B["k_full"][nq % STAGES].test(nq // STAGES) and
                       (nq < 2 or B["s_free"][s_idx(nq)].test((nq - 2) // 2 if s_buffers == 2 else nq - 1))):
                yield
            if k_stage[nq % STAGES] != nq:
                raise ProtocolError(f"QK^T({nq}) reads a K stage holding {k_stage[nq % STAGES]}")
            b = s_idx(nq)
            if s_unread[b]:
                raise ProtocolError(f"QK^T({nq}) overwrites S({s_buf[b]}) before every warp read it")
            k_reading[nq % STAGES] = nq
            events.append(("qk", nq))
            yield

    def pv():
        for np_ in range(n_tiles):
            while not (B["p_full"].test(np_) and B["v_full"][np_ % STAGES].test(np_ // STAGES)):
                yield
            if v_stage[np_ % STAGES] != np_ or p_buf["tile"] != np_:
                raise ProtocolError(f"P·V({np_}) reads V/P of another tile")
            v_reading[np_ % STAGES] = np_
            p_buf["reading"] = True
            events.append(("pv", np_))
            yield

    def softmax(w):
        for j in range(n_tiles):
            b = s_idx(j)
            while not B["s_full"][b].test(j // 2 if s_buffers == 2 else j):
                yield
            if s_buf[b] != j or w not in s_unread[b]:
                raise ProtocolError(f"warp {w} reads S({s_buf[b]}) for tile {j}")
            s_unread[b].discard(w)
            B["s_free"][b].arrive()
            yield
            slot = xslot[j % xmax_slots]
            partner = w ^ 1
            if slot.get(partner) is not None and slot[partner] < j and ("read", partner, slot[partner]) not in p_written:
                raise ProtocolError(f"warp {w} overwrites the max slot its partner has not read (tile {slot[partner]})")
            slot[w] = j
            B["xmax"][j % 2].arrive()
            while not B["xmax"][j % 2].test(j // 2):
                yield
            if slot.get(partner) != j:
                raise ProtocolError(f"warp {w} reads its partner's max of tile {slot.get(partner)} for tile {j}")
            p_written.add(("read", w, j))
            yield
            if j > 0 and wait_o_done:
                while not B["o_done"].test(j - 1):
                    yield
            if p_buf["reading"] and p_buf["tile"] != j:
                raise ProtocolError(f"P({j}) overwrites P({p_buf['tile']}) while P·V reads it")
            p_buf["tile"] = j
            B["p_full"].arrive()

    roles = {"prod": producer(), "qk": qk(), "pv": pv()}
    for w in range(SOFT):
        roles[("sm", w)] = softmax(w)
    idle = 0
    while roles or events:
        pick = rnd.randrange(len(roles) + len(events))
        if pick >= len(roles):
            kind, j = events.pop(pick - len(roles))
            st = j % STAGES
            if kind == "k":
                k_stage[st] = j
                B["k_full"][st].arrive()
            elif kind == "v":
                if v_reading[st] is not None:
                    raise ProtocolError(f"V({j}) lands over stage {st} while P·V({v_reading[st]}) reads it")
                v_stage[st] = j
                B["v_full"][st].arrive()
            elif kind == "qk":                     # QK^T(j) completes: S_FULL and the K stage's release
                b = s_idx(j)
                s_buf[b] = j
                s_unread[b] = set(range(SOFT))
                k_reading[st] = None
                B["s_full"][b].arrive()
                B["k_empty"][st].arrive()
            else:                                  # P·V(j) completes: the V stage's release and O_DONE
                v_reading[st] = None
                p_buf["reading"] = False
                B["v_empty"][st].arrive()
                B["o_done"].arrive()
            idle = 0
            continue
        key = list(roles)[pick]
        try:
            next(roles[key])
            idle += 1
        except StopIteration:
            del roles[key]
            idle = 0
        if idle > 20000:
            raise ProtocolError(f"deadlock; roles still running: {sorted(map(str, roles))}")


def test_prefill_protocol_holds():
    for seed in range(300):
        run_model(random.Random(seed).randint(1, 9), seed)


@pytest.mark.parametrize("mistake", [dict(wait_o_done=False), dict(s_buffers=1), dict(xmax_slots=1),
                                     dict(wait_v_empty=False)])
def test_planted_prefill_mistakes_are_caught(mistake):
    caught = 0
    for seed in range(200):
        try:
            run_model(random.Random(seed).randint(3, 9), seed, **mistake)
        except ProtocolError:
            caught += 1
    assert caught > 0, f"the model did not catch {mistake}"
