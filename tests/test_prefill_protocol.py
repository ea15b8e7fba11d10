"""Model check of the prefill attention kernel's synchronisation (CPU only).

The attention kernel of the decompress branch (csrc/prefill_attn.cu) runs
five roles per CTA: a TMA producer (Q into the third key stage, then a
3-deep key ring and a 2-deep value ring), a QK^T issuer, a P·V issuer that
waits until QK^T two tiles ahead is issued, and the softmax warps, two per
TMEM lane quarter, which swap their halves' row maxima through a
tile-parity slot and a named barrier of the pair.  TMEM holds Q, one score
buffer and two P buffers.  A parity wait that runs two phases ahead, a
buffer reused too early or a named barrier left waiting for a partner that
has gone shows up on the GPU as wrong numbers or a hang, not as a fault.

This file restates the protocol as a Python model (one lane quarter: its
two softmax warps) and runs it under random interleavings of the roles and
of the asynchronous completions (TMA copies landing, MMAs completing in
their issue order through one tensor pipe), with and without an abort
raised at a random step.  It checks that every read sees the tile it is
meant to (K, V, Q, S, P, the partner's maximum), that no buffer is
overwritten while a read of it is pending, that every parity wait passes
on its own phase, and that the roles always finish (no deadlock, no named
barrier waiting for ever).  Negative controls plant one mistake each and
must be caught.  The model computes none of the attention arithmetic.
"""
import random

import pytest

KST, VST = 3, 2          # key ring and value ring depths
QSTAGE = 2               # the key stage Q lands in
LAG = 2                  # P·V(t) waits until QK^T(t + LAG) is issued


class ProtocolError(RuntimeError):
    pass


class Barrier:
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


class NamedBarrier:
    """bar.sync / bar.arrive over two warps: a sync returns once two arrivals
    (syncs or arrives) of its generation are in."""

    def __init__(self):
        self.gen, self.count = 0, 0

    def arrive(self):
        self.count += 1
        if self.count == 2:
            self.gen, self.count = self.gen + 1, 0

    def sync(self):
        g = self.gen
        self.arrive()
        while self.gen == g:
            yield "named"


def run_model(n_tiles, seed, abort_at=None, no_abort_check=False, p_without_wait=False, qk_without_sfree=False,
              k2_without_q=False, single_xmax=False, rescale_every=5):
    rng = random.Random(seed)
    q_full, q_tmem = Barrier(1), Barrier(2)
    k_full = [Barrier(1) for _ in range(KST)]
    k_empty = [Barrier(1) for _ in range(KST)]
    v_full = [Barrier(1) for _ in range(VST)]
    v_empty = [Barrier(1) for _ in range(VST)]
    s_full, s_free = [Barrier(1), Barrier(1)], [Barrier(2), Barrier(2)]
    p_full, o_done = [Barrier(2), Barrier(2)], [Barrier(1), Barrier(1)]
    nbar = NamedBarrier()
    abort = [False]
    st = {"k": [None] * KST, "v": [None] * VST, "S": None, "P": [None, None], "xmax": {}, "qk_issued": -1,
          "q_copied": 0}
    in_flight, pipe = [], []     # copies; tensor-pipe queue in issue order
    reading = []                 # pending MMA reads: (kind, index, tile)

    def pending_read(kind, idx):
        return any(r[0] == kind and r[1] == idx for r in reading)

    # ------------------------------------------------------------ producer
    def producer():
        in_flight.append(("k", QSTAGE, "Q", q_full))
        q_full.arrive(expect_tx=1)
        nk = nv = 0
        while nv < n_tiles:
            if abort[0]:
                return
            progressed = False
            if nk < n_tiles:
                s = nk % KST
                if nk < KST:
                    ready = nk != QSTAGE or k2_without_q or q_tmem.test(0)
                else:
                    ready = k_empty[s].test((nk - KST) // KST)
                if ready:
                    if pending_read("k", s):
                        raise ProtocolError(f"key stage {s} refilled while QK^T still reads it")
                    if s == QSTAGE and st["q_copied"] < 2:
                        raise ProtocolError("key stage 2 refilled before Q was copied out of it")
                    k_full[s].arrive(expect_tx=1)
                    in_flight.append(("k", s, nk, k_full[s]))
                    nk += 1
                    progressed = True
            if nv < nk:
                s = nv % VST
                if nv < VST or v_empty[s].test((nv - VST) // VST):
                    if pending_read("v", s):
                        raise ProtocolError(f"value stage {s} refilled while P·V still reads it")
                    v_full[s].arrive(expect_tx=1)
                    in_flight.append(("v", s, nv, v_full[s]))
                    nv += 1
                    progressed = True
            yield "producer" if progressed else "wait"

    # ------------------------------------------------------------ QK^T issue
    def qk():
        while not q_tmem.test(0):
            if abort[0]:
                return
            yield "wait"
        for j in range(n_tiles):
            s = j % KST
            while not (k_full[s].test(j // KST) and
                       (j < 1 or qk_without_sfree or s_free[(j - 1) & 1].test((j - 1) >> 1))):
                if abort[0]:
                    return
                yield "wait"
            if st["k"][s] != j:
                raise ProtocolError(f"QK^T({j}) reads a key stage holding {st['k'][s]}")
            reading.append(("k", s, j))
            pipe.append(("qk", j))
            pipe.append(("arrive", [s_full[j & 1], k_empty[s]], ("k", s, j)))
            st["qk_issued"] = j
            yield "qk"

    # ------------------------------------------------------------ P·V issue
    def pv():
        for t in range(n_tiles):
            while not (p_full[t & 1].test(t >> 1) and v_full[t % VST].test(t // VST)):
                if abort[0]:
                    return
                yield "wait"
            while LAG > 0 and t + LAG < n_tiles and st["qk_issued"] < t + LAG:
                if abort[0]:
                    return
                yield "wait"
            if st["P"][t & 1] != ("full", t):
                raise ProtocolError(f"P·V({t}) reads P buffer {t & 1} holding {st['P'][t & 1]}")
            if st["v"][t % VST] != t:
                raise ProtocolError(f"P·V({t}) reads a value stage holding {st['v'][t % VST]}")
            reading.append(("p", t & 1, t))
            reading.append(("v", t % VST, t))
            pipe.append(("pv", t))
            pipe.append(("arrive", [v_empty[t % VST], o_done[t & 1]], ("pv", t, t)))
            yield "pv"

    # ------------------------------------------------------------ softmax warps
    def softmax(half):
        ok = True
        while not q_full.test(0):
            if abort[0]:
                ok = False
                break
            yield "wait"
        if ok:
            if st["k"][QSTAGE] != "Q":
                raise ProtocolError("Q copied from a stage that no longer holds it")
            st["q_copied"] += 1
            q_tmem.arrive()
            yield "copy"
        for j in range(n_tiles if ok else 0):
            sb = j & 1
            while not s_full[sb].test(j >> 1):
                if abort[0]:
                    ok = False
                    break
                yield "wait"
            if not ok:
                break
            if st["S"] != j:
                raise ProtocolError(f"softmax reads S holding {st['S']} for tile {j}")
            s_free[sb].arrive()
            yield "read"
            slot = 0 if single_xmax else sb
            key = (slot, half)
            if not abort[0] and key in st["xmax"] and st["xmax"][key][1] is False:
                raise ProtocolError("a maximum slot is overwritten before the partner read it")
            st["xmax"][key] = (j, False)
            if abort[0] and not no_abort_check:
                ok = False
                break
            yield from nbar.sync()
            partner = st["xmax"].get((slot, 1 - half))
            # after an abort the partner's single arrival releases this sync
            # without a value: the results are void (the error word is set)
            if not abort[0] and (partner is None or partner[0] != j):
                raise ProtocolError(f"tile {j}: the partner's maximum slot holds {partner}")
            st["xmax"][(slot, 1 - half)] = (j, True)
            yield "max"
            if j >= 2 and not p_without_wait:
                while not o_done[j & 1].test((j >> 1) - 1):
                    if abort[0]:
                        ok = False
                        break
                    yield "wait"
                if not ok:
                    break
            if j >= 1 and rng.randrange(rescale_every) == 0:
                while not o_done[(j - 1) & 1].test((j - 1) >> 1):
                    if abort[0]:
                        ok = False
                        break
                    yield "wait"
                if not ok:
                    break
                if any(e[0] == "pv" for e in pipe):
                    raise ProtocolError(f"O rescaled at tile {j} while a P·V still accumulates into it")
            if pending_read("p", j & 1):
                raise ProtocolError(f"P({j}) written while P·V still reads buffer {j & 1}")
            prev = st["P"][j & 1]
            st["P"][j & 1] = ("half", j) if prev != ("half", j) else ("full", j)
            p_full[j & 1].arrive()
            yield "p"
        if not ok:
            nbar.arrive()   # releases the partner's current or next sync

    def land(i):
        kind, s, tile, bar = in_flight.pop(i)
        st[kind][s] = tile
        bar.complete_tx(1)

    def complete():
        e = pipe.pop(0)
        if e[0] == "qk":
            st["S"] = e[1]
        elif e[0] == "arrive":
            kind, a, b = e[2]
            if kind == "k":
                reading.remove(("k", a, b))
            else:
                reading.remove(("p", b & 1, b))
                reading.remove(("v", b % VST, b))
            for bar in e[1]:
                bar.arrive()

    live = {"producer": producer(), "qk": qk(), "pv": pv(), "sm0": softmax(0), "sm1": softmax(1)}
    steps = idle = 0
    while live:
        steps += 1
        if abort_at is not None and steps == abort_at:
            abort[0] = True
        choices = list(live) + ["copy lands"] * (len(in_flight) > 0) + ["MMA completes"] * (len(pipe) > 0)
        c = rng.choice(choices)
        progressed = True
        if c == "copy lands":
            land(rng.randrange(len(in_flight)))
        elif c == "MMA completes":
            complete()
        else:
            try:
                progressed = next(live[c]) not in ("wait", "named")
            except StopIteration:
                del live[c]
        idle = 0 if progressed else idle + 1
        if idle > 2000:
            if not abort[0]:
                raise ProtocolError("deadlock: every role waits")
            raise ProtocolError("after the abort a role still waits (a named barrier without its partner?)")
    while pipe:
        complete()
    if not abort[0] and n_tiles > 0 and st["S"] != n_tiles - 1:
        raise ProtocolError("the last QK^T did not complete")
    return steps


@pytest.mark.parametrize("seed", range(120))
def test_prefill_protocol_random(seed):
    rng = random.Random(300 + seed)
    run_model(rng.randint(1, 9), seed)


@pytest.mark.parametrize("seed", range(120))
def test_prefill_protocol_abort(seed):
    rng = random.Random(600 + seed)
    n = rng.randint(1, 9)
    run_model(n, seed, abort_at=rng.randrange(1, 40 * n + 10))


def _caught(runs=80, with_abort=False, **kw):
    hits = 0
    for seed in range(runs):
        rng = random.Random(900 + seed)
        n = rng.randint(3, 9)
        try:
            run_model(n, seed, abort_at=rng.randrange(1, 40 * n + 10) if with_abort else None, **kw)
        except ProtocolError:
            hits += 1
    return hits


def test_control_p_written_without_waiting():
    assert _caught(p_without_wait=True) > 0


def test_control_qk_without_score_read():
    assert _caught(qk_without_sfree=True) > 0


def test_control_third_key_load_before_q_copy():
    assert _caught(k2_without_q=True) > 0


def test_control_one_maximum_slot():
    assert _caught(single_xmax=True) > 0


@pytest.mark.parametrize("seed", range(60))
def test_named_barrier_safe_without_the_abort_check(seed):
    """The kernel checks the abort flag before each max-exchange sync, but
    the protocol does not depend on it: a warp that leaves arrives once,
    which its partner's next sync consumes, and the partner cannot reach a
    second sync, since QK^T of the tile after needs both warps' score reads.
    So even without the check no abort leaves a warp waiting."""
    rng = random.Random(1200 + seed)
    n = rng.randint(2, 9)
    run_model(n, seed, abort_at=rng.randrange(1, 40 * n + 10), no_abort_check=True)
