"""CPU model of the backward kernels' synchronisation (csrc/backward.cu).

Each CTA of bwd_dkdv_kernel / bwd_dq_kernel has a TMA producer thread, an MMA
warp (one thread issues), a wait-helper warp and 8 compute warps. Two kinds of
barrier connect them:

* mbarriers (phase parity; the producer's copies and the MMA commits complete
  them): the stage rings of the streamed tiles, S/dP ready, the end of the
  accumulation;
* hardware named barriers (bar.arrive / bar.sync with a thread count; a sync
  blocks until the generation's count is reached and cannot time out):
  - P1 / P: the compute warps arrive once per block (P^T written; dS written),
    the MMA warp syncs;
  - Go / Ack: the helper waits on the mbarrier of the next streamed tile, arrives
    on Go, and syncs on Ack, which the MMA warp arrives on after its Go sync.

The model runs the kernels' loops as agents under random, unfair interleavings,
with copies and MMAs completing asynchronously in order. It checks that:
* no warp arrives twice on a named barrier within one generation, so no
  arrival runs a generation ahead;
* no parity wait passes on the wrong phase;
* no stage is overwritten while an MMA still has to read it, and no MMA reads
  a stage before its copy has landed;
* every MMA finds in each compute warp's part of the TMEM score regions what it
  reads, and nothing is written to a part while its warp works on it:
  - dK/dV kernel: S^T, P^T, dP^T or dS^T of the right block;
  - dQ kernel: S in two alternating regions, dP in a third, dS over S;
* the schedule always finishes, with no deadlock (a hang on the GPU).

Each of these changes makes it fail:
* taking out the Ack handshake;
* letting the helper hand a tile over without waiting for its copy;
* having it hand over the wrong tile;
* issuing the next block's S^T, or dK and the next dP^T, before the compute
  phase that frees their region (dK/dV);
* issuing S(j + 2) before dQ(j), or dP(j + 1) before phase 2 of block j (dQ).
"""
import random

import pytest


class _MBar:
    def __init__(self, name, count=1):
        self.name, self.count = name, count
        self.phase, self.pending, self.tx = 0, count, 0
        self.done = set()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done.add(self.phase)
            self.phase += 1
            self.pending = self.count

    def arrive(self, tx=0):
        if self.pending == 0:
            raise AssertionError(f"{self.name}: re-armed while phase {self.phase} is pending")
        self.tx += tx
        self.pending -= 1
        self._maybe_complete()

    def complete_tx(self, tx):
        self.tx -= tx
        self._maybe_complete()

    def ready(self, want):
        r = (self.phase & 1) != (want & 1)
        if r and want not in self.done:
            raise AssertionError(f"{self.name}: parity wait for phase {want} passed at phase {self.phase}")
        return r


class _NamedBar:
    """bar.arrive / bar.sync with a thread count, counted in warps of 32. A warp that arrives twice
    in one generation is a protocol error (the kernels never rely on it)."""

    def __init__(self, name, threads):
        self.name, self.need = name, threads // 32
        self.gen, self.who = 0, set()

    def arrive(self, warp):
        if warp in self.who:
            raise AssertionError(f"{self.name}: warp {warp} arrived twice in one generation")
        self.who.add(warp)
        if len(self.who) == self.need:
            self.gen += 1
            self.who = set()

    def sync(self, warp):
        """Arrive, then the caller waits until generation `target` has completed."""
        target = self.gen + 1
        self.arrive(warp)
        return target


def _run(agents, copies, mma_queue, on_mma, rnd, max_steps):
    waiting = [None] * len(agents)
    speed = [rnd.choice([1.0, 0.5, 0.1, 0.02]) for _ in range(len(agents) + 2)]
    frozen = [0] * (len(agents) + 2)

    def runs(i):
        if frozen[i] > 0:
            frozen[i] -= 1
            return False
        if rnd.random() < 0.002:
            frozen[i] = rnd.randint(1, 300)
            return False
        return rnd.random() < speed[i]

    for _ in range(max_steps):
        if copies and runs(len(agents)):
            bar, tx = copies.pop(0)
            bar.complete_tx(tx)
        if mma_queue and runs(len(agents) + 1):
            on_mma(mma_queue.pop(0))
        live = False
        for a in rnd.sample(range(len(agents)), len(agents)):
            if agents[a] is None:
                continue
            live = True
            if not runs(a):
                continue
            w = waiting[a]
            if w is not None:
                kind, obj, val = w
                if kind == "m" and not obj.ready(val):
                    continue
                if kind == "n" and obj.gen < val:
                    continue
                waiting[a] = None
            try:
                waiting[a] = next(agents[a])
            except StopIteration:
                agents[a] = None
        if not live and not copies and not mma_queue:
            return
    stuck = [(w[1].name, w[2]) if w else None for w in waiting]
    raise AssertionError(f"deadlock: no progress; waits per agent: {stuck}")


def _simulate_dkdv(n_it, seed, ack=True, helper_skew=0, helper_wait=True, max_steps=400000, compute_warps=8,
                   early=None):
    rnd = random.Random(seed)
    kv_full = _MBar("kv_full")
    q_full, q_empty = [_MBar(f"q_full[{i}]") for i in range(3)], [_MBar(f"q_empty[{i}]") for i in range(3)]
    do_full, do_empty = [_MBar(f"do_full[{i}]") for i in range(2)], [_MBar(f"do_empty[{i}]") for i in range(2)]
    s_ready, dp_ready, acc_done = _MBar("s_ready"), _MBar("dp_ready"), _MBar("acc_done")
    issuer_w, helper_w = compute_warps + 1, compute_warps + 2   # warp compute_warps is the TMA producer
    p1, pb = _NamedBar("P1", 32 * (compute_warps + 1)), _NamedBar("P", 32 * (compute_warps + 1))
    go, ackb = _NamedBar("Go", 64), _NamedBar("Ack", 64)
    cbar = _NamedBar("compute", 32 * compute_warps)
    copies, mma = [], []
    reads = {}                      # (tile kind, block) -> MMAs still to read it
    q_stage, do_stage = [None] * 3, [None] * 2

    def producer():
        kv_full.arrive(tx=1)
        copies.append((kv_full, 1))
        for it in range(n_it):
            sq, sd = it % 3, it & 1
            if it >= 3:
                yield ("m", q_empty[sq], it // 3 - 1)
                if reads.get(("q", q_stage[sq]), 0):
                    raise AssertionError("Q stage overwritten while still to be read")
            q_stage[sq] = it
            reads[("q", it)] = 2            # S^T(i), dK(i)
            q_full[sq].arrive(tx=1)
            copies.append((q_full[sq], 1))
            yield None
            if it >= 2:
                yield ("m", do_empty[sd], (it >> 1) - 1)
                if reads.get(("do", do_stage[sd]), 0):
                    raise AssertionError("dO stage overwritten while still to be read")
            do_stage[sd] = it
            reads[("do", it)] = 2           # dP^T(i), dV(i)
            do_full[sd].arrive(tx=1)
            copies.append((do_full[sd], 1))
            yield None

    def helper():
        for it in range(1 + helper_skew, n_it + helper_skew):
            k = min(it, n_it - 1)
            if helper_wait:
                yield ("m", q_full[k % 3], k // 3)
                yield ("m", do_full[k & 1], k >> 1)
            go.arrive(helper_w)
            if ack:
                yield ("n", ackb, ackb.sync(helper_w))
            yield None

    # TMEM: region S holds S^T(i), then P^T(i); region dP holds dP^T(i), then dS^T(i). Each compute
    # warp rewrites its own part of a region (its 32 lanes, its half of the columns), so the model
    # keeps one entry per (region, warp). An MMA writes or reads every part; a phase checks its own
    # part at its start and at its end, so a write that lands while a phase works is caught.
    tmem = {(r, w): None for r in ("S", "dP") for w in range(compute_warps)}

    def issuer():
        if n_it == 0:
            mma.append(("commit", acc_done))
            return
        yield ("m", kv_full, 0)
        yield ("m", q_full[0], 0)
        yield ("m", do_full[0], 0)
        mma.append(("read", ("q", 0)))                  # S^T(0)
        mma.append(("twrite", "S", ("S", 0)))
        mma.append(("commit", s_ready))
        mma.append(("read", ("do", 0)))                 # dP^T(0)
        mma.append(("twrite", "dP", ("dP", 0)))
        mma.append(("commit", dp_ready))
        for it in range(n_it):
            if early != "s":
                yield ("n", p1, p1.sync(issuer_w))
            mma.append(("read", ("do", it)))            # dV(i)
            mma.append(("tread", "S", ("P", it)))
            mma.append(("commit", do_empty[it & 1]))
            if it + 1 < n_it:
                yield ("n", go, go.sync(issuer_w))
                if ack:
                    ackb.arrive(issuer_w)
                mma.append(("read", ("q", it + 1)))     # S^T(i + 1)
                mma.append(("twrite", "S", ("S", it + 1)))
                mma.append(("commit", s_ready))
            if early == "s":
                yield ("n", p1, p1.sync(issuer_w))
            if early != "dp":
                yield ("n", pb, pb.sync(issuer_w))
            mma.append(("read", ("q", it)))             # dK(i)
            mma.append(("tread", "dP", ("dS", it)))
            mma.append(("commit", q_empty[it % 3]))
            if early == "dp":
                yield ("n", pb, pb.sync(issuer_w))
            if it + 1 < n_it:
                mma.append(("read", ("do", it + 1)))    # dP^T(i + 1)
                mma.append(("twrite", "dP", ("dP", it + 1)))
                mma.append(("commit", dp_ready))
        mma.append(("commit", acc_done))

    def phase(w, region, want, result):
        if tmem[region, w] != want:
            raise AssertionError(f"warp {w} found {tmem[region, w]} in region {region}, wanted {want}")
        yield None
        if tmem[region, w] != want:
            raise AssertionError(f"region {region} overwritten while warp {w} worked on {want}")
        tmem[region, w] = result

    def compute(w):
        for it in range(n_it):
            yield ("n", cbar, cbar.sync(w))
            yield ("n", cbar, cbar.sync(w))
            yield ("m", s_ready, it)
            yield from phase(w, "S", ("S", it), ("P", it))
            p1.arrive(w)
            yield ("m", dp_ready, it)
            yield from phase(w, "dP", ("dP", it), ("dS", it))
            pb.arrive(w)
            yield None
        if n_it > 0:
            yield ("m", acc_done, 0)

    def on_mma(op):
        kind, arg = op[0], op[1]
        if kind == "commit":
            arg.arrive()
        elif kind == "twrite":
            for w in range(compute_warps):
                tmem[arg, w] = op[2]
        elif kind == "tread":
            for w in range(compute_warps):
                if tmem[arg, w] != op[2]:
                    raise AssertionError(f"an MMA read {tmem[arg, w]} from warp {w}'s part of region {arg}, "
                                         f"wanted {op[2]}")
        else:
            which, j = arg
            landed = (j // 3) in q_full[j % 3].done if which == "q" else (j >> 1) in do_full[j & 1].done
            if not landed:
                raise AssertionError(f"an MMA read {which}({j}) before its copy landed")
            reads[arg] -= 1

    agents = [producer(), helper(), issuer()] + [compute(w) for w in range(compute_warps)]
    _run(agents, copies, mma, on_mma, rnd, max_steps)


def _simulate_dq(n_j, seed, ack=True, helper_wait=True, max_steps=400000, early=None):
    rnd = random.Random(seed)
    qd_full = _MBar("qd_full")
    k_full, k_empty = [_MBar(f"k_full[{i}]") for i in range(3)], [_MBar(f"k_empty[{i}]") for i in range(3)]
    v_full, v_empty = [_MBar(f"v_full[{i}]") for i in range(2)], [_MBar(f"v_empty[{i}]") for i in range(2)]
    s_ready, dp_ready, acc_done = [_MBar("s_ready[0]"), _MBar("s_ready[1]")], _MBar("dp_ready"), _MBar("acc_done")
    pb, go, ackb = _NamedBar("P", 288), _NamedBar("Go", 64), _NamedBar("Ack", 64)
    copies, mma = [], []
    reads = {}
    k_stage, v_stage = [None] * 3, [None] * 2
    # TMEM, one entry per (region, compute warp): S(j) goes to region R(j mod 2) and is read by
    # phase 1; dP(j) goes to region dP; phase 2 reads dP(j) and writes dS(j) over S(j); dQ(j) reads
    # dS(j). A phase checks its part at its start and at its end.
    tmem = {(r, w): None for r in ("R0", "R1", "dP") for w in range(8)}

    def producer():
        if n_j == 0:
            return
        qd_full.arrive(tx=1)
        copies.append((qd_full, 1))
        for j in range(n_j):
            sk, sv = j % 3, j & 1
            if j >= 3:
                yield ("m", k_empty[sk], j // 3 - 1)
                if reads.get(("k", k_stage[sk]), 0):
                    raise AssertionError("K stage overwritten while still to be read")
            k_stage[sk] = j
            reads[("k", j)] = 2          # S(j), dQ(j)
            k_full[sk].arrive(tx=1)
            copies.append((k_full[sk], 1))
            yield None
            if j >= 2:
                yield ("m", v_empty[sv], (j >> 1) - 1)
                if reads.get(("v", v_stage[sv]), 0):
                    raise AssertionError("V stage overwritten while still to be read")
            v_stage[sv] = j
            reads[("v", j)] = 1          # dP(j)
            v_full[sv].arrive(tx=1)
            copies.append((v_full[sv], 1))
            yield None

    def issue_s(j):
        mma.append(("read", ("k", j)))
        mma.append(("twrite", f"R{j & 1}", ("S", j)))
        mma.append(("commit", s_ready[j & 1]))

    def issue_dp(j):
        mma.append(("read", ("v", j)))
        mma.append(("twrite", "dP", ("dP", j)))
        mma.append(("commit", dp_ready))
        mma.append(("commit", v_empty[j & 1]))

    def issue_dq(j):
        mma.append(("read", ("k", j)))
        mma.append(("tread", f"R{j & 1}", ("dS", j)))
        mma.append(("commit", k_empty[j % 3]))

    def helper():
        for j in range(n_j):
            if j + 1 < n_j:
                if helper_wait:
                    yield ("m", v_full[(j + 1) & 1], (j + 1) >> 1)
                go.arrive(10)
                if ack:
                    yield ("n", ackb, ackb.sync(10))
            if j + 2 < n_j:
                if helper_wait:
                    yield ("m", k_full[(j + 2) % 3], (j + 2) // 3)
                go.arrive(10)
                if ack:
                    yield ("n", ackb, ackb.sync(10))
            yield None

    def issuer():
        if n_j > 0:
            yield ("m", qd_full, 0)
            yield ("m", k_full[0], 0)
            issue_s(0)
            yield ("m", v_full[0], 0)
            issue_dp(0)
            if n_j > 1:
                yield ("m", k_full[1], 0)
                issue_s(1)
        for j in range(n_j):
            if early != "dp":
                yield ("n", pb, pb.sync(9))
            if j + 1 < n_j:
                yield ("n", go, go.sync(9))
                if ack:
                    ackb.arrive(9)
                issue_dp(j + 1)
            if early == "dp":
                yield ("n", pb, pb.sync(9))
            if early != "s":
                issue_dq(j)
            if j + 2 < n_j:
                yield ("n", go, go.sync(9))
                if ack:
                    ackb.arrive(9)
                issue_s(j + 2)
            if early == "s":
                issue_dq(j)
        mma.append(("commit", acc_done))

    def check(w, region, want, what):
        if tmem[region, w] != want:
            raise AssertionError(f"warp {w} {what}: found {tmem[region, w]} in region {region}, wanted {want}")

    def compute(w):
        for j in range(n_j):
            r = f"R{j & 1}"
            yield ("m", s_ready[j & 1], j >> 1)
            check(w, r, ("S", j), "phase 1 start")
            yield None
            check(w, r, ("S", j), "phase 1 end")
            yield ("m", dp_ready, j)
            check(w, "dP", ("dP", j), "phase 2 start")
            check(w, r, ("S", j), "phase 2 start")
            yield None
            check(w, "dP", ("dP", j), "phase 2 end")
            check(w, r, ("S", j), "phase 2 end")
            tmem[r, w] = ("dS", j)
            pb.arrive(w)
            yield None
        yield ("m", acc_done, 0)

    def on_mma(op):
        kind, arg = op[0], op[1]
        if kind == "commit":
            arg.arrive()
        elif kind == "twrite":
            for w in range(8):
                tmem[arg, w] = op[2]
        elif kind == "tread":
            for w in range(8):
                if tmem[arg, w] != op[2]:
                    raise AssertionError(f"an MMA read {tmem[arg, w]} from warp {w}'s part of region {arg}, "
                                         f"wanted {op[2]}")
        else:
            which, j = arg
            landed = (j // 3) in k_full[j % 3].done if which == "k" else (j >> 1) in v_full[j & 1].done
            if not landed:
                raise AssertionError(f"an MMA read {which.upper()}({j}) before its copy landed")
            reads[arg] -= 1

    agents = [producer(), helper(), issuer()] + [compute(w) for w in range(8)]
    _run(agents, copies, mma, on_mma, rnd, max_steps)


@pytest.mark.parametrize("n", [0, 1, 2, 3, 4, 5, 9, 33])
def test_dkdv_protocol_is_sound(n):
    for s in range(12):
        _simulate_dkdv(n, 100 * n + s)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 9, 33])
def test_dq_protocol_is_sound(n):
    for s in range(12):
        _simulate_dq(n, 200 * n + s)


def _fails(fn, **kw):
    try:
        fn(**kw)
    except AssertionError:
        return True
    return False


def test_model_catches_a_helper_that_does_not_wait():
    # handing the tile over without waiting for its copy lets an MMA read a stage still in flight
    assert any(_fails(_simulate_dkdv, n_it=9, seed=s, helper_wait=False) for s in range(30))
    assert any(_fails(_simulate_dq, n_j=9, seed=s, helper_wait=False) for s in range(30))


def test_model_catches_a_missing_ack():
    # without the acknowledgement the helper can arrive on Go twice before the MMA warp syncs
    assert any(_fails(_simulate_dkdv, n_it=9, seed=s, ack=False) for s in range(30)) or \
        any(_fails(_simulate_dq, n_j=9, seed=s, ack=False) for s in range(30))


@pytest.mark.parametrize("early", ["s", "dp"])
def test_model_catches_a_region_overwritten_early(early):
    # S^T(i + 1) issued before phase 1 of block i has turned S^T(i) into P^T(i), or dK(i) and
    # dP^T(i + 1) issued before phase 2 has turned dP^T(i) into dS^T(i): the region tracking fails
    assert any(_fails(_simulate_dkdv, n_it=6, seed=s, early=early) for s in range(30))


@pytest.mark.parametrize("early", ["s", "dp"])
def test_dq_model_catches_a_region_overwritten_early(early):
    # S(j + 2) issued before dQ(j) has read dS(j) from the same region, or dP(j + 1) issued before
    # phase 2 of block j has read dP(j): the region tracking fails
    assert any(_fails(_simulate_dq, n_j=7, seed=s, early=early) for s in range(30))

