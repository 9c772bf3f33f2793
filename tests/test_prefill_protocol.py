"""CPU model of the prefill kernel's barrier protocol.

The prefill kernel (csrc/prefill.cu) is persistent: each CTA walks a sequence of
work units (two 128-row query tiles with nkv_0, nkv_1 key blocks; n = max of the
two, key blocks 0..n) and coordinates one TMA producer thread, one MMA thread
and two softmax warpgroups with mbarriers whose phases run on across units:

* G = index of a unit's key block 0 in the CTA's sequence of key blocks (grows
  by n + 1 per unit).
* q_full: one phase per unit (the unit's Q tiles landed). Before loading a
  unit's Q the producer waits for block G - 2 (the previous unit's last S MMAs).
* K/V ring: the unit's items 2j = K(j), 2j + 1 = V(j) go to consecutive slots;
  an item may overwrite its slot once the block that last read the slot's
  previous item is done (K(j) is read in block j, V(j) in block j + 1). Blocks
  complete in order, so the producer skips waits for blocks at or below the
  last one it saw complete (a stale wait could come after its barrier wrapped
  twice).
* kv_ready[(G + j) % R]: armed by the first item of block j (one arrive + the
  bytes of K(j) and V(j-1)), waited by the MMA side.
* Per block the MMA thread issues tile 1's GEMMs, then tile 0's.
  iter_done[(G + j) % R]: committed after the last MMA of block j; waited by the
  producer (slot and Q reuse) and by softmax group 0 (S_0(j) ready). Tile 0 is
  active in every unit with nkv_0 >= n - 1, so its waits never skip more than a
  few blocks of the ring.
* s_full1: one phase per S_1 block (tile 1 may be inactive in a unit, and then
  contributes no phase); o_done[q]: one phase per unit in which tile q is
  active; p_full[q]: one phase per P_q handoff. In the kernel the P handoff
  (and the data handoff from a helper warp to the MMA thread) are hardware
  named barriers that alternate strictly with the issuer's syncs; the model
  keeps them as barriers with the same phase order.

Waits use phase parity, so a ring of R barriers is only sound if no agent can
get R phases ahead of another on the same barrier. This model runs the same
index formulas under random interleavings of the agents and of the
asynchronous completions (copies, MMAs), and checks that no barrier is re-armed
while its phase is pending, that no parity wait succeeds on the wrong phase,
that no K/V slot or Q buffer is overwritten while an MMA still has to read it,
that a unit's first P.V product (which overwrites O_q) comes after the previous
unit's epilogue read O_q, and that the schedule never deadlocks. It also tracks
what each tile's TMEM regions hold:
* the softmax of block j must find S_q(j) in S_q, and O_q through block j - 1;
* P.V(j) must read P_q(j) there;
* the epilogue must read the final O_q;
* nothing may change while a phase works on it. The kernel's
configurations (5 slots for d = 128, 11 for d = 64, R = 8) must pass; a
too-shallow ring (R = 4 with 11 slots) must fail.
"""
import random

import pytest


class _Bar:
    def __init__(self, name):
        self.name = name
        self.phase = 0          # index of the current, not yet completed phase
        self.pending = 1        # arrivals still expected in this phase
        self.tx = 0             # transaction bytes still expected in this phase
        self.done = set()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done.add(self.phase)
            self.phase += 1
            self.pending = 1

    def arrive(self, tx=0):
        if self.pending == 0:
            raise AssertionError(f"{self.name}: re-armed while phase {self.phase} is pending")
        self.tx += tx
        self.pending -= 1
        self._maybe_complete()

    def complete_tx(self, tx):
        self.tx -= tx
        if self.tx < 0:
            raise AssertionError(f"{self.name}: transaction count underflow")
        self._maybe_complete()

    def parity_ready(self, want):
        ready = (self.phase & 1) != (want & 1)      # what the hardware parity test returns
        if ready and want not in self.done:
            raise AssertionError(f"{self.name}: parity wait for phase {want} passed at phase {self.phase}")
        return ready


def _simulate(k_slots, ring, units, seed, max_steps=2000000, skip_done_waits=True, counted_tile=1,
              s_before_pv=False):
    """units: list of (nkv_0, nkv_1) with max >= 1 and nkv_0 >= 1. `counted_tile` is the tile
    whose S-ready signal has its own barrier (one phase per S block of that tile); the other
    tile waits on iter_done. skip_done_waits=False, counted_tile=0 or s_before_pv=True (S_q(j)
    issued ahead of PV_q(j - 1)) switch off rules of the kernel's protocol, to show that the
    model catches their absence."""
    rnd = random.Random(seed)
    kv_ready = [_Bar(f"kv_ready[{r}]") for r in range(ring)]
    iter_done = [_Bar(f"iter_done[{r}]") for r in range(ring)]
    q_full = _Bar("q_full")
    s_full = _Bar(f"s_full{counted_tile}")
    o_done = [_Bar("o_done[0]"), _Bar("o_done[1]")]
    p_full = [_Bar("p_full[0]"), _Bar("p_full[1]")]
    copies = []          # (barrier, bytes) of issued copies not yet landed
    mma_queue = []       # issued MMA-side operations, completed in order
    reads_left = {}      # global item -> MMAs that still have to read it (issued or not)
    q_reads_left = [0]   # S MMAs of the current unit's Q not yet completed (issued or not)
    slot_item = [None] * k_slots
    epilogue_done = [-1, -1]   # last unit whose O_q the softmax warps have read
    last_active = [-1, -1]     # last unit in which tile q was active (issuer's view)
    # TMEM contents per tile: region S_q holds S_q(j) of unit u, which the softmax turns into
    # P_q(j) in place and PV_q(j) reads; O_q holds the product through block j (PV_q(j) done).
    tmem = {("S", 0): None, ("S", 1): None, ("O", 0): None, ("O", 1): None}

    # reads each item will get: K(j) by S_q(j) for tiles with j < nkv_q, V(j) by PV_q(j) likewise
    item_base = []
    ib = 0
    for n0, n1 in units:
        item_base.append(ib)
        n = max(n0, n1)
        for j in range(n):
            reads_left[ib + 2 * j] = (j < n0) + (j < n1)
            reads_left[ib + 2 * j + 1] = (j < n0) + (j < n1)
        ib += 2 * n

    def producer():
        G, slot, filled = 0, 0, 0
        rel = [None] * k_slots
        done_upto = [-1]   # blocks complete in order: no wait at or below the last one seen

        def wait_block(r):
            if r > done_upto[0] or not skip_done_waits:
                yield (iter_done[r % ring], r // ring)
                done_upto[0] = r

        for u, (n0, n1) in enumerate(units):
            n = max(n0, n1)
            if u > 0:
                yield from wait_block(G - 2)
                if q_reads_left[0]:
                    raise AssertionError(f"Q of unit {u - 1} overwritten while S MMAs still read it")
            q_reads_left[0] = (n0 + n1)
            nq = (n0 > 0) + (n1 > 0)
            q_full.arrive(tx=nq)
            copies.append((q_full, nq))
            for i in range(2 * n):
                if filled == k_slots:
                    yield from wait_block(rel[slot])
                    prev = slot_item[slot]
                    if reads_left[prev]:
                        raise AssertionError(f"slot of item {prev} overwritten while still to be read")
                else:
                    filled += 1
                it = (i + 1) >> 1
                rel[slot] = G + it
                rb = kv_ready[(G + it) % ring]
                if i == 0 or (i & 1):
                    rb.arrive(tx=(1 if it >= 1 else 0) + (1 if it < n else 0))
                slot_item[slot] = item_base[u] + i
                copies.append((rb, 1))
                slot = (slot + 1) % k_slots
                yield None
            G += n + 1

    def mma():
        G = 0
        pcount = [0, 0]
        for u, (n0, n1) in enumerate(units):
            n = max(n0, n1)
            ib = item_base[u]
            yield (q_full, u)
            order = ((1, n1), (0, n0)) if counted_tile == 1 else ((0, n0), (1, n1))
            for j in range(n + 1):
                yield (kv_ready[(G + j) % ring], (G + j) // ring)
                for q, nk in order:
                    def issue_s():
                        mma_queue.append(("read", ib + 2 * j))
                        mma_queue.append(("qread", None))
                        mma_queue.append(("twrite", (("S", q), ("S", u, j))))
                        if q == counted_tile:
                            mma_queue.append(("commit", s_full))
                    if s_before_pv and j < nk:
                        issue_s()
                    if j > 0 and j - 1 < nk:
                        yield (p_full[q], pcount[q])
                        pcount[q] += 1
                        if j == 1 and last_active[q] >= 0 and epilogue_done[q] < last_active[q]:
                            raise AssertionError(f"O_{q} overwritten before unit {last_active[q]}'s epilogue")
                        mma_queue.append(("read", ib + 2 * j - 1))
                        mma_queue.append(("tread", (("S", q), ("P", u, j - 1))))
                        mma_queue.append(("twrite", (("O", q), ("O", u, j - 1))))
                        if j == nk:
                            mma_queue.append(("commit", o_done[q]))
                    if not s_before_pv and j < nk:
                        issue_s()
                mma_queue.append(("commit", iter_done[(G + j) % ring]))
                yield None
            for q, nk in ((0, n0), (1, n1)):
                if nk > 0:
                    last_active[q] = u
            G += n + 1

    def softmax(q):
        G, sc, oc = 0, 0, 0
        for u, (n0, n1) in enumerate(units):
            n = max(n0, n1)
            nk = n1 if q else n0
            for j in range(nk):
                yield (s_full, sc + j) if q == counted_tile else (iter_done[(G + j) % ring], (G + j) // ring)
                # softmax of block j: reads S_q(j), writes P_q(j) over it, may rescale O_q, whose
                # product must then run through block j - 1 and stay untouched meanwhile
                for _ in range(2):
                    if tmem["S", q] != ("S", u, j):
                        raise AssertionError(f"softmax {q} found {tmem['S', q]} in S_{q}, wanted S({u}, {j})")
                    if j > 0 and tmem["O", q] != ("O", u, j - 1):
                        raise AssertionError(f"softmax {q} found {tmem['O', q]} in O_{q}, wanted O({u}, {j - 1})")
                    yield None
                tmem["S", q] = ("P", u, j)
                p_full[q].arrive()
                yield None
            if nk > 0:
                yield (o_done[q], oc)
                for _ in range(2):   # the epilogue reads the final O_q
                    if tmem["O", q] != ("O", u, nk - 1):
                        raise AssertionError(f"epilogue {q} found {tmem['O', q]} in O_{q}, wanted O({u}, {nk - 1})")
                    yield None
                epilogue_done[q] = u
                oc += 1
            sc += nk
            G += n + 1

    agents = [producer(), mma(), softmax(0), softmax(1)]
    waiting = [None] * len(agents)
    # Unfair schedules: every agent (and each completion stream) gets its own speed, and any
    # of them may freeze for a long stretch, so one side can fall far behind the others.
    speed = [rnd.choice([1.0, 0.5, 0.1, 0.02]) for _ in range(len(agents) + 2)]
    frozen = [0] * (len(agents) + 2)

    def runs(i):
        if frozen[i] > 0:
            frozen[i] -= 1
            return False
        if rnd.random() < 0.002:
            frozen[i] = rnd.randint(1, 400)
            return False
        return rnd.random() < speed[i]

    for _ in range(max_steps):
        if copies and runs(len(agents)):
            bar, tx = copies.pop(0)
            bar.complete_tx(tx)
        if mma_queue and runs(len(agents) + 1):
            kind, arg = mma_queue.pop(0)
            if kind == "commit":
                arg.arrive()
            elif kind == "read":
                reads_left[arg] -= 1
            elif kind == "twrite":
                tmem[arg[0]] = arg[1]
            elif kind == "tread":
                if tmem[arg[0]] != arg[1]:
                    raise AssertionError(f"an MMA read {tmem[arg[0]]} from {arg[0]}, wanted {arg[1]}")
            else:
                q_reads_left[0] -= 1
        live = False
        for a in rnd.sample(range(len(agents)), len(agents)):
            if agents[a] is None:
                continue
            live = True
            if not runs(a):
                continue
            if waiting[a] is not None:
                bar, phase = waiting[a]
                if not bar.parity_ready(phase):
                    continue
                waiting[a] = None
            try:
                waiting[a] = next(agents[a])
            except StopIteration:
                agents[a] = None
        if not live and not copies and not mma_queue:
            return
    stuck = [(w[0].name, w[1], w[0].phase) if w else None for w in waiting]
    raise AssertionError(f"deadlock: the schedule stopped making progress; waits (barrier, phase wanted, "
                         f"phase now) of producer, MMA, softmax 0, softmax 1: {stuck}")


def _unit_sequences(n, seed0, max_units=8):
    rnd = random.Random(seed0)
    for s in range(n):
        units = []
        for _ in range(rnd.randint(1, max_units)):
            nk0 = rnd.choice([1, 1, 2, 3, rnd.randint(1, 40)])   # short units stress the unit boundaries
            # the kernel's pairs: heads at the same rows, consecutive row tiles (causal), last tile inactive
            nk1 = rnd.choice([nk0, nk0, nk0 + 1, 0])
            units.append((nk0, nk1))
        yield units, s


@pytest.mark.parametrize("k_slots", [5, 11])
def test_kernel_configuration_is_sound(k_slots):
    for units, s in _unit_sequences(50, 1000 + k_slots):
        _simulate(k_slots, 8, units, s)


@pytest.mark.parametrize("k_slots", [5, 11])
def test_long_runs_of_one_block_units(k_slots):
    # every unit a single key block: the per-unit Q wait is all that keeps the producer close
    for s in range(10):
        _simulate(k_slots, 8, [(1, 1)] * 30 + [(1, 0)] * 5, 77 + s)


def test_model_catches_a_too_shallow_ring():
    failures = 0
    for units, s in _unit_sequences(30, 7, max_units=3):
        units = [(max(a, 20), max(b, 20) if b else 0) for a, b in units]
        try:
            _simulate(11, 4, units, s, max_steps=200000)
        except AssertionError:
            failures += 1
    assert failures > 0


def _fails(**kw):
    try:
        _simulate(**kw)
    except AssertionError:
        return True
    return False


def test_model_catches_a_missing_protocol_rule():
    # a long unit with tile 1 inactive: if tile 1 waited on the per-block ring, its next wait
    # would be many blocks away from its last one and could pass on a wrong phase or hang
    seq = [(27, 0), (1, 2), (1, 1), (2, 3)] * 3
    assert not any(_fails(k_slots=5, ring=8, units=seq, seed=s) for s in range(20))
    assert any(_fails(k_slots=5, ring=8, units=seq, seed=s, counted_tile=0, max_steps=300000) for s in range(20))
    # runs of one-block units, then a long one: a slot's release block was passed long ago
    seq = [(1, 0), (1, 0), (1, 1), (2, 2), (1, 1), (24, 25)]
    assert not _fails(k_slots=11, ring=8, units=seq, seed=7)
    assert _fails(k_slots=11, ring=8, units=seq, seed=7, skip_done_waits=False, max_steps=200000)


def test_model_catches_s_issued_before_the_previous_pv():
    # S_q(j) issued ahead of PV_q(j - 1) overwrites P_q(j - 1) before the P.V product reads it
    seq = [(3, 3), (2, 1), (4, 4)]
    assert not _fails(k_slots=5, ring=8, units=seq, seed=3)
    assert any(_fails(k_slots=5, ring=8, units=seq, seed=s, s_before_pv=True, max_steps=300000) for s in range(20))

