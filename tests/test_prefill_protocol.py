"""CPU model of the prefill kernel's barrier protocol.

The prefill kernel (csrc/prefill.cu) coordinates one TMA producer thread, one
MMA thread and two softmax warpgroups with mbarriers:

* K/V ring: item i (K(j) = item 2j, V(j) = item 2j + 1) goes to slot i % kSlots;
  item i may reuse its slot once key block r = (i - kSlots + 1) >> 1 is done.
* kv_ready[j % R]: armed by the producer (one arrive + the bytes of K(j) and
  V(j-1)) with the first item of block j, waited by the MMA thread.
* iter_done[j % R]: committed after the last MMA of key block j; waited by the
  producer (slot reuse) and by softmax group 1 (S_1(j) ready).
* s_full0 (S_0(j) ready) and p_full[q] (P_q(j) written), one phase per block.
  In the kernel the P handoff (and the data handoff from a helper warp to the
  MMA thread) are hardware named barriers that alternate strictly with the
  issuer's syncs; the model keeps them as barriers with the same phase order.

Waits use phase parity, so a ring of R barriers is only sound if no agent can
get R phases ahead of another on the same barrier. This model runs the same
index formulas under random interleavings of the agents and of the
asynchronous completions (copies, MMAs), and checks that no barrier is re-armed
while its phase is pending, that no parity wait succeeds on the wrong phase,
that no slot is overwritten while an MMA still reads it, and that the schedule
never deadlocks. The kernel's configurations (5 slots for d = 128, 11 for
d = 64, R = 8) must pass; a too-shallow ring (R = 4 with 11 slots) must fail.
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


def _simulate(k_slots, ring, nkv0, nkv1, seed, max_steps=400000):
    rnd = random.Random(seed)
    n_iter = max(nkv0, nkv1)
    kv_ready = [_Bar(f"kv_ready[{r}]") for r in range(ring)]
    iter_done = [_Bar(f"iter_done[{r}]") for r in range(ring)]
    s_full0 = _Bar("s_full0")
    p_full = [_Bar("p_full[0]"), _Bar("p_full[1]")]
    copies = []        # (barrier, bytes) of issued copies not yet landed
    mma_queue = []     # issued MMA-side operations, completed in order
    readers = {}       # item -> number of issued MMAs still reading it
    slot_of = {}

    def producer():
        for i in range(2 * n_iter):
            if i >= k_slots:
                r = (i - k_slots + 1) >> 1
                yield (iter_done[r % ring], r // ring)
                if readers.get(i - k_slots, 0):
                    raise AssertionError(f"slot of item {i - k_slots} reused while still read")
            it = (i + 1) >> 1
            rb = kv_ready[it % ring]
            if i == 0 or (i & 1):
                rb.arrive(tx=(1 if it >= 1 else 0) + (1 if it < n_iter else 0))
            slot_of[i] = i % k_slots
            copies.append((rb, 1))
            yield None

    def mma():
        for j in range(n_iter + 1):
            yield (kv_ready[j % ring], j // ring)
            for q, nk in ((0, nkv0), (1, nkv1)):
                if j > 0 and j - 1 < nk:
                    yield (p_full[q], j - 1)
                    readers[2 * j - 1] = readers.get(2 * j - 1, 0) + 1
                    mma_queue.append(("read_done", 2 * j - 1))
                if j < n_iter and j < nk:
                    readers[2 * j] = readers.get(2 * j, 0) + 1
                    mma_queue.append(("read_done", 2 * j))
                    if q == 0:
                        mma_queue.append(("commit", s_full0))
            mma_queue.append(("commit", iter_done[j % ring]))
            yield None

    def softmax(q, nk):
        for j in range(nk):
            yield (s_full0, j) if q == 0 else (iter_done[j % ring], j // ring)
            p_full[q].arrive()
            yield None

    agents = [producer(), mma(), softmax(0, nkv0), softmax(1, nkv1)]
    waiting = [None] * len(agents)
    for _ in range(max_steps):
        if copies and rnd.random() < 0.5:
            bar, tx = copies.pop(0)
            bar.complete_tx(tx)
        if mma_queue and rnd.random() < 0.5:
            kind, arg = mma_queue.pop(0)
            if kind == "commit":
                arg.arrive()
            else:
                readers[arg] -= 1
        live = False
        for a in rnd.sample(range(len(agents)), len(agents)):
            if agents[a] is None:
                continue
            live = True
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
    raise AssertionError("deadlock: the schedule stopped making progress")


def _cases(n, seed0):
    rnd = random.Random(seed0)
    for s in range(n):
        nk0 = rnd.randint(1, 40)
        nk1 = rnd.choice([nk0, nk0, nk0 + 1, 0])  # heads paired, row tiles paired, last tile inactive
        yield nk0, nk1, s


@pytest.mark.parametrize("k_slots", [5, 11])
def test_kernel_configuration_is_sound(k_slots):
    for nk0, nk1, s in _cases(60, 1000 + k_slots):
        _simulate(k_slots, 8, nk0, nk1, s)


def test_model_catches_a_too_shallow_ring():
    failures = 0
    for nk0, nk1, s in _cases(40, 7):
        try:
            _simulate(11, 4, nk0, nk1, s, max_steps=60000)
        except AssertionError:
            failures += 1
    assert failures > 0
