"""CPU model of the CTA-pair prefill kernel's barrier protocol (csrc/prefill_pair.cu).

The pair kernel runs as clusters of two CTAs. CTA 0's MMA thread issues M = 256 MMAs
whose operands and accumulators are half in each CTA, so the protocol spans both:

* Each CTA has its own TMA producer. Both walk the same units and key blocks and load
  their own halves into their own rings of slots, but every copy completes on CTA 0's
  barriers: q_full (one phase per unit) and kv_ready[(G + j) % R] (one phase per key
  block) count two arrivals per phase, one per producer, each adding its CTA's bytes.
* A producer reuses a slot, or its Q buffer, only after the block that last read it is
  done; it learns that from its own CTA's iter_done ring, which the issuer's commits
  complete in both CTAs at once (tcgen05.commit with a CTA mask). The same holds for
  s_full1 and o_done[q].
* CTA 0's helper warp waits on q_full and kv_ready, hands each block's data to the
  issuer through a pair of hardware named barriers (Data, then an acknowledgement), and
  for every P.V product relays CTA 1's P: it waits on p_peer[q] (one arrival per block
  from CTA 1's slot-q softmax) and arrives on CTA 0's named barrier P_q, where CTA 0's
  own slot-q softmax warps also arrive and the issuer syncs.
* Per block the issuer sends PV_1(j-1), S_1(j), PV_0(j-1), S_0(j). Each softmax warp
  group (two per CTA) reads S_q(j) from its own CTA's TMEM and writes P_q(j) in place.

The model runs these agents (two producers, helper, issuer, four softmax groups) under
random, unfair interleavings, with the copies and the MMAs completing asynchronously,
and checks: no mbarrier is re-armed while its phase is pending; no parity wait passes on
a wrong phase; no participant arrives twice in one generation of a named barrier; no
MMA reads a K/V half or a Q tile before its copy landed or after its slot was reused; per
CTA, the softmax finds S_q(j) and O_q through block j - 1, P.V reads P_q(j), the
epilogue reads the final O_q; and the schedule never deadlocks. The kernel's
configurations (9 slots with R = 8 at d = 128, 21 slots with R = 16 at d = 64) must
pass; removing a rule (the helper's wait for CTA 1's P, CTA 1's arrival on kv_ready, or
a deep enough ring) must fail.
"""
import random

import pytest


class _Bar:
    """An mbarrier: `count` arrivals plus the transaction bytes they announce complete a phase."""

    def __init__(self, name, count=1):
        self.name = name
        self.count = count
        self.phase = 0
        self.pending = count
        self.tx = 0
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
        # the hardware allows the bytes of a copy to land before its arrival announces them
        self.tx -= tx
        self._maybe_complete()

    def parity_ready(self, want):
        ready = (self.phase & 1) != (want & 1)
        if ready and want not in self.done:
            raise AssertionError(f"{self.name}: parity wait for phase {want} passed at phase {self.phase}")
        return ready


class _NamedBar:
    """A hardware named barrier: each participant arrives once per generation."""

    def __init__(self, name, participants):
        self.name = name
        self.participants = set(participants)
        self.arrived = set()
        self.gen = 0

    def arrive(self, who):
        if who in self.arrived:
            raise AssertionError(f"{self.name}: {who} arrived twice in generation {self.gen}")
        self.arrived.add(who)
        if self.arrived == self.participants:
            self.arrived = set()
            self.gen += 1


def _simulate(k_slots, ring, units, seed, max_steps=3000000, helper_waits_peer=True, peer_arms_kv=True):
    """units: list of (nkv_0, nkv_1), the key blocks slots 0 and 1 walk (nkv_0 >= 1,
    nkv_1 in {0, .., nkv_0 + 1}). helper_waits_peer=False and peer_arms_kv=False switch off
    rules of the protocol to show that the model catches their absence."""
    rnd = random.Random(seed)
    kv_ready = [_Bar(f"kv_ready[{r}]", 2 if peer_arms_kv else 1) for r in range(ring)]
    q_full = _Bar("q_full", 2)
    p_peer = [_Bar("p_peer[0]"), _Bar("p_peer[1]")]
    iter_done = [[_Bar(f"cta{c}.iter_done[{r}]") for r in range(ring)] for c in range(2)]
    s_full1 = [_Bar(f"cta{c}.s_full1") for c in range(2)]
    o_done = [[_Bar(f"cta{c}.o_done[{q}]") for q in range(2)] for c in range(2)]
    nb_data = _NamedBar("Data", ["helper", "issuer"])
    nb_ack = _NamedBar("DataAck", ["helper", "issuer"])
    nb_p = [_NamedBar(f"P_{q}", ["softmax0", "helper", "issuer"]) for q in range(2)]

    copies = []                  # (cta, item or ('Q', unit), barrier, bytes) not yet landed
    landed = set()               # (cta, item) whose copy landed and whose slot still holds it
    mma_queue = []
    reads_left = {}              # (cta, item) -> MMAs still to read it
    q_reads_left = [[0], [0]]    # per CTA: S MMAs of the current unit's Q not yet completed
    slot_item = [[None] * k_slots for _ in range(2)]
    epilogue_done = [[-1, -1], [-1, -1]]
    last_active = [-1, -1]
    tmem = [{("S", 0): None, ("S", 1): None, ("O", 0): None, ("O", 1): None} for _ in range(2)]

    item_base = []
    ib = 0
    for n0, n1 in units:
        item_base.append(ib)
        n = max(n0, n1)
        for j in range(n):
            for c in range(2):
                reads_left[c, ib + 2 * j] = (j < n0) + (j < n1)
                reads_left[c, ib + 2 * j + 1] = (j < n0) + (j < n1)
        ib += 2 * n

    def producer(c):
        G, slot, filled = 0, 0, 0
        rel = [None] * k_slots
        done_upto = [-1]

        def wait_block(r):
            if r > done_upto[0]:
                yield ("mbar", iter_done[c][r % ring], r // ring)
                done_upto[0] = r

        for u, (n0, n1) in enumerate(units):
            n = max(n0, n1)
            if u > 0:
                yield from wait_block(G - 2)
                if q_reads_left[c][0]:
                    raise AssertionError(f"CTA {c}: Q of unit {u - 1} overwritten while S MMAs still read it")
                landed.discard((c, ("Q", u - 1)))
            q_reads_left[c][0] = n0 + n1
            nq = (n0 > 0) + (n1 > 0)
            q_full.arrive(tx=nq)
            copies.append((c, ("Q", u), q_full, nq))
            for i in range(2 * n):
                if filled == k_slots:
                    yield from wait_block(rel[slot])
                    prev = slot_item[c][slot]
                    if reads_left[c, prev]:
                        raise AssertionError(f"CTA {c}: slot of item {prev} overwritten while still to be read")
                    landed.discard((c, prev))
                else:
                    filled += 1
                it = (i + 1) >> 1
                rel[slot] = G + it
                rb = kv_ready[(G + it) % ring]
                if (i == 0 or (i & 1)) and (c == 0 or peer_arms_kv):
                    rb.arrive(tx=(1 if it >= 1 else 0) + (1 if it < n else 0))
                slot_item[c][slot] = item_base[u] + i
                copies.append((c, item_base[u] + i, rb, 1))
                slot = (slot + 1) % k_slots
                yield None
            G += n + 1

    def helper():
        G = 0
        pc = [0, 0]
        for u, (n0, n1) in enumerate(units):
            n = max(n0, n1)
            yield ("mbar", q_full, u)
            for j in range(n + 1):
                if j <= n and (j < n or j > 0):
                    yield ("mbar", kv_ready[(G + j) % ring], (G + j) // ring)
                    nb_data.arrive("helper")
                    yield ("nb", nb_ack, nb_ack.gen, "helper")
                for q, nk in ((1, n1), (0, n0)):
                    if j > 0 and j - 1 < nk:
                        if helper_waits_peer:
                            yield ("mbar", p_peer[q], pc[q])
                        pc[q] += 1
                        nb_p[q].arrive("helper")
                        yield None
            G += n + 1

    def issuer():
        G = 0
        for u, (n0, n1) in enumerate(units):
            n = max(n0, n1)
            ib = item_base[u]
            for j in range(n + 1):
                if j <= n and (j < n or j > 0):
                    yield ("nb", nb_data, nb_data.gen, "issuer")
                    nb_ack.arrive("issuer")
                for q, nk in ((1, n1), (0, n0)):
                    if j > 0 and j - 1 < nk:
                        yield ("nb", nb_p[q], nb_p[q].gen, "issuer")
                        if j == 1 and last_active[q] >= 0 and min(epilogue_done[0][q], epilogue_done[1][q]) < last_active[q]:
                            raise AssertionError(f"O_{q} overwritten before unit {last_active[q]}'s epilogue")
                        mma_queue.append(("read", ib + 2 * j - 1))
                        mma_queue.append(("tread", (("S", q), ("P", u, j - 1))))
                        mma_queue.append(("twrite", (("O", q), ("O", u, j - 1))))
                        if j == nk:
                            mma_queue.append(("commit", [o_done[0][q], o_done[1][q]]))
                    if j < nk:
                        mma_queue.append(("read", ib + 2 * j))
                        mma_queue.append(("qread", u))
                        mma_queue.append(("twrite", (("S", q), ("S", u, j))))
                        if q == 1:
                            mma_queue.append(("commit", [s_full1[0], s_full1[1]]))
                mma_queue.append(("commit", [iter_done[0][(G + j) % ring], iter_done[1][(G + j) % ring]]))
                yield None
            for q, nk in ((0, n0), (1, n1)):
                if nk > 0:
                    last_active[q] = u
            G += n + 1

    def softmax(c, q):
        G, sc, oc = 0, 0, 0
        for u, (n0, n1) in enumerate(units):
            n = max(n0, n1)
            nk = n1 if q else n0
            for j in range(nk):
                if q == 1:
                    yield ("mbar", s_full1[c], sc + j)
                else:
                    yield ("mbar", iter_done[c][(G + j) % ring], (G + j) // ring)
                for _ in range(2):
                    if tmem[c]["S", q] != ("S", u, j):
                        raise AssertionError(f"CTA {c} softmax {q} found {tmem[c]['S', q]}, wanted S({u}, {j})")
                    if j > 0 and tmem[c]["O", q] != ("O", u, j - 1):
                        raise AssertionError(f"CTA {c} softmax {q} found {tmem[c]['O', q]}, wanted O({u}, {j - 1})")
                    yield None
                tmem[c]["S", q] = ("P", u, j)
                if c == 0:
                    nb_p[q].arrive("softmax0")
                else:
                    p_peer[q].arrive()
                yield None
            if nk > 0:
                yield ("mbar", o_done[c][q], oc)
                for _ in range(2):
                    if tmem[c]["O", q] != ("O", u, nk - 1):
                        raise AssertionError(f"CTA {c} epilogue {q} found {tmem[c]['O', q]}, wanted O({u}, {nk - 1})")
                    yield None
                epilogue_done[c][q] = u
                oc += 1
            sc += nk
            G += n + 1

    agents = [producer(0), producer(1), helper(), issuer(), softmax(0, 0), softmax(0, 1), softmax(1, 0),
              softmax(1, 1)]
    names = ["producer0", "producer1", "helper", "issuer", "softmax(0,0)", "softmax(0,1)", "softmax(1,0)",
             "softmax(1,1)"]
    waiting = [None] * len(agents)
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

    def ready(w):
        if w[0] == "mbar":
            return w[1].parity_ready(w[2])
        # named barrier sync: arrive (once) then wait for the generation to complete
        _, nb, gen, who = w
        if nb.gen == gen and who not in nb.arrived:
            nb.arrive(who)
        return nb.gen > gen

    for _ in range(max_steps):
        if copies and runs(len(agents)):
            k = rnd.randrange(len(copies)) if rnd.random() < 0.3 else 0   # copies may land out of order
            c, item, bar, tx = copies.pop(k)
            landed.add((c, item))
            bar.complete_tx(tx)
        if mma_queue and runs(len(agents) + 1):
            kind, arg = mma_queue.pop(0)
            if kind == "commit":
                for b in arg:
                    b.arrive()
            elif kind == "read":
                for c in range(2):
                    if (c, arg) not in landed:
                        raise AssertionError(f"an MMA read CTA {c}'s item {arg} before its copy landed")
                    reads_left[c, arg] -= 1
            elif kind == "qread":
                for c in range(2):
                    if (c, ("Q", arg)) not in landed:
                        raise AssertionError(f"an MMA read CTA {c}'s Q of unit {arg} before it landed")
                    q_reads_left[c][0] -= 1
            elif kind == "twrite":
                for c in range(2):
                    tmem[c][arg[0]] = arg[1]
            elif kind == "tread":
                for c in range(2):
                    if tmem[c][arg[0]] != arg[1]:
                        raise AssertionError(f"an MMA read {tmem[c][arg[0]]} from CTA {c}'s {arg[0]}, wanted {arg[1]}")
        live = False
        for a in rnd.sample(range(len(agents)), len(agents)):
            if agents[a] is None:
                continue
            live = True
            if not runs(a):
                continue
            if waiting[a] is not None:
                if not ready(waiting[a]):
                    continue
                waiting[a] = None
            try:
                waiting[a] = next(agents[a])
            except StopIteration:
                agents[a] = None
        if not live and not copies and not mma_queue:
            return
    stuck = {names[i]: (w[1].name, w[2]) if w else None for i, w in enumerate(waiting)}
    raise AssertionError(f"deadlock: the schedule stopped making progress; waits: {stuck}")


def _unit_sequences(n, seed0, max_units=8):
    rnd = random.Random(seed0)
    for s in range(n):
        units = []
        for _ in range(rnd.randint(1, max_units)):
            nk0 = rnd.choice([1, 1, 2, 3, rnd.randint(1, 40)])
            # slot 1 walks as many blocks as slot 0, one more (g odd, causal) or none (end of T)
            nk1 = rnd.choice([nk0, nk0, nk0 + 1, 0])
            units.append((nk0, nk1))
        yield units, s


@pytest.mark.parametrize("k_slots,ring", [(9, 8), (21, 16)])
def test_kernel_configuration_is_sound(k_slots, ring):
    for units, s in _unit_sequences(40, 2000 + k_slots):
        _simulate(k_slots, ring, units, s)


@pytest.mark.parametrize("k_slots,ring", [(9, 8), (21, 16)])
def test_long_runs_of_one_block_units(k_slots, ring):
    for s in range(8):
        _simulate(k_slots, ring, [(1, 1)] * 30 + [(1, 0)] * 5, 91 + s)


def _fails(**kw):
    try:
        _simulate(**kw)
    except AssertionError:
        return True
    return False


def test_model_catches_a_relay_without_the_peers_p():
    seq = [(3, 3), (2, 3), (4, 4)]
    assert not any(_fails(k_slots=9, ring=8, units=seq, seed=s) for s in range(10))
    assert any(_fails(k_slots=9, ring=8, units=seq, seed=s, helper_waits_peer=False, max_steps=400000)
               for s in range(20))


def test_model_catches_kv_ready_without_the_peers_arrival():
    seq = [(6, 6), (3, 4), (5, 5)]
    assert any(_fails(k_slots=9, ring=8, units=seq, seed=s, peer_arms_kv=False, max_steps=400000)
               for s in range(20))


def test_model_catches_a_too_shallow_ring():
    failures = 0
    for units, s in _unit_sequences(20, 9, max_units=3):
        units = [(max(a, 20), max(b, 20) if b else 0) for a, b in units]
        if _fails(k_slots=21, ring=8, units=units, seed=s, max_steps=300000):
            failures += 1
    assert failures > 0
