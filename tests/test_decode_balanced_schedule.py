"""CPU model of the balanced decode schedule (num_splits = 0): the partition of the key stream
into CTA ranges (BalancedPartition), the pieces each CTA walks, the partial slots they write
and the slots the merge reads. It restates the rules of decode_balanced_kernel /
decode_balanced_merge_kernel and checks, over random and degenerate length mixes, that every
tile of every segment is processed exactly once, that each cut segment's pieces are exactly
the slots the merge reads, in key order, and that no slot is written twice or read unwritten.
"""
import random

import pytest

TILE = 64


class Partition:
    """Equal ranges over Geff = min(G, NT) CTAs."""

    def __init__(self, NT, G):
        self.NT, self.Geff = NT, min(NT, G)

    def range(self, c):
        if c < self.Geff:
            return c * self.NT // self.Geff, (c + 1) * self.NT // self.Geff
        return 0, 0

    def cta_of(self, t):
        return ((t + 1) * self.Geff + self.NT - 1) // self.NT - 1


def tiles_of(L, Lcap):
    L = max(0, min(L, Lcap))
    return (L + TILE - 1) // TILE


def schedule(lens, Lcap, Y, G):
    pre = [0]
    for L in lens:
        pre.append(pre[-1] + tiles_of(L, Lcap))
    NT = Y * pre[-1]
    part = Partition(NT, G)

    def piece(t, hi):
        lo_b, hi_b = 0, len(lens)
        while hi_b - lo_b > 1:
            mid = (lo_b + hi_b) // 2
            if Y * pre[mid] <= t:
                lo_b = mid
            else:
                hi_b = mid
        b = lo_b
        n = pre[b + 1] - pre[b]
        row0 = Y * pre[b]
        y = (t - row0) // n
        seg0 = row0 + y * n
        return dict(b=b, y=y, n=n, seg0=seg0, t0=t, t1=min(hi, seg0 + n))

    writes = {}  # slot -> (b, y, t0, t1)
    finished = set()
    covered = []
    nonempty = []
    for c in range(G):
        lo, hi = part.range(c)
        if lo == hi:
            continue
        nonempty.append(c)
        t = lo
        while t < hi:
            pc = piece(t, hi)
            assert pc["n"] > 0
            covered.extend(range(pc["t0"], pc["t1"]))
            to_end = pc["t1"] == pc["seg0"] + pc["n"]
            whole = pc["t0"] == pc["seg0"] and to_end
            if whole:
                assert (pc["b"], pc["y"]) not in finished
                finished.add((pc["b"], pc["y"]))
            else:
                slot = 2 * c + (1 if to_end else 0)
                assert slot not in writes, f"slot {slot} written twice"
                writes[slot] = (pc["b"], pc["y"], pc["t0"], pc["t1"])
            t = pc["t1"]
    assert covered == list(range(NT)), "every tile once, in order"
    # the non-empty ranges are those of CTAs 0 .. Geff - 1: none empty between two that share
    # a segment
    assert nonempty == list(range(part.Geff))
    cta_of = part.cta_of

    reads = set()
    for b, L in enumerate(lens):
        n = tiles_of(L, Lcap)
        for y in range(Y):
            if n == 0:
                assert (b, y) not in finished
                continue
            seg0 = Y * pre[b] + y * n
            c_first, c_last = cta_of(seg0), cta_of(seg0 + n - 1)
            if c_first == c_last:
                assert (b, y) in finished
                continue
            assert (b, y) not in finished
            np_ = c_last - c_first + 1
            assert all(part.range(c)[0] < part.range(c)[1] for c in range(c_first, c_last + 1))
            slots = [2 * (c_first + k) if k < np_ - 1 else 2 * c_last + 1 for k in range(np_)]
            t = seg0
            for s in slots:
                assert s in writes, f"slot {s} read but never written"
                wb, wy, t0, t1 = writes[s]
                assert (wb, wy) == (b, y) and t0 == t, "pieces read in key order"
                t = t1
                reads.add(s)
            assert t == seg0 + n, "the pieces cover the segment"
    assert reads == set(writes), "every written slot is read by the merge"


@pytest.mark.parametrize("G", [1, 2, 7, 304])
@pytest.mark.parametrize("Y", [1, 2, 8])
def test_degenerate_mixes(G, Y):
    for lens in ([0], [1], [0, 0, 5], [64], [65], [32768], [1] * 40, [0, 100, 0, 3000, 64, 63],
                 [2048] * 16, [1, 2, 3, 4]):
        schedule(lens, 32768, Y, G)


def test_random_mixes():
    rng = random.Random(7)
    for _ in range(300):
        B = rng.randint(1, 40)
        Lcap = rng.choice([64, 100, 1024, 4096, 32768])
        lens = [rng.choice([0, 1, rng.randint(0, Lcap), Lcap, Lcap + 5, -2]) for _ in range(B)]
        schedule(lens, Lcap, rng.choice([1, 2, 3, 8, 16]), rng.choice([1, 3, 152, 304, 1000]))


def test_bench_workload_shapes():
    rng = random.Random(1004)
    lens = [rng.randint(8192, 32768) for _ in range(16)]
    schedule(lens, 32768, 8, 304)
    schedule([rng.randint(1024, 2048) for _ in range(16)], 2048, 8, 304)
