"""CPU model of the lane-pair store swap that writes O in the prefill's epilogue and dQ/dK/dV in
the backward (csrc/prefill.cu, bwd_store_row in csrc/backward.cu), when the output is 32-byte
aligned.

Each thread owns one row (its TMEM lane) and holds, per 32-column chunk, 16 words: the chunk's
first 32 bytes in words 0-7 and its second 32 bytes in words 8-15. Lanes 2i and 2i + 1 (rows r
and r + 1) exchange with one xor-1 shuffle per word: the even lane sends its second half and
keeps its first, the odd lane sends its first half and keeps its second. Afterwards words 0-7
are this lane's 32 bytes of the pair's even row and words 8-15 its 32 bytes of the odd row;
each lane stores them at (row_e, chunk, 32 * parity) and (row_e + 1, chunk, 32 * parity), only
for rows that exist. The model runs that exchange over whole warps with labelled words and
checks that every word of every existing row is written exactly once with its own value and
that no store touches a row past the end, for both head sizes, any number of valid rows in the
warp, and (for the backward) both column halves.
"""
import pytest


def _swap_and_store(rows, d, n_valid, col0=0, n_chunks=None, wrong_half=False):
    """rows: the warp's 32 row indices (lane = row order); n_valid rows exist (a prefix, as rows
    past Tq or Tk at the end of a tile). Returns {(row, word): value} of the stores."""
    words_per_row = d // 2              # bf16 pairs
    n_chunks = n_chunks if n_chunks is not None else d // 32
    mem = {}
    for cc in range(n_chunks):
        chunk = col0 // 32 + cc
        # every lane's 16 words of this chunk, labelled with (row, word index in the row)
        pk = [[(rows[l], chunk * 16 + k) for k in range(16)] for l in range(32)]
        sent = [[pk[l][k] if (l & 1) != wrong_half else pk[l][8 + k] for k in range(8)] for l in range(32)]
        for l in range(32):
            for k in range(8):
                r = sent[l ^ 1][k]      # __shfl_xor_sync(..., 1)
                if l & 1:
                    pk[l][k] = r
                else:
                    pk[l][8 + k] = r
        for l in range(32):
            odd = l & 1
            le = l & ~1
            row_e = rows[le]
            st_e, st_o = le < n_valid, le + 1 < n_valid
            base = chunk * 16 + (8 if odd else 0)  # word offset within the row
            for idx, (stores, row, src) in enumerate(((st_e, row_e, pk[l][0:8]), (st_o, rows[le + 1], pk[l][8:16]))):
                if not stores:
                    continue
                for k in range(8):
                    key = (row, base + k)
                    assert key not in mem, f"word {key} written twice"
                    assert base + k < words_per_row
                    mem[key] = src[k]
    return mem


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_valid", [32, 31, 17, 2, 1, 0])
def test_prefill_epilogue_swap(d, n_valid):
    rows = list(range(96, 128))          # warp 3 of a tile: rows 96..127 of the tile
    mem = _swap_and_store(rows, d, n_valid)
    for l in range(32):
        for w in range(d // 2):
            key = (rows[l], w)
            if l < n_valid:
                assert mem.get(key) == key, f"row {rows[l]} word {w}: {mem.get(key)}"
            else:
                assert key not in mem, f"row {rows[l]} past the end written"
    assert len(mem) == n_valid * d // 2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("half", [0, 1])
@pytest.mark.parametrize("n_valid", [32, 19, 1])
def test_backward_row_half_swap(d, half, n_valid):
    # bwd_store_row: a thread writes half `half` of its row, i.e. d/64 chunks from column half*d/2
    rows = list(range(32, 64))
    mem = _swap_and_store(rows, d, n_valid, col0=half * d // 2, n_chunks=d // 64)
    lo, hi = half * d // 4, (half + 1) * d // 4    # words of this half
    for l in range(32):
        for w in range(d // 2):
            key = (rows[l], w)
            if l < n_valid and lo <= w < hi:
                assert mem.get(key) == key
            else:
                assert key not in mem


def test_model_catches_a_swap_of_the_wrong_halves():
    rows = list(range(32))
    mem = _swap_and_store(rows, 128, 32, wrong_half=True)
    assert any(mem.get((r, w)) != (r, w) for r in rows for w in range(64))
