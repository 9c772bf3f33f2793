"""Float64 oracle for exact attention (prefill), flash-decoding and their parts.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definitions followed (all in float64, bf16 inputs decoded exactly):

* Scores  s_ij = scale * sum_k q_ik k_jk  over the visible keys V(i):
  all j < Tk, or, when causal, j <= i. The causal rule is the one of the
  reference implementation in "Module 07: Fused operators and FlashAttention",
  section "FlashAttention-naive in numpy" (entries above the diagonal are set
  to -inf), and of the lesson "FlashAttention: attention without the n x n
  matrix", section "Practice" (position i sees positions j <= i). For Tq != Tk
  the same rule is kept, aligned at the top-left corner.
* Three-pass safe softmax: m_i = max_j s_ij, l_i = sum_j exp(s_ij - m_i),
  O_i = sum_j exp(s_ij - m_i) v_j / l_i ("FlashAttention: attention without
  the n x n matrix", section "Online softmax: normalisation in one pass",
  first paragraph: find the max, sum the exponentials, divide).
* LSE_i = m_i + ln l_i = ln sum_j exp(s_ij) (same lesson, section "Backward
  pass: recomputing is cheaper than storing").
* GQA: g = Hq / Hkv query heads share one K/V head; query head h reads K/V
  head floor(h / g) ("Attention from the kernel's side", section "Prefill and
  decoding are different problems", grouped-query attention).
* Backward: the gradients by recomputation from the saved LSE ("FlashAttention:
  attention without the n x n matrix", section "Backward pass: recomputing is
  cheaper than storing"); see ``attention_backward``.
* Decode: one query per sequence attends to keys 0 .. L_b - 1 of its cache;
  flash-decoding splits the key range, each split keeps a partial (m, l, o),
  and the partials are merged with the same rescaling rule (same section,
  flash-decoding).
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np

NEG_INF = -math.inf


# ---------------------------------------------------------------------------
# Score-level cores (d = 1 worked examples feed these directly)
# ---------------------------------------------------------------------------

def scores_softmax_weighted(scores: Sequence[float], values) -> tuple[float | np.ndarray, float]:
    """Three-pass softmax-weighted sum of ``values`` for one row of scores.

    Returns (o, lse): o = sum_j softmax(s)_j v_j and lse = ln sum_j exp(s_j).
    Masked entries are given as -inf and contribute nothing.
    Source: "FlashAttention: attention without the n x n matrix", section
    "Online softmax: normalisation in one pass" (the three-pass safe softmax
    it starts from) and "Module 07", section "Online softmax: derivation",
    "What exactly has to be computed" (the O_i formula).
    """
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    m = s.max()                                  # pass 1: row maximum
    e = np.exp(s - m)                            # pass 2: exponentials and their sum
    l = e.sum()
    o = np.tensordot(e, v, axes=(0, 0)) / l      # pass 3: normalise (weighted sum)
    return o, float(m + math.log(l))


def online_softmax_blocks(scores: Sequence[float], values, block: int):
    """The block online-softmax recurrence on one row, returning every state.

    State after t blocks: (m_t, l_t, O_t) with l_t = sum exp(s - m_t) and
    O_t = sum exp(s - m_t) v over the blocks seen. Base m = -inf, l = 0, O = 0.
    Step for block B: m_new = max(m, max_B s); corr = exp(m - m_new);
    l <- l * corr + sum_B exp(s - m_new); O <- O * corr + sum_B exp(s - m_new) v.
    Final O / l.
    Source: "Module 07: Fused operators and FlashAttention", section
    "Online softmax: derivation" (Invariant, Step, Finalisation).

    Returns (o_final, states) where states[t] = dict(m, corr, l, O) after
    block t + 1.
    """
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    m = NEG_INF
    l = 0.0
    O = np.zeros(v.shape[1:], dtype=np.float64)
    states = []
    for j0 in range(0, len(s), block):
        sb = s[j0:j0 + block]
        vb = v[j0:j0 + block]
        m_new = max(m, float(sb.max()))
        corr = 0.0 if m == NEG_INF else math.exp(m - m_new)
        p = np.exp(sb - m_new)
        l = l * corr + float(p.sum())
        O = O * corr + np.tensordot(p, vb, axes=(0, 0))
        m = m_new
        states.append(dict(m=m, corr=corr, l=l, O=np.array(O)))
    return O / l, states


def online_normalizer(xs: Iterable[float]) -> tuple[float, float]:
    """One pass over a stream: m' = max(m, x), l' = l * e^(m - m') + e^(x - m').

    Source: "FlashAttention: attention without the n x n matrix", section
    "Online softmax: normalisation in one pass" (Milakov-Gimelshein update).
    """
    m, l = NEG_INF, 0.0
    for x in xs:
        m_new = max(m, x)
        l = (0.0 if m == NEG_INF else l * math.exp(m - m_new)) + math.exp(x - m_new)
        m = m_new
    return m, l


def online_weighted_stream(xs: Iterable[float], vs: Iterable[float]):
    """Online softmax with the value accumulator a' = a e^(m - m') + e^(x - m') v.

    Returns (m, l, a, o = a / l).
    Source: "FlashAttention: attention without the n x n matrix", section
    "Online softmax: normalisation in one pass" ("the main step for
    attention"); "Chapter 5", section 5.3.3, example 5-6 (the r = exp(m - m')
    rescaling of l and u).
    """
    m, l, a = NEG_INF, 0.0, 0.0
    for x, v in zip(xs, vs):
        m_new = max(m, x)
        r = 0.0 if m == NEG_INF else math.exp(m - m_new)
        w = math.exp(x - m_new)
        l = l * r + w
        a = a * r + w * v
        m = m_new
    return m, l, a, a / l


# ---------------------------------------------------------------------------
# Prefill attention
# ---------------------------------------------------------------------------

def _visible_mask(rows: np.ndarray, Tk: int, causal: bool) -> np.ndarray:
    cols = np.arange(Tk)[None, :]
    if causal:
        return cols <= rows[:, None]
    return np.ones((len(rows), Tk), dtype=bool)


def _rows_three_pass(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray,
                     rows: np.ndarray, causal: bool, scale: float):
    """Exact attention for the given query rows of one (batch, head)."""
    s = (q_rows @ k.T) * scale                           # [r, Tk] scores
    s = np.where(_visible_mask(rows, k.shape[0], causal), s, NEG_INF)
    m = s.max(axis=1, keepdims=True)                     # pass 1
    e = np.exp(s - m)                                    # pass 2
    l = e.sum(axis=1, keepdims=True)
    o = (e @ v) / l                                      # pass 3
    lse = (m + np.log(l))[:, 0]
    return o, lse


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
              scale: float, row_chunk: int = 1024):
    """Exact attention O = softmax(scale * Q K^T + mask) V and its LSE.

    q: [B, Hq, Tq, d], k and v: [B, Hkv, Tk, d] float64. Returns
    O [B, Hq, Tq, d] and LSE [B, Hq, Tq] (natural log of the scaled scores).
    Query rows are processed in chunks only to bound memory; every row is the
    plain three-pass softmax of its full score row.
    """
    B, Hq, Tq, d = q.shape
    Hkv = k.shape[1]
    assert Hq % Hkv == 0
    g = Hq // Hkv
    O = np.empty((B, Hq, Tq, v.shape[-1]), dtype=np.float64)
    L = np.empty((B, Hq, Tq), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            kvh = h // g
            for r0 in range(0, Tq, row_chunk):
                rows = np.arange(r0, min(r0 + row_chunk, Tq))
                o, lse = _rows_three_pass(q[b, h, rows], k[b, kvh], v[b, kvh], rows, causal, scale)
                O[b, h, rows] = o
                L[b, h, rows] = lse
    return O, L


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, b: int, h: int,
                   rows, causal: bool, scale: float):
    """Exact attention for selected query rows of one (batch, head) only.

    Used for sampled parity checks at sizes where the full oracle is too slow.
    """
    rows = np.asarray(rows, dtype=np.int64)
    g = q.shape[1] // k.shape[1]
    return _rows_three_pass(q[b, h, rows], k[b, h // g], v[b, h // g], rows, causal, scale)


def attention_online(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                     scale: float, Br: int, Bc: int):
    """Block-tiled attention with the online-softmax recurrence (FA-2 loop order).

    Outer loop over query blocks of Br rows, inner loop over key blocks of Bc
    keys; key blocks entirely above the diagonal are skipped when causal; the
    running (m, l, acc) are rescaled by exp(m_old - m_new); one division per
    row at the end. Used only to cross-check the three-pass definition.
    Source: "Module 07: Fused operators and FlashAttention", section
    "FlashAttention-2" (loop order, single division, causal skip) and
    "FlashAttention: attention without the n x n matrix", section "Forward
    pass of FlashAttention" (the block update of m, l and A).
    """
    B, Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    g = Hq // Hkv
    O = np.empty((B, Hq, Tq, v.shape[-1]))
    L = np.empty((B, Hq, Tq))
    for b in range(B):
        for h in range(Hq):
            K, V = k[b, h // g], v[b, h // g]
            for i0 in range(0, Tq, Br):
                Qi = q[b, h, i0:i0 + Br]
                nb = Qi.shape[0]
                rows = np.arange(i0, i0 + nb)
                m = np.full(nb, NEG_INF)
                l = np.zeros(nb)
                acc = np.zeros((nb, V.shape[1]))
                for j0 in range(0, Tk, Bc):
                    if causal and j0 > i0 + nb - 1:
                        break                                   # block fully above the diagonal
                    S = (Qi @ K[j0:j0 + Bc].T) * scale
                    cols = np.arange(j0, j0 + S.shape[1])
                    if causal:
                        S = np.where(cols[None, :] > rows[:, None], NEG_INF, S)  # mask before max
                    m_new = np.maximum(m, S.max(axis=1))
                    # A row whose every score so far is masked keeps m = -inf;
                    # exp(-inf - -inf) is avoided by using 0 as the base there.
                    base = np.where(np.isfinite(m_new), m_new, 0.0)
                    corr = np.exp(m - base)
                    P = np.exp(S - base[:, None])
                    l = l * corr + P.sum(axis=1)
                    acc = acc * corr[:, None] + P @ V[j0:j0 + Bc]
                    m = m_new
                O[b, h, i0:i0 + nb] = acc / l[:, None]
                L[b, h, i0:i0 + nb] = m + np.log(l)
    return O, L


def count_blocks(T: int, block_q: int, block_k: int, causal: bool) -> int:
    """Number of (query block, key block) pairs the tiled forward pass computes.

    Without a mask every pair; with the causal mask only pairs whose key block
    starts at or before the last row of the query block.
    Source: "FlashAttention: attention without the n x n matrix", section
    "Practice" (count_blocks contract) and section "Forward pass of
    FlashAttention" (causal mask paragraph).
    """
    n = 0
    for qs in range(0, T, block_q):
        qe = min(qs + block_q, T)
        for ks in range(0, T, block_k):
            if not causal or ks <= qe - 1:
                n += 1
    return n


# ---------------------------------------------------------------------------
# Decode (one query per sequence) and the split-KV merge
# ---------------------------------------------------------------------------

def decode(q: np.ndarray, kcache: np.ndarray, vcache: np.ndarray, seqlens, scale: float):
    """Exact single-query attention over the first L_b cached keys.

    q: [B, Hq, d]; kcache, vcache: [B, Hkv, Lcap, d]; seqlens: [B] with
    1 <= L_b <= Lcap. Returns O [B, Hq, d] and LSE [B, Hq].
    Source: "Attention from the kernel's side", section "Prefill and decoding
    are different problems" (one query per sequence, the whole cache streamed).
    """
    B, Hq, d = q.shape
    g = Hq // kcache.shape[1]
    O = np.empty((B, Hq, vcache.shape[-1]))
    L = np.empty((B, Hq))
    for b in range(B):
        n = int(seqlens[b])
        for h in range(Hq):
            s = (kcache[b, h // g, :n] @ q[b, h]) * scale
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            O[b, h] = (e @ vcache[b, h // g, :n]) / l
            L[b, h] = m + math.log(l)
    return O, L


def decode_split_merge(q, kcache, vcache, seqlens, scale: float, num_splits: int):
    """Flash-decoding in the oracle's own form: split the key range, merge partials.

    Split s covers keys [s*C, min((s+1)*C, L_b)) with C = ceil(Lcap / num_splits);
    each split keeps (m_s, l_s, o_s) with o_s unnormalised; the merge is
    M = max_s m_s, l = sum_s exp(m_s - M) l_s, o = sum_s exp(m_s - M) o_s,
    O = o / l, LSE = M + ln l. Empty splits contribute nothing.
    Source: "Attention from the kernel's side", section "Prefill and decoding
    are different problems" (flash-decoding: partial (m, l, o) per block of
    threads, merged by the same rescaling rule); the rule itself is the step of
    "Module 07", section "Online softmax: derivation".
    """
    B, Hq, d = q.shape
    Lcap = kcache.shape[2]
    g = Hq // kcache.shape[1]
    C = -(-Lcap // num_splits)
    O = np.empty((B, Hq, vcache.shape[-1]))
    L = np.empty((B, Hq))
    for b in range(B):
        n = int(seqlens[b])
        for h in range(Hq):
            parts = []
            for s_idx in range(num_splits):
                lo, hi = s_idx * C, min((s_idx + 1) * C, n)
                if lo >= hi:
                    parts.append((NEG_INF, 0.0, np.zeros(vcache.shape[-1])))
                    continue
                s = (kcache[b, h // g, lo:hi] @ q[b, h]) * scale
                m = s.max()
                e = np.exp(s - m)
                parts.append((m, e.sum(), e @ vcache[b, h // g, lo:hi]))
            M = max(p[0] for p in parts)
            l = 0.0
            o = np.zeros(vcache.shape[-1])
            for m_s, l_s, o_s in parts:                # fixed split order
                if m_s == NEG_INF:
                    continue
                r = math.exp(m_s - M)
                l += r * l_s
                o = o + r * o_s
            O[b, h] = o / l
            L[b, h] = M + math.log(l)
    return O, L


# ---------------------------------------------------------------------------
# Backward pass by recomputation from the saved LSE
# ---------------------------------------------------------------------------

def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, lse: np.ndarray,
                       do: np.ndarray, causal: bool, scale: float):
    """Gradients of O = softmax(scale Q K^T + mask) V with respect to Q, K, V.

    q, o, do: [B, Hq, Tq, d]; k, v: [B, Hkv, Tk, d]; lse: [B, Hq, Tq] (natural log, as
    the forward returns it). Returns dQ [B, Hq, Tq, d], dK and dV [B, Hkv, Tk, d]; the
    gradients of a K/V head are the sums over the g query heads that read it.
    Source: "FlashAttention: attention without the n x n matrix", section "Backward
    pass: recomputing is cheaper than storing": the scores are computed again, the
    probabilities recovered without normalisation as P_ij = exp(S_ij - L_i), then
    dV = P^T dO, dP = dO V^T, dS_ij = P_ij (dP_ij - D_i) with D_i = dO_i . O_i,
    dQ = dS K * scale, dK = dS^T Q * scale.
    """
    B, Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    g = Hq // Hkv
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    vis = _visible_mask(np.arange(Tq), Tk, causal)
    for b in range(B):
        for h in range(Hq):
            kk, vv = k[b, h // g], v[b, h // g]
            s = np.where(vis, (q[b, h] @ kk.T) * scale, NEG_INF)
            p = np.exp(s - lse[b, h][:, None])
            D = np.sum(do[b, h] * o[b, h], axis=1)
            dv[b, h // g] += p.T @ do[b, h]
            dp = do[b, h] @ vv.T
            ds = p * (dp - D[:, None])
            dq[b, h] = (ds @ kk) * scale
            dk[b, h // g] += (ds.T @ q[b, h]) * scale
    return dq, dk, dv


def attention_backward_rows(q, k, v, do, causal: bool, scale: float, b: int, kvh: int, q_rows, k_rows):
    """The gradients of ``attention_backward`` on selected rows of one K/V group, for sizes
    where the full gradients are too large: dQ on rows ``q_rows`` of each of the g query heads
    that read K/V head (b, kvh), and dK, dV on rows ``k_rows`` of that head. Each head's O, L
    and D_i = dO_i . O_i come from the full forward of that head (every query row).
    Returns dQ [g, len(q_rows), d], dK and dV [len(k_rows), d].
    """
    Hq, Tq = q.shape[1], q.shape[2]
    Hkv, Tk = k.shape[1], k.shape[2]
    g = Hq // Hkv
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    kk, vv = k[b, kvh], v[b, kvh]
    dq = np.zeros((g, len(q_rows), q.shape[3]))
    dk = np.zeros((len(k_rows), k.shape[3]))
    dv = np.zeros((len(k_rows), v.shape[3]))
    all_rows = np.arange(Tq)
    for gi in range(g):
        h = kvh * g + gi
        o, lse = attention_rows(q[b:b + 1, h:h + 1], k[b:b + 1, kvh:kvh + 1], v[b:b + 1, kvh:kvh + 1], 0, 0,
                                all_rows, causal, scale)
        D = np.sum(do[b, h] * o, axis=1)
        # dQ rows: full key range of each selected query row
        vis = _visible_mask(q_rows, Tk, causal)
        s = np.where(vis, (q[b, h, q_rows] @ kk.T) * scale, NEG_INF)
        p = np.exp(s - lse[q_rows][:, None])
        ds = p * (do[b, h, q_rows] @ vv.T - D[q_rows][:, None])
        dq[gi] = (ds @ kk) * scale
        # dK, dV rows: every query row against the selected keys
        visk = _visible_mask(all_rows, Tk, causal)[:, k_rows]
        sk = np.where(visk, (q[b, h] @ kk[k_rows].T) * scale, NEG_INF)
        pk = np.exp(sk - lse[:, None])
        dv += pk.T @ do[b, h]
        dsk = pk * (do[b, h] @ vv[k_rows].T - D[:, None])
        dk += (dsk.T @ q[b, h]) * scale
    return dq, dk, dv
