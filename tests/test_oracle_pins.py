"""Pins for the float64 oracle: what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers the
pages print for their worked examples (``tests/golden``), closed forms,
special cases that reduce to a known answer, brute force on tiny inputs, and
the identity between the block recurrence and the three-pass definition.
The cases are chosen so that a dropped term, a wrong sign, an off-by-one in
the causal rule, a wrong GQA head mapping, a transposed operand, a missing
scale or a misplaced eps fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import attention as A


# ---------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_module07_worked_example_row0(golden):
    g = golden["module07_row0"]
    o, states = oracle.online_softmax_blocks(g["scores"], g["values"], g["block"])
    s1, s2 = states
    b1, b2 = g["after_block1"], g["after_block2"]
    assert s1["m"] == b1["m"] and s1["corr"] == b1["corr"]
    assert abs(s1["l"] - b1["l"]) <= b1["tol"]
    assert abs(float(s1["O"]) - b1["O"]) <= b1["tol"]
    assert s2["m"] == b2["m"]
    assert abs(s2["corr"] - b2["corr"]) <= b2["tol"]
    assert abs(s2["l"] - b2["l"]) <= b2["tol"]
    assert abs(float(s2["O"]) - b2["O"]) <= b2["tol"]
    # the block-2 contributions printed beside the update
    p = np.exp(np.array(g["scores"][4:], float) - 5.0)
    assert abs(p.sum() - g["block2_sums"]["sum_p"]) <= g["block2_sums"]["tol"]
    assert abs(p @ np.array(g["values"][4:], float) - g["block2_sums"]["sum_pv"]) <= g["block2_sums"]["tol"]
    assert abs(float(o) - g["final"]["O_over_l"]) <= g["final"]["tol"]
    # the page checks the result against the plain softmax of the whole row
    o3, _ = oracle.scores_softmax_weighted(g["scores"], g["values"])
    assert abs(float(o3) - g["final"]["O_over_l"]) <= g["final"]["tol"]


def test_module07_row1_brute_force():
    # Row 1 of the same example has no printed answer; it is checked by an
    # explicit exp-weighted average with math.fsum (no max subtraction).
    s = [7, 1, 2, 0, 3, 2, 1, 0]
    v = list(range(1, 9))
    num = math.fsum(math.exp(x) * y for x, y in zip(s, v))
    den = math.fsum(math.exp(x) for x in s)
    o_blk, _ = oracle.online_softmax_blocks(s, v, 4)
    o3, lse = oracle.scores_softmax_weighted(s, v)
    assert abs(float(o_blk) - num / den) < 1e-13
    assert abs(float(o3) - num / den) < 1e-13
    assert abs(lse - math.log(den)) < 1e-13


def test_lesson_stream_example(golden):
    g = golden["lesson_stream_x132"]
    # step by step l and the rescale factor of the table
    for n in range(1, 4):
        m, l = oracle.online_normalizer(g["xs"][:n])
        assert abs(l - g["steps_l"][n - 1]) <= g["tol_l"]
    m, l, a, o = oracle.online_weighted_stream(g["xs"], g["vs"])
    assert m == g["m"]
    assert abs(l - g["l"]) <= g["tol_l"]
    assert abs(a - g["a"]) <= g["tol_a"]
    assert abs(o - g["o"]) <= g["tol_o"]
    # the printed probabilities e^(x - 3) / l
    p = [math.exp(x - m) / l for x in g["xs"]]
    for got, want in zip(p, g["probabilities"]):
        assert abs(got - want) <= g["tol_p"]
    assert abs(math.exp(1 - 3) - g["steps_factor"][1]) <= g["tol_l"]


def test_lesson_exercise_expected_print(golden):
    g = golden["lesson_exercise_main"]
    m, l = oracle.online_normalizer(iter(g["xs"]))
    assert m == g["m"]
    assert f"{l:.10f}".startswith(g["l_prefix"])


def test_chapter5_example_5_6(golden):
    g = golden["chapter5_example_5_6"]
    o, states = oracle.online_softmax_blocks(g["scores"], g["values"], 1)
    assert states[0]["m"] == g["after_first"]["m"]
    assert states[0]["l"] == g["after_first"]["l"]
    assert float(states[0]["O"]) == g["after_first"]["u"]
    assert abs(states[1]["corr"] - g["r"]) < 1e-15
    assert abs(states[1]["l"] - g["after_second"]["l"]) < 1e-15
    assert abs(float(states[1]["O"]) - g["after_second"]["u"]) < 1e-15
    assert abs(float(o) - g["result_num"] / g["result_den"]) < 1e-15
    m, l, a, o2 = oracle.online_weighted_stream(g["scores"], g["values"])
    assert abs(o2 - 7 / 3) < 1e-15


def test_block_counts_printed(golden):
    for c in golden["block_counts"]["cases"]:
        assert oracle.count_blocks(c["T"], c["bq"], c["bk"], c["causal"]) == c["blocks"]


def test_block_counts_closed_form():
    # n aligned blocks per side: n(n+1)/2 causal pairs, n^2 without the mask
    # (e.g. T = 2048 in blocks of 128: 16 * 17 / 2 = 136).
    for T, b in [(2048, 128), (1024, 64), (512, 128)]:
        n = T // b
        assert oracle.count_blocks(T, b, b, True) == n * (n + 1) // 2
        assert oracle.count_blocks(T, b, b, False) == n * n


def test_two_element_running_sum_closed_form():
    # running sum after (2, 5) with m = 5 is e^(2-5) + e^0 = 1 + e^-3 ~ 1.05
    m, l = oracle.online_normalizer([2.0, 5.0])
    assert m == 5.0
    assert abs(l - (1 + math.exp(-3))) < 1e-15
    assert round(l, 2) == 1.05


# ---------------------------------------------------------------------------
# Closed forms and special cases of the full attention oracle
# ---------------------------------------------------------------------------

def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


@pytest.mark.parametrize("causal", [False, True])
def test_single_key_returns_its_value(causal):
    q = _rand((1, 2, 1, 8), 1)
    k = _rand((1, 2, 1, 8), 2)
    v = _rand((1, 2, 1, 8), 3)
    scale = 0.37
    O, L = oracle.attention(q, k, v, causal, scale)
    assert np.array_equal(O, v)
    s00 = scale * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    assert np.allclose(L[:, :, 0], s00, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_return_that_constant(causal):
    q = _rand((1, 1, 20, 8), 4, 3.0)
    k = _rand((1, 1, 20, 8), 5)
    v = np.full((1, 1, 20, 8), -1.25)
    v[..., 3] = 7.5
    O, _ = oracle.attention(q, k, v, causal, 0.5)
    assert np.allclose(O, v[:, :, :1].repeat(20, axis=2), rtol=0, atol=1e-13)


def test_causal_row0_is_v0():
    q = _rand((2, 3, 17, 8), 6)
    k = _rand((2, 3, 17, 8), 7)
    v = _rand((2, 3, 17, 8), 8)
    O, L = oracle.attention(q, k, v, True, 0.3)
    assert np.array_equal(O[:, :, 0], v[:, :, 0])
    s00 = 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    assert np.allclose(L[:, :, 0], s00, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    T, d = 23, 4
    q = np.zeros((1, 1, T, d))
    k = _rand((1, 1, T, d), 9)
    v = _rand((1, 1, T, d), 10)
    O, L = oracle.attention(q, k, v, causal, 0.7)
    for i in range(T):
        n = i + 1 if causal else T
        assert np.allclose(O[0, 0, i], v[0, 0, :n].mean(axis=0), atol=1e-14)
        assert abs(L[0, 0, i] - math.log(n)) < 1e-14


def test_gqa_head_mapping_groups_contiguous_heads():
    # each K/V head carries its own constant value; query head h must see the
    # constant of K/V head floor(h / g)
    B, Hq, Hkv, T, d = 1, 8, 2, 9, 4
    q = _rand((B, Hq, T, d), 11)
    k = _rand((B, Hkv, T, d), 12)
    v = np.empty((B, Hkv, T, d))
    v[:, 0] = 3.0
    v[:, 1] = -5.0
    O, _ = oracle.attention(q, k, v, False, 0.5)
    for h in range(Hq):
        assert np.allclose(O[0, h], 3.0 if h // 4 == 0 else -5.0, atol=1e-13)


def test_noncausal_invariant_under_joint_key_permutation():
    q = _rand((1, 2, 11, 6), 13)
    k = _rand((1, 2, 11, 6), 14)
    v = _rand((1, 2, 11, 6), 15)
    perm = np.random.default_rng(16).permutation(11)
    O1, L1 = oracle.attention(q, k, v, False, 0.4)
    O2, L2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], False, 0.4)
    assert np.allclose(O1, O2, atol=1e-13) and np.allclose(L1, L2, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    q = _rand((1, 1, 40, 8), 17)
    k = _rand((1, 1, 40, 8), 18)
    v = _rand((1, 1, 40, 8), 19)
    scale = 1 / math.sqrt(8)
    _, L = oracle.attention(q, k, v, causal, scale)
    S = scale * q[0, 0] @ k[0, 0].T
    for i in range(40):
        n = i + 1 if causal else 40
        p = np.exp(S[i, :n] - L[0, 0, i])
        assert np.all(p >= 0)
        assert abs(p.sum() - 1.0) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_tiny(causal):
    # explicit loops, explicit exponentials summed with fsum, no max subtraction
    B, Hq, Hkv, Tq, Tk, d = 1, 4, 2, 7, 7, 3
    q = _rand((B, Hq, Tq, d), 20)
    k = _rand((B, Hkv, Tk, d), 21)
    v = _rand((B, Hkv, Tk, d), 22)
    scale = 0.61
    O, L = oracle.attention(q, k, v, causal, scale)
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        for i in range(Tq):
            js = [j for j in range(Tk) if (not causal or j <= i)]
            w = []
            for j in js:
                s = scale * math.fsum(q[0, h, i, t] * k[0, kv, j, t] for t in range(d))
                w.append(math.exp(s))
            den = math.fsum(w)
            for t in range(d):
                num = math.fsum(wj * v[0, kv, j, t] for wj, j in zip(w, js))
                assert abs(O[0, h, i, t] - num / den) < 1e-12
            assert abs(L[0, h, i] - math.log(den)) < 1e-12


def test_brute_force_rectangular_top_left_causal():
    # Tq != Tk: query i sees keys j <= i (top-left alignment)
    q = _rand((1, 1, 5, 2), 23)
    k = _rand((1, 1, 9, 2), 24)
    v = _rand((1, 1, 9, 2), 25)
    O, L = oracle.attention(q, k, v, True, 1.0)
    for i in range(5):
        w = [math.exp(math.fsum(q[0, 0, i] * k[0, 0, j])) for j in range(i + 1)]
        den = math.fsum(w)
        assert abs(L[0, 0, i] - math.log(den)) < 1e-12
        for t in range(2):
            assert abs(O[0, 0, i, t] - math.fsum(wj * v[0, 0, j, t] for j, wj in enumerate(w)) / den) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Br,Bc", [(7, 13), (32, 32), (16, 5), (64, 64)])
def test_recurrence_equals_three_pass(causal, Br, Bc):
    q = _rand((1, 2, 100, 16), 26)
    k = _rand((1, 1, 100, 16), 27)
    v = _rand((1, 1, 100, 16), 28)
    O1, L1 = oracle.attention(q, k, v, causal, 0.25)
    O2, L2 = oracle.attention_online(q, k, v, causal, 0.25, Br, Bc)
    assert np.max(np.abs(O1 - O2)) < 1e-12
    assert np.max(np.abs(L1 - L2)) < 1e-12


def test_peaked_scores_stay_finite():
    # Q scaled by 100: exp of the raw scores overflows in float32 (the pages'
    # arithmetic type for this check); the max-subtracted oracle stays finite
    q = _rand((1, 1, 64, 32), 29, 100.0)
    k = _rand((1, 1, 64, 32), 30)
    v = _rand((1, 1, 64, 32), 31)
    scale = 1 / math.sqrt(32)
    with np.errstate(over="ignore"):
        assert not np.all(np.isfinite(np.exp((scale * q[0, 0] @ k[0, 0].T).astype(np.float32))))
    for causal in (False, True):
        O, L = oracle.attention(q, k, v, causal, scale)
        assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
        O2, L2 = oracle.attention_online(q, k, v, causal, scale, 16, 16)
        assert np.max(np.abs(O - O2)) < 1e-10


def test_attention_rows_matches_full():
    q = _rand((2, 4, 50, 8), 32)
    k = _rand((2, 2, 50, 8), 33)
    v = _rand((2, 2, 50, 8), 34)
    O, L = oracle.attention(q, k, v, True, 0.3, row_chunk=16)
    rows = [0, 7, 31, 49]
    o, lse = oracle.attention_rows(q, k, v, 1, 3, rows, True, 0.3)
    assert np.max(np.abs(o - O[1, 3, rows])) < 1e-13
    assert np.max(np.abs(lse - L[1, 3, rows])) < 1e-13


# ---------------------------------------------------------------------------
# Decode
# ---------------------------------------------------------------------------

def test_decode_equals_last_prefill_row():
    B, Hq, Hkv, Lcap, d = 3, 4, 2, 40, 8
    k = _rand((B, Hkv, Lcap, d), 35)
    v = _rand((B, Hkv, Lcap, d), 36)
    q = _rand((B, Hq, d), 37)
    lens = [1, 17, 40]
    O, L = oracle.decode(q, k, v, lens, 0.35)
    for b, n in enumerate(lens):
        qp = np.zeros((1, Hq, n, d))
        qp[0, :, n - 1] = q[b]
        Op, Lp = oracle.attention(qp, k[b:b + 1, :, :n], v[b:b + 1, :, :n], True, 0.35)
        assert np.max(np.abs(Op[0, :, n - 1] - O[b])) < 1e-13
        assert np.max(np.abs(Lp[0, :, n - 1] - L[b])) < 1e-13


def test_decode_zero_query_is_mean_over_length():
    k = _rand((2, 1, 30, 4), 38)
    v = _rand((2, 1, 30, 4), 39)
    q = np.zeros((2, 2, 4))
    O, L = oracle.decode(q, k, v, [5, 30], 1.0)
    assert np.allclose(O[0, 1], v[0, 0, :5].mean(0), atol=1e-14)
    assert np.allclose(O[1, 0], v[1, 0].mean(0), atol=1e-14)
    assert abs(L[0, 0] - math.log(5)) < 1e-14 and abs(L[1, 1] - math.log(30)) < 1e-14


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 16, 64])
def test_split_merge_equals_decode(num_splits):
    B, Hq, Hkv, Lcap, d = 3, 8, 2, 64, 8
    k = _rand((B, Hkv, Lcap, d), 40)
    v = _rand((B, Hkv, Lcap, d), 41)
    q = _rand((B, Hq, d), 42, 2.0)
    lens = [1, 33, 64]
    O1, L1 = oracle.decode(q, k, v, lens, 0.5)
    O2, L2 = oracle.decode_split_merge(q, k, v, lens, 0.5, num_splits)
    assert np.max(np.abs(O1 - O2)) < 1e-12
    assert np.max(np.abs(L1 - L2)) < 1e-12


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rmsnorm_zeros_to_zeros():
    y = oracle.rmsnorm(np.zeros((4, 16)), np.ones(16), 1e-6)
    assert np.array_equal(y, np.zeros((4, 16)))


def test_rmsnorm_large_component_finite():
    x = _rand((3, 64), 43)
    x[0, 0] = 1e3
    y = oracle.rmsnorm(x, np.ones(64), 1e-6)
    assert np.all(np.isfinite(y))
    assert abs(y[0, 0] - 1e3 / math.sqrt((x[0] ** 2).mean() + 1e-6)) < 1e-9


def test_rmsnorm_unit_weight_gives_unit_rms():
    x = _rand((8, 512), 44)
    eps = 1e-6
    y = oracle.rmsnorm(x, np.ones(512), eps)
    ms = (x ** 2).mean(axis=1)
    rms = np.sqrt((y ** 2).mean(axis=1))
    assert np.allclose(rms, np.sqrt(ms / (ms + eps)), atol=1e-14)
    assert np.all(np.abs(rms - 1) < 1e-4)


def test_rmsnorm_constant_rows_eps_inside_root_mean_over_D():
    # row t is the constant c_t; y = c_t / sqrt(c_t^2 + eps) * w. A small c
    # separates eps-inside-the-root from eps-outside, and distinct rows
    # separate a mean over D from a mean over T.
    D, eps = 32, 1e-6
    c = np.array([1e-3, 2.0, -0.5])
    x = np.repeat(c[:, None], D, axis=1)
    w = np.linspace(0.5, 1.5, D)
    y = oracle.rmsnorm(x, w, eps)
    want = (c / np.sqrt(c * c + eps))[:, None] * w[None, :]
    assert np.allclose(y, want, rtol=0, atol=1e-14)
    assert abs(y[0, 0] / w[0] - 1 / math.sqrt(2)) < 1e-12


def test_rmsnorm_does_not_mutate_inputs():
    x = _rand((4, 8), 45)
    w = _rand((8,), 46)
    x0, w0 = x.copy(), w.copy()
    oracle.rmsnorm(x, w, 1e-6)
    assert np.array_equal(x, x0) and np.array_equal(w, w0)


def test_rmsnorm_residual_reduces_to_rmsnorm_and_to_closed_forms():
    # r = 0: exactly the plain RMSNorm; the sum is symmetric in x and r
    x, r = _rand((5, 64), 47), _rand((5, 64), 48)
    w = _rand((64,), 49)
    y0, h0 = oracle.rmsnorm_residual(x, np.zeros_like(x), w, 1e-6)
    assert np.array_equal(y0, oracle.rmsnorm(x, w, 1e-6)) and np.array_equal(h0, x)
    y1, h1 = oracle.rmsnorm_residual(x, r, w, 1e-6)
    y2, h2 = oracle.rmsnorm_residual(r, x, w, 1e-6)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)
    # x = -r cancels: h = 0 and y = 0 (0 / sqrt(eps))
    y3, h3 = oracle.rmsnorm_residual(x, -x, w, 1e-6)
    assert np.array_equal(h3, np.zeros_like(x)) and np.array_equal(y3, np.zeros_like(x))
    # constant rows again: x + r = c_t, y = c_t / sqrt(c_t^2 + eps) * w
    c = np.array([0.25, -3.0])
    xc = np.repeat((c / 2)[:, None], 16, axis=1)
    yc, _ = oracle.rmsnorm_residual(xc, xc, np.ones(16), 1e-6)
    assert np.allclose(yc, (c / np.sqrt(c * c + 1e-6))[:, None], rtol=0, atol=1e-14)
