"""Pins for the CPU oracle: values the pages print, closed forms, invariants
and pure-Python brute force.

Each test is chosen so that a plausible slip in ``oracle.attention`` -- a
dropped term, a wrong sign, a wrong index, a transposed operand, a wrong
log base, a mask on the wrong side of the diagonal -- fails at least one of
them. None of these tests re-types the oracle's formula with numpy.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import attention, attention_rows, flop_count
from oracle.online import online_attention, online_attention_row, online_softmax_trace


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _half_unit(decimals):
    return 0.5 * 10.0 ** (-decimals) + 1e-12


# ---------------------------------------------------------------------------
# Values printed on the pages
# ---------------------------------------------------------------------------

def test_worked_example_output_and_lse(golden_dir):
    """One query, three keys: the oracle's O and LSE must reproduce the
    printed output, and LSE = max + ln(l) with the printed l."""
    g = _load(golden_dir, "worked_example.json")
    tol = _half_unit(g["printed_decimals"])
    q = np.array([[1.0]])
    k = np.array(g["scores"])[:, None]          # q . k_j = score_j with scale 1
    v = np.array(g["values"])[:, None]
    o, lse = attention(q, k, v, scale=1.0)
    assert abs(o[0, 0] - g["out"]) <= tol
    assert abs(lse[0] - (max(g["scores"]) + math.log(g["l"]))) <= tol / g["l"] + 1e-9
    # The same case with a non-unit scale folded into the inputs: scale 2
    # with halved keys must give the identical answer.
    o2, lse2 = attention(q, k / 2.0, v, scale=2.0)
    assert abs(o2[0, 0] - o[0, 0]) < 1e-12 and abs(lse2[0] - lse[0]) < 1e-12


def test_worked_example_online_state(golden_dir):
    """Blocks of two then one: the running l, acc and output match the page."""
    g = _load(golden_dir, "worked_example.json")
    tol = _half_unit(g["printed_decimals"])
    s = np.array(g["scores"])
    v = np.array(g["values"])[:, None]
    out, l, acc, m = online_attention_row(s, v, block=g["blocks"][0])
    assert abs(l - g["l"]) <= tol
    assert abs(acc[0] - g["acc"]) <= tol
    assert abs(out[0] - g["out"]) <= tol
    assert m == max(g["scores"])
    # weights after the first block, relative to its max 2
    w1 = np.exp(s[:2] - g["max_after_first_block"])
    assert np.all(np.abs(w1 - g["weights_after_first_block"]) <= tol)
    # rescaled to the new max 3
    w3 = np.exp(s - m)
    assert np.all(np.abs(w3 - g["weights_rescaled_to_max_3"]) <= tol)


def test_step3_online_softmax_trace(golden_dir):
    g = _load(golden_dir, "online_softmax_step3.json")
    rng = np.random.default_rng(g["row_generator"]["numpy_default_rng_seed"])
    x = rng.standard_normal(g["row_generator"]["count"]) * g["row_generator"]["multiplier"]
    trace, probs = online_softmax_trace(x, g["chunk"])
    tol = _half_unit(g["trace_decimals"])
    assert len(trace) == len(g["trace_m_l"])
    for (m, l), (pm, pl) in zip(trace, g["trace_m_l"]):
        assert abs(m - pm) <= tol and abs(l - pl) <= tol
    # the ordinary softmax of the whole row, from the oracle (one query whose
    # scores are x: q = [1], keys = x, scale 1, values = identity rows)
    eye = np.eye(x.size)
    o, _ = attention(np.array([[1.0]]), x[:, None], eye, scale=1.0)
    assert np.abs(probs - o[0]).max() <= g["online_vs_reference_max_error"] + 1e-15
    # the deliberate mutant that forgets to rescale l
    _, bad = online_softmax_trace(x, g["chunk"], rescale_l=False)
    assert abs(np.abs(bad - o[0]).max() - g["no_rescale_max_error"]) < 1e-12
    with np.errstate(invalid="ignore"):
        assert math.isnan(float(np.exp(-np.inf - -np.inf)))


# ---------------------------------------------------------------------------
# Brute force: pure-Python loops with math.fsum on tiny inputs
# ---------------------------------------------------------------------------

def _brute(q, k, v, scale, causal):
    M, N, Dv = len(q), len(k), len(v[0]) if len(v) else 0
    o = [[0.0] * Dv for _ in range(M)]
    lse = [-math.inf] * M
    for i in range(M):
        vis = [j for j in range(N) if (not causal or j <= i)]
        if not vis:
            continue
        sc = {j: scale * math.fsum(q[i][d] * k[j][d] for d in range(len(q[i]))) for j in vis}
        mx = max(sc.values())
        w = {j: math.exp(sc[j] - mx) for j in vis}
        l = math.fsum(w.values())
        for d in range(Dv):
            o[i][d] = math.fsum(w[j] * v[j][d] for j in vis) / l
        lse[i] = mx + math.log(l)
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("M,N,D,causal,scale", [
    (1, 1, 1, False, 1.0), (3, 5, 2, False, 0.7), (5, 3, 4, True, 0.5),
    (8, 8, 8, True, 1 / math.sqrt(8)), (7, 6, 3, False, -1.3), (4, 7, 5, True, 2.5),
    (6, 8, 8, False, 1 / math.sqrt(8)),
])
def test_brute_force_tiny(M, N, D, causal, scale):
    rng = np.random.default_rng(1000 + M * 100 + N * 10 + D)
    q = rng.standard_normal((M, D)) * 1.5
    k = rng.standard_normal((N, D)) * 1.5
    v = rng.standard_normal((N, D + 1))          # value width differs from D
    o, lse = attention(q, k, v, scale, causal)
    bo, blse = _brute(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, blse, rtol=0, atol=1e-13)


def test_brute_force_batched_layout():
    """Leading [B, H] dims: each head is its own problem (no mixing)."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 3, 4, 5))
    k = rng.standard_normal((2, 3, 6, 5))
    v = rng.standard_normal((2, 3, 6, 5))
    o, lse = attention(q, k, v, 0.4, causal=True)
    for b in range(2):
        for h in range(3):
            bo, blse = _brute(q[b, h].tolist(), k[b, h].tolist(), v[b, h].tolist(), 0.4, True)
            np.testing.assert_allclose(o[b, h], bo, atol=1e-13, rtol=0)
            np.testing.assert_allclose(lse[b, h], blse, atol=1e-13, rtol=0)


# ---------------------------------------------------------------------------
# Closed forms and special cases
# ---------------------------------------------------------------------------

def test_single_key_returns_that_value():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((4, 6)), rng.standard_normal((1, 6)), rng.standard_normal((1, 6))
    o, lse = attention(q, k, v, 0.3)
    np.testing.assert_allclose(o, np.repeat(v, 4, axis=0), atol=1e-15)
    for i in range(4):
        assert abs(lse[i] - 0.3 * math.fsum(q[i, d] * k[0, d] for d in range(6))) < 1e-14


def test_identical_scores_give_mean_of_values():
    """All keys equal -> uniform weights -> O is the mean of V; LSE = s + ln N."""
    rng = np.random.default_rng(4)
    N = 37
    q = rng.standard_normal((5, 8))
    k = np.repeat(rng.standard_normal((1, 8)), N, axis=0)
    v = rng.standard_normal((N, 8))
    o, lse = attention(q, k, v, 0.5)
    mean = np.array([math.fsum(v[:, d]) / N for d in range(8)])
    np.testing.assert_allclose(o, np.repeat(mean[None], 5, axis=0), atol=1e-14)
    s = 0.5 * np.array([math.fsum(q[i] * k[0]) for i in range(5)])
    np.testing.assert_allclose(lse, s + math.log(N), atol=1e-13)


def test_zero_scale_is_uniform_and_causal_prefix_mean():
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal((6, 4)), rng.standard_normal((6, 4)), rng.standard_normal((6, 4))
    o, lse = attention(q, k, v, 0.0, causal=True)
    for i in range(6):
        want = [math.fsum(v[:i + 1, d]) / (i + 1) for d in range(4)]
        np.testing.assert_allclose(o[i], want, atol=1e-15)
        assert abs(lse[i] - math.log(i + 1)) < 1e-15


def test_causal_first_row_and_mask_side():
    """Row 0 sees only key 0; the last row of a square causal problem sees
    everything, so it equals the non-causal answer for that row."""
    rng = np.random.default_rng(6)
    q, k, v = rng.standard_normal((9, 4)), rng.standard_normal((9, 4)), rng.standard_normal((9, 4))
    o, lse = attention(q, k, v, 0.8, causal=True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    assert abs(lse[0] - 0.8 * math.fsum(q[0] * k[0])) < 1e-14
    o_full, lse_full = attention(q, k, v, 0.8, causal=False)
    np.testing.assert_allclose(o[-1], o_full[-1], atol=1e-14)
    assert abs(lse[-1] - lse_full[-1]) < 1e-14
    # changing a future key/value must not change an earlier row
    k2, v2 = k.copy(), v.copy()
    k2[5] += 10.0
    v2[5] -= 7.0
    o2, lse2 = attention(q, k2, v2, 0.8, causal=True)
    np.testing.assert_array_equal(o2[:5], o[:5])
    np.testing.assert_array_equal(lse2[:5], lse[:5])
    assert np.abs(o2[5:] - o[5:]).max() > 1e-3


def test_large_scale_selects_argmax_value():
    """As the scale grows, softmax becomes a hard argmax over the keys."""
    q = np.array([[1.0, 0.0]])
    k = np.array([[0.1, 0.0], [0.9, 0.0], [0.5, 0.0]])
    v = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])
    o, lse = attention(q, k, v, 200.0)
    np.testing.assert_allclose(o[0], v[1], atol=1e-30 + 1e-15)
    assert abs(lse[0] - 200.0 * 0.9) < 1e-15 + 200.0 * 0.9 * 1e-15


def test_empty_keys_give_zero_output_and_neg_inf_lse():
    q = np.ones((3, 4))
    k = np.zeros((0, 4))
    v = np.zeros((0, 4))
    o, lse = attention(q, k, v, 0.5)
    assert o.shape == (3, 4) and np.all(o == 0.0)
    assert np.all(np.isneginf(lse))


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def _scores_py(q, k, scale):
    return np.array([[scale * math.fsum(q[i] * k[j]) for j in range(len(k))] for i in range(len(q))])


def test_lse_normalises_softmax_rows():
    """sum_j exp(S_ij - LSE_i) = 1 and O = exp(S - LSE) V with S built in
    pure Python ("Module 08", recomputing P tiles from the saved L)."""
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal((7, 5)) * 2, rng.standard_normal((11, 5)) * 2, rng.standard_normal((11, 3))
    o, lse = attention(q, k, v, 0.6)
    s = _scores_py(q, k, 0.6)
    for i in range(7):
        p = [math.exp(s[i, j] - lse[i]) for j in range(11)]
        assert abs(math.fsum(p) - 1.0) < 1e-13
        for d in range(3):
            assert abs(math.fsum(p[j] * v[j, d] for j in range(11)) - o[i, d]) < 1e-13


def test_convex_hull_and_permutation_invariance():
    rng = np.random.default_rng(9)
    q, k, v = rng.standard_normal((10, 6)) * 3, rng.standard_normal((40, 6)) * 3, rng.standard_normal((40, 6))
    o, lse = attention(q, k, v, 0.4)
    assert np.all(o <= v.max(axis=0) + 1e-12) and np.all(o >= v.min(axis=0) - 1e-12)
    perm = rng.permutation(40)
    o2, lse2 = attention(q, k[perm], v[perm], 0.4)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)
    # causal: each row lies in the hull of its visible values only
    oc, _ = attention(q, k[:10], v[:10], 0.4, causal=True)
    for i in range(10):
        assert np.all(oc[i] <= v[:i + 1].max(axis=0) + 1e-12)
        assert np.all(oc[i] >= v[:i + 1].min(axis=0) - 1e-12)


def test_per_row_score_shift_moves_lse_only():
    """Adding a direction w to every key adds scale*q_i.w to all of row i's
    scores: O is unchanged and LSE_i moves by exactly that amount."""
    rng = np.random.default_rng(10)
    q, k, v = rng.standard_normal((6, 4)), rng.standard_normal((9, 4)), rng.standard_normal((9, 4))
    w = np.array([0.5, -1.0, 2.0, 0.25])
    o, lse = attention(q, k, v, 0.7)
    o2, lse2 = attention(q, k + w[None], v, 0.7)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    shift = np.array([0.7 * math.fsum(q[i] * w) for i in range(6)])
    np.testing.assert_allclose(lse2 - lse, shift, atol=1e-13)


def test_value_linearity():
    rng = np.random.default_rng(11)
    q, k = rng.standard_normal((5, 4)), rng.standard_normal((8, 4))
    v1, v2 = rng.standard_normal((8, 3)), rng.standard_normal((8, 3))
    o1, _ = attention(q, k, v1, 0.9, causal=True)
    o2, _ = attention(q, k, v2, 0.9, causal=True)
    o3, _ = attention(q, k, 2.0 * v1 - 3.0 * v2, 0.9, causal=True)
    np.testing.assert_allclose(o3, 2.0 * o1 - 3.0 * o2, atol=1e-13)


def test_attention_rows_matches_full_rows():
    rng = np.random.default_rng(12)
    q, k, v = rng.standard_normal((300, 8)), rng.standard_normal((300, 8)), rng.standard_normal((300, 8))
    o, lse = attention(q, k, v, 0.35, causal=True)
    rows = np.array([0, 1, 127, 128, 200, 299])
    orow, lrow = attention_rows(q, k, v, 0.35, True, rows)
    np.testing.assert_array_equal(orow, o[rows])
    np.testing.assert_array_equal(lrow, lse[rows])


def test_flop_count_convention():
    # "Module 08", Code Step 4: 256,000,000 matmul FLOPs at N = 1000, d = 64
    assert flop_count(1, 1, 1000, 1000, 64, False) == 256_000_000
    assert flop_count(1, 1, 1000, 1000, 64, True) == 128_000_000


# ---------------------------------------------------------------------------
# The online recurrence model and the mistakes the parity check must catch
# ---------------------------------------------------------------------------

def _max_err(a, b):
    return float(np.abs(np.asarray(a) - np.asarray(b)).max())


@pytest.mark.parametrize("base2", [False, True])
@pytest.mark.parametrize("causal", [False, True])
def test_online_model_reaches_definition(base2, causal):
    """The tiled recurrence equals materialised attention to fp64 rounding
    (the pages' Step 4 reports 2e-16..8e-16 for its tiled version)."""
    rng = np.random.default_rng(13)
    for n in (256, 1000):
        q, k, v = (rng.standard_normal((n, 64)) for _ in range(3))
        o, lse = attention(q, k, v, 1 / 8, causal)
        o2, lse2 = online_attention(q, k, v, 1 / 8, causal, block=196, base2=base2)
        assert _max_err(o, o2) < 1e-14
        assert _max_err(lse, lse2) < 1e-12


def test_forgotten_acc_alpha_only_shows_beyond_one_tile():
    """Dropping acc*alpha is exact while all keys fit in one tile and wrong
    once a later tile raises the max ("Things that break")."""
    rng = np.random.default_rng(14)
    q = rng.standard_normal((64, 32)) * 3
    k = rng.standard_normal((300, 32)) * 3
    v = rng.standard_normal((300, 32))
    o, _ = attention(q, k[:128], v[:128], 0.2)
    bad, _ = online_attention(q, k[:128], v[:128], 0.2, block=128, rescale_acc=False)
    assert _max_err(o, bad) < 1e-13                         # one tile: invisible
    o, _ = attention(q, k, v, 0.2)
    bad, _ = online_attention(q, k, v, 0.2, block=128, rescale_acc=False)
    assert _max_err(o, bad) > 1e-2                          # several tiles: caught


def test_mixed_exponent_bases_is_caught():
    rng = np.random.default_rng(15)
    q, k, v = rng.standard_normal((32, 16)) * 2, rng.standard_normal((400, 16)) * 2, rng.standard_normal((400, 16))
    o, _ = attention(q, k, v, 0.25)
    bad, _ = online_attention(q, k, v, 0.25, block=64, base2=True, alpha_base_e=True)
    assert _max_err(o, bad) > 1e-3


def test_reverse_tile_order_nan_without_guard_exact_with_guard():
    """"Module 08" Practice 2: causal, N = 300, blocks of 100 visited last to
    first. Rows 0..199 meet a fully masked block first: without a guard they
    become NaN; with an infinite max clamped to 0 they are exact."""
    rng = np.random.default_rng(16)
    n = 300
    q, k, v = (rng.standard_normal((n, 16)) for _ in range(3))
    o, lse = attention(q, k, v, 0.25, causal=True)
    bad, _ = online_attention(q, k, v, 0.25, True, block=100, reverse=True, guard=False)
    nan_rows = np.isnan(bad).any(axis=1)
    assert nan_rows.sum() == 200 and nan_rows[:200].all() and not nan_rows[200:].any()
    good, lse_g = online_attention(q, k, v, 0.25, True, block=100, reverse=True, guard=True)
    assert _max_err(o, good) < 1e-13 and _max_err(lse, lse_g) < 1e-12
