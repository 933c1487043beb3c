"""Pins of the backward oracle (oracle.backward.attention_bwd), CPU only.

None of these re-types the oracle's formulas: the gradients are checked
against central finite differences of the FORWARD oracle (the definition of
a derivative), against closed forms of special cases, and against the
recompute identity of "Module 08: FlashAttention and Memory-Efficient
Kernels", Code Step 6 (P rebuilt as exp(S - L) equals the stored P).
"""

import math

import numpy as np
import pytest

from oracle import attention, attention_bwd, bwd_flop_count


def _loss(q, k, v, g, scale, causal):
    o, _ = attention(q, k, v, scale, causal)
    return float(np.sum(o * g))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("M,N,D", [(3, 4, 2), (5, 5, 3), (1, 6, 4), (6, 2, 2)])
def test_gradients_match_finite_differences(M, N, D, causal):
    rng = np.random.default_rng(M * 100 + N * 10 + D + causal)
    q, k, v = (rng.standard_normal(s) for s in ((2, M, D), (2, N, D), (2, N, D)))
    g = rng.standard_normal((2, M, D))            # dL/dO of L = sum(O * g)
    scale = 0.7
    dq, dk, dv = attention_bwd(q, k, v, g, scale, causal)
    h = 1e-6
    for x, grad in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            fp = _loss(q, k, v, g, scale, causal)
            x[idx] = old - h
            fm = _loss(q, k, v, g, scale, causal)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8)


def test_identical_keys_give_zero_dq_and_mean_dv():
    # all scores of a row equal: P = 1/N, the row's softmax is flat, so Q has
    # no influence (dQ = 0) and every V row receives the mean of dO.
    rng = np.random.default_rng(7)
    M, N, D = 4, 5, 3
    q = rng.standard_normal((M, D))
    k = np.tile(rng.standard_normal((1, D)), (N, 1))
    v = rng.standard_normal((N, D))
    g = rng.standard_normal((M, D))
    dq, dk, dv = attention_bwd(q, k, v, g, 0.9, False)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dv, np.tile(g.sum(0) / N, (N, 1)), rtol=1e-13, atol=1e-14)


def test_zero_output_gradient_gives_zero_gradients():
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal((3, 4)), rng.standard_normal((6, 4)), rng.standard_normal((6, 4))
    for x in attention_bwd(q, k, v, np.zeros((3, 4)), 0.5, True):
        assert np.all(x == 0)


def test_single_key_routes_all_gradient_to_v():
    # one key: P = 1, O = V_0 for every row; dV_0 = sum of dO, dQ = dK = 0
    rng = np.random.default_rng(9)
    q, k, v = rng.standard_normal((4, 3)), rng.standard_normal((1, 3)), rng.standard_normal((1, 3))
    g = rng.standard_normal((4, 3))
    dq, dk, dv = attention_bwd(q, k, v, g, 1.3, False)
    np.testing.assert_allclose(dq, 0.0, atol=1e-14)
    np.testing.assert_allclose(dk, 0.0, atol=1e-14)
    np.testing.assert_allclose(dv, g.sum(0, keepdims=True), rtol=1e-13)


def test_causal_future_keys_get_no_gradient_from_earlier_rows():
    # with one query row (row 0) only key 0 is visible: every other key and
    # value row gets zero gradient
    rng = np.random.default_rng(10)
    q, k, v = rng.standard_normal((1, 4)), rng.standard_normal((5, 4)), rng.standard_normal((5, 4))
    g = rng.standard_normal((1, 4))
    dq, dk, dv = attention_bwd(q, k, v, g, 0.8, True)
    assert np.all(dk[1:] == 0) and np.all(dv[1:] == 0)
    np.testing.assert_allclose(dv[0], g[0], rtol=1e-13)


def test_recomputed_p_matches_stored_p():
    # Code Step 6: P rebuilt tile by tile as exp(S - L) from Q, K and the one
    # number per row equals the softmax of the full score matrix
    rng = np.random.default_rng(0)
    N, d = 300, 16
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    scale = 1 / math.sqrt(d)
    _, lse = attention(q, k, v, scale, False)
    s = scale * q @ k.T
    p_full = np.exp(s - s.max(1, keepdims=True))
    p_full /= p_full.sum(1, keepdims=True)
    worst = 0.0
    for i in range(0, N, 64):
        for j in range(0, N, 100):
            tile = np.exp(scale * q[i:i + 64] @ k[j:j + 100].T - lse[i:i + 64, None])
            worst = max(worst, float(np.abs(tile - p_full[i:i + 64, j:j + 100]).max()))
    assert worst < 1e-14


def test_bwd_flop_count_is_five_products():
    # Practice 3: four products in the standard backward plus the recomputed Q K^T
    assert bwd_flop_count(1, 1, 10, 20, 8, False) == 5 * 2 * 10 * 20 * 8
    assert bwd_flop_count(2, 3, 10, 20, 8, True) == 0.5 * 6 * 5 * 2 * 10 * 20 * 8
