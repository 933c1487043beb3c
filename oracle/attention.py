"""Materialised attention in float64: the parity oracle for fa_fwd.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA path never
imports this module.

What is computed, for every (batch, head) and every query row i
--------------------------------------------------------------------
Written from the plain definition of attention on the pages:

* "Module 08: FlashAttention and Memory-Efficient Kernels", section
  "Where the time goes in standard attention": S = QK^T/sqrt(d),
  P = softmax(S) row by row, O = PV; and its Code Step 1 ("the library"),
  whose standard attention subtracts the row maximum before the exponential
  and masks causal scores above the diagonal with -inf.
* Same page, section "The backward pass: recompute instead of store": the
  one number per row that is kept is the log-sum-exp L = m + log(l).
* "FlashAttention in Triton: A Tile-by-Tile Walkthrough", section
  "First, what does attention actually do?": Q has M rows, K and V have N
  rows, all of width D; O is M x D.

Steps, in float64 on the inputs exactly as given (bf16 inputs arrive already
rounded and are upcast without change):

1. S = scale * Q K^T                        (M x N)
2. causal: S[i, j] = -inf where j > i        (top-left alignment, j <= i kept)
3. m_i   = max_j S[i, j]
4. P     = exp(S - m_i)
5. l_i   = sum_j P[i, j]
6. O_i   = (sum_j P[i, j] V_j) / l_i
7. LSE_i = m_i + ln(l_i)

A row with no visible key (N = 0) has m_i = -inf and l_i = 0; the pages
prescribe no value for it (they only say the kernel must not produce NaN),
and this oracle's reading is O_i = 0 and LSE_i = -inf.

``scale`` is an explicit argument; the pages' launcher uses 1/sqrt(D).

Rows are computed independently of one another, so ``attention_rows`` may
evaluate any subset of rows (used for the 64K-token causal workload, whose
full score matrix would not fit in memory); the arithmetic per row is the
same seven steps.
"""

from __future__ import annotations

import numpy as np

__all__ = ["attention", "attention_rows", "flop_count"]

# Rows per chunk when a head is too large to materialise at once. Chunking
# over rows does not change any row's arithmetic.
_ROW_CHUNK = 2048


def _one_head(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
              causal: bool, rows: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Steps 1-7 for the query rows ``rows`` of one head (float64 out)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_keys = k.shape[0]
    d_v = v.shape[1]
    o = np.zeros((rows.size, d_v), dtype=np.float64)
    lse = np.full(rows.size, -np.inf, dtype=np.float64)
    if n_keys == 0 or rows.size == 0:
        return o, lse
    for lo in range(0, rows.size, _ROW_CHUNK):
        r = rows[lo:lo + _ROW_CHUNK]
        # 1. scaled scores
        s = scale * (q[r] @ k.T)
        # 2. causal mask: key j is visible to query i only when j <= i
        if causal:
            cols = np.arange(n_keys)[None, :]
            s = np.where(cols <= r[:, None], s, -np.inf)
        # 3. row maximum (a row with no visible key keeps -inf)
        m = s.max(axis=1)
        visible = np.isfinite(m)
        m_sub = np.where(visible, m, 0.0)
        # 4. unnormalised probabilities
        p = np.exp(s - m_sub[:, None])
        # 5. row sums
        l = p.sum(axis=1)
        # 6. normalised output
        acc = p @ v
        o_chunk = np.zeros_like(acc)
        o_chunk[visible] = acc[visible] / l[visible, None]
        # 7. log-sum-exp
        lse_chunk = np.full(r.size, -np.inf)
        lse_chunk[visible] = m[visible] + np.log(l[visible])
        o[lo:lo + r.size] = o_chunk
        lse[lo:lo + r.size] = lse_chunk
    return o, lse


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
              causal: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """O and LSE of softmax(scale * Q K^T) V, materialised, in float64.

    Parameters
    ----------
    q : array [..., M, D]
    k : array [..., N, D]
    v : array [..., N, Dv]
        Any leading batch/head dimensions, identical for q, k and v.
    scale : float
        Multiplies Q K^T before the softmax.
    causal : bool
        Top-left causal mask (query i sees keys j <= i).

    Returns
    -------
    (O [..., M, Dv] float64, LSE [..., M] float64, natural log)
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    lead = q.shape[:-2]
    if k.shape[:-2] != lead or v.shape[:-2] != lead:
        raise ValueError("q, k and v must share their leading dimensions")
    if k.shape[-2] != v.shape[-2]:
        raise ValueError("k and v must have the same number of rows")
    if q.shape[-1] != k.shape[-1]:
        raise ValueError("q and k must have the same width")
    m_rows = q.shape[-2]
    heads = int(np.prod(lead, dtype=np.int64))
    qf = q.reshape((heads,) + q.shape[-2:])
    kf = k.reshape((heads,) + k.shape[-2:])
    vf = v.reshape((heads,) + v.shape[-2:])
    o = np.empty((qf.shape[0], m_rows, v.shape[-1]), dtype=np.float64)
    lse = np.empty((qf.shape[0], m_rows), dtype=np.float64)
    rows = np.arange(m_rows)
    for h in range(qf.shape[0]):
        o[h], lse[h] = _one_head(qf[h], kf[h], vf[h], scale, causal, rows)
    return o.reshape(lead + o.shape[-2:]), lse.reshape(lead + (m_rows,))


def attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                   causal: bool, rows) -> tuple[np.ndarray, np.ndarray]:
    """O and LSE for the selected query rows of ONE head, in float64.

    ``q`` is [M, D] (only rows ``rows`` are read), ``k`` and ``v`` are
    [N, D]. Row indices keep their meaning in the causal mask, so row i sees
    keys 0..i. Returns (O [len(rows), D], LSE [len(rows)]).
    """
    rows = np.asarray(rows, dtype=np.int64)
    return _one_head(q, k, v, scale, causal, rows)


def flop_count(B: int, H: int, M: int, N: int, D: int, causal: bool) -> float:
    """Matmul FLOPs of the forward pass, the metric's convention.

    Two matmuls (QK^T and PV) of 2*M*N*D each, per head ("Module 08", Code
    Step 4, which counts 2*N*N*d + 2*N*N*d for the standard pass); causal
    attention is counted as half of that.
    """
    f = 4.0 * B * H * M * N * D
    return f * 0.5 if causal else f
