"""Gradients of materialised attention in float64: the parity oracle for
fa_bwd.

TEST INFRASTRUCTURE ONLY (see the package docstring): the CUDA path never
imports this module.

What is computed
----------------
"Module 08: FlashAttention and Memory-Efficient Kernels", section "The
backward pass: recompute instead of store", and its Code Step 6: the backward
pass needs P; instead of keeping it, it rebuilds P from Q, K and the one
number per row kept by the forward pass, L = m + log(l), as P = exp(S - L).
The same page's Practice 3 counts the work: the standard backward has four
N x N x d matrix products and FlashAttention's recomputes Q K^T once more.

The pages give no formula for the gradients themselves; they are the plain
derivative of O = P V with P = softmax(S), S = scale * Q K^T (causal scores
above the diagonal masked), for a loss whose gradient with respect to O is
dO. For every (batch, head), in float64 on the inputs exactly as given:

1. S  = scale * Q K^T, causal mask with -inf (as the forward oracle)
2. P  = exp(S - L)              with L the forward's log-sum-exp (rebuilt here)
3. dV = P^T dO                  (N x D)
4. dP = dO V^T                  (M x N)
5. Dl_i = sum_j P_ij dP_ij      (= sum_d dO_id O_id, O = P V)
6. dS = P * (dP - Dl)           (the softmax Jacobian applied row by row)
7. dQ = scale * dS K,  dK = scale * dS^T Q

A row with no visible key has P = 0 and contributes nothing.
"""

from __future__ import annotations

import numpy as np

from .attention import attention

__all__ = ["attention_bwd", "bwd_flop_count"]


def attention_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray, scale: float,
                  causal: bool = False) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """dQ, dK, dV of softmax(scale * Q K^T) V for the output gradient ``do``.

    q, do : [..., M, D];  k, v : [..., N, D]; any identical leading dims.
    Returns float64 arrays shaped like q, k and v.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lead = q.shape[:-2]
    M, D = q.shape[-2:]
    N = k.shape[-2]
    if k.shape[:-2] != lead or v.shape[:-2] != lead or do.shape != q.shape[:-1] + (v.shape[-1],):
        raise ValueError("shapes of q, k, v and do do not match")
    _, lse = attention(q, k, v, scale, causal)               # step 2's L, from the forward definition
    heads = int(np.prod(lead, dtype=np.int64))
    qf, kf, vf = (x.reshape((heads,) + x.shape[-2:]) for x in (q, k, v))
    dof = do.reshape((heads,) + do.shape[-2:])
    lf = lse.reshape(heads, M)
    dq = np.zeros_like(qf)
    dk = np.zeros_like(kf)
    dv = np.zeros_like(vf)
    for h in range(heads):
        s = scale * (qf[h] @ kf[h].T)
        if causal:
            s = np.where(np.arange(N)[None, :] > np.arange(M)[:, None], -np.inf, s)
        with np.errstate(invalid="ignore"):
            p = np.exp(s - lf[h][:, None])                     # step 2
        p = np.where(np.isfinite(lf[h])[:, None], p, 0.0)      # rows without keys: P = 0
        dv[h] = p.T @ dof[h]                                   # step 3
        dp = dof[h] @ vf[h].T                                  # step 4
        dl = np.sum(p * dp, axis=1, keepdims=True)             # step 5
        ds = p * (dp - dl)                                     # step 6
        dq[h] = scale * (ds @ kf[h])                           # step 7
        dk[h] = scale * (ds.T @ qf[h])
    return dq.reshape(q.shape), dk.reshape(k.shape), dv.reshape(v.shape)


def bwd_flop_count(B: int, H: int, M: int, N: int, D: int, causal: bool) -> float:
    """Matmul FLOPs of the recomputing backward pass: five M x N x D
    products of 2*M*N*D each per head (Practice 3: the standard backward's
    four plus the recomputed Q K^T); causal counted as half."""
    f = 10.0 * B * H * M * N * D
    return f * 0.5 if causal else f
