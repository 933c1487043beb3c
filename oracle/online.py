"""Model of the streaming (online) softmax recurrence, with plantable mistakes.

TEST INFRASTRUCTURE ONLY (see the package docstring). This is NOT the parity
oracle -- ``oracle.attention`` is. It models, in float64 and in the pages'
own notation, the per-row recurrence that a FlashAttention kernel runs over
tiles of keys, so that tests can show two things on the CPU:

* with every switch at its default the recurrence reaches the plain
  definition (up to rounding), and
* each mistake the pages warn about is caught by the same comparison the GPU
  parity tests make, and only under the conditions the pages say it shows.

The recurrence (keys visited one tile at a time; m = -inf, l = 0, acc = 0
at the start), from "FlashAttention-style kernel" section "The loop",
"Module 08: FlashAttention and Memory-Efficient Kernels" section "Tiling and
the online softmax", and "FlashAttention in Triton: A Tile-by-Tile
Walkthrough" section "How can softmax work a tile at a time?":

    m_new = max(m, max(s))            s: the tile's scaled scores
    alpha = exp(m - m_new)            rescales what was accumulated so far
    p     = exp(s - m_new)
    l     = l * alpha + sum(p)
    acc   = acc * alpha + p @ V_tile
    m     = m_new
    out   = acc / l                   once, after the last tile

Switches (each plants one mistake named on the pages):

``rescale_acc=False``
    drops acc * alpha ("FlashAttention-style kernel", "Things that break":
    right while the keys fit in one tile, wrong beyond it).
``rescale_l=False``
    drops l * alpha (the deliberate mutant of "Module 08" Code Step 3).
``base2=True, alpha_base_e=True``
    a base-two kernel (scores pre-multiplied by log2 e, exp2 everywhere)
    whose alpha is computed with base e ("Things that break": a smooth
    wrong factor).
``reverse=True``
    visits the key tiles last-to-first ("Module 08", Practice 2).
``guard=False``
    subtracts an infinite running max as is, so a tile row with no visible
    key gives exp(-inf - (-inf)) = NaN ("Module 08", Code Step 3 and
    "Common mistakes"). With ``guard=True`` an infinite max is clamped to 0
    before it is subtracted.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = ["online_softmax_trace", "online_attention_row", "online_attention"]

_LOG2E = 1.0 / math.log(2.0)


def online_softmax_trace(x, chunk: int, rescale_l: bool = True):
    """Online softmax of one row ``x`` seen ``chunk`` entries at a time.

    Returns ``(trace, probs)``: ``trace`` lists (m, l) after every chunk and
    ``probs`` is exp(x - m) / l with the final m and l ("Module 08", Code
    Step 3).
    """
    x = np.asarray(x, dtype=np.float64)
    m, l = -np.inf, 0.0
    trace = []
    for start in range(0, x.size, chunk):
        c = x[start:start + chunk]
        m_new = max(m, float(c.max()))
        if rescale_l:
            l = l * math.exp(m - m_new) + float(np.exp(c - m_new).sum())
        else:
            l = l + float(np.exp(c - m_new).sum())
        m = m_new
        trace.append((m, l))
    return trace, np.exp(x - m) / l


def online_attention_row(s, v, block: int, rescale_acc: bool = True):
    """Recurrence for one query row with already-scaled scores ``s`` [N] and
    values ``v`` [N, Dv]; keys are taken ``block`` at a time.

    Returns ``(out, l, acc, m)`` with the final running state, as in the
    worked example of "FlashAttention in Triton: A Tile-by-Tile Walkthrough"
    (scores [1, 2, 3], values [10, 20, 30], blocks of two and one).
    """
    s = np.asarray(s, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64).reshape(s.size, -1)
    m, l = -np.inf, 0.0
    acc = np.zeros(v.shape[1])
    for start in range(0, s.size, block):
        c = s[start:start + block]
        m_new = max(m, float(c.max()))
        alpha = math.exp(m - m_new)
        p = np.exp(c - m_new)
        l = l * alpha + float(p.sum())
        acc = (acc * alpha if rescale_acc else acc) + p @ v[start:start + block]
        m = m_new
    return acc / l, l, acc, m


def online_attention(q, k, v, scale: float, causal: bool = False,
                     block: int = 128, *, rescale_acc: bool = True,
                     rescale_l: bool = True, base2: bool = False,
                     alpha_base_e: bool = False, reverse: bool = False,
                     guard: bool = True):
    """Tiled recurrence over key tiles for one head, all rows at once.

    ``q`` [M, D], ``k`` and ``v`` [N, D]. Returns (O [M, Dv], LSE [M]) in
    float64; LSE = m + ln l in natural-log units whichever base is used.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_rows, n_keys = q.shape[0], k.shape[0]
    rows = np.arange(n_rows)[:, None]
    c = scale * _LOG2E if base2 else scale
    expf = np.exp2 if base2 else np.exp

    m = np.full(n_rows, -np.inf)
    l = np.zeros(n_rows)
    acc = np.zeros((n_rows, v.shape[1]))
    starts = list(range(0, n_keys, block))
    if reverse:
        starts = starts[::-1]
    with np.errstate(invalid="ignore"):
        for j in starts:
            kj, vj = k[j:j + block], v[j:j + block]
            s = c * (q @ kj.T)
            if causal:
                cols = np.arange(j, j + kj.shape[0])[None, :]
                s = np.where(cols <= rows, s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            m_sub = np.where(np.isfinite(m_new), m_new, 0.0) if guard else m_new
            if base2 and alpha_base_e:
                alpha = np.exp(m - m_sub)
            else:
                alpha = expf(m - m_sub)
            p = expf(s - m_sub[:, None])
            l = (l * alpha if rescale_l else l) + p.sum(axis=1)
            acc = (acc * alpha[:, None] if rescale_acc else acc) + p @ vj
            m = m_new
        out = acc / l[:, None]
        log_l = np.log2(l) if base2 else np.log(l)
        lse = (m + log_l) * (math.log(2.0) if base2 else 1.0)
    return out, lse
