"""Seeded synthetic inputs for fa_fwd: the one module the kernels' callers and
the oracle's tests share.

It holds no attention arithmetic, only random draws and the bf16 storage
format. Every tensor is drawn per (batch, head) from its own numpy PCG64
stream, seeded by ``SeedSequence([workload_id, tensor_id, bh])`` with
tensor_id 0 for Q, 1 for K and 2 for V, as float32 ``standard_normal`` times
the workload's sigma; bf16 workloads then round each value to bf16
(round-to-nearest-even). Drawing per head lets a test regenerate any single
head without the others (the 64K-token workload's sampled rows).

The workloads are the five shapes the attention pages motivate: the
single-head fp32 problem of "FlashAttention in Triton: A Tile-by-Tile
Walkthrough", the GPT-2-medium attention shape quoted in "Module 08:
FlashAttention and Memory-Efficient Kernels" (section "What FlashAttention
changes"), a causal 4K-token shape, a ragged cross-attention shape with
peaked logits and a 64K-token causal shape.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = ["Workload", "WORKLOADS", "head_tensor", "make_inputs",
           "round_to_bf16", "bf16_bits", "sample_rows"]


@dataclass(frozen=True)
class Workload:
    name: str
    wid: int            # seed component
    B: int
    H: int
    M: int              # query rows per head
    N: int              # key/value rows per head
    D: int              # head dimension
    dtype: str          # "f32" or "bf16"
    causal: bool
    sigma_qk: float = 1.0
    sigma_v: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        f = 4.0 * self.B * self.H * self.M * self.N * self.D
        return f * 0.5 if self.causal else f

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "M": self.M,
                "N": self.N, "D": self.D, "causal": self.causal,
                "dtype": self.dtype, "sigma_qk": self.sigma_qk,
                "sigma_v": self.sigma_v, "scale": self.scale}


WORKLOADS = {w.name: w for w in [
    Workload("f32_single_head_m256_n512_d64", 1, 1, 1, 256, 512, 64, "f32", False),
    Workload("gpt2m_b64_h16_s1024_d64", 2, 64, 16, 1024, 1024, 64, "bf16", False),
    Workload("causal_b8_h32_s4096_d128", 3, 8, 32, 4096, 4096, 128, "bf16", True),
    Workload("cross_b2_h8_m1000_n3000_d96_peaked", 4, 2, 8, 1000, 3000, 96,
             "bf16", False, sigma_qk=3.0),
    Workload("long_causal_b1_h8_s65536_d64", 5, 1, 8, 65536, 65536, 64, "bf16", True),
    # The GPT-2-medium and causal 4K shapes in fp32, for the fp32 paths.
    Workload("f32_gpt2m_b64_h16_s1024_d64", 6, 64, 16, 1024, 1024, 64, "f32", False),
    Workload("f32_causal_b8_h32_s4096_d128", 7, 8, 32, 4096, 4096, 128, "f32", True),
]}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 out."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).copy()
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    u &= np.uint32(0xFFFF0000)
    return u.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of float32 values that are bf16-exact."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> np.uint32(16)).astype(np.uint16)


def head_tensor(wid: int, tensor_id: int, bh: int, rows: int, D: int,
                sigma: float, dtype: str) -> np.ndarray:
    """One head's [rows, D] tensor, float32 (bf16-exact when dtype is bf16)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([wid, tensor_id, bh])))
    x = rng.standard_normal((rows, D), dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return round_to_bf16(x) if dtype == "bf16" else x


def make_inputs(w: Workload, heads=None):
    """Q [B,H,M,D], K and V [B,H,N,D] as float32 arrays for workload ``w``.

    With ``heads`` (a list of flat b*H+h indices) only those heads are drawn
    and the arrays are [len(heads), rows, D].
    """
    bhs = range(w.B * w.H) if heads is None else list(heads)
    n = len(bhs)
    q = np.empty((n, w.M, w.D), dtype=np.float32)
    k = np.empty((n, w.N, w.D), dtype=np.float32)
    v = np.empty((n, w.N, w.D), dtype=np.float32)
    for i, bh in enumerate(bhs):
        q[i] = head_tensor(w.wid, 0, bh, w.M, w.D, w.sigma_qk, w.dtype)
        k[i] = head_tensor(w.wid, 1, bh, w.N, w.D, w.sigma_qk, w.dtype)
        v[i] = head_tensor(w.wid, 2, bh, w.N, w.D, w.sigma_v, w.dtype)
    if heads is None:
        q = q.reshape(w.B, w.H, w.M, w.D)
        k = k.reshape(w.B, w.H, w.N, w.D)
        v = v.reshape(w.B, w.H, w.N, w.D)
    return q, k, v


def sample_rows(wid: int, bh: int, M: int, count: int = 256) -> np.ndarray:
    """Sorted distinct query rows to check on a head too large to materialise.

    Always includes rows 0, 1, 127, 128 and M-1 (tile edges and the causal
    diagonal's first tiles); the rest are drawn from the head's own stream.
    """
    fixed = {r for r in (0, 1, 127, 128, M - 1) if 0 <= r < M}
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([wid, 99, bh])))
    extra = rng.choice(M, size=min(count, M), replace=False)
    rows = list(fixed)
    for r in extra:
        if len(rows) >= min(count, M):
            break
        if int(r) not in fixed:
            rows.append(int(r))
    return np.array(sorted(rows), dtype=np.int64)
