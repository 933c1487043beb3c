"""Memory-traffic model of the attention forward pass (CPU only, no GPU).

Counts the elements (or bytes) that move between HBM and the chip for three
loop orders, each twice: once by walking the loops and adding up what every
step reads and writes ("counted"), once in closed form. The two must agree
exactly; the tests also hold them to the table the pages print.

* Standard attention: the three-kernel forward of "Module 08: FlashAttention
  and Memory-Efficient Kernels", Code Step 5 ("count HBM traffic"): read Q, K;
  write S; read S; write P; read P, V; write O, i.e. 4Nd + 4N^2 elements.
* Algorithm 1 of the FlashAttention paper, as the same page's Code Step 1
  tiles it: K/V blocks of Bc rows in the outer loop, Q blocks of Br rows in
  the inner loop, with O, l and m read from and written back to HBM at every
  inner step. Closed form (Code Step 5): 2Nd + Tc (3Nd + 4N), Tc = ceil(N/Bc).
  Block sizes from an on-chip budget of M elements: Bc = ceil(M / 4d),
  Br = min(Bc, d) (Code Step 1, block_sizes).
* The swapped order of the same page's "Project" (FlashAttention-2): Q blocks
  outside, K/V blocks inside, O and the running (m, l) kept on chip and O
  divided once at the end. Each Q block reads all K/V rows it can see once;
  Q is read and O written once: 2Md + 2 Tr N d for M = N, Tr = ceil(M/Br)
  (+ M for the log-sum-exp this library also writes).

``kernel_traffic`` applies the last order to this library's own bf16 kernel
schedule (units of two 128-row query tiles that share each 128-key K/V tile
load; causal units stop at the diagonal), giving the bytes the kernel moves
from L2 into the SMs and the bytes it must move to and from HBM at least (Q,
K, V read once, O and LSE written once), the figure the roofline's DRAM
counters are compared with.

A causal tile is skipped when it lies entirely above the diagonal (top-left
alignment: key j visible to query i iff j <= i), as in Code Step 1.
"""

from __future__ import annotations

import math
from dataclasses import dataclass


def block_sizes(sram_elems: int, d: int) -> tuple[int, int]:
    """(Br, Bc) for an on-chip budget of ``sram_elems`` elements: Bc = ceil(M/4d), Br = min(Bc, d)."""
    if sram_elems <= 0 or d <= 0:
        raise ValueError("block_sizes needs a positive budget and head dimension")
    bc = -(-sram_elems // (4 * d))
    return min(bc, d), bc


# ------------------------------------------------------------ standard
def standard_traffic(n: int, d: int) -> int:
    """Elements the three-kernel forward moves: 4Nd + 4N^2 (closed form)."""
    return 4 * n * d + 4 * n * n


def standard_count(n: int, d: int) -> int:
    """The same, step by step: kernel 1 reads Q and K and writes S; kernel 2
    reads S and writes P; kernel 3 reads P and V and writes O."""
    k1 = (n * d) + (n * d) + (n * n)
    k2 = (n * n) + (n * n)
    k3 = (n * n) + (n * d) + (n * d)
    return k1 + k2 + k3


# --------------------------------------------------------- Algorithm 1
@dataclass
class Counts:
    reads: int = 0
    writes: int = 0

    @property
    def total(self) -> int:
        return self.reads + self.writes


def alg1_traffic(n: int, d: int, bc: int) -> int:
    """Closed form for Algorithm 1 (non-causal): 2Nd + Tc (3Nd + 4N)."""
    tc = math.ceil(n / bc)
    return 2 * n * d + tc * (3 * n * d + 4 * n)


def alg1_count(n: int, d: int, br: int, bc: int, causal: bool = False) -> Counts:
    """Walks Algorithm 1's loops and counts elements moved.

    Outer step j (a K/V block of bc_j rows) reads K_j and V_j. Each inner step
    i that is not skipped reads Q_i and O_i (br_i x d each) and l_i, m_i
    (br_i each), and writes O_i, l_i and m_i back.
    """
    c = Counts()
    for j0 in range(0, n, bc):
        bcj = min(bc, n - j0)
        c.reads += 2 * bcj * d
        for i0 in range(0, n, br):
            bri = min(br, n - i0)
            if causal and j0 > i0 + br - 1:
                continue
            c.reads += 2 * bri * d + 2 * bri
            c.writes += bri * d + 2 * bri
    return c


# ------------------------------------------------ FlashAttention-2 order
def fa2_traffic(m: int, n: int, d: int, br: int, lse: bool = True) -> int:
    """Closed form for the swapped order (non-causal): Q read and O written
    once, K and V read once per Q block: 2Md + 2 Tr N d (+ M for LSE)."""
    tr = math.ceil(m / br)
    return 2 * m * d + 2 * tr * n * d + (m if lse else 0)


def fa2_count(m: int, n: int, d: int, br: int, bc: int, causal: bool = False, lse: bool = True) -> Counts:
    """Walks the swapped loops: per Q block, read Q_i, then every K/V block it
    can see (whole blocks of bc rows, stopping after the one holding its last
    row's diagonal when causal), then write O_i (and its LSE)."""
    c = Counts()
    for i0 in range(0, m, br):
        bri = min(br, m - i0)
        c.reads += bri * d
        for j0 in range(0, n, bc):
            if causal and j0 > i0 + bri - 1:
                break
            c.reads += 2 * min(bc, n - j0) * d
        c.writes += bri * d + (bri if lse else 0)
    return c


# ------------------------------------------------- this library's kernel
@dataclass
class KernelTraffic:
    l2_to_sm_bytes: int       # Q once per unit + every K/V tile a unit loads
    hbm_min_bytes: int        # Q, K, V read once; O and LSE written once
    written_bytes: int        # O and LSE
    key_tiles_loaded: int     # K/V tile loads over all units


def kernel_traffic(b: int, h: int, m: int, n: int, d: int, causal: bool, elem_bytes: int = 2,
                   tile: int = 128, tiles_per_unit: int = 2) -> KernelTraffic:
    """Bytes of the bf16 forward kernel's schedule for one launch.

    A unit is ``tiles_per_unit`` query tiles of ``tile`` rows of one head; it
    loads each K/V tile once for all its query tiles, as many tiles as its
    longest query tile visits (all ceil(N/tile) when not causal; up to and
    including the diagonal tile when causal). Rows past N or M are
    zero-filled by the copy engine and move no memory.
    """
    nkv = math.ceil(n / tile) if n > 0 else 0
    tiles_loaded = 0
    kv_rows = 0
    for q0 in range(0, m, tile * tiles_per_unit):
        nmax = 0
        for t in range(tiles_per_unit):
            qt = q0 + t * tile
            if qt >= m:
                continue
            nt = min(nkv, qt // tile + 1) if causal else nkv
            nmax = max(nmax, nt)
        tiles_loaded += nmax
        kv_rows += min(n, nmax * tile)
    heads = b * h
    q_bytes = heads * m * d * elem_bytes
    o_bytes = heads * m * d * elem_bytes
    lse_bytes = heads * m * 4
    l2_to_sm = q_bytes + heads * 2 * kv_rows * d * elem_bytes
    hbm_min = q_bytes + 2 * heads * n * d * elem_bytes + o_bytes + lse_bytes
    return KernelTraffic(l2_to_sm_bytes=l2_to_sm, hbm_min_bytes=hbm_min, written_bytes=o_bytes + lse_bytes,
                         key_tiles_loaded=heads * tiles_loaded)
