"""The memory-traffic model (flashattention_fa_fwd_gb300.traffic) on the CPU.

Counted traffic (the loops walked step by step) must equal each closed form
exactly, and both must reproduce the table of "Module 08: FlashAttention and
Memory-Efficient Kernels", Code Step 5, within half a unit of its last printed
digit. The kernel-schedule model is checked against sums worked out by hand.
"""

import json
import math
import os

import pytest

from flashattention_fa_fwd_gb300 import traffic as T

MIB = 2 ** 20


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "traffic_step5.json")) as f:
        return json.load(f)


def test_block_sizes_match_pages(golden_dir):
    g = _golden(golden_dir)
    assert T.block_sizes(g["sram_elems"], g["d"]) == (g["Br"], g["Bc"])
    for row in g["budget_sweep"]:
        assert T.block_sizes(row["sram_elems"], g["d"])[1] == row["Bc"]


def test_step5_table(golden_dir):
    g = _golden(golden_dir)
    d, bc, br = g["d"], g["Bc"], g["Br"]
    for row in g["table"]:
        n = row["N"]
        std = T.standard_traffic(n, d)
        tiled = T.alg1_count(n, d, br, bc).total
        assert abs(std * 2 / MIB - row["standard_mib"]) <= 0.05 + 1e-9
        assert abs(tiled * 2 / MIB - row["tiled_mib"]) <= 0.05 + 1e-9
        assert abs(std / tiled - row["ratio"]) <= 0.05 + 1e-9
    growth = T.alg1_traffic(8192, d, bc) / T.alg1_traffic(4096, d, bc)
    assert abs(growth - g["growth_4096_to_8192"]) <= 0.005 + 1e-9


def test_step5_budget_sweep(golden_dir):
    g = _golden(golden_dir)
    for row in g["budget_sweep"]:
        _, bc = T.block_sizes(row["sram_elems"], g["d"])
        mib = T.alg1_traffic(g["budget_sweep_N"], g["d"], bc) * 2 / MIB
        assert abs(mib - row["tiled_mib"]) <= 0.05 + 1e-9


@pytest.mark.parametrize("n", [1, 7, 64, 100, 196, 197, 511, 1000])
@pytest.mark.parametrize("d,br,bc", [(64, 64, 196), (16, 5, 9), (32, 32, 32), (8, 3, 50)])
def test_alg1_counted_equals_closed_form(n, d, br, bc):
    assert T.alg1_count(n, d, br, bc).total == T.alg1_traffic(n, d, bc)


@pytest.mark.parametrize("n,d", [(1, 1), (5, 3), (512, 64), (1000, 96)])
def test_standard_counted_equals_closed_form(n, d):
    assert T.standard_count(n, d) == T.standard_traffic(n, d)


@pytest.mark.parametrize("m,n", [(1, 1), (64, 64), (100, 333), (513, 200)])
@pytest.mark.parametrize("d,br,bc", [(64, 64, 128), (16, 7, 5)])
def test_fa2_counted_equals_closed_form(m, n, d, br, bc):
    assert T.fa2_count(m, n, d, br, bc).total == T.fa2_traffic(m, n, d, br)
    assert T.fa2_count(m, n, d, br, bc, lse=False).total == T.fa2_traffic(m, n, d, br, lse=False)


def _causal_keys_brute(m, n, br, bc):
    """K/V rows the swapped order reads under top-left causal masking, from
    per-row visibility: a Q block needs every K/V block holding a key <= its
    last row."""
    rows = 0
    for i0 in range(0, m, br):
        last = min(i0 + br, m) - 1
        need = [j0 for j0 in range(0, n, bc) if any(j0 + k <= last for k in range(min(bc, n - j0)))]
        rows += sum(min(bc, n - j0) for j0 in need)
    return rows


@pytest.mark.parametrize("m,n,br,bc", [(10, 10, 3, 4), (37, 37, 8, 5), (64, 100, 16, 16), (100, 40, 7, 9)])
def test_fa2_causal_counts_visible_blocks(m, n, br, bc):
    d = 4
    c = T.fa2_count(m, n, d, br, bc, causal=True)
    q_and_o = 2 * m * d + m
    assert c.total - q_and_o == 2 * d * _causal_keys_brute(m, n, br, bc)
    assert c.total <= T.fa2_count(m, n, d, br, bc).total


@pytest.mark.parametrize("n,br,bc", [(50, 8, 8), (300, 64, 196), (257, 16, 40)])
def test_alg1_causal_skips_tiles_above_the_diagonal(n, br, bc):
    d = 8
    full = T.alg1_count(n, d, br, bc)
    causal = T.alg1_count(n, d, br, bc, causal=True)
    assert causal.total < full.total
    # A (K/V block, Q block) step is kept when the block holds a visible key:
    # j0 <= the Q block's last row. Each kept step moves Q_i, O_i in and O_i
    # out (3 br d) plus l_i, m_i in and out (4 br); K and V are read once.
    kept = [(j0, i0) for j0 in range(0, n, bc) for i0 in range(0, n, br) if j0 <= i0 + br - 1]
    assert 0 < len(kept) < math.ceil(n / bc) * math.ceil(n / br)
    inner = sum(3 * min(br, n - i0) * d + 4 * min(br, n - i0) for _, i0 in kept)
    assert causal.total == 2 * n * d + inner


def test_kernel_model_noncausal():
    b, h, m, n, d = 2, 3, 1000, 777, 64
    k = T.kernel_traffic(b, h, m, n, d, causal=False)
    units = math.ceil(m / 256)
    assert k.key_tiles_loaded == b * h * units * math.ceil(n / 128)
    assert k.hbm_min_bytes == b * h * (m * d * 2 * 2 + 2 * n * d * 2 + m * 4)
    assert k.l2_to_sm_bytes == b * h * (m * d * 2 + units * 2 * n * d * 2)


def test_kernel_model_causal_square():
    # S = 4096: 16 units per head; unit p (rows 256p .. 256p + 255) loads
    # 2p + 2 key tiles, 272 per head in all.
    b, h, s, d = 2, 32, 4096, 128
    k = T.kernel_traffic(b, h, s, s, d, causal=True)
    assert k.key_tiles_loaded == b * h * sum(2 * p + 2 for p in range(16))
    assert k.l2_to_sm_bytes == b * h * (s * d * 2 + 272 * 2 * 128 * d * 2)
    assert k.written_bytes == b * h * s * (d * 2 + 4)


def test_orders_compared_at_the_pages_budget():
    # Same blocks (Br = 64, Bc = 196, d = 64): Algorithm 1 re-reads Q, O, l, m
    # once per K/V block; the swapped order re-reads K, V once per Q block.
    # With Br = d < Bc there are more Q blocks than K/V blocks, and the
    # swapped order moves more elements; with equal blocks it moves fewer.
    n, d = 4096, 64
    assert T.fa2_count(n, n, d, 64, 196).total > T.alg1_count(n, d, 64, 196).total
    assert T.fa2_count(n, n, d, 196, 196).total < T.alg1_count(n, d, 196, 196).total
