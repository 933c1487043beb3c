// bf16 FlashAttention forward for sm_103a: TMA-fed shared-memory tiles,
// tcgen05 MMAs with fp32 accumulators in tensor memory, warp-specialised
// load / MMA / softmax / epilogue roles, persistent CTAs.
//
// Algorithm ("FlashAttention-style kernel", section "The loop"; "Module 08:
// FlashAttention and Memory-Efficient Kernels", sections "Tiling and the
// online softmax" and "Related ideas"): a query tile stays resident while
// key/value tiles stream past it; per row the kernel carries the running
// max m, the running sum l and the unnormalised output acc, rescales l and
// acc by alpha = exp2(m_old - m_new) when the max grows (see "Running max"
// below), and divides by l once at the end. log2(e) is folded into the score
// scale so that each score costs one FMA and one base-two exponential. The per-row log-sum-exp
// m + log(l) is written next to O ("Module 08", section "The backward pass").
//
// Work unit: one (batch*head, pair of 128-row query tiles), or one query
// tile when every tile of the problem fits on its own SM (Bf16Params::single;
// tile 1 then stays idle). Each CTA is
// persistent (one per SM) and claims units one at a time from a global
// counter, in an order that puts the longest causal units of a group of
// heads first (unit_info), so that CTAs finish within one short unit of each
// other. The CTA's TMA thread claims each unit and passes its index to the
// other roles through a small ring in shared memory (UNIT_FULL / UNIT_EMPTY).
// The two query tiles t = 0, 1 of a unit are processed in ping-pong: while
// the softmax of one tile runs, the tensor core works on the other tile.
//
// Roles (512 threads, 4 warpgroups; registers re-split with setmaxnreg):
//   WG0 (warps 0-3)   softmax of query tile 0   (thread = row = TMEM lane)
//   WG1 (warps 4-7)   softmax of query tile 1
//   WG2 (warps 8-11)  epilogue (O / l, LSE) of the previous unit while the
//                     next one runs
//   WG3 (warps 12-15) warp 12: TMA producer; warp 13: tensor-memory owner
//                     and MMA issuer; warp 14: K/V gate (waits for K/V
//                     tiles in the MMA thread's place); warp 15 idle
//
// Tensor memory (512 columns, 128 lanes, lane = query row of the tile):
//   [  0,128)  S_0 (fp32 scores of tile 0); P_0 (bf16, packed in pairs)
//              overwrites its first 64 columns after softmax
//   [128,256)  S_1 / P_1
//   [256,256+D) O_0 accumulator      [384,384+D) O_1 accumulator
//
// Per key/value tile j the MMA warp issues, in this order:
//   O_0 += P_0(j-1) V(j-1);  S_0 = Q_0 K(j)^T;  O_1 += P_1(j-1) V(j-1);
//   S_1 = Q_1 K(j)^T
// tcgen05 MMAs from one thread execute in issue order, so S_t(j) only
// overwrites P_t(j-1) after the product that reads it, and the commit that
// announces S_t(j) also guarantees that O_t holds every earlier product
// (which is what lets the softmax rescale O_t before P_t(j) V(j)).
//
// Running max: a row's reference m (shared by l and acc) moves only when a
// tile raises the row max by more than 2^8; then alpha = exp2(m_old - m_new)
// rescales l and acc, as in the pages' recurrence. Below that the stale
// reference is exact for O = acc / l and LSE = m + log l; the one bf16
// effect it has -- the tile's largest weight can exceed 1 and is rounded
// when it enters P V -- is compensated by normalising O with l_o, which
// counts each tile's largest weight as rounded.
//
// Hand-offs (mbarriers): S_FULL (MMA -> softmax of tile 0), ITER (one MMA
// commit per key tile step: announces S_1 to the softmax of tile 1 and frees
// the step's K/V stages for the producer), P_FULL (softmax -> MMA; for tile 0
// also the gate's "V(j-1) and K(j) have landed"), per unit ST_FULL /
// ST_EMPTY (softmax <-> epilogue: m, l, l_o), O_DONE (MMA -> epilogue),
// O_FREE (epilogue -> MMA: O_t may be overwritten by the next unit), Q_FULL /
// Q_EMPTY and KV_FULL (TMA), UNIT_FULL / UNIT_EMPTY (the ring of claimed unit
// indices). While the tensor core streams its operands from shared memory,
// every mbarrier poll or commit of the MMA thread takes 100-160 cycles, during
// which the tensor pipe (about three MMAs deep) runs dry; the thread
// therefore makes only four such calls per step in the steady state (two P
// waits, the S_0 commit and the step's ITER commit), none back to back.
//
// Causal (top-left, key j visible to query i when j <= i): key tiles wholly
// above the diagonal are never loaded or multiplied; the diagonal tile and a
// ragged last key tile are masked with -inf in registers ("FlashAttention-
// style kernel", section "Causal masking"). A row whose running max is still
// -inf uses 0 in its place so that exp2(-inf - -inf) never forms ("Module
// 08", "Common mistakes"). Query rows >= M and key rows >= N are zero-filled
// by TMA, and their scores masked or their outputs not stored.
//
// Every wait is bounded (see ptx.cuh): on a time-out the kernel sets the
// device status word, all roles leave their loops, in-flight copies and
// MMAs are drained, and tensor memory is freed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

template <int D>
struct Bf16Cfg {
    static_assert(D == 64 || D == 96 || D == 128, "head dimension");
    static constexpr int BM = 128;                     // query rows per tile
    static constexpr int BN = 128;                     // key rows per tile
    static constexpr int PANELS = (D + 63) / 64;       // 64-column swizzle panels
    static constexpr int PANEL_BYTES = 128 * 128;      // 128 rows x 128 B
    static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
    static constexpr int QB = (D <= 64) ? 2 : 1;       // Q buffers (units in flight)
    static constexpr int NS = (D <= 64) ? 8 : 4;       // K/V ring stages
    static constexpr int THREADS = 512;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL0 = 256, O_COL1 = 384;
    static constexpr int QK_STEPS = D / 16;            // MMA K-steps of Q K^T
    static constexpr int PV_STEPS = BN / 16;           // MMA K-steps of P V
    // shared memory layout (offsets from a 1024-byte aligned base)
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = Q_OFF + QB * 2 * TILE_BYTES;
    static constexpr int STATS_OFF = KV_OFF + NS * TILE_BYTES;      // float [2 t][3 (m, l, l_o)][128]
    static constexpr int BAR_OFF = STATS_OFF + 2 * 3 * 128 * 4;
    // barrier slots
    // ITER: ring of per-iteration completion barriers (one MMA commit per key
    // tile step); it releases K/V stages and announces S_1.
    static constexpr int ITERS = 8;
    static constexpr int KV_FULL = 0, ITER = NS, Q_FULL = NS + ITERS, Q_EMPTY = Q_FULL + QB;
    static constexpr int S_FULL = Q_EMPTY + QB;                     // S_0 only
    static constexpr int P_FULL = S_FULL + 1, O_DONE = P_FULL + 2;
    static constexpr int O_FREE = O_DONE + 2, ST_FULL = O_FREE + 2, ST_EMPTY = ST_FULL + 2;
    static constexpr int DRAIN = ST_EMPTY + 2;
    static constexpr int UNIT_SLOTS = 4;                            // ring of claimed unit indices
    static constexpr int UNIT_FULL = DRAIN + 1, UNIT_EMPTY = UNIT_FULL + UNIT_SLOTS;
    // Readers of a ring slot: the MMA thread, one lane of each of the four
    // warps of both softmax warpgroups and of the epilogue warpgroup, and the
    // K/V gate thread.
    static constexpr int UNIT_READERS = 1 + 3 * 4 + 1;
    static constexpr int NUM_BARS = UNIT_EMPTY + UNIT_SLOTS;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;         // tensor-memory base, abort flag
    static constexpr int RING_OFF = MISC_OFF + 16;                  // int [UNIT_SLOTS]
    static constexpr int SMEM_USED = RING_OFF + UNIT_SLOTS * 4;
    // + slack to align the base up to 1024 B (the 128-byte swizzle atom).
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Register split per warpgroup (setmaxnreg); sums to 512 x 128, the launch's
// registers, and to 512 per SM sub-partition (one warp of each group).
constexpr int kRegsSoftmax = 176, kRegsEpilogue = 64, kRegsLoadMma = 96;
static_assert(2 * kRegsSoftmax + kRegsEpilogue + kRegsLoadMma == 4 * 128, "register split");

// A row's running max (the reference of its l and acc) only moves when a
// tile raises the max by more than this, in base-2 units (a factor 256).
constexpr float kRescaleLog2 = 8.0f;

struct Unit {
    int bh, q0, n0, n1, nmax;
    int split, kv_lo;   // key-range split of the unit and its first key tile
};

template <bool CAUSAL>
__device__ __forceinline__ Unit unit_info(int u, const Bf16Params& p) {
    Unit U;
    int pair;
    U.split = u % p.splits;
    u /= p.splits;
    if (CAUSAL) {
        // Heads in groups of heads_per_group; inside a group the longest
        // query tiles (largest pair index) come first.
        const int group_units = p.heads_per_group * p.n_pairs;
        const int g = u / group_units;
        const int r = u - g * group_units;
        const int hg = min(p.heads_per_group, p.bh_count - g * p.heads_per_group);
        pair = p.n_pairs - 1 - r / hg;
        U.bh = g * p.heads_per_group + r % hg;
    } else {
        U.bh = u / p.n_pairs;
        pair = u - U.bh * p.n_pairs;
    }
    // A unit is a pair of 128-row query tiles, or one tile (tile 1 unused)
    // when the launch runs in single-tile units.
    U.q0 = pair * (p.single ? 128 : 256);
    const int nkv = (p.N + 127) / 128;
    // This split's key tiles are [kv_lo, kv_hi).
    const int per = (nkv + p.splits - 1) / p.splits;
    U.kv_lo = min(nkv, U.split * per);
    const int kv_hi = min(nkv, U.kv_lo + per);
    // Key tiles each query tile visits (0 when the tile lies beyond M or
    // the split holds none of its visible keys).
    const int lim0 = CAUSAL ? min(kv_hi, U.q0 / 128 + 1) : kv_hi;
    const int lim1 = CAUSAL ? min(kv_hi, (U.q0 + 128) / 128 + 1) : kv_hi;
    U.n0 = (U.q0 >= p.M) ? 0 : max(0, lim0 - U.kv_lo);
    U.n1 = (p.single || U.q0 + 128 >= p.M) ? 0 : max(0, lim1 - U.kv_lo);
    U.nmax = max(U.n0, U.n1);
    return U;
}

struct Ctx {
    uint32_t bar0;        // shared address of barrier 0
    uint8_t* sQ;
    uint8_t* sKV;
    float* stats_sm;      // [2 t][3 (m, l, l_o)][128]
    uint32_t tmem;
    volatile int* abort;
    uint32_t* err;
    __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * static_cast<uint32_t>(i); }
    __device__ __forceinline__ bool wait(int i, int parity) const {
        return mbar_wait(bar(i), static_cast<uint32_t>(parity) & 1u, abort, err);
    }
    // Whole-warp wait: every lane polls, and all agree on the outcome.
    __device__ __forceinline__ bool wait_warp(int i, int parity) const {
        return __all_sync(0xffffffffu, wait(i, parity));
    }
    // Per-thread arrive (the hand-off barriers count the 128 threads of a
    // warpgroup).
    __device__ __forceinline__ void arrive_warp(int i) const { mbar_arrive(bar(i)); }
    volatile int* ring;   // claimed unit indices, -1 = no more units
};

// The sequence of units this CTA processes, as every role but the TMA thread
// reads it from the ring: next() returns the following unit index, or -1
// when there are no more units (or the pipeline was aborted). `whole_warp`
// readers call it with all 32 lanes and arrive once per warp; the MMA thread
// calls it alone.
template <int SLOTS, int FULL, int EMPTY>
struct UnitReader {
    int k = 0;
    __device__ __forceinline__ int next(const Ctx& c, bool whole_warp) {
        const int slot = k % SLOTS;
        const int phase = k / SLOTS;
        ++k;
        const bool ok = whole_warp ? c.wait_warp(FULL + slot, phase) : c.wait(FULL + slot, phase);
        if (!ok) return -1;
        const int u = c.ring[slot];
        if (whole_warp) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(c.bar(EMPTY + slot));
        } else {
            mbar_arrive(c.bar(EMPTY + slot));
        }
        return u;
    }
};

// ----------------------------------------------------------- TMA producer
template <int D, bool CAUSAL>
__device__ __forceinline__ void producer_role(const CUtensorMap* mq, const CUtensorMap* mk, const CUtensorMap* mv,
                                              const Bf16Params& p, const Ctx& c) {
    using C = Bf16Cfg<D>;
    const uint64_t pol_q = policy_evict_first();
    const uint64_t pol_kv = policy_evict_last();
    int kv_idx = 0, qit = 0;
    int it_base = 0;         // MMA iteration of the current unit's first key tile step
    int rel[C::NS];          // per stage: the MMA iteration whose commit frees its last load
    bool ok = true;
    // Claims the CTA's next unit and publishes it in the ring (-1 once the
    // units are used up). A CTA's first unit is its own index (the grid
    // never has more CTAs than units); the rest come from the global
    // counter, which numbers the units after the first gridDim.x.
    int claimed = 0;
    auto claim = [&]() -> int {
        const int slot = claimed % C::UNIT_SLOTS;
        if (claimed >= C::UNIT_SLOTS && !c.wait(C::UNIT_EMPTY + slot, claimed / C::UNIT_SLOTS - 1)) return -2;
        int v = (claimed == 0) ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(p.sched, 1);
        if (v >= p.num_units) v = -1;
        c.ring[slot] = v;
        mbar_arrive(c.bar(C::UNIT_FULL + slot));
        ++claimed;
        return v;
    };
    int u = claim();
    while (u >= 0 && ok) {
        // The following unit is claimed one ahead, so that its Q tiles can be
        // pulled into L2 while this unit runs.
        const int u_next = claim();
        if (u_next == -2) {
            ok = false;
            break;
        }
        const Unit U = unit_info<CAUSAL>(u, p);
        if (U.nmax == 0) {
            u = u_next;
            continue;
        }
        const int qb = qit % C::QB;
        if (qit >= C::QB && !c.wait(C::Q_EMPTY + qb, qit / C::QB - 1)) {
            ok = false;
            break;
        }
        const int nq = (U.n0 > 0 ? 1 : 0) + (U.n1 > 0 ? 1 : 0);
        mbar_arrive_expect_tx(c.bar(C::Q_FULL + qb), nq * C::TILE_BYTES);
        for (int t = 0; t < 2; ++t) {
            if ((t ? U.n1 : U.n0) == 0) continue;
            for (int pn = 0; pn < C::PANELS; ++pn)
                tma_load_3d(smem_u32(c.sQ + (qb * 2 + t) * C::TILE_BYTES + pn * C::PANEL_BYTES), mq,
                            c.bar(C::Q_FULL + qb), pn * 64, U.q0 + 128 * t, U.bh, pol_q);
        }
        ++qit;
        if (C::QB == 1) {
            // One Q buffer: the next unit's Q tiles can only be loaded once
            // this unit's last Q K^T product is done. Pull them into L2 now so
            // that load does not wait on HBM.
            if (u_next >= 0) {
                const Unit N = unit_info<CAUSAL>(u_next, p);
                for (int t = 0; t < 2; ++t) {
                    if ((t ? N.n1 : N.n0) == 0) continue;
                    for (int pn = 0; pn < C::PANELS; ++pn) tma_prefetch_l2_3d(mq, pn * 64, N.q0 + 128 * t, N.bh);
                }
            }
        }
        for (int j = 0; j < U.nmax && ok; ++j) {
            for (int which = 0; which < 2; ++which) {
                const int stage = kv_idx % C::NS;
                const int round = kv_idx / C::NS;
                if (round > 0 && !c.wait(C::ITER + rel[stage] % C::ITERS, rel[stage] / C::ITERS)) {
                    ok = false;
                    break;
                }
                // K(j) is last read in step j of the unit, V(j) in step j + 1.
                rel[stage] = it_base + j + which;
                mbar_arrive_expect_tx(c.bar(C::KV_FULL + stage), C::TILE_BYTES);
                const CUtensorMap* m = which ? mv : mk;
                for (int pn = 0; pn < C::PANELS; ++pn)
                    tma_load_3d(smem_u32(c.sKV + stage * C::TILE_BYTES + pn * C::PANEL_BYTES), m,
                                c.bar(C::KV_FULL + stage), pn * 64, (U.kv_lo + j) * C::BN, U.bh, pol_kv);
                ++kv_idx;
            }
        }
        it_base += U.nmax + 1;
        u = u_next;
    }
    // Every copy issued must land before this CTA's shared memory is
    // released: wait for the last fill of each stage and of each Q buffer.
    for (int s = 0; s < C::NS && s < kv_idx; ++s) {
        const int last = s + ((kv_idx - 1 - s) / C::NS) * C::NS;
        mbar_wait_drain(c.bar(C::KV_FULL + s), (last / C::NS) & 1);
    }
    for (int b = 0; b < C::QB && b < qit; ++b) {
        const int last = b + ((qit - 1 - b) / C::QB) * C::QB;
        mbar_wait_drain(c.bar(C::Q_FULL + b), (last / C::QB) & 1);
    }
}

// ------------------------------------------------------------- MMA issuer
template <int D, bool CAUSAL>
__device__ __forceinline__ void mma_role(const Bf16Params& p, const Ctx& c) {
    using C = Bf16Cfg<D>;
    constexpr uint32_t id_s = idesc_bf16_f32(128, C::BN, false);
    constexpr uint32_t id_o = idesc_bf16_f32(128, D, true);
    constexpr uint32_t kPanel = C::PANEL_BYTES >> 4;
    const uint32_t sq = smem_u32(c.sQ);
    const uint32_t skv = smem_u32(c.sKV);
    // Descriptor templates with a zero start address; adding (address >> 4)
    // fills the 14-bit start field (shared addresses are < 256 KB).
    const uint64_t desc_k = smem_desc_sw128(0, 16, 1024);
    const uint64_t desc_v = smem_desc_sw128(0, C::PANEL_BYTES, 1024);
    // S_t = Q_t K^T: Q and K tiles K-major, 128-byte swizzle; a 16-column
    // K-step advances 32 B inside a 64-column panel, 4 steps a panel.
    auto issue_s = [&](uint32_t s_col, uint64_t dq, uint64_t dk) {
#pragma unroll
        for (int kk = 0; kk < C::QK_STEPS; ++kk) {
            const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 2;
            mma_ss(c.tmem + s_col, dq + off, dk + off, id_s, kk > 0 ? 1u : 0u);
        }
    };
    // O_t (+)= P_t V: P from tensor memory (aliasing S_t), V MN-major with
    // 128-byte swizzle (LBO = the 64-column panel stride, SBO = 8 rows of
    // 128 B); 16 keys per step. The first product of a unit overwrites O_t.
    auto issue_pv = [&](uint32_t o_col, uint32_t s_col, uint64_t dv, bool first) {
#pragma unroll
        for (int kk = 0; kk < C::PV_STEPS; ++kk)
            mma_ts(c.tmem + o_col, c.tmem + s_col + kk * 8, dv + kk * (2048 >> 4), id_o, (first && kk == 0) ? 0u : 1u);
    };
    int kv_idx = 0, qit = 0;
    int itr = 0;            // key tile steps issued (one ITER commit each)
    int pv0 = 0, pv1 = 0;   // P V products issued per query tile
    int uo0 = 0, uo1 = 0;   // units whose last product was committed, per tile
    bool ok = true;
    UnitReader<C::UNIT_SLOTS, C::UNIT_FULL, C::UNIT_EMPTY> units;
    while (ok) {
        const int u = units.next(c, false);
        if (u < 0) break;
        const Unit U = unit_info<CAUSAL>(u, p);
        if (U.nmax == 0) continue;
        const int n0 = U.n0, n1 = U.n1, nm = U.nmax;
        const int qb = qit % C::QB;
        if (!c.wait(C::Q_FULL + qb, qit / C::QB)) {
            ok = false;
            break;
        }
        tc_fence_after();
        const uint64_t dq0 = desc_k + ((sq + (qb * 2 + 0) * C::TILE_BYTES) >> 4);
        const uint64_t dq1 = desc_k + ((sq + (qb * 2 + 1) * C::TILE_BYTES) >> 4);
        // Key tile step j: K(j) sits in ring slot kidx = kv_idx + 2j, V(j-1)
        // in slot kidx - 1.
        for (int j = 0; j <= nm; ++j) {
            const int kidx = kv_idx + 2 * j;
            const int kst = kidx % C::NS, vst = (kidx + C::NS - 1) % C::NS;
            const uint64_t dk = desc_k + ((skv + kst * C::TILE_BYTES) >> 4);
            const uint64_t dv = desc_v + ((skv + vst * C::TILE_BYTES) >> 4);
            // When tile 0 has a P V product in this step, its P_FULL phase
            // also certifies V(j-1) and K(j) (the gate thread arrives on it
            // once both have landed); otherwise wait for them here.
            if (j == 0 || j > n0) {
                if ((j >= 1 && !c.wait(C::KV_FULL + vst, (kidx - 1) / C::NS)) ||
                    (j < nm && !c.wait(C::KV_FULL + kst, kidx / C::NS))) {
                    ok = false;
                    break;
                }
            }
            if (j >= 1 && j <= n0) {
                if (!c.wait(C::P_FULL + 0, pv0) || (j == 1 && uo0 > 0 && !c.wait(C::O_FREE + 0, uo0 - 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(C::O_COL0, C::S_COL0, dv, j == 1);
                ++pv0;
                if (j == n0) {
                    mma_commit(c.bar(C::O_DONE + 0));
                    ++uo0;
                }
            }
            if (j < n0) {
                tc_fence_after();
                issue_s(C::S_COL0, dq0, dk);
                mma_commit(c.bar(C::S_FULL));
            }
            if (j >= 1 && j <= n1) {
                if (!c.wait(C::P_FULL + 1, pv1) || (j == 1 && uo1 > 0 && !c.wait(C::O_FREE + 1, uo1 - 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_pv(C::O_COL1, C::S_COL1, dv, j == 1);
                ++pv1;
                if (j == n1) {
                    mma_commit(c.bar(C::O_DONE + 1));
                    ++uo1;
                }
            } else if (j >= 1 && n1 == 0 && !p.single) {
                // Tile 1 lies beyond M: its softmax's empty hand-off keeps
                // it in step (tile1_lockstep).
                if (!c.wait(C::P_FULL + 1, pv1)) {
                    ok = false;
                    break;
                }
                ++pv1;
            }
            if (j < n1) {
                tc_fence_after();
                issue_s(C::S_COL1, dq1, dk);
            }
            if (j == nm - 1) mma_commit(c.bar(C::Q_EMPTY + qb));
            // One commit per step: S_1(j) is ready, and K(j) and V(j-1) are
            // free once every product issued so far has completed.
            mma_commit(c.bar(C::ITER + itr % C::ITERS));
            ++itr;
        }
        kv_idx += 2 * nm;
        ++qit;
    }
    // All MMAs issued must finish before tensor memory is freed.
    mma_commit(c.bar(C::DRAIN));
    mbar_wait_drain(c.bar(C::DRAIN), 0);
}

// ---------------------------------------------------------------- softmax
// Tile 1's softmax for a pair whose tile 1 lies beyond M: it steps with the
// MMA thread anyway, waiting for each of the unit's `n` steps and handing
// over an empty P, so that it is never more than two steps ahead of the
// MMA thread. The ITER ring is waited on by phase parity, which only tells
// phase k from k + 1; skipping the unit's steps could put tile 1 ITERS or
// more steps ahead, where a phase not yet begun reads as complete. Kept out
// of line so that the softmax's own loop keeps its registers.
template <int ITERS>
__device__ __noinline__ bool tile1_lockstep(uint32_t iter0, uint32_t p_full1, volatile int* abort, uint32_t* err,
                                            int itb, int n) {
    for (int j = 0; j < n; ++j) {
        const int s = itb + j;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(iter0 + 8u * static_cast<uint32_t>(s % ITERS),
                                                          static_cast<uint32_t>(s / ITERS) & 1u, abort, err));
        if (!ok) return false;
        mbar_arrive(p_full1);
    }
    return true;
}

template <int D, bool CAUSAL>
__device__ __forceinline__ void softmax_role(int t, const Bf16Params& p, const Ctx& c) {
    using C = Bf16Cfg<D>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = (warp & 3) * 32 + lane;                   // row in the tile = TMEM lane
    const uint32_t lane_base = c.tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_addr = lane_base + (t ? C::S_COL1 : C::S_COL0);
    const float cl2 = p.scale_log2;
    const uint64_t c2 = f2_pack(cl2, cl2);
    int s_cnt = 0, st_cnt = 0;
    int it_base = 0;   // MMA step of the current unit's first key tile
    bool ok = true;
    UnitReader<C::UNIT_SLOTS, C::UNIT_FULL, C::UNIT_EMPTY> units;
    while (ok) {
        const int u = units.next(c, true);
        if (u < 0) break;
        const Unit U = unit_info<CAUSAL>(u, p);
        const int itb = it_base;
        if (U.nmax > 0) it_base += U.nmax + 1;
        const int ntile = t ? U.n1 : U.n0;
        if (t == 1 && ntile == 0 && U.nmax > 0 && !p.single) {
            ok = tile1_lockstep<C::ITERS>(c.bar(C::ITER), c.bar(C::P_FULL + 1), c.abort, c.err, itb, U.nmax);
            continue;
        }
        if (ntile == 0) continue;
        const int qt0 = U.q0 + 128 * t;                     // first row of the tile
        const int qrow = qt0 + r;
        float m_run = -INFINITY;   // running max of scaled scores, base-2 units
        float l_run = 0.f;         // running sum of exp2(score - m_run)
        float lo_run = 0.f;        // l with each tile's largest weight as rounded to bf16
        for (int j = 0; j < ntile; ++j) {
            // Every lane must agree: the tensor-memory loads below are
            // warp-collective.
            // S_0(j) has its own barrier; S_1(j) is announced by step j's
            // ITER commit (sound while tile 1 stays within ITERS - 1 steps of
            // the MMA thread, which the lockstep below guarantees).
            const bool s_ok = t == 0 ? c.wait_warp(C::S_FULL, s_cnt)
                                     : c.wait_warp(C::ITER + (itb + j) % C::ITERS, (itb + j) / C::ITERS);
            if (!s_ok) {
                ok = false;
                break;
            }
            ++s_cnt;
            tc_fence_after();
            uint32_t s[128];
            // Row max from the tensor-memory loads themselves (tcgen05.ld.red,
            // one maximum per 32 columns); a masked tile's maximum is taken
            // again after masking.
            float rr[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                tmem_ld_red_max_x32(s_addr + 32 * q4, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * q4]), rr[q4]);
            tmem_ld_wait(s);
            asm volatile("" : "+f"(rr[0]), "+f"(rr[1]), "+f"(rr[2]), "+f"(rr[3]));
            const int kv0 = (U.kv_lo + j) * C::BN;
            const bool need_mask = (kv0 + C::BN > p.N) || (CAUSAL && kv0 + C::BN - 1 > qt0);
            float mx = fmaxf(fmaxf(rr[0], rr[1]), fmaxf(rr[2], rr[3]));
            if (need_mask) {
                int lim = p.N - kv0;                         // key columns < N
                if (CAUSAL) lim = min(lim, qrow - kv0 + 1);  // key <= query
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i >= lim) s[i] = __float_as_uint(-INFINITY);
                float mx0 = fmaxf(__uint_as_float(s[0]), __uint_as_float(s[1]));
                float mx1 = fmaxf(__uint_as_float(s[2]), __uint_as_float(s[3]));
#pragma unroll
                for (int i = 4; i < 128; i += 4) {
                    mx0 = fmax3(mx0, __uint_as_float(s[i + 0]), __uint_as_float(s[i + 1]));
                    mx1 = fmax3(mx1, __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
                }
                mx = fmaxf(mx0, mx1);
            }
            // Running max m_run: the common reference of l and acc. It moves
            // only when a tile raises the row max by more than kRescaleLog2
            // (then alpha rescales what was accumulated, as on the pages);
            // below that p = exp2(s*c - m_run) <= 2^kRescaleLog2 and nothing
            // needs rescaling, which makes the rescale of O rare.
            const float m_tile = mx * cl2;                         // -inf if all masked
            const bool grow = m_tile > m_run + kRescaleLog2;       // first visible tile: m_run = -inf
            const float m_new = grow ? m_tile : m_run;
            const float alpha = grow ? ex2(m_run - m_new) : 1.f;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;   // no -inf - -inf
            const uint64_t neg2 = f2_pack(-m_use, -m_use);
            uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
            uint32_t pk[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2, neg2);
                float x0, x1;
                f2_unpack(x2, x0, x1);
                const float p0 = ex2(x0);
                const float p1 = ex2(x1);
                acc2[i & 3] = f2_add(acc2[i & 3], f2_pack(p0, p1));
                pk[i] = pack_bf16x2(p0, p1);
            }
            // The tile's largest weight exactly as the MMA will see it (same
            // FMA and exp2 as in the loop, then bf16): its rounding error
            // goes into l_o, the normaliser of O, so a dominant key is not
            // misweighted when the reference is stale (p_max may be > 1).
            const float pmax = ex2(fmaf(mx, cl2, -m_use));
            const float pmax_b = __uint_as_float(pack_bf16x2(pmax, 0.f) << 16);
            tmem_st_x32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            // A moved reference: rescale this warp's rows of O. S_t(j) was
            // issued after P_t(j-1) V(j-1), so that product has landed; tile 0
            // of a unit has no accumulator yet (its first product overwrites).
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
                const uint32_t o_addr = lane_base + (t ? C::O_COL1 : C::O_COL0);
                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    tmem_ld_x32(o_addr + cc * 32, ov);
                    tmem_ld_wait(ov);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float lo, hi;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(ov[2 * i]), __uint_as_float(ov[2 * i + 1])), a2, 0ull), lo, hi);
                        ov[2 * i] = __float_as_uint(lo);
                        ov[2 * i + 1] = __float_as_uint(hi);
                    }
                    tmem_st_x32(o_addr + cc * 32, ov);
                }
            }
            float sa, sb, sc, sd;
            f2_unpack(f2_add(acc2[0], acc2[1]), sa, sb);
            f2_unpack(f2_add(acc2[2], acc2[3]), sc, sd);
            const float lsum = (sa + sb) + (sc + sd);
            l_run = l_run * alpha + lsum;
            lo_run = lo_run * alpha + (lsum + (pmax_b - pmax));
            m_run = m_new;
            tmem_st_wait();
            tc_fence_before();
            c.arrive_warp(C::P_FULL + t);
        }
        if (!ok) break;
        // Final statistics of this tile for the epilogue, once it has read
        // the previous unit's (ST_EMPTY): that also keeps ST_FULL at most one
        // phase ahead of its waiter.
        if (st_cnt > 0 && !c.wait_warp(C::ST_EMPTY + t, st_cnt - 1)) break;
        float* st = c.stats_sm + t * 384;
        st[r] = m_run;
        st[128 + r] = l_run;
        st[256 + r] = lo_run;
        c.arrive_warp(C::ST_FULL + t);
        ++st_cnt;
    }
}

// ------------------------------------------------------------ K/V gate
// Waits, in the MMA thread's place, for the K/V tiles of each step in which
// query tile 0 has a P V product: step j + 1 reads V(j) and K(j + 1) (if
// any), and the MMA thread waits on P_FULL_0 phase of tile j before it
// issues anything in that step. The gate arrives on that phase (its 129th
// arrival, next to the 128 softmax threads) once both tiles have landed,
// then waits for the phase to complete before it arrives again. Shared-
// memory polls are slow while the tensor core streams its operands, so
// every one taken off the MMA thread leaves the tensor pipe fed longer.
template <int D, bool CAUSAL>
__device__ __forceinline__ void gate_role(const Bf16Params& p, const Ctx& c) {
    using C = Bf16Cfg<D>;
    int kv_idx = 0;   // loads issued before the current unit (the producer's count)
    int pc = 0;       // P_FULL_0 phases
    UnitReader<C::UNIT_SLOTS, C::UNIT_FULL, C::UNIT_EMPTY> units;
    while (true) {
        const int u = units.next(c, false);
        if (u < 0) break;
        const Unit U = unit_info<CAUSAL>(u, p);
        if (U.nmax == 0) continue;
        bool ok = true;
        for (int j = 0; j < U.n0 && ok; ++j) {
            const int lv = kv_idx + 2 * j + 1;   // V(j); K(j + 1) follows it
            ok = c.wait(C::KV_FULL + lv % C::NS, lv / C::NS) &&
                 (j + 1 >= U.nmax || c.wait(C::KV_FULL + (lv + 1) % C::NS, (lv + 1) / C::NS));
            if (!ok) break;
            mbar_arrive(c.bar(C::P_FULL + 0));
            ok = c.wait(C::P_FULL + 0, pc);
            ++pc;
        }
        if (!ok) break;
        kv_idx += 2 * U.nmax;
    }
}

// --------------------------------------------------------------- epilogue
// Per unit and query tile: O = acc / l_o in bf16 (or the split's fp32 partial
// result), LSE = ln2 * (m + log2 l).
template <int D, bool CAUSAL>
__device__ __forceinline__ void epilogue_role(const Bf16Params& p, const Ctx& c) {
    using C = Bf16Cfg<D>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int st_cnt[2] = {0, 0}, od_cnt[2] = {0, 0};
    bool ok = true;
    UnitReader<C::UNIT_SLOTS, C::UNIT_FULL, C::UNIT_EMPTY> units;
    while (ok) {
        const int u = units.next(c, true);
        if (u < 0) break;
        const Unit U = unit_info<CAUSAL>(u, p);
        // Epilogue: O = acc / l in bf16, LSE = ln2 * (m + log2 l).
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int nt = t ? U.n1 : U.n0;
            const int qt0 = U.q0 + 128 * t;
            // Tile 1 of a single-tile unit is another unit's query tile.
            if (!ok || qt0 >= p.M || (t == 1 && p.single)) continue;
            float m_fin = -INFINITY, l_fin = 0.f, lo_fin = 0.f;
            if (nt > 0) {
                bool w = c.wait_warp(C::ST_FULL + t, st_cnt[t]);
                w = w && c.wait_warp(C::O_DONE + t, od_cnt[t]);
                if (!w) {
                    ok = false;
                    break;
                }
                const float* st = c.stats_sm + t * 384;
                m_fin = st[r];
                l_fin = st[128 + r];
                lo_fin = st[256 + r];
                c.arrive_warp(C::ST_EMPTY + t);
                ++st_cnt[t];
                ++od_cnt[t];
                tc_fence_after();
            }
            const int qrow = qt0 + r;
            const bool store = qrow < p.M;
            const float inv_l = (lo_fin > 0.f) ? 1.f / lo_fin : 0.f;
            const float lse_val = (l_fin > 0.f) ? (m_fin + log2f(l_fin)) * 0.69314718055994531f : -INFINITY;
            const uint32_t o_addr = c.tmem + lane_base + (t ? C::O_COL1 : C::O_COL0);
            const size_t row_idx = static_cast<size_t>(U.bh) * p.M + (store ? qrow : 0);
            if (p.splits == 1) {
                uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + row_idx * D;   // bf16 bits
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    if (nt > 0) {
                        tmem_ld_x32(o_addr + cc * 32, ov);
                        tmem_ld_wait(ov);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = 0u;
                    }
                    uint32_t pkd[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pkd[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
                    if (store) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
                    }
                }
                if (store) p.lse[row_idx] = lse_val;
            } else {
                // Split-KV: this split's normalised fp32 O and its LSE go to
                // the workspace; a second kernel merges the splits.
                const size_t ws_row = static_cast<size_t>(U.split) * p.bh_count * p.M + row_idx;
                float* orow = p.ws_o + ws_row * D;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    if (nt > 0) {
                        tmem_ld_x32(o_addr + cc * 32, ov);
                        tmem_ld_wait(ov);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = 0u;
                    }
                    if (store) {
                        float4* dst = reinterpret_cast<float4*>(orow + cc * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(ov[4 * i]) * inv_l, __uint_as_float(ov[4 * i + 1]) * inv_l,
                                                 __uint_as_float(ov[4 * i + 2]) * inv_l, __uint_as_float(ov[4 * i + 3]) * inv_l);
                    }
                }
                if (store) p.ws_lse[ws_row] = lse_val;
            }
            if (nt > 0) {
                tc_fence_before();
                c.arrive_warp(C::O_FREE + t);
            }
        }
    }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(Bf16Cfg<D>::THREADS, 1)
fa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const Bf16Params p) {
    using C = Bf16Cfg<D>;
    // All shared state lives in the dynamic window (no static shared
    // variables), aligned up to 1024 B inside the launch's slack.
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t& tmem_base_sh = *reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    int& abort_sh = *reinterpret_cast<int*>(smem + C::MISC_OFF + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    Ctx c;
    c.bar0 = smem_u32(smem + C::BAR_OFF);
    c.sQ = smem + C::Q_OFF;
    c.sKV = smem + C::KV_OFF;
    c.stats_sm = reinterpret_cast<float*>(smem + C::STATS_OFF);
    c.abort = &abort_sh;
    c.err = p.err;
    c.ring = reinterpret_cast<volatile int*>(smem + C::RING_OFF);

    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int s = 0; s < C::NS; ++s) mbar_init(c.bar(C::KV_FULL + s), 1);
        for (int s = 0; s < C::ITERS; ++s) mbar_init(c.bar(C::ITER + s), 1);
        for (int b = 0; b < C::QB; ++b) {
            mbar_init(c.bar(C::Q_FULL + b), 1);
            mbar_init(c.bar(C::Q_EMPTY + b), 1);
        }
        mbar_init(c.bar(C::S_FULL), 1);
        mbar_init(c.bar(C::P_FULL + 0), 128 + 1);   // softmax of tile 0 + the K/V gate
        mbar_init(c.bar(C::P_FULL + 1), 128);
        for (int t = 0; t < 2; ++t) {
            mbar_init(c.bar(C::O_DONE + t), 1);
            mbar_init(c.bar(C::O_FREE + t), 128);
            mbar_init(c.bar(C::ST_FULL + t), 128);
            mbar_init(c.bar(C::ST_EMPTY + t), 128);
        }
        mbar_init(c.bar(C::DRAIN), 1);
        for (int s = 0; s < C::UNIT_SLOTS; ++s) {
            mbar_init(c.bar(C::UNIT_FULL + s), 1);
            mbar_init(c.bar(C::UNIT_EMPTY + s), C::UNIT_READERS);
        }
        fence_barrier_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(&tmem_base_sh), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 12 && lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = tmem_base_sh;

    const int wg = warp >> 2;
    if (wg < 2) {
        setmaxnreg_inc<kRegsSoftmax>();
        softmax_role<D, CAUSAL>(wg, p, c);
    } else if (wg == 2) {
        setmaxnreg_dec<kRegsEpilogue>();
        epilogue_role<D, CAUSAL>(p, c);
    } else {
        setmaxnreg_dec<kRegsLoadMma>();
        if (warp == 12) {
            if (lane == 0) producer_role<D, CAUSAL>(&map_q, &map_k, &map_v, p, c);
            __syncwarp();
        } else if (warp == 13) {
            if (lane == 0) mma_role<D, CAUSAL>(p, c);
            __syncwarp();
        } else if (warp == 14) {
            if (lane == 0) gate_role<D, CAUSAL>(p, c);
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after();
        tmem_dealloc(c.tmem, C::TMEM_COLS);
    }
    // The last CTA to finish resets the unit counter for the next launch that
    // uses it; every CTA's claims precede its count here.
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            atomicExch(p.sched, 0);
            atomicExch(p.sched + 1, 0);
        }
    }
}

inline int sm_count_cached() {
    static std::atomic<int> counts[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

template <int D>
cudaError_t launch_bf16(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const Bf16Params& p,
                        bool causal, cudaStream_t stream) {
    using C = Bf16Cfg<D>;
    const int sms = sm_count_cached();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = p.num_units < sms ? p.num_units : sms;   // persistent: one CTA per SM
    auto kern = causal ? fa_fwd_bf16_kernel<D, true> : fa_fwd_bf16_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

}  // namespace fa
