// bf16 FlashAttention forward for head dimension 64 on sm_103a: one 128-row
// query tile per CTA, 64-key steps, four CTAs per SM.
//
// Same algorithm and numerics as fa_bf16_kernel.cuh ("FlashAttention-style
// kernel", section "The loop"; "Module 08: FlashAttention and
// Memory-Efficient Kernels", sections "Tiling and the online softmax" and
// "Related ideas"): a query tile stays resident while key/value tiles stream
// past it; per row the running max m, sum l and unnormalised output acc,
// rescaled by alpha = exp2(m_old - m_new) when the max grows by more than
// 2^8; O = acc / l_o and LSE = m + log l written once at the end.
//
// Why a separate kernel at D = 64: a 128 x 64 S tile and a 128 x 64 O
// accumulator take 128 tensor-memory columns, so four CTAs fit on one SM
// (512 columns), each with its own MMA thread. A single CTA's step is a
// serial chain (S = Q K^T, softmax, P V, next S), but four independent
// chains keep the shared tensor pipe busy: while one CTA's softmax runs or
// its MMA thread waits on a barrier, the others' products execute. With two
// query tiles in one CTA (fa_bf16_kernel.cuh) one thread issues every
// product and each of its barrier polls or commits leaves the pipe idle.
//
// Roles (256 threads, registers re-split with setmaxnreg per warpgroup):
//   warps 0-3  softmax of the tile (thread = row = tensor-memory lane) and,
//              at the end of a unit, its epilogue (O / l_o, LSE)
//   warp 4     TMA producer (Q once per unit; K and V 64-row tiles)
//   warp 5     tensor-memory owner and MMA issuer
//   warp 6     K/V gate: waits for V(j-1) and K(j) in the MMA thread's place
//              and arrives on P_FULL next to the 128 softmax threads
//   warp 7     idle (completes the second warpgroup)
//
// Tensor memory (128 columns): [0, 64) S (fp32; P overwrites its first 32
// columns as bf16 pairs after the softmax), [64, 128) O.
//
// Per unit the MMA thread runs steps j = 0 .. n (n = key tiles of 64):
//   step j: O += P(j-1) V(j-1) (j >= 1); S = Q K(j)^T (j < n); one ITER
//   commit, which announces S(j) to the softmax and frees K(j) and V(j-1).
// K(j), V(j) are the unit's j-th key tile in visiting order: tile
// (first + j) mod n (unit_info).
// One thread's MMAs run in issue order, so S(j) overwrites P(j-1) only after
// the product that reads it.
//
// Every wait is bounded (ptx.cuh); on a time-out the kernel sets the device
// status word, every role leaves its loop, in-flight copies and MMAs are
// drained, and tensor memory is freed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace q1 {

struct Cfg {
    static constexpr int D = 64;
    static constexpr int BM = 128;                 // query rows per CTA tile
    static constexpr int BN = 64;                  // keys per step
    static constexpr int THREADS = 256;
    static constexpr int CTAS_PER_SM = 4;
    static constexpr uint32_t TMEM_COLS = 128;
    static constexpr uint32_t S_COL = 0, O_COL = 64;
    static constexpr int Q_BYTES = BM * 128;       // 128 rows x 64 bf16
    static constexpr int KV_BYTES = BN * 128;      // 64 rows x 64 bf16
    static constexpr int NS = 4;                   // K/V ring stages
    static constexpr int ITERS = 8;                // ring of per-step commit barriers
    static constexpr int Q_OFF = 0;
    static constexpr int KV_OFF = Q_OFF + Q_BYTES;
    static constexpr int BAR_OFF = KV_OFF + NS * KV_BYTES;
    static constexpr int KV_FULL = 0, ITER = NS, Q_FULL = ITER + ITERS, Q_EMPTY = Q_FULL + 1;
    static constexpr int P_FULL = Q_EMPTY + 1, O_DONE = P_FULL + 1, O_FREE = O_DONE + 1, DRAIN = O_FREE + 1;
    static constexpr int UNIT_SLOTS = 4;
    static constexpr int UNIT_FULL = DRAIN + 1, UNIT_EMPTY = UNIT_FULL + UNIT_SLOTS;
    // Readers of a unit-ring slot: one lane of each softmax warp, the MMA
    // thread and the gate thread.
    static constexpr int UNIT_READERS = 4 + 1 + 1;
    static constexpr int NUM_BARS = UNIT_EMPTY + UNIT_SLOTS;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;   // tensor-memory base, abort flag
    static constexpr int RING_OFF = MISC_OFF + 16;
    static constexpr int SMEM_USED = RING_OFF + UNIT_SLOTS * 4;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;       // + slack to align the base to 1024 B
    static_assert(SMEM_BYTES * CTAS_PER_SM + CTAS_PER_SM * 1024 <= 233472, "shared memory for four CTAs");
};

// Launch registers: 65536 / (4 CTAs x 256 threads) = 64. setmaxnreg works
// on whole warpgroups: the softmax warpgroup raises its warps to 88, the
// other one (producer, MMA, gate and an idle warp) drops to 40:
// 128 x 88 + 128 x 40 = 256 x 64.
constexpr int kLaunchRegs = 64;
constexpr int kRegsSoftmax = 88, kRegsOther = 40;
static_assert(128 * kRegsSoftmax + 128 * kRegsOther == Cfg::THREADS * kLaunchRegs, "register split");
static_assert(Cfg::THREADS * kLaunchRegs * Cfg::CTAS_PER_SM == 65536, "launch registers");

constexpr float kRescaleLog2 = 8.0f;

struct Unit {
    int bh, q0, n;   // head, first query row, 64-key steps
    int first;       // key tile of step 0; step j visits tile (first + j) mod n
};

template <bool CAUSAL>
__device__ __forceinline__ Unit unit_info(int u, const Bf16Params& p, int n_tiles) {
    Unit U;
    int qt;
    if (CAUSAL) {
        // Groups of heads_per_group heads; inside a group the longest query
        // tiles (largest index) come first, so the last units are short.
        const int group_units = p.heads_per_group * n_tiles;
        const int g = u / group_units;
        const int r = u - g * group_units;
        const int hg = min(p.heads_per_group, p.bh_count - g * p.heads_per_group);
        qt = n_tiles - 1 - r / hg;
        U.bh = g * p.heads_per_group + r % hg;
    } else {
        U.bh = u / n_tiles;
        qt = u - U.bh * n_tiles;
    }
    U.q0 = qt * Cfg::BM;
    const int nkv = (p.N + Cfg::BN - 1) / Cfg::BN;
    // Key tiles the tile visits: all, or (top-left causal) those with a key
    // <= the tile's last row.
    U.n = CAUSAL ? min(nkv, (U.q0 + Cfg::BM - 1) / Cfg::BN + 1) : nkv;
    // The online softmax does not depend on the order of the key tiles, so
    // each unit starts at an offset in [0, 8) hashed from its query tile:
    // CTAs working on one head at the same time then read different K/V
    // lines instead of the same ones (measured +2 %). The head index plays
    // no part, so a call over a subset of the heads gives the same bits.
    const uint32_t h = static_cast<uint32_t>(qt) * 2654435761u;
    U.first = U.n > 0 ? static_cast<int>((h >> 8) % static_cast<uint32_t>(min(U.n, 8))) : 0;
    return U;
}

// mbar_wait with the abort flag and the clock read only after every 16
// unsuccessful polls: a waiting warp here shares its SM sub-partition with
// three other CTAs' softmax warps, and the cheaper loop leaves them more
// issue slots (measured +2-4 % at D = 64; slower for the two-tile kernel).
__device__ __forceinline__ bool wait_batched(uint32_t bar, uint32_t parity, volatile int* abort, uint32_t* err_word) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            if (err_word) atomicOr(err_word, DEV_ERR_TIMEOUT);
            return false;
        }
    }
}

struct Ctx {
    uint32_t bar0;
    uint8_t* sQ;
    uint8_t* sKV;
    uint32_t tmem;
    volatile int* abort;
    uint32_t* err;
    volatile int* ring;
    __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * static_cast<uint32_t>(i); }
    __device__ __forceinline__ bool wait(int i, int parity) const {
        return wait_batched(bar(i), static_cast<uint32_t>(parity) & 1u, abort, err);
    }
    __device__ __forceinline__ bool wait_warp(int i, int parity) const {
        return __all_sync(0xffffffffu, wait(i, parity));
    }
};

// The CTA's sequence of units as every role but the producer reads it from
// the ring (-1 when there are no more, or the pipeline was aborted).
struct UnitReader {
    int k = 0;
    __device__ __forceinline__ int next(const Ctx& c, bool whole_warp) {
        const int slot = k % Cfg::UNIT_SLOTS;
        const int phase = k / Cfg::UNIT_SLOTS;
        ++k;
        const bool ok = whole_warp ? c.wait_warp(Cfg::UNIT_FULL + slot, phase) : c.wait(Cfg::UNIT_FULL + slot, phase);
        if (!ok) return -1;
        const int u = c.ring[slot];
        if (whole_warp) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(c.bar(Cfg::UNIT_EMPTY + slot));
        } else {
            mbar_arrive(c.bar(Cfg::UNIT_EMPTY + slot));
        }
        return u;
    }
};

// ----------------------------------------------------------- TMA producer
template <bool CAUSAL>
__device__ __forceinline__ void producer_role(const CUtensorMap* mq, const CUtensorMap* mk, const CUtensorMap* mv,
                                              const Bf16Params& p, const Ctx& c, int n_tiles) {
    using C = Cfg;
    const uint64_t pol_q = policy_evict_first();
    const uint64_t pol_kv = policy_evict_last();
    int kv_idx = 0, qit = 0, it_base = 0;
    int rel[C::NS];   // per stage: the MMA step whose commit frees its last load
    bool ok = true;
    int claimed = 0;
    // A CTA's first unit is its own index; later ones come from the counter,
    // which numbers the units after the first gridDim.x.
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
        const int u_next = claim();
        if (u_next == -2) break;
        const Unit U = unit_info<CAUSAL>(u, p, n_tiles);
        if (U.n > 0) {
            if (qit >= 1 && !c.wait(C::Q_EMPTY, qit - 1)) break;
            mbar_arrive_expect_tx(c.bar(C::Q_FULL), C::Q_BYTES);
            tma_load_3d(smem_u32(c.sQ), mq, c.bar(C::Q_FULL), 0, U.q0, U.bh, pol_q);
            ++qit;
            // The next unit's Q tile into L2 while this unit runs.
            if (u_next >= 0) {
                const Unit N = unit_info<CAUSAL>(u_next, p, n_tiles);
                if (N.n > 0) tma_prefetch_l2_3d(mq, 0, N.q0, N.bh);
            }
            for (int j = 0; j < U.n && ok; ++j) {
                for (int which = 0; which < 2; ++which) {
                    const int stage = kv_idx % C::NS;
                    const int round = kv_idx / C::NS;
                    if (round > 0 && !c.wait(C::ITER + rel[stage] % C::ITERS, rel[stage] / C::ITERS)) {
                        ok = false;
                        break;
                    }
                    // K(j) is last read in step j, V(j) in step j + 1.
                    rel[stage] = it_base + j + which;
                    mbar_arrive_expect_tx(c.bar(C::KV_FULL + stage), C::KV_BYTES);
                    const int t = (j + U.first < U.n) ? j + U.first : j + U.first - U.n;   // key tile
                    tma_load_3d(smem_u32(c.sKV + stage * C::KV_BYTES), which ? mv : mk, c.bar(C::KV_FULL + stage), 0,
                                t * C::BN, U.bh, pol_kv);
                    ++kv_idx;
                }
            }
            it_base += U.n + 1;
        }
        u = u_next;
    }
    // Every copy issued must land before the CTA's shared memory is released.
    for (int s = 0; s < C::NS && s < kv_idx; ++s) {
        const int last = s + ((kv_idx - 1 - s) / C::NS) * C::NS;
        mbar_wait_drain(c.bar(C::KV_FULL + s), (last / C::NS) & 1);
    }
    if (qit > 0) mbar_wait_drain(c.bar(C::Q_FULL), (qit - 1) & 1);
}

// ------------------------------------------------------------- MMA issuer
template <bool CAUSAL>
__device__ __forceinline__ void mma_role(const Bf16Params& p, const Ctx& c, int n_tiles) {
    using C = Cfg;
    constexpr uint32_t id_s = idesc_bf16_f32(128, C::BN, false);
    constexpr uint32_t id_o = idesc_bf16_f32(128, C::D, true);
    const uint32_t sq = smem_u32(c.sQ);
    const uint32_t skv = smem_u32(c.sKV);
    // S = Q K^T: Q (128 rows) and K (64 rows) K-major, 128-byte swizzle, one
    // 64-column panel each; a 16-column K-step advances 32 B.
    const uint64_t dq = smem_desc_sw128(0, 16, 1024) + (sq >> 4);
    const uint64_t desc_k = smem_desc_sw128(0, 16, 1024);
    // O += P V: P from tensor memory, V (64 keys x 64 columns) MN-major; a
    // 16-key step advances 16 rows of 128 B.
    const uint64_t desc_v = smem_desc_sw128(0, C::KV_BYTES, 1024);
    int kv_idx = 0, qit = 0, itr = 0, pv = 0, uo = 0;
    bool ok = true;
    UnitReader units;
    while (ok) {
        const int u = units.next(c, false);
        if (u < 0) break;
        const Unit U = unit_info<CAUSAL>(u, p, n_tiles);
        if (U.n == 0) continue;
        const int n = U.n;
        if (!c.wait(C::Q_FULL, qit)) break;
        tc_fence_after();
        for (int j = 0; j <= n; ++j) {
            const int kidx = kv_idx + 2 * j;
            const int kst = kidx % C::NS, vst = (kidx + C::NS - 1) % C::NS;
            const uint64_t dk = desc_k + ((skv + kst * C::KV_BYTES) >> 4);
            const uint64_t dv = desc_v + ((skv + vst * C::KV_BYTES) >> 4);
            if (j == 0) {
                // The gate certifies K/V only together with a P hand-off.
                if (!c.wait(C::KV_FULL + kst, kidx / C::NS)) {
                    ok = false;
                    break;
                }
            } else {
                // P(j-1) is in tensor memory; the gate's arrival on the same
                // phase says V(j-1) and K(j) (if any) have landed. The unit's
                // first product overwrites O: the epilogue must have read it.
                if (!c.wait(C::P_FULL, pv) || (j == 1 && uo > 0 && !c.wait(C::O_FREE, uo - 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    mma_ts(c.tmem + C::O_COL, c.tmem + C::S_COL + kk * 8, dv + kk * (2048 >> 4), id_o,
                           (j == 1 && kk == 0) ? 0u : 1u);
                ++pv;
                if (j == n) {
                    mma_commit(c.bar(C::O_DONE));
                    ++uo;
                }
            }
            if (j < n) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < C::D / 16; ++kk)
                    mma_ss(c.tmem + C::S_COL, dq + kk * 2, dk + kk * 2, id_s, kk > 0 ? 1u : 0u);
            }
            if (j == n - 1) mma_commit(c.bar(C::Q_EMPTY));
            // S(j) is ready, and K(j), V(j-1) are free, once every product
            // issued so far has completed.
            mma_commit(c.bar(C::ITER + itr % C::ITERS));
            ++itr;
        }
        kv_idx += 2 * n;
        ++qit;
    }
    mma_commit(c.bar(C::DRAIN));
    mbar_wait_drain(c.bar(C::DRAIN), 0);
}

// ------------------------------------------------------------ K/V gate
// For step j >= 1 of a unit the MMA thread waits only on P_FULL; the gate
// adds its arrival to that phase once V(j-1) and K(j) (if j < n) have landed,
// then waits for the phase to complete before it arrives again.
template <bool CAUSAL>
__device__ __forceinline__ void gate_role(const Bf16Params& p, const Ctx& c, int n_tiles) {
    using C = Cfg;
    int kv_idx = 0, pc = 0;
    UnitReader units;
    while (true) {
        const int u = units.next(c, false);
        if (u < 0) break;
        const Unit U = unit_info<CAUSAL>(u, p, n_tiles);
        if (U.n == 0) continue;
        bool ok = true;
        for (int j = 1; j <= U.n && ok; ++j) {
            const int lv = kv_idx + 2 * j - 1;   // V(j-1); K(j) follows it
            ok = c.wait(C::KV_FULL + lv % C::NS, lv / C::NS) &&
                 (j == U.n || c.wait(C::KV_FULL + (lv + 1) % C::NS, (lv + 1) / C::NS));
            if (!ok) break;
            mbar_arrive(c.bar(C::P_FULL));
            ok = c.wait(C::P_FULL, pc);
            ++pc;
        }
        if (!ok) break;
        kv_idx += 2 * U.n;
    }
}

// ----------------------------------------------- softmax and epilogue
template <bool CAUSAL>
__device__ __forceinline__ void softmax_role(const Bf16Params& p, const Ctx& c, int n_tiles) {
    using C = Cfg;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = warp * 32 + lane;                          // row = tensor-memory lane
    const uint32_t lane_base = c.tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t s_addr = lane_base + C::S_COL;
    const uint32_t o_addr = lane_base + C::O_COL;
    const float cl2 = p.scale_log2;
    const uint64_t c2 = f2_pack(cl2, cl2);
    int it_base = 0, od = 0;
    bool ok = true;
    UnitReader units;
    while (ok) {
        const int u = units.next(c, true);
        if (u < 0) break;
        const Unit U = unit_info<CAUSAL>(u, p, n_tiles);
        const int qrow = U.q0 + r;
        if (U.n == 0) {
            // No keys (N = 0): O = 0 and LSE = -inf; nothing else runs.
            if (qrow < p.M) {
                const size_t row_idx = static_cast<size_t>(U.bh) * p.M + qrow;
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.o) + row_idx * C::D);
#pragma unroll
                for (int i = 0; i < C::D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
                p.lse[row_idx] = -INFINITY;
            }
            continue;
        }
        const int itb = it_base;
        it_base += U.n + 1;
        float m_run = -INFINITY;   // running max (base 2), the reference of l and acc
        float l_run = 0.f;         // running sum of exp2(score - m_run)
        float lo_run = 0.f;        // l with each tile's largest weight as rounded to bf16
        for (int j = 0; j < U.n; ++j) {
            // S(j) is announced by step j's ITER commit.
            if (!c.wait_warp(C::ITER + (itb + j) % C::ITERS, (itb + j) / C::ITERS)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[64];
            // Row max from the tensor-memory loads themselves (tcgen05.ld.red,
            // +6-9 % against a max3 chain); a masked tile's maximum is taken
            // again after masking.
            float r0, r1;
            tmem_ld_red_max_x32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]), r0);
            tmem_ld_red_max_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]), r1);
            tmem_ld_wait(s);
            asm volatile("" : "+f"(r0), "+f"(r1));
            const int kv0 = ((j + U.first < U.n) ? j + U.first : j + U.first - U.n) * C::BN;
            float mx = fmaxf(r0, r1);
            if ((kv0 + C::BN > p.N) || (CAUSAL && kv0 + C::BN - 1 > U.q0)) {
                int lim = p.N - kv0;                             // key columns < N
                if (CAUSAL) lim = min(lim, qrow - kv0 + 1);      // key <= query
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i >= lim) s[i] = __float_as_uint(-INFINITY);
                float mx0 = fmaxf(__uint_as_float(s[0]), __uint_as_float(s[1]));
                float mx1 = fmaxf(__uint_as_float(s[2]), __uint_as_float(s[3]));
#pragma unroll
                for (int i = 4; i < 64; i += 4) {
                    mx0 = fmax3(mx0, __uint_as_float(s[i + 0]), __uint_as_float(s[i + 1]));
                    mx1 = fmax3(mx1, __uint_as_float(s[i + 2]), __uint_as_float(s[i + 3]));
                }
                mx = fmaxf(mx0, mx1);
            }
            // The reference moves only when the tile raises the row max by
            // more than kRescaleLog2; then alpha rescales l and acc.
            const float m_tile = mx * cl2;                           // -inf if all masked
            const bool grow = m_tile > m_run + kRescaleLog2;
            const float m_new = grow ? m_tile : m_run;
            const float alpha = grow ? ex2(m_run - m_new) : 1.f;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no -inf - -inf
            const uint64_t neg2 = f2_pack(-m_use, -m_use);
            uint64_t acc2[2] = {0ull, 0ull};
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])), c2, neg2);
                float x0, x1;
                f2_unpack(x2, x0, x1);
                const float p0 = ex2(x0);
                const float p1 = ex2(x1);
                acc2[i & 1] = f2_add(acc2[i & 1], f2_pack(p0, p1));
                pk[i] = pack_bf16x2(p0, p1);
            }
            // The tile's largest weight as the MMA will see it (bf16): its
            // rounding goes into l_o, the normaliser of O.
            const float pmax = ex2(fmaf(mx, cl2, -m_use));
            const float pmax_b = __uint_as_float(pack_bf16x2(pmax, 0.f) << 16);
            tmem_st_x32(s_addr, pk);
            // A moved reference: rescale this warp's rows of O. S(j) was
            // issued after P(j-1) V(j-1), so that product has landed.
            if (j > 0 && __any_sync(0xffffffffu, grow)) {
                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
                for (int cc = 0; cc < C::D / 32; ++cc) {
                    uint32_t ov[32];
                    tmem_ld_x32(o_addr + cc * 32, ov);
                    tmem_ld_wait(ov);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float lo, hi;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(ov[2 * i]), __uint_as_float(ov[2 * i + 1])), a2, 0ull),
                                  lo, hi);
                        ov[2 * i] = __float_as_uint(lo);
                        ov[2 * i + 1] = __float_as_uint(hi);
                    }
                    tmem_st_x32(o_addr + cc * 32, ov);
                }
            }
            float sa, sb;
            f2_unpack(f2_add(acc2[0], acc2[1]), sa, sb);
            const float lsum = sa + sb;
            l_run = l_run * alpha + lsum;
            lo_run = lo_run * alpha + (lsum + (pmax_b - pmax));
            m_run = m_new;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(c.bar(C::P_FULL));
        }
        if (!ok) break;
        // Epilogue: O = acc / l_o in bf16, LSE = ln2 * (m + log2 l), once the
        // unit's last P V product has landed (O_DONE).
        if (!c.wait_warp(C::O_DONE, od)) break;
        ++od;
        tc_fence_after();
        const bool store = qrow < p.M;
        const float inv_l = (lo_run > 0.f) ? 1.f / lo_run : 0.f;
        const float lse_val = (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        const size_t row_idx = static_cast<size_t>(U.bh) * p.M + (store ? qrow : 0);
        uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + row_idx * C::D;   // bf16 bits
#pragma unroll 1
        for (int cc = 0; cc < C::D / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld_x32(o_addr + cc * 32, ov);
            tmem_ld_wait(ov);
            if (store) {
                uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(pack_bf16x2(__uint_as_float(ov[8 * i + 0]) * inv_l, __uint_as_float(ov[8 * i + 1]) * inv_l),
                                        pack_bf16x2(__uint_as_float(ov[8 * i + 2]) * inv_l, __uint_as_float(ov[8 * i + 3]) * inv_l),
                                        pack_bf16x2(__uint_as_float(ov[8 * i + 4]) * inv_l, __uint_as_float(ov[8 * i + 5]) * inv_l),
                                        pack_bf16x2(__uint_as_float(ov[8 * i + 6]) * inv_l, __uint_as_float(ov[8 * i + 7]) * inv_l));
            }
        }
        if (store) p.lse[row_idx] = lse_val;
        tc_fence_before();
        mbar_arrive(c.bar(C::O_FREE));
    }
}

template <bool CAUSAL>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::CTAS_PER_SM)
fa_fwd_bf16_q1_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const Bf16Params p) {
    using C = Cfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint32_t& tmem_base_sh = *reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    int& abort_sh = *reinterpret_cast<int*>(smem + C::MISC_OFF + 4);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_tiles = (p.M + C::BM - 1) / C::BM;
    Ctx c;
    c.bar0 = smem_u32(smem + C::BAR_OFF);
    c.sQ = smem + C::Q_OFF;
    c.sKV = smem + C::KV_OFF;
    c.abort = &abort_sh;
    c.err = p.err;
    c.ring = reinterpret_cast<volatile int*>(smem + C::RING_OFF);
    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int s = 0; s < C::NS; ++s) mbar_init(c.bar(C::KV_FULL + s), 1);
        for (int s = 0; s < C::ITERS; ++s) mbar_init(c.bar(C::ITER + s), 1);
        mbar_init(c.bar(C::Q_FULL), 1);
        mbar_init(c.bar(C::Q_EMPTY), 1);
        mbar_init(c.bar(C::P_FULL), 128 + 1);   // the softmax threads + the K/V gate
        mbar_init(c.bar(C::O_DONE), 1);
        mbar_init(c.bar(C::O_FREE), 128);
        mbar_init(c.bar(C::DRAIN), 1);
        for (int s = 0; s < C::UNIT_SLOTS; ++s) {
            mbar_init(c.bar(C::UNIT_FULL + s), 1);
            mbar_init(c.bar(C::UNIT_EMPTY + s), C::UNIT_READERS);
        }
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(&tmem_base_sh), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = tmem_base_sh;
    if (warp < 4) {
        setmaxnreg_inc<kRegsSoftmax>();
        softmax_role<CAUSAL>(p, c, n_tiles);
    } else {
        setmaxnreg_dec<kRegsOther>();
        if (warp == 4) {
            if (lane == 0) producer_role<CAUSAL>(&map_q, &map_k, &map_v, p, c, n_tiles);
        } else if (warp == 5) {
            if (lane == 0) mma_role<CAUSAL>(p, c, n_tiles);
        } else if (warp == 6) {
            if (lane == 0) gate_role<CAUSAL>(p, c, n_tiles);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(c.tmem, C::TMEM_COLS);
    }
    // The last CTA to finish resets the unit counter for the next launch that
    // uses it.
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            atomicExch(p.sched, 0);
            atomicExch(p.sched + 1, 0);
        }
    }
}

}  // namespace q1

// The D = 64 forward without key splits: maps of Q ({64, 128, 1} box) and of
// K and V ({64, 64, 1} boxes), 128-byte swizzle.
inline cudaError_t launch_bf16_q1(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const Bf16Params& p, bool causal, cudaStream_t stream, int sms) {
    using C = q1::Cfg;
    const int cap = sms * C::CTAS_PER_SM;
    const int grid = p.num_units < cap ? p.num_units : cap;   // persistent: four CTAs per SM
    auto kern = causal ? q1::fa_fwd_bf16_q1_kernel<true> : q1::fa_fwd_bf16_q1_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

}  // namespace fa
