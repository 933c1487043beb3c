// Backward pass of the bf16 forward on the tensor cores (tcgen05, TMA).
//
// "Module 08: FlashAttention and Memory-Efficient Kernels", section "The
// backward pass: recompute instead of store" and Code Step 6: every tile of P
// is rebuilt on chip as exp(S - L) from Q, K and the forward's per-row
// log-sum-exp L; nothing N x N is read or written. With that P and the
// output gradient dO:
//   dV = P^T dO,  dP = dO V^T,  Dl_i = sum_d dO_id O_id,
//   dS = P * (dP - Dl),  dQ = scale dS K,  dK = scale dS^T Q.
// Two kernels after the row dots Dl (bwd_rowdot, shared with the CUDA-core
// version), each over whole 128 x 128 tiles, bf16 operands, fp32
// accumulators in tensor memory:
//   bwd_tc_dkdv: one CTA per 128-key tile of a head. It computes the
//     transposed products S^T = K Q_i^T and dP^T = V dO_i^T, so that tensor-
//     memory lane t (rebuild thread t) owns key t: the thread rebuilds its
//     row of P^T and dS^T over the tile's 128 queries (L and Dl of those
//     queries staged in shared memory), writes both back as bf16 over the
//     first half of their own columns, and the MMA accumulates dV += P^T dO_i
//     and dK += dS^T Q_i with those as the A operand straight from tensor
//     memory. S^T of the next query tile is issued as soon as dV has read
//     P^T, dP^T of the next as soon as dK has read dS^T, so the rebuild of
//     one product's operand runs under the other's MMAs.
//   bwd_tc_dq: one CTA per 128-row query tile, the forward's orientation:
//     S = Q K_j^T, dP = dO V_j^T, dS into tensor memory over dP, dQ += dS
//     K_j; S of the next key tile is issued once the rebuild has read S.
// Each output is written by one CTA, so the result is deterministic and no
// atomics are needed; the price is that S and dP are computed twice (seven
// products per tile pair instead of five).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kT = 128;            // rows of every tile (queries or keys)
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
    // Warps [0, 4 NWG): NWG warpgroups that rebuild P and dS, each over W of
    // a tile's 128 columns, and write the results; then the TMA warp and the
    // MMA warp.
    static constexpr int NWG = 2;
    static constexpr int W = kT / NWG;                   // 64 columns per warpgroup
    static constexpr int TMA_WARP = 4 * NWG, MMA_WARP = 4 * NWG + 1;
    static constexpr int THREADS = 32 * (4 * NWG + 2);
    static constexpr int PANELS = (D + 63) / 64;         // 64-column TMA boxes per tile row
    static constexpr int PANEL = kT * 128;               // 128 rows x 128 B
    static constexpr int TILE = PANELS * PANEL;
    // A ring stage: two tiles (Q and dO, or K and V) and, in the dK/dV
    // kernel, the base-2 LSE and Dl of the stage's 128 queries.
    static constexpr int VEC = 2 * kT * 4;
    static constexpr int STAGE = 2 * TILE + 1024;
    static constexpr int STAGES = (D <= 64) ? 4 : 2;
    static constexpr int FIX_OFF = 0;                    // the CTA's resident pair (K and V, or Q and dO)
    static constexpr int RING_OFF = 2 * TILE;
    static constexpr int BAR_OFF = RING_OFF + STAGES * STAGE;
    // FULL[s]: stage s landed. DPE[s]: dP^T of the tile in stage s computed,
    // which also means the previous tile's dK product is done, so that
    // tile's stage is free (the rebuild and the producer both wait on it).
    // S_FULL: S^T landed; P_FULL, DS_FULL: the rebuild threads wrote P^T,
    // dS^T (NWG x 128 arrivals each).
    static constexpr int FIX_FULL = 0, FULL = 1, DPE = 1 + STAGES;
    static constexpr int S_FULL = 1 + 2 * STAGES, P_FULL = S_FULL + 1, DS_FULL = P_FULL + 1;
    static constexpr int DONE = DS_FULL + 1, DRAIN = DONE + 1;
    // The persistent dK/dV kernel: a unit's K and V no longer read
    // (FIX_EMPTY, a commit), its dV and dK read out of tensor memory by the
    // epilogue (ACC_FREE, NWG x 128 arrivals), and a ring of claimed units
    // (written by the TMA thread, read by the MMA thread and every rebuild
    // warp).
    static constexpr int FIX_EMPTY = DRAIN + 1, ACC_FREE = FIX_EMPTY + 1;
    static constexpr int UNIT_SLOTS = 4, UNIT_READERS = 4 * NWG + 1;
    static constexpr int UNIT_FULL = ACC_FREE + 1, UNIT_EMPTY = UNIT_FULL + UNIT_SLOTS;
    // OWN_P (D = 64, where tensor memory has room): P^T gets 64 columns of
    // its own, so S^T of the next tile can follow as soon as the rebuild has
    // read S^T (S_READ, NWG x 128 arrivals); P^T(k+1) is written once dV(k)
    // has read P^T(k) (P_FREE, a commit).
    static constexpr bool OWN_P = D == 64;
    static constexpr int S_READ = UNIT_EMPTY + UNIT_SLOTS, P_FREE = S_READ + 1;
    static constexpr int NUM_BARS = P_FREE + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;   // tensor-memory base, abort flag, unit ring
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 4 * UNIT_SLOTS + 1024;
    // Tensor memory of the dK/dV kernel: S^T (128 columns; warpgroup wg
    // writes its 64 queries of P^T, bf16 pairs, over columns [64 wg, 64 wg +
    // 32), inside what it read itself), dP^T (likewise dS^T), then dV, dK;
    // with OWN_P, P^T sits in its own 64 columns at TP (warpgroup wg at
    // [TP + 32 wg, TP + 32 wg + 32)) before the accumulators.
    static constexpr uint32_t TS = 0, TDP = 128, TP = 256, TACC = OWN_P ? 320 : 256;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t ID_SS = idesc_bf16_f32(128, kT, false);   // 128 x 128, both K-major
    static constexpr uint32_t ID_ACC = idesc_bf16_f32(128, D, true);    // 128 x D, B MN-major
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(TACC + 2 * D <= TMEM_COLS, "tensor memory");
};

struct BwdCtx {
    uint32_t bar0;
    volatile int* abort;
    uint32_t* err;
    __device__ uint32_t bar(int i) const { return bar0 + 8u * static_cast<uint32_t>(i); }
    __device__ bool wait(int i, int parity) const { return mbar_wait(bar(i), static_cast<uint32_t>(parity) & 1u, abort, err); }
    __device__ bool wait_warp(int i, int parity) const { return __all_sync(0xffffffffu, wait(i, parity)); }
};

// Loads one 128 x D tile (PANELS boxes of 64 columns) of head bh starting at
// row `row` into shared memory at `dst`; completion on `bar`.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar, int row, int bh,
                                          uint64_t pol) {
#pragma unroll
    for (int pn = 0; pn < BwdCfg<D>::PANELS; ++pn)
        tma_load_3d(dst + pn * BwdCfg<D>::PANEL, map, bar, pn * 64, row, bh, pol);
}

// Descriptor templates (zero start address; add address >> 4). K-major
// operand: a 16-column K-step advances 32 B inside a 64-column panel, four
// steps a panel. MN-major operand (its rows are the K dimension): LBO = the
// panel stride along N, SBO = 8 rows; a 16-row K-step advances 2048 B.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr) { return smem_desc_sw128(0, 16, 1024) + (addr >> 4); }
template <int D>
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t addr) {
    return smem_desc_sw128(0, BwdCfg<D>::PANEL, 1024) + (addr >> 4);
}
template <int D>
__device__ __forceinline__ uint32_t kstep(int kk) {
    return (kk >> 2) * (BwdCfg<D>::PANEL >> 4) + (kk & 3) * 2;
}

// D[128 x 128] = A[128 x D] B[128 x D]^T, both K-major tiles in shared memory.
template <int D>
__device__ __forceinline__ void mma_tile_nt(uint32_t d_tmem, uint32_t a, uint32_t b) {
    const uint64_t da = desc_kmajor(a), db = desc_kmajor(b);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(d_tmem, da + kstep<D>(kk), db + kstep<D>(kk), BwdCfg<D>::ID_SS, kk > 0 ? 1u : 0u);
}

// Acc[128 x D] (+)= A[128 x 128] (bf16 pairs in tensor memory) B[128 x D]
// (a tile in shared memory read MN-major: its rows are the K dimension). A's
// 16-column K-steps sit at a_tmem + 8 kk (SPLIT false: 64 contiguous
// columns) or, SPLIT, as two 32-column halves 64 columns apart (one per
// rebuild warpgroup).
template <int D, bool SPLIT>
__device__ __forceinline__ void mma_tile_acc(uint32_t acc, uint32_t a_tmem, uint32_t b, bool first) {
    const uint64_t db = desc_mnmajor<D>(b);
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk) {
        const uint32_t a = SPLIT ? a_tmem + (kk >> 2) * 64 + (kk & 3) * 8 : a_tmem + kk * 8;
        mma_ts(acc, a, db + kk * (2048 >> 4), BwdCfg<D>::ID_ACC, (first && kk == 0) ? 0u : 1u);
    }
}

// This thread's row of a 128 x D fp32 accumulator (its tensor-memory lane),
// times `mul`, to global memory; zeros when `have` is false.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t tm_acc, bool have, bool in, float* dst, float mul,
                                              int cc_lo = 0, int cc_hi = D / 32) {
#pragma unroll 1
    for (int cc = cc_lo; cc < cc_hi; ++cc) {
        uint32_t r[32];
        if (have) {
            tmem_ld_x32(tm_acc + cc * 32, r);
            tmem_ld_wait(r);
        }
        if (in) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
                if (have) {
                    w.x = __uint_as_float(r[4 * i + 0]) * mul;
                    w.y = __uint_as_float(r[4 * i + 1]) * mul;
                    w.z = __uint_as_float(r[4 * i + 2]) * mul;
                    w.w = __uint_as_float(r[4 * i + 3]) * mul;
                }
                *reinterpret_cast<float4*>(dst + cc * 32 + 4 * i) = w;
            }
        }
    }
}

// This thread's W = 64 columns of a 128-column fp32 buffer in tensor memory.
__device__ __forceinline__ void load_share(uint32_t taddr, uint32_t (&r)[64]) {
    tmem_ld_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tmem_ld_x32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tmem_ld_wait(r);
}

// p = exp2(s * cs - L2) over a share's 64 columns, zero outside columns
// [lo, hi) when MASK. L2 is per column (dK/dV kernel: `l2` points at the
// share's first query, 16-byte aligned) or per row (dQ kernel: l2_row).
template <bool PER_COLUMN, bool MASK>
__device__ __forceinline__ void rebuild_p(const uint32_t (&sr)[64], float cs, const float* l2, float l2_row, int lo,
                                          int hi, float (&pv)[64]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float lv[4];
        if (PER_COLUMN) {
            const float4 a = *reinterpret_cast<const float4*>(l2 + 4 * i);
            lv[0] = a.x, lv[1] = a.y, lv[2] = a.z, lv[3] = a.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) lv[e] = l2_row;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 4 * i + e;
            const float x = ex2(fmaf(__uint_as_float(sr[c]), cs, -lv[e]));
            pv[c] = (!MASK || (c >= lo && c < hi)) ? x : 0.f;
        }
    }
}

// p = exp2(s * cs - L2) over 32 columns with per-column L2 (16-byte
// aligned), zero outside columns [lo, hi) when MASK.
template <bool MASK>
__device__ __forceinline__ void rebuild_p32(const uint32_t (&sr)[32], float cs, const float* l2, int lo, int hi,
                                            float* pv) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 a = *reinterpret_cast<const float4*>(l2 + 4 * i);
        const float lv[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 4 * i + e;
            const float x = ex2(fmaf(__uint_as_float(sr[c]), cs, -lv[e]));
            pv[c] = (!MASK || (c >= lo && c < hi)) ? x : 0.f;
        }
    }
}

// ds = p (dp - Dl) over a share's 64 columns as 32 bf16 pairs; Dl per column
// (`dl`, 16-byte aligned) or per row (dl_row).
template <bool PER_COLUMN>
__device__ __forceinline__ void rebuild_ds(const float (&pv)[64], const uint32_t (&dr)[64], const float* dl,
                                           float dl_row, uint32_t (&dd)[32]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float dv[4];
        if (PER_COLUMN) {
            const float4 b = *reinterpret_cast<const float4*>(dl + 4 * i);
            dv[0] = b.x, dv[1] = b.y, dv[2] = b.z, dv[3] = b.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) dv[e] = dl_row;
        }
        float d[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) d[e] = pv[4 * i + e] * (__uint_as_float(dr[4 * i + e]) - dv[e]);
        dd[2 * i] = pack_bf16x2(d[0], d[1]);
        dd[2 * i + 1] = pack_bf16x2(d[2], d[3]);
    }
}

// One warpgroup's share of streamed tile k of the dK/dV kernel: P^T from
// S^T, then (once dP^T(k) has landed, DPE) dS^T from dP^T, each written as
// bf16 pairs over the first 32 of the 64 columns the warpgroup read (P^T:
// into its own columns with OWN_P, once dV(k-1) has read them). L2 and Dl
// per column (`l2`, `dl`: the share's first query, 16-byte aligned).
// Returns false if a wait gave up.
template <int D>
__device__ __forceinline__ bool rebuild_dkdv(const BwdCtx& c, int wg, int k, uint32_t ts, uint32_t tdp, float cs,
                                             const float* l2, const float* dl, int lo, int hi) {
    using C = BwdCfg<D>;
    // P in two halves of 32 queries (fewer live registers); both halves are
    // read before P^T is written over the first of them.
    float pv[64];
    const bool full = lo <= 0 && hi >= 64;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t sr[32];
        tmem_ld_x32(ts + 64 * wg + 32 * h, sr);
        tmem_ld_wait(sr);
        if (C::OWN_P && h == 1) {   // S^T read: the next tile's S^T may follow
            tc_fence_before();
            mbar_arrive(c.bar(C::S_READ));
        }
        if (full)
            rebuild_p32<false>(sr, cs, l2 + 32 * h, lo - 32 * h, hi - 32 * h, pv + 32 * h);
        else
            rebuild_p32<true>(sr, cs, l2 + 32 * h, lo - 32 * h, hi - 32 * h, pv + 32 * h);
    }
    {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(pv[2 * i], pv[2 * i + 1]);
        if (C::OWN_P) {
            if (k > 0) {
                if (!c.wait_warp(C::P_FREE, k - 1)) return false;
                tc_fence_after();
            }
            tmem_st_x32(ts + C::TP + 32 * wg, pk);
        } else {
            tmem_st_x32(ts + 64 * wg, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(c.bar(C::P_FULL));
    }
    if (!c.wait_warp(C::DPE + k % C::STAGES, k / C::STAGES)) return false;
    tc_fence_after();
    // Two halves of 32 queries (fewer live registers): half h reads dP^T
    // columns [32 h, 32 h + 32) of the share and writes its 16 columns of dS^T
    // at [16 h, 16 h + 16), which half 0 has already read.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t dr[32], dd[16];
        tmem_ld_x32(tdp + 64 * wg + 32 * h, dr);
        tmem_ld_wait(dr);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 b4 = *reinterpret_cast<const float4*>(dl + 32 * h + 4 * i);
            const float dv[4] = {b4.x, b4.y, b4.z, b4.w};
            float q[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) q[e] = pv[32 * h + 4 * i + e] * (__uint_as_float(dr[4 * i + e]) - dv[e]);
            dd[2 * i] = pack_bf16x2(q[0], q[1]);
            dd[2 * i + 1] = pack_bf16x2(q[2], q[3]);
        }
        tmem_st_x16(tdp + 64 * wg + 16 * h, dd);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(c.bar(C::DS_FULL));
    return true;
}

// Shared prologue: barriers, tensor memory.
template <int D>
__device__ __forceinline__ uint32_t bwd_setup(const BwdCtx& c, uint32_t* misc) {
    using C = BwdCfg<D>;
    if (threadIdx.x == 0) {
        mbar_init(c.bar(C::FIX_FULL), 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(c.bar(C::FULL + s), 1);
            mbar_init(c.bar(C::DPE + s), 1);
        }
        mbar_init(c.bar(C::S_FULL), 1);
        mbar_init(c.bar(C::P_FULL), C::NWG * kT);
        mbar_init(c.bar(C::DS_FULL), C::NWG * kT);
        mbar_init(c.bar(C::DONE), 1);
        mbar_init(c.bar(C::DRAIN), 1);
        mbar_init(c.bar(C::FIX_EMPTY), 1);
        mbar_init(c.bar(C::ACC_FREE), C::NWG * kT);
        mbar_init(c.bar(C::S_READ), C::NWG * kT);
        mbar_init(c.bar(C::P_FREE), 1);
        for (int s = 0; s < C::UNIT_SLOTS; ++s) {
            mbar_init(c.bar(C::UNIT_FULL + s), 1);
            mbar_init(c.bar(C::UNIT_EMPTY + s), C::UNIT_READERS);
        }
        misc[1] = 0;
        fence_barrier_init();
    }
    if (threadIdx.x / 32 == C::MMA_WARP) {
        tmem_alloc(smem_u32(misc), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return misc[0];
}

template <int D>
__device__ __forceinline__ void bwd_teardown(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x / 32 == BwdCfg<D>::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, BwdCfg<D>::TMEM_COLS);
    }
}

// A unit of the dK/dV kernel: one 128-key tile of a head and the query
// tiles that see it. Causal units come in groups of 8 heads, key tile 0
// (the most query tiles) first, so that the last units to be claimed are the
// shortest while the streamed Q and dO tiles of the heads in flight stay in
// L2.
struct DkdvUnit {
    int bh, kt, nq;
};

__device__ __forceinline__ DkdvUnit dkdv_unit(int u, const BwdParams& p, int ktiles, int mtiles) {
    DkdvUnit U;
    if (p.causal) {
        constexpr int kHeads = 8;
        const int gu = kHeads * ktiles;
        const int g = u / gu, r = u - g * gu;
        const int hg = min(kHeads, p.bh_count - g * kHeads);
        U.kt = r / hg;
        U.bh = g * kHeads + r % hg;
    } else {
        U.bh = u / ktiles;
        U.kt = u - U.bh * ktiles;
    }
    const int i0 = p.causal ? U.kt : 0;   // query tiles with rows >= the tile's first key
    U.nq = mtiles > i0 ? mtiles - i0 : 0;
    return U;
}

// Reads the CTA's sequence of units from the ring (-1 when there are no
// more, or a wait gave up).
template <int D>
struct DkdvUnitReader {
    int k = 0;
    __device__ __forceinline__ int next(const BwdCtx& c, const volatile int* ring, bool whole_warp) {
        using C = BwdCfg<D>;
        const int slot = k % C::UNIT_SLOTS, phase = k / C::UNIT_SLOTS;
        ++k;
        const bool ok = whole_warp ? c.wait_warp(C::UNIT_FULL + slot, phase) : c.wait(C::UNIT_FULL + slot, phase);
        if (!ok) return -1;
        const int u = ring[slot];
        if (whole_warp) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(c.bar(C::UNIT_EMPTY + slot));
        } else {
            mbar_arrive(c.bar(C::UNIT_EMPTY + slot));
        }
        return u;
    }
};

// ------------------------------------------------------------ dK, dV kernel
// Persistent: one CTA per SM claims units (its own index first, then from
// the launch's work counter). The TMA thread loads a unit's K and V once it
// has claimed it and the previous unit's last S^T and dP^T products are done
// (FIX_EMPTY), so that load, and the next unit's first products, overlap
// the previous unit's last tile and its epilogue; the stage ring and every
// per-tile barrier run on over unit boundaries.
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
bwd_tc_dkdv(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(sm);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
    volatile int* ring = reinterpret_cast<volatile int*>(misc + 4);
    BwdCtx c;
    c.bar0 = s0 + C::BAR_OFF;
    c.abort = reinterpret_cast<volatile int*>(misc + 1);
    c.err = p.err;
    const int warp = threadIdx.x / 32;
    const int ktiles = (p.N + kT - 1) / kT;
    const int mtiles = p.Mpad / kT;
    const int units = p.bh_count * ktiles;
    const uint32_t tmem = bwd_setup<D>(c, misc);
    if (warp < C::TMA_WARP) {
        // Thread t of warpgroup wg owns key key0 + t (tensor-memory lane t)
        // and queries [W wg, W wg + W) of every streamed tile.
        const int wg = warp >> 2, t = threadIdx.x & 127;
        const uint32_t tm = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const float cs = p.scale * kLog2e;
        constexpr int kHalfWg = C::NWG / 2, kPer = (D / 32 + kHalfWg - 1) / kHalfWg;
        const int part = wg % kHalfWg;
        const int clo = min(D / 32, part * kPer), chi = min(D / 32, clo + kPer);
        DkdvUnitReader<D> units_in;
        int kg = 0, uc = 0;   // streamed tiles and non-empty units so far
        bool ok = true;
        while (ok) {
            const int u = units_in.next(c, ring, true);
            if (u < 0) break;
            const DkdvUnit U = dkdv_unit(u, p, ktiles, mtiles);
            const int key = U.kt * kT + t;
            const int i0 = p.causal ? U.kt : 0;
            const bool in = key < p.N;
#pragma unroll 1
            for (int k = 0; k < U.nq && ok; ++k) {
                const int g = kg + k, s = g % C::STAGES;
                const int q0 = (i0 + k) * kT + C::W * wg;   // this share's first query
                // The stage's LSE2 / Dl arrived with its tiles (FULL), which
                // the MMA thread waited for before S_FULL; wait here too so
                // that the copies are visible to this thread.
                if (!c.wait_warp(C::FULL + s, g / C::STAGES) || !c.wait_warp(C::S_FULL, g)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float* l2 =
                    reinterpret_cast<const float*>(sm + C::RING_OFF + s * C::STAGE + 2 * C::TILE) + C::W * wg;
                const float* dl = l2 + kT;
                // Visible queries: column c with q0 + c >= key (causal); rows
                // past M have L2 = +inf; a key past N sees nothing.
                const int lo = p.causal ? key - q0 : 0;
                const int hi = in ? C::W : 0;
                ok = rebuild_dkdv<D>(c, wg, g, tm + C::TS, tm + C::TDP, cs, l2, dl, lo, hi);
            }
            if (!ok) break;
            if (U.nq > 0) {
                if (!c.wait_warp(C::DONE, uc)) break;
                tc_fence_after();
            }
            // The first half of the warpgroups writes dV, the second dK, each
            // a share of the chunks (zeros for a key no query sees). One call
            // site: two inlined copies kept more registers live and spilled.
            const bool second = wg >= kHalfWg;
            float* dst = (second ? p.dk : p.dv) + (static_cast<int64_t>(U.bh) * p.N + key) * D;
            store_acc_row<D>(tm + C::TACC + (second ? static_cast<uint32_t>(D) : 0u), U.nq > 0, in, dst,
                             second ? p.scale : 1.f, clo, chi);
            if (U.nq > 0) {
                tc_fence_before();
                mbar_arrive(c.bar(C::ACC_FREE));
                kg += U.nq;
                ++uc;
            }
        }
    } else if (warp == C::TMA_WARP) {
        if ((threadIdx.x & 31) == 0) {
            const uint64_t pol = policy_evict_last();
            int claimed = 0;
            auto claim = [&]() -> int {
                const int slot = claimed % C::UNIT_SLOTS;
                if (claimed >= C::UNIT_SLOTS && !c.wait(C::UNIT_EMPTY + slot, claimed / C::UNIT_SLOTS - 1)) return -2;
                int v = (claimed == 0) ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(p.sched, 1);
                if (v >= units) v = -1;
                ring[slot] = v;
                mbar_arrive(c.bar(C::UNIT_FULL + slot));
                ++claimed;
                return v;
            };
            int sg = 0, uf = 0;   // stages issued, non-empty units loaded
            bool ok = true;
            int u = claim();
            while (u >= 0 && ok) {
                const int u_next = claim();   // one ahead: the other roles see it early
                if (u_next == -2) break;
                const DkdvUnit U = dkdv_unit(u, p, ktiles, mtiles);
                if (U.nq > 0) {
                    const int i0 = p.causal ? U.kt : 0;
                    if (uf > 0 && !c.wait(C::FIX_EMPTY, uf - 1)) break;
                    mbar_arrive_expect_tx(c.bar(C::FIX_FULL), 2 * C::TILE);
                    load_tile<D>(s0 + C::FIX_OFF, &map_k, c.bar(C::FIX_FULL), U.kt * kT, U.bh, pol);
                    load_tile<D>(s0 + C::FIX_OFF + C::TILE, &map_v, c.bar(C::FIX_FULL), U.kt * kT, U.bh, pol);
                    const int64_t vec_row = static_cast<int64_t>(U.bh) * p.Mpad + i0 * kT;
#pragma unroll 1
                    for (int k = 0; k < U.nq; ++k) {
                        const int g = sg + k, s = g % C::STAGES;
                        // Stage s last held tile g - STAGES, whose dK product is
                        // done once dP^T(g - STAGES + 1) is.
                        const int f = g - C::STAGES + 1;
                        if (g >= C::STAGES && !c.wait(C::DPE + f % C::STAGES, f / C::STAGES)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = s0 + C::RING_OFF + s * C::STAGE;
                        mbar_arrive_expect_tx(c.bar(C::FULL + s), 2 * C::TILE + C::VEC);
                        load_tile<D>(dst, &map_q, c.bar(C::FULL + s), (i0 + k) * kT, U.bh, pol);
                        load_tile<D>(dst + C::TILE, &map_do, c.bar(C::FULL + s), (i0 + k) * kT, U.bh, pol);
                        bulk_load(dst + 2 * C::TILE, p.lse2 + vec_row + k * kT, kT * 4, c.bar(C::FULL + s));
                        bulk_load(dst + 2 * C::TILE + kT * 4, p.delta + vec_row + k * kT, kT * 4, c.bar(C::FULL + s));
                    }
                    if (!ok) break;
                    sg += U.nq;
                    ++uf;
                }
                u = u_next;
            }
            // Every copy issued must land before shared memory is released.
            if (uf > 0) mbar_wait_drain(c.bar(C::FIX_FULL), (uf - 1) & 1);
            for (int s = 0; s < C::STAGES && s < sg; ++s) {
                const int last = s + ((sg - 1 - s) / C::STAGES) * C::STAGES;
                mbar_wait_drain(c.bar(C::FULL + s), (last / C::STAGES) & 1);
            }
        }
    } else if ((threadIdx.x & 31) == 0) {
        // MMA thread. Per streamed query tile k of a unit, in this order:
        //   dV += P^T(k) dO(k)        once the rebuild wrote P^T over S^T
        //   S^T(k+1) = K Q(k+1)^T     S's columns are free once dV(k) read P^T
        //   dK += dS^T(k) Q(k)        once the rebuild wrote dS^T over dP^T
        //   dP^T(k+1) = V dO(k+1)^T   dP's columns are free once dK(k) read dS^T
        // so the rebuild of tile k+1's P overlaps dK(k) and dP^T(k+1), and its
        // dS overlaps dV(k+1) and S^T(k+2). One thread's MMAs run in issue
        // order, which is what makes each overwrite safe, and why DPE (the
        // commit after dP^T(k+1)) also frees tile k's stage. A unit's first
        // dV overwrites the accumulators, so it waits for the previous unit's
        // epilogue (ACC_FREE).
        const uint32_t kt_s = s0 + C::FIX_OFF, vt_s = kt_s + C::TILE;
        auto stage = [&](int g) -> uint32_t { return s0 + C::RING_OFF + (g % C::STAGES) * C::STAGE; };
        auto issue_s = [&](int g) -> bool {
            if (!c.wait(C::FULL + g % C::STAGES, g / C::STAGES)) return false;
            tc_fence_after();
            mma_tile_nt<D>(tmem + C::TS, kt_s, stage(g));
            mma_commit(c.bar(C::S_FULL));
            return true;
        };
        auto issue_dp = [&](int g) {
            mma_tile_nt<D>(tmem + C::TDP, vt_s, stage(g) + C::TILE);
            mma_commit(c.bar(C::DPE + g % C::STAGES));
        };
        DkdvUnitReader<D> units_in;
        int kg = 0, uf = 0;
        bool ok = true;
        while (ok) {
            const int u = units_in.next(c, ring, false);
            if (u < 0) break;
            const DkdvUnit U = dkdv_unit(u, p, ktiles, mtiles);
            if (U.nq == 0) continue;
            if (!c.wait(C::FIX_FULL, uf)) break;
            tc_fence_after();
            if (!issue_s(kg)) break;
            issue_dp(kg);
            if (U.nq == 1) mma_commit(c.bar(C::FIX_EMPTY));   // K and V read by S^T(0), dP^T(0) only
#pragma unroll 1
            for (int k = 0; k < U.nq; ++k) {
                const int g = kg + k;
                const uint32_t qt = stage(g), dot = qt + C::TILE;
                // OWN_P: S^T(k+1) as soon as the rebuild has read S^T(k).
                if (C::OWN_P && k + 1 < U.nq && (!c.wait(C::S_READ, g) || !issue_s(g + 1))) {
                    ok = false;
                    break;
                }
                if (!c.wait(C::P_FULL, g) || (k == 0 && uf > 0 && !c.wait(C::ACC_FREE, uf - 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (C::OWN_P) {
                    mma_tile_acc<D, false>(tmem + C::TACC, tmem + C::TP, dot, k == 0);
                    mma_commit(c.bar(C::P_FREE));
                } else {
                    mma_tile_acc<D, true>(tmem + C::TACC, tmem + C::TS, dot, k == 0);
                    if (k + 1 < U.nq && !issue_s(g + 1)) {
                        ok = false;
                        break;
                    }
                }
                if (!c.wait(C::DS_FULL, g)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                mma_tile_acc<D, true>(tmem + C::TACC + D, tmem + C::TDP, qt, k == 0);
                if (k == U.nq - 1) mma_commit(c.bar(C::DONE));
                if (k + 1 < U.nq) {
                    issue_dp(g + 1);
                    if (k + 2 == U.nq) mma_commit(c.bar(C::FIX_EMPTY));   // the unit's last K, V reads
                }
            }
            kg += U.nq;
            ++uf;
        }
        mma_commit(c.bar(C::DRAIN));
        mbar_wait_drain(c.bar(C::DRAIN), 0);
    }
    bwd_teardown<D>(tmem);
    // The last CTA to finish resets the unit counter for the next launch
    // that uses it; every CTA's claims precede its count here.
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            atomicExch(p.sched, 0);
            atomicExch(p.sched + 1, 0);
        }
    }
}

// --------------------------------------------------------------- dQ kernel
// Its own layout: Q and dO resident; K and V in separate rings, since V(j)
// is last read by dP(j) while K(j) stays until dQ(j) (with one ring of two
// K/V stages at D = 128 the next tile's S waited for its load); dS in its
// own tensor-memory columns, so that S(j+1) and dP(j+1) can follow as soon
// as the rebuild has read S(j) and dP(j). The MMA thread's barrier
// operations cost it ~100 cycles each while the tensor core streams shared
// memory, so every barrier here serves as many waiters as it can:
//   KFULL[s]  K(j) and V(j) landed (one barrier per K slot)
//   SDP[v]    S(j) and dP(j) computed, V slot v free (one per V slot)
//   KEMPTY[s] dQ(j) done: K slot s free and dS's columns free
//   DP_READ   the rebuild has read S(j) and dP(j)
//   DS_FULL   the rebuild has written dS(j)
template <int D>
struct DqCfg {
    using B = BwdCfg<D>;
    static constexpr int KST = (D <= 64) ? 4 : 3;        // K ring stages
    static constexpr int VST = (D <= 64) ? 4 : 2;        // V ring stages
    static constexpr int FIX_OFF = 0;                    // Q, dO
    static constexpr int K_OFF = 2 * B::TILE;
    static constexpr int V_OFF = K_OFF + KST * B::TILE;
    static constexpr int BAR_OFF = V_OFF + VST * B::TILE;
    static constexpr int FIX_FULL = 0, KFULL = 1, KEMPTY = KFULL + KST, SDP = KEMPTY + KST;
    static constexpr int DP_READ = SDP + VST, DS_FULL = DP_READ + 1, DONE = DS_FULL + 1, DRAIN = DONE + 1;
    static constexpr int NUM_BARS = DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
    // Tensor memory: S, dP (128 columns each), dS (bf16 pairs, 64), dQ (D).
    static constexpr uint32_t TS = 0, TDP = 128, TDS = 256, TACC = 320;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(TACC + D <= B::TMEM_COLS, "tensor memory");
};

template <int D>
__device__ __forceinline__ uint32_t dq_setup(const BwdCtx& c, uint32_t* misc) {
    using C = DqCfg<D>;
    if (threadIdx.x == 0) {
        mbar_init(c.bar(C::FIX_FULL), 1);
        for (int s = 0; s < C::KST; ++s) {
            mbar_init(c.bar(C::KFULL + s), 1);
            mbar_init(c.bar(C::KEMPTY + s), 1);
        }
        for (int s = 0; s < C::VST; ++s) mbar_init(c.bar(C::SDP + s), 1);
        mbar_init(c.bar(C::DP_READ), BwdCfg<D>::NWG * kT);
        mbar_init(c.bar(C::DS_FULL), BwdCfg<D>::NWG * kT);
        mbar_init(c.bar(C::DONE), 1);
        mbar_init(c.bar(C::DRAIN), 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (threadIdx.x / 32 == BwdCfg<D>::MMA_WARP) {
        tmem_alloc(smem_u32(misc), BwdCfg<D>::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return misc[0];
}

// TMA thread of the dQ kernel: Q and dO once, then K(j) and V(j) of the
// n streamed key tiles into their rings, both signalled on K(j)'s slot.
template <int D>
__device__ __forceinline__ void dq_producer(const BwdCtx& c, uint32_t s0, const CUtensorMap* mq, const CUtensorMap* mdo,
                                            int r0, const CUtensorMap* mk, const CUtensorMap* mv, int n, int bh) {
    using C = DqCfg<D>;
    using B = BwdCfg<D>;
    const uint64_t pol = policy_evict_last();
    mbar_arrive_expect_tx(c.bar(C::FIX_FULL), 2 * B::TILE);
    load_tile<D>(s0 + C::FIX_OFF, mq, c.bar(C::FIX_FULL), r0, bh, pol);
    load_tile<D>(s0 + C::FIX_OFF + B::TILE, mdo, c.bar(C::FIX_FULL), r0, bh, pol);
    int kn = 0;
#pragma unroll 1
    for (int j = 0; j < n; ++j) {
        const int ks = j % C::KST, vs = j % C::VST;
        // K slot: free once dQ(j - KST) is done; V slot: once dP(j - VST) is.
        if (j >= C::KST && !c.wait(C::KEMPTY + ks, j / C::KST - 1)) break;
        if (j >= C::VST && !c.wait(C::SDP + vs, j / C::VST - 1)) break;
        mbar_arrive_expect_tx(c.bar(C::KFULL + ks), 2 * B::TILE);
        load_tile<D>(s0 + C::K_OFF + ks * B::TILE, mk, c.bar(C::KFULL + ks), j * kT, bh, pol);
        load_tile<D>(s0 + C::V_OFF + vs * B::TILE, mv, c.bar(C::KFULL + ks), j * kT, bh, pol);
        ++kn;
    }
    mbar_wait_drain(c.bar(C::FIX_FULL), 0);
    for (int s = 0; s < C::KST && s < kn; ++s) {
        const int last = s + ((kn - 1 - s) / C::KST) * C::KST;
        mbar_wait_drain(c.bar(C::KFULL + s), (last / C::KST) & 1);
    }
}

template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
bwd_tc_dq(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
          const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
    using B = BwdCfg<D>;
    using C = DqCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(sm);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
    BwdCtx c;
    c.bar0 = s0 + C::BAR_OFF;
    c.abort = reinterpret_cast<volatile int*>(misc + 1);
    c.err = p.err;
    const int warp = threadIdx.x / 32;
    const int mtiles = p.Mpad / kT;
    const int bh = static_cast<int>(blockIdx.x / mtiles);
    const int r0 = static_cast<int>(blockIdx.x % mtiles) * kT;
    // Key tiles any row of this tile sees: all, or (causal) keys up to its
    // last row.
    const int kend = p.causal ? min(p.N, min(p.M, r0 + kT)) : p.N;
    const int nk = (kend + kT - 1) / kT;
    const uint32_t tmem = dq_setup<D>(c, misc);
    if (warp < B::TMA_WARP) {
        // Thread t of warpgroup wg owns query row r0 + t (tensor-memory lane
        // t) and keys [W wg, W wg + W) of every streamed tile.
        const int wg = warp >> 2, t = threadIdx.x & 127;
        const int row = r0 + t;
        const uint32_t tm = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const float cs = p.scale * kLog2e;
        const int64_t prow = static_cast<int64_t>(bh) * p.Mpad + row;
        const float l2 = p.lse2[prow], dl = p.delta[prow];   // +inf / 0 past M
        const int lim = p.causal ? min(p.N, row + 1) : p.N;   // keys [0, lim) visible
        bool ok = true;
#pragma unroll 1
        for (int j = 0; j < nk && ok; ++j) {
            if (!c.wait_warp(C::SDP + j % C::VST, j / C::VST)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int hi = lim - (j * kT + B::W * wg);   // this share's keys: j * 128 + W wg + column
            float pv[64];
            uint32_t dd[32];
            {
                uint32_t sr[64], dr[64];
                load_share(tm + C::TS + 64 * wg, sr);
                load_share(tm + C::TDP + 64 * wg, dr);
                tc_fence_before();
                mbar_arrive(c.bar(C::DP_READ));
                if (hi >= 64)
                    rebuild_p<false, false>(sr, cs, nullptr, l2, 0, hi, pv);
                else
                    rebuild_p<false, true>(sr, cs, nullptr, l2, 0, hi, pv);
                rebuild_ds<false>(pv, dr, nullptr, dl, dd);
            }
            // dS(j-1) must have been read by dQ(j-1) before it is overwritten.
            if (j > 0) {
                if (!c.wait_warp(C::KEMPTY + (j - 1) % C::KST, (j - 1) / C::KST)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            tmem_st_x32(tm + C::TDS + 32 * wg, dd);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(c.bar(C::DS_FULL));
        }
        if (ok && nk > 0) {
            ok = c.wait_warp(C::DONE, 0);
            tc_fence_after();
        }
        if (ok) {   // each warpgroup writes a share of the row's 32-column chunks
            constexpr int kPer = (D / 32 + B::NWG - 1) / B::NWG;
            const int clo = min(D / 32, wg * kPer), chi = min(D / 32, clo + kPer);
            store_acc_row<D>(tm + C::TACC, nk > 0, row < p.M, p.dq + (static_cast<int64_t>(bh) * p.M + row) * D,
                             p.scale, clo, chi);
        }
    } else if (warp == B::TMA_WARP) {
        if ((threadIdx.x & 31) == 0 && nk > 0) dq_producer<D>(c, s0, &map_q, &map_do, r0, &map_k, &map_v, nk, bh);
    } else if ((threadIdx.x & 31) == 0) {
        // MMA thread. Per streamed key tile j, in this order:
        //   S(j+1) = Q K(j+1)^T, dP(j+1) = dO V(j+1)^T   once the rebuild has
        //                                                 read S(j) and dP(j)
        //   dQ += dS(j) K(j)                              once it wrote dS(j)
        // so both products of tile j+1 run during tile j's rebuild.
        bool ok = nk > 0 && c.wait(C::FIX_FULL, 0);
        const uint32_t qt = s0 + C::FIX_OFF, dot = qt + B::TILE;
        auto kslot = [&](int j) -> uint32_t { return s0 + C::K_OFF + (j % C::KST) * B::TILE; };
        auto issue_sdp = [&](int j) -> bool {
            if (!c.wait(C::KFULL + j % C::KST, j / C::KST)) return false;
            tc_fence_after();
            mma_tile_nt<D>(tmem + C::TS, qt, kslot(j));
            mma_tile_nt<D>(tmem + C::TDP, dot, s0 + C::V_OFF + (j % C::VST) * B::TILE);
            mma_commit(c.bar(C::SDP + j % C::VST));
            return true;
        };
        if (ok) ok = issue_sdp(0);
#pragma unroll 1
        for (int j = 0; ok && j < nk; ++j) {
            if (j + 1 < nk && (!c.wait(C::DP_READ, j) || !issue_sdp(j + 1))) break;
            if (!c.wait(C::DS_FULL, j)) break;
            tc_fence_after();
            mma_tile_acc<D, false>(tmem + C::TACC, tmem + C::TDS, kslot(j), j == 0);
            mma_commit(c.bar(C::KEMPTY + j % C::KST));
            if (j == nk - 1) mma_commit(c.bar(C::DONE));
        }
        mma_commit(c.bar(C::DRAIN));
        mbar_wait_drain(c.bar(C::DRAIN), 0);
    }
    bwd_teardown<D>(tmem);
}

template <int D>
cudaError_t launch_bwd_tc_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                            const BwdParams& p, cudaStream_t s) {
    using C = BwdCfg<D>;
    const int64_t kv_blocks = static_cast<int64_t>(p.bh_count) * ((p.N + kT - 1) / kT);
    const int64_t q_blocks = static_cast<int64_t>(p.bh_count) * (p.Mpad / kT);
    if (kv_blocks > 0x7fffffffLL || q_blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // Set on every call: the attribute belongs to the current device's context.
    cudaError_t e = cudaFuncSetAttribute(bwd_tc_dkdv<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd_tc_dq<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (kv_blocks > 0) {
        if (p.sched == nullptr) return cudaErrorInvalidValue;   // the persistent kernel needs its counters
        int dev = 0, sms = 0;
        e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int64_t grid = kv_blocks < sms ? kv_blocks : sms;   // persistent: one CTA per SM
        bwd_tc_dkdv<D><<<static_cast<unsigned>(grid), C::THREADS, C::SMEM_BYTES, s>>>(q, k, v, dout, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    bwd_tc_dq<D><<<static_cast<unsigned>(q_blocks), C::THREADS, DqCfg<D>::SMEM_BYTES, s>>>(q, k, v, dout, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                          const BwdParams& p, cudaStream_t s) {
    switch (p.D) {
        case 64: return launch_bwd_tc_t<64>(q, k, v, dout, p, s);
        case 96: return launch_bwd_tc_t<96>(q, k, v, dout, p, s);
        case 128: return launch_bwd_tc_t<128>(q, k, v, dout, p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
