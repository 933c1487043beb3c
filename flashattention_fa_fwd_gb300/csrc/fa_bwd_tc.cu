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
// version), each over 128 x 128 tiles, bf16 operands, fp32 accumulators in
// tensor memory:
//   bwd_tc_dkdv: one CTA per 128-key tile of a head. It computes the
//     transposed products S^T = K Q_i^T and dP^T = V dO_i^T, so that tensor-
//     memory lane t (softmax thread t) owns key t: the thread rebuilds its row
//     of P^T and dS^T over the tile's 128 queries (L and Dl of those queries
//     staged in shared memory), writes both back as bf16 over their own
//     columns, and the MMA accumulates dV += P^T dO_i and dK += dS^T Q_i with
//     those as the A operand straight from tensor memory.
//   bwd_tc_dq: one CTA per 128-row query tile, the forward's orientation:
//     S = Q K_j^T, dP = dO V_j^T, dS into tensor memory, dQ += dS K_j.
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
    // a buffer's 64 columns, and write the results; then the TMA warp and the
    // MMA warp. (Four warpgroups of 16 columns measured slower than two of 32
    // at D = 64 as well as at D = 128.)
    static constexpr int NWG = 2;
    static constexpr int W = 64 / NWG;
    static_assert(W == 32, "the rebuild moves 32 columns per tensor-memory load");
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
    static constexpr int FIX_FULL = 0, FULL = 1, EMPTY = 1 + STAGES, S_FULL = 1 + 2 * STAGES;   // S_FULL, P_FULL: one per S buffer
    static constexpr int P_FULL = S_FULL + 2, S_READ = P_FULL + 2, DONE = S_READ + 2, DRAIN = DONE + 1;
    static constexpr int NUM_BARS = DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;
    // Every 128-row streamed tile is handled as two 64-row halves, each with
    // its own S and dP buffer, so that one half's rebuild of P and dS runs
    // while the other half's products are computed. Tensor memory: S buffers
    // (then P, bf16 pairs in their first 32 columns) at 0 and 64, dP buffers
    // (then dS) at 128 and 192, then the accumulators (dV and dK, or dQ).
    static constexpr int HALF_ROWS = 64;
    static constexpr int HALF_BYTES = HALF_ROWS * 128;   // a half's row offset inside every panel
    static constexpr uint32_t TS = 0, TDP = 128, TACC = 256;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t ID_SS = idesc_bf16_f32(128, HALF_ROWS, false);  // 128 x 64, both K-major
    static constexpr uint32_t ID_ACC = idesc_bf16_f32(128, D, true);     // 128 x D, B MN-major
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

// D[128 x 64] = A[128 x D] B[64 x D]^T, both K-major in shared memory (B:
// half a tile, `b` already offset to its first row).
template <int D>
__device__ __forceinline__ void mma_tile_nt(uint32_t d_tmem, uint32_t a, uint32_t b) {
    const uint64_t da = desc_kmajor(a), db = desc_kmajor(b);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(d_tmem, da + kstep<D>(kk), db + kstep<D>(kk), BwdCfg<D>::ID_SS, kk > 0 ? 1u : 0u);
}

// Acc[128 x D] (+)= A[128 x 64] (bf16 pairs in tensor memory) B[64 x D]
// (half a tile in shared memory read MN-major: its rows are the K dimension).
template <int D>
__device__ __forceinline__ void mma_tile_acc(uint32_t acc, uint32_t a_tmem, uint32_t b, bool first) {
    const uint64_t db = desc_mnmajor<D>(b);
#pragma unroll
    for (int kk = 0; kk < BwdCfg<D>::HALF_ROWS / 16; ++kk)
        mma_ts(acc, a_tmem + kk * 8, db + kk * (2048 >> 4), BwdCfg<D>::ID_ACC, (first && kk == 0) ? 0u : 1u);
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

// Rebuilds W columns of this thread's row of P and dS from S and dP in
// tensor memory: p = exp2(s * cs - L2), zero outside columns [lo, hi) of the
// share when MASK; ds = p (dp - Dl). L2 and Dl are per column (dK/dV kernel,
// `l2` and `dl` pointing at the share's first column, 16-byte aligned) or
// per row (dQ kernel).
template <int W, bool PER_COLUMN, bool MASK>
__device__ __forceinline__ void rebuild_chunk(const uint32_t (&sr)[W], const uint32_t (&dr)[W], float cs,
                                              const float* l2, const float* dl, float l2_row, float dl_row, int lo,
                                              int hi, uint32_t (&pp)[W / 2], uint32_t (&dd)[W / 2]) {
#pragma unroll
    for (int i = 0; i < W / 4; ++i) {
        float lv[4], dv[4];
        if (PER_COLUMN) {
            const float4 a = *reinterpret_cast<const float4*>(l2 + 4 * i);
            const float4 b = *reinterpret_cast<const float4*>(dl + 4 * i);
            lv[0] = a.x, lv[1] = a.y, lv[2] = a.z, lv[3] = a.w;
            dv[0] = b.x, dv[1] = b.y, dv[2] = b.z, dv[3] = b.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) lv[e] = l2_row, dv[e] = dl_row;
        }
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = 4 * i + e;
            pv[e] = ex2(fmaf(__uint_as_float(sr[c]), cs, -lv[e]));
            if (MASK) pv[e] = (c >= lo && c < hi) ? pv[e] : 0.f;
        }
        pp[2 * i] = pack_bf16x2(pv[0], pv[1]);
        pp[2 * i + 1] = pack_bf16x2(pv[2], pv[3]);
        dd[2 * i] = pack_bf16x2(pv[0] * (__uint_as_float(dr[4 * i]) - dv[0]), pv[1] * (__uint_as_float(dr[4 * i + 1]) - dv[1]));
        dd[2 * i + 1] =
            pack_bf16x2(pv[2] * (__uint_as_float(dr[4 * i + 2]) - dv[2]), pv[3] * (__uint_as_float(dr[4 * i + 3]) - dv[3]));
    }
}

// One warpgroup's share of a buffer: loads its W columns of S and dP,
// rebuilds P and dS and writes the bf16 pairs over columns [W/2 wg, W/2 (wg
// + 1)) of the same buffers. Those columns were read by a lower warpgroup,
// so every warpgroup signals S_READ once its loads are done and all but the
// first wait for it before writing (the first writes inside its own
// columns). Returns false if a wait gave up.
template <int D, bool PER_COLUMN, bool WRITE_P>
__device__ __forceinline__ bool rebuild_share(const BwdCtx& c, int wg, int b, int phase, uint32_t ts, uint32_t tdp,
                                              float cs, const float* l2, const float* dl, float l2_row, float dl_row,
                                              int lo, int hi) {
    using C = BwdCfg<D>;
    constexpr int W = C::W;
    uint32_t sr[W], dr[W], pp[W / 2], dd[W / 2];
    tmem_ld_x32(ts + W * wg, sr);
    tmem_ld_x32(tdp + W * wg, dr);
    tmem_ld_wait(sr);
    tmem_ld_wait(dr);
    tc_fence_before();
    mbar_arrive(c.bar(C::S_READ + b));
    if (lo <= 0 && hi >= W)
        rebuild_chunk<W, PER_COLUMN, false>(sr, dr, cs, l2, dl, l2_row, dl_row, lo, hi, pp, dd);
    else
        rebuild_chunk<W, PER_COLUMN, true>(sr, dr, cs, l2, dl, l2_row, dl_row, lo, hi, pp, dd);
    if (wg > 0) {
        if (!c.wait_warp(C::S_READ + b, phase)) return false;
        tc_fence_after();
    }
    if (WRITE_P) tmem_st_x16(ts + (W / 2) * wg, pp);
    tmem_st_x16((WRITE_P ? tdp : ts) + (W / 2) * wg, dd);
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(c.bar(C::P_FULL + b));
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
            mbar_init(c.bar(C::EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(c.bar(C::S_FULL + b), 1);
            mbar_init(c.bar(C::P_FULL + b), C::NWG * kT);
            mbar_init(c.bar(C::S_READ + b), C::NWG * kT);
        }
        mbar_init(c.bar(C::DONE), 1);
        mbar_init(c.bar(C::DRAIN), 1);
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

// TMA thread: the resident pair once, then `n` streamed pairs (rows r0 +
// 128 k), each with (when vec) the 128 padded LSE2 / Dl values at vec_row +
// 128 k of the workspace arrays.
template <int D>
__device__ __forceinline__ void bwd_producer(const BwdCtx& c, uint32_t s0, const CUtensorMap* f0, const CUtensorMap* f1,
                                             int fix_row, const CUtensorMap* r0m, const CUtensorMap* r1m, int r0, int n,
                                             int bh, const float* lse2, const float* delta, int64_t vec_row) {
    using C = BwdCfg<D>;
    const uint64_t pol = policy_evict_last();
    mbar_arrive_expect_tx(c.bar(C::FIX_FULL), 2 * C::TILE);
    load_tile<D>(s0 + C::FIX_OFF, f0, c.bar(C::FIX_FULL), fix_row, bh, pol);
    load_tile<D>(s0 + C::FIX_OFF + C::TILE, f1, c.bar(C::FIX_FULL), fix_row, bh, pol);
    int issued = 0;
#pragma unroll 1
    for (int k = 0; k < n; ++k) {
        const int s = k % C::STAGES;
        if (k >= C::STAGES && !c.wait(C::EMPTY + s, k / C::STAGES - 1)) break;
        const uint32_t dst = s0 + C::RING_OFF + s * C::STAGE;
        mbar_arrive_expect_tx(c.bar(C::FULL + s), 2 * C::TILE + (lse2 ? C::VEC : 0));
        load_tile<D>(dst, r0m, c.bar(C::FULL + s), r0 + k * kT, bh, pol);
        load_tile<D>(dst + C::TILE, r1m, c.bar(C::FULL + s), r0 + k * kT, bh, pol);
        if (lse2) {
            bulk_load(dst + 2 * C::TILE, lse2 + vec_row + k * kT, kT * 4, c.bar(C::FULL + s));
            bulk_load(dst + 2 * C::TILE + kT * 4, delta + vec_row + k * kT, kT * 4, c.bar(C::FULL + s));
        }
        ++issued;
    }
    mbar_wait_drain(c.bar(C::FIX_FULL), 0);
    for (int s = 0; s < C::STAGES && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / C::STAGES) * C::STAGES;
        mbar_wait_drain(c.bar(C::FULL + s), (last / C::STAGES) & 1);
    }
}

// ------------------------------------------------------------ dK, dV kernel
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
bwd_tc_dkdv(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
            const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(sm);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
    BwdCtx c;
    c.bar0 = s0 + C::BAR_OFF;
    c.abort = reinterpret_cast<volatile int*>(misc + 1);
    c.err = p.err;
    const int warp = threadIdx.x / 32;
    const int ktiles = (p.N + kT - 1) / kT;
    const int bh = static_cast<int>(blockIdx.x / ktiles);
    const int key0 = static_cast<int>(blockIdx.x % ktiles) * kT;
    const int mtiles = p.Mpad / kT;
    // Query tiles holding a row that sees a key of this tile: all, or
    // (top-left causal) those with rows >= key0.
    const int i0 = p.causal ? key0 / kT : 0;
    const int nq = mtiles > i0 ? mtiles - i0 : 0;
    const uint32_t tmem = bwd_setup<D>(c, misc);
    if (warp < C::TMA_WARP) {
        // Thread t of warpgroup wg owns key key0 + t (tensor-memory lane t)
        // and columns [W wg, W wg + W) of every 64-query half.
        const int wg = warp >> 2, t = threadIdx.x & 127;
        const int key = key0 + t;
        const uint32_t tm = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const float cs = p.scale * kLog2e;
        bool ok = true;
#pragma unroll 1
        for (int g = 0; g < 2 * nq && ok; ++g) {
            const int k = g >> 1, h = g & 1, b = g & 1;   // query tile, half, S/dP buffer
            const int s = k % C::STAGES;
            const int q0 = (i0 + k) * kT + h * C::HALF_ROWS + C::W * wg;   // this share's first query
            // The stage's LSE2 / Dl arrived with its tiles (FULL), which the
            // MMA thread waited for before S_FULL; wait here too so that the
            // copies are visible to this thread.
            if (!c.wait_warp(C::FULL + s, k / C::STAGES) || !c.wait_warp(C::S_FULL + b, g >> 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float* l2 = reinterpret_cast<const float*>(sm + C::RING_OFF + s * C::STAGE + 2 * C::TILE) +
                              h * C::HALF_ROWS + C::W * wg;
            const float* dl = l2 + kT;
            // Visible queries: column c with q0 + c >= key (causal); rows past
            // M have L2 = +inf; a key past N sees nothing.
            const int lo = p.causal ? key - q0 : 0;
            const int hi = key < p.N ? C::W : 0;
            ok = rebuild_share<D, true, true>(c, wg, b, g >> 1, tm + C::TS + b * 64, tm + C::TDP + b * 64, cs, l2, dl,
                                              0.f, 0.f, lo, hi);
        }
        if (ok && nq > 0) {
            ok = c.wait_warp(C::DONE, 0);
            tc_fence_after();
        }
        if (ok) {   // the first half of the warpgroups writes dV, the second dK, each a share of the chunks
            const bool in = key < p.N;
            const int64_t off = (static_cast<int64_t>(bh) * p.N + key) * D;
            constexpr int kHalfWg = C::NWG / 2, kPer = (D / 32 + kHalfWg - 1) / kHalfWg;
            const int part = wg % kHalfWg;
            const int clo = min(D / 32, part * kPer), chi = min(D / 32, clo + kPer);
            if (wg < kHalfWg)
                store_acc_row<D>(tm + C::TACC, nq > 0, in, p.dv + off, 1.f, clo, chi);
            else
                store_acc_row<D>(tm + C::TACC + D, nq > 0, in, p.dk + off, p.scale, clo, chi);
        }
    } else if (warp == C::TMA_WARP) {
        if ((threadIdx.x & 31) == 0 && nq > 0)
            bwd_producer<D>(c, s0, &map_k, &map_v, key0, &map_q, &map_do, i0 * kT, nq, bh, p.lse2, p.delta,
                            static_cast<int64_t>(bh) * p.Mpad + i0 * kT);
    } else if ((threadIdx.x & 31) == 0) {
        // MMA thread. Per half query tile g: S^T = K Q^T and dP^T = V dO^T
        // into buffer g & 1; once the softmax threads have turned them into
        // P^T and dS^T (bf16, in place): dV += P^T dO, dK += dS^T Q. Half
        // g + 1's products are issued before half g's gradient products, so
        // its rebuild overlaps them; a buffer is rewritten (half g + 2) only
        // after half g's gradient products, which read it (one thread's MMAs
        // run in order).
        bool ok = nq > 0 && c.wait(C::FIX_FULL, 0);
        const uint32_t kt = s0 + C::FIX_OFF, vt = kt + C::TILE;
        auto issue_sdp = [&](int g) -> bool {
            const int k = g >> 1, h = g & 1, s = k % C::STAGES;
            if (h == 0 && !c.wait(C::FULL + s, k / C::STAGES)) return false;
            tc_fence_after();
            const uint32_t qt = s0 + C::RING_OFF + s * C::STAGE + h * C::HALF_BYTES, dot = qt + C::TILE;
            mma_tile_nt<D>(tmem + C::TS + (g & 1) * 64, kt, qt);
            mma_tile_nt<D>(tmem + C::TDP + (g & 1) * 64, vt, dot);
            mma_commit(c.bar(C::S_FULL + (g & 1)));
            return true;
        };
        auto issue_grad = [&](int g) -> bool {
            const int k = g >> 1, h = g & 1, s = k % C::STAGES;
            if (!c.wait(C::P_FULL + (g & 1), g >> 1)) return false;
            tc_fence_after();
            const uint32_t qt = s0 + C::RING_OFF + s * C::STAGE + h * C::HALF_BYTES, dot = qt + C::TILE;
            mma_tile_acc<D>(tmem + C::TACC, tmem + C::TS + (g & 1) * 64, dot, g == 0);
            mma_tile_acc<D>(tmem + C::TACC + D, tmem + C::TDP + (g & 1) * 64, qt, g == 0);
            if (h == 1) mma_commit(c.bar(C::EMPTY + s));
            if (g == 2 * nq - 1) mma_commit(c.bar(C::DONE));
            return true;
        };
        if (ok) ok = issue_sdp(0);
#pragma unroll 1
        for (int g = 0; ok && g < 2 * nq; ++g) {
            if (g + 1 < 2 * nq && !issue_sdp(g + 1)) break;
            ok = issue_grad(g);
        }
        mma_commit(c.bar(C::DRAIN));
        mbar_wait_drain(c.bar(C::DRAIN), 0);
    }
    bwd_teardown<D>(tmem);
}

// --------------------------------------------------------------- dQ kernel
template <int D>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
bwd_tc_dq(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
          const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do, const BwdParams p) {
    using C = BwdCfg<D>;
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
    const uint32_t tmem = bwd_setup<D>(c, misc);
    if (warp < C::TMA_WARP) {
        // Thread t of warpgroup wg owns query row r0 + t (tensor-memory lane
        // t) and columns [W wg, W wg + W) of every 64-key half.
        const int wg = warp >> 2, t = threadIdx.x & 127;
        const int row = r0 + t;
        const uint32_t tm = tmem + (static_cast<uint32_t>(t & ~31) << 16);
        const float cs = p.scale * kLog2e;
        const int64_t prow = static_cast<int64_t>(bh) * p.Mpad + row;
        const float l2 = p.lse2[prow], dl = p.delta[prow];   // +inf / 0 past M
        const int lim = p.causal ? min(p.N, row + 1) : p.N;   // keys [0, lim) visible
        bool ok = true;
#pragma unroll 1
        for (int g = 0; g < 2 * nk && ok; ++g) {
            const int b = g & 1;
            if (!c.wait_warp(C::S_FULL + b, g >> 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int hi = lim - (g * C::HALF_ROWS + C::W * wg);   // this share's keys: g * 64 + W wg + column
            ok = rebuild_share<D, false, false>(c, wg, b, g >> 1, tm + C::TS + b * 64, tm + C::TDP + b * 64, cs,
                                                nullptr, nullptr, l2, dl, 0, hi);
        }
        if (ok && nk > 0) {
            ok = c.wait_warp(C::DONE, 0);
            tc_fence_after();
        }
        if (ok) {   // each warpgroup writes a share of the row's 32-column chunks
            constexpr int kPer = (D / 32 + C::NWG - 1) / C::NWG;
            const int clo = min(D / 32, wg * kPer), chi = min(D / 32, clo + kPer);
            store_acc_row<D>(tm + C::TACC, nk > 0, row < p.M, p.dq + (static_cast<int64_t>(bh) * p.M + row) * D,
                             p.scale, clo, chi);
        }
    } else if (warp == C::TMA_WARP) {
        if ((threadIdx.x & 31) == 0 && nk > 0)
            bwd_producer<D>(c, s0, &map_q, &map_do, r0, &map_k, &map_v, 0, nk, bh, nullptr, nullptr, 0);
    } else if ((threadIdx.x & 31) == 0) {
        // MMA thread. Per half key tile g: S = Q K^T and dP = dO V^T into
        // buffer g & 1; once the softmax threads have written dS (bf16, over
        // S): dQ += dS K. Issue order as in the dK/dV kernel.
        bool ok = nk > 0 && c.wait(C::FIX_FULL, 0);
        const uint32_t qt = s0 + C::FIX_OFF, dot = qt + C::TILE;
        auto issue_sdp = [&](int g) -> bool {
            const int k = g >> 1, h = g & 1, s = k % C::STAGES;
            if (h == 0 && !c.wait(C::FULL + s, k / C::STAGES)) return false;
            tc_fence_after();
            const uint32_t kt = s0 + C::RING_OFF + s * C::STAGE + h * C::HALF_BYTES, vt = kt + C::TILE;
            mma_tile_nt<D>(tmem + C::TS + (g & 1) * 64, qt, kt);
            mma_tile_nt<D>(tmem + C::TDP + (g & 1) * 64, dot, vt);
            mma_commit(c.bar(C::S_FULL + (g & 1)));
            return true;
        };
        auto issue_grad = [&](int g) -> bool {
            const int k = g >> 1, h = g & 1, s = k % C::STAGES;
            if (!c.wait(C::P_FULL + (g & 1), g >> 1)) return false;
            tc_fence_after();
            const uint32_t kt = s0 + C::RING_OFF + s * C::STAGE + h * C::HALF_BYTES;
            mma_tile_acc<D>(tmem + C::TACC, tmem + C::TS + (g & 1) * 64, kt, g == 0);
            if (h == 1) mma_commit(c.bar(C::EMPTY + s));
            if (g == 2 * nk - 1) mma_commit(c.bar(C::DONE));
            return true;
        };
        if (ok) ok = issue_sdp(0);
#pragma unroll 1
        for (int g = 0; ok && g < 2 * nk; ++g) {
            if (g + 1 < 2 * nk && !issue_sdp(g + 1)) break;
            ok = issue_grad(g);
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
    if (e == cudaSuccess) e = cudaFuncSetAttribute(bwd_tc_dq<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (kv_blocks > 0) {
        bwd_tc_dkdv<D><<<static_cast<unsigned>(kv_blocks), C::THREADS, C::SMEM_BYTES, s>>>(q, k, v, dout, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    bwd_tc_dq<D><<<static_cast<unsigned>(q_blocks), C::THREADS, C::SMEM_BYTES, s>>>(q, k, v, dout, p);
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
