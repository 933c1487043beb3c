// fp32 attention forward on the tensor cores: three TF32 products per matrix
// product.
//
// "FlashAttention in Triton: A Tile-by-Tile Walkthrough" computes both dots of
// its fp32 problem in IEEE fp32 on the CUDA cores and ends up slower than the
// library kernel it is compared with. This path keeps the streaming softmax of
// "FlashAttention-style kernel" (section "The loop") and moves the two
// products onto tcgen05, which reads fp32 operands as TF32 (sign, exponent and
// the top 10 of 23 mantissa bits). Every fp32 x is split as
//   x = hi + lo,  hi = x rounded to 11 significant bits,  lo = x - hi (exact),
// and a product A B is taken as  A_lo B_hi + A_hi B_lo + A_hi B_hi,  small
// terms first, into an fp32 accumulator. The dropped A_lo B_lo term and the
// truncation of lo to TF32 are each about 2^-22 relative to the product, so
// the result is close to fp32 accuracy at a sixth of the bf16 tensor rate.
//
// Two kernels:
//   x3_split: K and V, per 64-key block, into hi and lo images laid out as
//             the MMA reads them (K-major, 128-byte swizzle: K as 64 keys x
//             32-column panels, V transposed to D rows x 32-key panels), so
//             the attention kernel loads them with plain bulk copies.
//   x3_fwd:   one CTA per 128-row query tile. The four softmax warps split
//             their Q rows into tensor memory (the A operand of S = Q K^T),
//             then run the online softmax one 64-key block at a time: P_hi
//             goes back into the block's S columns of tensor memory and
//             P_lo into shared memory, the two A operands of P V. Two warps
//             stream the K and the V images through rings of their own (a K
//             slot is free again as soon as its S product completes, so K
//             runs ahead), one thread issues the MMAs: S(j+1) is computed
//             while the softmax works on S(j). A TF32 MMA of 128 rows costs
//             about as much at N = 32 as at N = 64, so the 64-key block
//             halves the S instructions per key.
// Masking (top-left causal, key tail), the safe max, the rare rescale of the
// accumulator (only when a row's max grows by more than 2^8) and the final
// division follow the bf16 kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kBM = 128;              // query rows per CTA: one per softmax thread and TMEM lane
constexpr int kThreads = 224;         // 4 softmax warps, the K load warp, the MMA warp, the V load warp
constexpr int kSplitThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // a row's reference max moves only when it grows by more

// x = hi + lo with hi holding the 11 leading significant bits of x (rounded
// to nearest, ties away from zero, on the magnitude) and lo the exact rest.
// Finite inputs below 2^127 in magnitude.
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
    hi = __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xffffe000u);
    lo = x - hi;
}

// Position (in floats) of element (row r, column c) inside one K-major,
// 128-byte-swizzled panel of 32 fp32 columns: the 16-byte unit c / 4 of row
// r is stored at unit (c / 4) xor (r mod 8).
__host__ __device__ constexpr int swz(int r, int c) { return r * 32 + (((c >> 2) ^ (r & 7)) << 2) + (c & 3); }

// Keys per block: 64 (two 128-byte swizzle panels of fp32) for D >= 96;
// 32 below, where a CTA's tensor memory then fits in half of the SM's and two
// CTAs share an SM. A TF32 MMA of 128 rows costs about as much at N = 32 as
// at N = 64, so the wider block halves the S instructions per key.
template <int D>
struct X3Cfg {
    static constexpr int BN = (D >= 96) ? 64 : 32;
    static constexpr int PANELS = BN / 32;                   // 128-byte panels along the keys
    static constexpr int HALF = BN * D * 4;                  // bytes of one K or V^T part (hi or lo)
    static constexpr int SLOT = 2 * HALF;                    // one ring slot: hi and lo of K, or of V^T
    static constexpr int K_PANEL = BN * 128;                 // BN keys x 128 B
    static constexpr int V_PANEL = D * 128;                  // D rows x 128 B (32 keys)
    static constexpr int P_PANEL = kBM * 128;                // 128 rows x 128 B (32 keys)
    static constexpr int P_OFF = 0;                          // P_lo: PANELS panels
    static constexpr int K_OFF = PANELS * P_PANEL;
    // Ring slots: D = 128 fits three (two for K, which is needed first, one
    // for V); D <= 64 keeps each CTA under half of the SM's shared memory.
    static constexpr int FIT = (232448 - 2048 - K_OFF) / SLOT;
    static constexpr int NK = (D <= 64) ? 3 : (FIT >= 8 ? 4 : (FIT + 1) / 2);
    static constexpr int NV = (D <= 64) ? 2 : (FIT >= 8 ? 4 : FIT / 2);
    static constexpr int V_OFF = K_OFF + NK * SLOT;
    static constexpr int BAR_OFF = V_OFF + NV * SLOT;
    static constexpr int K_FULL = 0, K_EMPTY = NK, V_FULL = 2 * NK, V_EMPTY = 2 * NK + NV, Q_READY = 2 * NK + 2 * NV;
    static constexpr int S_FULL = Q_READY + 1, P_FULL = S_FULL + 2, O_DONE = P_FULL + 1, DRAIN = O_DONE + 1;
    static constexpr int NUM_BARS = DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;  // tensor-memory base, abort flag
    static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack to align the base to 1024 B
    // Tensor-memory columns: Q hi, Q lo, O, two S buffers (each later P_hi).
    static constexpr uint32_t QH = 0, QL = D, OC = 2 * D, SC0 = 3 * D, SC1 = 3 * D + BN;
    static constexpr uint32_t TMEM_COLS = (3 * D + 2 * BN <= 256) ? 256 : 512;
    static_assert(D % 32 == 0 && D >= 32 && D <= 128, "D");
    static_assert(NK >= 1 && NV >= 1, "ring slots");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(D > 64 || SMEM_BYTES <= 232448 / 2 - 1024, "two CTAs per SM");
};

// K/V images of one key block: [K hi | K lo | V^T hi | V^T lo], each BN * D
// floats. K parts: D/32 panels of BN keys x 32 columns. V^T parts: BN/32
// panels (32 keys each) of D rows x 32 keys.
template <int D>
__global__ void __launch_bounds__(kSplitThreads) x3_split(const float* __restrict__ k, const float* __restrict__ v,
                                                          float* __restrict__ ws, int N, int nt) {
    constexpr int kBN = X3Cfg<D>::BN;
    constexpr int HALF = kBN * D;
    const int64_t blk = blockIdx.x;            // head * nt + key block
    const int64_t head = blk / nt;
    const int j = static_cast<int>(blk - head * nt);
    const float* kh = k + head * N * D;
    const float* vh = v + head * N * D;
    float* out = ws + blk * (4 * HALF);
    // K: one float4 of a key row per item; reads coalesce along the row.
    constexpr int KU = D / 4;
    for (int i = threadIdx.x; i < kBN * KU; i += kSplitThreads) {
        const int r = i / KU, c = (i % KU) * 4;
        const int key = j * kBN + r;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (key < N) x = *reinterpret_cast<const float4*>(kh + static_cast<int64_t>(key) * D + c);
        float4 h, l;
        split_tf32(x.x, h.x, l.x);
        split_tf32(x.y, h.y, l.y);
        split_tf32(x.z, h.z, l.z);
        split_tf32(x.w, h.w, l.w);
        const int dst = (c >> 5) * (kBN * 32) + swz(r, c & 31);
        *reinterpret_cast<float4*>(out + dst) = h;
        *reinterpret_cast<float4*>(out + HALF + dst) = l;
    }
    // V^T: the block's rows are staged in shared memory (coalesced float4
    // reads), then each item takes four consecutive keys of one column d;
    // the keys run fastest across the threads, so the eight 16-byte units of
    // one 128-byte output row are written by neighbouring threads.
    __shared__ float sv[kBN][D + 1];   // +1: column reads spread over the banks
    for (int i = threadIdx.x; i < kBN * KU; i += kSplitThreads) {
        const int r = i / KU, c = (i % KU) * 4;
        const int key = j * kBN + r;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (key < N) x = *reinterpret_cast<const float4*>(vh + static_cast<int64_t>(key) * D + c);
        sv[r][c + 0] = x.x;
        sv[r][c + 1] = x.y;
        sv[r][c + 2] = x.z;
        sv[r][c + 3] = x.w;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < D * (kBN / 4); i += kSplitThreads) {
        const int c = (i % (kBN / 4)) * 4, d = i / (kBN / 4);   // c: key within the block
        float4 h, l;
        split_tf32(sv[c + 0][d], h.x, l.x);
        split_tf32(sv[c + 1][d], h.y, l.y);
        split_tf32(sv[c + 2][d], h.z, l.z);
        split_tf32(sv[c + 3][d], h.w, l.w);
        const int dst = (c >> 5) * (D * 32) + swz(d, c & 31);
        *reinterpret_cast<float4*>(out + 2 * HALF + dst) = h;
        *reinterpret_cast<float4*>(out + 3 * HALF + dst) = l;
    }
}

// Per-CTA view of the barriers and the abort flag.
struct X3Ctx {
    uint32_t bar0;
    volatile int* abort;
    uint32_t* err;
    __device__ uint32_t bar(int i) const { return bar0 + 8u * static_cast<uint32_t>(i); }
    __device__ bool wait(int i, int parity) const { return mbar_wait(bar(i), static_cast<uint32_t>(parity) & 1u, abort, err); }
    // Warp-uniform result, for code that runs warp-collective tcgen05 loads next.
    __device__ bool wait_warp(int i, int parity) const { return __all_sync(0xffffffffu, wait(i, parity)); }
};

// Pairwise reductions over a row's BN values (short dependency chains).
template <int BN>
__device__ __forceinline__ float tree_max(const float (&x)[BN]) {
    float m[BN / 2];
#pragma unroll
    for (int i = 0; i < BN / 2; ++i) m[i] = fmaxf(x[i], x[i + BN / 2]);
#pragma unroll
    for (int w = BN / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    return m[0];
}
template <int BN>
__device__ __forceinline__ float tree_sum(const float (&x)[BN]) {
    float m[BN / 2];
#pragma unroll
    for (int i = 0; i < BN / 2; ++i) m[i] = x[i] + x[i + BN / 2];
#pragma unroll
    for (int w = BN / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] += m[i + w];
    return m[0];
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// ------------------------------------------------------------ softmax warps
// Thread t of warps 0-3 owns query row r0 + t and tensor-memory lane t.
template <int D>
__device__ __forceinline__ void x3_softmax(const X3Params& p, const X3Ctx& c, uint32_t s0, uint32_t tmem, int bh,
                                           int r0, int nb) {
    using C = X3Cfg<D>;
    constexpr int kBN = C::BN;
    const int t = threadIdx.x;
    const int row = r0 + t;
    const bool in = row < p.M;
    const uint32_t tm = tmem + (static_cast<uint32_t>(t & ~31) << 16);
    const int64_t row_off = (static_cast<int64_t>(bh) * p.M + row) * D;
    // Q row -> hi and lo parts in tensor memory (rows past M are zero).
    if (nb > 0) {
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (in) x = *reinterpret_cast<const float4*>(p.q + row_off + cc * 32 + i * 4);
                const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float h, l;
                    split_tf32(xs[e], h, l);
                    hi[i * 4 + e] = __float_as_uint(h);
                    lo[i * 4 + e] = __float_as_uint(l);
                }
            }
            tmem_st_x32(tm + C::QH + cc * 32, hi);
            tmem_st_x32(tm + C::QL + cc * 32, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(c.bar(C::Q_READY));
    }
    const float cs = p.scale * kLog2e;
    const int lim = p.causal ? min(p.N, row + 1) : p.N;   // keys [0, lim) are visible
    const uint32_t prow = s0 + C::P_OFF + t * 128;
    const uint32_t sw = t & 7;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < nb; ++j) {
        const int sb = j & 1;
        const uint32_t scol = tm + (sb ? C::SC1 : C::SC0);
        if (!c.wait_warp(C::S_FULL + sb, j >> 1)) {
            ok = false;
            break;
        }
        tc_fence_after();
        float x[kBN];
        {
            uint32_t sr[C::PANELS][32];
#pragma unroll
            for (int h = 0; h < C::PANELS; ++h) tmem_ld_x32(scol + h * 32, sr[h]);
#pragma unroll
            for (int h = 0; h < C::PANELS; ++h) tmem_ld_wait(sr[h]);
            const int key0 = j * kBN;
            if (key0 + kBN <= lim) {   // every key of the block visible to this row
#pragma unroll
                for (int h = 0; h < C::PANELS; ++h)
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[h * 32 + i] = __uint_as_float(sr[h][i]) * cs;
            } else {
#pragma unroll
                for (int h = 0; h < C::PANELS; ++h)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        x[h * 32 + i] = (key0 + h * 32 + i < lim) ? __uint_as_float(sr[h][i]) * cs : -INFINITY;
            }
        }
        const float mx = tree_max<kBN>(x);
        float m_new = m_ref;
        bool resc = false;
        if (mx > m_ref + kRescaleLog2) {
            m_new = mx;
            resc = j > 0;
        }
        const float m_s = (m_new == -INFINITY) ? 0.f : m_new;
#pragma unroll
        for (int i = 0; i < kBN; ++i) x[i] = ex2(x[i] - m_s);
        const float sum = tree_sum<kBN>(x);
        const float alpha = resc ? ex2(m_ref - m_new) : 1.f;
        l = l * alpha + sum;
        // P V of the previous block has completed: O is final for it and
        // the P_lo buffer is free.
        if (j > 0) {
            if (!c.wait_warp(C::O_DONE, j - 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
        }
        if (__any_sync(0xffffffffu, resc)) {   // the warp rescales together; alpha = 1 leaves a row as it is
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld_x32(tm + C::OC + cc * 32, o);
                tmem_ld_wait(o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st_x32(tm + C::OC + cc * 32, o);
            }
        }
        // P = hi + lo: hi over this block's S columns, lo into row t of the
        // shared-memory panels (32 keys each).
#pragma unroll
        for (int half = 0; half < C::PANELS; ++half) {
            uint32_t hb[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                float h[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    split_tf32(x[half * 32 + u * 4 + e], h[e], lo[e]);
                    hb[u * 4 + e] = __float_as_uint(h[e]);
                }
                const uint32_t a = prow + half * C::P_PANEL + ((static_cast<uint32_t>(u) ^ sw) << 4);
                st_shared_v4(a, lo[0], lo[1], lo[2], lo[3]);
            }
            tmem_st_x32(scol + half * 32, hb);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(c.bar(C::P_FULL));
        m_ref = m_new;
    }
    if (ok && nb > 0) {
        ok = c.wait_warp(C::O_DONE, nb - 1);
        tc_fence_after();
    }
    if (!ok) return;
    // Epilogue: O = acc / l, LSE = ln 2 * m + ln l (natural log of the
    // scaled scores' exponential sum); a row that saw no key gets O = 0 and
    // LSE = -inf.
    float* orow = p.o + row_off;
#pragma unroll 1
    for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        if (nb > 0) {
            tmem_ld_x32(tm + C::OC + cc * 32, o);
            tmem_ld_wait(o);
        }
        if (in) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
                if (nb > 0 && l > 0.f) {
                    w.x = __uint_as_float(o[i * 4 + 0]) / l;
                    w.y = __uint_as_float(o[i * 4 + 1]) / l;
                    w.z = __uint_as_float(o[i * 4 + 2]) / l;
                    w.w = __uint_as_float(o[i * 4 + 3]) / l;
                }
                *reinterpret_cast<float4*>(orow + cc * 32 + i * 4) = w;
            }
        }
    }
    if (in) p.lse[static_cast<int64_t>(bh) * p.M + row] = (nb > 0 && l > 0.f) ? m_ref * kLn2 + logf(l) : -INFINITY;
}

// -------------------------------------------------------------- load warps
// Streams one half of every key block's image (part 0: K hi and lo; part 1:
// V^T hi and lo) through its ring of `ns` slots.
template <int D>
__device__ __forceinline__ void x3_producer(const X3Params& p, const X3Ctx& c, uint32_t s0, int bh, int nb, int nt,
                                            int part) {
    using C = X3Cfg<D>;
    const int ns = part ? C::NV : C::NK;
    const int full = part ? C::V_FULL : C::K_FULL, empty = part ? C::V_EMPTY : C::K_EMPTY;
    const uint32_t ring = s0 + (part ? C::V_OFF : C::K_OFF);
    const uint8_t* img = p.ws + static_cast<int64_t>(bh) * nt * (2 * C::SLOT) + part * C::SLOT;
    int issued = 0;
#pragma unroll 1
    for (int j = 0; j < nb; ++j) {
        const int st = j % ns;
        if (j >= ns && !c.wait(empty + st, j / ns - 1)) break;
        const uint8_t* src = img + static_cast<int64_t>(j) * (2 * C::SLOT);
        mbar_arrive_expect_tx(c.bar(full + st), C::SLOT);
        bulk_load(ring + st * C::SLOT, src, C::HALF, c.bar(full + st));
        bulk_load(ring + st * C::SLOT + C::HALF, src + C::HALF, C::HALF, c.bar(full + st));
        ++issued;
    }
    // Every copy issued lands before the CTA's shared memory is released.
    for (int s = 0; s < ns && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / ns) * ns;
        mbar_wait_drain(c.bar(full + s), (last / ns) & 1);
    }
}

// --------------------------------------------------------------- MMA thread
template <int D>
__device__ __forceinline__ void x3_mma(const X3Ctx& c, uint32_t s0, uint32_t tmem, int nb) {
    using C = X3Cfg<D>;
    constexpr int kBN = C::BN;
    constexpr uint32_t id_s = idesc_tf32_f32(kBM, kBN);
    constexpr uint32_t id_o = idesc_tf32_f32(kBM, D);
    // Descriptor template with a zero start address; adding (address >> 4)
    // fills the 14-bit start field. K-major, 128-byte swizzle: SBO = 8 rows
    // of 128 B; an 8-column (32-byte) K-step advances the start by 2, every
    // fourth step moves to the next 128-byte panel.
    const uint64_t dz = smem_desc_sw128(0, 16, 1024);
    constexpr uint32_t kPanelK = C::K_PANEL >> 4, kPanelV = C::V_PANEL >> 4, kPanelP = C::P_PANEL >> 4;
    // S(j) = Q_lo K_hi^T + Q_hi K_lo^T + Q_hi K_hi^T, Q from tensor memory.
    // Buffer j & 1 last held P_hi(j - 2), whose P V products were issued
    // before this (the tensor pipe runs one thread's MMAs in order) and whose
    // softmax finished before they were.
    auto issue_s = [&](int j) -> bool {
        const int st = j % C::NK, sb = j & 1;
        if (!c.wait(C::K_FULL + st, j / C::NK)) return false;
        tc_fence_after();
        const uint32_t kb = s0 + C::K_OFF + st * C::SLOT;
        const uint64_t dkh = dz + (kb >> 4), dkl = dz + ((kb + C::HALF) >> 4);
        const uint32_t scol = tmem + (sb ? C::SC1 : C::SC0);
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk) {
            const uint32_t off = (kk >> 2) * kPanelK + (kk & 3) * 2;
            mma_ts_tf32(scol, tmem + C::QL + kk * 8, dkh + off, id_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk) {
            const uint32_t off = (kk >> 2) * kPanelK + (kk & 3) * 2;
            mma_ts_tf32(scol, tmem + C::QH + kk * 8, dkl + off, id_s, 1u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk) {
            const uint32_t off = (kk >> 2) * kPanelK + (kk & 3) * 2;
            mma_ts_tf32(scol, tmem + C::QH + kk * 8, dkh + off, id_s, 1u);
        }
        mma_commit(c.bar(C::S_FULL + sb));
        mma_commit(c.bar(C::K_EMPTY + st));
        return true;
    };
    // O (+)= P_lo V_hi + P_hi V_lo + P_hi V_hi: P_lo from shared memory, P_hi
    // from the block's S columns, V^T K-major; the first product of the tile
    // overwrites O.
    auto issue_pv = [&](int j) -> bool {
        const int st = j % C::NV;
        if (!c.wait(C::V_FULL + st, j / C::NV) || !c.wait(C::P_FULL, j)) return false;
        tc_fence_after();
        const uint32_t vb = s0 + C::V_OFF + st * C::SLOT;
        const uint64_t dvh = dz + (vb >> 4), dvl = dz + ((vb + C::HALF) >> 4);
        const uint64_t dpl = dz + ((s0 + C::P_OFF) >> 4);
        const uint32_t pcol = tmem + ((j & 1) ? C::SC1 : C::SC0);
        const uint32_t ocol = tmem + C::OC;
#pragma unroll
        for (int kk = 0; kk < kBN / 8; ++kk)
            mma_ss_tf32(ocol, dpl + (kk >> 2) * kPanelP + (kk & 3) * 2, dvh + (kk >> 2) * kPanelV + (kk & 3) * 2, id_o,
                        (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kBN / 8; ++kk)
            mma_ts_tf32(ocol, pcol + kk * 8, dvl + (kk >> 2) * kPanelV + (kk & 3) * 2, id_o, 1u);
#pragma unroll
        for (int kk = 0; kk < kBN / 8; ++kk)
            mma_ts_tf32(ocol, pcol + kk * 8, dvh + (kk >> 2) * kPanelV + (kk & 3) * 2, id_o, 1u);
        mma_commit(c.bar(C::O_DONE));
        mma_commit(c.bar(C::V_EMPTY + st));
        return true;
    };
    bool ok = nb > 0 && c.wait(C::Q_READY, 0);
    if (ok) {
        tc_fence_after();
        ok = issue_s(0);
    }
#pragma unroll 1
    for (int j = 0; ok && j < nb; ++j) {
        if (j + 1 < nb && !issue_s(j + 1)) break;
        ok = issue_pv(j);
    }
    // Every MMA issued completes before tensor or shared memory is released.
    mma_commit(c.bar(C::DRAIN));
    mbar_wait_drain(c.bar(C::DRAIN), 0);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) x3_fwd(const X3Params p) {
    using C = X3Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s0 = smem_u32(sm);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
    X3Ctx c;
    c.bar0 = s0 + C::BAR_OFF;
    c.abort = reinterpret_cast<volatile int*>(misc + 1);
    c.err = p.err;
    const int warp = threadIdx.x / 32;
    // The query tiles of one head are adjacent, heaviest (last, under the
    // causal mask) first: the CTAs resident at one time cover a few heads,
    // whose K/V images stay in L2 while all their query tiles read them.
    const int mtiles = (p.M + kBM - 1) / kBM;
    const int mt = mtiles - 1 - static_cast<int>(blockIdx.x % mtiles);
    const int bh = static_cast<int>(blockIdx.x / mtiles);
    const int r0 = mt * kBM;
    const int kend = p.causal ? min(p.N, min(p.M, r0 + kBM)) : p.N;
    const int nb = (kend + C::BN - 1) / C::BN;
    const int nt = (p.N + C::BN - 1) / C::BN;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NK; ++i) {
            mbar_init(c.bar(C::K_FULL + i), 1);
            mbar_init(c.bar(C::K_EMPTY + i), 1);
        }
        for (int i = 0; i < C::NV; ++i) {
            mbar_init(c.bar(C::V_FULL + i), 1);
            mbar_init(c.bar(C::V_EMPTY + i), 1);
        }
        mbar_init(c.bar(C::Q_READY), kBM);
        mbar_init(c.bar(C::S_FULL + 0), 1);
        mbar_init(c.bar(C::S_FULL + 1), 1);
        mbar_init(c.bar(C::P_FULL), kBM);
        mbar_init(c.bar(C::O_DONE), 1);
        mbar_init(c.bar(C::DRAIN), 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(misc), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    if (warp < 4) {
        x3_softmax<D>(p, c, s0, tmem, bh, r0, nb);
    } else if (warp == 4 || warp == 6) {
        if ((threadIdx.x & 31) == 0) x3_producer<D>(p, c, s0, bh, nb, nt, warp == 6 ? 1 : 0);
    } else if ((threadIdx.x & 31) == 0) {
        x3_mma<D>(c, s0, tmem, nb);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_x3_t(const X3Params& p, cudaStream_t s) {
    using C = X3Cfg<D>;
    const int64_t nt = (static_cast<int64_t>(p.N) + C::BN - 1) / C::BN;
    const int64_t split_blocks = static_cast<int64_t>(p.bh_count) * nt;
    const int64_t blocks = static_cast<int64_t>(p.bh_count) * ((static_cast<int64_t>(p.M) + kBM - 1) / kBM);
    if (split_blocks > 0x7fffffffLL || blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (split_blocks > 0) {
        x3_split<D><<<static_cast<unsigned>(split_blocks), kSplitThreads, 0, s>>>(p.k, p.v, reinterpret_cast<float*>(p.ws),
                                                                                 p.N, static_cast<int>(nt));
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // Set on every call: the attribute belongs to the current device's context.
    const cudaError_t e = cudaFuncSetAttribute(x3_fwd<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    x3_fwd<D><<<static_cast<unsigned>(blocks), kThreads, C::SMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int64_t x3_workspace_bytes(int64_t bh, int64_t N, int64_t D) {
    const int64_t bn = (D >= 96) ? X3Cfg<128>::BN : X3Cfg<64>::BN;   // the key block of X3Cfg<D>
    const int64_t nt = (N + bn - 1) / bn;
    return bh * nt * 4 * bn * D * static_cast<int64_t>(sizeof(float));
}

cudaError_t launch_x3(const X3Params& p, cudaStream_t s) {
    switch (p.D) {
        case 32: return launch_x3_t<32>(p, s);
        case 64: return launch_x3_t<64>(p, s);
        case 96: return launch_x3_t<96>(p, s);
        case 128: return launch_x3_t<128>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
