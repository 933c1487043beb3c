// Backward pass of the attention forward, on the CUDA cores (fp32 arithmetic).
//
// "Module 08: FlashAttention and Memory-Efficient Kernels", section "The
// backward pass: recompute instead of store" and Code Step 6: the forward
// keeps one number per row, L = m + log(l), and the backward rebuilds every
// tile of P on chip as exp(S - L) from Q and K instead of reading a stored
// N x N matrix. With that P, for an output gradient dO:
//   dV = P^T dO,  dP = dO V^T,  Dl_i = sum_d dO_id O_id,
//   dS = P * (dP - Dl),  dQ = scale dS K,  dK = scale dS^T Q.
// Three kernels, each reading bf16 inputs and accumulating in fp32:
//   bwd_rowdot: Dl_i for every query row (one warp per row), with the LSE in
//               base 2, into a workspace padded to 128-row tiles (it also
//               feeds the tensor-core kernels of fa_bwd_tc.cu);
//   bwd_dkdv:   one CTA per 64-key tile of one head; query rows stream through
//               shared memory in chunks; dK and dV of the tile stay in
//               registers (eight threads per key at D = 128, four below,
//               each holding its share of D);
//   bwd_dq:     one CTA per 64-row query tile; key rows stream through shared
//               memory; dQ stays in registers.
// The two main kernels both rebuild P (and dP) -- seven products' worth of
// work against the five of Practice 3 -- so that no output needs atomics and
// the result is deterministic. The scores use the hardware exp2 with log2(e)
// folded into the scale, as the forward does.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kTile = 64;      // keys (dK/dV kernel) or query rows (dQ kernel) per CTA
// Threads sharing one key or row, each over DV / parts of D: eight at D = 128
// (fewer registers, twice the warps), four below (fewer shuffles).
template <int DV>
__host__ __device__ constexpr int parts() { return DV >= 128 ? 8 : 4; }
template <int DV>
__host__ __device__ constexpr int threads() { return kTile * parts<DV>(); }
constexpr int kChunk = 32;     // rows streamed through shared memory per step
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ld_bf16(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Sum over the P consecutive lanes that share a key or row.
template <int P>
__device__ __forceinline__ float part_sum(float x) {
#pragma unroll
    for (int off = 1; off < P; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Hardware base-2 exponential (MUFU), as in the forward kernel.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One warp per row of the padded [BH, Mpad] layout: Dl = sum_d dO * O and
// the LSE in base-2 units; rows past M get Dl = 0 and LSE = +inf (P = 0).
__global__ void bwd_rowdot(const BwdParams p) {
    const int64_t prow = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (prow >= static_cast<int64_t>(p.bh_count) * p.Mpad) return;
    const int64_t bh = prow / p.Mpad;
    const int r = static_cast<int>(prow - bh * p.Mpad);
    if (r >= p.M) {
        if (lane == 0) {
            p.delta[prow] = 0.f;
            p.lse2[prow] = INFINITY;
        }
        return;
    }
    const int64_t row = bh * p.M + r;
    const __nv_bfloat16* o = p.o + row * p.D;
    const __nv_bfloat16* d = p.dout + row * p.D;
    float s = 0.f;
    if ((p.D & 3) == 0) {   // rows 8-byte aligned: four bf16 per lane and load
        for (int i = lane * 4; i < p.D; i += 128) {
            const uint2 ov = *reinterpret_cast<const uint2*>(o + i), dv = *reinterpret_cast<const uint2*>(d + i);
            const float2 o0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov.x));
            const float2 o1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov.y));
            const float2 d0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dv.x));
            const float2 d1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dv.y));
            s = fmaf(o0.x, d0.x, fmaf(o0.y, d0.y, fmaf(o1.x, d1.x, fmaf(o1.y, d1.y, s))));
        }
    } else {
        for (int i = lane; i < p.D; i += 32) s = fmaf(ld_bf16(o + i), ld_bf16(d + i), s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
        p.delta[prow] = s;
        p.lse2[prow] = p.lse[row] * kLog2e;
    }
}

// The same for D = 8 LR (LR = 8 or 16 lanes per row, 16-byte loads; O and dO
// 16-byte aligned): a warp takes 32 / LR rows at a time and issues the loads
// of four such groups before reducing any, so that enough bytes are in
// flight to run near the HBM rate (one warp per row with 8-byte loads kept
// too few requests outstanding: 3.0 TB/s at D = 128, 1.6 at D = 64).
template <int LR>
__global__ void __launch_bounds__(256) bwd_rowdot_vec(const BwdParams p) {
    constexpr int D = 8 * LR, RPW = 32 / LR, U = 4, G = U * RPW;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LR, l = lane % LR;
    const int64_t total = static_cast<int64_t>(p.bh_count) * p.Mpad;
    const int64_t base = (static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32) * G;
    uint4 ov[U], dv[U];
    int64_t prow[U], row[U];
    bool live[U];
    float lse[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        prow[u] = base + u * RPW + sub;
        const int64_t bh = prow[u] / p.Mpad;
        const int r = static_cast<int>(prow[u] - bh * p.Mpad);
        live[u] = prow[u] < total && r < p.M;
        row[u] = bh * p.M + r;
        ov[u] = dv[u] = make_uint4(0u, 0u, 0u, 0u);
        lse[u] = INFINITY;
        if (live[u]) {
            ov[u] = *reinterpret_cast<const uint4*>(p.o + row[u] * D + 8 * l);
            dv[u] = *reinterpret_cast<const uint4*>(p.dout + row[u] * D + 8 * l);
            if (l == 0) lse[u] = p.lse[row[u]] * kLog2e;
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t ow[4] = {ov[u].x, ov[u].y, ov[u].z, ov[u].w};
        const uint32_t dw[4] = {dv[u].x, dv[u].y, dv[u].z, dv[u].w};
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[i]));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[i]));
            s = fmaf(a.x, b.x, fmaf(a.y, b.y, s));
        }
#pragma unroll
        for (int off = LR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (l == 0 && prow[u] < total) {
            p.delta[prow[u]] = live[u] ? s : 0.f;
            p.lse2[prow[u]] = lse[u];   // +inf past M: P = 0
        }
    }
}

// Copies `rows` rows of width D (bf16, row-major) starting at row r0 into
// shared memory as fp32 [kChunk][DV], zero-filling rows >= limit and
// columns >= D.
template <int DV>
__device__ __forceinline__ void stage(float* dst, const __nv_bfloat16* src, int r0, int limit, int D) {
    for (int i = threadIdx.x; i < kChunk * DV; i += threads<DV>()) {
        const int r = i / DV, c = i % DV;
        dst[i] = (r0 + r < limit && c < D) ? ld_bf16(src + static_cast<int64_t>(r0 + r) * D + c) : 0.f;
    }
}

template <int DV>
__global__ void __launch_bounds__(threads<DV>()) bwd_dkdv(const BwdParams p) {
    constexpr int P = parts<DV>();
    constexpr int W = DV / P;
    __shared__ float sq[kChunk * DV], sdo[kChunk * DV], slse[kChunk], sdl[kChunk];
    const int tiles = (p.N + kTile - 1) / kTile;
    const int bh = blockIdx.x / tiles;
    const int key0 = (blockIdx.x - bh * tiles) * kTile;
    const int key = key0 + threadIdx.x / P;
    const int c0 = (threadIdx.x % P) * W;            // this thread's columns [c0, c0 + W)
    const bool kvalid = key < p.N;
    const int64_t kv_base = static_cast<int64_t>(bh) * p.N * p.D;
    const int64_t q_base = static_cast<int64_t>(bh) * p.M * p.D;
    float kr[W], vr[W], dk[W], dv[W];
#pragma unroll
    for (int c = 0; c < W; ++c) {
        const bool in = kvalid && c0 + c < p.D;
        kr[c] = in ? ld_bf16(p.k + kv_base + static_cast<int64_t>(key) * p.D + c0 + c) : 0.f;
        vr[c] = in ? ld_bf16(p.v + kv_base + static_cast<int64_t>(key) * p.D + c0 + c) : 0.f;
        dk[c] = 0.f;
        dv[c] = 0.f;
    }
    const float cs = p.scale * kLog2e;
    // Query rows that can see a key of this tile: all, or (causal) rows >= key0.
    const int row_lo = p.causal ? key0 : 0;
    for (int r0 = row_lo; r0 < p.M; r0 += kChunk) {
        __syncthreads();
        stage<DV>(sq, p.q + q_base, r0, p.M, p.D);
        stage<DV>(sdo, p.dout + q_base, r0, p.M, p.D);
        for (int i = threadIdx.x; i < kChunk; i += threads<DV>()) {
            const bool in = r0 + i < p.M;
            const int64_t row = static_cast<int64_t>(bh) * p.M + r0 + i;
            slse[i] = in ? p.lse[row] : -INFINITY;
            sdl[i] = in ? p.delta[static_cast<int64_t>(bh) * p.Mpad + r0 + i] : 0.f;
        }
        __syncthreads();
        for (int i = 0; i < kChunk; ++i) {
            const int row = r0 + i;
            const float* qi = sq + i * DV + c0;
            const float* doi = sdo + i * DV + c0;
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < W; ++c) {
                s = fmaf(kr[c], qi[c], s);
                dp = fmaf(vr[c], doi[c], dp);
            }
            s = part_sum<P>(s);
            dp = part_sum<P>(dp);
            const bool vis = kvalid && row < p.M && (!p.causal || key <= row) && slse[i] != -INFINITY;
            const float pr = vis ? ex2(fmaf(s, cs, -slse[i] * kLog2e)) : 0.f;
            const float ds = pr * (dp - sdl[i]);
#pragma unroll
            for (int c = 0; c < W; ++c) {
                dv[c] = fmaf(pr, doi[c], dv[c]);
                dk[c] = fmaf(ds, qi[c], dk[c]);
            }
        }
    }
    if (!kvalid) return;
    const int64_t out = kv_base + static_cast<int64_t>(key) * p.D;
#pragma unroll
    for (int c = 0; c < W; ++c) {
        if (c0 + c < p.D) {
            p.dk[out + c0 + c] = dk[c] * p.scale;
            p.dv[out + c0 + c] = dv[c];
        }
    }
}

template <int DV>
__global__ void __launch_bounds__(threads<DV>()) bwd_dq(const BwdParams p) {
    constexpr int P = parts<DV>();
    constexpr int W = DV / P;
    __shared__ float sk[kChunk * DV], sv[kChunk * DV];
    const int tiles = (p.M + kTile - 1) / kTile;
    const int bh = blockIdx.x / tiles;
    const int row0 = (blockIdx.x - bh * tiles) * kTile;
    const int row = row0 + threadIdx.x / P;
    const int c0 = (threadIdx.x % P) * W;
    const bool rvalid = row < p.M;
    const int64_t q_base = static_cast<int64_t>(bh) * p.M * p.D;
    const int64_t kv_base = static_cast<int64_t>(bh) * p.N * p.D;
    float qr[W], dor[W], dq[W];
#pragma unroll
    for (int c = 0; c < W; ++c) {
        const bool in = rvalid && c0 + c < p.D;
        qr[c] = in ? ld_bf16(p.q + q_base + static_cast<int64_t>(row) * p.D + c0 + c) : 0.f;
        dor[c] = in ? ld_bf16(p.dout + q_base + static_cast<int64_t>(row) * p.D + c0 + c) : 0.f;
        dq[c] = 0.f;
    }
    const float lse = rvalid ? p.lse[static_cast<int64_t>(bh) * p.M + row] : -INFINITY;
    const float dl = rvalid ? p.delta[static_cast<int64_t>(bh) * p.Mpad + row] : 0.f;
    const float cs = p.scale * kLog2e;
    // Keys any row of this tile can see: all, or (causal) keys <= its last row.
    const int key_hi = p.causal ? min(p.N, min(p.M, row0 + kTile)) : p.N;
    for (int k0 = 0; k0 < key_hi; k0 += kChunk) {
        __syncthreads();
        stage<DV>(sk, p.k + kv_base, k0, p.N, p.D);
        stage<DV>(sv, p.v + kv_base, k0, p.N, p.D);
        __syncthreads();
        for (int j = 0; j < kChunk; ++j) {
            const int key = k0 + j;
            const float* kj = sk + j * DV + c0;
            const float* vj = sv + j * DV + c0;
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < W; ++c) {
                s = fmaf(qr[c], kj[c], s);
                dp = fmaf(dor[c], vj[c], dp);
            }
            s = part_sum<P>(s);
            dp = part_sum<P>(dp);
            const bool vis = rvalid && key < p.N && (!p.causal || key <= row) && lse != -INFINITY;
            const float pr = vis ? ex2(fmaf(s, cs, -lse * kLog2e)) : 0.f;
            const float ds = pr * (dp - dl);
#pragma unroll
            for (int c = 0; c < W; ++c) dq[c] = fmaf(ds, kj[c], dq[c]);
        }
    }
    if (!rvalid) return;
    const int64_t out = q_base + static_cast<int64_t>(row) * p.D;
#pragma unroll
    for (int c = 0; c < W; ++c)
        if (c0 + c < p.D) p.dq[out + c0 + c] = dq[c] * p.scale;
}

template <int DV>
cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t s) {
    const int64_t kv_blocks = static_cast<int64_t>(p.bh_count) * ((p.N + kTile - 1) / kTile);
    const int64_t q_blocks = static_cast<int64_t>(p.bh_count) * ((p.M + kTile - 1) / kTile);
    if (kv_blocks > 0x7fffffffLL || q_blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (kv_blocks > 0) bwd_dkdv<DV><<<static_cast<unsigned>(kv_blocks), threads<DV>(), 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dq<DV><<<static_cast<unsigned>(q_blocks), threads<DV>(), 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_rowdot(const BwdParams& p, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(p.bh_count) * p.Mpad;
    const bool aligned = ((reinterpret_cast<uintptr_t>(p.o) | reinterpret_cast<uintptr_t>(p.dout)) & 15u) == 0;
    if (aligned && (p.D == 64 || p.D == 128)) {
        const int rows_per_block = 8 * 4 * (p.D == 64 ? 4 : 2);   // warps x groups x rows per group
        const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        if (p.D == 64)
            bwd_rowdot_vec<8><<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
        else
            bwd_rowdot_vec<16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
        return cudaGetLastError();
    }
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    bwd_rowdot<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdParams& p, cudaStream_t s) {
    if (p.D <= 32) return launch_bwd_t<32>(p, s);
    if (p.D <= 64) return launch_bwd_t<64>(p, s);
    return launch_bwd_t<128>(p, s);
}

}  // namespace fa
