// fp32 attention forward on the CUDA cores, exact fp32 arithmetic.
//
// The single-head fp32 problem of "FlashAttention in Triton: A Tile-by-Tile
// Walkthrough" (its kernel computes both dots in IEEE fp32 and streams key
// tiles through a running max, sum and accumulator), generalised to a
// [B, H] batch and the top-left causal mask. Each thread owns one query row;
// a block stages 32-key tiles of K and V in shared memory, and every thread
// runs the streaming softmax of "FlashAttention-style kernel" (section "The
// loop") over them, with log2(e) folded into the scale and exp2f. Products
// are plain fp32 fused multiply-adds (no TF32, no tensor cores); the final
// division is IEEE.
//
// Compiled without fast-math: exp2f and log2f are the full-accuracy CUDA
// functions.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kRows = 64;    // query rows (threads) per block
constexpr int kKeys = 32;    // keys per shared-memory tile

template <int DMAX>
__global__ void __launch_bounds__(kRows)
fa_fwd_f32_kernel(const F32Params p, bool causal) {
    extern __shared__ float sm[];
    float* sK = sm;                    // [kKeys][DMAX]
    float* sV = sm + kKeys * DMAX;     // [kKeys][DMAX]

    const int row_blocks = (p.M + kRows - 1) / kRows;
    const int bh = blockIdx.x / row_blocks;
    const int row0 = (blockIdx.x - bh * row_blocks) * kRows;
    const int row = row0 + threadIdx.x;
    const bool valid = row < p.M;
    const int D = p.D;
    const float* qh = p.q + static_cast<size_t>(bh) * p.M * D;
    const float* kh = p.k + static_cast<size_t>(bh) * p.N * D;
    const float* vh = p.v + static_cast<size_t>(bh) * p.N * D;

    float q[DMAX], acc[DMAX];
#pragma unroll
    for (int d = 0; d < DMAX; ++d) {
        q[d] = (valid && d < D) ? qh[static_cast<size_t>(row) * D + d] : 0.f;
        acc[d] = 0.f;
    }
    const float c = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;

    // Keys any row of this block can see.
    int n_keys = p.N;
    if (causal) n_keys = min(n_keys, min(row0 + kRows, p.M));

    for (int k0 = 0; k0 < n_keys; k0 += kKeys) {
        __syncthreads();
        for (int i = threadIdx.x; i < kKeys * DMAX; i += kRows) {
            const int kr = i / DMAX, d = i % DMAX;
            const bool in = (k0 + kr < p.N) && d < D;
            sK[i] = in ? kh[static_cast<size_t>(k0 + kr) * D + d] : 0.f;
            sV[i] = in ? vh[static_cast<size_t>(k0 + kr) * D + d] : 0.f;
        }
        __syncthreads();

        float s[kKeys];
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < kKeys; ++j) {
            float dot = 0.f;
#pragma unroll
            for (int d = 0; d < DMAX; ++d) dot = fmaf(q[d], sK[j * DMAX + d], dot);
            const int key = k0 + j;
            const bool vis = key < p.N && (!causal || key <= row);
            s[j] = vis ? dot * c : -INFINITY;
            mx = fmaxf(mx, s[j]);
        }
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;   // fully masked so far
        const float alpha = exp2f(m_run - m_use);
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < kKeys; ++j) {
            s[j] = exp2f(s[j] - m_use);
            psum += s[j];
        }
        l_run = l_run * alpha + psum;
#pragma unroll
        for (int d = 0; d < DMAX; ++d) {
            float a = acc[d] * alpha;
#pragma unroll
            for (int j = 0; j < kKeys; ++j) a = fmaf(s[j], sV[j * DMAX + d], a);
            acc[d] = a;
        }
        m_run = m_new;
    }

    if (valid) {
        float* orow = p.o + (static_cast<size_t>(bh) * p.M + row) * D;
#pragma unroll
        for (int d = 0; d < DMAX; ++d)
            if (d < D) orow[d] = (l_run > 0.f) ? acc[d] / l_run : 0.f;
        p.lse[static_cast<size_t>(bh) * p.M + row] =
            (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }
}

template <int DMAX>
cudaError_t launch_f32_t(const F32Params& p, bool causal, cudaStream_t s) {
    const int smem = 2 * kKeys * DMAX * static_cast<int>(sizeof(float));
    auto kern = fa_fwd_f32_kernel<DMAX>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    const long long blocks = static_cast<long long>((p.M + kRows - 1) / kRows) * p.bh_count;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(blocks), kRows, smem, s>>>(p, causal);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_f32(const F32Params& p, bool causal, cudaStream_t s) {
    if (p.D <= 32) return launch_f32_t<32>(p, causal, s);
    if (p.D <= 64) return launch_f32_t<64>(p, causal, s);
    return launch_f32_t<128>(p, causal, s);
}

}  // namespace fa
