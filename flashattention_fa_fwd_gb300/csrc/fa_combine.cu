// Merge of split-KV partial results.
//
// Softmax of a concatenation from the softmaxes of its pieces ("Module 08:
// FlashAttention and Memory-Efficient Kernels", section "Tiling and the
// online softmax"): if split s of a row's keys gives the normalised output
// O_s and log-sum-exp LSE_s, the whole row has
//     LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
// One warp per row; lane l handles columns 4l .. 4l + 3 (D <= 128, a
// multiple of 4), reading every split's partial output with one 16-byte load
// issued before any weight is known and writing four bf16 values at once
// (memory bound: splits * D * 4 bytes in, D * 2 + 4 bytes out).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kMaxSplits = 32;
constexpr int kRowsPerBlock = 8;

__device__ __forceinline__ uint32_t bf16_bits(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;   // round to nearest even (finite values)
}

__global__ void __launch_bounds__(32 * kRowsPerBlock)
fa_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, uint16_t* __restrict__ o,
                  float* __restrict__ lse, int64_t rows, int D, int splits) {
    // Launched as a programmatic dependent of the split kernel: wait here
    // until that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;
    // Lane s holds LSE_s; the row's LSE by a max-shifted sum over the lanes.
    const float l_s = (lane < splits) ? ws_lse[static_cast<int64_t>(lane) * rows + row] : -INFINITY;
    const int d = 4 * lane;
    const bool cols = d < D;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float mx = l_s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float e = (l_s == -INFINITY) ? 0.f : expf(l_s - mx);
    float sum = e;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const bool any = mx != -INFINITY;
    const float total = any ? mx + logf(sum) : -INFINITY;
    const float w_lane = any ? e / sum : 0.f;   // exp(LSE_s - LSE) of lane s
    // Four splits at a time: their loads are in flight together. A split
    // with weight 0 (no visible key) contributes nothing, whatever it holds.
    for (int s0 = 0; s0 < splits; s0 += 4) {
        float4 x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            x[i] = (cols && s0 + i < splits)
                       ? *reinterpret_cast<const float4*>(ws_o + (static_cast<int64_t>(s0 + i) * rows + row) * D + d)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float w = __shfl_sync(0xffffffffu, w_lane, (s0 + i) & 31);
            if (s0 + i < splits && w != 0.f) {
                acc.x = fmaf(w, x[i].x, acc.x);
                acc.y = fmaf(w, x[i].y, acc.y);
                acc.z = fmaf(w, x[i].z, acc.z);
                acc.w = fmaf(w, x[i].w, acc.w);
            }
        }
    }
    if (cols) {
        const uint2 packed = make_uint2(bf16_bits(acc.x) | (bf16_bits(acc.y) << 16),
                                        bf16_bits(acc.z) | (bf16_bits(acc.w) << 16));
        *reinterpret_cast<uint2*>(o + row * D + d) = packed;
    }
    if (lane == 0) lse[row] = total;
}

}  // namespace

cudaError_t launch_combine(const float* ws_o, const float* ws_lse, void* o, float* lse, int64_t rows, int D,
                           int splits, cudaStream_t s) {
    if (splits < 1 || splits > kMaxSplits || D > 128 || D % 4 != 0) return cudaErrorInvalidValue;
    const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (blocks == 0) return cudaSuccess;
    // Programmatic dependent launch: the merge's launch overlaps the end of
    // the split kernel; the kernel waits for that grid before reading.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(32 * kRowsPerBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fa_combine_kernel, ws_o, ws_lse, static_cast<uint16_t*>(o), lse, rows, D, splits);
}

}  // namespace fa
