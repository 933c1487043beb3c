// Merge of split-KV partial results.
//
// Softmax of a concatenation from the softmaxes of its pieces ("Module 08:
// FlashAttention and Memory-Efficient Kernels", section "Tiling and the
// online softmax"): if split s of a row's keys gives the normalised output
// O_s and log-sum-exp LSE_s, the whole row has
//     LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
// One warp per row; lanes read the row's partial outputs with coalesced
// loads (memory bound: splits * D * 4 bytes in, D * 2 + 4 bytes out).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kMaxSplits = 32;
constexpr int kRowsPerBlock = 8;

__global__ void __launch_bounds__(32 * kRowsPerBlock)
fa_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, uint16_t* __restrict__ o,
                  float* __restrict__ lse, int64_t rows, int D, int splits) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;
    // Lane s holds LSE_s; the row's LSE by a max-shifted sum over the lanes.
    const float l_s = (lane < splits) ? ws_lse[static_cast<int64_t>(lane) * rows + row] : -INFINITY;
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
    for (int d = lane; d < D; d += 32) {
        float acc = 0.f;
        for (int s = 0; s < splits; ++s) {
            const float w = __shfl_sync(0xffffffffu, w_lane, s);
            if (w != 0.f) acc = fmaf(w, ws_o[(static_cast<int64_t>(s) * rows + row) * D + d], acc);
        }
        const uint32_t u = __float_as_uint(acc);
        // fp32 -> bf16, round to nearest even (finite values)
        o[row * D + d] = static_cast<uint16_t>((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
    }
    if (lane == 0) lse[row] = total;
}

}  // namespace

cudaError_t launch_combine(const float* ws_o, const float* ws_lse, void* o, float* lse, int64_t rows, int D,
                           int splits, cudaStream_t s) {
    if (splits < 1 || splits > kMaxSplits) return cudaErrorInvalidValue;
    const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (blocks == 0) return cudaSuccess;
    fa_combine_kernel<<<static_cast<unsigned>(blocks), 32 * kRowsPerBlock, 0, s>>>(
        ws_o, ws_lse, static_cast<uint16_t*>(o), lse, rows, D, splits);
    return cudaGetLastError();
}

}  // namespace fa
