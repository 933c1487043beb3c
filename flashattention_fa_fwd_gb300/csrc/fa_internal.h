// Internal interface between the host entry points (fa_api.cu) and the
// kernel translation units. Not installed; not part of the C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fa {

// Bits a kernel ORs into the per-device status word.
constexpr uint32_t DEV_ERR_TIMEOUT = 1u;  // a pipeline wait ran out of time

// Arguments of the bf16 tensor-core kernel that are not tensor maps.
struct Bf16Params {
    void* o;             // [BH, M, D] bf16
    float* lse;          // [BH, M] fp32
    uint32_t* err;       // device status word
    int bh_count;        // B * H
    int M;
    int N;
    int n_pairs;         // query-tile units per head: ceil(M / 256) pairs of 128-row
                         // tiles, or ceil(M / 128) single tiles when `single`
    int single;          // 1: units of one query tile (tile 1 idle), when every
                         // tile fits on its own SM; a row's arithmetic is the
                         // same either way
    int splits;          // key-range splits per unit (1 = no split)
    int num_units;       // bh_count * n_pairs * splits
    float* ws_o;         // splits > 1: [splits, BH, M, D] fp32 partial outputs
    float* ws_lse;       // splits > 1: [splits, BH, M] fp32 partial log-sum-exps
    int heads_per_group; // causal unit order: heads that share a group (longest units first within it)
    float scale_log2;    // scale * log2(e)
    int* sched;          // [2]: next unit to claim, CTAs finished. Zero when the
                         // launch starts; the launch's last CTA sets both back
                         // to zero, so a slot serves one running launch at a time.
};

// Launches the bf16 kernel for head dimension D (64, 96 or 128); the three
// maps are 3-D {D, rows, B*H} bf16 maps with a {64, rows, 1} box and 128-byte
// swizzle: 128 rows for Q, and for K and V except at D = 64 without key
// splits (kv_box_rows), whose kernel streams 64-key tiles. Returns the launch
// error.
constexpr int kv_box_rows(int64_t D, int splits) { return (D == 64 && splits == 1) ? 64 : 128; }

cudaError_t launch_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const Bf16Params& p, bool causal, cudaStream_t s);
cudaError_t launch_bf16_d96(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const Bf16Params& p, bool causal, cudaStream_t s);
cudaError_t launch_bf16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const Bf16Params& p, bool causal, cudaStream_t s);

// Arguments of the fp32 CUDA-core kernel.
struct F32Params {
    const float* q;
    const float* k;
    const float* v;
    float* o;
    float* lse;
    int bh_count;
    int M;
    int N;
    int D;
    float scale_log2;
};

cudaError_t launch_f32(const F32Params& p, bool causal, cudaStream_t s);

// Arguments of the backward kernels: bf16 inputs of the forward plus its O,
// LSE and the output gradient dO; fp32 gradients out.
struct BwdParams {
    const __nv_bfloat16* q;      // [BH, M, D]
    const __nv_bfloat16* k;      // [BH, N, D]
    const __nv_bfloat16* v;      // [BH, N, D]
    const __nv_bfloat16* o;      // [BH, M, D] forward output
    const __nv_bfloat16* dout;   // [BH, M, D] gradient of the loss with respect to O
    const float* lse;            // [BH, M] forward log-sum-exp (natural log)
    float* delta;                // [BH, Mpad] workspace: sum_d dO * O per row (0 past M)
    float* lse2;                 // [BH, Mpad] workspace: lse * log2(e) (+inf past M)
    uint32_t* err;               // device status word (tensor-core kernels' bounded waits)
    int Mpad;                    // M rounded up to a multiple of 128
    float* dq;                   // [BH, M, D]
    float* dk;                   // [BH, N, D]
    float* dv;                   // [BH, N, D]
    int bh_count;
    int M;
    int N;
    int D;
    float scale;
    int causal;
    int* sched;                  // [2] work counters of the persistent dK/dV kernel
                                 // (as Bf16Params::sched)
};

// Row dots Dl and the padded base-2 LSE (both into the workspace) on `s`.
cudaError_t launch_bwd_rowdot(const BwdParams& p, cudaStream_t s);

// The CUDA-core dK/dV and dQ kernels (after launch_bwd_rowdot) on `s`.
cudaError_t launch_bwd(const BwdParams& p, cudaStream_t s);

// The tensor-core dK/dV and dQ kernels (after launch_bwd_rowdot) on `s`, for
// D in {64, 96, 128}; maps are fa_fwd's bf16 {D, rows, B*H} maps of Q, K, V
// and dO.
cudaError_t launch_bwd_tc(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                          const BwdParams& p, cudaStream_t s);

// Arguments of the fp32 tensor-core path (three TF32 products per matrix
// product): fp32 Q, K, V in, fp32 O and LSE out.
struct X3Params {
    const float* q;   // [BH, M, D]
    const float* k;   // [BH, N, D]
    const float* v;   // [BH, N, D]
    float* o;         // [BH, M, D]
    float* lse;       // [BH, M]
    uint8_t* ws;      // K and V split into TF32 hi/lo parts, 32-key tile images (x3_workspace_bytes)
    uint32_t* err;    // device status word
    int bh_count;
    int M;
    int N;
    int D;            // 32, 64, 96 or 128
    float scale;
    int causal;
};

// Bytes of the K/V image workspace for B*H heads of N keys of width D.
int64_t x3_workspace_bytes(int64_t bh, int64_t N, int64_t D);

// Launches the split pre-pass and the attention kernel on `s`.
cudaError_t launch_x3(const X3Params& p, cudaStream_t s);

// Merges split-KV partial results: for every row, LSE = ln sum_s exp(LSE_s)
// and O = sum_s exp(LSE_s - LSE) O_s, written as bf16 O and fp32 LSE.
cudaError_t launch_combine(const float* ws_o, const float* ws_lse, void* o, float* lse, int64_t rows, int D,
                           int splits, cudaStream_t s);

}  // namespace fa
