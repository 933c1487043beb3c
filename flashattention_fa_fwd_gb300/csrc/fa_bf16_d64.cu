// Instantiation of the bf16 tensor-core kernels for head dimension 64: one
// query tile per CTA and four CTAs per SM (fa_bf16_q1.cuh) for the forward
// itself; the two-tile kernel (fa_bf16_kernel.cuh) for key-range splits.
#include "fa_bf16_kernel.cuh"
#include "fa_bf16_q1.cuh"

namespace fa {

cudaError_t launch_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const Bf16Params& p, bool causal, cudaStream_t s) {
    if (p.splits > 1) return launch_bf16<64>(q, k, v, p, causal, s);
    const int sms = sm_count_cached();
    if (sms <= 0) return cudaErrorInvalidDevice;
    Bf16Params p1 = p;
    p1.num_units = p.bh_count * ((p.M + q1::Cfg::BM - 1) / q1::Cfg::BM);   // one query tile per unit
    return launch_bf16_q1(q, k, v, p1, causal, s, sms);
}

}  // namespace fa
