// Instantiation of the bf16 tensor-core kernel for head dimension 64.
#include "fa_bf16_kernel.cuh"

namespace fa {

cudaError_t launch_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const Bf16Params& p, bool causal, cudaStream_t s) {
    return launch_bf16<64>(q, k, v, p, causal, s);
}

}  // namespace fa
