"""fa_fwd: a FlashAttention forward pass for one NVIDIA GB300 GPU (sm_103a).

The computation lives in ``libfa_fwd.so`` (hand-written CUDA: a tcgen05 /
TMA kernel for bf16, an exact-fp32 CUDA-core kernel, a tensor-core fp32
path built from three TF32 products, and a CUDA-core backward), behind the C ABI of
``include/fa_fwd.h``. This package is its thin Python binding plus the seeded
input generator the tests and the benchmark share. Importing it does not load
the library; the first call does, and raises if it has not been built.
"""

from ._binding import (FA_ERR_CUDA, FA_ERR_INVALID_ARG, FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED, FA_OK,  # noqa: F401
                       FaError, fa_bwd, fa_bwd_raw, fa_bwd_workspace_bytes, fa_fwd, fa_fwd_f32, fa_fwd_f32_raw,
                       fa_fwd_f32x3, fa_fwd_f32x3_raw, fa_fwd_f32x3_workspace_bytes,
                       fa_fwd_host, fa_fwd_host_raw,
                       fa_fwd_host_workspace_bytes, fa_fwd_noalloc, fa_fwd_noalloc_raw,
                       fa_fwd_raw, fa_fwd_splitkv, fa_fwd_splitkv_raw, fa_fwd_splitkv_suggest,
                       fa_fwd_splitkv_workspace_bytes, fa_get_device_status,
                       fa_last_error, fa_selftest_wait_timeout, fa_status_string, library_path, load_library)
