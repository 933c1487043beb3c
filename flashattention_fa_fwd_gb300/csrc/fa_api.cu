// Host side of libfa_fwd.so: the C ABI declared in include/fa_fwd.h.
//
// Validates arguments before anything touches the GPU, builds the TMA
// tensor maps, picks the kernel for the head dimension and launches it on
// the caller's stream. The library never synchronises inside fa_fwd /
// fa_fwd_f32 and allocates nothing per call; the only allocation is one small
// block of device state per device (the status word and the work counters
// of the bf16 kernel's unit scheduler), made on the first call on that
// device.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <atomic>
#include <cstdio>
#include <mutex>

#include "fa_fwd.h"
#include "fa_internal.h"
#include "ptx.cuh"

#define FA_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local char g_msg[512] = "";

fa_status fail(fa_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
// Work-counter slots of the bf16 kernel's unit scheduler. An ordinary launch
// takes the next of kSchedSlots slots in turn; before it reuses a slot, its
// stream waits for the event recorded after the slot's previous launch, so
// two running launches never share a counter (a 65th launch in flight
// queues behind the first instead). A launch captured into a CUDA graph
// cannot wait on events recorded outside the capture: it takes the next of
// kGraphSlots slots reserved for captured launches, which ordinary launches
// never touch.
constexpr int kSchedSlots = 64;
constexpr int kGraphSlots = 64;
struct DeviceState {
    uint32_t status;                   // the device status word
    uint32_t pad;
    int sched[kSchedSlots][2];         // per launch: next unit, CTAs finished
    int graph_sched[kGraphSlots][2];   // the same, for launches captured into graphs
};
struct SlotRing {
    std::mutex mu[kSchedSlots];        // held from a slot's wait to its event record
    cudaEvent_t done[kSchedSlots] = {};// recorded after the slot's last launch
};
std::mutex g_mu;
uint32_t* g_status_word[kMaxDevices] = {};
DeviceState* g_state[kMaxDevices] = {};
SlotRing g_slots[kMaxDevices];
std::atomic<uint32_t> g_launch_seq[kMaxDevices];
std::atomic<uint32_t> g_graph_seq[kMaxDevices];
int g_arch[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
// Device address, per device, of fa_fwd_noalloc's static scratch array
// (looked up on that entry point's first call on the device); word 0 is its
// status word, which fa_get_device_status also reads.
uint32_t* g_noalloc_scratch_addr[kMaxDevices] = {};

// Per-device set-up on first use: architecture check, device state (status
// word, work counters), and the driver's tensor-map encoder (fetched through
// the runtime, so the library does not link libcuda).
fa_status device_setup(bool need_encoder, uint32_t** status_word) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_arch[dev] == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        g_arch[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_arch[dev] != 1) return fail(FA_ERR_UNSUPPORTED, "device %d is not sm_103 (this library is built for sm_103a only)", dev);
    if (g_state[dev] == nullptr) {
        DeviceState* w = nullptr;
        e = cudaMalloc(&w, sizeof(DeviceState));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(device state)");
        e = cudaMemset(w, 0, sizeof(DeviceState));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaFree(w);
            return cuda_fail(e, "clearing the device state");
        }
        g_state[dev] = w;
        g_status_word[dev] = &w->status;
    }
    if (need_encoder && g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *status_word = g_status_word[dev];
    return FA_OK;
}

// Runs launch(sched) -- one launch of the bf16 kernel on stream `s` -- with a
// work-counter pair that no other running launch uses (device_setup must
// have succeeded on the current device). Ordinary launches cycle through
// kSchedSlots pairs: the stream first waits for the event recorded after the
// pair's previous launch, and the event is recorded again after this one,
// all under the slot's lock so that concurrent host threads cannot
// interleave their waits and records. Launches captured into a graph cycle
// through kGraphSlots pairs of their own without events (a capture cannot
// wait on an event recorded outside it); a graph's launch keeps its pair for
// every replay, so replays of the same graph must not overlap one another
// (as for any graph whose nodes share memory).
template <class Launch>
fa_status with_sched_slot(cudaStream_t s, Launch&& launch) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    DeviceState* state = g_state[dev];
    if (cs != cudaStreamCaptureStatusNone) {
        const uint32_t slot = g_graph_seq[dev].fetch_add(1, std::memory_order_relaxed) % kGraphSlots;
        return launch(state->graph_sched[slot]);
    }
    const uint32_t slot = g_launch_seq[dev].fetch_add(1, std::memory_order_relaxed) % kSchedSlots;
    SlotRing& ring = g_slots[dev];
    std::lock_guard<std::mutex> lock(ring.mu[slot]);
    if (ring.done[slot] == nullptr) {
        e = cudaEventCreateWithFlags(&ring.done[slot], cudaEventDisableTiming);
        if (e != cudaSuccess) {
            ring.done[slot] = nullptr;
            return cuda_fail(e, "creating a work-counter event");
        }
    } else {
        e = cudaStreamWaitEvent(s, ring.done[slot], 0);
        if (e != cudaSuccess) return cuda_fail(e, "waiting for the work counters' previous launch");
    }
    const fa_status st = launch(state->sched[slot]);
    if (st != FA_OK) return st;
    e = cudaEventRecord(ring.done[slot], s);
    if (e != cudaSuccess) return cuda_fail(e, "recording the work counters' event");
    return FA_OK;
}

// Causal units are claimed longest first inside groups of this many heads:
// small enough that the groups in flight keep their K and V in L2, large
// enough that the last group has many more units than CTAs, so the short
// units balance the end of the launch (8-head groups left CTAs idle for 4 %
// of a causal 4K launch at D = 128; 16 measured +2.1 %).
constexpr int64_t kCausalHeadsPerGroup = 16;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    if (abytes <= 0 || bbytes <= 0 || a == nullptr || b == nullptr) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

// Shape and pointer checks shared by both entry points. Sets *empty when
// there is nothing to compute.
fa_status validate(const void* q, const void* k, const void* v, const void* o, const void* lse, int64_t B,
                   int64_t H, int64_t M, int64_t N, int64_t D, float scale, int64_t elem, bool* empty) {
    if (B < 0 || H < 0 || M < 0 || N < 0) return fail(FA_ERR_INVALID_ARG, "B, H, M and N must be >= 0");
    if (D < 1) return fail(FA_ERR_INVALID_ARG, "D must be >= 1 (got %lld)", (long long)D);
    if (!std::isfinite(scale) || !(scale > 0.f))
        return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0 (got %g)", (double)scale);
    const int64_t kInt = 0x7fffffff;
    if (B > kInt || H > kInt || M > kInt || N > kInt || D > kInt || (H > 0 && B > kInt / H))
        return fail(FA_ERR_INVALID_ARG, "sizes exceed the 32-bit index range");
    const int64_t bh = B * H;
    // byte counts must fit in int64
    const int64_t lim = INT64_MAX / 16;
    if ((bh > 0 && M > lim / bh) || (bh > 0 && N > lim / bh) || (bh * M > 0 && D > lim / (bh * M)) ||
        (bh * N > 0 && D > lim / (bh * N)))
        return fail(FA_ERR_INVALID_ARG, "tensor sizes overflow");
    const int64_t qbytes = bh * M * D * elem, kvbytes = bh * N * D * elem, lbytes = bh * M * 4;
    *empty = (bh == 0 || M == 0);
    if (*empty) return FA_OK;
    if (q == nullptr || o == nullptr || lse == nullptr) return fail(FA_ERR_INVALID_ARG, "q, o and lse must not be null");
    if (N > 0 && (k == nullptr || v == nullptr)) return fail(FA_ERR_INVALID_ARG, "k and v must not be null when N > 0");
    if (!aligned(q, 16) || !aligned(o, 16) || (N > 0 && (!aligned(k, 16) || !aligned(v, 16))))
        return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
    if (!aligned(lse, 4)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    if (overlaps(o, qbytes, q, qbytes) || overlaps(o, qbytes, k, kvbytes) || overlaps(o, qbytes, v, kvbytes) ||
        overlaps(lse, lbytes, q, qbytes) || overlaps(lse, lbytes, k, kvbytes) || overlaps(lse, lbytes, v, kvbytes) ||
        overlaps(o, qbytes, lse, lbytes))
        return fail(FA_ERR_INVALID_ARG, "o and lse must not overlap the inputs or each other");
    return FA_OK;
}

// 3-D {D, rows, B*H} bf16 map, box_rows x 64-column box, 128-byte swizzle.
fa_status encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t bh, int64_t D, int box_rows = 128) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(bh)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(rows * D * 2)};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                          elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return FA_OK;
}

constexpr double kLog2e = 1.4426950408889634;

}  // namespace

namespace {

// The bf16 forward on device buffers whose arguments have been checked:
// tensor maps, parameters and the launch on `s`.
fa_status launch_fwd_checked(const void* q, const void* k, const void* v, void* o, float* lse, int64_t bh,
                             int64_t M, int64_t N, int64_t D, float scale, int causal, cudaStream_t s);

}  // namespace

FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                        int64_t M, int64_t N, int64_t D, float scale, int causal, void* stream) {
    bool empty = false;
    fa_status st = validate(q, k, v, o, lse, B, H, M, N, D, scale, 2, &empty);
    if (st != FA_OK) return st;
    if (D != 64 && D != 96 && D != 128)
        return fail(FA_ERR_UNSUPPORTED, "bf16 fa_fwd supports D in {64, 96, 128} (got %lld)", (long long)D);
    if (empty) return FA_OK;
    return launch_fwd_checked(q, k, v, o, lse, B * H, M, N, D, scale, causal, static_cast<cudaStream_t>(stream));
}

namespace {

// Work units of the two-tile kernel without key splits: pairs of 128-row
// query tiles, or single tiles when every tile fits on its own SM. A CTA
// steps one tile through the keys in ~3/4 of the time it takes for a pair,
// so single tiles win while they need one wave and pairs would leave SMs
// idle (the cross-attention workload: 64 pairs, 128 tiles, 152 SMs; +7 %),
// and lose once they need two. A row's arithmetic is the same either way,
// so the choice never changes a result. At D = 64 the one-tile kernel runs
// and sets its own units.
void set_units(fa::Bf16Params& p, int64_t bh, int64_t M) {
    const int64_t pairs = (M + 255) / 256, tiles = (M + 127) / 128;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 0;
    p.single = (tiles > pairs && bh * tiles <= sms) ? 1 : 0;
    p.n_pairs = static_cast<int>(p.single ? tiles : pairs);
    p.splits = 1;
    p.num_units = static_cast<int>(bh * p.n_pairs);
}

fa_status launch_fwd_checked(const void* q, const void* k, const void* v, void* o, float* lse, int64_t bh,
                             int64_t M, int64_t N, int64_t D, float scale, int causal, cudaStream_t s) {
    fa_status st;
    const int64_t n_pairs = (M + 255) / 256;
    if (bh * n_pairs > 0x7fffffffLL) return fail(FA_ERR_UNSUPPORTED, "too many query tiles for one launch");
    uint32_t* word = nullptr;
    st = device_setup(true, &word);
    if (st != FA_OK) return st;

    CUtensorMap mq, mk, mv;
    if ((st = encode_map(&mq, q, M, bh, D)) != FA_OK) return st;
    if (N > 0) {
        if ((st = encode_map(&mk, k, N, bh, D, fa::kv_box_rows(D, 1))) != FA_OK) return st;
        if ((st = encode_map(&mv, v, N, bh, D, fa::kv_box_rows(D, 1))) != FA_OK) return st;
    } else {
        mk = mq;  // never read: no key tiles exist
        mv = mq;
    }
    fa::Bf16Params p;
    p.o = o;
    p.lse = lse;
    p.err = word;
    p.bh_count = static_cast<int>(bh);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    set_units(p, bh, M);
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    p.heads_per_group = static_cast<int>(bh < kCausalHeadsPerGroup ? bh : kCausalHeadsPerGroup);
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    return with_sched_slot(s, [&](int* sched) -> fa_status {
        p.sched = sched;
        cudaError_t e;
        switch (D) {
            case 64: e = fa::launch_bf16_d64(mq, mk, mv, p, causal != 0, s); break;
            case 96: e = fa::launch_bf16_d96(mq, mk, mv, p, causal != 0, s); break;
            default: e = fa::launch_bf16_d128(mq, mk, mv, p, causal != 0, s); break;
        }
        return e == cudaSuccess ? FA_OK : cuda_fail(e, "launching the bf16 kernel");
    });
}

}  // namespace

FA_API fa_status fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int64_t B,
                            int64_t H, int64_t M, int64_t N, int64_t D, float scale, int causal, void* stream) {
    bool empty = false;
    fa_status st = validate(q, k, v, o, lse, B, H, M, N, D, scale, 4, &empty);
    if (st != FA_OK) return st;
    if (D > 128) return fail(FA_ERR_UNSUPPORTED, "fp32 fa_fwd_f32 supports D <= 128 (got %lld)", (long long)D);
    if (empty) return FA_OK;
    uint32_t* word = nullptr;
    st = device_setup(false, &word);
    if (st != FA_OK) return st;
    fa::F32Params p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.bh_count = static_cast<int>(B * H);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.D = static_cast<int>(D);
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    cudaError_t e = fa::launch_f32(p, causal != 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "launching the fp32 kernel");
    return FA_OK;
}

FA_API int64_t fa_fwd_f32x3_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D) {
    if (B < 0 || H < 0 || N < 0 || D < 0) return -1;
    if (B > 0x7fffffff || H > 0x7fffffff || N > 0x7fffffff || D > 256) return -1;
    return fa::x3_workspace_bytes(B * H, N, D);
}

FA_API fa_status fa_fwd_f32x3(const float* q, const float* k, const float* v, float* o, float* lse, int64_t B,
                              int64_t H, int64_t M, int64_t N, int64_t D, float scale, int causal, void* workspace,
                              int64_t workspace_bytes, void* stream) {
    bool empty = false;
    fa_status st = validate(q, k, v, o, lse, B, H, M, N, D, scale, 4, &empty);
    if (st != FA_OK) return st;
    if (D != 32 && D != 64 && D != 96 && D != 128)
        return fail(FA_ERR_UNSUPPORTED, "fa_fwd_f32x3 supports D in {32, 64, 96, 128} (got %lld)", (long long)D);
    if (empty) return FA_OK;
    const int64_t bh = B * H;
    const int64_t need = fa_fwd_f32x3_workspace_bytes(B, H, N, D);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need))
        return fail(FA_ERR_INVALID_ARG, "workspace of %lld bytes needed (got %lld)", (long long)need,
                    (long long)workspace_bytes);
    if (need > 0 && !aligned(workspace, 128)) return fail(FA_ERR_INVALID_ARG, "workspace must be 128-byte aligned");
    const int64_t qb = bh * M * D * 4, kb = bh * N * D * 4;
    if (overlaps(workspace, need, q, qb) || overlaps(workspace, need, k, kb) || overlaps(workspace, need, v, kb) ||
        overlaps(workspace, need, o, qb) || overlaps(workspace, need, lse, bh * M * 4))
        return fail(FA_ERR_INVALID_ARG, "workspace must not overlap the tensors");
    uint32_t* word = nullptr;
    if ((st = device_setup(false, &word)) != FA_OK) return st;
    fa::X3Params p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.ws = static_cast<uint8_t*>(workspace);
    p.err = word;
    p.bh_count = static_cast<int>(bh);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.D = static_cast<int>(D);
    p.scale = scale;
    p.causal = causal != 0;
    const cudaError_t e = fa::launch_x3(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "launching the fp32 tensor-core kernels");
    return FA_OK;
}

FA_API fa_status fa_get_device_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return FA_OK;
    // Two status words: the one in the library's device state (every entry
    // point but fa_fwd_noalloc) and word 0 of fa_fwd_noalloc's static array.
    // Reading and clearing them allocates nothing.
    uint32_t* words[2];
    {
        std::lock_guard<std::mutex> lock(g_mu);
        words[0] = g_status_word[dev];
        words[1] = g_noalloc_scratch_addr[dev];
    }
    uint32_t h = 0;
    for (uint32_t* w : words) {
        if (w == nullptr) continue;
        uint32_t x = 0;
        e = cudaMemcpy(&x, w, sizeof(x), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
        if (x != 0) {
            e = cudaMemset(w, 0, sizeof(uint32_t));
            if (e == cudaSuccess) e = cudaDeviceSynchronize();
            if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
            h |= x;
        }
    }
    if (h & fa::DEV_ERR_TIMEOUT) return fail(FA_ERR_TIMEOUT, "a kernel gave up waiting on its pipeline (status 0x%x)", h);
    if (h != 0) return fail(FA_ERR_CUDA, "device status word 0x%x", h);
    return FA_OK;
}

FA_API const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
        default: return "FA_ERR_UNKNOWN";
    }
}

FA_API const char* fa_last_error(void) { return g_msg; }

// ---------------------------------------------------------------------------
// Split-KV: each query tile's keys are cut into `num_splits` contiguous ranges
// processed by different CTAs, which write partial results into a caller-
// provided workspace; a merge kernel combines them. Worth it when B*H*M is
// too small to fill the GPU (few query tiles, long keys).
// ---------------------------------------------------------------------------
namespace {

int64_t splitkv_bytes(int64_t bh, int64_t M, int64_t D, int64_t splits) {
    return splits * bh * M * (D + 1) * static_cast<int64_t>(sizeof(float));
}

}  // namespace

FA_API int64_t fa_fwd_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t M, int64_t D, int num_splits) {
    if (B < 0 || H < 0 || M < 0 || D < 1 || num_splits < 1) return -1;
    if (num_splits == 1) return 0;
    return splitkv_bytes(B * H, M, D, num_splits);
}

FA_API int fa_fwd_splitkv_suggest(int64_t B, int64_t H, int64_t M, int64_t N, int causal) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    const int64_t units = B * H * ((M + 255) / 256);
    const int64_t nkv = (N + 127) / 128;
    if (units <= 0 || nkv < 4 || causal) return 1;
    int64_t s = sms / units;                 // fill the SMs once, no more
    if (s > nkv / 2) s = nkv / 2;            // at least two key tiles per split
    if (s > 16) s = 16;
    return s < 1 ? 1 : static_cast<int>(s);
}

FA_API fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                                int64_t H, int64_t M, int64_t N, int64_t D, float scale, int causal, int num_splits,
                                void* workspace, int64_t workspace_bytes, void* stream) {
    bool empty = false;
    fa_status st = validate(q, k, v, o, lse, B, H, M, N, D, scale, 2, &empty);
    if (st != FA_OK) return st;
    if (D != 64 && D != 96 && D != 128)
        return fail(FA_ERR_UNSUPPORTED, "bf16 fa_fwd_splitkv supports D in {64, 96, 128} (got %lld)", (long long)D);
    if (num_splits < 1 || num_splits > 16)
        return fail(FA_ERR_INVALID_ARG, "num_splits must be in [1, 16] (got %d)", num_splits);
    if (num_splits == 1) return fa_fwd(q, k, v, o, lse, B, H, M, N, D, scale, causal, stream);
    const int64_t bh = B * H;
    const int64_t need = splitkv_bytes(bh, M, D, num_splits);
    if (empty) return FA_OK;
    if (workspace == nullptr || workspace_bytes < need)
        return fail(FA_ERR_INVALID_ARG, "workspace of %lld bytes needed (got %lld)", (long long)need,
                    (long long)workspace_bytes);
    if (!aligned(workspace, 16)) return fail(FA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    const int64_t qbytes = bh * M * D * 2, kvbytes = bh * N * D * 2;
    if (overlaps(workspace, need, q, qbytes) || overlaps(workspace, need, k, kvbytes) ||
        overlaps(workspace, need, v, kvbytes) || overlaps(workspace, need, o, qbytes) ||
        overlaps(workspace, need, lse, bh * M * 4))
        return fail(FA_ERR_INVALID_ARG, "workspace must not overlap the tensors");
    const int64_t n_pairs = (M + 255) / 256;
    if (bh * n_pairs * num_splits > 0x7fffffffLL) return fail(FA_ERR_UNSUPPORTED, "too many work units for one launch");
    uint32_t* word = nullptr;
    st = device_setup(true, &word);
    if (st != FA_OK) return st;
    CUtensorMap mq, mk, mv;
    if ((st = encode_map(&mq, q, M, bh, D)) != FA_OK) return st;
    if (N > 0) {
        if ((st = encode_map(&mk, k, N, bh, D, fa::kv_box_rows(D, num_splits))) != FA_OK) return st;
        if ((st = encode_map(&mv, v, N, bh, D, fa::kv_box_rows(D, num_splits))) != FA_OK) return st;
    } else {
        mk = mq;
        mv = mq;
    }
    fa::Bf16Params p;
    p.o = o;
    p.lse = lse;
    p.err = word;
    p.bh_count = static_cast<int>(bh);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.n_pairs = static_cast<int>(n_pairs);
    p.single = 0;
    p.splits = num_splits;
    p.num_units = static_cast<int>(bh * n_pairs * num_splits);
    p.ws_o = static_cast<float*>(workspace);
    p.ws_lse = p.ws_o + num_splits * bh * M * D;
    p.heads_per_group = static_cast<int>(bh < kCausalHeadsPerGroup ? bh : kCausalHeadsPerGroup);
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = with_sched_slot(s, [&](int* sched) -> fa_status {
        p.sched = sched;
        cudaError_t err;
        switch (D) {
            case 64: err = fa::launch_bf16_d64(mq, mk, mv, p, causal != 0, s); break;
            case 96: err = fa::launch_bf16_d96(mq, mk, mv, p, causal != 0, s); break;
            default: err = fa::launch_bf16_d128(mq, mk, mv, p, causal != 0, s); break;
        }
        return err == cudaSuccess ? FA_OK : cuda_fail(err, "launching the bf16 kernel");
    });
    if (st != FA_OK) return st;
    cudaError_t e = fa::launch_combine(p.ws_o, p.ws_lse, o, lse, bh * M, static_cast<int>(D), num_splits, s);
    if (e != cudaSuccess) return cuda_fail(e, "launching the split merge");
    return FA_OK;
}

// ---------------------------------------------------------------------------
// fa_fwd_noalloc: the bf16 forward for callers that cannot allocate device
// memory.
//
// fa_fwd keeps the kernel's scratch memory (its status word and the work
// counters its CTAs claim units from) in a buffer it cudaMallocs on its
// first call on each device. Some callers
// cannot allow that: applications whose own caching allocator or memory
// pool already owns all device memory (a cudaMalloc from a library can fail
// or defragment their pool), serving loops that must not take the implicit
// device synchronisation a cudaMalloc/cudaFree can cause, and processes
// under a fixed device-memory quota. This variant runs the same kernel with
// its scratch in a file-scope static device array instead, so it never
// calls cudaMalloc, cudaFree or any allocating routine.
//
// The array (kNoAllocScratchWords 32-bit words, 256 bytes) lives on every
// GPU that loads the library until the process exits. Host code cannot use
// the array's name as a device address; the first call on each device looks
// the address up with cudaGetSymbolAddress (with that device current) and
// caches it, so that first call should come before any stream capture. All
// calls share the array and it keeps the last call's contents: each call
// clears the two scheduler counters the kernel expects to start at zero
// (cudaMemsetAsync on the caller's stream, before the launch); the status
// word (word 0) keeps a recorded failure until fa_get_device_status reads
// and clears it. Calls that overlap on the GPU (concurrent streams, or
// several host threads) race on the array: they share the unit counter, so
// work units can be skipped or done twice and O and LSE can be wrong.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocScratchWords = 64;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchWords];

// Words of scratch the bf16 kernel needs, whatever the problem size: its
// status word (word 0) and the two counters of its unit scheduler (words 1
// and 2: next unit to claim, CTAs finished).
constexpr int kBf16ScratchWords = 3;

fa_status noalloc_setup(uint32_t** scratch) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_arch[dev] == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        g_arch[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_arch[dev] != 1) return fail(FA_ERR_UNSUPPORTED, "device %d is not sm_103 (this library is built for sm_103a only)", dev);
    if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (g_noalloc_scratch_addr[dev] == nullptr) {
        uint32_t* ptr = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_noalloc_scratch_addr[dev] = ptr;
    }
    *scratch = g_noalloc_scratch_addr[dev];
    return FA_OK;
}

}  // namespace

FA_API fa_status fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                                int64_t H, int64_t M, int64_t N, int64_t D, float scale, int causal,
                                void* stream) {
    bool empty = false;
    fa_status st = validate(q, k, v, o, lse, B, H, M, N, D, scale, 2, &empty);
    if (st != FA_OK) return st;
    if (D != 64 && D != 96 && D != 128)
        return fail(FA_ERR_UNSUPPORTED, "bf16 fa_fwd_noalloc supports D in {64, 96, 128} (got %lld)", (long long)D);
    if (kBf16ScratchWords > kNoAllocScratchWords)
        return fail(FA_ERR_UNSUPPORTED, "the kernel needs %d scratch words; the static buffer holds %d",
                    kBf16ScratchWords, kNoAllocScratchWords);
    if (empty) return FA_OK;
    const int64_t bh = B * H;
    const int64_t n_pairs = (M + 255) / 256;
    if (bh * n_pairs > 0x7fffffffLL) return fail(FA_ERR_UNSUPPORTED, "too many query tiles for one launch");
    uint32_t* scratch = nullptr;
    st = noalloc_setup(&scratch);
    if (st != FA_OK) return st;

    CUtensorMap mq, mk, mv;
    if ((st = encode_map(&mq, q, M, bh, D)) != FA_OK) return st;
    if (N > 0) {
        if ((st = encode_map(&mk, k, N, bh, D, fa::kv_box_rows(D, 1))) != FA_OK) return st;
        if ((st = encode_map(&mv, v, N, bh, D, fa::kv_box_rows(D, 1))) != FA_OK) return st;
    } else {
        mk = mq;
        mv = mq;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Word 0, the status word, stays as it is until fa_get_device_status
    // reads and clears it; the two scheduler counters must start at zero.
    cudaError_t e = cudaMemsetAsync(scratch + 1, 0, (kBf16ScratchWords - 1) * sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the static scratch");
    fa::Bf16Params p;
    p.o = o;
    p.lse = lse;
    p.err = scratch;
    p.bh_count = static_cast<int>(bh);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    set_units(p, bh, M);
    p.ws_o = nullptr;
    p.ws_lse = nullptr;
    p.heads_per_group = static_cast<int>(bh < kCausalHeadsPerGroup ? bh : kCausalHeadsPerGroup);
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * kLog2e);
    p.sched = reinterpret_cast<int*>(scratch + 1);
    switch (D) {
        case 64: e = fa::launch_bf16_d64(mq, mk, mv, p, causal != 0, s); break;
        case 96: e = fa::launch_bf16_d96(mq, mk, mv, p, causal != 0, s); break;
        default: e = fa::launch_bf16_d128(mq, mk, mv, p, causal != 0, s); break;
    }
    if (e != cudaSuccess) return cuda_fail(e, "launching the bf16 kernel");
    return FA_OK;
}

// ---------------------------------------------------------------------------
// fa_fwd_host: the bf16 forward on host buffers, with the copies overlapped.
//
// The heads (b, h) are processed in chunks of `heads_per_chunk` through two
// slots of a caller-provided device workspace. Two library-owned streams per
// device carry the copies: chunk c's Q, K, V go host -> device on the first
// while the kernel runs chunk c - 1 on the caller's stream and chunk c - 2's
// O and LSE go device -> host on the second. Events order a slot's reuse:
// its inputs are overwritten only after the kernel that read them, its
// outputs only after they were copied out. The call is asynchronous on the
// caller's stream: the auxiliary streams first wait for an event recorded
// on it, and it finally waits for the last copy.
// ---------------------------------------------------------------------------
namespace {

constexpr int kHostSlots = 2;

struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_ready[kHostSlots] = {}, comp_done[kHostSlots] = {}, out_done[kHostSlots] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

struct SlotLayout {
    int64_t q, k, v, o, lse, bytes;   // offsets within a slot, slot size
};

SlotLayout slot_layout(int64_t hc, int64_t M, int64_t N, int64_t D) {
    SlotLayout L;
    L.q = 0;
    L.k = L.q + align256(hc * M * D * 2);
    L.v = L.k + align256(hc * N * D * 2);
    L.o = L.v + align256(hc * N * D * 2);
    L.lse = L.o + align256(hc * M * D * 2);
    L.bytes = L.lse + align256(hc * M * 4);
    return L;
}

// Heads per chunk when the caller leaves it to the library: up to eight
// chunks, but none with less than ~32 MB of inputs (smaller chunks cost more
// in per-chunk launches and copy latency than their overlap saves).
int64_t default_chunk(int64_t bh, int64_t M, int64_t N, int64_t D) {
    const int64_t in_bytes = bh * (M + 2 * N) * D * 2;
    int64_t chunks = (in_bytes + (32ll << 20) - 1) / (32ll << 20);
    chunks = chunks < 1 ? 1 : (chunks > 8 ? 8 : chunks);
    if (chunks > bh) chunks = bh;
    return (bh + chunks - 1) / chunks;
}

fa_status pipe_setup(int dev, HostPipe** out) {
    HostPipe& P = g_pipe[dev];
    if (!P.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&P.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&P.out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&P.start, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&P.end, cudaEventDisableTiming);
        for (int s = 0; s < kHostSlots && e == cudaSuccess; ++s) {
            e = cudaEventCreateWithFlags(&P.in_ready[s], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&P.comp_done[s], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&P.out_done[s], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return cuda_fail(e, "creating the copy streams and events");
        P.ready = true;
    }
    *out = &P;
    return FA_OK;
}

}  // namespace

FA_API int64_t fa_fwd_host_workspace_bytes(int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                                           int64_t heads_per_chunk) {
    if (B < 0 || H < 0 || M < 0 || N < 0 || D < 1 || heads_per_chunk < 0) return -1;
    const int64_t bh = B * H;
    if (bh == 0 || M == 0) return 0;
    int64_t hc = heads_per_chunk == 0 ? default_chunk(bh, M, N, D) : heads_per_chunk;
    if (hc > bh) hc = bh;
    return kHostSlots * slot_layout(hc, M, N, D).bytes;
}

FA_API fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                             int64_t H, int64_t M, int64_t N, int64_t D, float scale, int causal,
                             int64_t heads_per_chunk, void* workspace, int64_t workspace_bytes, void* stream) {
    bool empty = false;
    fa_status st = validate(q, k, v, o, lse, B, H, M, N, D, scale, 2, &empty);
    if (st != FA_OK) return st;
    if (D != 64 && D != 96 && D != 128)
        return fail(FA_ERR_UNSUPPORTED, "bf16 fa_fwd_host supports D in {64, 96, 128} (got %lld)", (long long)D);
    if (heads_per_chunk < 0) return fail(FA_ERR_INVALID_ARG, "heads_per_chunk must be >= 0");
    if (empty) return FA_OK;
    const int64_t bh = B * H;
    int64_t hc = heads_per_chunk == 0 ? default_chunk(bh, M, N, D) : heads_per_chunk;
    if (hc > bh) hc = bh;
    const SlotLayout L = slot_layout(hc, M, N, D);
    if (workspace == nullptr || workspace_bytes < kHostSlots * L.bytes)
        return fail(FA_ERR_INVALID_ARG, "workspace of %lld bytes needed (got %lld)",
                    (long long)(kHostSlots * L.bytes), (long long)workspace_bytes);
    if (!aligned(workspace, 256)) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    // Whole calls are enqueued one at a time, so that each call's waits
    // refer to its own event records.
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe* P = nullptr;
    if ((st = pipe_setup(dev, &P)) != FA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto check = [&](cudaError_t err, const char* what) -> bool {
        if (err != cudaSuccess) {
            cuda_fail(err, what);
            return false;
        }
        return true;
    };
    if (!check(cudaEventRecord(P->start, s), "cudaEventRecord") ||
        !check(cudaStreamWaitEvent(P->in, P->start, 0), "cudaStreamWaitEvent") ||
        !check(cudaStreamWaitEvent(P->out, P->start, 0), "cudaStreamWaitEvent"))
        return FA_ERR_CUDA;
    const uint8_t* hq = static_cast<const uint8_t*>(q);
    const uint8_t* hk = static_cast<const uint8_t*>(k);
    const uint8_t* hv = static_cast<const uint8_t*>(v);
    uint8_t* ho = static_cast<uint8_t*>(o);
    uint8_t* hl = reinterpret_cast<uint8_t*>(lse);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int64_t qrow = M * D * 2, krow = N * D * 2, lrow = M * 4;   // bytes per head
    int64_t chunk = 0;
    for (int64_t h0 = 0; h0 < bh; h0 += hc, ++chunk) {
        const int64_t n = (bh - h0 < hc) ? bh - h0 : hc;
        const int slot = static_cast<int>(chunk % kHostSlots);
        uint8_t* base = ws + slot * L.bytes;
        // inputs: the slot's previous kernel must have read them
        if (chunk >= kHostSlots && !check(cudaStreamWaitEvent(P->in, P->comp_done[slot], 0), "cudaStreamWaitEvent"))
            return FA_ERR_CUDA;
        if (!check(cudaMemcpyAsync(base + L.q, hq + h0 * qrow, n * qrow, cudaMemcpyHostToDevice, P->in), "copying q") ||
            (N > 0 && !check(cudaMemcpyAsync(base + L.k, hk + h0 * krow, n * krow, cudaMemcpyHostToDevice, P->in),
                             "copying k")) ||
            (N > 0 && !check(cudaMemcpyAsync(base + L.v, hv + h0 * krow, n * krow, cudaMemcpyHostToDevice, P->in),
                             "copying v")) ||
            !check(cudaEventRecord(P->in_ready[slot], P->in), "cudaEventRecord"))
            return FA_ERR_CUDA;
        // kernel: inputs landed, and the slot's previous outputs were copied out
        if (!check(cudaStreamWaitEvent(s, P->in_ready[slot], 0), "cudaStreamWaitEvent") ||
            (chunk >= kHostSlots && !check(cudaStreamWaitEvent(s, P->out_done[slot], 0), "cudaStreamWaitEvent")))
            return FA_ERR_CUDA;
        st = launch_fwd_checked(base + L.q, base + L.k, base + L.v, base + L.o,
                                reinterpret_cast<float*>(base + L.lse), n, M, N, D, scale, causal, s);
        if (st != FA_OK) return st;
        if (!check(cudaEventRecord(P->comp_done[slot], s), "cudaEventRecord") ||
            !check(cudaStreamWaitEvent(P->out, P->comp_done[slot], 0), "cudaStreamWaitEvent") ||
            !check(cudaMemcpyAsync(ho + h0 * qrow, base + L.o, n * qrow, cudaMemcpyDeviceToHost, P->out), "copying o") ||
            !check(cudaMemcpyAsync(hl + h0 * lrow, base + L.lse, n * lrow, cudaMemcpyDeviceToHost, P->out),
                   "copying lse") ||
            !check(cudaEventRecord(P->out_done[slot], P->out), "cudaEventRecord"))
            return FA_ERR_CUDA;
    }
    if (!check(cudaEventRecord(P->end, P->out), "cudaEventRecord") ||
        !check(cudaStreamWaitEvent(s, P->end, 0), "cudaStreamWaitEvent"))
        return FA_ERR_CUDA;
    return FA_OK;
}

// ---------------------------------------------------------------------------
// Self-test of the failure path: a kernel waits, with the attention kernels'
// bounded wait, on a barrier phase that nothing completes. The wait must give
// up after `limit_ns`, OR FA timeout into the status word and return, leaving
// the context usable; fa_get_device_status() then reports FA_ERR_TIMEOUT.
// ---------------------------------------------------------------------------
namespace {

__global__ void selftest_wait_kernel(uint32_t* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        fa::mbar_init(fa::smem_u32(&bar), 1);
        fa::fence_barrier_init();
    }
    __syncthreads();
    // Nothing ever arrives on `bar`.
    if (threadIdx.x == 0) (void)fa::mbar_wait(fa::smem_u32(&bar), 0, &abort_flag, err, limit_ns);
}

}  // namespace

FA_API fa_status fa_selftest_wait_timeout(int64_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000)
        return fail(FA_ERR_INVALID_ARG, "limit_us must be in [1, 1000000] (got %lld)", (long long)limit_us);
    uint32_t* word = nullptr;
    fa_status st = device_setup(false, &word);
    if (st != FA_OK) return st;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(word,
                                                                        static_cast<uint64_t>(limit_us) * 1000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launching the wait self-test");
    return FA_OK;
}

// ---------------------------------------------------------------------------
// fa_bwd: gradients of the bf16 forward (see fa_bwd.cu).
// ---------------------------------------------------------------------------
FA_API int64_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t M) {
    if (B < 0 || H < 0 || M < 0) return -1;
    const int64_t mpad = (M + 127) / 128 * 128;   // Dl and the base-2 LSE, padded to 128-row tiles
    return 2 * B * H * mpad * static_cast<int64_t>(sizeof(float));
}

FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, float* dq, float* dk, float* dv, int64_t B, int64_t H, int64_t M,
                        int64_t N, int64_t D, float scale, int causal, void* workspace, int64_t workspace_bytes,
                        void* stream) {
    bool empty = false;
    // q, k, v and the forward's o / lse pass the forward's checks.
    fa_status st = validate(q, k, v, o, lse, B, H, M, N, D, scale, 2, &empty);
    if (st != FA_OK) return st;
    if (D > 128) return fail(FA_ERR_UNSUPPORTED, "fa_bwd supports D <= 128 (got %lld)", (long long)D);
    const int64_t bh = B * H;
    const int64_t need = fa_bwd_workspace_bytes(B, H, M);
    if (bh == 0 || (M == 0 && N == 0)) return FA_OK;
    if ((M > 0 && (dout == nullptr || dq == nullptr)) || (N > 0 && (dk == nullptr || dv == nullptr)))
        return fail(FA_ERR_INVALID_ARG, "dout, dq, dk and dv must not be null for non-empty tensors");
    if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
        return fail(FA_ERR_INVALID_ARG, "dout, dq, dk and dv must be 16-byte aligned");
    if (M > 0 && (workspace == nullptr || workspace_bytes < need))
        return fail(FA_ERR_INVALID_ARG, "workspace of %lld bytes needed (got %lld)", (long long)need,
                    (long long)workspace_bytes);
    if (M > 0 && !aligned(workspace, 16)) return fail(FA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    const int64_t qb = bh * M * D * 4, kb = bh * N * D * 4;
    if (overlaps(dq, qb, dk, kb) || overlaps(dq, qb, dv, kb) || overlaps(dk, kb, dv, kb) ||
        overlaps(dq, qb, q, bh * M * D * 2) || overlaps(dk, kb, k, bh * N * D * 2) || overlaps(dv, kb, v, bh * N * D * 2) ||
        overlaps(workspace, need, dq, qb) || overlaps(workspace, need, dk, kb) || overlaps(workspace, need, dv, kb))
        return fail(FA_ERR_INVALID_ARG, "the gradients and the workspace must not overlap each other or the inputs");
    // D in {64, 96, 128}: the tensor-core kernels (TMA maps); other D: the
    // CUDA-core kernels.
    const bool tc = (D == 64 || D == 96 || D == 128);
    uint32_t* word = nullptr;
    if ((st = device_setup(tc, &word)) != FA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (M == 0) {   // no query rows: every key gets zero gradient
        e = cudaMemsetAsync(dk, 0, kb, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kb, s);
        return e == cudaSuccess ? FA_OK : cuda_fail(e, "clearing dk and dv");
    }
    fa::BwdParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.o = static_cast<const __nv_bfloat16*>(o);
    p.dout = static_cast<const __nv_bfloat16*>(dout);
    p.lse = lse;
    p.Mpad = static_cast<int>((M + 127) / 128 * 128);
    p.delta = static_cast<float*>(workspace);
    p.lse2 = p.delta + bh * p.Mpad;
    p.err = word;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.bh_count = static_cast<int>(bh);
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.D = static_cast<int>(D);
    p.scale = scale;
    p.causal = causal != 0;
    p.sched = nullptr;
    e = fa::launch_bwd_rowdot(p, s);
    if (e == cudaSuccess && !tc) e = fa::launch_bwd(p, s);
    if (e == cudaSuccess && tc) {
        CUtensorMap mq, mk, mv, mdo;
        if ((st = encode_map(&mq, q, M, bh, D)) != FA_OK || (st = encode_map(&mdo, dout, M, bh, D)) != FA_OK) return st;
        if (N > 0) {
            if ((st = encode_map(&mk, k, N, bh, D)) != FA_OK || (st = encode_map(&mv, v, N, bh, D)) != FA_OK) return st;
        } else {
            mk = mq;  // never read: no key tiles exist
            mv = mq;
        }
        // The persistent dK/dV kernel claims its units from a work-counter
        // pair, used as for the forward (the dQ kernel after it uses none).
        if (e == cudaSuccess)
            return with_sched_slot(s, [&](int* sched) -> fa_status {
                p.sched = sched;
                const cudaError_t e2 = fa::launch_bwd_tc(mq, mk, mv, mdo, p, s);
                return e2 == cudaSuccess ? FA_OK : cuda_fail(e2, "launching the backward kernels");
            });
    }
    if (e != cudaSuccess) return cuda_fail(e, "launching the backward kernels");
    return FA_OK;
}
