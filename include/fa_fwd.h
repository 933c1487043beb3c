/*
 * fa_fwd.h -- C ABI of libfa_fwd.so, the FlashAttention forward pass for one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The operation (what every entry point below computes)
 * -----------------------------------------------------
 * For every batch b < B and head h < H, with Q_bh an M x D matrix and K_bh,
 * V_bh N x D matrices:
 *
 *     S   = scale * Q_bh K_bh^T                          (M x N, never stored)
 *     S[i][j] = -inf where causal and j > i              (top-left causal mask)
 *     O_bh[i]  = sum_j softmax_j(S[i]) * V_bh[j]          (M x D)
 *     LSE_bh[i] = max_j S[i][j] + ln sum_j exp(S[i][j] - max_j S[i][j])
 *
 * Sources: attention as S = QK^T/sqrt(d), P = softmax(S), O = PV and the
 * per-row log-sum-exp L = m + log(l) kept for the backward pass are from
 * "Module 08: FlashAttention and Memory-Efficient Kernels" (sections "Where
 * the time goes in standard attention" and "The backward pass: recompute
 * instead of store"); the M-row query / N-row key problem statement and the
 * caller-preallocated output are from "FlashAttention in Triton: A
 * Tile-by-Tile Walkthrough" (sections "First, what does attention actually
 * do?" and "Full Triton implementation"); the (batch, heads, sequence,
 * head_dim) layout is the one of "Module 08" Code Step 7; the causal mask
 * keeps key j for query i when j <= i as in "Module 08" Code Step 1. The
 * pages show only square causal masks; for M != N this library keeps the
 * same top-left rule (j <= i).
 *
 * A row with no visible key (only possible when N == 0) gets O = 0 and
 * LSE = -inf. LSE is in natural-log units of the scaled scores.
 *
 * Layout and ownership (all entry points)
 * ---------------------------------------
 *   q   : [B, H, M, D] contiguous, device memory
 *   k,v : [B, H, N, D] contiguous, device memory
 *   o   : [B, H, M, D] contiguous, device memory, written
 *   lse : [B, H, M]    contiguous fp32, device memory, written
 * The caller allocates and owns every buffer; o and lse must not overlap
 * the inputs or each other. `stream` is a cudaStream_t (NULL = the legacy
 * default stream). Calls are asynchronous on `stream` and never
 * synchronise; the results are ready when the stream reaches them.
 *
 * The library allocates nothing per call. On its first call on a device it
 * allocates one small block of device state for that device (1032 bytes),
 * which it keeps until the process exits: a status word, into which
 * device-side failures (a pipeline wait that ran out of time) are OR-ed and
 * which fa_get_device_status() reads, and 128 pairs of work counters that
 * the persistent kernels' CTAs use to claim work units. Each bf16 forward
 * launch (fa_fwd, fa_fwd_splitkv, fa_fwd_host) and each tensor-core fa_bwd
 * call takes the next of 64 pairs in turn and leaves it at zero when it ends; before reusing a pair, the launch's stream waits
 * for an event recorded after the pair's previous launch, so any number of
 * launches may be in flight on any streams and host threads without two
 * running launches sharing a pair (the 65th queues behind the first). A
 * launch captured into a CUDA graph takes the next of the other 64 pairs
 * and keeps it for every replay of the graph: replays of graphs that hold
 * the same pair must not overlap (captures 1 and 65 on a device share one).
 *
 * Errors
 * ------
 * Arguments are checked on the host before anything is launched; a failed
 * check launches nothing and returns:
 *   FA_ERR_INVALID_ARG  a null pointer (unless the tensor it names is
 *                       empty), B, H or M < 0, N < 0, D < 1, a scale that is
 *                       not finite and > 0, a pointer that is not 16-byte
 *                       aligned, or sizes whose byte counts overflow.
 *   FA_ERR_UNSUPPORTED  a head dimension the entry point has no kernel for,
 *                       or a current device that is not sm_103.
 *   FA_ERR_CUDA         a CUDA runtime or driver call failed (details in
 *                       fa_last_error()).
 * B, H or M equal to 0 is a legal empty problem: nothing is launched and
 * FA_OK is returned.
 */
#ifndef FA_FWD_H_
#define FA_FWD_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,
    FA_ERR_UNSUPPORTED = 2,
    FA_ERR_CUDA = 3,
    FA_ERR_TIMEOUT = 4
} fa_status;

/*
 * bf16 attention forward on the tensor cores (tcgen05, accumulators in
 * tensor memory). q, k, v and o hold bf16 values; lse is fp32. Scores,
 * the running max and sum and the output accumulator are fp32; the
 * probabilities are rounded to bf16 before they multiply V (the pages'
 * tutorial loop casts p to 16 bits for that product: "FlashAttention-style
 * kernel", section "The loop").
 *
 * D must be 64, 96 or 128 (FA_ERR_UNSUPPORTED otherwise). The algorithm is
 * the streaming softmax of "FlashAttention-style kernel" ("The loop", with
 * its base-two exponent and log2(e) folded into the scale) with the
 * FlashAttention-2 work split of "Module 08" (section "Related ideas"):
 * each 128-row query tile stays on chip while 128-row key/value tiles
 * stream past it, and causal key tiles that lie wholly above the diagonal
 * are skipped ("FlashAttention-style kernel", section "Causal masking").
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                 float scale, int causal, void* stream);

/*
 * fp32 attention forward on the CUDA cores with exact fp32 fused
 * multiply-adds (no TF32): the single-head fp32 problem of "FlashAttention
 * in Triton: A Tile-by-Tile Walkthrough" (its kernel computes its dots in
 * IEEE fp32), generalised to [B, H] and the causal mask. All buffers fp32.
 * D must be in [1, 128]. Problems with few rows also cut the keys across
 * the CTAs of a thread-block cluster and merge the partial results with the
 * softmax-of-a-concatenation rule of "Module 08: FlashAttention and
 * Memory-Efficient Kernels" (section "Tiling and the online softmax"), in a
 * fixed order: results are deterministic. One kernel launch, no workspace.
 */
fa_status fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                     int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                     float scale, int causal, void* stream);

/*
 * fp32 attention forward on the tensor cores: the result of fa_fwd_f32 (same
 * arguments, layouts and semantics) with both matrix products on tcgen05 as
 * three TF32 products. Every fp32 input x is split as x = hi + lo, hi = x
 * rounded to 11 significant bits, lo = x - hi, and a product A B is taken as
 * A_lo B_hi + A_hi B_lo + A_hi B_hi in fp32: near-fp32 accuracy (the dropped
 * A_lo B_lo term is ~2^-22 of the product) where fa_fwd_f32's exact FMAs are
 * CUDA-core bound. This is the fast fp32 path that "FlashAttention in
 * Triton: A Tile-by-Tile Walkthrough" lacks: its IEEE-fp32 kernel ends up
 * slower than the library attention it is compared with.
 *
 *   q, k, v, o, lse  as fa_fwd_f32 (fp32, contiguous, 16-byte aligned; lse 4)
 *   D                32, 64, 96 or 128 (others: FA_ERR_UNSUPPORTED)
 *   workspace        device memory owned by the caller, 128-byte aligned, at
 *                    least fa_fwd_f32x3_workspace_bytes(B, H, N, D) bytes;
 *                    receives K and V split into hi/lo tile images (it may
 *                    be null when that size is 0, i.e. N = 0)
 *
 * Inputs must be finite and below 2^127 in magnitude. Asynchronous on
 * `stream`: two kernels (the split, then the attention), never
 * synchronises. Errors: fa_fwd_f32's checks, plus FA_ERR_INVALID_ARG for a
 * missing, short or misaligned workspace or one that overlaps a tensor;
 * device wait timeouts surface through fa_get_device_status.
 */
fa_status fa_fwd_f32x3(const float* q, const float* k, const float* v, float* o, float* lse,
                       int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                       float scale, int causal, void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes fa_fwd_f32x3 needs: 16 bytes per (head, key, column) with
 * the keys padded to the kernel's key block, 64 for D >= 96 and 32 below
 * (-1 for negative sizes). Needs no GPU. */
int64_t fa_fwd_f32x3_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D);

/*
 * Split-KV bf16 forward: the same result as fa_fwd (same arguments, layouts
 * and checks), computed by cutting each query tile's keys into `num_splits`
 * contiguous ranges that different CTAs process in parallel, then merging
 * the partial results with the softmax-of-a-concatenation algebra of
 * "Module 08: FlashAttention and Memory-Efficient Kernels" (section "Tiling
 * and the online softmax"): LSE = ln sum_s exp(LSE_s), O = sum_s
 * exp(LSE_s - LSE) O_s. Useful when B*H*ceil(M/256) is below the SM count
 * (few query tiles, long keys; "FlashAttention in Triton: A Tile-by-Tile
 * Walkthrough", section "What the H100 run showed", on exposing more
 * parallel work).
 *
 *   num_splits       1..16; 1 is exactly fa_fwd (the workspace is unused)
 *   workspace        device memory owned by the caller, 16-byte aligned,
 *                    at least fa_fwd_splitkv_workspace_bytes(...) bytes, not
 *                    overlapping the tensors; it holds fp32 partial outputs
 *                    and log-sum-exps and is overwritten by every call
 *
 * Launches two kernels on `stream` (the split kernel, then the merge).
 * Errors as fa_fwd, plus FA_ERR_INVALID_ARG for num_splits outside [1, 16]
 * or a missing, short, misaligned or overlapping workspace.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                         float scale, int causal, int num_splits,
                         void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes fa_fwd_splitkv needs: num_splits * B*H*M * (D + 1) * 4
 * (0 when num_splits == 1; -1 for invalid arguments). Needs no GPU. */
int64_t fa_fwd_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t M, int64_t D, int num_splits);

/* A split count that fills the current device's SMs once with
 * B*H*ceil(M/256)*splits units, keeping at least two 128-key tiles per
 * split; 1 for causal problems or when no split helps. */
int fa_fwd_splitkv_suggest(int64_t B, int64_t H, int64_t M, int64_t N, int causal);

/*
 * bf16 forward on HOST buffers: the result of fa_fwd (same layouts, checks
 * and results) for q, k, v, o and lse in host memory, with the host <-> device
 * copies overlapped with the computation. It is how the library is used when
 * the tensors live on the host; the pages' statement of the problem ("FlashAttention
 * in Triton: A Tile-by-Tile Walkthrough", section "Full Triton implementation":
 * `solve` writes a preallocated output) does not say where they live.
 *
 * The B*H heads are processed in chunks of `heads_per_chunk` (0 = the
 * library's choice: up to eight chunks, none with less than ~32 MB of
 * q, k, v) through two slots of a
 * caller-owned device workspace: while the kernel runs one chunk on
 * `stream`, the next chunk's q, k, v are copied in and the previous chunk's
 * o, lse copied out on two streams the library creates once per device.
 *
 *   q, k, v, o, lse  host memory, 16-byte aligned (lse 4); page-locked
 *                    (cudaHostAlloc / pinned) for the copies to overlap --
 *                    pageable memory works, with the driver's synchronous
 *                    staging
 *   heads_per_chunk  >= 0
 *   workspace        device memory owned by the caller, 256-byte aligned, at
 *                    least fa_fwd_host_workspace_bytes(...) bytes
 *
 * Asynchronous on `stream`: the host buffers must stay valid and unchanged,
 * and o and lse are only complete, once the stream reaches the point of the
 * call (e.g. after cudaStreamSynchronize(stream)). Calls that may run at the
 * same time on different streams need different workspaces. Errors as
 * fa_fwd, plus FA_ERR_INVALID_ARG for a negative heads_per_chunk or a
 * missing, short or misaligned workspace, and FA_ERR_CUDA if creating the
 * library's streams or events, or enqueueing a copy, fails.
 */
fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                      int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                      float scale, int causal, int64_t heads_per_chunk,
                      void* workspace, int64_t workspace_bytes, void* stream);

/* Device workspace bytes fa_fwd_host needs: two slots, each holding one
 * chunk's q, k, v, o (bf16) and lse (fp32), every array padded to 256 bytes
 * (0 for an empty problem; -1 for invalid arguments). Needs no GPU. */
int64_t fa_fwd_host_workspace_bytes(int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                                    int64_t heads_per_chunk);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * words (the library's device state and, once fa_fwd_noalloc has run on the
 * device, word 0 of its static array). Returns FA_ERR_TIMEOUT if a kernel
 * launched since the last call gave up on a pipeline wait (its outputs are
 * then undefined), FA_ERR_CUDA if the synchronisation itself failed, FA_OK
 * otherwise.
 */
fa_status fa_get_device_status(void* stream);

/*
 * fa_fwd_noalloc: the bf16 forward of fa_fwd (same arguments, layouts,
 * checks and results) for callers that cannot allocate device memory. The
 * pages have no counterpart to this entry point; it exists for the library's
 * users.
 *
 * Who needs it: fa_fwd cudaMallocs a small block of device state (its status
 * word and work counters) on its first call on each device. Applications whose caching allocator or memory pool owns all
 * device memory, serving loops that must avoid the implicit device-wide
 * synchronisation a cudaMalloc can cause, and processes under a fixed
 * device-memory quota cannot allow that. This entry point calls no
 * cudaMalloc, cudaFree or other allocating routine: the kernel's scratch (its
 * status word and the two counters its CTAs claim work units from) lives in
 * a file-scope static device array of 64 32-bit words (256 bytes), which
 * every GPU that loads the library holds until the process exits. No
 * problem size needs more than those three words; a kernel needing more
 * than the array holds would be rejected with FA_ERR_UNSUPPORTED.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture. Every call clears the two work
 * counters on `stream` before its launch. All calls share the one array, so
 * calls that overlap on the GPU (other streams, other host threads) race on
 * it: they share the work counters, so units of work can be skipped or done
 * twice and O and LSE can be wrong. Keep such calls on one stream, or order
 * them with events. A device-side pipeline timeout in this variant leaves O
 * and LSE undefined and is OR-ed into word 0 of the array, which keeps it
 * until fa_get_device_status() reads and clears it (that call reads both
 * this word and fa_fwd's, with plain copies that allocate nothing).
 */
fa_status fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                         int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                         float scale, int causal, void* stream);

/*
 * Backward pass of fa_fwd: the gradients dQ, dK, dV of a loss whose gradient
 * with respect to O is `dout`. "Module 08: FlashAttention and
 * Memory-Efficient Kernels", section "The backward pass: recompute instead of
 * store" and Code Step 6: nothing N x N is stored by the forward; every tile
 * of P is rebuilt as exp(S - L) from Q, K and the forward's per-row
 * log-sum-exp L (`lse`). With that P: dV = P^T dO, dP = dO V^T,
 * dS = P * (dP - rowsum(dO * O)), dQ = scale dS K, dK = scale dS^T Q.
 * D in {64, 96, 128} runs on the tensor cores (tcgen05, TMA): a persistent
 * kernel whose CTAs take 128-key tiles in turn computes S^T = K Q^T and
 * dP^T = V dO^T, rebuilds P^T and dS^T (bf16) in tensor memory and
 * accumulates dV, dK there (its CTAs claim tiles from one of the work-counter
 * pairs described above); one kernel per 128-row query tile does the same
 * for dQ. Other D run on the CUDA cores in fp32. Both are deterministic (each
 * output written by one CTA, no atomics).
 *
 *   q, k, v          the forward's bf16 inputs, [B,H,M,D] / [B,H,N,D]
 *   o, lse           the forward's outputs for them (bf16 O, fp32 LSE)
 *   dout             bf16 [B,H,M,D]
 *   dq               fp32 [B,H,M,D], written
 *   dk, dv           fp32 [B,H,N,D], written (rows no query sees get 0)
 *   workspace        device memory owned by the caller, 16-byte aligned,
 *                    at least fa_bwd_workspace_bytes(B, H, M) bytes
 *   D                1..128
 *
 * Asynchronous on `stream`, never synchronises. Errors: the forward's
 * checks on q, k, v, o, lse and the sizes, plus FA_ERR_INVALID_ARG for a
 * null or misaligned dout / dq / dk / dv, a missing or short workspace, or
 * gradients that overlap each other, the inputs or the workspace, and
 * FA_ERR_UNSUPPORTED for D > 128.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, float* dq, float* dk, float* dv,
                 int64_t B, int64_t H, int64_t M, int64_t N, int64_t D,
                 float scale, int causal, void* workspace, int64_t workspace_bytes, void* stream);

/* Workspace bytes fa_bwd needs: two fp32 values per (head, query row) with
 * the rows padded to a multiple of 128 (-1 for negative sizes).
 * Needs no GPU. */
int64_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t M);

/*
 * Self-test of the library's failure detection (the pages have no
 * counterpart: it checks this library's own bounded waits). Launches on
 * `stream` one small kernel that waits, with the same bounded barrier wait
 * the attention kernels use, on a barrier phase that nothing completes; after
 * `limit_us` microseconds (1 .. 1000000) the wait gives up, records a timeout
 * in the device status word and the kernel returns normally. A following
 * fa_get_device_status() must return FA_ERR_TIMEOUT (and clear the word), and
 * the CUDA context stays usable. Nothing faults, traps or hangs.
 * Returns FA_ERR_INVALID_ARG for limit_us outside [1, 1000000], otherwise
 * as fa_fwd's launch.
 */
fa_status fa_selftest_wait_timeout(int64_t limit_us, void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(int status);

/* Detail of the last non-OK status returned on the calling thread (static
 * per-thread buffer, valid until the thread's next call into the library). */
const char* fa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_FWD_H_ */
