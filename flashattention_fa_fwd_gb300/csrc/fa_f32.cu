// fp32 attention forward on the CUDA cores, exact fp32 arithmetic.
//
// The single-head fp32 problem of "FlashAttention in Triton: A Tile-by-Tile
// Walkthrough" (its kernel computes both dots in IEEE fp32 and streams key
// tiles through a running max, sum and accumulator), generalised to a
// [B, H] batch and the top-left causal mask, with the streaming softmax of
// "FlashAttention-style kernel" (section "The loop": exp2 with log2(e) folded
// into the scale) over 32-key tiles of K and V staged in shared memory.
// Products are plain fp32 fused multiply-adds (no TF32), dot products over D
// in order; the final division is IEEE. Three kernels:
//   fa_fwd_f32_rows:  one thread per query row (many rows);
//   fa_fwd_f32_warps: one warp per query row (few rows): the lanes take one
//                     key each for the score, the warp updates the running
//                     max and sum, then the lanes split D for acc += p V.
//   fa_fwd_f32_split: the warp-per-row loop with the keys cut across the
//                     CTAs of a cluster (very few rows), partial results
//                     merged through distributed shared memory.
//
// Compiled without fast-math: exp2f and log2f are the full-accuracy CUDA
// functions.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kRows = 64;    // query rows (threads) per block of the thread-per-row kernel
constexpr int kKeys = 32;    // keys per shared-memory tile

// Thread per row, for problems with enough rows to fill the GPU.

template <int DMAX>
__global__ void __launch_bounds__(kRows)
fa_fwd_f32_rows(const F32Params p, bool causal) {
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
cudaError_t launch_rows_t(const F32Params& p, bool causal, cudaStream_t s) {
    const int smem = 2 * kKeys * DMAX * static_cast<int>(sizeof(float));
    auto kern = fa_fwd_f32_rows<DMAX>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    const long long blocks = static_cast<long long>((p.M + kRows - 1) / kRows) * p.bh_count;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(blocks), kRows, smem, s>>>(p, causal);
    return cudaGetLastError();
}

constexpr int kWarps = 4;    // query rows (warps) per block of the warp-per-row kernel

// Warp per row, for problems with too few rows to fill the GPU one thread per
// row. K/V tiles are double-buffered: the next tile's loads are in flight
// (in registers) while the current one is used.
template <int DMAX>
__global__ void __launch_bounds__(kWarps * 32)
fa_fwd_f32_warps(const F32Params p, bool causal) {
    constexpr int LD = DMAX + 4;       // padded row: distinct rows hit distinct banks
    constexpr int PER = kKeys * DMAX / (kWarps * 32);   // tile elements per thread
    extern __shared__ float sm[];
    float* sK = sm;                    // [2][kKeys][LD]
    float* sV = sK + 2 * kKeys * LD;   // [2][kKeys][LD]
    float* sQ = sV + 2 * kKeys * LD;   // [kWarps][DMAX]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_blocks = (p.M + kWarps - 1) / kWarps;
    const int bh = blockIdx.x / row_blocks;
    const int row0 = (blockIdx.x - bh * row_blocks) * kWarps;
    const int row = row0 + warp;
    const bool valid = row < p.M;
    const int D = p.D;
    const float* qh = p.q + static_cast<size_t>(bh) * p.M * D;
    const float* kh = p.k + static_cast<size_t>(bh) * p.N * D;
    const float* vh = p.v + static_cast<size_t>(bh) * p.N * D;

    float* q = sQ + warp * DMAX;
    for (int d = lane; d < DMAX; d += 32) q[d] = (valid && d < D) ? qh[static_cast<size_t>(row) * D + d] : 0.f;
    constexpr int DL = DMAX / 32;      // output columns per lane: lane + 32 i
    float acc[DL];
#pragma unroll
    for (int i = 0; i < DL; ++i) acc[i] = 0.f;
    const float c = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;

    // Keys any row of this block can see.
    int n_keys = p.N;
    if (causal) n_keys = min(n_keys, min(row0 + kWarps, p.M));

    // Tile loads: element e = threadIdx.x + 128 i of the tile (row e / DMAX,
    // column e % DMAX), coalesced along the rows.
    float rk[PER], rv[PER];
    auto load = [&](int k0) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = threadIdx.x + i * kWarps * 32, kr = e / DMAX, d = e % DMAX;
            const bool in = (k0 + kr < p.N) && d < D;
            rk[i] = in ? kh[static_cast<size_t>(k0 + kr) * D + d] : 0.f;
            rv[i] = in ? vh[static_cast<size_t>(k0 + kr) * D + d] : 0.f;
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = threadIdx.x + i * kWarps * 32, kr = e / DMAX, d = e % DMAX;
            sK[(buf * kKeys + kr) * LD + d] = rk[i];
            sV[(buf * kKeys + kr) * LD + d] = rv[i];
        }
    };
    if (n_keys > 0) {
        load(0);
        store(0);
    }
    __syncthreads();
    for (int k0 = 0, buf = 0; k0 < n_keys; k0 += kKeys, buf ^= 1) {
        const bool more = k0 + kKeys < n_keys;
        if (more) load(k0 + kKeys);    // in flight while this tile is used
        const float* tk = sK + buf * kKeys * LD;
        const float* tv = sV + buf * kKeys * LD;

        // Score of key k0 + lane: q . k over d in order.
        const float4* q4 = reinterpret_cast<const float4*>(q);
        const float4* k4 = reinterpret_cast<const float4*>(tk + lane * LD);
        float dot = 0.f;
#pragma unroll
        for (int d4 = 0; d4 < DMAX / 4; ++d4) {
            const float4 a = q4[d4], b = k4[d4];
            dot = fmaf(a.x, b.x, dot);
            dot = fmaf(a.y, b.y, dot);
            dot = fmaf(a.z, b.z, dot);
            dot = fmaf(a.w, b.w, dot);
        }
        const int key = k0 + lane;
        const bool vis = key < p.N && (!causal || key <= row);
        const float s = vis ? dot * c : -INFINITY;
        float mx = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;   // fully masked so far
        const float alpha = exp2f(m_run - m_use);
        const float pl = exp2f(s - m_use);
        float psum = pl;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l_run = l_run * alpha + psum;
        // acc += p V over the tile's keys in order; lane owns columns lane + 32 i.
#pragma unroll
        for (int i = 0; i < DL; ++i) acc[i] *= alpha;
#pragma unroll 8
        for (int j = 0; j < kKeys; ++j) {
            const float pj = __shfl_sync(0xffffffffu, pl, j);
#pragma unroll
            for (int i = 0; i < DL; ++i) acc[i] = fmaf(pj, tv[j * LD + lane + 32 * i], acc[i]);
        }
        m_run = m_new;
        if (more) store(buf ^ 1);      // the other buffer was last read a tile ago
        __syncthreads();
    }

    if (valid) {
        float* orow = p.o + (static_cast<size_t>(bh) * p.M + row) * D;
#pragma unroll
        for (int i = 0; i < DL; ++i) {
            const int d = lane + 32 * i;
            if (d < D) orow[d] = (l_run > 0.f) ? acc[i] / l_run : 0.f;
        }
        if (lane == 0)
            p.lse[static_cast<size_t>(bh) * p.M + row] =
                (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }
}

template <int DMAX>
cudaError_t launch_warps_t(const F32Params& p, bool causal, cudaStream_t s) {
    const int smem = (4 * kKeys * (DMAX + 4) + kWarps * DMAX) * static_cast<int>(sizeof(float));
    auto kern = fa_fwd_f32_warps<DMAX>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    const long long blocks = static_cast<long long>((p.M + kWarps - 1) / kWarps) * p.bh_count;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(blocks), kWarps * 32, smem, s>>>(p, causal);
    return cudaGetLastError();
}

constexpr int kSplitRows = 8;   // query rows (warps) per CTA of the key-split kernel
constexpr int kMaxSplits = 8;   // CTAs per cluster: the portable cluster size

// Warp per row with the keys cut across the CTAs of a thread-block cluster,
// for problems whose rows alone cannot fill the GPU. CTA `split` of a
// cluster runs the warp-per-row loop above over key tiles
// [split * tiles_per_split, (split + 1) * tiles_per_split) for the cluster's
// kSplitRows rows and leaves its (acc, m, l) per row in shared memory; the
// cluster then merges them through distributed shared memory with the
// softmax-of-a-concatenation rule of "Module 08: FlashAttention and
// Memory-Efficient Kernels" (section "Tiling and the online softmax"):
// m = max_s m_s, l = sum_s 2^(m_s - m) l_s, acc = sum_s 2^(m_s - m) acc_s,
// summed over s in order. Every CTA passes the same two cluster barriers.
template <int DMAX>
__global__ void __launch_bounds__(kSplitRows * 32)
fa_fwd_f32_split(const F32Params p, bool causal, int tiles_per_split) {
    namespace cg = cooperative_groups;
    constexpr int NT = kSplitRows * 32;
    constexpr int LD = DMAX + 4;       // padded row: distinct rows hit distinct banks
    constexpr int PER = kKeys * DMAX / NT;   // tile elements per thread
    constexpr int PART = DMAX + 2;     // a row's partial: acc[DMAX], m, l
    extern __shared__ float sm[];
    float* sK = sm;                    // [2][kKeys][LD]
    float* sV = sK + 2 * kKeys * LD;   // [2][kKeys][LD]
    float* sQ = sV + 2 * kKeys * LD;   // [kSplitRows][DMAX]
    float* part = sQ + kSplitRows * DMAX;   // [kSplitRows][PART]

    cg::cluster_group cluster = cg::this_cluster();
    const int split = static_cast<int>(cluster.block_rank());
    const int splits = static_cast<int>(cluster.num_blocks());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_groups = (p.M + kSplitRows - 1) / kSplitRows;
    const int group = blockIdx.x / splits;
    const int bh = group / row_groups;
    const int row0 = (group - bh * row_groups) * kSplitRows;
    const int row = row0 + warp;
    const bool valid = row < p.M;
    const int D = p.D;
    const float* qh = p.q + static_cast<size_t>(bh) * p.M * D;
    const float* kh = p.k + static_cast<size_t>(bh) * p.N * D;
    const float* vh = p.v + static_cast<size_t>(bh) * p.N * D;

    constexpr int DL = DMAX / 32;      // output columns per lane: lane + 32 i
    float acc[DL];
#pragma unroll
    for (int i = 0; i < DL; ++i) acc[i] = 0.f;
    const float c = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;

    // This CTA's keys: its split's tiles, cut at N and, under the causal
    // mask, at the last key any row of the CTA sees. Split boundaries are
    // tile boundaries, so no tile holds another split's keys.
    const int k_lo = split * tiles_per_split * kKeys;
    int k_hi = min(p.N, k_lo + tiles_per_split * kKeys);
    if (causal) k_hi = min(k_hi, min(row0 + kSplitRows, p.M));

    float rk[PER], rv[PER];
    auto load = [&](int k0) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = threadIdx.x + i * NT, kr = e / DMAX, d = e % DMAX;
            const bool in = (k0 + kr < p.N) && d < D;
            rk[i] = in ? kh[static_cast<size_t>(k0 + kr) * D + d] : 0.f;
            rv[i] = in ? vh[static_cast<size_t>(k0 + kr) * D + d] : 0.f;
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = threadIdx.x + i * NT, kr = e / DMAX, d = e % DMAX;
            sK[(buf * kKeys + kr) * LD + d] = rk[i];
            sV[(buf * kKeys + kr) * LD + d] = rv[i];
        }
    };
    // The first tile's loads and the query row's are in flight together.
    if (k_lo < k_hi) load(k_lo);
    float* q = sQ + warp * DMAX;
    for (int d = lane; d < DMAX; d += 32) q[d] = (valid && d < D) ? qh[static_cast<size_t>(row) * D + d] : 0.f;
    if (k_lo < k_hi) store(0);
    __syncthreads();
    for (int k0 = k_lo, buf = 0; k0 < k_hi; k0 += kKeys, buf ^= 1) {
        const bool more = k0 + kKeys < k_hi;
        if (more) load(k0 + kKeys);    // in flight while this tile is used
        const float* tk = sK + buf * kKeys * LD;
        const float* tv = sV + buf * kKeys * LD;

        // Score of key k0 + lane: q . k over d in order.
        const float4* q4 = reinterpret_cast<const float4*>(q);
        const float4* k4 = reinterpret_cast<const float4*>(tk + lane * LD);
        float dot = 0.f;
#pragma unroll
        for (int d4 = 0; d4 < DMAX / 4; ++d4) {
            const float4 a = q4[d4], b = k4[d4];
            dot = fmaf(a.x, b.x, dot);
            dot = fmaf(a.y, b.y, dot);
            dot = fmaf(a.z, b.z, dot);
            dot = fmaf(a.w, b.w, dot);
        }
        const int key = k0 + lane;
        const bool vis = key < p.N && (!causal || key <= row);
        const float s = vis ? dot * c : -INFINITY;
        float mx = s;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;   // fully masked so far
        const float alpha = exp2f(m_run - m_use);
        const float pl = exp2f(s - m_use);
        float psum = pl;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l_run = l_run * alpha + psum;
#pragma unroll
        for (int i = 0; i < DL; ++i) acc[i] *= alpha;
#pragma unroll 8
        for (int j = 0; j < kKeys; ++j) {
            const float pj = __shfl_sync(0xffffffffu, pl, j);
#pragma unroll
            for (int i = 0; i < DL; ++i) acc[i] = fmaf(pj, tv[j * LD + lane + 32 * i], acc[i]);
        }
        m_run = m_new;
        if (more) store(buf ^ 1);      // the other buffer was last read a tile ago
        __syncthreads();
    }

    // This CTA's partial of each of its rows (m = -inf, l = 0, acc = 0 when
    // the split holds none of the row's keys).
    float* mine = part + warp * PART;
#pragma unroll
    for (int i = 0; i < DL; ++i) mine[lane + 32 * i] = acc[i];
    if (lane == 0) {
        mine[DMAX] = m_run;
        mine[DMAX + 1] = l_run;
    }
    cluster.sync();   // every partial written, and visible to the cluster

    // Row `warp` is merged by the cluster's CTA warp % splits. Every remote
    // load is issued before any result is used: lane t fetches split t's m
    // and l, each lane its columns of every split's acc.
    if (valid && warp % splits == split) {
        float mt = -INFINITY, lt = 0.f;
        if (lane < splits) {
            const float* pt = cluster.map_shared_rank(part, lane) + warp * PART;
            mt = pt[DMAX];
            lt = pt[DMAX + 1];
        }
        float pa[kMaxSplits][DL];
#pragma unroll
        for (int t = 0; t < kMaxSplits; ++t) {
            const float* pt = cluster.map_shared_rank(part, t < splits ? t : 0) + warp * PART;
#pragma unroll
            for (int i = 0; i < DL; ++i) pa[t][i] = (t < splits) ? pt[lane + 32 * i] : 0.f;
        }
        float m = mt;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float m_use = (m == -INFINITY) ? 0.f : m;
        const float wt = exp2f(mt - m_use);   // 0 for an empty split and for lanes >= splits
        float l = 0.f, o[DL];
#pragma unroll
        for (int i = 0; i < DL; ++i) o[i] = 0.f;
#pragma unroll
        for (int t = 0; t < kMaxSplits; ++t) {
            const float w = __shfl_sync(0xffffffffu, wt, t);
            if (t < splits) {
                l = fmaf(w, __shfl_sync(0xffffffffu, lt, t), l);
#pragma unroll
                for (int i = 0; i < DL; ++i) o[i] = fmaf(w, pa[t][i], o[i]);
            }
        }
        float* orow = p.o + (static_cast<size_t>(bh) * p.M + row) * D;
#pragma unroll
        for (int i = 0; i < DL; ++i) {
            const int d = lane + 32 * i;
            if (d < D) orow[d] = (l > 0.f) ? o[i] / l : 0.f;
        }
        if (lane == 0)
            p.lse[static_cast<size_t>(bh) * p.M + row] =
                (l > 0.f) ? (m_use + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
    cluster.sync();   // no CTA leaves while another still reads its partials
}

// The current device's ordinal and SM count (0 SMs if they cannot be read).
int device_sms(int* dev_out) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    *dev_out = dev;
    return n;
}

// Whether a cluster of `splits` CTAs of the key-split kernel can be resident
// on the device at all (a partitioned GPU may offer fewer SMs per cluster);
// asked once per device, head-dimension class and cluster size. When it
// cannot, the warp-per-row kernel runs instead.
constexpr int kMaxDev = 64;
std::atomic<int> g_cluster_ok[kMaxDev][3][4];   // 0 unknown, 1 yes, -1 no

// Launches the key-split kernel; sets *launched to false, launching nothing,
// when its clusters cannot be scheduled on this device.
template <int DMAX>
cudaError_t launch_split_t(const F32Params& p, bool causal, int splits, int tiles_per_split, cudaStream_t s,
                           int dev, bool* launched) {
    *launched = false;
    const int smem = (4 * kKeys * (DMAX + 4) + kSplitRows * DMAX + kSplitRows * (DMAX + 2)) * static_cast<int>(sizeof(float));
    auto kern = fa_fwd_f32_split<DMAX>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    const long long groups = static_cast<long long>((p.M + kSplitRows - 1) / kSplitRows) * p.bh_count;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(groups * splits));
    cfg.blockDim = dim3(kSplitRows * 32);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int di = DMAX == 32 ? 0 : (DMAX == 64 ? 1 : 2), si = splits == 2 ? 0 : (splits == 4 ? 1 : 2);
    std::atomic<int>* ok = (dev >= 0 && dev < kMaxDev) ? &g_cluster_ok[dev][di][si] : nullptr;
    int known = ok ? ok->load(std::memory_order_relaxed) : 0;
    if (known == 0) {
        int clusters = 0;
        const cudaError_t oe = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (oe != cudaSuccess) (void)cudaGetLastError();   // not a launch: nothing to report
        known = (oe == cudaSuccess && clusters > 0) ? 1 : -1;
        if (ok) ok->store(known, std::memory_order_relaxed);
    }
    if (known < 0) return cudaSuccess;
    *launched = true;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p, causal, tiles_per_split);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// The key-split cluster count for a problem: doubled (up to the portable
// cluster size) while the CTAs stay under two per SM and every split keeps
// at least one 32-key tile; 1 means no split.
int f32_key_splits(long long bh_count, long long M, long long N, int sms) {
    const long long groups = (M + kSplitRows - 1) / kSplitRows * bh_count;
    const long long tiles = (N + kKeys - 1) / kKeys;
    int splits = 1;
    while (splits < kMaxSplits && groups * splits < 2LL * sms && 2 * splits <= tiles) splits *= 2;
    return splits;
}

// Thread per row once there are enough rows for four blocks on every SM;
// below that warp per row, where the thread-per-row kernel would leave most
// SMs idle and wait on its long dependent dot products; and with the keys
// also cut across a cluster when the rows' warps alone fill less than two
// CTAs per SM.
cudaError_t launch_f32(const F32Params& p, bool causal, cudaStream_t s) {
    int dev = -1;
    int sms = device_sms(&dev);
    if (sms <= 0) sms = 152;
    const bool many = static_cast<long long>(p.bh_count) * p.M >= static_cast<long long>(sms) * 4 * kRows;
    const int splits = many ? 1 : f32_key_splits(p.bh_count, p.M, p.N, sms);
    if (splits > 1) {
        const int tiles = (p.N + kKeys - 1) / kKeys;
        const int per = (tiles + splits - 1) / splits;
        bool launched = false;
        cudaError_t e;
        if (p.D <= 32) e = launch_split_t<32>(p, causal, splits, per, s, dev, &launched);
        else if (p.D <= 64) e = launch_split_t<64>(p, causal, splits, per, s, dev, &launched);
        else e = launch_split_t<128>(p, causal, splits, per, s, dev, &launched);
        if (e != cudaSuccess || launched) return e;
    }
    if (p.D <= 32) return many ? launch_rows_t<32>(p, causal, s) : launch_warps_t<32>(p, causal, s);
    if (p.D <= 64) return many ? launch_rows_t<64>(p, causal, s) : launch_warps_t<64>(p, causal, s);
    return many ? launch_rows_t<128>(p, causal, s) : launch_warps_t<128>(p, causal, s);
}

}  // namespace fa
