// bf16 FlashAttention forward for sm_103a: TMA-fed shared-memory tiles,
// tcgen05 MMAs with fp32 accumulators in tensor memory, warp-specialised
// load / MMA / softmax roles.
//
// Algorithm ("FlashAttention-style kernel", section "The loop"; "Module 08:
// FlashAttention and Memory-Efficient Kernels", sections "Tiling and the
// online softmax" and "Related ideas"): a query tile stays resident while
// key/value tiles stream past it; per row the kernel carries the running
// max m, the running sum l and the unnormalised output acc, rescales l and
// acc by alpha = exp2(m_old - m_new) whenever the max grows, and divides by
// l once at the end. log2(e) is folded into the score scale so that each
// score costs one FMA and one base-two exponential. The per-row log-sum-exp
// m + log(l) is written next to O ("Module 08", section "The backward pass").
//
// Work unit: one (batch*head, pair of 128-row query tiles). The two query
// tiles (t = 0, 1) are processed in ping-pong so that the tensor core works
// on one tile's matmuls while the other tile's softmax runs.
//
// Roles (320 threads):
//   warps 0-3  softmax for query tile 0 (thread = one query row = one TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q once, then K_j, V_j into a ring of stages
//   warp  9    tensor-memory owner and MMA issuer
//
// Tensor memory (512 columns, 128 lanes, lane = query row of the tile):
//   [  0,128)  S_0 (fp32 scores of tile 0); P_0 (bf16, packed in pairs)
//              overwrites its first 64 columns after softmax
//   [128,256)  S_1 / P_1
//   [256,256+D) O_0 accumulator      [384,384+D) O_1 accumulator
//
// Per key/value tile j the MMA warp issues, in this order:
//   O_0 += P_0(j-1) V(j-1);  S_0 = Q_0 K(j)^T;  O_1 += P_1(j-1) V(j-1);
//   S_1 = Q_1 K(j)^T
// tcgen05 MMAs from one thread execute in issue order, so S_t(j) only
// overwrites P_t(j-1) after the product that reads it, and the commit that
// announces S_t(j) also guarantees that O_t holds every earlier product
// (which is what lets softmax t rescale O_t before releasing P_t(j)).
//
// Causal (top-left, key j visible to query i when j <= i): key tiles wholly
// above the diagonal are never loaded or multiplied; the diagonal tile and a
// ragged last key tile are masked with -inf in registers ("FlashAttention-
// style kernel", section "Causal masking"). A row whose running max is still
// -inf uses 0 in its place so that exp2(-inf - -inf) never forms ("Module
// 08", "Common mistakes"). Query rows >= M and key rows >= N are zero-filled
// by TMA, and their scores masked or their outputs not stored.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

template <int D>
struct Bf16Cfg {
    static_assert(D == 64 || D == 96 || D == 128, "head dimension");
    static constexpr int BM = 128;                     // query rows per tile
    static constexpr int BN = 128;                     // key rows per tile
    static constexpr int PANELS = (D + 63) / 64;       // 64-column swizzle panels
    static constexpr int PANEL_BYTES = 128 * 128;      // 128 rows x 128 B
    static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;
    static constexpr int NS = (D <= 64) ? 8 : 5;       // K/V ring stages
    static constexpr int NUM_BARS = 2 * NS + 8;
    static constexpr int SMEM_BYTES = 1024 + (2 + NS) * TILE_BYTES + NUM_BARS * 8;
    static constexpr int THREADS = 320;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL0 = 256, O_COL1 = 384;
    static constexpr int QK_STEPS = D / 16;            // MMA K-steps of Q K^T
    static constexpr int PV_STEPS = BN / 16;           // MMA K-steps of P V
};

// Barrier slots in shared memory.
template <int NS>
struct Bars {
    static constexpr int full = 0;            // [NS] K/V stage loaded
    static constexpr int empty = NS;          // [NS] K/V stage released
    static constexpr int q_full = 2 * NS;     // Q tiles loaded
    static constexpr int s_full = 2 * NS + 1; // [2] S_t ready in TMEM
    static constexpr int p_ready = 2 * NS + 3;// [2] P_t stored and O_t rescaled
    static constexpr int o_done = 2 * NS + 5; // [2] last P V of tile t complete
    static constexpr int drain = 2 * NS + 7;  // all MMAs complete (exit)
};

__device__ __forceinline__ void decode_unit(int u, int bh_count, int n_pairs, int heads_per_group,
                                            bool causal, int& bh, int& pair) {
    if (causal) {
        // Heads in groups of heads_per_group; inside a group the longest
        // query tiles (largest pair index) come first.
        const int group_units = heads_per_group * n_pairs;
        const int g = u / group_units;
        const int r = u - g * group_units;
        const int hg = min(heads_per_group, bh_count - g * heads_per_group);
        pair = n_pairs - 1 - r / hg;
        bh = g * heads_per_group + r % hg;
    } else {
        bh = u / n_pairs;
        pair = u - bh * n_pairs;
    }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(Bf16Cfg<D>::THREADS, 1)
fa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const Bf16Params p) {
    using C = Bf16Cfg<D>;
    using B = Bars<C::NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                                  // 2 tiles
    uint8_t* sKV = smem + 2 * C::TILE_BYTES;             // NS tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::NS * C::TILE_BYTES);
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    volatile int* abort_flag = &abort_sh;
    auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

    int bh, pair;
    decode_unit(blockIdx.x, p.bh_count, p.n_pairs, p.heads_per_group, CAUSAL, bh, pair);
    const int q0 = pair * 256;
    const int nkv = (p.N + C::BN - 1) / C::BN;
    int n_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qs = q0 + 128 * t;
        if (qs >= p.M) n_t[t] = 0;
        else n_t[t] = CAUSAL ? min(nkv, qs / C::BN + 1) : nkv;
    }
    const int nmax = max(n_t[0], n_t[1]);

    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(bar(B::full + s), 1);
            mbar_init(bar(B::empty + s), 1);
        }
        mbar_init(bar(B::q_full), 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B::s_full + t), 1);
            mbar_init(bar(B::p_ready + t), 128);
            mbar_init(bar(B::o_done + t), 1);
        }
        mbar_init(bar(B::drain), 1);
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(&tmem_base_sh), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 8) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            const int nq = (n_t[0] > 0 ? 1 : 0) + (n_t[1] > 0 ? 1 : 0);
            if (nq > 0) {
                mbar_arrive_expect_tx(bar(B::q_full), nq * C::TILE_BYTES);
                for (int t = 0; t < 2; ++t) {
                    if (n_t[t] == 0) continue;
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_3d(smem_u32(sQ + t * C::TILE_BYTES + pn * C::PANEL_BYTES), &map_q,
                                    bar(B::q_full), pn * 64, q0 + 128 * t, bh, pol_q);
                }
            }
            int idx = 0;
            bool ok = true;
            for (int j = 0; j < nmax && ok; ++j) {
                for (int which = 0; which < 2; ++which) {
                    const int stage = idx % C::NS;
                    const int round = idx / C::NS;
                    if (round > 0 && !mbar_wait(bar(B::empty + stage), (round - 1) & 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(B::full + stage), C::TILE_BYTES);
                    const CUtensorMap* m = which ? &map_v : &map_k;
                    for (int pn = 0; pn < C::PANELS; ++pn)
                        tma_load_3d(smem_u32(sKV + stage * C::TILE_BYTES + pn * C::PANEL_BYTES), m,
                                    bar(B::full + stage), pn * 64, j * C::BN, bh, pol_kv);
                    ++idx;
                }
            }
            // Every copy issued must land before this CTA's shared memory is
            // released: wait for the last fill of each stage and for Q.
            for (int s = 0; s < C::NS && s < idx; ++s) {
                const int last = s + ((idx - 1 - s) / C::NS) * C::NS;
                mbar_wait_drain(bar(B::full + s), (last / C::NS) & 1);
            }
            if (nq > 0) mbar_wait_drain(bar(B::q_full), 0);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ----------------------------------------------------- MMA issuer
        if (lane == 0 && nmax > 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(128, C::BN, false);
            constexpr uint32_t id_o = idesc_bf16_f32(128, D, true);
            const uint32_t sq = smem_u32(sQ);
            const uint32_t skv = smem_u32(sKV);
            const uint32_t s_col[2] = {C::S_COL0, C::S_COL1};
            const uint32_t o_col[2] = {C::O_COL0, C::O_COL1};
            bool ok = mbar_wait(bar(B::q_full), 0, abort_flag, p.err);
            tc_fence_after();
            for (int j = 0; j <= nmax && ok; ++j) {
                const int kidx = 2 * j, vidx = 2 * j - 1;
                const int kst = kidx % C::NS, vst = (vidx + C::NS) % C::NS;
                if (j < nmax && !mbar_wait(bar(B::full + kst), (kidx / C::NS) & 1, abort_flag, p.err)) break;
                if (j >= 1 && !mbar_wait(bar(B::full + vst), (vidx / C::NS) & 1, abort_flag, p.err)) break;
                tc_fence_after();
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j >= 1 && j - 1 < n_t[t]) {
                        if (!mbar_wait(bar(B::p_ready + t), (j - 1) & 1, abort_flag, p.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t vb = skv + vst * C::TILE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                            const uint64_t bd = smem_desc_sw128(vb + kk * 2048, C::PANEL_BYTES, 1024);
                            mma_ts(tmem + o_col[t], tmem + s_col[t] + kk * 8, bd, id_o,
                                   (j > 1 || kk > 0) ? 1u : 0u);
                        }
                        if (j - 1 == n_t[t] - 1) mma_commit(bar(B::o_done + t));
                    }
                    if (j < n_t[t]) {
                        const uint32_t qb = sq + t * C::TILE_BYTES;
                        const uint32_t kb = skv + kst * C::TILE_BYTES;
#pragma unroll
                        for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                            const uint32_t off = (kk >> 2) * C::PANEL_BYTES + (kk & 3) * 32;
                            const uint64_t ad = smem_desc_sw128(qb + off, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(kb + off, 16, 1024);
                            mma_ss(tmem + s_col[t], ad, bd, id_s, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(B::s_full + t));
                    }
                }
                if (!ok) break;
                if (j < nmax) mma_commit(bar(B::empty + kst));
                if (j >= 1) mma_commit(bar(B::empty + vst));
            }
            // All MMAs issued must finish before tensor memory is freed.
            mma_commit(bar(B::drain));
            mbar_wait_drain(bar(B::drain), 0);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- softmax
        const int t = warp >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;                       // row in the tile
        const int qrow = q0 + 128 * t + r;                  // query row
        const int ntile = n_t[t];
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + (t ? C::S_COL1 : C::S_COL0);
        const uint32_t o_addr = tmem + lane_base + (t ? C::O_COL1 : C::O_COL0);
        const float c = p.scale_log2;
        float m_run = -INFINITY;   // running max of scaled scores, base-2 units
        float l_run = 0.f;         // running sum of exp2(score - m_run)
        bool ok = true;

        for (int j = 0; j < ntile; ++j) {
            // Every lane must agree: the tensor-memory loads below are
            // warp-collective.
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B::s_full + t), j & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[128];
            {
                uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
                uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
                uint32_t (&cc)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[64]);
                uint32_t (&d)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[96]);
                tmem_ld_x32(s_addr + 0, a);
                tmem_ld_x32(s_addr + 32, b);
                tmem_ld_x32(s_addr + 64, cc);
                tmem_ld_x32(s_addr + 96, d);
                tmem_ld_wait(s);
            }
            const int kv0 = j * C::BN;
            const bool need_mask = (kv0 + C::BN > p.N) || (CAUSAL && kv0 + C::BN - 1 > q0 + 128 * t);
            if (need_mask) {
                int lim = p.N - kv0;                         // key columns < N
                if (CAUSAL) lim = min(lim, qrow - kv0 + 1);  // key <= query
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i >= lim) s[i] = __float_as_uint(-INFINITY);
            }
            float mx = __uint_as_float(s[0]);
#pragma unroll
            for (int i = 1; i < 128; ++i) mx = fmaxf(mx, __uint_as_float(s[i]));
            const float m_new = fmaxf(m_run, mx * c);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m_run - m_use);
            const float neg = -m_use;
            float sum0 = 0.f, sum1 = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const float p0 = ex2(fmaf(__uint_as_float(s[2 * i]), c, neg));
                const float p1 = ex2(fmaf(__uint_as_float(s[2 * i + 1]), c, neg));
                sum0 += p0;
                sum1 += p1;
                pk[i] = pack_bf16x2(p0, p1);
            }
            l_run = l_run * alpha + (sum0 + sum1);
            m_run = m_new;
            tmem_st_x32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            // Rescale the output accumulator to the new max (tile 0 has no
            // accumulator yet: its first product overwrites O).
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    tmem_ld_x32(o_addr + cc * 32, ov);
                    tmem_ld_wait(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st_x32(o_addr + cc * 32, ov);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(B::p_ready + t));
        }

        // ---------------------------------------------------------- epilogue
        if (ok && ntile > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::o_done + t), 0, abort_flag, p.err));
            tc_fence_after();
        }
        if (ok && q0 + 128 * t < p.M) {
            const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
            const bool store = qrow < p.M;
            uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +   // bf16 bits
                             (static_cast<size_t>(bh) * p.M + (store ? qrow : 0)) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                if (ntile > 0) {
                    tmem_ld_x32(o_addr + cc * 32, ov);
                    tmem_ld_wait(ov);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = 0u;
                }
                uint32_t pkd[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pkd[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
                }
            }
            if (store) {
                // LSE in natural-log units: ln2 * (m + log2 l); -inf when no key was visible.
                p.lse[static_cast<size_t>(bh) * p.M + qrow] =
                    (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_bf16(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const Bf16Params& p,
                        bool causal, cudaStream_t stream) {
    using C = Bf16Cfg<D>;
    const int units = p.bh_count * p.n_pairs;
    auto kern = causal ? fa_fwd_bf16_kernel<D, true> : fa_fwd_bf16_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<units, C::THREADS, C::SMEM_BYTES, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

}  // namespace fa
