// kt_decode_dev.cuh -- block- and warp-level pieces of the single-launch
// decode kernel (kt_mxfp4_moe_decode): routing one token with one warp, the
// stable permutation of up to kDecodeMaxSlots slots by one CTA, and a grid
// barrier with a deadline.
//
// The routing and permutation compute exactly what route_topk_kernel and the
// permutation kernels of kt_route_permute.cu compute (same selection order,
// same fp64 weight arithmetic and summation order, same stable ranks), so the
// decode kernel's ids, weights and indices equal the multi-launch path's.
#pragma once

#include <cmath>

#include "kt_common.cuh"
#include "kt_internal.h"

namespace kt {

// Route one token with one warp: k rounds of a warp arg-max over its E
// logits (value descending, index ascending; lane l holds experts l, l+32,
// ... in EPL registers, EPL a power of two >= ceil(E / 32)), then the gating
// weights in fp64, rounded to f32 once: the softmax over the k selected
// logits (renormalize) or the full softmax over E taken at them.  Top-k
// routing as in the DeepSeek-V4-Flash (top-6 of 256) and Kimi-K3 (top-16 of
// 896) layers the pages name.  kShared: the logits row (and nothing else)
// is in shared memory.
template <int EPL, bool kShared>
__device__ __forceinline__ void route_token_warp_t(const float* __restrict__ row, int E, int k, int renormalize,
                                                   int32_t* __restrict__ ids, float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    constexpr int kNone = 0x7fffffff;
    float v[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? (kShared ? row[e] : __ldg(row + e)) : -INFINITY;
    }
    uint32_t taken = 0;
    int my_id = 0;
    float my_v = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = kNone;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u)) {
                if (bi == kNone || v[i] > bv) {
                    bv = v[i];
                    bi = e;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (oi != kNone && (bi == kNone || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_id = bi;
            my_v = bv;
        }
    }
    if (lane < k) ids[lane] = my_id;
    const double lmax = static_cast<double>(__shfl_sync(0xffffffffu, my_v, 0));
    const double ex = (lane < k) ? exp(static_cast<double>(my_v) - lmax) : 0.0;
    double part = 0.0;
    if (renormalize) {
        for (int jj = 0; jj < k; ++jj) part += __shfl_sync(0xffffffffu, ex, jj);
    } else {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) part += exp(static_cast<double>(v[i]) - lmax);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    }
    if (lane < k) w[lane] = static_cast<float>(ex / part);
}

template <bool kShared = false>
__device__ __forceinline__ void route_token_warp(const float* __restrict__ row, int E, int k, int renormalize,
                                                 int32_t* __restrict__ ids, float* __restrict__ w) {
    const int epl = (E + 31) >> 5;   // E <= 1024 keeps this <= 32
    if (epl <= 1) route_token_warp_t<1, kShared>(row, E, k, renormalize, ids, w);
    else if (epl <= 2) route_token_warp_t<2, kShared>(row, E, k, renormalize, ids, w);
    else if (epl <= 4) route_token_warp_t<4, kShared>(row, E, k, renormalize, ids, w);
    else if (epl <= 8) route_token_warp_t<8, kShared>(row, E, k, renormalize, ids, w);
    else if (epl <= 16) route_token_warp_t<16, kShared>(row, E, k, renormalize, ids, w);
    else route_token_warp_t<32, kShared>(row, E, k, renormalize, ids, w);
}

// Stable token-to-expert permutation of S <= kDecodeMaxSlots slots by one
// CTA of nwarps warps (the histogram -> exclusive scan -> stable scatter of
// the permutation step): warp w owns the contiguous slots
// [w * seg, (w + 1) * seg) and counts them per expert into row w of s_cnt
// ([nwarps][E] ints of shared memory); thread t then owns experts
// [4t, 4t + 4) for the scans that give expert_offsets and chunk_prefix; each
// warp finally sweeps its slots again in slot order and ranks equal experts
// with match.any.  Writes expert_offsets [E+1], chunk_prefix [E+1], perm [S]
// (-1 past the valid rows), inv_perm [S] (-1 for an id outside [0, E)).
// kShared: ids and the four outputs are in shared memory (otherwise ids were
// written earlier in the same launch and are read past L1).
constexpr int kDecodeMaxSlots = KT_DECODE_MAX_SLOTS;

__device__ __forceinline__ int block_exclusive_scan(int x, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = static_cast<int>(blockDim.x) >> 5;
    int inc = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int wv = lane < nwarps ? s_warp[lane] : 0;
        int winc = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, winc, off);
            if (lane >= off) winc += y;
        }
        if (lane < nwarps) s_warp[lane] = winc - wv;
        if (lane == 31) s_warp[32] = winc;
    }
    __syncthreads();
    const int res = s_warp[warp] + inc - x;
    *total = s_warp[32];
    __syncthreads();
    return res;
}

template <bool kShared = false>
__device__ __forceinline__ void permute_block(const int32_t* __restrict__ ids, int S, int E,
                                              int32_t* __restrict__ offsets, int32_t* __restrict__ chunk_prefix,
                                              int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm, int* err,
                                              int* s_cnt, int* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = static_cast<int>(blockDim.x) >> 5;
    for (int i = threadIdx.x; i < nwarps * E; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();
    const int seg = ((S + nwarps - 1) / nwarps + 31) & ~31;
    const int s0 = warp * seg;
    const int s1 = min(S, s0 + seg);
    int* cnt = s_cnt + warp * E;
    bool bad = false;
    for (int r = s0; r < s1; r += 32) {   // warp-uniform bounds
        const int s = r + lane;
        int e = -1;
        if (s < s1) {
            e = kShared ? ids[s] : __ldcg(ids + s);   // written earlier in the same launch
            if (e < 0 || e >= E) {
                bad = true;
                e = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
        __syncwarp();
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, KT_DEVERR_BAD_EXPERT_ID);
    __syncthreads();
    // experts [4t, 4t + 4) of thread t: counts over warps -> per-warp bases (relative to the expert)
    int tot[4], nch[4];
    int my_tot = 0, my_nch = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = 4 * static_cast<int>(threadIdx.x) + u;
        int run = 0;
        if (e < E) {
            for (int ww = 0; ww < nwarps; ++ww) {
                const int c = s_cnt[ww * E + e];
                s_cnt[ww * E + e] = run;
                run += c;
            }
        }
        tot[u] = run;
        nch[u] = (run + kChunkRows - 1) / kChunkRows;
        my_tot += tot[u];
        my_nch += nch[u];
    }
    int total_cnt, total_ch;
    int off = block_exclusive_scan(my_tot, s_warp, &total_cnt);
    int cpre = block_exclusive_scan(my_nch, s_warp, &total_ch);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = 4 * static_cast<int>(threadIdx.x) + u;
        if (e < E) {
            offsets[e] = off;
            chunk_prefix[e] = cpre;
            for (int ww = 0; ww < nwarps; ++ww) s_cnt[ww * E + e] += off;
        }
        off += tot[u];
        cpre += nch[u];
    }
    if (threadIdx.x == 0) {
        offsets[E] = total_cnt;
        chunk_prefix[E] = total_ch;
    }
    __syncthreads();
    for (int r = s0; r < s1; r += 32) {
        const int s = r + lane;
        int e = -1;
        if (s < s1) {
            e = kShared ? ids[s] : __ldcg(ids + s);
            if (e < 0 || e >= E) e = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int before = (e >= 0) ? cnt[e] : 0;
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] = before + __popc(peers);
        __syncwarp();
        if (s < s1) {
            const int pos = (e >= 0) ? before + rank : -1;
            inv_perm[s] = pos;
            if (pos >= 0) perm[pos] = s;
        }
    }
    for (int p = total_cnt + threadIdx.x; p < S; p += blockDim.x) perm[p] = -1;
}

// Grid-wide barrier of a cooperative launch (every CTA resident): the
// calling CTA arrives on *ctr once and waits until it reaches `target`
// (the caller counts barriers: target = barrier number x gridDim.x), with a
// deadline.  Memory written before the barrier by any CTA is visible after
// it, to the generic proxy and (fence.proxy.async) to TMA loads.  On expiry
// sets KT_DEVERR_TIMEOUT_GRID and the CTA's abort flag and returns false;
// returns false at once when the abort flag is already up.
__device__ __forceinline__ bool grid_barrier(unsigned* ctr, unsigned target, volatile int* abort_flag, int* err,
                                             uint64_t limit_ns) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
            if (v >= target) break;
            if (*abort_flag || globaltimer_ns() - t0 > limit_ns) {
                set_error(err, KT_DEVERR_TIMEOUT_GRID);
                *abort_flag = 1;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
    }
    __syncthreads();
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return *abort_flag == 0;
}

}  // namespace kt
