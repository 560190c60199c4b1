// kt_route_permute.cu -- route (top-k + softmax weights) and the
// deterministic token-to-expert permutation.
//
// Routing follows the top-k expert selection of the DeepSeek-V4-Flash
// (256 experts, top-6) and Kimi-K3 (896 experts, top-16) MoE layers named in
// "[MXFP4 layerwise prefill] SM 8.6 (Ampere) excluded by capability
// whitelist" (Environment) and "Kimi-K3 SM120 FlashInfer MXFP4 MoE" (Phase 0
// audit table).  The permutation groups slots by expert so that each expert's
// rows are contiguous ("different expert hits", Kimi-K3 README, later hard
// gates, item 5); within an expert, rows keep slot order, which makes every
// index bit-reproducible.
#include <cmath>

#include "kt_common.cuh"
#include "kt_internal.h"

namespace kt {

// ------------------------------------------------------------------ route
// One warp per token, eight tokens per block.  Lane l holds logits l, l+32,
// ...; k rounds of a warp arg-max (value descending, index ascending) pick
// the experts in order.  Weights are exp(l_j - l_max) / sum in fp64 (the
// difference of two f32 logits is exact in fp64), then rounded to f32.
// GB300 runs fp64 at a small fraction of its fp32 rate and a warp-wide fp64
// instruction costs the same with 6 lanes active as with 32, so for the
// default renormalised weights the fp64 work runs in a second phase with one
// thread per (token, selected expert) of the block: top-6 packs 48 exps into
// 2 warps instead of 8.
// EPL = expert slots per lane, a power of two >= ceil(E / 32): the candidate
// scans run over EPL slots, not 32 (E = 256 needs 8).
constexpr int kRouteTokensPerBlock = 8;

template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int renormalize, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float s_v[kRouteTokensPerBlock][32];     // selected logits, in selection order
    __shared__ double s_ex[kRouteTokensPerBlock][32];   // their exp(l_j - l_max)
    __shared__ double s_part[kRouteTokensPerBlock];     // per-token sum
    const int tb = static_cast<int>(threadIdx.x >> 5);  // token within the block
    const int t = static_cast<int>(blockIdx.x) * kRouteTokensPerBlock + tb;
    const int lane = threadIdx.x & 31;
    const bool active = t < T;
    float v[EPL];
    int my_id = 0;
    float my_v = 0.f;
    if (active) {
        const float* row = logits + static_cast<size_t>(t) * E;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = (e < E) ? row[e] : -INFINITY;
        }
        constexpr int kNone = 0x7fffffff;
        uint32_t taken = 0;
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
        if (lane < k) ids[static_cast<size_t>(t) * k + lane] = my_id;
    }
    if (!renormalize) {
        // full softmax over all E logits (a flag): every lane's logits enter the sum
        if (!active) return;
        const double lmax = static_cast<double>(__shfl_sync(0xffffffffu, my_v, 0));
        const double ex = (lane < k) ? exp(static_cast<double>(my_v) - lmax) : 0.0;
        double part = 0.0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) part += exp(static_cast<double>(v[i]) - lmax);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane < k) w[static_cast<size_t>(t) * k + lane] = static_cast<float>(ex / part);
        return;
    }
    if (active && lane < k) s_v[tb][lane] = my_v;
    __syncthreads();
    const int nt = min(kRouteTokensPerBlock, T - static_cast<int>(blockIdx.x) * kRouteTokensPerBlock);
    const int i = static_cast<int>(threadIdx.x);
    const bool mine = i < nt * k;
    const int ti = mine ? i / k : 0;
    const int j = mine ? i - ti * k : 0;
    double ex = 0.0;
    if (mine) {
        ex = exp(static_cast<double>(s_v[ti][j]) - static_cast<double>(s_v[ti][0]));
        s_ex[ti][j] = ex;
    }
    __syncthreads();
    if (i < nt) {
        double part = 0.0;
        for (int jj = 0; jj < k; ++jj) part += s_ex[i][jj];
        s_part[i] = part;
    }
    __syncthreads();
    if (mine) {
        const size_t tt = static_cast<size_t>(blockIdx.x) * kRouteTokensPerBlock + ti;
        w[tt * k + j] = static_cast<float>(ex / s_part[ti]);
    }
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int renormalize, int32_t* ids, float* w,
                              cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int blocks = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
    const int epl = (E + 31) / 32;   // E <= kMaxExperts = 1024 keeps this <= 32
    auto go = [&](auto kernel) {
        return launch_chained(kernel, dim3(blocks), dim3(256), 0, s, logits, T, E, k, renormalize, ids, w);
    };
    cudaError_t e;
    if (epl <= 1) e = go(route_topk_kernel<1>);
    else if (epl <= 2) e = go(route_topk_kernel<2>);
    else if (epl <= 4) e = go(route_topk_kernel<4>);
    else if (epl <= 8) e = go(route_topk_kernel<8>);
    else if (epl <= 16) e = go(route_topk_kernel<16>);
    else e = go(route_topk_kernel<32>);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------------------------------ permute
// Pass 1: per-tile expert histogram (tile = kPermTile consecutive slots).
__global__ void __launch_bounds__(256) perm_hist_kernel(const int32_t* __restrict__ ids, long long S, int E,
                                                        int32_t* __restrict__ hist, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ int sh_count[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) sh_count[e] = 0;
    __syncthreads();
    const long long base = static_cast<long long>(blockIdx.x) * kPermTile;
    int bad = 0;
    for (int i = threadIdx.x; i < kPermTile; i += blockDim.x) {
        const long long s = base + i;
        if (s < S) {
            const int e = ids[s];
            if (e >= 0 && e < E) atomicAdd(&sh_count[e], 1);
            else bad = 1;
        }
    }
    if (bad) set_error(err, KT_DEVERR_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<size_t>(blockIdx.x) * E + e] = sh_count[e];
}

// Exclusive scan over the 1024 threads of a block; returns the thread's
// exclusive prefix and writes the block total to *total (all threads).
__device__ __forceinline__ int block_exclusive_scan_1024(int x, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int wv = s_warp[lane];
        int winc = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, winc, off);
            if (lane >= off) winc += y;
        }
        s_warp[lane] = winc - wv;                 // exclusive prefix of warp totals
        if (lane == 31) s_warp[32] = winc;        // block total
    }
    __syncthreads();
    const int res = s_warp[warp] + inc - x;
    *total = s_warp[32];
    __syncthreads();
    return res;
}

// Pass 2 (one block of 1024 threads, thread = expert): in-place exclusive
// prefix of each expert's tile counts, expert offsets, token-chunk prefix.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ hist, int ntiles, int E, long long S,
                                                         int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ chunk_prefix,
                                                         int32_t* __restrict__ perm) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int s_warp[33];
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int t0 = 0; t0 < ntiles; t0 += 8) {
            int h[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) h[u] = (t0 + u < ntiles) ? hist[static_cast<size_t>(t0 + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (t0 + u < ntiles) {
                    hist[static_cast<size_t>(t0 + u) * E + e] = run;
                    run += h[u];
                }
            }
        }
    }
    const int cnt = (e < E) ? run : 0;
    const int nch = (cnt + kChunkRows - 1) / kChunkRows;
    int total_cnt, total_ch;
    const int off = block_exclusive_scan_1024(cnt, s_warp, &total_cnt);
    const int cpre = block_exclusive_scan_1024(nch, s_warp, &total_ch);
    if (e < E) {
        offsets[e] = off;
        chunk_prefix[e] = cpre;
    }
    if (e == 0) {
        offsets[E] = total_cnt;
        chunk_prefix[E] = total_ch;
    }
    for (long long p = total_cnt + threadIdx.x; p < S; p += blockDim.x) perm[p] = -1;
}

// Pass 3 (one block of 128 threads per tile): the tile's ids and the
// per-expert bases (expert offset + tile prefix) are staged in shared memory
// first.  Warp w owns the tile's slots [256 w, 256 w + 256): it counts them
// per expert (match.any, one lane per distinct expert adding the round's
// count), an exclusive prefix over the four warps turns the counts into
// per-warp bases, and each warp then sweeps its slots in slot order, ranking
// peers with match.any, so equal experts keep slot order across rounds and
// warps.  Ranks and outputs are written back by all 128 threads.
constexpr int kScatterWarps = 4;
constexpr int kScatterSeg = kPermTile / kScatterWarps;

__global__ void __launch_bounds__(128) perm_scatter_kernel(const int32_t* __restrict__ ids, long long S, int E,
                                                           const int32_t* __restrict__ tile_base,
                                                           const int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ perm,
                                                           int32_t* __restrict__ inv_perm) {
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ int sh[];
    int* s_base = sh;                      // [E]   offsets[e] + tile prefix
    int* s_id = sh + E;                    // [kPermTile] expert of each slot (-1 invalid / past S)
    int* s_pos = s_id + kPermTile;         // [kPermTile] permuted row of each slot
    int* s_w = s_pos + kPermTile;          // [kScatterWarps][E] per-warp counts, then running bases
    const long long base = static_cast<long long>(blockIdx.x) * kPermTile;
    const int32_t* tb = tile_base + static_cast<size_t>(blockIdx.x) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_base[e] = offsets[e] + tb[e];
    for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) s_w[i] = 0;
    for (int i = threadIdx.x; i < kPermTile; i += blockDim.x) {
        const long long s = base + i;
        int e = -1;
        if (s < S) {
            e = ids[s];
            if (e < 0 || e >= E) e = -1;
        }
        s_id[i] = e;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int* cnt = s_w + warp * E;
    const int i0 = warp * kScatterSeg;
    for (int r = 0; r < kScatterSeg / 32; ++r) {
        const int e = s_id[i0 + r * 32 + lane];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = s_base[e];
        for (int w = 0; w < kScatterWarps; ++w) {
            const int c = s_w[w * E + e];
            s_w[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int r = 0; r < kScatterSeg / 32; ++r) {
        const int e = s_id[i0 + r * 32 + lane];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int before = (e >= 0) ? cnt[e] : 0;
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] = before + __popc(peers);
        __syncwarp();
        s_pos[i0 + r * 32 + lane] = (e >= 0) ? before + rank : -1;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kPermTile; i += blockDim.x) {
        const long long s = base + i;
        if (s >= S) break;
        const int pos = s_pos[i];
        inv_perm[s] = pos;
        if (pos >= 0) perm[pos] = static_cast<int32_t>(s);
    }
}

// Single-block permutation for S <= kPermFusedMaxSlots: the three passes
// above in one launch of 1024 threads.  At decode sizes it takes 9-10 us
// against 15-18 us for the three launches on GB300; its sequential rounds
// lose beyond a few thousand slots (46 us against 23-26 us at 24576).  Warp w owns the contiguous slots
// [w * seg, (w + 1) * seg) (seg = ceil(S / 32) rounded up to 32) and keeps
// its per-expert counts in row w of a [32][E] shared-memory table:
//   1. each warp counts its slots, 32 per round, one lane per distinct expert
//      (match.any) adding the round's count;
//   2. thread e turns column e into exclusive bases over warps, and a block
//      scan gives expert_offsets and chunk_prefix;
//   3. each warp sweeps its slots again in slot order, ranking peers with
//      match.any, so equal experts keep slot order across rounds and warps.
constexpr int kPermFusedMaxSlots = 2048;
constexpr int kPermFusedUnroll = 4;   // rounds whose ids are loaded together

__global__ void __launch_bounds__(1024) perm_fused_kernel(const int32_t* __restrict__ ids, int S, int E,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ chunk_prefix,
                                                          int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm,
                                                          int* err) {
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ int s_cnt[];   // [32][E]: counts, then bases
    __shared__ int s_warp[33];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();
    const int seg = ((S + 31) / 32 + 31) & ~31;
    const int s0 = warp * seg;
    const int s1 = min(S, s0 + seg);
    int* cnt = s_cnt + warp * E;
    bool bad = false;
    // expert of slot s, or -1 outside [s0, s1) or for an id outside [0, E)
    auto load = [&](int s, bool& flag) {
        if (s >= s1) return -1;
        const int e = __ldg(ids + s);
        if (e < 0 || e >= E) {
            flag = true;
            return -1;
        }
        return e;
    };
    for (int r = s0; r < s1; r += 32 * kPermFusedUnroll) {   // warp-uniform bounds
        int e4[kPermFusedUnroll];
#pragma unroll
        for (int u = 0; u < kPermFusedUnroll; ++u) e4[u] = load(r + 32 * u + lane, bad);
#pragma unroll
        for (int u = 0; u < kPermFusedUnroll; ++u) {
            const unsigned peers = __match_any_sync(0xffffffffu, e4[u]);
            if (e4[u] >= 0 && lane == __ffs(peers) - 1) cnt[e4[u]] += __popc(peers);
            __syncwarp();
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, KT_DEVERR_BAD_EXPERT_ID);
    __syncthreads();
    const int e = threadIdx.x;   // E <= kMaxExperts = blockDim.x
    int tot = 0;
    if (e < E) {
        for (int w = 0; w < 32; ++w) {
            const int c = s_cnt[w * E + e];
            s_cnt[w * E + e] = tot;
            tot += c;
        }
    }
    const int nch = (tot + kChunkRows - 1) / kChunkRows;
    int total_cnt, total_ch;
    const int off = block_exclusive_scan_1024(tot, s_warp, &total_cnt);
    const int cpre = block_exclusive_scan_1024(nch, s_warp, &total_ch);
    if (e < E) {
        offsets[e] = off;
        chunk_prefix[e] = cpre;
        for (int w = 0; w < 32; ++w) s_cnt[w * E + e] += off;
    }
    if (e == 0) {
        offsets[E] = total_cnt;
        chunk_prefix[E] = total_ch;
    }
    __syncthreads();
    bool unused = false;
    for (int r = s0; r < s1; r += 32 * kPermFusedUnroll) {
        int e4[kPermFusedUnroll];
#pragma unroll
        for (int u = 0; u < kPermFusedUnroll; ++u) e4[u] = load(r + 32 * u + lane, unused);
#pragma unroll
        for (int u = 0; u < kPermFusedUnroll; ++u) {
            const int ee = e4[u];
            const unsigned peers = __match_any_sync(0xffffffffu, ee);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int before = (ee >= 0) ? cnt[ee] : 0;
            __syncwarp();
            if (ee >= 0 && lane == __ffs(peers) - 1) cnt[ee] = before + __popc(peers);
            __syncwarp();
            const int sl = r + 32 * u + lane;
            if (sl < s1) {
                const int pos = (ee >= 0) ? before + rank : -1;
                inv_perm[sl] = pos;
                if (pos >= 0) perm[pos] = sl;
            }
        }
    }
    for (int p = total_cnt + threadIdx.x; p < S; p += blockDim.x) perm[p] = -1;
}

cudaError_t launch_permute(const int32_t* ids, long long S, int E, int32_t* hist, int32_t* expert_offsets,
                           int32_t* chunk_prefix, int32_t* perm, int32_t* inv_perm, int* err, cudaStream_t s) {
    const int ntiles = perm_tiles(S);
    if (S <= kPermFusedMaxSlots) {
        static bool attr_set[64] = {};
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev >= 0 && dev < 64 && !attr_set[dev]) {
            const cudaError_t ea = cudaFuncSetAttribute(perm_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                        32 * kMaxExperts * static_cast<int>(sizeof(int)));
            if (ea != cudaSuccess) return ea;
            attr_set[dev] = true;
        }
        if (S > 0) {
            const cudaError_t e = launch_chained(perm_fused_kernel, dim3(1), dim3(1024), 32 * E * sizeof(int), s, ids,
                                                 static_cast<int>(S), E, expert_offsets, chunk_prefix, perm,
                                                 inv_perm, err);
            count_launches(1);
            return e != cudaSuccess ? e : cudaGetLastError();
        }
    }
    if (ntiles > 0) {
        cudaError_t e = launch_chained(perm_hist_kernel, dim3(ntiles), dim3(256), E * sizeof(int), s, ids, S, E, hist,
                                       err);
        count_launches(1);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_chained(perm_scan_kernel, dim3(1), dim3(1024), 0, s, hist, ntiles, E, S, expert_offsets,
                                   chunk_prefix, perm);
    count_launches(1);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ntiles > 0) {
        e = launch_chained(perm_scatter_kernel, dim3(ntiles), dim3(128),
                           ((1 + kScatterWarps) * E + 2 * kPermTile) * sizeof(int), s, ids, S, E, hist,
                           expert_offsets, perm, inv_perm);
        count_launches(1);
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    return e;
}

// Token-chunk prefix from expert offsets alone (one block, thread = expert).
__global__ void __launch_bounds__(1024) chunk_prefix_kernel(const int32_t* __restrict__ offsets, int E,
                                                            int32_t* __restrict__ chunk_prefix) {
    __shared__ int s_warp[33];
    const int e = threadIdx.x;
    const int cnt = (e < E) ? offsets[e + 1] - offsets[e] : 0;
    const int nch = cnt > 0 ? (cnt + kChunkRows - 1) / kChunkRows : 0;
    int total;
    const int cpre = block_exclusive_scan_1024(nch, s_warp, &total);
    if (e < E) chunk_prefix[e] = cpre;
    if (e == 0) chunk_prefix[E] = total;
}

cudaError_t launch_chunk_prefix(const int32_t* expert_offsets, int E, int32_t* chunk_prefix, cudaStream_t s) {
    chunk_prefix_kernel<<<1, 1024, 0, s>>>(expert_offsets, E, chunk_prefix);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace kt
