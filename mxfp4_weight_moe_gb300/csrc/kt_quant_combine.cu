// kt_quant_combine.cu -- the HBM-bound ends of the layer: MXFP8 activation
// quantisation fused with the permuted scatter, and the final top-k combine.
//
// MXFP8 (e4m3 elements, one e8m0 scale per 32 along H) is the activation
// format of the "MXFP8 activation x MXFP4 weight fused MoE" ("Kimi-K3 SM120
// FlashInfer MXFP4 MoE", Goal).  The shared exponent follows the OCP MX v1.0
// rule floor(log2 amax) - 8 and elements are converted with round-to-
// nearest-even, saturating at +-448.
#include "kt_common.cuh"
#include "kt_decode_dev.cuh"
#include "kt_internal.h"
#include "kt_quant_dev.cuh"

namespace kt {

// One warp per (token row, pass of 1024 elements) (quant_token_warp in kt_quant_dev.cuh).
// With `offsets` given, one extra block (the last) also derives chunk_prefix
// [E+1] from expert_offsets [E+1]: the chunks of kChunkRows rows each expert's
// rows split into, as an exclusive prefix sum (what the permutation kernels
// write), for a forward that reuses a routing call's permutation.
__global__ void __launch_bounds__(256) quant_scatter_kernel(const uint16_t* __restrict__ hidden, int T, int H, int k,
                                                            const int32_t* __restrict__ inv_perm,
                                                            uint8_t* __restrict__ a1, uint8_t* __restrict__ a1_sf,
                                                            int S4, const int32_t* __restrict__ offsets, int E,
                                                            int32_t* __restrict__ chunk_prefix) {
    griddep_wait();
    griddep_launch_dependents();
    if (offsets != nullptr && blockIdx.x == gridDim.x - 1) {
        __shared__ int s_warp[33];
        constexpr int kPer = (kMaxExperts + 255) / 256;   // experts per thread
        int nch[kPer];
        int mine = 0;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = static_cast<int>(threadIdx.x) * kPer + u;
            const int cnt = e < E ? offsets[e + 1] - offsets[e] : 0;
            nch[u] = cnt > 0 ? (cnt + kChunkRows - 1) / kChunkRows : 0;
            mine += nch[u];
        }
        int total;
        int run = block_exclusive_scan(mine, s_warp, &total);
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int e = static_cast<int>(threadIdx.x) * kPer + u;
            if (e < E) chunk_prefix[e] = run;
            run += nch[u];
        }
        if (threadIdx.x == 0) chunk_prefix[E] = total;
        return;
    }
    __shared__ int s_dst[8][kMaxTopK];
    const int wib = threadIdx.x >> 5;
    const int per_row = quant_items_per_row(H);
    const long long item = static_cast<long long>(blockIdx.x) * 8 + wib;
    if (item >= static_cast<long long>(T) * per_row) return;   // whole warp
    const int t = static_cast<int>(item / per_row);
    const int c = static_cast<int>(item - static_cast<long long>(t) * per_row);
    quant_token_warp(hidden, t, H, k, inv_perm, a1, a1_sf, S4, s_dst[wib], c, c + 1);
}

cudaError_t launch_quant_scatter(const uint16_t* hidden, int T, int H, int k, const int32_t* inv_perm, uint8_t* a1,
                                 uint8_t* a1_sf, int S4, cudaStream_t s, const int32_t* offsets, int E,
                                 int32_t* chunk_prefix) {
    if (T <= 0) return cudaSuccess;
    const long long items = static_cast<long long>(T) * quant_items_per_row(H);
    const unsigned blocks = static_cast<unsigned>((items + 7) / 8) + (offsets != nullptr ? 1u : 0u);
    const cudaError_t e = launch_chained(quant_scatter_kernel, dim3(blocks), dim3(256), 0, s, hidden, T, H, k, inv_perm,
                                         a1, a1_sf, S4, offsets, E, chunk_prefix);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Plain [S, K/32] scale bytes -> K-step-major u32 [K/128][S4] (one thread per
// row and K step; rows S..S4-1 are zero).
__global__ void __launch_bounds__(256) sf_to_kstep_major_kernel(const uint8_t* __restrict__ plain, int S, int K,
                                                                uint32_t* __restrict__ out, int S4) {
    const int nks = K / 128;
    const long long n = static_cast<long long>(nks) * S4;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int ks = static_cast<int>(i / S4);
        const int r = static_cast<int>(i % S4);
        uint32_t v = 0;
        if (r < S) {
            const uint8_t* src = plain + static_cast<size_t>(r) * (K / 32) + ks * 4;
            v = static_cast<uint32_t>(src[0]) | (static_cast<uint32_t>(src[1]) << 8) |
                (static_cast<uint32_t>(src[2]) << 16) | (static_cast<uint32_t>(src[3]) << 24);
        }
        out[i] = v;
    }
}

cudaError_t launch_sf_to_kstep_major(const uint8_t* plain, int S, int K, uint8_t* out, int S4, cudaStream_t s) {
    const long long n = static_cast<long long>(K / 128) * S4;
    if (n <= 0) return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    sf_to_kstep_major_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(plain, S, K, reinterpret_cast<uint32_t*>(out),
                                                                      S4);
    count_launches(1);
    return cudaGetLastError();
}

// out[t, h] = bf16( sum_j y[t*k + j, h] ) (combine_rows in kt_quant_dev.cuh).
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ ids,
                                                      int T, int H, int k, int E, uint16_t* __restrict__ out) {
    griddep_wait();
    griddep_launch_dependents();
    combine_rows<false>(y, ids, T, H, k, E, out, static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x,
                        static_cast<long long>(gridDim.x) * blockDim.x);
}

cudaError_t launch_combine(const uint16_t* y, const int32_t* ids, int T, int H, int k, int E, uint16_t* out,
                           cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const long long n = static_cast<long long>(T) * (H / 8);
    long long blocks = (n + 255) / 256;
    const long long cap = static_cast<long long>(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    const cudaError_t e = launch_chained(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, y, ids,
                                         T, H, k, E, out);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kt
