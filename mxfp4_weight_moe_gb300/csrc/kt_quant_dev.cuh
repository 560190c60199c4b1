// kt_quant_dev.cuh -- MXFP8 quantisation of one bf16 token row by one warp,
// written to the token's k permuted rows (the activation-quantisation step of
// the layer).  Shared by the standalone quantiser kernel and the fused
// single-launch decode kernel.
//
// MXFP8 (e4m3 elements, one e8m0 scale per 32 along H) is the activation
// format of the "MXFP8 activation x MXFP4 weight fused MoE" ("Kimi-K3 SM120
// FlashInfer MXFP4 MoE", Goal).  The shared exponent follows the OCP MX v1.0
// rule floor(log2 amax) - 8 and elements are converted with round-to-
// nearest-even, saturating at +-448.
#pragma once

#include "kt_common.cuh"

namespace kt {

// Passes of 32 blocks (1024 elements) of one token row that one warp-level
// work item of the quantiser takes: a row of H elements is ceil(H / 1024)
// items, so that decode-sized batches spread over many warps.
constexpr int kQuantPass = 32;
__host__ __device__ __forceinline__ int quant_items_per_row(int H) { return ((H >> 5) + kQuantPass - 1) / kQuantPass; }

// Lane l quantises 32-element blocks b0 + l of the passes in [pass0, pass1)
// (64 contiguous input bytes each); the 32 codes + scale byte go to every
// permuted row the token's k slots map to (inv_perm; a slot of -1 is
// skipped).  The codes of a pass of 32 blocks (1 KB per row) are exchanged
// through shuffles once, so that each store instruction writes 512
// contiguous bytes of a row: one 16-byte store per lane at a 32-byte stride
// left half-filled sectors and measured 25-33 % slower on GB300.
// s_dst: kMaxTopK ints of shared memory owned by the warp.  kSharedInv:
// inv_perm is in shared memory (otherwise it was written earlier in the same
// launch, or by an earlier kernel, and is read past L1).
template <bool kSharedInv = false>
__device__ __forceinline__ void quant_token_warp(const uint16_t* __restrict__ hidden, int t, int H, int k,
                                                 const int32_t* __restrict__ inv_perm, uint8_t* __restrict__ a1,
                                                 uint8_t* __restrict__ a1_sf, int S4, int* s_dst, int pass0 = 0,
                                                 int pass1 = 1 << 30) {
    const int lane = threadIdx.x & 31;
    if (lane < k)
        s_dst[lane] = kSharedInv ? inv_perm[static_cast<size_t>(t) * k + lane]
                                 : __ldcg(inv_perm + static_cast<size_t>(t) * k + lane);
    __syncwarp();
    const int nblk_row = H >> 5;
    const int bend = min(nblk_row, pass1 * kQuantPass);
    const int nblk = bend;
    const uint16_t* row = hidden + static_cast<size_t>(t) * H;
    // warp-uniform passes of 32 blocks: lane l converts block b0 + l (if it
    // exists); the next pass's block is loaded before this one is converted
    uint4 nxt[4] = {};
    const int bstart = pass0 * kQuantPass;
    if (bstart + lane < nblk) {
#pragma unroll
        for (int i = 0; i < 4; ++i) nxt[i] = __ldcs(reinterpret_cast<const uint4*>(row + (bstart + lane) * 32) + i);
    }
    for (int b0 = bstart; b0 < nblk; b0 += 32) {
        const int b = b0 + lane;
        const bool mine = b < nblk;
        uint32_t wv[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 q = nxt[i];
            wv[4 * i + 0] = q.x;
            wv[4 * i + 1] = q.y;
            wv[4 * i + 2] = q.z;
            wv[4 * i + 3] = q.w;
        }
        if (b + 32 < nblk) {
#pragma unroll
            for (int i = 0; i < 4; ++i) nxt[i] = __ldcs(reinterpret_cast<const uint4*>(row + (b + 32) * 32) + i);
        }
        float x[32];
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            x[2 * i] = __uint_as_float(wv[i] << 16);
            x[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
            amax = max(amax, __float_as_uint(x[2 * i]) & 0x7FFFFFFFu);
            amax = max(amax, __float_as_uint(x[2 * i + 1]) & 0x7FFFFFFFu);
        }
        const int X = mx_e4m3_block_exponent(amax);
        const float sc = exp2_neg(X);
        uint32_t codes[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = f32x2_to_e4m3x2_satfinite(x[4 * i] * sc, x[4 * i + 1] * sc);
            const uint32_t hi = f32x2_to_e4m3x2_satfinite(x[4 * i + 2] * sc, x[4 * i + 3] * sc);
            codes[i] = lo | (hi << 16);
        }
        const uint32_t sb = static_cast<uint32_t>(X + 127) & 0xFFu;
        const bool full = b0 + 32 <= nblk;   // warp-uniform
        if (full) {
            // lane l stores bytes [16 l, 16 l + 16) and [512 + 16 l, ...) of the pass's
            // 1 KB per row, taken from the owning lanes (l / 2 and 16 + l / 2, half l % 2)
            const int src0 = lane >> 1, src1 = 16 + (lane >> 1);
            const bool hi = lane & 1;
            uint32_t w0[4], w1[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo0 = __shfl_sync(0xffffffffu, codes[i], src0);
                const uint32_t hi0 = __shfl_sync(0xffffffffu, codes[4 + i], src0);
                const uint32_t lo1 = __shfl_sync(0xffffffffu, codes[i], src1);
                const uint32_t hi1 = __shfl_sync(0xffffffffu, codes[4 + i], src1);
                w0[i] = hi ? hi0 : lo0;
                w1[i] = hi ? hi1 : lo1;
            }
            const uint4 st0 = make_uint4(w0[0], w0[1], w0[2], w0[3]);
            const uint4 st1 = make_uint4(w1[0], w1[1], w1[2], w1[3]);
            // the scale bytes of blocks 4j..4j+3 packed into one word by lane 4j
            uint32_t sword = sb;
            sword |= __shfl_down_sync(0xffffffffu, sb, 1) << 8;
            sword |= __shfl_down_sync(0xffffffffu, sb, 2) << 16;
            sword |= __shfl_down_sync(0xffffffffu, sb, 3) << 24;
            for (int j = 0; j < k; ++j) {
                const int p = s_dst[j];
                if (p < 0) continue;
                uint4* rowp = reinterpret_cast<uint4*>(a1 + static_cast<size_t>(p) * H + b0 * 32);
                rowp[lane] = st0;
                rowp[32 + lane] = st1;
                if ((lane & 3) == 0)
                    reinterpret_cast<uint32_t*>(a1_sf)[static_cast<size_t>(b >> 2) * S4 + p] = sword;
            }
        } else if (mine) {
            for (int j = 0; j < k; ++j) {
                const int p = s_dst[j];
                if (p < 0) continue;
                uint4* dst = reinterpret_cast<uint4*>(a1 + static_cast<size_t>(p) * H + b * 32);
                dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
                dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
                a1_sf[((static_cast<size_t>(b >> 2) * S4 + p) << 2) + (b & 3)] = static_cast<uint8_t>(sb);
            }
        }
    }
}

// The top-k combine: out[t, h] = bf16( sum_j y[t*k + j, h] ) over the slots
// with a valid id, summed in fp32 in slot order (y rows were already
// multiplied by topk_w).  Work item idx = (token, 8 columns), items first,
// first + step, ...  kCoherent: y and ids were written earlier in the same
// launch (read through L2).
template <bool kCoherent>
__device__ __forceinline__ void combine_rows(const uint16_t* __restrict__ y, const int32_t* __restrict__ ids, int T,
                                             int H, int k, int E, uint16_t* __restrict__ out, long long first,
                                             long long step) {
    const int h8n = H >> 3;
    const long long n = static_cast<long long>(T) * h8n;
    for (long long idx = first; idx < n; idx += step) {
        const int t = static_cast<int>(idx / h8n);
        const int h8 = static_cast<int>(idx % h8n);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        // slots in order (the sum order is fixed); loads of four slots are in flight together
        for (int j0 = 0; j0 < k; j0 += 4) {
            uint4 q[4];
            bool use[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u;
                int e = -1;
                if (j < k) e = kCoherent ? __ldcg(ids + static_cast<size_t>(t) * k + j)
                                         : __ldg(ids + static_cast<size_t>(t) * k + j);
                use[u] = e >= 0 && e < E;
                const uint4* src = reinterpret_cast<const uint4*>(y + (static_cast<size_t>(t) * k + j) * H + h8 * 8);
                q[u] = use[u] ? (kCoherent ? __ldcg(src) : __ldcs(src)) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (!use[u]) continue;
                const uint32_t wv[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] += __uint_as_float(wv[i] << 16);
                    acc[2 * i + 1] += __uint_as_float(wv[i] & 0xFFFF0000u);
                }
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
            o[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        *reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + h8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace kt
