// kt_gemm_mx.cu -- persistent grouped GEMM on the 5th-generation tensor
// cores: D = W[e] (MXFP4, e2m1 + e8m0/32) x A[rows of expert e] (MXFP8,
// e4m3 + e8m0/32), fp32 accumulators in tensor memory, with three fused
// epilogues (raw fp32 store; FC1 SwiGLU + MXFP8 requant; FC2 topk-weighted
// store in slot order).
//
// This is the "MXFP8 activation x MXFP4 weight fused MoE" GEMM of "Kimi-K3
// SM120 FlashInfer MXFP4 MoE" (Goal), with the gated FC1 of twice the FC2
// inter size (on-device evidence) and the SwiGLU gate (Phase 0 audit,
// item 4), built for sm_103a rather than the SM120 CUTLASS or Ampere Marlin
// kernels the pages discuss.
//
// Tile = 128 weight rows (MMA M) x up to 256 token rows of one expert
// (MMA N, a multiple of 16), K streamed in steps of 128.  Weights sit on the
// M side ("swap AB") so that experts with few tokens waste little MMA work.
// For FC1 the 128 weight rows are 64 gate rows and the matching 64 up rows,
// so SwiGLU needs only the accumulator tile.
//
// Warp roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0     producer: TMA loads of the fp4 weight tile (unpacked by the
//              16U4_ALIGN16B tensor map type: each 16-byte shared-memory
//              chunk holds 8 bytes = 16 packed values, then an 8-byte gap the
//              copy leaves untouched) and of the e4m3 token tile, 4-byte
//              cp.async gathers of both scale-factor tiles into the 128x4
//              block layout
//   warp 1     one thread issues tcgen05.cp (scales -> tensor memory) and
//              tcgen05.mma (4 per K step), commits to the pipeline barriers
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//              32*(w%4)..+31), fused math, global stores
// Every barrier wait has a deadline; on expiry the role records itself in
// the device error word and the CTA winds down and frees its tensor memory.
#include <cudaTypedefs.h>

#include <mutex>

#include "kt_common.cuh"
#include "kt_internal.h"

namespace kt {

constexpr int kStages = 4;
constexpr int kBK = 128;                     // K elements per pipeline stage
constexpr int kSmemA = 128 * kBK;            // 16 KB: 128 rows x 128 bytes (fp4 unpacked)
// The unpacking TMA counts the packed global bytes as transaction bytes
// (half the shared-memory footprint): 128 rows x 64 bytes per stage.
constexpr int kTxA = 128 * kBK / 2;
constexpr int kSmemB = kTileTokens * kBK;    // 32 KB: 256 rows x 128 bytes
constexpr int kOffSFA = kSmemA + kSmemB;     // 512 B scale block for the 128 weight rows
constexpr int kOffSFB = kOffSFA + 512;       // 2 x 512 B scale blocks for 256 token rows
constexpr int kStageBytes = 51200;           // rounded up to a 1 KB multiple
constexpr int kEpiBytes = 32 * 64 * 4 + 2 * 32 * 32;   // SwiGLU exchange + byte transpose
constexpr int kBarBytes = 256;
constexpr int kSmemTotal = 1024 + kStages * kStageBytes + kEpiBytes + kBarBytes;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSF = 256;            // scale columns: 16 per stage after the accumulator
static_assert(kOffSFB + 1024 <= kStageBytes, "stage layout");
static_assert(kSmemTotal <= 232448, "shared memory budget");

struct TileInfo {
    int e, f, r0, nvalid, nmma;
};

struct KParams {
    const int32_t* expert_offsets;
    const int32_t* chunk_prefix;
    int E, K, rows_w, I, S, n_ftiles, H;
    const uint8_t* w_sf;
    const uint8_t* act_sf;
    uint8_t* a2;
    uint8_t* a2_sf;
    uint16_t* y;
    const int32_t* perm;
    const float* topk_w;
    float* raw_out;
    int* err;
    uint64_t wait_limit_ns;
    int debug_flags;
};

// Tile u -> (expert, feature tile, token chunk); token chunks of one
// (expert, feature tile) are adjacent so concurrent CTAs share weight tiles
// through L2.  chunk c of an expert with `cnt` rows split into nc chunks covers
// rows [c*cnt/nc, (c+1)*cnt/nc).
__device__ __forceinline__ void decode_tile(const KParams& p, int u, TileInfo& ti) {
    const int v = u / p.n_ftiles;
    int lo = 1, hi = p.E;                   // first e' with chunk_prefix[e'] > v
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.chunk_prefix + mid) > v) hi = mid;
        else lo = mid + 1;
    }
    const int e = lo - 1;
    const int c0 = __ldg(p.chunk_prefix + e);
    const int nc = __ldg(p.chunk_prefix + e + 1) - c0;
    const int local = u - p.n_ftiles * c0;
    ti.e = e;
    ti.f = local / nc;
    const int c = local - ti.f * nc;
    const int off = __ldg(p.expert_offsets + e);
    const int cnt = __ldg(p.expert_offsets + e + 1) - off;
    const int a = static_cast<int>(static_cast<long long>(c) * cnt / nc);
    const int b = static_cast<int>(static_cast<long long>(c + 1) * cnt / nc);
    ti.r0 = off + a;
    ti.nvalid = b - a;
    ti.nmma = (ti.nvalid + 15) & ~15;
}

template <int MODE>
__device__ __forceinline__ void weight_rows(const KParams& p, const TileInfo& ti, int& rowA0, int& rowA1) {
    if (MODE == static_cast<int>(GemmEpilogue::SwiGLU)) {
        rowA0 = ti.e * p.rows_w + ti.f * 64;           // gate rows
        rowA1 = ti.e * p.rows_w + p.I + ti.f * 64;     // matching up rows
    } else {
        rowA0 = ti.e * p.rows_w + ti.f * 128;
        rowA1 = rowA0 + 64;
    }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_act,
                   const __grid_constant__ KParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t s_base = smem_u32(smem);
    uint8_t* epi = smem + kStages * kStageBytes;
    uint8_t* bars = epi + kEpiBytes;
    const uint32_t bar_base = smem_u32(bars);
    // barrier addresses: full[4] empty[4] acc_full acc_empty drain
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (kStages + s); };
    const uint32_t acc_full = bar_base + 8u * (2 * kStages);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t drain_bar = acc_full + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 128);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 136);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1 + 32);   // producer's expect_tx arrive + 32 cp.async arrivals
            mbar_init(empty_bar(s), 1);       // tcgen05.commit
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);              // one arrive per epilogue warp
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tc_alloc(smem_u32(tmem_slot), kTmemCols);
        tc_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_w);
        tma_prefetch_map(&map_act);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int total = p.n_ftiles * __ldg(p.chunk_prefix + p.E);
    const int nk = p.K / kBK;
    const int ksf = p.K / 32;   // scale bytes per row

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        const uint64_t pol_w = l2_policy_evict_first();
        const uint64_t pol_a = l2_policy_evict_last();
        for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
            TileInfo ti;
            decode_tile(p, u, ti);
            int rowA0, rowA1;
            weight_rows<MODE>(p, ti, rowA0, rowA1);
            const uint32_t tx = static_cast<uint32_t>(kTxA + ti.nmma * kBK);
            const int nsfb = (ti.nmma + 31) >> 5;
            for (int kb = 0; kb < nk; ++kb) {
                ok = __all_sync(0xffffffffu, mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit_ns));
                if (!ok) break;
                if ((p.debug_flags & KT_DEBUG_WITHHOLD_STAGE) && u == static_cast<int>(blockIdx.x) && kb == 0) {
                    // test hook: leave this stage unfilled and unsignalled
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
                fence_proxy_async_smem();
                const uint32_t sA = s_base + stage * kStageBytes;
                const uint32_t sB = sA + kSmemA;
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(stage), tx);
                    tma_load_2d_hint(sA, &map_w, full_bar(stage), kb * kBK, rowA0, pol_w);
                    tma_load_2d_hint(sA + kSmemA / 2, &map_w, full_bar(stage), kb * kBK, rowA1, pol_w);
                    for (int i = 0; i < ti.nmma / 16; ++i)
                        tma_load_2d_hint(sB + i * 16 * kBK, &map_act, full_bar(stage), kb * kBK, ti.r0 + 16 * i,
                                         pol_a);
                }
                // weight scales: row r of the tile -> byte (r%32)*16 + (r/32)*4 of the 512-byte block
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane + 32 * i;
                    const int grow = (r < 64) ? rowA0 + r : rowA1 + (r - 64);
                    cp_async_4(sA + kOffSFA + lane * 16 + i * 4, p.w_sf + static_cast<size_t>(grow) * ksf + kb * 4, 4);
                }
                // token scales: rows beyond the tile's valid rows are zero-filled
                for (int i = 0; i < nsfb; ++i) {
                    const int t = lane + 32 * i;
                    const bool valid = t < ti.nvalid;
                    const uint8_t* src = valid ? p.act_sf + static_cast<size_t>(ti.r0 + t) * ksf + kb * 4 : p.act_sf;
                    cp_async_4(sA + kOffSFB + (i >> 2) * 512 + lane * 16 + (i & 3) * 4, src, valid ? 4u : 0u);
                }
                cp_async_arrive_noinc(full_bar(stage));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            if (lane == 0) set_error(p.err, KT_DEVERR_TIMEOUT_LOAD);
            *abort_flag = 1;
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, issued = false;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                TileInfo ti;
                decode_tile(p, u, ti);
                issued = true;
                ok = mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag, p.wait_limit_ns);
                if (!ok) break;
                tc_fence_after();
                for (int kb = 0; kb < nk; ++kb) {
                    ok = mbar_wait(full_bar(stage), phase, abort_flag, p.wait_limit_ns);
                    if (!ok) break;
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t sA = s_base + stage * kStageBytes;
                    const uint32_t sB = sA + kSmemA;
                    const uint32_t t_sfa = tmem + kTmemSF + stage * 16;
                    const uint32_t t_sfb = t_sfa + 4;
                    tc_cp_32x128b_warpx4(t_sfa, sdesc_sf_block(sA + kOffSFA));
                    tc_cp_32x128b_warpx4(t_sfb, sdesc_sf_block(sA + kOffSFB));
                    if (ti.nmma > 128) tc_cp_32x128b_warpx4(t_sfb + 4, sdesc_sf_block(sA + kOffSFB + 512));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        tc_mma_mxf8f6f4(tmem, sdesc_k_sw128(sA + 32 * j), sdesc_k_sw128(sB + 32 * j),
                                        idesc_mx_e2m1_e4m3(ti.nmma, static_cast<uint32_t>(j)), t_sfa, t_sfb,
                                        (kb | j) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty_bar(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(acc_full);
                acc_phase ^= 1u;
            }
            if (!ok) {
                set_error(p.err, KT_DEVERR_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            // every tcgen05 operation issued above completes before teardown
            if (issued) {
                tc_commit(drain_bar);
                mbar_wait(drain_bar, 0, abort_flag, p.wait_limit_ns);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                        // tensor-memory lane quadrant
        const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16);
        uint32_t acc_phase = 0;
        bool ok = true;
        float* xch = reinterpret_cast<float*>(epi);            // [32 tokens][64 features]
        uint8_t* bt = epi + 32 * 64 * 4;                        // [2][32 tokens][32 features]
        for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
            TileInfo ti;
            decode_tile(p, u, ti);
            ok = __all_sync(0xffffffffu, mbar_wait(acc_full, acc_phase, abort_flag, p.wait_limit_ns));
            if (!ok) break;
            tc_fence_after();
            for (int c0 = 0; c0 < ti.nvalid; c0 += 32) {
                uint32_t v[32];
                tc_ld_32x32b_x32(trow + static_cast<uint32_t>(c0), v);
                tc_wait_ld();
                if (MODE == static_cast<int>(GemmEpilogue::Raw)) {
                    const int n = ti.f * 128 + q * 32 + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (c0 + j < ti.nvalid)
                            p.raw_out[static_cast<size_t>(ti.r0 + c0 + j) * p.rows_w + n] = __uint_as_float(v[j]);
                    }
                } else if (MODE == static_cast<int>(GemmEpilogue::Combine)) {
                    const int h = ti.f * 128 + q * 32 + lane;
                    int slot = 0;
                    float wt = 0.f;
                    if (c0 + lane < ti.nvalid) {
                        slot = __ldg(p.perm + ti.r0 + c0 + lane);
                        wt = __ldg(p.topk_w + slot);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int s = __shfl_sync(0xffffffffu, slot, j);
                        const float wj = __shfl_sync(0xffffffffu, wt, j);
                        if (c0 + j < ti.nvalid) {
                            const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[j]) * wj);
                            p.y[static_cast<size_t>(s) * p.H + h] = *reinterpret_cast<const uint16_t*>(&b);
                        }
                    }
                } else {
                    // SwiGLU: quadrants 0,1 hold gate rows, 2,3 the matching up rows.
                    if (q < 2) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float g = __uint_as_float(v[j]);
                            xch[j * 64 + q * 32 + lane] = g / (1.0f + __expf(-g));
                        }
                    }
                    named_bar_sync(1, 128);
                    if (q >= 2) {
                        uint8_t* my_bt = bt + (q - 2) * 1024;
                        uint8_t my_scale = 0;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float hv = xch[j * 64 + (q - 2) * 32 + lane] * __uint_as_float(v[j]);
                            const uint32_t am = __reduce_max_sync(0xffffffffu, __float_as_uint(hv) & 0x7FFFFFFFu);
                            const int X = mx_e4m3_block_exponent(am);
                            my_bt[j * 32 + lane] = f32_to_e4m3_satfinite(hv * exp2_neg(X));
                            if (lane == j) my_scale = static_cast<uint8_t>(X + 127);
                        }
                        __syncwarp();
                        if (c0 + lane < ti.nvalid) {
                            const size_t row = static_cast<size_t>(ti.r0 + c0 + lane);
                            const int col = ti.f * 64 + (q - 2) * 32;
                            const uint4* srcv = reinterpret_cast<const uint4*>(my_bt + lane * 32);
                            uint4* dst = reinterpret_cast<uint4*>(p.a2 + row * p.I + col);
                            dst[0] = srcv[0];
                            dst[1] = srcv[1];
                            p.a2_sf[row * (p.I / 32) + col / 32] = my_scale;
                        }
                        __syncwarp();
                    }
                    named_bar_sync(2, 128);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            acc_phase ^= 1u;
        }
        if (!ok) {
            if (lane == 0) set_error(p.err, KT_DEVERR_TIMEOUT_EPI);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) __nanosleep(1000000);   // let any copy still in flight land before teardown
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// fp4x2 [rows, K/2] bytes, read as K 4-bit elements per row; each 64-row x
// 128-element box lands in shared memory unpacked to one byte per element
// (16U4_ALIGN16B: 8 data bytes then an 8-byte gap), 128-byte swizzled.
static CUresult make_map_fp4(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {K / 2};
    cuuint32_t box[2] = {128, 64};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// e4m3 [rows, K] bytes; 16-row x 128-byte boxes, 128-byte swizzled.
static CUresult make_map_u8(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {K};
    cuuint32_t box[2] = {128, 16};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int MODE>
static cudaError_t launch_mode(const CUtensorMap& mw, const CUtensorMap& ma, const KParams& kp, cudaStream_t s) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemTotal);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    mx_gemm_kernel<MODE><<<sm_count(), kThreads, kSmemTotal, s>>>(mw, ma, kp);
    count_launches(1);
    return cudaGetLastError();
}

kt_status launch_gemm(const GemmArgs& a, cudaStream_t s) {
    if (a.S <= 0) return KT_OK;
    alignas(64) CUtensorMap mw;
    alignas(64) CUtensorMap ma;
    const uint64_t wrows = static_cast<uint64_t>(a.E) * a.rows_w;
    if (make_map_fp4(&mw, a.w, a.K, wrows) != CUDA_SUCCESS) return KT_ERR_CUDA;
    if (make_map_u8(&ma, a.act, a.K, a.S) != CUDA_SUCCESS) return KT_ERR_CUDA;
    KParams kp{};
    kp.expert_offsets = a.expert_offsets;
    kp.chunk_prefix = a.chunk_prefix;
    kp.E = a.E;
    kp.K = a.K;
    kp.rows_w = a.rows_w;
    kp.I = a.I;
    kp.S = a.S;
    kp.H = a.H;
    kp.n_ftiles = (a.mode == GemmEpilogue::SwiGLU) ? a.I / 64 : a.rows_w / 128;
    kp.w_sf = a.w_sf;
    kp.act_sf = a.act_sf;
    kp.a2 = a.a2;
    kp.a2_sf = a.a2_sf;
    kp.y = a.y;
    kp.perm = a.perm;
    kp.topk_w = a.topk_w;
    kp.raw_out = a.raw_out;
    kp.err = a.err;
    const DebugSettings dbg = debug_settings();
    kp.wait_limit_ns = dbg.wait_limit_ns;
    kp.debug_flags = dbg.flags;
    cudaError_t e;
    switch (a.mode) {
        case GemmEpilogue::Raw: e = launch_mode<0>(mw, ma, kp, s); break;
        case GemmEpilogue::SwiGLU: e = launch_mode<1>(mw, ma, kp, s); break;
        default: e = launch_mode<2>(mw, ma, kp, s); break;
    }
    return cuda_status(e);
}

}  // namespace kt
