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
// Tile = 128 weight rows (MMA M) x up to kTileTokens token rows of one expert
// (MMA N, a multiple of 16), K streamed in steps of 128.  Weights sit on the
// M side ("swap AB") so that experts with few tokens waste little MMA work.
// For FC1 the 128 weight rows are 64 gate rows and the matching 64 up rows,
// so SwiGLU needs only the accumulator tile.
//
// Warp roles (224 threads, one CTA per SM, persistent over tiles):
//   warp 0     TMA producer: one lane issues, per K step, one TMA for the
//              whole fp4 weight tile (for FC1 a 3-D view of w13 puts the 64
//              gate rows and the 64 matching up rows in one box; the
//              16U4_ALIGN16B type unpacks it to one byte per element in
//              shared memory: 8 data bytes then an 8-byte gap the copy leaves
//              untouched, and counts the packed bytes as transaction bytes)
//              and at most four boxes (128/64/32/16 rows) for the e4m3 token
//              tile.
//   warp 1     one thread issues tcgen05.cp (scales -> tensor memory) and
//              tcgen05.mma (4 per K step) and commits to the barriers.
//   warp 2     scale warp: per 4 K steps it TMA-loads the weight scales
//              (16-byte rows of the plain [rows, K/32] layout) and the token
//              scales (the K-step-major u32 layout the quantisers write) into
//              a staging buffer, builds the 128x4 scale blocks the MMA reads,
//              and prefetches the weight bytes of a later group of K steps
//              into L2.
//   warps 3-6  epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//              32*(w%4)..+31), fused math, global stores.  Two accumulator
//              buffers let one tile's epilogue overlap the next main loop.
// Every barrier wait has a deadline; on expiry the role records itself in
// the device error word and the CTA winds down and frees its tensor memory.
#include <cudaTypedefs.h>

#include <mutex>

#include "kt_common.cuh"
#include "kt_internal.h"

namespace kt {

constexpr int kStages = 4;
constexpr int kBK = 128;                      // K elements per pipeline stage
constexpr int kSmemA = 128 * kBK;             // 16 KB: 128 rows x 128 bytes (fp4 unpacked)
constexpr int kTxA = 128 * kBK / 2;           // the unpacking TMA counts packed bytes
constexpr int kSmemB = kTileTokens * kBK;     // 28 KB: up to 224 token rows x 128 bytes
constexpr int kStageBytes = kSmemA + kSmemB;  // 44 KB
constexpr int kGroup = 4;                     // K steps per scale group
constexpr int kSfStep = 512 + 1024;           // per K step: weight block + up to 2 token blocks
constexpr int kSfBytes = kGroup * kSfStep;    // one scale-block buffer (two of them)
constexpr int kStgSFA = 128 * 16;             // staging: 128 weight rows x 16 scale bytes
constexpr int kStgSFB = kGroup * 256 * 4;     // staging: 4 K steps x 256 token rows x u32
constexpr int kStgBytes = kStgSFA + kStgSFB;  // one staging buffer (two of them)
constexpr int kEpiBytes = 10240;              // FC1 exchange + transposes / FC2 transpose
constexpr int kBarBytes = 256;
constexpr int kSmemTotal = 1024 + kStages * kStageBytes + 2 * kSfBytes + 2 * kStgBytes + kEpiBytes + kBarBytes;
constexpr int kThreads = 224;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kTileTokens;    // accumulator buffer b at column b * kAccCols
constexpr uint32_t kTmemSF = 2 * kAccCols;    // scale columns: 12 per stage after both accumulators
constexpr int kPrefetchGroups = 2;            // scale-warp L2 prefetch distance, in groups of K steps
static_assert(kStageBytes % 1024 == 0, "stage alignment");
static_assert(kSmemTotal <= 232448, "shared memory budget");
static_assert(kTmemSF + 12 * kStages <= kTmemCols, "tensor memory budget");
static_assert(kTileTokens % 32 == 0 && kTileTokens + 3 <= 256 && kTileTokens <= 240, "token tile");

struct TileInfo {
    int e, f, r0, nvalid, nmma;
};

struct KParams {
    const int32_t* expert_offsets;
    const int32_t* chunk_prefix;
    int E, K, rows_w, I, S, S4, n_ftiles, H;
    const uint8_t* w_sf;      // plain [E * rows_w, K/32] (read directly when K % 512 != 0)
    int sfa_tma;              // 1: weight scales staged by TMA; 0: 4-byte cp.async gathers
    uint8_t* a2;
    uint8_t* a2_sf;           // K-step-major u32 [I/128][S4]
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

// Coordinates of a tile's weight rows: for FC1 (3-D view [2E][I][K] of w13)
// (y, z) = (64 f, 2 e) selects the 64 gate rows and the 64 matching up rows;
// otherwise (2-D view [E * rows_w][K]) y = e * rows_w + 128 f.
template <int MODE>
__device__ __forceinline__ void weight_coords(const KParams& p, const TileInfo& ti, int& y, int& z) {
    if (MODE == static_cast<int>(GemmEpilogue::SwiGLU)) {
        y = ti.f * 64;
        z = 2 * ti.e;
    } else {
        y = ti.e * p.rows_w + ti.f * 128;
        z = 0;
    }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Load (or prefetch) a weight-side box: 3-D for FC1, 2-D otherwise.
template <int MODE>
__device__ __forceinline__ void load_weight_box(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                int z) {
    if (MODE == static_cast<int>(GemmEpilogue::SwiGLU)) tma_load_3d(dst, map, bar, x, y, z);
    else tma_load_2d(dst, map, bar, x, y);
}
template <int MODE>
__device__ __forceinline__ void prefetch_weight_box(const CUtensorMap* map, int x, int y, int z) {
    if (MODE == static_cast<int>(GemmEpilogue::SwiGLU)) tma_prefetch_l2_3d(map, x, y, z);
    else tma_prefetch_l2_2d(map, x, y);
}

// Walks the (tile, group of kGroup K steps) sequence of one CTA.
template <int MODE>
struct GroupCursor {
    int u, g;          // tile id and group index within the tile
    TileInfo ti;
    int wy, wz;
    bool valid;
    __device__ __forceinline__ void start(const KParams& p, int total) {
        u = blockIdx.x;
        g = 0;
        load(p, total);
    }
    __device__ __forceinline__ void load(const KParams& p, int total) {
        valid = u < total;
        if (valid) {
            decode_tile(p, u, ti);
            weight_coords<MODE>(p, ti, wy, wz);
        }
    }
    __device__ __forceinline__ void advance(const KParams& p, int total, int ngroups) {
        if (++g == ngroups) {
            g = 0;
            u += gridDim.x;
            load(p, total);
        }
    }
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_b16,
                   const __grid_constant__ CUtensorMap map_b32, const __grid_constant__ CUtensorMap map_b64,
                   const __grid_constant__ CUtensorMap map_b128, const __grid_constant__ CUtensorMap map_wpf,
                   const __grid_constant__ CUtensorMap map_wsf, const __grid_constant__ CUtensorMap map_asf,
                   const __grid_constant__ KParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t s_base = smem_u32(smem);
    uint8_t* sfbuf = smem + kStages * kStageBytes;        // two scale-block buffers
    uint8_t* stg = sfbuf + 2 * kSfBytes;                   // two staging buffers
    uint8_t* epi = stg + 2 * kStgBytes;
    uint8_t* bars = epi + kEpiBytes;
    const uint32_t bar_base = smem_u32(bars);
    // barriers: full[4] empty[4] sf_full[2] sf_empty[2] stg[2] acc_full[2] acc_empty[2] drain
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (4 + s); };
    auto sf_full = [&](int b) { return bar_base + 8u * (8 + b); };
    auto sf_empty = [&](int b) { return bar_base + 8u * (10 + b); };
    auto stg_bar = [&](int b) { return bar_base + 8u * (12 + b); };
    auto acc_full = [&](int b) { return bar_base + 8u * (14 + b); };
    auto acc_empty = [&](int b) { return bar_base + 8u * (16 + b); };
    const uint32_t drain_bar = bar_base + 8u * 18;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 192);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 200);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);      // producer's arrive.expect_tx
            mbar_init(empty_bar(s), 1);     // tcgen05.commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sf_full(b), 32);      // one arrive per scale-warp lane
            mbar_init(sf_empty(b), 1);      // tcgen05.commit
            mbar_init(stg_bar(b), 1);       // scale warp's arrive.expect_tx
            mbar_init(acc_full(b), 1);      // tcgen05.commit
            mbar_init(acc_empty(b), 4);     // one arrive per epilogue warp
        }
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
        tma_prefetch_map(&map_b16);
        tma_prefetch_map(&map_b32);
        tma_prefetch_map(&map_b64);
        tma_prefetch_map(&map_b128);
    }
    if (warp == 2 && lane == 0) {
        tma_prefetch_map(&map_wpf);
        tma_prefetch_map(&map_asf);
        if (p.sfa_tma) tma_prefetch_map(&map_wsf);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int total = p.n_ftiles * __ldg(p.chunk_prefix + p.E);
    const int nk = p.K / kBK;
    const int ngroups = (nk + kGroup - 1) / kGroup;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_a = l2_policy_evict_last();
            const CUtensorMap* bmaps[4] = {&map_b16, &map_b32, &map_b64, &map_b128};
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                TileInfo ti;
                decode_tile(p, u, ti);
                int wy, wz;
                weight_coords<MODE>(p, ti, wy, wz);
                const uint32_t tx = static_cast<uint32_t>(kTxA + ti.nmma * kBK);
                for (int kb = 0; kb < nk; ++kb) {
                    ok = mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit_ns);
                    if (!ok) break;
                    const bool withhold = (p.debug_flags & KT_DEBUG_WITHHOLD_STAGE) &&
                                          u == static_cast<int>(blockIdx.x) && kb == 0;
                    if (!withhold) {   // test hook: a withheld stage is neither loaded nor signalled
                        const uint32_t sA = s_base + stage * kStageBytes;
                        const uint32_t sB = sA + kSmemA;
                        mbar_arrive_expect_tx(full_bar(stage), tx);
                        if (MODE == static_cast<int>(GemmEpilogue::SwiGLU)) {
                            asm volatile(
                                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(sA),
                                "l"(reinterpret_cast<uint64_t>(&map_w)), "r"(full_bar(stage)), "r"(kb * kBK),
                                "r"(wy), "r"(wz), "l"(pol_w)
                                : "memory");
                        } else {
                            tma_load_2d_hint(sA, &map_w, full_bar(stage), kb * kBK, wy, pol_w);
                        }
                        int rdone = 0;
#pragma unroll
                        for (int bi = 3; bi >= 0; --bi) {
                            const int rows = 16 << bi;
                            if (ti.nmma - rdone >= rows) {
                                tma_load_2d_hint(sB + rdone * kBK, bmaps[bi], full_bar(stage), kb * kBK,
                                                 ti.r0 + rdone, pol_a);
                                rdone += rows;
                            }
                        }
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                set_error(p.err, KT_DEVERR_TIMEOUT_LOAD);
                *abort_flag = 1;
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ scale warp
        uint32_t stg_ph[2] = {0u, 0u}, sfe_ph[2] = {0u, 0u};
        bool ok = true;
        const uint32_t stg_tx = static_cast<uint32_t>(kStgSFB + (p.sfa_tma ? kStgSFA : 0));
        const int ksf = p.K / 32;
        GroupCursor<MODE> cur, nxt, pf;
        cur.start(p, total);
        nxt = cur;
        pf = cur;
        auto issue_staging = [&](const GroupCursor<MODE>& c, int buf) {
            if (lane == 0 && c.valid) {
                const uint32_t dst = smem_u32(stg + buf * kStgBytes);
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(stg_bar(buf), stg_tx);
                if (p.sfa_tma) load_weight_box<MODE>(dst, &map_wsf, stg_bar(buf), c.g * 16, c.wy, c.wz);
                tma_load_2d(dst + kStgSFA, &map_asf, stg_bar(buf), c.ti.r0 & ~3, c.g * kGroup);
            }
        };
        auto prefetch_group = [&](const GroupCursor<MODE>& c) {
            if (lane == 0 && c.valid) prefetch_weight_box<MODE>(&map_wpf, c.g * (kGroup * kBK / 2), c.wy, c.wz);
        };
        for (int i = 0; i < kPrefetchGroups; ++i) {
            prefetch_group(pf);
            pf.advance(p, total, ngroups);
        }
        issue_staging(cur, 0);
        int buf = 0;
        while (cur.valid && ok) {
            nxt = cur;
            nxt.advance(p, total, ngroups);
            __syncwarp();                      // every lane is done with the buffer refilled next
            issue_staging(nxt, buf ^ 1);
            prefetch_group(pf);
            pf.advance(p, total, ngroups);
            ok = __all_sync(0xffffffffu, mbar_wait(stg_bar(buf), stg_ph[buf], abort_flag, p.wait_limit_ns));
            if (!ok) break;
            ok = __all_sync(0xffffffffu, mbar_wait(sf_empty(buf), sfe_ph[buf] ^ 1u, abort_flag, p.wait_limit_ns));
            if (!ok) break;
            const TileInfo& ti = cur.ti;
            const uint8_t* sb = stg + buf * kStgBytes;
            uint8_t* sfo = sfbuf + buf * kSfBytes;
            const int kb0 = cur.g * kGroup;
            const int nkk = min(kGroup, nk - kb0);
            const int shift = ti.r0 & 3;
            const int natoms = ti.nmma > 128 ? 2 : 1;
            for (int kk = 0; kk < nkk; ++kk) {
                uint8_t* blk = sfo + kk * kSfStep;
                // weight scales: tile row r -> byte (r%32)*16 + (r/32)*4 of the 512-byte block
                if (p.sfa_tma) {
                    uint32_t w4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        w4[i] = *reinterpret_cast<const uint32_t*>(sb + (lane + 32 * i) * 16 + kk * 4);
                    *reinterpret_cast<uint4*>(blk + lane * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = lane + 32 * i;
                        size_t grow;
                        if (MODE == static_cast<int>(GemmEpilogue::SwiGLU))
                            grow = static_cast<size_t>(ti.e) * p.rows_w + (r < 64 ? 0 : p.I) + ti.f * 64 + (r & 63);
                        else
                            grow = static_cast<size_t>(ti.e) * p.rows_w + ti.f * 128 + r;
                        cp_async_4(smem_u32(blk + lane * 16 + i * 4), p.w_sf + grow * ksf + (kb0 + kk) * 4, 4);
                    }
                }
                // token scales from the K-step-major staging rows (shifted by r0 % 4)
                const uint32_t* arow = reinterpret_cast<const uint32_t*>(sb + kStgSFA) + kk * 256 + shift;
                for (int a = 0; a < natoms; ++a) {
                    uint32_t t4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int t = 128 * a + lane + 32 * i;
                        t4[i] = (t < ti.nvalid) ? arow[t] : 0u;
                    }
                    *reinterpret_cast<uint4*>(blk + 512 + a * 512 + lane * 16) =
                        make_uint4(t4[0], t4[1], t4[2], t4[3]);
                }
            }
            fence_proxy_async_smem();
            if (p.sfa_tma) mbar_arrive(sf_full(buf));
            else cp_async_arrive_noinc(sf_full(buf));
            stg_ph[buf] ^= 1u;
            sfe_ph[buf] ^= 1u;
            buf ^= 1;
            cur = nxt;
        }
        if (!ok) {
            if (lane == 0) set_error(p.err, KT_DEVERR_TIMEOUT_LOAD);
            *abort_flag = 1;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, sb = 0, it = 0;
            uint32_t phase = 0;
            uint32_t acc_ph[2] = {0u, 0u}, sf_ph[2] = {0u, 0u};
            bool ok = true, issued = false;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++it) {
                TileInfo ti;
                decode_tile(p, u, ti);
                const int ab = it & 1;
                issued = true;
                ok = mbar_wait(acc_empty(ab), acc_ph[ab] ^ 1u, abort_flag, p.wait_limit_ns);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + ab * kAccCols;
                const uint32_t idesc0 = idesc_mx_e2m1_e4m3(ti.nmma, 0);
                for (int kb = 0; kb < nk; ++kb) {
                    const int kk = kb & (kGroup - 1);
                    if (kk == 0) {
                        ok = mbar_wait(sf_full(sb), sf_ph[sb], abort_flag, p.wait_limit_ns);
                        if (!ok) break;
                        fence_proxy_async_smem();   // scale blocks were written through the generic proxy
                    }
                    ok = mbar_wait(full_bar(stage), phase, abort_flag, p.wait_limit_ns);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sA = s_base + stage * kStageBytes;
                    const uint32_t sB = sA + kSmemA;
                    const uint32_t sF = smem_u32(sfbuf + sb * kSfBytes + kk * kSfStep);
                    const uint32_t t_sfa = tmem + kTmemSF + stage * 12;
                    const uint32_t t_sfb = t_sfa + 4;
                    tc_cp_32x128b_warpx4(t_sfa, sdesc_sf_block(sF));
                    tc_cp_32x128b_warpx4(t_sfb, sdesc_sf_block(sF + 512));
                    if (ti.nmma > 128) tc_cp_32x128b_warpx4(t_sfb + 4, sdesc_sf_block(sF + 1024));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t idesc =
                            idesc0 | (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
                        tc_mma_mxf8f6f4(d_tmem, sdesc_k_sw128(sA + 32 * j), sdesc_k_sw128(sB + 32 * j), idesc, t_sfa,
                                        t_sfb, (kb | j) != 0 ? 1u : 0u);
                    }
                    tc_commit(empty_bar(stage));
                    if (kk == kGroup - 1 || kb == nk - 1) {
                        tc_commit(sf_empty(sb));
                        sf_ph[sb] ^= 1u;
                        sb ^= 1;
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(acc_full(ab));
                acc_ph[ab] ^= 1u;
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
        // ------------------------------------------------------------ epilogue (warps 3-6)
        const int q = warp & 3;                        // tensor-memory lane quadrant
        uint32_t acc_ph[2] = {0u, 0u};
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++it) {
            TileInfo ti;
            decode_tile(p, u, ti);
            const int ab = it & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(acc_full(ab), acc_ph[ab], abort_flag, p.wait_limit_ns));
            if (!ok) break;
            tc_fence_after();
            const uint32_t trow = tmem + ab * kAccCols + (static_cast<uint32_t>(32 * q) << 16);
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
                    // weight, round to bf16 and transpose through shared memory so each
                    // lane writes 64 contiguous bytes of one token's output row
                    uint8_t* tb = epi + q * 2560;   // [32 tokens][80 bytes]
                    int slot = 0;
                    float wt = 0.f;
                    if (c0 + lane < ti.nvalid) {
                        slot = __ldg(p.perm + ti.r0 + c0 + lane);
                        wt = __ldg(p.topk_w + slot);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float wj = __shfl_sync(0xffffffffu, wt, j);
                        const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[j]) * wj);
                        *reinterpret_cast<__nv_bfloat16*>(tb + j * 80 + lane * 2) = b;
                    }
                    __syncwarp();
                    if (c0 + lane < ti.nvalid) {
                        const uint4* src = reinterpret_cast<const uint4*>(tb + lane * 80);
                        uint4* dst =
                            reinterpret_cast<uint4*>(p.y + static_cast<size_t>(slot) * p.H + ti.f * 128 + q * 32);
                        dst[0] = src[0];
                        dst[1] = src[1];
                        dst[2] = src[2];
                        dst[3] = src[3];
                    }
                    __syncwarp();
                } else {
                    // SwiGLU.  Quadrants 0,1 hold gate rows (features 32q + lane of the
                    // tile), 2,3 the matching up rows.  The pair (q, q+2) splits the 32
                    // tokens: the gate warp finishes tokens 0-15, the up warp 16-31,
                    // each taking the partner's half of the values through shared memory.
                    const int pair = q & 1;
                    const bool gate = q < 2;
                    float* X = reinterpret_cast<float*>(epi) + pair * 512;          // silu(gate), tokens 16-31
                    float* Y = reinterpret_cast<float*>(epi) + 1024 + pair * 512;   // up, tokens 0-15
                    if (gate) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float g = __uint_as_float(v[16 + j]);
                            X[j * 32 + lane] = g / (1.0f + __expf(-g));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) Y[j * 32 + lane] = __uint_as_float(v[j]);
                    }
                    named_bar_sync(1, 128);
                    uint8_t* my_bt = epi + 8192 + q * 512;   // [16 tokens][32 features]
                    uint8_t my_scale = 0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float hv;
                        if (gate) {
                            const float g = __uint_as_float(v[j]);
                            hv = g / (1.0f + __expf(-g)) * Y[j * 32 + lane];
                        } else {
                            hv = X[j * 32 + lane] * __uint_as_float(v[16 + j]);
                        }
                        const uint32_t am = __reduce_max_sync(0xffffffffu, __float_as_uint(hv) & 0x7FFFFFFFu);
                        const int X8 = mx_e4m3_block_exponent(am);
                        my_bt[j * 32 + lane] = f32_to_e4m3_satfinite(hv * exp2_neg(X8));
                        if (lane == j) my_scale = static_cast<uint8_t>(X8 + 127);
                    }
                    __syncwarp();
                    const int tok = c0 + (gate ? 0 : 16) + lane;
                    if (lane < 16 && tok < ti.nvalid) {
                        const size_t row = static_cast<size_t>(ti.r0 + tok);
                        const int col = ti.f * 64 + pair * 32;
                        const uint4* srcv = reinterpret_cast<const uint4*>(my_bt + lane * 32);
                        uint4* dst = reinterpret_cast<uint4*>(p.a2 + row * p.I + col);
                        dst[0] = srcv[0];
                        dst[1] = srcv[1];
                        const int blk = col >> 5;
                        p.a2_sf[((static_cast<size_t>(blk >> 2) * p.S4 + row) << 2) + (blk & 3)] = my_scale;
                    }
                    named_bar_sync(2, 128);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(ab));
            acc_ph[ab] ^= 1u;
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

// rank-2 or rank-3 tiled map (dims/box innermost first; strides in bytes for dims 1..rank-1)
static bool encode(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t b[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) st[i] = strides[i];
    return fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
static cudaError_t launch_mode(const CUtensorMap* maps, const KParams& kp, cudaStream_t s) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemTotal);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    mx_gemm_kernel<MODE><<<sm_count(), kThreads, kSmemTotal, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4],
                                                                   maps[5], maps[6], maps[7], kp);
    count_launches(1);
    return cudaGetLastError();
}

kt_status launch_gemm(const GemmArgs& a, cudaStream_t s) {
    if (a.S <= 0) return KT_OK;
    // 0 weight tile (fp4 unpacked), 1-4 token boxes of 16/32/64/128 rows,
    // 5 weight bytes for the L2 prefetch, 6 weight scales (16-byte rows),
    // 7 token scales (K-step-major u32)
    alignas(64) CUtensorMap maps[8];
    const bool fc1 = a.mode == GemmEpilogue::SwiGLU;
    const uint64_t K = static_cast<uint64_t>(a.K);
    const uint64_t wrows = static_cast<uint64_t>(a.E) * a.rows_w;
    const int S4 = sf_rows(a.S);
    const bool sfa_tma = (a.K % 512) == 0;
    bool ok = true;
    if (fc1) {
        // w13 viewed as [2E][I][K]: (z = 2e + half, y = row within the half)
        const uint64_t dw[3] = {K, static_cast<uint64_t>(a.I), 2ull * a.E};
        const uint64_t sw[2] = {K / 2, static_cast<uint64_t>(a.I) * (K / 2)};
        const uint32_t bw[3] = {128, 64, 2};
        ok = ok && encode(&maps[0], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, a.w, 3, dw, sw, bw,
                          CU_TENSOR_MAP_SWIZZLE_128B);
        const uint64_t dp[3] = {K / 2, static_cast<uint64_t>(a.I), 2ull * a.E};
        const uint32_t bp[3] = {static_cast<uint32_t>(kGroup * kBK / 2), 64, 2};
        ok = ok && encode(&maps[5], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w, 3, dp, sw, bp, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (sfa_tma) {
            const uint64_t ds[3] = {K / 32, static_cast<uint64_t>(a.I), 2ull * a.E};
            const uint64_t ss[2] = {K / 32, static_cast<uint64_t>(a.I) * (K / 32)};
            const uint32_t bs[3] = {16, 64, 2};
            ok = ok && encode(&maps[6], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_sf, 3, ds, ss, bs,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
        }
    } else {
        const uint64_t dw[2] = {K, wrows};
        const uint64_t sw[1] = {K / 2};
        const uint32_t bw[2] = {128, 128};
        ok = ok && encode(&maps[0], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, a.w, 2, dw, sw, bw,
                          CU_TENSOR_MAP_SWIZZLE_128B);
        const uint64_t dp[2] = {K / 2, wrows};
        const uint32_t bp[2] = {static_cast<uint32_t>(kGroup * kBK / 2), 128};
        ok = ok && encode(&maps[5], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w, 2, dp, sw, bp, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (sfa_tma) {
            const uint64_t ds[2] = {K / 32, wrows};
            const uint64_t ss[1] = {K / 32};
            const uint32_t bs[2] = {16, 128};
            ok = ok && encode(&maps[6], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_sf, 2, ds, ss, bs,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
        }
    }
    if (!sfa_tma) maps[6] = maps[5];   // not used on this path
    for (int bi = 0; bi < 4; ++bi) {
        const uint64_t db[2] = {K, static_cast<uint64_t>(a.S)};
        const uint64_t sb[1] = {K};
        const uint32_t bb[2] = {128, 16u << bi};
        ok = ok && encode(&maps[1 + bi], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.act, 2, db, sb, bb,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    }
    {
        const uint64_t da[2] = {static_cast<uint64_t>(S4), K / kBK};
        const uint64_t sa[1] = {static_cast<uint64_t>(S4) * 4};
        const uint32_t ba[2] = {256, static_cast<uint32_t>(kGroup)};
        ok = ok && encode(&maps[7], CU_TENSOR_MAP_DATA_TYPE_UINT32, a.act_sf, 2, da, sa, ba,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok) return report(KT_ERR_CUDA, "tensor map encoding failed");
    KParams kp{};
    kp.expert_offsets = a.expert_offsets;
    kp.chunk_prefix = a.chunk_prefix;
    kp.E = a.E;
    kp.K = a.K;
    kp.rows_w = a.rows_w;
    kp.I = a.I;
    kp.S = a.S;
    kp.S4 = S4;
    kp.H = a.H;
    kp.n_ftiles = fc1 ? a.I / 64 : a.rows_w / 128;
    kp.w_sf = a.w_sf;
    kp.sfa_tma = sfa_tma ? 1 : 0;
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
        case GemmEpilogue::Raw: e = launch_mode<0>(maps, kp, s); break;
        case GemmEpilogue::SwiGLU: e = launch_mode<1>(maps, kp, s); break;
        default: e = launch_mode<2>(maps, kp, s); break;
    }
    return cuda_status(e);
}

}  // namespace kt
