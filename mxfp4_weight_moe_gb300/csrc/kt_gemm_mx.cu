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
// (MMA N, a multiple of 16), K streamed in stages of 256 (tiles of at most
// kSmallN token rows) or 128 (larger tiles, so that four stages fit in
// flight).  Weights sit on the M side ("swap AB") so that experts with few
// tokens waste little MMA work.  For FC1 the 128 weight rows are 64 gate rows
// and the matching 64 up rows, so SwiGLU needs only the accumulator tile.  A
// tile's token rows start at the expert's first row rounded down to a
// multiple of 8 (up to 7 leading rows of the previous expert ride along and
// are discarded), so that its token box decomposes into whole 8-row groups.
//
// Pipeline.  One stage is a weight tile of 128 rows x kqs*128 fp4 (one TMA
// box; the 16U4_ALIGN16B type unpacks it to one byte per element in shared
// memory and counts the packed bytes as transaction bytes) plus the token
// tile of N rows x kqs*128 e4m3 bytes, kqs = 2 or 1 K-quads of 128.  Both sit
// back to back in one ring of shared memory whose stages take only the bytes
// they need.  Two producer threads share the ring bookkeeping: one loads
// weight tiles, the other token tiles; both arrive on the stage's full
// barrier.  On GB300 one thread that waits on a barrier, arrives on another
// and issues a TMA manages about one stage per 250 ns, so the producer is
// split and small-N stages carry 16 KB of packed weights.
//
// Clusters.  The CTAs of a cluster (cl = 1, 2 or 4) work on the same token
// chunk with consecutive feature tiles.  Each loads 1/cl of the token rows
// and multicasts them to all, so a token row leaves L2 once per cluster
// instead of once per feature tile; each CTA's MMA commit releases the stage
// in every CTA of the cluster (the empty barriers count cl arrivals).
//
// Shared-memory operand layouts (K-major, 128-byte swizzle):
//   weights  [K quad q][128 rows][128 B]                 (rows 128 B apart)
//   tokens   [8-row group g][K quad q][8 rows][128 B]    (groups kqs KB apart)
// so the MMA descriptor of quad q starts at the quad's first row with 1024 B
// (weights) or kqs * 1024 B (tokens) between 8-row groups.
//
// Warp roles (288 threads, one CTA per SM, persistent over tiles):
//   warp 0     weight producer (one lane): one 3-D (FC1: 4-D) TMA box with
//              the stage's K quads of the weight tile.
//   warp 1     MMA issuer: the whole warp follows the pipeline, one elected
//              lane issues tcgen05.cp (scales -> tensor memory) and
//              tcgen05.mma (4 per K quad) and commits to the barriers.
//   warps 2, 8 scale warps (alternate groups): per group of 4 K-quads each TMA-loads the weight
//              scales (16-byte rows of the plain [rows, K/32] layout) and the
//              token scales (the K-step-major u32 layout the quantisers
//              write) into a staging ring ahead of use, builds the 128x4
//              scale blocks the MMA reads, and prefetches the weight bytes of
//              a later group into L2.
//   warp 3     token producer (one lane): one 4-D TMA box per stage with
//              this CTA's share of the tile's token rows (a map per share
//              size), multicast to the cluster.
//   warps 4-7  epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//              32*(w%4)..+31), fused math, global stores.  Two accumulator
//              buffers let one tile's epilogue overlap the next main loop.
// Every barrier wait has a deadline; on expiry the role records itself in
// the device error word and the CTA winds down and frees its tensor memory.
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "kt_common.cuh"
#include "kt_decode_dev.cuh"
#include "kt_internal.h"
#include "kt_quant_dev.cuh"

namespace kt {

constexpr int kQuadW = 128 * 128;             // one K quad of the weight tile in shared memory (fp4 unpacked)
constexpr uint32_t kQuadWTx = 128 * 128 / 2;  // ... and its transaction bytes (the unpacking TMA counts packed bytes)
// Build-time tuning: the largest tile (token rows) that uses two-quad stages,
// and the largest cluster the launcher may pick.  Measured on GB300 (FC1+FC2
// of the DSV4-shaped, Kimi-K3-shaped T=16 and T=8192 layers): 96 beats 0 and
// 192; clusters of 2 beat 1 and 4.
#ifndef KT_GEMM_SMALL_N
#define KT_GEMM_SMALL_N 96
#endif
#ifndef KT_GEMM_MAX_CLUSTER
#define KT_GEMM_MAX_CLUSTER 2
#endif
constexpr int kSmallN = KT_GEMM_SMALL_N;      // tiles of at most this many token rows use two-quad stages
constexpr int kGemmMaxCluster = KT_GEMM_MAX_CLUSTER;
constexpr int kRing = 176 * 1024;             // stage ring: weight tile + token tile per stage
constexpr int kMaxCluster = 4;
static_assert(kGemmMaxCluster == 1 || kGemmMaxCluster == 2 || kGemmMaxCluster == 4, "cluster size");
constexpr int kSlots = 4;                     // stages in flight at most (barrier pairs, tensor-memory scale slots)
constexpr int kGroup = 4;                     // K quads per scale group
constexpr int kSfQuad = 512 + 1024;           // per quad: weight scale block + up to 2 token blocks
constexpr int kSfBytes = kGroup * kSfQuad;    // one scale-block buffer (two of them)
constexpr int kStgSFA = 128 * 16;             // staging: 128 weight rows x 16 scale bytes
constexpr int kStgSFB = kGroup * kTileTokens * 4;   // staging: 4 quads x tile token rows x u32
constexpr int kStgBytes = kStgSFA + kStgSFB;  // one staging buffer
constexpr int kStgBufs = 4;                   // staging: two buffers per scale warp
constexpr int kScaleWarp2 = 8;                // second scale warp (odd groups)
constexpr int kEpiBytes = 10240;              // FC1 exchange + transposes / FC2 transpose
constexpr int kBarBytes = 512;
constexpr int kTabBytes = (kMaxExperts + 1) * 4 + 8;   // chunk_prefix, staged per CTA
constexpr int kSmemTotal = 1024 + kRing + 2 * kSfBytes + kStgBufs * kStgBytes + kEpiBytes + kBarBytes + kTabBytes;
constexpr int kThreads = 288;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kTileTokens;    // accumulator buffer b at column b * kAccCols
constexpr uint32_t kTmemSF = 2 * kAccCols;    // scale columns after both accumulators
constexpr uint32_t kSfQuadCols = 12;          // per K quad: 4 weight + 8 token scale columns
constexpr uint32_t kSfGroupCols = kGroup * kSfQuadCols;   // one scale group's tensor-memory buffer (two of them)
constexpr int kPrefetchGroups = 2;            // scale-warp L2 prefetch distance, in groups (decode-sized launches)
constexpr int kPrefetchNearRows = 64;         // launches with this many token rows per expert prefetch at distance 0
// the largest stage always fits once every earlier stage is released
static_assert(2 * kQuadW + kSmallN * 256 <= kRing && kQuadW + kTileTokens * 128 <= kRing, "stage ring");
static_assert(kSmemTotal <= 232448, "shared memory budget");
static_assert(kTmemSF + 2 * kSfGroupCols <= kTmemCols, "tensor memory budget");
static_assert(kTileTokens % (8 * kMaxCluster) == 0 && kTileTokens <= 256 && kChunkRows + 7 <= kTileTokens,
              "token tile");

constexpr int kMaxShare = kTileTokens / 8;   // 8-row groups one CTA loads per stage, at most

struct TileInfo {
    int e, f;
    int r_al;     // first token row of the tile (a multiple of 8)
    int lead;     // rows of another expert before the tile's own: columns [lead, lead + nvalid) are valid
    int nvalid;
    int nmma;     // MMA N: lead + nvalid rounded up to a multiple of 16 and of 8 * cluster size
    int kqs;      // K quads (128 K) per pipeline stage: 2 for small N, 1 otherwise
};

// Tensor maps of one launch (all in kernel parameter space).
struct GemmMaps {
    CUtensorMap w[2];      // weight tile, 1 or 2 K quads per box
    CUtensorMap t[2][kMaxShare];   // token rows: [quads per stage - 1][8-row groups per box - 1]
    CUtensorMap wpf;       // packed weight bytes for the L2 prefetch
    CUtensorMap wsf;       // weight scales, 16-byte rows
    CUtensorMap asf;       // token scales, K-step-major u32
};

struct KParams {
    const int32_t* expert_offsets;
    const int32_t* chunk_prefix;
    int E, K, rows_w, I, S, S4, n_ftiles, H;
    int cl;                   // CTAs per cluster (1, 2 or 4); n_ftiles % cl == 0
    int nfg;                  // feature-tile groups per chunk: n_ftiles / cl
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
    int interleaved;          // FC1: w13 rows interleave gate / up (row 2i gate i, row 2i+1 up i)
    int act;                  // FC1: 0 SwiGLU, 1 clamped SwiGLU
    float alpha, limit;       // clamped SwiGLU parameters
    int pf_near;              // 1: each group's weights are prefetched into L2 as its scales are built
};

// The routing tables a CTA decodes its work units from.  chunk_prefix is
// staged in shared memory at kernel start (a binary search over global
// memory costs several microseconds of dependent loads at every tile
// start); expert_offsets stays in global memory (two loads per tile).
struct Tables {
    const int32_t* cp;   // chunk_prefix [E+1], shared memory
    const int32_t* eo;   // expert_offsets [E+1], global memory
};

// MODE of the single-launch decode kernel: FC1 with the SwiGLU epilogue as
// pass 0, then FC2 with the weighted-store epilogue as pass 1, in one launch.
constexpr int kFused = 3;

// Loads of routing tables and FC2 epilogue inputs.  The other modes read data
// that earlier launches wrote, through the read-only cache.  The fused kernel
// writes them itself earlier in the same launch, before a grid barrier that
// orders them (release / acquire at GPU scope); no SM reads these addresses
// before that barrier, so no stale line can be cached, and an ordinary cached
// load (ld.global.ca) sees the written values.
template <int MODE, typename T>
__device__ __forceinline__ T ld_table(const T* ptr) {
    if (MODE == kFused) return __ldca(ptr);
    return __ldg(ptr);
}

template <int MODE>
__device__ __forceinline__ bool pass_fc1(int pass) {
    return MODE == static_cast<int>(GemmEpilogue::SwiGLU) || (MODE == kFused && pass == 0);
}

// One GEMM pass of a launch: its parameters, tensor maps and work counts.
struct Pass {
    const KParams* p;
    const GemmMaps* m;
    int total;     // work units of the grid's clusters
    int nq;        // K quads per tile
    int ngroups;   // scale groups (kGroup quads) per tile
    bool fc1;      // FC1 weight views (gate / up) and the SwiGLU epilogue
};

// Work unit u of a cluster -> (expert, feature-tile group, token chunk); the
// CTA of cluster rank r takes feature tile group * cl + r.  Token chunks of
// one (expert, feature-tile group) are adjacent so concurrent clusters share
// weight tiles through L2.  chunk c of an expert with `cnt` rows split into
// nc chunks covers rows [c*cnt/nc, (c+1)*cnt/nc).
template <int MODE>
__device__ __forceinline__ void decode_tile(const KParams& p, const Tables& tb, int u, int rank, TileInfo& ti) {
    const int v = u / p.nfg;
    int lo = 1, hi = p.E;                   // first e' with chunk_prefix[e'] > v
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (tb.cp[mid] > v) hi = mid;
        else lo = mid + 1;
    }
    const int e = lo - 1;
    const int c0 = tb.cp[e];
    const int nc = tb.cp[e + 1] - c0;
    const int local = u - p.nfg * c0;
    ti.e = e;
    const int fg = local / nc;
    ti.f = fg * p.cl + rank;
    const int c = local - fg * nc;
    const int off = ld_table<MODE>(tb.eo + e);
    const int cnt = ld_table<MODE>(tb.eo + e + 1) - off;
    const int a = static_cast<int>(static_cast<long long>(c) * cnt / nc);
    const int b = static_cast<int>(static_cast<long long>(c + 1) * cnt / nc);
    const int r0 = off + a;
    ti.r_al = r0 & ~7;
    ti.lead = r0 - ti.r_al;
    ti.nvalid = b - a;
    const int gran = p.cl > 2 ? 8 * p.cl : 16;
    ti.nmma = (ti.lead + ti.nvalid + gran - 1) / gran * gran;
    ti.kqs = ti.nmma <= kSmallN ? 2 : 1;
}

__device__ __forceinline__ uint32_t stage_bytes(const TileInfo& ti) {
    return static_cast<uint32_t>(ti.kqs * (kQuadW + ti.nmma * 128));
}

// Coordinates of a tile's weight rows: for FC1 with gate | up halves (view
// [2E][I][K] of w13) (y, z) = (64 f, 2 e) selects the 64 gate rows and the 64
// matching up rows; for FC1 with interleaved rows (view [E][2][I][K], the
// [2] being row parity) (y, z) = (64 f, e); otherwise (view [E * rows_w][K])
// y = e * rows_w + 128 f.  Either FC1 view lands the 64 gate rows and then
// the 64 up rows in shared memory, so the MMA and epilogue are the same.
__device__ __forceinline__ void weight_coords(bool fc1, const KParams& p, const TileInfo& ti, int& y, int& z) {
    if (fc1) {
        y = ti.f * 64;
        z = p.interleaved ? ti.e : 2 * ti.e;
    } else {
        y = ti.e * p.rows_w + ti.f * 128;
        z = 0;
    }
}

// SiLU with the fast reciprocal-based division (the division's 2-ulp error is
// far below the MXFP8 step the result is quantised to next).
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// The gated activation h = gate_fn(g) * up_fn(u): SwiGLU (act 0) is
// silu(g) * u; the clamped SwiGLU of GPT-OSS-format checkpoints (act 1) is
// g' * sigmoid(alpha g') * (u' + 1) with g' = min(g, limit) and
// u' = clamp(u, -limit, limit).
__device__ __forceinline__ float gate_fn(float g, int act, float alpha, float limit) {
    if (act == 0) return silu(g);
    const float gc = fminf(g, limit);
    return __fdividef(gc, 1.0f + __expf(-alpha * gc));
}
__device__ __forceinline__ float up_fn(float u, int act, float limit) {
    if (act == 0) return u;
    return fminf(fmaxf(u, -limit), limit) + 1.0f;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// One lane of a fully active warp (the same lane every call).
__device__ __forceinline__ bool elect_one_sync() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.b32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z, int w, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z, int w, int v, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z,
                                            int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
        "[%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

// The same box delivered to the same shared-memory offset (and barrier
// offset) in every CTA of `mask` within the cluster.
__device__ __forceinline__ void tma_load_4d_mc_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                    int z, int w, uint16_t mask, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7, %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w), "h"(mask), "l"(policy)
        : "memory");
}

// Arrive once on the barrier at offset `bar` of every CTA in `mask` when all
// tcgen05 operations this thread issued so far have completed.
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// non-tensor bulk prefetch of `bytes` contiguous bytes into L2 (address and size multiples of 16)
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
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

__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int x, int y, int z, int w) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

// Load (or prefetch) a box of the weight-scale / weight-prefetch maps: for
// FC1 3-D (gate | up halves, z = 2e) or 4-D (interleaved rows, parity 0,
// expert z); 2-D otherwise.
__device__ __forceinline__ void load_weight_box(bool fc1, uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                                int y, int z, bool inter) {
    if (fc1) {
        if (inter) tma_load_4d(dst, map, bar, x, y, 0, z);
        else tma_load_3d(dst, map, bar, x, y, z);
    } else {
        tma_load_2d(dst, map, bar, x, y);
    }
}
__device__ __forceinline__ void prefetch_weight_box(bool fc1, const CUtensorMap* map, int x, int y, int z, bool inter) {
    if (fc1) {
        if (inter) tma_prefetch_l2_4d(map, x, y, 0, z);
        else tma_prefetch_l2_3d(map, x, y, z);
    } else {
        tma_prefetch_l2_2d(map, x, y);
    }
}

// K-major, 128-byte-swizzled operand descriptor with `sbo` bytes between
// 8-row groups (1024 when rows are packed, kqs * 1024 for the token layout).
__device__ __forceinline__ uint64_t sdesc_sw128_sbo(uint32_t saddr, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);          // bits 0-13  start address >> 4
    d |= static_cast<uint64_t>(16u >> 4) << 16;                    // bits 16-29 leading byte offset (unused)
    d |= static_cast<uint64_t>(sbo >> 4) << 32;                    // bits 32-45 stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                          // bits 46-48 fixed 0b001
    d |= static_cast<uint64_t>(2u) << 61;                          // bits 61-63 swizzle: 128B
    return d;
}

// Placement of stages in the ring: a stage of `need` bytes starts at the
// head, or at the ring start if it would cross the end.  This is the
// consumer's view (the ring offset only); RingProducer places identically.
struct PhysRing {
    uint32_t phys = 0;
    __device__ __forceinline__ uint32_t place(uint32_t need) {
        if (phys + need > static_cast<uint32_t>(kRing)) phys = 0;
        const uint32_t start = phys;
        phys += need;
        return start;
    }
};

// Producer-side bookkeeping of the ring: stage gi (counted in `gi`) uses
// barrier slot `slot` in lap `lap` (gi % kSlots and gi / kSlots, kept
// incrementally), its bytes end at virtual offset end_of(slot), bytes before
// `tail` are free and stages below `released` have completed.  Both producer
// threads run the same stage sequence and so agree on every placement, and
// the MMA warp's PhysRing reproduces the physical offsets.  The issuing
// thread is alone on its warp's critical path, so the placement does no
// 64-bit division per stage.
struct RingProducer {
    uint64_t head = 0;    // virtual end of the last placed stage
    uint32_t phys = 0;    // head % kRing
    uint64_t b_end0 = 0, b_end1 = 0, b_end2 = 0, b_end3 = 0, b_end4 = 0;   // registers, not a local array
    uint64_t tail = 0;
    long long gi = 0, released = 0;
    int slot = 0;
    uint32_t lap = 0;
    static_assert(kSlots <= 5, "one end offset per slot");
    __device__ __forceinline__ uint64_t end_of(int s) const {
        return s == 0 ? b_end0 : s == 1 ? b_end1 : s == 2 ? b_end2 : s == 3 ? b_end3 : b_end4;
    }
    __device__ __forceinline__ void set_end(int s, uint64_t v) {
        if (s == 0) b_end0 = v;
        else if (s == 1) b_end1 = v;
        else if (s == 2) b_end2 = v;
        else if (s == 3) b_end3 = v;
        else b_end4 = v;
    }
    // Waits until stage gi's barrier slot and ring bytes are free, then places it: `off` is its
    // offset in the ring and `s` its barrier slot, and the next call places stage gi + 1.  Returns
    // false on timeout (or abort).
    __device__ __forceinline__ bool acquire(uint32_t need, uint32_t empty_base, const volatile int* abort_flag,
                                            uint64_t limit, uint32_t& off, int& s) {
        if (!mbar_wait(empty_base + 8u * slot, (lap & 1u) ^ 1u, abort_flag, limit)) return false;
        if (gi >= kSlots) {   // stage gi - kSlots (and every earlier one) is done
            tail = end_of(slot);
            if (released < gi - kSlots + 1) released = gi - kSlots + 1;
        }
        uint64_t start = head;
        uint32_t p = phys;
        if (p + need > static_cast<uint32_t>(kRing)) {   // a stage never wraps: start the next lap
            start += kRing - p;
            p = 0;
        }
        while (start + need - tail > static_cast<uint64_t>(kRing)) {
            // wait for the oldest stage still holding ring bytes (the rare path: mixed stage sizes)
            const long long j = released;
            const int js = static_cast<int>(j % kSlots);
            if (!mbar_wait(empty_base + 8u * js, static_cast<uint32_t>((j / kSlots) & 1), abort_flag, limit))
                return false;
            tail = end_of(js);
            released = j + 1;
        }
        head = start + need;
        phys = p + need;
        set_end(slot, head);
        off = p;
        s = slot;
        if (++slot == kSlots) {
            slot = 0;
            ++lap;
        }
        ++gi;
        return true;
    }
};

// Walks the (pass, work unit, group of kGroup K quads) sequence of one CTA:
// every unit of pass 0, then every unit of pass 1.
template <int MODE, int NP>
struct GroupCursor {
    int pass, u, g;    // pass, work unit and group index within the tile
    TileInfo ti;
    int wy, wz;
    bool valid;
    int first, rank, stride;
    Tables tb;
    const Pass* P;
    __device__ __forceinline__ void start(const Pass* P_, const Tables& tb_, int first_, int rank_, int stride_) {
        P = P_;
        tb = tb_;
        first = first_;
        rank = rank_;
        stride = stride_;
        pass = 0;
        u = first;
        g = 0;
        load();
    }
    __device__ __forceinline__ void load() {
        while (pass < NP && u >= P[pass].total) {
            ++pass;
            u = first;
        }
        valid = pass < NP;
        if (valid) {
            decode_tile<MODE>(*P[pass].p, tb, u, rank, ti);
            weight_coords(P[pass].fc1, *P[pass].p, ti, wy, wz);
        }
    }
    __device__ __forceinline__ void advance() {
        if (++g == P[pass].ngroups) {
            g = 0;
            u += stride;
            load();
        }
    }
};

// Everything the fused decode kernel adds to the two GEMM passes: routing,
// permutation and quantisation before them, the k-way combine after them,
// and the counters of its grid barriers (all device pointers; the counters
// are zero at launch).
struct DecodeArgs {
    const float* logits;
    const uint16_t* hidden;
    int T, H, E, k, renormalize;
    int32_t* ids;
    float* w;
    int32_t* offsets;
    int32_t* chunk_prefix;
    int32_t* perm;
    int32_t* inv_perm;
    uint8_t* a1;
    uint8_t* a1_sf;
    int S4;
    const uint16_t* y;
    uint16_t* out;
    unsigned* grid_ctr;   // grid barriers: barrier b completes at b * gridDim.x arrivals
    unsigned* fc1_done;   // FC1 epilogue warps done: gridDim.x * 4 arrivals
    // the layer's weight arrays (w13, w13 scales, w2, w2 scales), prefetched into L2 at launch when
    // the whole layer is small enough to stay there (bytes 0 otherwise)
    const uint8_t* l2_pf[4];
    unsigned l2_pf_bytes[4];
};

// Decode prologue with replicated routing: for at most kReplTokens tokens whose T * E logits fit in
// kReplLogits floats, every CTA routes all T tokens and permutes all S slots in its own shared memory
// (the stage ring is free until the GEMM passes start), so that only the quantised rows A1 need a grid
// barrier before FC1.  CTA 0 publishes ids, weights and the permutation.  Measured on GB300: 1.0-1.2 us
// faster than routing across the grid at T = 1; at T = 32 the CTA's warps share one SM's fp64 pipe
// for the gating weights and routing alone took 15 us.  Offsets (bytes) into the ring:
constexpr int kReplTokens = 4;
constexpr int kReplLogits = 16384;
constexpr int kRpLogits = 0;
constexpr int kRpIds = kRpLogits + kReplLogits * 4;
constexpr int kRpW = kRpIds + kDecodeMaxSlots * 4;
constexpr int kRpPerm = kRpW + kDecodeMaxSlots * 4;
constexpr int kRpInv = kRpPerm + kDecodeMaxSlots * 4;
constexpr int kRpOff = kRpInv + kDecodeMaxSlots * 4;
constexpr int kRpCnt = kRpOff + ((kMaxExperts + 1) * 4 + 511) / 512 * 512;
static_assert(kRpCnt + (kThreads / 32) * kMaxExperts * 4 <= kRing, "replicated decode prologue fits the ring");
static_assert(4 * kThreads >= kMaxExperts, "permute_block: four experts per thread");
// L2 prefetch of the layer's weights at launch: at most this many bytes in all, in pieces of at most
// kL2PfPiece bytes per instruction
constexpr unsigned long long kL2PfMaxBytes = 64ull << 20;
constexpr unsigned kL2PfPiece = 64u << 10;

// Spin (one thread) until *ctr reaches target, with a deadline; then make
// the generic-proxy writes behind the counter visible to TMA loads.
__device__ __forceinline__ bool wait_count(unsigned* ctr, unsigned target, volatile int* abort_flag, int* err,
                                           uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) break;
        if (*abort_flag || globaltimer_ns() - t0 > limit_ns) {
            set_error(err, KT_DEVERR_TIMEOUT_GRID);
            *abort_flag = 1;
            return false;
        }
        __nanosleep(64);
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// The persistent warp-specialised GEMM over NP passes (NP = 1: one grouped
// GEMM; NP = 2 with MODE kFused: FC1 then FC2 of the decode kernel, whose
// prologue and combine phases also run here, d != nullptr).  M[i] and PP[i]
// live in kernel parameter space.
template <int MODE, int NP, bool NEAR>
__device__ __forceinline__ void gemm_body(const GemmMaps* M, const KParams* PP, const DecodeArgs* d) {
    const KParams& p = PP[0];   // fields every pass shares (E, cl, tables, error word, wait limits)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t ring_base = smem_u32(smem);             // stage ring
    uint8_t* sfbuf = smem + kRing;                         // two scale-block buffers
    uint8_t* stg = sfbuf + 2 * kSfBytes;                   // staging ring
    uint8_t* epi = stg + kStgBufs * kStgBytes;
    uint8_t* bars = epi + kEpiBytes;
    const uint32_t bar_base = smem_u32(bars);
    int32_t* s_cp = reinterpret_cast<int32_t*>(bars + kBarBytes);
    const Tables tb{s_cp, p.expert_offsets};
    // barriers: full[S] empty[S] sf_full[2] sf_empty[2] stg[3] acc_full[2] acc_empty[2] drain
    const uint32_t full_base = bar_base;
    const uint32_t empty_base = bar_base + 8u * kSlots;
    auto full_bar = [&](int s) { return full_base + 8u * s; };
    auto empty_bar = [&](int s) { return empty_base + 8u * s; };
    auto sf_full = [&](int b) { return bar_base + 8u * (2 * kSlots + b); };
    auto sf_empty = [&](int b) { return bar_base + 8u * (2 * kSlots + 2 + b); };
    auto stg_bar = [&](int b) { return bar_base + 8u * (2 * kSlots + 4 + b); };
    auto acc_full = [&](int b) { return bar_base + 8u * (2 * kSlots + 4 + kStgBufs + b); };
    auto acc_empty = [&](int b) { return bar_base + 8u * (2 * kSlots + 6 + kStgBufs + b); };
    const uint32_t drain_bar = bar_base + 8u * (2 * kSlots + 8 + kStgBufs);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 480);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 488);
    static_assert(8 * (2 * kSlots + 9 + kStgBufs) <= 480, "barrier area");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cl = p.cl;
    const int rank = cl > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int first = static_cast<int>(blockIdx.x) / cl;      // this cluster's first work unit
    const int stride = static_cast<int>(gridDim.x) / cl;      // clusters in the grid
    const uint16_t cl_mask = static_cast<uint16_t>((1u << cl) - 1u);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(full_bar(s), 2);      // one arrive.expect_tx per producer thread
            mbar_init(empty_bar(s), cl);    // one tcgen05.commit per CTA of the cluster
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sf_full(b), 1);       // the scale warp's tcgen05.commit of its scale copies
            mbar_init(sf_empty(b), 1);      // tcgen05.commit
            mbar_init(acc_full(b), 1);      // tcgen05.commit
            mbar_init(acc_empty(b), 4);     // one arrive per epilogue warp
        }
        for (int b = 0; b < kStgBufs; ++b) mbar_init(stg_bar(b), 1);   // scale warp's arrive.expect_tx
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    // the first global-memory access: the previous kernel in the stream has completed
    griddep_wait();
    griddep_launch_dependents();
    if (MODE != kFused) {
        for (int i = threadIdx.x; i <= p.E; i += kThreads) s_cp[i] = __ldg(p.chunk_prefix + i);
    }
    if (warp == 1) {
        tc_alloc(smem_u32(tmem_slot), kTmemCols);
        tc_relinquish();
    }
    for (int i = 0; i < NP; ++i) {
        const GemmMaps& mm = M[i];
        if (warp == 0 && lane == 0) {
            tma_prefetch_map(&mm.w[0]);
            tma_prefetch_map(&mm.w[1]);
        }
        if (warp == 3) {
            for (int j = lane; j < 2 * kMaxShare; j += 32) tma_prefetch_map(&mm.t[j / kMaxShare][j % kMaxShare]);
        }
        if (warp == 2 && lane == 0) {
            tma_prefetch_map(&mm.wpf);
            tma_prefetch_map(&mm.asf);
            if (PP[i].sfa_tma) tma_prefetch_map(&mm.wsf);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (cl > 1) cluster_sync_all();   // every CTA's barriers exist before any multicast lands
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    unsigned dec_bars = 0;   // grid barriers the decode prologue has passed
    if (MODE == kFused) {
        // ---------------------------------------------------------- decode prologue
        const int nw = kThreads / 32;
        const int gw = static_cast<int>(blockIdx.x) * nw + warp;
        const int nwg = static_cast<int>(gridDim.x) * nw;
        const unsigned g = gridDim.x;
        const int S = d->T * d->k;
        int* s_warp = reinterpret_cast<int*>(epi);        // 33 ints
        int* s_dst = reinterpret_cast<int*>(epi) + 64 + warp * kMaxTopK;
        const int per_row = quant_items_per_row(d->H);
        if (warp == 2 && lane == 0) {
            // the layer's weights into L2 while the prologue runs (the FC1 and FC2 passes then load them
            // from L2): this CTA's 1/gridDim share of each array
            for (int a = 0; a < 4; ++a) {
                const unsigned long long n = d->l2_pf_bytes[a];
                const unsigned long long share = ((n + g - 1) / g + 15) & ~15ull;
                const unsigned long long lo = share * blockIdx.x;
                const unsigned long long hi = lo + share < n ? lo + share : n;
                for (unsigned long long o = lo; o < hi; o += kL2PfPiece) {
                    const unsigned len = static_cast<unsigned>(hi - o < kL2PfPiece ? hi - o : kL2PfPiece);
                    bulk_prefetch_l2(d->l2_pf[a] + o, len);
                }
            }
        }
        if (d->T <= kReplTokens && d->T * d->E <= kReplLogits) {
            // replicated routing and permutation in this CTA's shared memory, then its share of the
            // quantisation, then one grid barrier
            float* s_lg = reinterpret_cast<float*>(smem + kRpLogits);
            int32_t* s_ids = reinterpret_cast<int32_t*>(smem + kRpIds);
            float* s_w = reinterpret_cast<float*>(smem + kRpW);
            int32_t* s_perm = reinterpret_cast<int32_t*>(smem + kRpPerm);
            int32_t* s_inv = reinterpret_cast<int32_t*>(smem + kRpInv);
            int32_t* s_off = reinterpret_cast<int32_t*>(smem + kRpOff);
            const int nlg = d->T * d->E;
            for (int i = threadIdx.x; i < nlg; i += kThreads) s_lg[i] = __ldg(d->logits + i);
            __syncthreads();
            for (int t = warp; t < d->T; t += nw)
                route_token_warp<true>(s_lg + static_cast<size_t>(t) * d->E, d->E, d->k, d->renormalize,
                                       s_ids + t * d->k, s_w + t * d->k);
            __syncthreads();
            permute_block<true>(s_ids, S, d->E, s_off, s_cp, s_perm, s_inv, p.err,
                                reinterpret_cast<int*>(smem + kRpCnt), s_warp);
            __syncthreads();
            if (blockIdx.x == 0) {
                for (int i = threadIdx.x; i < S; i += kThreads) {
                    d->ids[i] = s_ids[i];
                    d->w[i] = s_w[i];
                    d->perm[i] = s_perm[i];
                    d->inv_perm[i] = s_inv[i];
                }
                for (int i = threadIdx.x; i <= d->E; i += kThreads) {
                    d->offsets[i] = s_off[i];
                    d->chunk_prefix[i] = s_cp[i];
                }
            }
            for (int item = gw; item < d->T * per_row; item += nwg) {
                const int t = item / per_row, c = item - (item / per_row) * per_row;
                quant_token_warp<true>(d->hidden, t, d->H, d->k, s_inv, d->a1, d->a1_sf, d->S4, s_dst, c, c + 1);
            }
            grid_barrier(d->grid_ctr, 1 * g, abort_flag, p.err, p.wait_limit_ns);
            dec_bars = 1;
        } else {
            // route (a warp per token), grid barrier, permute (CTA 0, the stage ring as scratch), grid
            // barrier, quantise A1 (a warp per (token, 1024 elements)), grid barrier; then every CTA
            // stages chunk_prefix like the other modes.
            for (int t = gw; t < d->T; t += nwg)
                route_token_warp(d->logits + static_cast<size_t>(t) * d->E, d->E, d->k, d->renormalize,
                                 d->ids + static_cast<size_t>(t) * d->k, d->w + static_cast<size_t>(t) * d->k);
            grid_barrier(d->grid_ctr, 1 * g, abort_flag, p.err, p.wait_limit_ns);
            if (blockIdx.x == 0 && !*abort_flag)
                permute_block(d->ids, S, d->E, d->offsets, d->chunk_prefix, d->perm, d->inv_perm, p.err,
                              reinterpret_cast<int*>(smem), s_warp);
            grid_barrier(d->grid_ctr, 2 * g, abort_flag, p.err, p.wait_limit_ns);
            if (!*abort_flag) {
                for (int item = gw; item < d->T * per_row; item += nwg) {
                    const int t = item / per_row, c = item - (item / per_row) * per_row;
                    quant_token_warp(d->hidden, t, d->H, d->k, d->inv_perm, d->a1, d->a1_sf, d->S4, s_dst, c,
                                     c + 1);
                }
            }
            grid_barrier(d->grid_ctr, 3 * g, abort_flag, p.err, p.wait_limit_ns);
            dec_bars = 3;
            for (int i = threadIdx.x; i <= p.E; i += kThreads) s_cp[i] = __ldcg(d->chunk_prefix + i);
        }
        // the ring held generic-proxy scratch: order it before the TMA writes of the GEMM passes
        fence_proxy_async_smem();
        __syncthreads();
    }

    Pass P[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        P[i].p = &PP[i];
        P[i].m = &M[i];
        P[i].total = *abort_flag ? 0 : PP[i].nfg * s_cp[p.E];   // work units of the grid's clusters
        P[i].nq = PP[i].K / 128;
        P[i].ngroups = (P[i].nq + kGroup - 1) / kGroup;
        P[i].fc1 = pass_fc1<MODE>(i);
    }

    // Work units of pass i, from kernel parameter space (the producer, MMA and epilogue loops below unroll
    // their pass loop, so PP[pass] resolves to a parameter at a fixed offset; the table P is only indexed
    // at run time by the scale warps' cursor)
    const int units_all = *abort_flag ? 0 : s_cp[p.E];
    auto pass_total = [&](int i) { return PP[i].nfg * units_all; };

    if (warp == 0 || warp == 3) {
        // ------------------------------------------------------------ producers (one lane each)
        if (lane == 0) {
            const bool weights = warp == 0;
            bool ok = true;
            // weight tiles are read once per token chunk of their expert, by adjacent work units that run
            // at about the same time: normal priority keeps them in L2 between those reads (evict-first
            // measured 1-2 % slower on device memory and made host-resident weights cross the host link
            // once per chunk)
            const uint64_t pol_w = l2_policy_evict_normal();
            const uint64_t pol_a = l2_policy_evict_last();
            RingProducer rp;
#pragma unroll
            for (int pass = 0; pass < NP; ++pass) {
            if (!ok) break;
            const KParams& pp = PP[pass];
            const GemmMaps& mm = M[pass];
            const bool fc1p = pass_fc1<MODE>(pass);
            const bool inter = fc1p && pp.interleaved;
            const int nq = pp.K / 128;
            const int total = pass_total(pass);
            // FC2 token rows (A2) are written by every CTA's FC1 epilogue in this launch
            if (MODE == kFused && pass == 1 && !weights)
                ok = wait_count(d->fc1_done, gridDim.x * 4u, abort_flag, p.err, p.wait_limit_ns);
            for (int u = first; u < total && ok; u += stride) {
                TileInfo ti;
                decode_tile<MODE>(pp, tb, u, rank, ti);
                int wy, wz;
                weight_coords(fc1p, pp, ti, wy, wz);
                const uint32_t need = stage_bytes(ti);
                const int nk = (nq + ti.kqs - 1) / ti.kqs;
                const int share = (ti.nmma >> 3) / cl;            // 8-row groups this CTA loads
                const int g0 = (ti.r_al >> 3) + rank * share;
                const uint32_t gstride = static_cast<uint32_t>(ti.kqs) * 1024u;   // bytes per 8-row group
                const CUtensorMap* tm = &mm.t[ti.kqs - 1][share - 1];   // one box covers this CTA's share
                for (int kb = 0; kb < nk; ++kb) {
                    uint32_t off;
                    int slot;
                    if (!rp.acquire(need, empty_base, abort_flag, p.wait_limit_ns, off, slot)) {
                        ok = false;
                        break;
                    }
                    const bool withhold =
                        (p.debug_flags & KT_DEBUG_WITHHOLD_STAGE) && pass == 0 && u == first && kb == 0;
                    if (withhold) continue;   // test hook: a withheld stage is neither loaded nor signalled
                    const uint32_t dst = ring_base + off;
                    const int kq0 = kb * ti.kqs;
                    if (weights) {
                        mbar_arrive_expect_tx(full_bar(slot), kQuadWTx * ti.kqs);
                        const CUtensorMap* wm = &mm.w[ti.kqs - 1];
                        if (inter)
                            tma_load_5d_hint(dst, wm, full_bar(slot), 0, wy, 0, wz, kq0, pol_w);
                        else if (fc1p)
                            tma_load_4d_hint(dst, wm, full_bar(slot), 0, wy, wz, kq0, pol_w);
                        else
                            tma_load_3d_hint(dst, wm, full_bar(slot), 0, wy, kq0, pol_w);
                    } else {
                        // this CTA's expected bytes: the whole token tile, from every CTA's share
                        mbar_arrive_expect_tx(full_bar(slot), static_cast<uint32_t>(ti.nmma * 128 * ti.kqs));
                        const uint32_t tdst = dst + static_cast<uint32_t>(ti.kqs * kQuadW) +
                                              static_cast<uint32_t>(rank * share) * gstride;
                        if (cl > 1)
                            tma_load_4d_mc_hint(tdst, tm, full_bar(slot), 0, 0, kq0, g0, cl_mask, pol_a);
                        else
                            tma_load_4d_hint(tdst, tm, full_bar(slot), 0, 0, kq0, g0, pol_a);
                    }
                }
            }
            }
            if (!ok) {
                set_error(p.err, KT_DEVERR_TIMEOUT_LOAD);
                *abort_flag = 1;
            }
        }
    } else if (warp == 2 || warp == kScaleWarp2) {
        // ------------------------------------------------------------ scale warps
        // Warp 2 builds the even groups, warp 8 the odd ones; group g uses
        // scale-block buffer g & 1, so each warp owns one buffer and two
        // staging buffers.  (One warp alone paced the pipeline on GB300.)
        const int sw = warp == 2 ? 0 : 1;
        uint32_t stg_ph = 0u, sfe_ph = 0u;   // one parity bit per buffer
        bool ok = true;
        bool a2_ready = MODE != kFused;      // fused: FC2's token scales exist once every FC1 epilogue is done
        GroupCursor<MODE, NP> cur, ahead, pf;
        cur.start(P, tb, first, rank, stride);
        if (sw) cur.advance();
        ahead = cur;
        pf = cur;
        auto advance2 = [&](GroupCursor<MODE, NP>& c) {
            c.advance();
            c.advance();
        };
        // Fused kernel: the staging of the first FC2 group is deferred until that group is the one
        // being built, and then waits for every CTA's FC1 epilogue.  (Waiting when it is issued, a
        // group ahead, would hold back this CTA's last FC1 group, and with it every CTA's FC2.)
        GroupCursor<MODE, NP> deferred;
        int deferred_buf = -1;
        auto issue_staging = [&](const GroupCursor<MODE, NP>& c, int buf) {
            if (MODE == kFused && c.valid && c.pass == 1 && !a2_ready) {
                deferred = c;
                deferred_buf = buf;
                return;
            }
            if (lane == 0 && c.valid) {
                const KParams& pp = *P[c.pass].p;
                const GemmMaps& mm = *P[c.pass].m;
                const uint32_t dst = smem_u32(stg + buf * kStgBytes);
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(stg_bar(buf), static_cast<uint32_t>(kStgSFB + (pp.sfa_tma ? kStgSFA : 0)));
                if (pp.sfa_tma)
                    load_weight_box(P[c.pass].fc1, dst, &mm.wsf, stg_bar(buf), c.g * 16, c.wy, c.wz,
                                    pp.interleaved != 0);
                tma_load_2d(dst + kStgSFA, &mm.asf, stg_bar(buf), c.ti.r_al, c.g * kGroup);
            }
        };
        // L2 prefetch of a group's packed weight bytes: whole 128-byte lines, four K quads of each row at
        // once, where the stage boxes later read one or two quads of each row.  Prefill-sized launches
        // (NEAR) prefetch each group as its scales are built, which measured faster than any distance
        // ahead; decode-sized launches (2-quad stages, a few rows per tile) kPrefetchGroups of this warp's
        // groups ahead.
        constexpr bool pf_near = NEAR;
        auto prefetch_group = [&](const GroupCursor<MODE, NP>& c) {
            if (lane == 0 && c.valid)
                prefetch_weight_box(P[c.pass].fc1, &P[c.pass].m->wpf, c.g * (kGroup * 128 / 2), c.wy, c.wz,
                                    P[c.pass].p->interleaved != 0);
        };
        if (!pf_near) {
            for (int i = 0; i < kPrefetchGroups; ++i) {   // this warp's next groups
                prefetch_group(pf);
                advance2(pf);
            }
        }
        issue_staging(ahead, 2 * sw);   // staging for this warp's first group
        advance2(ahead);
        int lidx = 0;                   // this warp's groups so far (global group 2 * lidx + sw)
        while (cur.valid && ok) {
            const int sbuf = 2 * sw + (lidx & 1);   // staging buffer of this group
            const int fbuf = sw;                    // scale-block buffer of this group
            __syncwarp();                           // every lane is done with the buffer refilled next
            if (MODE == kFused && deferred_buf >= 0) {
                // the deferred group is this one (it was staged into sbuf's turn): every earlier group of
                // this warp is built, so wait for every CTA's A2 and stage it before the next is staged
                bool ready = true;
                if (lane == 0) ready = wait_count(d->fc1_done, gridDim.x * 4u, abort_flag, p.err, p.wait_limit_ns);
                ok = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
                if (!ok) break;
                a2_ready = true;
                issue_staging(deferred, deferred_buf);
                deferred_buf = -1;
            }
            issue_staging(ahead, 2 * sw + ((lidx + 1) & 1));
            advance2(ahead);
            if (pf_near) {
                prefetch_group(cur);
            } else {
                prefetch_group(pf);
                advance2(pf);
            }
            ok = __all_sync(0xffffffffu, mbar_wait(stg_bar(sbuf), (stg_ph >> sbuf) & 1u, abort_flag,
                                                   p.wait_limit_ns));
            if (!ok) break;
            ok = __all_sync(0xffffffffu, mbar_wait(sf_empty(fbuf), ((sfe_ph >> fbuf) & 1u) ^ 1u, abort_flag,
                                                   p.wait_limit_ns));
            if (!ok) break;
            const TileInfo& ti = cur.ti;
            const KParams& pp = *P[cur.pass].p;
            const int nq = P[cur.pass].nq;
            const int ksf = pp.K / 32;
            const uint8_t* sb = stg + sbuf * kStgBytes;
            uint8_t* sfo = sfbuf + fbuf * kSfBytes;
            const int kq0 = cur.g * kGroup;
            const int nkk = min(kGroup, nq - kq0);
            const int natoms = ti.nmma > 128 ? 2 : 1;
            const int lo = ti.lead, hi = ti.lead + ti.nvalid;
            // weight scales: staging row r holds the 16 scale bytes of the group (word kk = quad kk); one
            // 16-byte load per row serves all four quads (consecutive rows per lane: no bank conflicts)
            uint4 wrow[4];
            if (pp.sfa_tma) {
#pragma unroll
                for (int i = 0; i < 4; ++i) wrow[i] = *reinterpret_cast<const uint4*>(sb + (lane + 32 * i) * 16);
            }
#pragma unroll
            for (int kk = 0; kk < kGroup; ++kk) {
                if (kk >= nkk) break;
                uint8_t* blk = sfo + kk * kSfQuad;
                // tile row r -> byte (r%32)*16 + (r/32)*4 of the 512-byte block
                if (pp.sfa_tma) {
                    auto word = [&](const uint4& v) { return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w; };
                    *reinterpret_cast<uint4*>(blk + lane * 16) =
                        make_uint4(word(wrow[0]), word(wrow[1]), word(wrow[2]), word(wrow[3]));
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = lane + 32 * i;
                        size_t grow;
                        if (P[cur.pass].fc1 && pp.interleaved)
                            grow = static_cast<size_t>(ti.e) * pp.rows_w + 2 * (ti.f * 64 + (r & 63)) + (r < 64 ? 0 : 1);
                        else if (P[cur.pass].fc1)
                            grow = static_cast<size_t>(ti.e) * pp.rows_w + (r < 64 ? 0 : pp.I) + ti.f * 64 + (r & 63);
                        else
                            grow = static_cast<size_t>(ti.e) * pp.rows_w + ti.f * 128 + r;
                        cp_async_4(smem_u32(blk + lane * 16 + i * 4), pp.w_sf + grow * ksf + (kq0 + kk) * 4, 4);
                    }
                }
                // token scales from the K-step-major staging rows (tile column t = row r_al + t)
                const uint32_t* arow = reinterpret_cast<const uint32_t*>(sb + kStgSFA) + kk * kTileTokens;
                for (int a = 0; a < natoms; ++a) {
                    uint32_t t4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int t = 128 * a + lane + 32 * i;
                        t4[i] = (t >= lo && t < hi) ? arow[t] : 0u;
                    }
                    *reinterpret_cast<uint4*>(blk + 512 + a * 512 + lane * 16) =
                        make_uint4(t4[0], t4[1], t4[2], t4[3]);
                }
            }
            // The scale warp copies the group's blocks into its tensor-memory scale buffer itself
            // (tcgen05.cp), and the copies' commit completes sf_full: the MMA warp then issues
            // nothing but MMAs.  Each copy puts one 32-row x 16-byte block into all four lane
            // quadrants, the layout block-scaled MMAs read scale factors from.
            if (!pp.sfa_tma) asm volatile("cp.async.wait_all;" ::: "memory");
            fence_proxy_async_smem();
            __syncwarp();
            tc_fence_after();
            if (elect_one_sync()) {
                const uint64_t dF0 = sdesc_sf_block(smem_u32(sfo));
                const uint32_t t_buf = tmem + kTmemSF + static_cast<uint32_t>(fbuf) * kSfGroupCols;
                for (int kk = 0; kk < nkk; ++kk) {
                    const uint64_t dF = dF0 + static_cast<uint64_t>((kk * kSfQuad) >> 4);
                    const uint32_t t_sfa = t_buf + static_cast<uint32_t>(kk) * kSfQuadCols;
                    tc_cp_32x128b_warpx4(t_sfa, dF);
                    tc_cp_32x128b_warpx4(t_sfa + 4, dF + (512 >> 4));
                    if (natoms > 1) tc_cp_32x128b_warpx4(t_sfa + 8, dF + (1024 >> 4));
                }
                tc_commit(sf_full(fbuf));
            }
            __syncwarp();
            stg_ph ^= 1u << sbuf;
            sfe_ph ^= 1u << fbuf;
            ++lidx;
            advance2(cur);
        }
        if (!ok) {
            if (lane == 0) set_error(p.err, KT_DEVERR_TIMEOUT_LOAD);
            *abort_flag = 1;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp follows the pipeline (measured faster on GB300 than one
        // lane running it alone); one elected lane issues the tensor-core work.
        {
            auto wait = [&](uint32_t bar, uint32_t par) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(bar, par, abort_flag, p.wait_limit_ns));
            };
            auto leader = [&]() -> bool { return elect_one_sync(); };
            auto wsync = [&]() { __syncwarp(); };
            int sb = 0, it = 0;
            int slot = 0;                       // pipeline slot of the next stage ...
            uint32_t full_ph = 0u;              // ... and the parity its full barrier completes with
            PhysRing ring;
            uint32_t acc_ph = 0u, sf_ph = 0u;   // one parity bit per buffer
            bool ok = true, issued = false;
            // Shared-memory descriptors with a zero start address: a stage adds its address >> 4
            // (bits 0-13; shared addresses stay below 256 KB, so nothing carries out), and each
            // 32-byte K step of a quad adds 2.  The issuing lane runs alone, so its instruction
            // chain is kept short: no descriptor is rebuilt inside the stage loop.
            const uint64_t dA_t = sdesc_sw128_sbo(0u, 1024);
#pragma unroll
            for (int pass = 0; pass < NP; ++pass) {
            if (!ok) break;
            const int nq = PP[pass].K / 128;
            const int total = pass_total(pass);
            for (int u = first; u < total && ok; u += stride, ++it) {
                TileInfo ti;
                decode_tile<MODE>(PP[pass], tb, u, rank, ti);
                const int ab = it & 1;
                issued = true;
                ok = wait(acc_empty(ab), ((acc_ph >> ab) & 1u) ^ 1u);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + ab * kAccCols;
                const uint32_t idesc0 = idesc_mx_e2m1_e4m3(ti.nmma, 0);
                const uint32_t need = stage_bytes(ti);
                const int nk = (nq + ti.kqs - 1) / ti.kqs;
                const uint64_t dB_t = sdesc_sw128_sbo(0u, static_cast<uint32_t>(ti.kqs) * 1024u);
                const uint32_t b_off16 = static_cast<uint32_t>(ti.kqs * kQuadW) >> 4;
                for (int kb = 0; kb < nk && ok; ++kb) {
                    const uint32_t off = ring.place(need);
                    const int kq0 = kb * ti.kqs;
                    const int nqs = min(ti.kqs, nq - kq0);     // K quads in this stage
                    const int kq_last = kq0 + nqs - 1;
                    // a stage never straddles scale groups: it starts a group when kq0 % kGroup == 0
                    const bool group_start = (kq0 & (kGroup - 1)) == 0;
                    const bool group_end = (kq_last & (kGroup - 1)) == kGroup - 1 || kq_last == nq - 1;
                    ok = wait(full_bar(slot), full_ph);
                    if (!ok) break;
                    if (group_start) {   // the group's scales are in tensor memory
                        ok = wait(sf_full(sb), (sf_ph >> sb) & 1u);
                        if (!ok) break;
                    }
                    tc_fence_after();
                    if (leader()) {
                        const uint64_t sa = static_cast<uint64_t>((ring_base + off) >> 4);
                        const uint32_t t_sf = tmem + kTmemSF + static_cast<uint32_t>(sb) * kSfGroupCols;
                        auto issue_quad = [&](int q) {
                            const int kq = kq0 + q;
                            const uint32_t t_sfa = t_sf + static_cast<uint32_t>(kq & (kGroup - 1)) * kSfQuadCols;
                            const uint64_t dB = dB_t + sa + b_off16 + static_cast<uint64_t>(q * (1024 >> 4));
                            const uint64_t dA = dA_t + sa + static_cast<uint64_t>(q * (kQuadW >> 4));
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t idesc =
                                    idesc0 | (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
                                tc_mma_mxf8f6f4(d_tmem, dA + static_cast<uint64_t>(2 * j),
                                                dB + static_cast<uint64_t>(2 * j), idesc, t_sfa, t_sfa + 4,
                                                (kq == 0 && j == 0) ? 0u : 1u);
                            }
                        };
                        issue_quad(0);
                        if (nqs > 1) issue_quad(1);
                        if (group_end) tc_commit(sf_empty(sb));
                        if (cl > 1) tc_commit_mc(empty_bar(slot), cl_mask);   // frees the stage in every CTA
                        else tc_commit(empty_bar(slot));
                    }
                    // no warp sync here: the next barrier wait is a full-warp vote
                    if (group_end) {
                        sf_ph ^= 1u << sb;
                        sb ^= 1;
                    }
                    if (++slot == kSlots) {
                        slot = 0;
                        full_ph ^= 1u;
                    }
                }
                if (!ok) break;
                if (leader()) tc_commit(acc_full(ab));
                wsync();
                acc_ph ^= 1u << ab;
            }
            }
            if (!ok) {
                if (lane == 0) set_error(p.err, KT_DEVERR_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            // every tcgen05 operation issued above completes before teardown
            if (issued) {
                if (leader()) tc_commit(drain_bar);
                wsync();
                wait(drain_bar, 0);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 4-7)
        const int q = warp & 3;                        // tensor-memory lane quadrant
        uint32_t acc_ph = 0u;                          // one parity bit per buffer
        int it = 0;
        bool ok = true;
#pragma unroll
        for (int pass = 0; pass < NP; ++pass) {
        const KParams& pp = PP[pass];
        const int ek = MODE == kFused ? (pass == 0 ? static_cast<int>(GemmEpilogue::SwiGLU)
                                                   : static_cast<int>(GemmEpilogue::Combine))
                                      : MODE;
        const int total = pass_total(pass);
        for (int u = first; u < total && ok; u += stride, ++it) {
            TileInfo ti;
            decode_tile<MODE>(pp, tb, u, rank, ti);
            const int ab = it & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(acc_full(ab), (acc_ph >> ab) & 1u, abort_flag, p.wait_limit_ns));
            if (!ok) break;
            tc_fence_after();
            const uint32_t trow = tmem + ab * kAccCols + (static_cast<uint32_t>(32 * q) << 16);
            const int lo = ti.lead, hi = ti.lead + ti.nvalid;
            for (int c0 = 0; c0 < hi; c0 += 32) {
                uint32_t v[32];
                tc_ld_32x32b_x32(trow + static_cast<uint32_t>(c0), v);
                tc_wait_ld();
                if (ek == static_cast<int>(GemmEpilogue::Raw)) {
                    const int n = ti.f * 128 + q * 32 + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (c0 + j >= lo && c0 + j < hi)
                            pp.raw_out[static_cast<size_t>(ti.r_al + c0 + j) * pp.rows_w + n] = __uint_as_float(v[j]);
                    }
                } else if (ek == static_cast<int>(GemmEpilogue::Combine)) {
                    // weight, round to bf16 and transpose through shared memory so each
                    // lane writes 64 contiguous bytes of one token's output row
                    uint8_t* tb = epi + q * 2560;   // [32 tokens][80 bytes]
                    const bool mine = c0 + lane >= lo && c0 + lane < hi;
                    int slot = 0;
                    float wt = 0.f;
                    if (mine) {
                        slot = ld_table<MODE>(pp.perm + ti.r_al + c0 + lane);
                        wt = ld_table<MODE>(pp.topk_w + slot);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float wj = __shfl_sync(0xffffffffu, wt, j);
                        const __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(v[j]) * wj);
                        *reinterpret_cast<__nv_bfloat16*>(tb + j * 80 + lane * 2) = b;
                    }
                    __syncwarp();
                    // four lanes per token row: each store instruction writes 8 rows x 64
                    // contiguous bytes (full sectors; one lane per row left each 32-byte
                    // sector half-written per instruction)
                    const int mine_i = mine ? 1 : 0;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int tk = r * 8 + (lane >> 2);
                        const int sl = __shfl_sync(0xffffffffu, slot, tk);
                        const int mk = __shfl_sync(0xffffffffu, mine_i, tk);
                        if (mk) {
                            const uint4 val = *reinterpret_cast<const uint4*>(tb + tk * 80 + (lane & 3) * 16);
                            uint4* dst = reinterpret_cast<uint4*>(pp.y + static_cast<size_t>(sl) * pp.H + ti.f * 128 +
                                                                  q * 32) +
                                         (lane & 3);
                            *dst = val;
                        }
                    }
                    __syncwarp();
                } else {
                    // SwiGLU.  Quadrants 0,1 hold gate rows (features 32q + lane of the
                    // tile), 2,3 the matching up rows.  The pair (q, q+2) splits the 32
                    // columns: the gate warp finishes columns 0-15, the up warp 16-31,
                    // each taking the partner's half of the values through shared memory.
                    const int pair = q & 1;
                    const bool gate = q < 2;
                    float* X = reinterpret_cast<float*>(epi) + pair * 512;          // silu(gate), columns 16-31
                    float* Y = reinterpret_cast<float*>(epi) + 1024 + pair * 512;   // up, columns 0-15
                    const int act = pp.act;
                    const float alpha = pp.alpha, limit = pp.limit;
                    if (gate) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            X[j * 32 + lane] = gate_fn(__uint_as_float(v[16 + j]), act, alpha, limit);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) Y[j * 32 + lane] = up_fn(__uint_as_float(v[j]), act, limit);
                    }
                    named_bar_sync(1, 128);
                    uint8_t* my_bt = epi + 8192 + q * 512;   // [16 columns][32 features]
                    // three independent passes (h, block amax, codes) so the 16 columns overlap
                    float hv[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        hv[j] = gate ? gate_fn(__uint_as_float(v[j]), act, alpha, limit) * Y[j * 32 + lane]
                                     : X[j * 32 + lane] * up_fn(__uint_as_float(v[16 + j]), act, limit);
                    uint32_t am[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        am[j] = __reduce_max_sync(0xffffffffu, __float_as_uint(hv[j]) & 0x7FFFFFFFu);
                    uint8_t my_scale = 0;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const int X0 = mx_e4m3_block_exponent(am[j]);
                        const int X1 = mx_e4m3_block_exponent(am[j + 1]);
                        const uint16_t c2 = f32x2_to_e4m3x2_satfinite(hv[j] * exp2_neg(X0), hv[j + 1] * exp2_neg(X1));
                        my_bt[j * 32 + lane] = static_cast<uint8_t>(c2 & 0xFFu);
                        my_bt[(j + 1) * 32 + lane] = static_cast<uint8_t>(c2 >> 8);
                        if (lane == j) my_scale = static_cast<uint8_t>(X0 + 127);
                        if (lane == j + 1) my_scale = static_cast<uint8_t>(X1 + 127);
                    }
                    __syncwarp();
                    const int col_t = c0 + (gate ? 0 : 16) + lane;
                    if (lane < 16 && col_t >= lo && col_t < hi) {
                        const size_t row = static_cast<size_t>(ti.r_al + col_t);
                        const int col = ti.f * 64 + pair * 32;
                        const uint4* srcv = reinterpret_cast<const uint4*>(my_bt + lane * 32);
                        uint4* dst = reinterpret_cast<uint4*>(pp.a2 + row * pp.I + col);
                        dst[0] = srcv[0];
                        dst[1] = srcv[1];
                        const int blk = col >> 5;
                        pp.a2_sf[((static_cast<size_t>(blk >> 2) * pp.S4 + row) << 2) + (blk & 3)] = my_scale;
                    }
                    named_bar_sync(2, 128);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(ab));
            acc_ph ^= 1u << ab;
        }
        if (MODE == kFused && pass == 0) {
            // this warp's A2 rows are written: make them visible to every CTA's FC2 TMA loads
            __syncwarp();
            if (lane == 0) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __threadfence();
                atomicAdd(d->fc1_done, 1u);
            }
        }
        }
        if (!ok) {
            if (lane == 0) set_error(p.err, KT_DEVERR_TIMEOUT_EPI);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (MODE == kFused) {
        // ---------------------------------------------------------- decode combine
        // every CTA's FC2 epilogue has written its weighted rows y: out[t] = sum_j y[t*k + j]
        grid_barrier(d->grid_ctr, (dec_bars + 1) * gridDim.x, abort_flag, p.err, p.wait_limit_ns);
        if (!*abort_flag)
            combine_rows<true>(d->y, d->ids, d->T, d->H, d->k, d->E, d->out,
                               static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x,
                               static_cast<long long>(gridDim.x) * kThreads);
    }
    if (*abort_flag) __nanosleep(1000000);   // let any copy or commit still in flight land before teardown
    // no CTA leaves while a peer may still multicast into it or arrive on its barriers
    if (cl > 1) cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, kTmemCols);
    }
}

// NEAR: the L2 weight prefetch of prefill-sized launches (see the scale warps)
template <int MODE, bool NEAR>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ KParams p) {
    gemm_body<MODE, 1, NEAR>(&maps, &p, nullptr);
}

// The single-launch decode kernel: routing, permutation, quantisation, FC1,
// FC2 and the combine, as one cooperative launch with one CTA per SM.
struct DecodeParams {
    GemmMaps maps[2];
    KParams p[2];
    DecodeArgs d;
};

__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ DecodeParams dp) {
    gemm_body<kFused, 2, false>(dp.maps, dp.p, &dp.d);
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

// tiled map of rank 2-5 (dims/box innermost first; strides in bytes for dims 1..rank-1)
constexpr int kMaxMapRank = 5;
static bool encode(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn || rank < 1 || rank > kMaxMapRank) return false;
    cuuint64_t d[kMaxMapRank], st[kMaxMapRank - 1];
    cuuint32_t b[kMaxMapRank], es[kMaxMapRank] = {1, 1, 1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) st[i] = strides[i];
    return fn(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest cluster size (up to `want`) whose co-resident clusters of one CTA
// per SM cover at least 15/16 of the SMs; asked of the driver once per device.
template <int MODE>
static int pick_cluster(int want, int* grid) {
    static int best_c[64][3] = {}, best_g[64][3] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const int sms = sm_count();
    const int idx = want >= 4 ? 2 : want >= 2 ? 1 : 0;
    if (dev < 64 && best_c[dev][idx] != 0) {
        *grid = best_g[dev][idx];
        return best_c[dev][idx];
    }
    int c_pick = 1, g_pick = sms;
    for (int c = want; c >= 2; c /= 2) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(sms / c * c));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemTotal;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(c);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, mx_gemm_kernel<MODE, false>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (nclusters * c * 16 >= sms * 15) {
            c_pick = c;
            g_pick = nclusters * c;
            break;
        }
    }
    if (dev < 64) {
        best_c[dev][idx] = c_pick;
        best_g[dev][idx] = g_pick;
    }
    *grid = g_pick;
    return c_pick;
}

template <int MODE>
static cudaError_t launch_mode(const GemmMaps& maps, KParams kp, int max_cluster, cudaStream_t s) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(mx_gemm_kernel<MODE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemTotal);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(mx_gemm_kernel<MODE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemTotal);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    int want = 1;
    if (kp.n_ftiles % 4 == 0 && max_cluster >= 4) want = 4;
    else if (kp.n_ftiles % 2 == 0 && max_cluster >= 2) want = 2;
    int grid = sm_count();
    const int c = want > 1 ? pick_cluster<MODE>(want, &grid) : 1;
    kp.cl = c;
    kp.nfg = kp.n_ftiles / c;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemTotal;
    cfg.stream = s;
    // programmatic stream serialization: the CTAs may start (barriers, tensor
    // memory) while the previous kernel finishes; they wait before reading
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(c);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = c > 1 ? 2 : 1;
    cudaError_t e = kp.pf_near ? cudaLaunchKernelEx(&cfg, mx_gemm_kernel<MODE, true>, maps, kp)
                               : cudaLaunchKernelEx(&cfg, mx_gemm_kernel<MODE, false>, maps, kp);
    count_launches(1);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Every tensor map of one launch.  The maps are a pure function of the
// pointers and sizes they describe, so they are cached (MapCache below).
static bool encode_maps(const GemmArgs& a, GemmMaps& maps) {
    const bool fc1 = a.mode == GemmEpilogue::SwiGLU;
    const uint64_t K = static_cast<uint64_t>(a.K);
    const uint64_t wrows = static_cast<uint64_t>(a.E) * a.rows_w;
    const int S4 = sf_rows(a.S);
    const bool sfa_tma = (a.K % 512) == 0;
    bool ok = true;
    const bool inter = fc1 && a.interleaved;
    // Weight tiles: the unpacking type (one byte per element in shared memory, 64 packed bytes per row per
    // K quad read) in the 128-byte swizzle the MMA reads; x counts elements.
    const CUtensorMapDataType wt = CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
    const uint64_t wx = 128;
    const CUtensorMapSwizzle wsw = CU_TENSOR_MAP_SWIZZLE_128B;
    for (int kq = 1; kq <= 2; ++kq) {
        if (inter) {
            // interleaved w13 viewed as [K/128 quad][E][2 parity][I][128]: row 2i + parity of expert e
            const uint64_t dw[5] = {wx, static_cast<uint64_t>(a.I), 2, static_cast<uint64_t>(a.E), K / 128};
            const uint64_t sw[4] = {K, K / 2, static_cast<uint64_t>(a.I) * K, 64};
            const uint32_t bw[5] = {static_cast<uint32_t>(wx), 64, 2, 1, static_cast<uint32_t>(kq)};
            ok = ok && encode(&maps.w[kq - 1], wt, a.w, 5, dw, sw, bw, wsw);
        } else if (fc1) {
            // w13 viewed as [K/128 quad][2E][I][128]: (z = 2e + gate/up, y = row within the half)
            const uint64_t dw[4] = {wx, static_cast<uint64_t>(a.I), 2ull * a.E, K / 128};
            const uint64_t sw[3] = {K / 2, static_cast<uint64_t>(a.I) * (K / 2), 64};
            const uint32_t bw[4] = {static_cast<uint32_t>(wx), 64, 2, static_cast<uint32_t>(kq)};
            ok = ok && encode(&maps.w[kq - 1], wt, a.w, 4, dw, sw, bw, wsw);
        } else {
            // w viewed as [K/128 quad][E * rows_w][128]
            const uint64_t dw[3] = {wx, wrows, K / 128};
            const uint64_t sw[2] = {K / 2, 64};
            const uint32_t bw[3] = {static_cast<uint32_t>(wx), 128, static_cast<uint32_t>(kq)};
            ok = ok && encode(&maps.w[kq - 1], wt, a.w, 3, dw, sw, bw, wsw);
        }
        // activations viewed as [S8/8 group][K/128 quad][8 rows][128]; rows up
        // to S8 = S rounded up to 8 must be addressable (callers pad the buffer)
        const uint64_t S8 = (static_cast<uint64_t>(a.S) + 7) / 8 * 8;
        for (int g = 1; g <= kMaxShare; ++g) {
            const uint64_t db[4] = {128, 8, K / 128, S8 / 8};
            const uint64_t sb[3] = {K, 128, 8 * K};
            const uint32_t bb[4] = {128, 8, static_cast<uint32_t>(kq), static_cast<uint32_t>(g)};
            ok = ok && encode(&maps.t[kq - 1][g - 1], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.act, 4, db, sb, bb,
                              CU_TENSOR_MAP_SWIZZLE_128B);
        }
    }
    if (inter) {
        const uint64_t dp[4] = {K / 2, static_cast<uint64_t>(a.I), 2, static_cast<uint64_t>(a.E)};
        const uint64_t sp[3] = {K, K / 2, static_cast<uint64_t>(a.I) * K};
        const uint32_t bp[4] = {static_cast<uint32_t>(kGroup * 128 / 2), 64, 2, 1};
        ok = ok && encode(&maps.wpf, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w, 4, dp, sp, bp, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (sfa_tma) {
            const uint64_t ds[4] = {K / 32, static_cast<uint64_t>(a.I), 2, static_cast<uint64_t>(a.E)};
            const uint64_t ss[3] = {K / 16, K / 32, static_cast<uint64_t>(a.I) * (K / 16)};
            const uint32_t bs[4] = {16, 64, 2, 1};
            ok = ok && encode(&maps.wsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_sf, 4, ds, ss, bs,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
        }
    } else if (fc1) {
        const uint64_t dp[3] = {K / 2, static_cast<uint64_t>(a.I), 2ull * a.E};
        const uint64_t sp[2] = {K / 2, static_cast<uint64_t>(a.I) * (K / 2)};
        const uint32_t bp[3] = {static_cast<uint32_t>(kGroup * 128 / 2), 64, 2};
        ok = ok && encode(&maps.wpf, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w, 3, dp, sp, bp, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (sfa_tma) {
            const uint64_t ds[3] = {K / 32, static_cast<uint64_t>(a.I), 2ull * a.E};
            const uint64_t ss[2] = {K / 32, static_cast<uint64_t>(a.I) * (K / 32)};
            const uint32_t bs[3] = {16, 64, 2};
            ok = ok && encode(&maps.wsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_sf, 3, ds, ss, bs,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
        }
    } else {
        const uint64_t dp[2] = {K / 2, wrows};
        const uint64_t sp[1] = {K / 2};
        const uint32_t bp[2] = {static_cast<uint32_t>(kGroup * 128 / 2), 128};
        ok = ok && encode(&maps.wpf, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w, 2, dp, sp, bp, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (sfa_tma) {
            const uint64_t ds[2] = {K / 32, wrows};
            const uint64_t ss[1] = {K / 32};
            const uint32_t bs[2] = {16, 128};
            ok = ok && encode(&maps.wsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w_sf, 2, ds, ss, bs,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
        }
    }
    if (!sfa_tma) maps.wsf = maps.wpf;   // not used on this path
    {
        const uint64_t da[2] = {static_cast<uint64_t>(S4), K / 128};
        const uint64_t sa[1] = {static_cast<uint64_t>(S4) * 4};
        const uint32_t ba[2] = {static_cast<uint32_t>(kTileTokens), static_cast<uint32_t>(kGroup)};
        ok = ok && encode(&maps.asf, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.act_sf, 2, da, sa, ba,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    return ok;
}

// Tensor maps cached per (device, epilogue, layout, pointers, sizes): a
// decode-sized forward would otherwise spend much of its host time encoding
// the same ~53 maps per GEMM launch on every call.  The key holds everything
// a map depends on (a map is bytes: the addresses and sizes it describes,
// valid in any context), so an entry never goes stale; re-allocated memory
// at the same address with the same sizes maps to the same bytes.  Bounded:
// the table is cleared when it reaches kMapCacheEntries.
struct MapKey {
    int dev, mode, interleaved, K, E, rows_w, I, S;
    const void *w, *w_sf, *act, *act_sf;
    bool operator==(const MapKey& o) const {
        return dev == o.dev && mode == o.mode && interleaved == o.interleaved && K == o.K && E == o.E &&
               rows_w == o.rows_w && I == o.I && S == o.S && w == o.w && w_sf == o.w_sf && act == o.act &&
               act_sf == o.act_sf;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = 1469598103934665603ull;
        auto mix = [&h](uint64_t v) {
            h ^= v;
            h *= 1099511628211ull;
        };
        mix(static_cast<uint64_t>(k.dev));
        mix(static_cast<uint64_t>(k.mode) | (static_cast<uint64_t>(k.interleaved) << 8));
        mix(static_cast<uint64_t>(k.K));
        mix(static_cast<uint64_t>(k.E));
        mix(static_cast<uint64_t>(k.rows_w));
        mix(static_cast<uint64_t>(k.I));
        mix(static_cast<uint64_t>(k.S));
        mix(reinterpret_cast<uintptr_t>(k.w));
        mix(reinterpret_cast<uintptr_t>(k.w_sf));
        mix(reinterpret_cast<uintptr_t>(k.act));
        mix(reinterpret_cast<uintptr_t>(k.act_sf));
        return static_cast<size_t>(h);
    }
};
constexpr size_t kMapCacheEntries = 256;
static std::mutex g_map_mu;
static std::unordered_map<MapKey, GemmMaps, MapKeyHash>& map_cache() {
    static std::unordered_map<MapKey, GemmMaps, MapKeyHash> m;
    return m;
}

#ifndef KT_MAP_CACHE
#define KT_MAP_CACHE 1
#endif

static bool get_maps(const GemmArgs& a, GemmMaps& maps) {
    if (!KT_MAP_CACHE) return encode_maps(a, maps);
    int dev = 0;
    cudaGetDevice(&dev);
    const MapKey key{dev, static_cast<int>(a.mode), a.mode == GemmEpilogue::SwiGLU ? a.interleaved : 0, a.K, a.E,
                     a.rows_w, a.I, a.S, a.w, a.w_sf, a.act, a.act_sf};
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        auto it = map_cache().find(key);
        if (it != map_cache().end()) {
            maps = it->second;
            return true;
        }
    }
    if (!encode_maps(a, maps)) return false;
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (map_cache().size() >= kMapCacheEntries) map_cache().clear();
    map_cache().emplace(key, maps);
    return true;
}

// Kernel parameters of one GEMM pass (cluster size and feature-tile groups
// are set by the launcher).
static void fill_params(const GemmArgs& a, KParams& kp) {
    const bool fc1 = a.mode == GemmEpilogue::SwiGLU;
    const bool inter = fc1 && a.interleaved;
    const int S4 = sf_rows(a.S);
    const bool sfa_tma = (a.K % 512) == 0;
    kp = KParams{};
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
    kp.interleaved = inter ? 1 : 0;
    kp.pf_near = static_cast<long long>(a.S) >= static_cast<long long>(kPrefetchNearRows) * a.E ? 1 : 0;
    kp.act = fc1 ? a.activation : 0;
    kp.alpha = a.alpha;
    kp.limit = a.limit;
    kp.cl = 1;
    kp.nfg = kp.n_ftiles;
}

kt_status launch_gemm(const GemmArgs& a, cudaStream_t s) {
    if (a.S <= 0) return KT_OK;
    alignas(64) GemmMaps maps;
    if (!get_maps(a, maps)) return report(KT_ERR_CUDA, "tensor map encoding failed");
    KParams kp;
    fill_params(a, kp);
    const int max_cluster = kGemmMaxCluster;
    cudaError_t e;
    switch (a.mode) {
        case GemmEpilogue::Raw: e = launch_mode<0>(maps, kp, max_cluster, s); break;
        case GemmEpilogue::SwiGLU: e = launch_mode<1>(maps, kp, max_cluster, s); break;
        default: e = launch_mode<2>(maps, kp, max_cluster, s); break;
    }
    return cuda_status(e);
}

kt_status launch_decode(const GemmArgs& fc1, const GemmArgs& fc2, const DecodeInputs& in, cudaStream_t s) {
    alignas(64) DecodeParams dp;
    if (!get_maps(fc1, dp.maps[0]) || !get_maps(fc2, dp.maps[1]))
        return report(KT_ERR_CUDA, "tensor map encoding failed");
    fill_params(fc1, dp.p[0]);
    fill_params(fc2, dp.p[1]);
    DecodeArgs& d = dp.d;
    d.logits = in.logits;
    d.hidden = in.hidden;
    d.T = in.T;
    d.H = in.H;
    d.E = in.E;
    d.k = in.k;
    d.renormalize = in.renormalize;
    d.ids = in.ids;
    d.w = in.w;
    d.offsets = in.offsets;
    d.chunk_prefix = in.chunk_prefix;
    d.perm = in.perm;
    d.inv_perm = in.inv_perm;
    d.a1 = in.a1;
    d.a1_sf = in.a1_sf;
    d.S4 = sf_rows(static_cast<long long>(in.T) * in.k);
    d.y = in.y;
    d.out = in.out;
    d.grid_ctr = in.grid_ctr;
    d.fc1_done = in.fc1_done;
    const unsigned long long pf[4] = {
        static_cast<unsigned long long>(fc1.E) * fc1.rows_w * (fc1.K / 2),
        static_cast<unsigned long long>(fc1.E) * fc1.rows_w * (fc1.K / 32),
        static_cast<unsigned long long>(fc2.E) * fc2.rows_w * (fc2.K / 2),
        static_cast<unsigned long long>(fc2.E) * fc2.rows_w * (fc2.K / 32)};
    const bool pf_on = pf[0] + pf[1] + pf[2] + pf[3] <= kL2PfMaxBytes;
    const uint8_t* pf_ptr[4] = {fc1.w, fc1.w_sf, fc2.w, fc2.w_sf};
    for (int a = 0; a < 4; ++a) {
        // 16-byte aligned pieces only (every weight array is; a pointer that is not is skipped)
        const bool ok = pf_on && (reinterpret_cast<uintptr_t>(pf_ptr[a]) & 15u) == 0 && (pf[a] & 15u) == 0;
        d.l2_pf[a] = pf_ptr[a];
        d.l2_pf_bytes[a] = ok ? static_cast<unsigned>(pf[a]) : 0u;
    }
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(moe_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kSmemTotal);
        if (e != cudaSuccess) return cuda_status(e);
        attr_set[dev] = true;
    }
    // one CTA per SM, all resident at once (cooperative): the kernel's grid barriers wait on every CTA
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(sm_count()));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemTotal;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, moe_decode_kernel, dp);
    count_launches(1);
    return cuda_status(e != cudaSuccess ? e : cudaGetLastError());
}

}  // namespace kt
