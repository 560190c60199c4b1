// kt_internal.h -- host-side declarations shared by the library's
// translation units: workspace layout, kernel launchers and tensor maps.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kt_moe.h"

namespace kt {

// Token rows of one GEMM tile (the MMA N extent; two accumulator buffers of
// this many columns fit in tensor memory next to the scale columns), the
// most rows of one expert a tile covers (a tile starts at its first row
// rounded down to a multiple of 8, so kChunkRows + 7 <= kTileTokens), and
// the number of slots one permutation tile handles.
constexpr int kTileTokens = 192;
constexpr int kChunkRows = 176;
constexpr int kPermTile = 1024;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int perm_tiles(long long S) { return static_cast<int>((S + kPermTile - 1) / kPermTile); }

// Activation scales (A1, A2) are stored K-step-major: a u32 array
// [K/128][S4] whose word (ks, p) holds the four e8m0 bytes of row p for the
// 32-element blocks 4ks..4ks+3 (block b in byte b % 4).  S4 = S rounded up to
// a multiple of 4 keeps every row of the array 16-byte aligned for TMA.
inline int sf_rows(long long S) { return static_cast<int>((S + 3) / 4 * 4); }

// Activation code buffers (A1, A2) hold S rounded up to a multiple of 8 rows:
// the GEMM loads token rows in whole groups of 8.
inline long long act_rows(long long S) { return (S + 7) / 8 * 8; }

// Workspace carving (offsets relative to the 256-byte aligned base).
bool ws_layout(int T, int H, int I, int E, int k, kt_ws_layout* L);
// Routing workspace: error word, hist [tiles * E], chunk prefix [E + 1].
struct RouteWs {
    size_t err, hist, chunk_prefix, total;
};
bool route_ws_layout(int T, int E, int k, RouteWs* L);

// Launch with programmatic stream serialization: the kernel may begin while
// its predecessor in the stream runs, and waits for it (griddep_wait) before
// touching global memory.  Used for every kernel of the routing and forward
// paths.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------- launchers
// All return cudaSuccess or the launch error; none synchronises.
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int renormalize, int32_t* ids, float* w,
                              cudaStream_t s);
// Permutation of S = T*k slots: histogram -> scan -> stable scatter (one
// single-block launch up to 2048 slots, three launches above).
// Writes expert_offsets [E+1], chunk_prefix [E+1] (token chunks of at most
// kChunkRows rows per expert), perm [S], inv_perm [S]; hist is scratch of
// perm_tiles(S) * E ints; err collects KT_DEVERR_BAD_EXPERT_ID.
cudaError_t launch_permute(const int32_t* ids, long long S, int E, int32_t* hist, int32_t* expert_offsets,
                           int32_t* chunk_prefix, int32_t* perm, int32_t* inv_perm, int* err, cudaStream_t s);
// chunk_prefix [E+1] from expert_offsets alone (for the diagnostic GEMM).
cudaError_t launch_chunk_prefix(const int32_t* expert_offsets, int E, int32_t* chunk_prefix, cudaStream_t s);
// MXFP8 quantisation of hidden rows, each written to its k permuted rows
// (codes [S, H]; scales K-step-major with S4 = sf_rows(S)).  With `offsets`
// (expert_offsets [E+1]) the same launch also writes chunk_prefix [E+1].
cudaError_t launch_quant_scatter(const uint16_t* hidden, int T, int H, int k, const int32_t* inv_perm, uint8_t* a1,
                                 uint8_t* a1_sf, int S4, cudaStream_t s, const int32_t* offsets = nullptr, int E = 0,
                                 int32_t* chunk_prefix = nullptr);
// Plain [S, K/32] scale bytes -> K-step-major layout (diagnostic GEMM entry).
cudaError_t launch_sf_to_kstep_major(const uint8_t* plain, int S, int K, uint8_t* out, int S4, cudaStream_t s);
// out[t] = sum over valid slots of y[t*k + j] (y already weighted).
cudaError_t launch_combine(const uint16_t* y, const int32_t* ids, int T, int H, int k, int E, uint16_t* out,
                           cudaStream_t s);

enum class GemmEpilogue : int { Raw = 0, SwiGLU = 1, Combine = 2 };

struct GemmArgs {
    GemmEpilogue mode;
    const int32_t* expert_offsets;  // [E+1] permuted row ranges
    const int32_t* chunk_prefix;    // [E+1]
    int E;
    int K;            // contraction length, % 128 == 0
    int rows_w;       // weight rows per expert (2I for FC1, H for FC2, N for Raw)
    int I;            // FC2 inter size (SwiGLU: up rows start at I)
    int S;            // activation rows
    const uint8_t* w;      // fp4x2 [E, rows_w, K/2]
    const uint8_t* w_sf;   // e8m0  [E, rows_w, K/32]
    const uint8_t* act;    // e4m3  [S, K]
    const uint8_t* act_sf; // e8m0, K-step-major u32 [K/128][sf_rows(S)]
    // SwiGLU outputs: A2 e4m3 [S, I] + e8m0 K-step-major [I/128][sf_rows(S)]
    uint8_t* a2;
    uint8_t* a2_sf;
    // Combine outputs: y bf16 [S, H] in slot order, scaled by topk_w
    uint16_t* y;
    const int32_t* perm;
    const float* topk_w;
    int H;
    // Raw output: f32 [S, rows_w]
    float* raw_out;
    int* err;
    // SwiGLU: w13 gate/up row layout and gated activation (kt_moe_options)
    int interleaved = 0;
    int activation = 0;
    float alpha = 1.0f, limit = 0.0f;
};

// Test-hook settings (kt_moe_debug_configure), read at each GEMM launch.
struct DebugSettings {
    uint64_t wait_limit_ns;
    int flags;
};
DebugSettings debug_settings();

// Encodes the tensor maps and launches the persistent tcgen05 GEMM.
// Returns KT_OK, KT_ERR_CUDA (launch / map encoding failure).
kt_status launch_gemm(const GemmArgs& a, cudaStream_t s);

// The single-launch decode kernel (route -> permute -> quantise -> FC1 ->
// FC2 -> combine), for T * k <= kDecodeMaxSlots slots.  fc1 / fc2 are the two
// GEMM passes as launch_gemm takes them (their routing tables are written by
// the kernel itself); grid_ctr and fc1_done are zeroed device counters.
struct DecodeInputs {
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
    const uint16_t* y;
    uint16_t* out;
    unsigned* grid_ctr;
    unsigned* fc1_done;
};
kt_status launch_decode(const GemmArgs& fc1, const GemmArgs& fc2, const DecodeInputs& in, cudaStream_t s);

// Device properties cached per device.
int sm_count();

// Argument checks of the routing entry points (shape limits, null pointers,
// 4-byte alignment), in that order; KT_OK also for T == 0.  Records the
// failing check as kt_last_error().
kt_status check_route_args(const float* logits, int T, int E, int k, const int32_t* topk_ids, const float* topk_w,
                           const int32_t* expert_offsets, const int32_t* perm, const int32_t* inv_perm);

// Status helper: map a CUDA error to KT_ERR_CUDA, remembering the last one.
kt_status cuda_status(cudaError_t e);
// Record `msg` as this thread's kt_last_error() text and return `st`.
kt_status report(kt_status st, const char* msg);

// Measurement hooks (kt_profile.cpp): launch counter and, when profiling is
// enabled, CUDA events recorded on the stream around one stage (RAII).
void count_launches(int n);
class StageTimer {
  public:
    StageTimer(int stage, cudaStream_t s);
    ~StageTimer();
    StageTimer(const StageTimer&) = delete;
    StageTimer& operator=(const StageTimer&) = delete;

  private:
    int stage_;
    cudaStream_t s_;
    cudaEvent_t end_;
};

}  // namespace kt
