/*
 * kt_moe.h -- C ABI of the GB300 (sm_103a) fused MXFP4-weight MoE layer.
 *
 * The layer (one mixture-of-experts block of a DeepSeek-V4-Flash- or
 * Kimi-K3-shaped model) computes, for T tokens of hidden size H routed top-k
 * over E experts of FC2 inter size I:
 *
 *   route:    topk_ids, topk_w = top-k of router logits, softmax weights
 *   permute:  slots s = t*k + j grouped by expert (stable), expert offsets
 *   quant:    A1 = MXFP8(hidden)            e4m3 + e8m0 per 32 along H
 *   FC1:      G|U = A1 . w13[e]^T           w13 = gate rows | up rows (2I)
 *   SwiGLU:   h = silu(G) * U;  A2 = MXFP8(h) (e8m0 per 32 along I)
 *   FC2:      Y = A2 . w2[e]^T
 *   combine:  out[t] = sum_j topk_w[t, j] * Y[slot t*k+j]
 *
 * Sources: "[MXFP4 layerwise prefill] SM 8.6 (Ampere) excluded by capability
 * whitelist" (KTransformers issue 2172; Summary, Impact and Environment:
 * native-MXFP4 DeepSeek-V4-Flash, 256 experts / top-6, 43 MoE layers, the
 * per-layer "load experts -> compute -> sync" chain and the double-buffered
 * layerwise prefill it wants instead) and "Kimi-K3 SM120 FlashInfer MXFP4
 * MoE" (Goal: MXFP8 activation x MXFP4 weight fused MoE; on-device evidence:
 * gated FC1 inter size = 2 x FC2 inter size; Phase 0 audit, item 4: SwiGLU
 * gated layout).  Element formats follow the OCP MX v1.0 specification:
 * MXFP4 = e2m1 elements, MXFP8 = e4m3 elements, one e8m0 scale per 32.
 *
 * Data formats at this boundary (all row-major, C order):
 *   bf16       uint16_t bit patterns of bfloat16
 *   fp4x2      uint8_t, two e2m1 values per byte: element 2i in bits 0-3,
 *              element 2i+1 in bits 4-7
 *   e8m0       uint8_t scale byte s meaning 2^(s-127); 255 (NaN) not allowed
 *   e4m3       uint8_t OCP E4M3FN code
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller
 *     owns every buffer.  `stream` is a cudaStream_t passed as void*
 *     (NULL = the legacy default stream).
 *   - Calls are asynchronous on `stream` and never synchronise the device
 *     (except kt_moe_read_device_error, which reads one word back).
 *   - Arguments are checked before anything is launched; a failed check
 *     returns an error and launches nothing.
 *   - The forward and routing calls allocate no device memory: scratch
 *     lives in the caller's workspace `ws` (see kt_moe_workspace_bytes).
 *   - A workspace may be reused by consecutive calls on one stream; calls
 *     that share a workspace must not overlap on the GPU.
 *   - Kernels are built for sm_103a only; other devices get KT_ERR_CUDA.
 *   - Every kernel is launched with programmatic stream serialization (it
 *     may be scheduled while the previous work in the stream finishes) and
 *     waits for that work to complete before it touches memory, so stream
 *     order is kept; each also lets the next launch in the stream start
 *     early, which matters only to a caller kernel that opts in to the
 *     same mechanism, and which must then wait before reading our outputs.
 */
#ifndef KT_MOE_H
#define KT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int kt_status;

#define KT_OK 0
#define KT_ERR_INVALID_ARG (-1)       /* null pointer, negative size, k out of range */
#define KT_ERR_UNSUPPORTED_SHAPE (-2) /* H or I not a multiple of 128, E > 1024, k > 32, ... */
#define KT_ERR_WORKSPACE (-3)         /* ws too small or not 256-byte aligned */
#define KT_ERR_CUDA (-4)              /* a CUDA runtime/driver call or launch failed */
#define KT_ERR_TIMEOUT (-5)           /* a host-side wait passed its deadline */
#define KT_ERR_DEVICE_TIMEOUT (-6)    /* a kernel's bounded wait expired (device error word) */
#define KT_ERR_ALIGNMENT (-7)         /* a pointer is not aligned as documented */
#define KT_ERR_BAD_EXPERT_ID (-8)     /* device error word: a topk id was outside [0, E) */

/* Bits of the device error word (kt_moe_read_device_error). */
#define KT_DEVERR_BAD_EXPERT_ID 0x1   /* an id outside [0, E): that slot contributed 0 */
#define KT_DEVERR_TIMEOUT_LOAD 0x2    /* GEMM producer wait expired */
#define KT_DEVERR_TIMEOUT_MMA 0x4     /* GEMM MMA-issuer wait expired */
#define KT_DEVERR_TIMEOUT_EPI 0x8     /* GEMM epilogue wait expired */
#define KT_DEVERR_TIMEOUT_GRID 0x10   /* decode kernel: a grid-wide barrier wait expired */

/* Human-readable name of a status code (static string, never NULL). */
const char* kt_status_string(kt_status status);

/* Detail of the last failed call on this host thread (argument check that
 * failed, or the CUDA error string); "" when none.  Valid until the next call. */
const char* kt_last_error(void);

/* ------------------------------------------------------------------ */
/* Routing + permutation (route and permute steps).                   */
/* ------------------------------------------------------------------ */

/* Workspace bytes kt_moe_route_permute needs for T tokens, E experts, top-k. */
size_t kt_moe_route_workspace_bytes(int T, int E, int k);

/*
 * Top-k routing and the token-to-expert permutation.
 *   logits         f32 [T, E]  router logits (finite)
 *   renormalize    1: topk_w = softmax over the k selected logits
 *                  0: topk_w = full softmax over E, taken at the selected experts
 *   topk_ids       i32 [T, k]  out: experts by (logit desc, index asc)
 *   topk_w         f32 [T, k]  out: gating weights (computed in fp64, rounded)
 *   expert_offsets i32 [E+1]   out: exclusive prefix of per-expert slot counts
 *   perm           i32 [T*k]   out: perm[p] = slot s = t*k+j of permuted row p,
 *                              grouped by expert, stable in slot order
 *   inv_perm       i32 [T*k]   out: inv_perm[s] = p
 *   ws, ws_bytes   scratch, >= kt_moe_route_workspace_bytes(T, E, k), 256-B aligned
 * Limits: 1 <= k <= min(E, 32), E <= 1024, T >= 0 (T == 0 is a no-op).
 * Errors: KT_ERR_INVALID_ARG, KT_ERR_UNSUPPORTED_SHAPE, KT_ERR_WORKSPACE,
 * KT_ERR_ALIGNMENT (pointers must be 4-byte aligned), KT_ERR_CUDA.
 */
kt_status kt_moe_route_permute(const float* logits, int T, int E, int k, int renormalize,
                               int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                               int32_t* perm, int32_t* inv_perm,
                               void* ws, size_t ws_bytes, void* stream);

/*
 * Routing + permutation for callers that cannot allocate device memory.
 *
 * No counterpart on the pages: this is a convenience of this library.  Some
 * callers have no way to hand over a scratch workspace and must not call
 * cudaMalloc themselves -- for instance a plugin whose host framework owns
 * all device memory and gives the plugin no workspace, or a latency-bound
 * serving loop where cudaMalloc's implicit device synchronisation is not
 * acceptable.  This entry point computes exactly what kt_moe_route_permute
 * computes (same kernels, same outputs), but its scratch lives in a
 * file-scope device array of KT_NOALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library holds until the process exits.
 *   - Arguments, outputs, limits and errors as for kt_moe_route_permute,
 *     without ws/ws_bytes, checked in the same order (shape, null
 *     pointers, alignment).  Then sizes whose scratch need
 *     (kt_moe_route_workspace_bytes(T, E, k)) exceeds
 *     KT_NOALLOC_SCRATCH_BYTES return KT_ERR_WORKSPACE before anything runs
 *     (1 MiB covers, e.g., T = 8192 tokens with E = 896, k = 16).
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Every call looks up the array's device address in the current
 *     device's context (cudaGetSymbolAddress, a host-side lookup), so the
 *     address stays right after a context reset.  The first call on a
 *     device may also load the library's device code into that context.
 *   - All calls share the one array and leave their scratch in it; each call
 *     clears the error word it uses and fully rewrites the rest before
 *     reading it.  Calls that overlap on the GPU (other streams, other host
 *     threads) race on the array: serialise them.
 *   - kt_moe_read_device_error cannot see this array; the outputs are the
 *     same as kt_moe_route_permute's, whose error word reports bad ids.
 */
#define KT_NOALLOC_SCRATCH_BYTES (1u << 20)
kt_status kt_moe_route_permute_noalloc(const float* logits, int T, int E, int k, int renormalize,
                                       int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                                       int32_t* perm, int32_t* inv_perm, void* stream);

/* ------------------------------------------------------------------ */
/* The fused layer forward (quant, FC1 + SwiGLU + requant, FC2 +      */
/* combine; it re-derives the permutation from topk_ids).             */
/* ------------------------------------------------------------------ */

/* Workspace bytes kt_mxfp4_moe_forward needs (0 if a size is invalid). */
size_t kt_moe_workspace_bytes(int T, int H, int I, int E, int k);

/*
 * One MoE layer forward on one GPU.
 *   hidden   bf16  [T, H]            activations
 *   topk_ids i32   [T, k]            expert of each slot; ids outside [0, E)
 *                                    are skipped (that slot adds 0) and set
 *                                    KT_DEVERR_BAD_EXPERT_ID
 *   topk_w   f32   [T, k]            gating weights
 *   w13      fp4x2 [E, 2I, H/2]      FC1 weights: rows [0, I) gate, [I, 2I) up
 *   w13_sf   e8m0  [E, 2I, H/32]
 *   w2       fp4x2 [E, H, I/2]       FC2 weights
 *   w2_sf    e8m0  [E, H, I/32]
 *   out      bf16  [T, H]            result (written, not accumulated)
 *   ws       >= kt_moe_workspace_bytes(T, H, I, E, k) bytes, 256-B aligned
 * Shape limits: H % 128 == 0, I % 128 == 0, 1 <= k <= min(E, 32),
 * E <= 1024, T >= 0 (T == 0 returns KT_OK and launches nothing).
 * The gated FC1 has 2I rows per expert, twice the FC2 inter size I; the
 * signature carries I once, so that relation holds by construction.
 * Alignment: hidden/out/topk_*: 16 B; w13/w2: 32 B; w13_sf/w2_sf: 16 B.
 * Errors: KT_ERR_INVALID_ARG, KT_ERR_UNSUPPORTED_SHAPE, KT_ERR_ALIGNMENT,
 * KT_ERR_WORKSPACE, KT_ERR_CUDA.  Device-side conditions are reported
 * through the error word (kt_moe_read_device_error), which every forward
 * call clears first.
 */
kt_status kt_mxfp4_moe_forward(const uint16_t* hidden, int T, int H,
                               const int32_t* topk_ids, const float* topk_w, int k,
                               const uint8_t* w13, const uint8_t* w13_sf,
                               const uint8_t* w2, const uint8_t* w2_sf, int E, int I,
                               uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/*
 * Options of the gated FC1 (kt_mxfp4_moe_forward_ex).
 *
 * "Kimi-K3 SM120 FlashInfer MXFP4 MoE" (Phase 0 audit conclusions, item 4)
 * notes that the SM120 MXFP4 path it audits keeps the weight layout and the
 * parameters of GPT-OSS's SwiGLU.  Those are read as the published GPT-OSS
 * definition:
 *   gate_up_layout  KT_GATE_UP_HALVES:      w13 rows [0, I) gate, [I, 2I) up
 *                   KT_GATE_UP_INTERLEAVED: w13 row 2i is gate i, row 2i+1 up i
 *                   (w13_sf rows follow the same order)
 *   activation      KT_ACT_SWIGLU:          h = silu(g) * u
 *                   KT_ACT_SWIGLU_CLAMPED:  g' = min(g, limit),
 *                                           u' = min(max(u, -limit), limit),
 *                                           h = g' * sigmoid(alpha * g') * (u' + 1)
 *   alpha, limit    parameters of KT_ACT_SWIGLU_CLAMPED (GPT-OSS: 1.702, 7.0);
 *                   both finite, limit > 0; ignored by KT_ACT_SWIGLU.
 * The two choices are independent.  A NULL options pointer means
 * {KT_GATE_UP_HALVES, KT_ACT_SWIGLU}, which is what kt_mxfp4_moe_forward does.
 */
#define KT_GATE_UP_HALVES 0
#define KT_GATE_UP_INTERLEAVED 1
#define KT_ACT_SWIGLU 0
#define KT_ACT_SWIGLU_CLAMPED 1
typedef struct kt_moe_options {
    int gate_up_layout;
    int activation;
    float alpha;
    float limit;
} kt_moe_options;

/*
 * kt_mxfp4_moe_forward with the gated-FC1 options above (opts is a HOST
 * pointer, read during the call; NULL = defaults).  Arguments, limits,
 * ownership and errors as kt_mxfp4_moe_forward, plus KT_ERR_INVALID_ARG for
 * an unknown layout or activation or an invalid alpha / limit.
 */
kt_status kt_mxfp4_moe_forward_ex(const uint16_t* hidden, int T, int H,
                                  const int32_t* topk_ids, const float* topk_w, int k,
                                  const uint8_t* w13, const uint8_t* w13_sf,
                                  const uint8_t* w2, const uint8_t* w2_sf, int E, int I,
                                  uint16_t* out, void* ws, size_t ws_bytes,
                                  const kt_moe_options* opts, void* stream);

/*
 * kt_mxfp4_moe_forward_ex on a routing that kt_moe_route_permute (or
 * kt_moe_route_permute_noalloc) has already permuted (a convenience of this
 * library; the pages route and run the layer as two steps, and this entry
 * point only avoids redoing the first one's permutation): expert_offsets [E+1],
 * perm [S] and inv_perm [S] (S = T * k; device pointers, 16-byte aligned)
 * are that call's outputs for the same topk_ids and are used as they are,
 * so the forward skips its own histogram -> scan -> scatter (three launches;
 * one small launch derives the per-expert chunk counts instead).  Results
 * are bit-identical to kt_mxfp4_moe_forward_ex.  The arrays must be exactly
 * those outputs: the GEMMs take row ranges from them without re-checking.
 * Other arguments, limits, ownership and errors as kt_mxfp4_moe_forward_ex;
 * a NULL routing array is KT_ERR_INVALID_ARG.
 */
kt_status kt_mxfp4_moe_forward_routed(const uint16_t* hidden, int T, int H,
                                      const int32_t* topk_ids, const float* topk_w, int k,
                                      const int32_t* expert_offsets, const int32_t* perm,
                                      const int32_t* inv_perm,
                                      const uint8_t* w13, const uint8_t* w13_sf,
                                      const uint8_t* w2, const uint8_t* w2_sf, int E, int I,
                                      uint16_t* out, void* ws, size_t ws_bytes,
                                      const kt_moe_options* opts, void* stream);

/*
 * Single-launch decode: routing, permutation and the layer forward in ONE
 * kernel launch, for decode-sized batches (T * k <= KT_DECODE_MAX_SLOTS).
 * It computes exactly what kt_moe_route_permute followed by
 * kt_mxfp4_moe_forward_ex compute (same ids, weights, permutation and
 * kernels' arithmetic), without their separate launches: one cooperative kernel
 * with one CTA per SM runs route -> permute -> MXFP8 quantisation -> FC1 +
 * SwiGLU -> FC2 -> combine, with grid-wide barriers (each wait bounded by the
 * same deadline as the GEMM barriers; an expired wait sets
 * KT_DEVERR_TIMEOUT_GRID and the kernel returns).
 * ("Kimi-K3 SM120 FlashInfer MXFP4 MoE", later hard gates, item 5: token
 * counts 1/2/8/32 and CUDA Graph capture/replay.)
 *   logits      f32 [T, E] router logits; renormalize as for
 *               kt_moe_route_permute
 *   hidden .. w2_sf, opts   as for kt_mxfp4_moe_forward_ex
 *   topk_ids    i32 [T, k] out;  topk_w f32 [T, k] out (16-byte aligned)
 *   out         bf16 [T, H] out
 *   ws          >= kt_moe_workspace_bytes(T, H, I, E, k), 256-byte aligned,
 *               same layout (kt_moe_workspace_layout); bytes 64-191 of its
 *               error region hold the kernel's barrier counters
 * Errors as kt_mxfp4_moe_forward_ex, plus KT_ERR_UNSUPPORTED_SHAPE when
 * T * k > KT_DECODE_MAX_SLOTS.  Needs every SM free for one CTA (a
 * cooperative launch): KT_ERR_CUDA when the device cannot co-schedule it.
 */
#define KT_DECODE_MAX_SLOTS 2048
kt_status kt_mxfp4_moe_decode(const float* logits, const uint16_t* hidden, int T, int H, int E, int k, int I,
                              int renormalize, const uint8_t* w13, const uint8_t* w13_sf,
                              const uint8_t* w2, const uint8_t* w2_sf,
                              int32_t* topk_ids, float* topk_w, uint16_t* out,
                              void* ws, size_t ws_bytes, const kt_moe_options* opts, void* stream);

/*
 * Byte offsets of the forward's intermediates inside its workspace, so that
 * tests and tools can read them after a call (all relative to ws):
 *   err            i32 device error word
 *   expert_offsets i32 [E+1]      chunk_prefix i32 [E+1] (token chunks per expert)
 *   perm, inv_perm i32 [S]        S = T*k
 *   hist           i32 [tiles*E]  permutation scratch
 *   a1 e4m3 [S, H]  (rows in permuted order; the buffer has room for S
 *                   rounded up to a multiple of 8 rows, the GEMM reads
 *                   token rows in groups of 8 and discards the padding)
 *   a1_sf           A1's e8m0 scales, K-step-major: u32 [H/128][S4] with
 *                   S4 = S rounded up to a multiple of 4; word (ks, p) holds
 *                   row p's scale bytes for 32-blocks 4ks..4ks+3 (block b in
 *                   byte b % 4)
 *   a2 e4m3 [S, I] (padded like a1), a2_sf likewise u32 [I/128][S4]
 *                   (rows in permuted order)
 *   y  bf16 [S, H]  topk_w-weighted FC2 output, rows in slot order
 */
typedef struct kt_ws_layout {
    size_t err, expert_offsets, chunk_prefix, perm, inv_perm, hist;
    size_t a1, a1_sf, a2, a2_sf, y;
    size_t total;
} kt_ws_layout;

kt_status kt_moe_workspace_layout(int T, int H, int I, int E, int k, kt_ws_layout* layout);

/*
 * Copy the device error word of a forward (or routing) workspace to *code
 * (host int).  Synchronises `stream` first; returns KT_OK, or
 * KT_ERR_DEVICE_TIMEOUT / KT_ERR_BAD_EXPERT_ID when the word has those bits.
 */
kt_status kt_moe_read_device_error(const void* ws, int* code, void* stream);

/*
 * Diagnostic entry: the block-scaled grouped GEMM alone, fp32 out.
 *   act     e4m3 [S, K] + act_sf e8m0 [S, K/32]  rows grouped by expert
 *   expert_offsets i32 [E+1] (device)            row ranges per expert
 *   w       fp4x2 [E, N, K/2] + w_sf e8m0 [E, N, K/32]
 *   out     f32 [S, N]: out[p, n] = sum_K act[p] * w[e(p), n] (block-scaled);
 *           rows outside [expert_offsets[0], expert_offsets[E]) untouched
 *   ws      >= kt_mx_gemm_workspace_bytes(S, K, E) bytes (holds the chunk
 *           prefix, the scales in K-step-major order and a copy of act padded
 *           to a multiple of 8 rows)
 * Limits: K % 128 == 0, N % 128 == 0, E <= 1024.
 */
size_t kt_mx_gemm_workspace_bytes(int S, int K, int E);
kt_status kt_mx_grouped_gemm_f32(const uint8_t* act, const uint8_t* act_sf, int S, int K,
                                 const int32_t* expert_offsets,
                                 const uint8_t* w, const uint8_t* w_sf, int E, int N,
                                 float* out, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ */
/* Measurement hooks.                                                 */
/* ------------------------------------------------------------------ */

/* Number of kernels this library has launched in this process so far. */
uint64_t kt_moe_kernel_launches(void);

/* Stages of one layer, in launch order (index into kt_moe_profile_read). */
#define KT_STAGE_ROUTE 0     /* top-k routing (kt_moe_route_permute only) */
#define KT_STAGE_PERMUTE 1   /* histogram + scan + stable scatter */
#define KT_STAGE_QUANT 2     /* MXFP8 activation quantisation + scatter */
#define KT_STAGE_FC1 3       /* FC1 grouped GEMM + SwiGLU + MXFP8 requant */
#define KT_STAGE_FC2 4       /* FC2 grouped GEMM + weighted store */
#define KT_STAGE_COMBINE 5   /* top-k combine -> bf16 out */
#define KT_NUM_STAGES 6

/*
 * Stage timing.  While enabled, every route/forward call records CUDA
 * events on its own stream around each stage (recording adds no device
 * work and no synchronisation).  kt_moe_profile_read synchronises on the
 * last event, adds each stage's elapsed time over all calls since
 * enabling into stage_ms[KT_NUM_STAGES] (host array, milliseconds) and the
 * number of calls that ran each stage into calls[KT_NUM_STAGES].
 * Enabling (again) discards earlier records.  Not thread-safe.
 */
kt_status kt_moe_profile_enable(int enable);
kt_status kt_moe_profile_read(double* stage_ms, int* calls);
/*
 * As kt_moe_profile_enable, recording only the stages whose bit
 * (1 << KT_STAGE_*) is set in stage_mask; 0 disables.  Each recorded stage
 * adds two event records to the stream, so a caller timing whole steps can
 * record just the stage it needs.  Bits at or above KT_NUM_STAGES:
 * KT_ERR_INVALID_ARG.
 */
kt_status kt_moe_profile_enable_stages(uint32_t stage_mask);

/*
 * Test hook for the device-side failure path.  wait_limit_us bounds every
 * barrier wait inside the GEMM kernels (0 restores the default of 2 s).
 * flags = KT_DEBUG_WITHHOLD_STAGE makes each GEMM CTA's producer withhold
 * the first pipeline stage of its first tile (nothing is loaded into it and
 * it is never signalled), so the MMA issuer's wait runs out: the kernel
 * records KT_DEVERR_TIMEOUT_* in the error word, frees its tensor memory
 * and returns; the CUDA context stays usable.  Process-wide; 0 disables.
 */
#define KT_DEBUG_WITHHOLD_STAGE 0x1
kt_status kt_moe_debug_configure(uint64_t wait_limit_us, int flags);

/* ------------------------------------------------------------------ */
/* Layerwise prefill: stream layer l+1's experts host -> device while  */
/* layer l computes (issue 2172, Background / motivation).             */
/* ------------------------------------------------------------------ */

typedef struct kt_layerwise kt_layerwise;

/* Bytes of one layer's packed expert store: w13 | w13_sf | w2 | w2_sf,
 * each region starting at a 256-byte multiple (offsets via
 * kt_layerwise_pack_offsets). */
size_t kt_layerwise_pack_bytes(int H, int I, int E);
kt_status kt_layerwise_pack_offsets(int H, int I, int E, size_t* w13, size_t* w13_sf,
                                    size_t* w2, size_t* w2_sf);

/*
 * Create a layerwise context for L layers.  host_packs[l] is a HOST pointer
 * (pinned, e.g. cudaHostAlloc) to layer l's pack; the array is copied, the
 * packs are not and must outlive the context.  The context allocates (and
 * destroy frees) two device pack slots, the per-call workspace for up to
 * T_max tokens, two ping-pong hidden buffers, routing buffers, one copy
 * stream and its events.  Uses the current device.
 */
kt_status kt_layerwise_create(kt_layerwise** ctx, int L, int H, int I, int E, int k, int T_max,
                              const void* const* host_packs);

/*
 * Run all L layers: h_0 = hidden, h_{l+1} = MoE_l(h_l), out = h_L.
 *   hidden bf16 [T, H] (device), logits: HOST array of L device pointers,
 *   each f32 [T, E]; out bf16 [T, H] (device); T <= T_max.
 * serialized_control = 0: double-buffered streaming -- the copy stream
 *   uploads layer l+1 into the other slot while `stream` computes layer l.
 * serialized_control = 1: the per-layer "upload all experts -> compute ->
 *   synchronise" chain, kept as the measurement control.
 * Routing uses renormalized top-k softmax.  Returns after enqueueing all
 * work (serialized_control = 1 also synchronises per layer); host waits are
 * bounded and return KT_ERR_TIMEOUT.
 */
kt_status kt_layerwise_prefill(kt_layerwise* ctx, const uint16_t* hidden, const float* const* logits,
                               uint16_t* out, int T, int serialized_control, void* stream);

/*
 * Zero-copy variant of kt_layerwise_create for hosts whose memory the GPU
 * reads coherently (a Grace-Blackwell node over NVLink-C2C).  Same arguments;
 * each host_packs[l] must be pinned (cudaHostAlloc or cudaHostRegister) and
 * 256-byte aligned.  No device slots and no copy stream traffic: in
 * kt_layerwise_prefill the GEMMs of layer l read its packed experts in place
 * from host_packs[l] (through its device address, cudaHostGetDevicePointer),
 * so the host link is crossed by the GEMM's own loads.  Everything else
 * (workspace, routing buffers, hidden ping-pong buffers) is as for
 * kt_layerwise_create.  Errors: KT_ERR_INVALID_ARG when a pack is not pinned,
 * not mapped or misaligned; otherwise as kt_layerwise_create.
 * This is the zero-copy form of the double-buffered layerwise prefill that
 * issue 2172 (Background / motivation) asks for in place of the per-layer
 * "load -> compute -> sync" chain of its Impact section.
 */
kt_status kt_layerwise_create_zero_copy(kt_layerwise** ctx, int L, int H, int I, int E, int k, int T_max,
                                        const void* const* host_packs);

/*
 * Per-layer timing of the next prefills (measurement hook).  enable = 1
 * creates 4*L+1 CUDA events; every later kt_layerwise_prefill records, per
 * layer, events around its copy (on the copy stream) and around its compute
 * (routing + forward, on the caller's stream), plus one start event.
 * kt_layerwise_read_timing synchronises on the last layer's events and
 * writes, for the most recent prefill: copy_ms[l] and compute_ms[l] (HOST
 * arrays of L doubles, milliseconds; copy_ms is 0 in zero-copy mode) and
 * *span_ms, the time from the start event to the end of the last layer.
 * enable = 0 frees the events.  Not thread-safe.
 */
kt_status kt_layerwise_enable_timing(kt_layerwise* ctx, int enable);
kt_status kt_layerwise_read_timing(kt_layerwise* ctx, double* copy_ms, double* compute_ms, double* span_ms);

/* Test hook: make the copy step of layer `layer` report KT_ERR_CUDA
 * (-1 disables).  The pipeline must drain both streams and return it.
 * In zero-copy mode the same layer's step reports it before its compute. */
kt_status kt_layerwise_inject_copy_failure(kt_layerwise* ctx, int layer);

kt_status kt_layerwise_destroy(kt_layerwise* ctx);

#ifdef __cplusplus
}
#endif

#endif /* KT_MOE_H */
