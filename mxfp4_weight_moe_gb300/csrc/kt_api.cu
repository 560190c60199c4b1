// kt_api.cu -- the C ABI declared in include/kt_moe.h: argument checks,
// workspace carving and the launch sequence of one MoE layer forward
// (permute -> quantise+scatter -> FC1+SwiGLU+requant -> FC2 -> combine).
#include <cstdarg>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kt_internal.h"

namespace kt {

static thread_local char g_last_error[256] = "";

static kt_status fail(kt_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
static kt_status fail(kt_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

kt_status report(kt_status st, const char* msg) {
    snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
    return st;
}

kt_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return KT_OK;
    snprintf(g_last_error, sizeof(g_last_error), "CUDA error %d: %s", static_cast<int>(e), cudaGetErrorString(e));
    return KT_ERR_CUDA;
}

int sm_count() {
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (counts[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        counts[dev] = n > 0 ? n : 1;
    }
    return counts[dev];
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool ws_layout(int T, int H, int I, int E, int k, kt_ws_layout* L) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return false;
    const size_t S = static_cast<size_t>(T) * static_cast<size_t>(k);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 1024);
        return o;
    };
    L->err = take(256);
    L->expert_offsets = take(sizeof(int32_t) * (E + 1));
    L->chunk_prefix = take(sizeof(int32_t) * (E + 1));
    L->perm = take(sizeof(int32_t) * S);
    L->inv_perm = take(sizeof(int32_t) * S);
    L->hist = take(sizeof(int32_t) * static_cast<size_t>(perm_tiles(static_cast<long long>(S))) * E);
    const size_t S4 = static_cast<size_t>(sf_rows(static_cast<long long>(S)));
    const size_t S8 = static_cast<size_t>(act_rows(static_cast<long long>(S)));
    L->a1 = take(S8 * H);
    L->a1_sf = take(S4 * (H / 32));
    L->a2 = take(S8 * I);
    L->a2_sf = take(S4 * (I / 32));
    L->y = take(S * H * sizeof(uint16_t));
    L->total = off;
    return true;
}

bool route_ws_layout(int T, int E, int k, RouteWs* L) {
    if (T < 0 || E <= 0 || k <= 0) return false;
    const long long S = static_cast<long long>(T) * k;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 1024);
        return o;
    };
    L->err = take(256);
    L->hist = take(sizeof(int32_t) * static_cast<size_t>(perm_tiles(S)) * E);
    L->chunk_prefix = take(sizeof(int32_t) * (E + 1));
    L->total = off;
    return true;
}

static kt_status check_route_shape(int T, int E, int k) {
    if (T < 0) return fail(KT_ERR_INVALID_ARG, "T=%d must be >= 0", T);
    if (E <= 0 || k <= 0) return fail(KT_ERR_INVALID_ARG, "E=%d and k=%d must be positive", E, k);
    if (k > E) return fail(KT_ERR_INVALID_ARG, "k=%d exceeds E=%d", k, E);
    if (E > kMaxExperts) return fail(KT_ERR_UNSUPPORTED_SHAPE, "E=%d above the supported %d", E, kMaxExperts);
    if (k > kMaxTopK) return fail(KT_ERR_UNSUPPORTED_SHAPE, "k=%d above the supported %d", k, kMaxTopK);
    if (static_cast<long long>(T) * k > INT_MAX / 2)
        return fail(KT_ERR_UNSUPPORTED_SHAPE, "T*k=%lld slots too many", static_cast<long long>(T) * k);
    return KT_OK;
}

kt_status check_route_args(const float* logits, int T, int E, int k, const int32_t* topk_ids, const float* topk_w,
                           const int32_t* expert_offsets, const int32_t* perm, const int32_t* inv_perm) {
    kt_status st = check_route_shape(T, E, k);
    if (st != KT_OK || T == 0) return st;
    if (!logits || !topk_ids || !topk_w || !expert_offsets || !perm || !inv_perm)
        return fail(KT_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(expert_offsets, 4) ||
        !aligned(perm, 4) || !aligned(inv_perm, 4))
        return fail(KT_ERR_ALIGNMENT, "routing pointers must be 4-byte aligned");
    return KT_OK;
}

}  // namespace kt

using namespace kt;

extern "C" {

const char* kt_status_string(kt_status s) {
    switch (s) {
        case KT_OK: return "KT_OK";
        case KT_ERR_INVALID_ARG: return "KT_ERR_INVALID_ARG";
        case KT_ERR_UNSUPPORTED_SHAPE: return "KT_ERR_UNSUPPORTED_SHAPE";
        case KT_ERR_WORKSPACE: return "KT_ERR_WORKSPACE";
        case KT_ERR_CUDA: return "KT_ERR_CUDA";
        case KT_ERR_TIMEOUT: return "KT_ERR_TIMEOUT";
        case KT_ERR_DEVICE_TIMEOUT: return "KT_ERR_DEVICE_TIMEOUT";
        case KT_ERR_ALIGNMENT: return "KT_ERR_ALIGNMENT";
        case KT_ERR_BAD_EXPERT_ID: return "KT_ERR_BAD_EXPERT_ID";
        default: return "KT_ERR_UNKNOWN";
    }
}

const char* kt_last_error(void) { return g_last_error; }

size_t kt_moe_route_workspace_bytes(int T, int E, int k) {
    RouteWs L;
    if (check_route_shape(T, E, k) != KT_OK || !route_ws_layout(T, E, k, &L)) return 0;
    return L.total;
}

kt_status kt_moe_route_permute(const float* logits, int T, int E, int k, int renormalize, int32_t* topk_ids,
                               float* topk_w, int32_t* expert_offsets, int32_t* perm, int32_t* inv_perm, void* ws,
                               size_t ws_bytes, void* stream) {
    g_last_error[0] = '\0';
    kt_status st = check_route_args(logits, T, E, k, topk_ids, topk_w, expert_offsets, perm, inv_perm);
    if (st != KT_OK || T == 0) return st;
    if (!ws) return fail(KT_ERR_INVALID_ARG, "null pointer argument");
    RouteWs L;
    route_ws_layout(T, E, k, &L);
    if (!aligned(ws, 256)) return fail(KT_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < L.total) return fail(KT_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, L.total);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    int* err = reinterpret_cast<int*>(base + L.err);
    if ((st = cuda_status(cudaMemsetAsync(err, 0, sizeof(int), s))) != KT_OK) return st;
    {
        StageTimer timer(KT_STAGE_ROUTE, s);
        if ((st = cuda_status(launch_route_topk(logits, T, E, k, renormalize ? 1 : 0, topk_ids, topk_w, s))) !=
            KT_OK)
            return st;
    }
    StageTimer timer(KT_STAGE_PERMUTE, s);
    return cuda_status(launch_permute(topk_ids, static_cast<long long>(T) * k, E,
                                      reinterpret_cast<int32_t*>(base + L.hist), expert_offsets,
                                      reinterpret_cast<int32_t*>(base + L.chunk_prefix), perm, inv_perm, err, s));
}

size_t kt_moe_workspace_bytes(int T, int H, int I, int E, int k) {
    kt_ws_layout L;
    if (check_route_shape(T, E, k) != KT_OK) return 0;
    if (H <= 0 || I <= 0 || H % 128 || I % 128) return 0;
    if (!ws_layout(T, H, I, E, k, &L)) return 0;
    return L.total;
}

kt_status kt_moe_workspace_layout(int T, int H, int I, int E, int k, kt_ws_layout* layout) {
    if (!layout) return fail(KT_ERR_INVALID_ARG, "null layout");
    if (kt_moe_workspace_bytes(T, H, I, E, k) == 0 && T != 0)
        return fail(KT_ERR_UNSUPPORTED_SHAPE, "invalid sizes");
    if (!ws_layout(T, H, I, E, k, layout)) return fail(KT_ERR_INVALID_ARG, "invalid sizes");
    return KT_OK;
}

kt_status kt_mxfp4_moe_forward(const uint16_t* hidden, int T, int H, const int32_t* topk_ids, const float* topk_w,
                               int k, const uint8_t* w13, const uint8_t* w13_sf, const uint8_t* w2,
                               const uint8_t* w2_sf, int E, int I, uint16_t* out, void* ws, size_t ws_bytes,
                               void* stream) {
    return kt_mxfp4_moe_forward_ex(hidden, T, H, topk_ids, topk_w, k, w13, w13_sf, w2, w2_sf, E, I, out, ws, ws_bytes,
                                   nullptr, stream);
}

// The forward behind kt_mxfp4_moe_forward_ex (routed == false: the permutation is derived here from
// topk_ids) and kt_mxfp4_moe_forward_routed (routed == true: r_offsets / r_perm / r_inv_perm are the
// routing call's outputs).
static kt_status forward_impl(const uint16_t* hidden, int T, int H, const int32_t* topk_ids, const float* topk_w,
                              int k, bool routed, const int32_t* r_offsets, const int32_t* r_perm,
                              const int32_t* r_inv_perm, const uint8_t* w13, const uint8_t* w13_sf,
                              const uint8_t* w2, const uint8_t* w2_sf, int E, int I, uint16_t* out, void* ws,
                              size_t ws_bytes, const kt_moe_options* opts, void* stream) {
    g_last_error[0] = '\0';
    kt_moe_options o{KT_GATE_UP_HALVES, KT_ACT_SWIGLU, 1.0f, 0.0f};
    if (opts) o = *opts;
    if (o.gate_up_layout != KT_GATE_UP_HALVES && o.gate_up_layout != KT_GATE_UP_INTERLEAVED)
        return fail(KT_ERR_INVALID_ARG, "gate_up_layout=%d is not a KT_GATE_UP_* value", o.gate_up_layout);
    if (o.activation != KT_ACT_SWIGLU && o.activation != KT_ACT_SWIGLU_CLAMPED)
        return fail(KT_ERR_INVALID_ARG, "activation=%d is not a KT_ACT_* value", o.activation);
    if (o.activation == KT_ACT_SWIGLU_CLAMPED &&
        !(std::isfinite(o.alpha) && std::isfinite(o.limit) && o.limit > 0.0f))
        return fail(KT_ERR_INVALID_ARG, "clamped SwiGLU needs a finite alpha and a finite limit > 0");
    kt_status st = check_route_shape(T, E, k);
    if (st != KT_OK) return st;
    if (H <= 0 || I <= 0) return fail(KT_ERR_INVALID_ARG, "H=%d and I=%d must be positive", H, I);
    if (H % 128 || I % 128)
        return fail(KT_ERR_UNSUPPORTED_SHAPE, "H=%d and I=%d must be multiples of 128", H, I);
    if (static_cast<long long>(E) * 2 * I > INT_MAX / 2 || static_cast<long long>(E) * H > INT_MAX / 2)
        return fail(KT_ERR_UNSUPPORTED_SHAPE, "E*2I or E*H too large");
    if (T == 0) return KT_OK;
    if (!hidden || !topk_ids || !topk_w || !w13 || !w13_sf || !w2 || !w2_sf || !out || !ws)
        return fail(KT_ERR_INVALID_ARG, "null pointer argument");
    if (routed && (!r_offsets || !r_perm || !r_inv_perm))
        return fail(KT_ERR_INVALID_ARG, "null routing array (expert_offsets, perm, inv_perm)");
    if (!aligned(hidden, 16) || !aligned(out, 16) || !aligned(topk_ids, 16) || !aligned(topk_w, 16))
        return fail(KT_ERR_ALIGNMENT, "hidden, out, topk_ids and topk_w must be 16-byte aligned");
    if (routed && (!aligned(r_offsets, 16) || !aligned(r_perm, 16) || !aligned(r_inv_perm, 16)))
        return fail(KT_ERR_ALIGNMENT, "expert_offsets, perm and inv_perm must be 16-byte aligned");
    if (!aligned(w13, 32) || !aligned(w2, 32))
        return fail(KT_ERR_ALIGNMENT, "w13 and w2 must be 32-byte aligned");
    if (!aligned(w13_sf, 16) || !aligned(w2_sf, 16))
        return fail(KT_ERR_ALIGNMENT, "w13_sf and w2_sf must be 16-byte aligned");
    kt_ws_layout L;
    ws_layout(T, H, I, E, k, &L);
    if (!aligned(ws, 256)) return fail(KT_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < L.total) return fail(KT_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, L.total);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    int* err = reinterpret_cast<int*>(base + L.err);
    const int32_t* offsets = routed ? r_offsets : reinterpret_cast<int32_t*>(base + L.expert_offsets);
    int32_t* chunk_prefix = reinterpret_cast<int32_t*>(base + L.chunk_prefix);
    const int32_t* perm = routed ? r_perm : reinterpret_cast<int32_t*>(base + L.perm);
    const int32_t* inv_perm = routed ? r_inv_perm : reinterpret_cast<int32_t*>(base + L.inv_perm);
    uint8_t* a1 = base + L.a1;
    uint8_t* a1_sf = base + L.a1_sf;
    uint8_t* a2 = base + L.a2;
    uint8_t* a2_sf = base + L.a2_sf;
    uint16_t* y = reinterpret_cast<uint16_t*>(base + L.y);
    const long long S = static_cast<long long>(T) * k;

    if ((st = cuda_status(cudaMemsetAsync(err, 0, sizeof(int), s))) != KT_OK) return st;
    if (!routed) {
        StageTimer timer(KT_STAGE_PERMUTE, s);
        if ((st = cuda_status(launch_permute(topk_ids, S, E, reinterpret_cast<int32_t*>(base + L.hist),
                                             reinterpret_cast<int32_t*>(base + L.expert_offsets), chunk_prefix,
                                             reinterpret_cast<int32_t*>(base + L.perm),
                                             reinterpret_cast<int32_t*>(base + L.inv_perm), err, s))) != KT_OK)
            return st;
    }
    {
        // on a given routing, the quantiser's launch also derives the per-expert chunk counts
        StageTimer timer(KT_STAGE_QUANT, s);
        if ((st = cuda_status(launch_quant_scatter(hidden, T, H, k, inv_perm, a1, a1_sf, sf_rows(S), s,
                                                   routed ? offsets : nullptr, E, chunk_prefix))) != KT_OK)
            return st;
    }

    GemmArgs fc1{};
    fc1.mode = GemmEpilogue::SwiGLU;
    fc1.expert_offsets = offsets;
    fc1.chunk_prefix = chunk_prefix;
    fc1.E = E;
    fc1.K = H;
    fc1.rows_w = 2 * I;
    fc1.I = I;
    fc1.S = static_cast<int>(S);
    fc1.H = H;
    fc1.w = w13;
    fc1.w_sf = w13_sf;
    fc1.act = a1;
    fc1.act_sf = a1_sf;
    fc1.a2 = a2;
    fc1.a2_sf = a2_sf;
    fc1.err = err;
    fc1.interleaved = o.gate_up_layout == KT_GATE_UP_INTERLEAVED ? 1 : 0;
    fc1.activation = o.activation;
    fc1.alpha = o.alpha;
    fc1.limit = o.limit;
    {
        StageTimer timer(KT_STAGE_FC1, s);
        if ((st = launch_gemm(fc1, s)) != KT_OK) return st;
    }

    GemmArgs fc2{};
    fc2.mode = GemmEpilogue::Combine;
    fc2.expert_offsets = offsets;
    fc2.chunk_prefix = chunk_prefix;
    fc2.E = E;
    fc2.K = I;
    fc2.rows_w = H;
    fc2.I = I;
    fc2.S = static_cast<int>(S);
    fc2.H = H;
    fc2.w = w2;
    fc2.w_sf = w2_sf;
    fc2.act = a2;
    fc2.act_sf = a2_sf;
    fc2.y = y;
    fc2.perm = perm;
    fc2.topk_w = topk_w;
    fc2.err = err;
    {
        StageTimer timer(KT_STAGE_FC2, s);
        if ((st = launch_gemm(fc2, s)) != KT_OK) return st;
    }
    StageTimer timer(KT_STAGE_COMBINE, s);
    return cuda_status(launch_combine(y, topk_ids, T, H, k, E, out, s));
}

kt_status kt_mxfp4_moe_forward_ex(const uint16_t* hidden, int T, int H, const int32_t* topk_ids,
                                  const float* topk_w, int k, const uint8_t* w13, const uint8_t* w13_sf,
                                  const uint8_t* w2, const uint8_t* w2_sf, int E, int I, uint16_t* out, void* ws,
                                  size_t ws_bytes, const kt_moe_options* opts, void* stream) {
    return forward_impl(hidden, T, H, topk_ids, topk_w, k, false, nullptr, nullptr, nullptr, w13, w13_sf, w2, w2_sf,
                        E, I, out, ws, ws_bytes, opts, stream);
}

kt_status kt_mxfp4_moe_forward_routed(const uint16_t* hidden, int T, int H, const int32_t* topk_ids,
                                      const float* topk_w, int k, const int32_t* expert_offsets, const int32_t* perm,
                                      const int32_t* inv_perm, const uint8_t* w13, const uint8_t* w13_sf,
                                      const uint8_t* w2, const uint8_t* w2_sf, int E, int I, uint16_t* out, void* ws,
                                      size_t ws_bytes, const kt_moe_options* opts, void* stream) {
    return forward_impl(hidden, T, H, topk_ids, topk_w, k, true, expert_offsets, perm, inv_perm, w13, w13_sf, w2,
                        w2_sf, E, I, out, ws, ws_bytes, opts, stream);
}

kt_status kt_mxfp4_moe_decode(const float* logits, const uint16_t* hidden, int T, int H, int E, int k, int I,
                              int renormalize, const uint8_t* w13, const uint8_t* w13_sf, const uint8_t* w2,
                              const uint8_t* w2_sf, int32_t* topk_ids, float* topk_w, uint16_t* out, void* ws,
                              size_t ws_bytes, const kt_moe_options* opts, void* stream) {
    g_last_error[0] = '\0';
    kt_moe_options o{KT_GATE_UP_HALVES, KT_ACT_SWIGLU, 1.0f, 0.0f};
    if (opts) o = *opts;
    if (o.gate_up_layout != KT_GATE_UP_HALVES && o.gate_up_layout != KT_GATE_UP_INTERLEAVED)
        return fail(KT_ERR_INVALID_ARG, "gate_up_layout=%d is not a KT_GATE_UP_* value", o.gate_up_layout);
    if (o.activation != KT_ACT_SWIGLU && o.activation != KT_ACT_SWIGLU_CLAMPED)
        return fail(KT_ERR_INVALID_ARG, "activation=%d is not a KT_ACT_* value", o.activation);
    if (o.activation == KT_ACT_SWIGLU_CLAMPED &&
        !(std::isfinite(o.alpha) && std::isfinite(o.limit) && o.limit > 0.0f))
        return fail(KT_ERR_INVALID_ARG, "clamped SwiGLU needs a finite alpha and a finite limit > 0");
    kt_status st = check_route_shape(T, E, k);
    if (st != KT_OK) return st;
    if (H <= 0 || I <= 0) return fail(KT_ERR_INVALID_ARG, "H=%d and I=%d must be positive", H, I);
    if (H % 128 || I % 128)
        return fail(KT_ERR_UNSUPPORTED_SHAPE, "H=%d and I=%d must be multiples of 128", H, I);
    if (static_cast<long long>(E) * 2 * I > INT_MAX / 2 || static_cast<long long>(E) * H > INT_MAX / 2)
        return fail(KT_ERR_UNSUPPORTED_SHAPE, "E*2I or E*H too large");
    if (static_cast<long long>(T) * k > KT_DECODE_MAX_SLOTS)
        return fail(KT_ERR_UNSUPPORTED_SHAPE, "T*k=%lld slots above the decode kernel's %d",
                    static_cast<long long>(T) * k, KT_DECODE_MAX_SLOTS);
    if (T == 0) return KT_OK;
    if (!logits || !hidden || !topk_ids || !topk_w || !w13 || !w13_sf || !w2 || !w2_sf || !out || !ws)
        return fail(KT_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(logits, 4) || !aligned(hidden, 16) || !aligned(out, 16) || !aligned(topk_ids, 16) ||
        !aligned(topk_w, 16))
        return fail(KT_ERR_ALIGNMENT, "logits must be 4-byte and hidden, out, topk_ids, topk_w 16-byte aligned");
    if (!aligned(w13, 32) || !aligned(w2, 32))
        return fail(KT_ERR_ALIGNMENT, "w13 and w2 must be 32-byte aligned");
    if (!aligned(w13_sf, 16) || !aligned(w2_sf, 16))
        return fail(KT_ERR_ALIGNMENT, "w13_sf and w2_sf must be 16-byte aligned");
    kt_ws_layout L;
    ws_layout(T, H, I, E, k, &L);
    if (!aligned(ws, 256)) return fail(KT_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < L.total) return fail(KT_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, L.total);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    int* err = reinterpret_cast<int*>(base + L.err);
    int32_t* offsets = reinterpret_cast<int32_t*>(base + L.expert_offsets);
    int32_t* chunk_prefix = reinterpret_cast<int32_t*>(base + L.chunk_prefix);
    int32_t* perm = reinterpret_cast<int32_t*>(base + L.perm);
    const long long S = static_cast<long long>(T) * k;
    // the error word and the kernel's two grid counters share the 256-byte error region
    if ((st = cuda_status(cudaMemsetAsync(base + L.err, 0, 256, s))) != KT_OK) return st;

    GemmArgs fc1{};
    fc1.mode = GemmEpilogue::SwiGLU;
    fc1.expert_offsets = offsets;
    fc1.chunk_prefix = chunk_prefix;
    fc1.E = E;
    fc1.K = H;
    fc1.rows_w = 2 * I;
    fc1.I = I;
    fc1.S = static_cast<int>(S);
    fc1.H = H;
    fc1.w = w13;
    fc1.w_sf = w13_sf;
    fc1.act = base + L.a1;
    fc1.act_sf = base + L.a1_sf;
    fc1.a2 = base + L.a2;
    fc1.a2_sf = base + L.a2_sf;
    fc1.err = err;
    fc1.interleaved = o.gate_up_layout == KT_GATE_UP_INTERLEAVED ? 1 : 0;
    fc1.activation = o.activation;
    fc1.alpha = o.alpha;
    fc1.limit = o.limit;
    GemmArgs fc2{};
    fc2.mode = GemmEpilogue::Combine;
    fc2.expert_offsets = offsets;
    fc2.chunk_prefix = chunk_prefix;
    fc2.E = E;
    fc2.K = I;
    fc2.rows_w = H;
    fc2.I = I;
    fc2.S = static_cast<int>(S);
    fc2.H = H;
    fc2.w = w2;
    fc2.w_sf = w2_sf;
    fc2.act = base + L.a2;
    fc2.act_sf = base + L.a2_sf;
    fc2.y = reinterpret_cast<uint16_t*>(base + L.y);
    fc2.perm = perm;
    fc2.topk_w = topk_w;
    fc2.err = err;
    DecodeInputs in{};
    in.logits = logits;
    in.hidden = hidden;
    in.T = T;
    in.H = H;
    in.E = E;
    in.k = k;
    in.renormalize = renormalize ? 1 : 0;
    in.ids = topk_ids;
    in.w = topk_w;
    in.offsets = offsets;
    in.chunk_prefix = chunk_prefix;
    in.perm = perm;
    in.inv_perm = reinterpret_cast<int32_t*>(base + L.inv_perm);
    in.a1 = base + L.a1;
    in.a1_sf = base + L.a1_sf;
    in.y = reinterpret_cast<const uint16_t*>(base + L.y);
    in.out = out;
    in.grid_ctr = reinterpret_cast<unsigned*>(base + L.err + 64);
    in.fc1_done = reinterpret_cast<unsigned*>(base + L.err + 128);
    return launch_decode(fc1, fc2, in, s);
}

kt_status kt_moe_read_device_error(const void* ws, int* code, void* stream) {
    g_last_error[0] = '\0';
    if (!ws || !code) return fail(KT_ERR_INVALID_ARG, "null pointer argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kt_status st = cuda_status(cudaStreamSynchronize(s));
    if (st != KT_OK) return st;
    int v = 0;
    if ((st = cuda_status(cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost))) != KT_OK) return st;
    *code = v;
    if (v & (KT_DEVERR_TIMEOUT_LOAD | KT_DEVERR_TIMEOUT_MMA | KT_DEVERR_TIMEOUT_EPI | KT_DEVERR_TIMEOUT_GRID))
        return fail(KT_ERR_DEVICE_TIMEOUT, "device error word 0x%x", v);
    if (v & KT_DEVERR_BAD_EXPERT_ID) return fail(KT_ERR_BAD_EXPERT_ID, "device error word 0x%x", v);
    return KT_OK;
}

// error word | chunk prefix [E+1] | K-step-major scales | activation codes padded to act_rows(S) rows
size_t kt_mx_gemm_workspace_bytes(int S, int K, int E) {
    if (S < 0 || K <= 0 || K % 128 || E <= 0 || E > kMaxExperts) return 0;
    return 1024 + align_up(sizeof(int32_t) * (E + 1), 1024) +
           align_up(static_cast<size_t>(sf_rows(S)) * (K / 32), 1024) +
           align_up(static_cast<size_t>(act_rows(S)) * K, 1024);
}

kt_status kt_mx_grouped_gemm_f32(const uint8_t* act, const uint8_t* act_sf, int S, int K,
                                 const int32_t* expert_offsets, const uint8_t* w, const uint8_t* w_sf, int E, int N,
                                 float* out, void* ws, size_t ws_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (S < 0 || K <= 0 || N <= 0 || E <= 0) return fail(KT_ERR_INVALID_ARG, "invalid sizes");
    if (K % 128 || N % 128) return fail(KT_ERR_UNSUPPORTED_SHAPE, "K=%d and N=%d must be multiples of 128", K, N);
    if (E > kMaxExperts) return fail(KT_ERR_UNSUPPORTED_SHAPE, "E=%d above the supported %d", E, kMaxExperts);
    if (S == 0) return KT_OK;
    if (!act || !act_sf || !expert_offsets || !w || !w_sf || !out || !ws)
        return fail(KT_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(act, 16) || !aligned(w, 32) || !aligned(act_sf, 4) || !aligned(w_sf, 4) || !aligned(out, 16))
        return fail(KT_ERR_ALIGNMENT, "misaligned pointer");
    if (!aligned(ws, 256)) return fail(KT_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < kt_mx_gemm_workspace_bytes(S, K, E)) return fail(KT_ERR_WORKSPACE, "workspace too small");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(ws);
    int* err = reinterpret_cast<int*>(base);
    int32_t* chunk_prefix = reinterpret_cast<int32_t*>(base + 1024);
    uint8_t* sf_km = base + 1024 + align_up(sizeof(int32_t) * (E + 1), 1024);
    uint8_t* act_pad = sf_km + align_up(static_cast<size_t>(sf_rows(S)) * (K / 32), 1024);
    kt_status st;
    if ((st = cuda_status(cudaMemsetAsync(err, 0, sizeof(int), s))) != KT_OK) return st;
    if ((st = cuda_status(cudaMemcpyAsync(act_pad, act, static_cast<size_t>(S) * K, cudaMemcpyDeviceToDevice, s))) !=
        KT_OK)
        return st;
    if ((st = cuda_status(launch_chunk_prefix(expert_offsets, E, chunk_prefix, s))) != KT_OK) return st;
    if ((st = cuda_status(launch_sf_to_kstep_major(act_sf, S, K, sf_km, sf_rows(S), s))) != KT_OK) return st;
    GemmArgs g{};
    g.mode = GemmEpilogue::Raw;
    g.expert_offsets = expert_offsets;
    g.chunk_prefix = chunk_prefix;
    g.E = E;
    g.K = K;
    g.rows_w = N;
    g.I = 0;
    g.S = S;
    g.H = 0;
    g.w = w;
    g.w_sf = w_sf;
    g.act = act_pad;
    g.act_sf = sf_km;
    g.raw_out = out;
    g.err = err;
    return launch_gemm(g, s);
}

}  // extern "C"
