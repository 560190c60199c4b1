// kt_layerwise.cpp -- single-GPU layerwise prefill: while layer l computes on
// the caller's stream, a copy stream uploads layer l+1's packed experts from
// pinned host memory into the other of two device slots.
//
// "[MXFP4 layerwise prefill] SM 8.6 (Ampere) excluded by capability
// whitelist", Impact: the fallback per layer uploads all 256 experts,
// computes, then synchronises before the next layer -- a serialised
// per-layer transfer chain; Background / motivation: a double-buffered
// layerwise prefill is what should hide that chain.  Both are implemented:
// serialized_control = 1 reproduces the chain as the measurement control,
// serialized_control = 0 double-buffers.  Events order the two streams:
//   copy(l+1) into slot (l+1)%2 waits for consumed[(l+1)%2] (layer l-1 done)
//   compute(l) waits for copied[l%2]
// Host-side waits poll with a deadline and return KT_ERR_TIMEOUT.
//
// Zero-copy mode (a GB300 node's Grace host memory is coherent with the GPU
// over NVLink-C2C): no device slots and no copies; each layer's GEMMs read
// its packed experts in place from the pinned host pack, through the host
// pack's device address.  Only host memory that this process pinned is
// read; nothing is multicast.
//
// Optional per-layer timing: events on the copy stream around each layer's
// copy and on the compute stream around each layer's compute, read back by
// kt_layerwise_read_timing.
#include <chrono>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include <cuda_runtime.h>

#include "kt_internal.h"

struct kt_layerwise {
    int L = 0, H = 0, I = 0, E = 0, k = 0, T_max = 0, dev = 0;
    std::vector<const void*> host_packs;
    size_t pack_bytes = 0, off_w13 = 0, off_w13_sf = 0, off_w2 = 0, off_w2_sf = 0;
    void* slot[2] = {nullptr, nullptr};
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t copied[2] = {nullptr, nullptr};
    cudaEvent_t consumed[2] = {nullptr, nullptr};
    void* ws = nullptr;
    size_t ws_bytes = 0;
    void* route_ws = nullptr;
    size_t route_ws_bytes = 0;
    uint16_t* hbuf[2] = {nullptr, nullptr};
    int32_t* ids = nullptr;
    float* w = nullptr;
    int32_t* offsets = nullptr;
    int32_t* perm = nullptr;
    int32_t* inv_perm = nullptr;
    int inject_layer = -1;
    int zero_copy = 0;
    std::vector<const void*> dev_packs;   // zero-copy: device addresses of the host packs
    bool timing = false;
    std::vector<cudaEvent_t> ev;          // timing: [copy_b, copy_e, comp_b, comp_e] per layer, then start
};

namespace {

constexpr double kHostWaitLimitS = 120.0;

kt_status wait_stream(cudaStream_t s) {
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t e = cudaStreamQuery(s);
        if (e == cudaSuccess) return KT_OK;
        if (e != cudaErrorNotReady) return kt::cuda_status(e);
        const double el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
        if (el > kHostWaitLimitS) return KT_ERR_TIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
}

void pack_offsets(int H, int I, int E, size_t* o13, size_t* o13s, size_t* o2, size_t* o2s, size_t* total) {
    size_t off = 0;
    auto take = [&](size_t b) {
        const size_t o = off;
        off = kt::align_up(off + b, 256);
        return o;
    };
    *o13 = take(static_cast<size_t>(E) * 2 * I * (H / 2));
    *o13s = take(static_cast<size_t>(E) * 2 * I * (H / 32));
    *o2 = take(static_cast<size_t>(E) * H * (I / 2));
    *o2s = take(static_cast<size_t>(E) * H * (I / 32));
    *total = off;
}

void free_timing(kt_layerwise* c) {
    for (cudaEvent_t e : c->ev)
        if (e) cudaEventDestroy(e);
    c->ev.clear();
}

void free_ctx(kt_layerwise* c) {
    if (!c) return;
    free_timing(c);
    for (int i = 0; i < 2; ++i) {
        if (c->slot[i]) cudaFree(c->slot[i]);
        if (c->hbuf[i]) cudaFree(c->hbuf[i]);
        if (c->copied[i]) cudaEventDestroy(c->copied[i]);
        if (c->consumed[i]) cudaEventDestroy(c->consumed[i]);
    }
    if (c->ws) cudaFree(c->ws);
    if (c->route_ws) cudaFree(c->route_ws);
    if (c->ids) cudaFree(c->ids);
    if (c->w) cudaFree(c->w);
    if (c->offsets) cudaFree(c->offsets);
    if (c->perm) cudaFree(c->perm);
    if (c->inv_perm) cudaFree(c->inv_perm);
    if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
    delete c;
}

}  // namespace

extern "C" {

size_t kt_layerwise_pack_bytes(int H, int I, int E) {
    if (H <= 0 || I <= 0 || E <= 0 || H % 128 || I % 128) return 0;
    size_t a, b, c, d, t;
    pack_offsets(H, I, E, &a, &b, &c, &d, &t);
    return t;
}

kt_status kt_layerwise_pack_offsets(int H, int I, int E, size_t* w13, size_t* w13_sf, size_t* w2, size_t* w2_sf) {
    if (!w13 || !w13_sf || !w2 || !w2_sf) return KT_ERR_INVALID_ARG;
    if (H <= 0 || I <= 0 || E <= 0) return KT_ERR_INVALID_ARG;
    if (H % 128 || I % 128) return KT_ERR_UNSUPPORTED_SHAPE;
    size_t t;
    pack_offsets(H, I, E, w13, w13_sf, w2, w2_sf, &t);
    return KT_OK;
}

static kt_status create_ctx(kt_layerwise** out, int L, int H, int I, int E, int k, int T_max,
                            const void* const* host_packs, int zero_copy) {
    if (!out || !host_packs || L <= 0 || T_max <= 0) return KT_ERR_INVALID_ARG;
    *out = nullptr;
    if (kt_moe_workspace_bytes(T_max, H, I, E, k) == 0) return KT_ERR_UNSUPPORTED_SHAPE;
    for (int l = 0; l < L; ++l)
        if (!host_packs[l]) return KT_ERR_INVALID_ARG;
    kt_layerwise* c = new (std::nothrow) kt_layerwise();
    if (!c) return KT_ERR_INVALID_ARG;
    c->host_packs.assign(host_packs, host_packs + L);
    c->L = L;
    c->H = H;
    c->I = I;
    c->E = E;
    c->k = k;
    c->T_max = T_max;
    c->inject_layer = -1;
    c->zero_copy = zero_copy ? 1 : 0;
    cudaGetDevice(&c->dev);
    pack_offsets(H, I, E, &c->off_w13, &c->off_w13_sf, &c->off_w2, &c->off_w2_sf, &c->pack_bytes);
    c->ws_bytes = kt_moe_workspace_bytes(T_max, H, I, E, k);
    c->route_ws_bytes = kt_moe_route_workspace_bytes(T_max, E, k);
    const size_t S = static_cast<size_t>(T_max) * k;
    bool ok = true;
    if (c->zero_copy) {
        // the device address of each pinned host pack (fails for memory that is not pinned)
        for (int l = 0; l < L && ok; ++l) {
            void* d = nullptr;
            const cudaError_t e = cudaHostGetDevicePointer(&d, const_cast<void*>(host_packs[l]), 0);
            if (e != cudaSuccess || d == nullptr || (reinterpret_cast<uintptr_t>(d) & 255u) != 0) {
                cudaGetLastError();
                free_ctx(c);
                return kt::report(KT_ERR_INVALID_ARG,
                                  "zero-copy layerwise needs pinned, device-mapped, 256-byte aligned host packs");
            }
            c->dev_packs.push_back(d);
        }
    }
    for (int i = 0; i < 2 && ok; ++i) {
        if (!c->zero_copy) ok = ok && cudaMalloc(&c->slot[i], c->pack_bytes) == cudaSuccess;
        ok = ok && cudaMalloc(reinterpret_cast<void**>(&c->hbuf[i]), sizeof(uint16_t) * T_max * H) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->copied[i], cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->consumed[i], cudaEventDisableTiming) == cudaSuccess;
    }
    ok = ok && cudaMalloc(&c->ws, c->ws_bytes) == cudaSuccess;
    ok = ok && cudaMalloc(&c->route_ws, c->route_ws_bytes) == cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void**>(&c->ids), sizeof(int32_t) * S) == cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void**>(&c->w), sizeof(float) * S) == cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void**>(&c->offsets), sizeof(int32_t) * (E + 1)) == cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void**>(&c->perm), sizeof(int32_t) * S) == cudaSuccess;
    ok = ok && cudaMalloc(reinterpret_cast<void**>(&c->inv_perm), sizeof(int32_t) * S) == cudaSuccess;
    ok = ok && cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking) == cudaSuccess;
    if (!ok) {
        const cudaError_t e = cudaGetLastError();
        free_ctx(c);
        return kt::cuda_status(e == cudaSuccess ? cudaErrorMemoryAllocation : e);
    }
    *out = c;
    return KT_OK;
}

kt_status kt_layerwise_create(kt_layerwise** out, int L, int H, int I, int E, int k, int T_max,
                              const void* const* host_packs) {
    return create_ctx(out, L, H, I, E, k, T_max, host_packs, 0);
}

kt_status kt_layerwise_create_zero_copy(kt_layerwise** out, int L, int H, int I, int E, int k, int T_max,
                                        const void* const* host_packs) {
    return create_ctx(out, L, H, I, E, k, T_max, host_packs, 1);
}

kt_status kt_layerwise_enable_timing(kt_layerwise* c, int enable) {
    if (!c) return KT_ERR_INVALID_ARG;
    free_timing(c);
    c->timing = false;
    if (!enable) return KT_OK;
    c->ev.assign(static_cast<size_t>(4 * c->L + 1), nullptr);
    for (auto& e : c->ev) {
        if (cudaEventCreate(&e) != cudaSuccess) {
            const cudaError_t err = cudaGetLastError();
            free_timing(c);
            return kt::cuda_status(err);
        }
    }
    c->timing = true;
    return KT_OK;
}

kt_status kt_layerwise_read_timing(kt_layerwise* c, double* copy_ms, double* compute_ms, double* span_ms) {
    if (!c || !copy_ms || !compute_ms || !span_ms) return KT_ERR_INVALID_ARG;
    if (!c->timing) return kt::report(KT_ERR_INVALID_ARG, "timing is not enabled");
    kt_status st;
    const cudaEvent_t start = c->ev[4 * c->L];
    float last = 0.f;
    for (int l = 0; l < c->L; ++l) {
        float a = 0.f, b = 0.f, e_end = 0.f;
        if ((st = kt::cuda_status(cudaEventSynchronize(c->ev[4 * l + 3]))) != KT_OK) return st;
        if (c->zero_copy) {
            copy_ms[l] = 0.0;
        } else {
            if ((st = kt::cuda_status(cudaEventElapsedTime(&a, c->ev[4 * l], c->ev[4 * l + 1]))) != KT_OK) return st;
            copy_ms[l] = a;
        }
        if ((st = kt::cuda_status(cudaEventElapsedTime(&b, c->ev[4 * l + 2], c->ev[4 * l + 3]))) != KT_OK) return st;
        compute_ms[l] = b;
        if ((st = kt::cuda_status(cudaEventElapsedTime(&e_end, start, c->ev[4 * l + 3]))) != KT_OK) return st;
        if (e_end > last) last = e_end;
    }
    *span_ms = last;
    return KT_OK;
}

kt_status kt_layerwise_inject_copy_failure(kt_layerwise* c, int layer) {
    if (!c) return KT_ERR_INVALID_ARG;
    c->inject_layer = layer;
    return KT_OK;
}

static kt_status enqueue_copy(kt_layerwise* c, int l, cudaStream_t s, bool wait_consumed) {
    if (l == c->inject_layer) return KT_ERR_CUDA;   // test hook: the copy step of this layer fails
    const int b = l & 1;
    kt_status st;
    if (wait_consumed && (st = kt::cuda_status(cudaStreamWaitEvent(s, c->consumed[b], 0))) != KT_OK) return st;
    if (c->timing && (st = kt::cuda_status(cudaEventRecord(c->ev[4 * l], s))) != KT_OK) return st;
    if ((st = kt::cuda_status(cudaMemcpyAsync(c->slot[b], c->host_packs[l], c->pack_bytes, cudaMemcpyHostToDevice,
                                              s))) != KT_OK)
        return st;
    if (c->timing && (st = kt::cuda_status(cudaEventRecord(c->ev[4 * l + 1], s))) != KT_OK) return st;
    return kt::cuda_status(cudaEventRecord(c->copied[b], s));
}

static kt_status compute_layer(kt_layerwise* c, int l, const uint16_t* in, const float* logits, uint16_t* outp,
                               int T, cudaStream_t s) {
    const int b = l & 1;
    const uint8_t* base = static_cast<const uint8_t*>(c->zero_copy ? c->dev_packs[l] : c->slot[b]);
    kt_status st;
    if (c->timing && (st = kt::cuda_status(cudaEventRecord(c->ev[4 * l + 2], s))) != KT_OK) return st;
    st = kt_moe_route_permute(logits, T, c->E, c->k, 1, c->ids, c->w, c->offsets, c->perm, c->inv_perm,
                                        c->route_ws, c->route_ws_bytes, s);
    if (st != KT_OK) return st;
    st = kt_mxfp4_moe_forward(in, T, c->H, c->ids, c->w, c->k, base + c->off_w13, base + c->off_w13_sf,
                              base + c->off_w2, base + c->off_w2_sf, c->E, c->I, outp, c->ws, c->ws_bytes, s);
    if (st == KT_OK && c->timing) st = kt::cuda_status(cudaEventRecord(c->ev[4 * l + 3], s));
    return st;
}

kt_status kt_layerwise_prefill(kt_layerwise* c, const uint16_t* hidden, const float* const* logits, uint16_t* out,
                               int T, int serialized_control, void* stream) {
    if (!c || !hidden || !logits || !out || T < 0 || T > c->T_max) return KT_ERR_INVALID_ARG;
    for (int l = 0; l < c->L; ++l)
        if (!logits[l]) return KT_ERR_INVALID_ARG;
    if (T == 0) return KT_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kt_status st = KT_OK;
    if (c->timing) {
        // the copy stream's first copy and the compute stream's first layer both follow this event
        st = kt::cuda_status(cudaEventRecord(c->ev[4 * c->L], s));
        if (st == KT_OK && !c->zero_copy) st = kt::cuda_status(cudaStreamWaitEvent(c->copy_stream, c->ev[4 * c->L], 0));
        if (st != KT_OK) return st;
    }
    for (int l = 0; l < c->L && st == KT_OK; ++l) {
        const uint16_t* in = (l == 0) ? hidden : c->hbuf[(l - 1) & 1];
        uint16_t* o = (l == c->L - 1) ? out : c->hbuf[l & 1];
        if (c->zero_copy) {
            // the GEMMs read the layer's experts in place: no copy and no slot to wait for
            if (l == c->inject_layer) st = KT_ERR_CUDA;
            if (st == KT_OK) st = compute_layer(c, l, in, logits[l], o, T, s);
            if (st == KT_OK && serialized_control) st = wait_stream(s);
        } else if (serialized_control) {
            // upload all experts -> compute -> synchronise, one layer at a time
            st = enqueue_copy(c, l, s, false);
            if (st == KT_OK) st = compute_layer(c, l, in, logits[l], o, T, s);
            if (st == KT_OK) st = wait_stream(s);
        } else {
            if (l == 0) st = enqueue_copy(c, 0, c->copy_stream, true);
            if (st == KT_OK && l + 1 < c->L) st = enqueue_copy(c, l + 1, c->copy_stream, true);
            if (st == KT_OK) st = kt::cuda_status(cudaStreamWaitEvent(s, c->copied[l & 1], 0));
            if (st == KT_OK) st = compute_layer(c, l, in, logits[l], o, T, s);
            if (st == KT_OK) st = kt::cuda_status(cudaEventRecord(c->consumed[l & 1], s));
        }
    }
    if (st != KT_OK) {
        // drain both streams so no copy or kernel is left in flight
        wait_stream(c->copy_stream);
        wait_stream(s);
    }
    return st;
}

kt_status kt_layerwise_destroy(kt_layerwise* c) {
    if (!c) return KT_ERR_INVALID_ARG;
    cudaSetDevice(c->dev);
    wait_stream(c->copy_stream);
    free_ctx(c);
    return KT_OK;
}

}  // extern "C"
