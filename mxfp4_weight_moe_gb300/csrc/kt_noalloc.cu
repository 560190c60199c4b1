// kt_noalloc.cu -- routing + permutation with library-owned scratch, for
// callers that cannot allocate device memory (see kt_moe_route_permute_noalloc
// in kt_moe.h).  The scratch is a file-scope device array; host code gets its
// device address once per device with cudaGetSymbolAddress (the array's name
// in host code is only a host-side stand-in, never a device address) and
// hands that address to the same kernels kt_moe_route_permute launches.
#include <cstdio>
#include <mutex>

#include "kt_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_route_scratch[KT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (looked up once per
// device); nullptr and the CUDA status on failure.
void* scratch_address(kt_status* st) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = kt::cuda_status(e);
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *st = KT_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess || p == nullptr) {
            *st = kt::cuda_status(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    *st = KT_OK;
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" kt_status kt_moe_route_permute_noalloc(const float* logits, int T, int E, int k, int renormalize,
                                                  int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                                                  int32_t* perm, int32_t* inv_perm, void* stream) {
    // The size limit is checked before anything touches the GPU.
    if (T > 0 && E > 0 && k > 0) {
        const size_t need = kt_moe_route_workspace_bytes(T, E, k);
        if (need > KT_NOALLOC_SCRATCH_BYTES) {
            char msg[256];
            snprintf(msg, sizeof(msg),
                     "T=%d E=%d k=%d needs %zu bytes of routing scratch, above the %u-byte static scratch of "
                     "kt_moe_route_permute_noalloc; use kt_moe_route_permute with a workspace",
                     T, E, k, need, KT_NOALLOC_SCRATCH_BYTES);
            return kt::report(KT_ERR_WORKSPACE, msg);
        }
    }
    if (T <= 0 || E <= 0 || k <= 0 || kt_moe_route_workspace_bytes(T, E, k) == 0)
        return kt_moe_route_permute(logits, T, E, k, renormalize, topk_ids, topk_w, expert_offsets, perm, inv_perm,
                                    nullptr, 0, stream);   // argument errors / T == 0, nothing launched
    kt_status st;
    void* scratch = scratch_address(&st);
    if (!scratch) return st;
    return kt_moe_route_permute(logits, T, E, k, renormalize, topk_ids, topk_w, expert_offsets, perm, inv_perm,
                                scratch, KT_NOALLOC_SCRATCH_BYTES, stream);
}
