// kt_noalloc.cu -- routing + permutation with library-owned scratch, for
// callers that cannot allocate device memory (see kt_moe_route_permute_noalloc
// in kt_moe.h).  The scratch is a file-scope device array.  In host code the
// array's name is only a host-side stand-in, never a device address, so every
// call asks the runtime for the array's device address in the current
// device's context (cudaGetSymbolAddress, a host-side lookup) and hands that
// address to the same kernels kt_moe_route_permute launches.  Looking it up
// on every call, rather than caching it, keeps the address valid after the
// context is torn down and re-created (cudaDeviceReset) in the same process.
#include <cstdio>

#include "kt_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_route_scratch[KT_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" kt_status kt_moe_route_permute_noalloc(const float* logits, int T, int E, int k, int renormalize,
                                                  int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                                                  int32_t* perm, int32_t* inv_perm, void* stream) {
    // argument checks first (as kt_moe_route_permute orders them), then the size limit, before any GPU work
    kt_status st = kt::check_route_args(logits, T, E, k, topk_ids, topk_w, expert_offsets, perm, inv_perm);
    if (st != KT_OK || T == 0) return st;
    const size_t need = kt_moe_route_workspace_bytes(T, E, k);
    if (need > KT_NOALLOC_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "T=%d E=%d k=%d needs %zu bytes of routing scratch, above the %u-byte static scratch of "
                 "kt_moe_route_permute_noalloc; use kt_moe_route_permute with a workspace",
                 T, E, k, need, KT_NOALLOC_SCRATCH_BYTES);
        return kt::report(KT_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&scratch, g_route_scratch);
    if (e != cudaSuccess || scratch == nullptr) {
        cudaGetLastError();
        return kt::cuda_status(e == cudaSuccess ? cudaErrorInvalidSymbol : e);
    }
    return kt_moe_route_permute(logits, T, E, k, renormalize, topk_ids, topk_w, expert_offsets, perm, inv_perm,
                                scratch, KT_NOALLOC_SCRATCH_BYTES, stream);
}
