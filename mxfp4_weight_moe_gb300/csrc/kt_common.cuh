// kt_common.cuh -- sm_103a device helpers shared by the MoE kernels:
// mbarrier waits with deadlines, TMA tile loads, 4-byte cp.async gathers and
// the tcgen05 (5th-generation tensor core) instructions, all as inline PTX.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kt_moe.h"

namespace kt {

// Default longest any single barrier wait may take before the kernel gives
// up, records the failing role in the device error word and returns.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ launch chaining
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream still runs.
// griddep_wait() returns once the predecessor grid has completed and its
// memory is visible (at once for a kernel launched without that attribute),
// so every kernel calls it before its first global-memory access;
// griddep_launch_dependents() then lets the next kernel start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One bounded try_wait: the thread may suspend until the phase completes, for
// at most kMbarSuspendNs.  Measured on GB300: without the hint (a system-
// dependent suspend limit) the GEMM's stage loop ran 7 % slower on the
// Kimi-K3-shaped and DeepSeek-V4-shaped layers than with any hint from 16 to
// 256 ns, so a waiter evidently does not always resume as soon as the TMA
// bytes or the tcgen05.commit land.
constexpr uint32_t kMbarSuspendNs = 64;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2, %3;\n\t"
        "selp.b32 %0, 1, 0, P1;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(kMbarSuspendNs)
        : "memory");
    return ok != 0;
}

// Wait for the phase with parity `parity` to complete.  Returns false when
// the deadline passes or another role of the CTA raised *abort_flag; the
// barrier's state is then left as is and the caller must wind down.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    uint32_t it = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++it & 15u) == 0u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ TMA / cp.async
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA load of one box at element coordinates (x, y) into shared
// memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 4-byte global -> shared copy; src_bytes = 0 writes zeros (no global read).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Arrive on `bar` once all of this thread's earlier cp.async copies landed
// (counts against the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// Copy a 32-row x 128-bit shared-memory block into tensor memory, replicated
// into all four 32-lane quadrants (the layout block scale factors use).
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// D[tmem] (+)= A[smem] x B[smem]^T with per-32 e8m0 block scales from tmem.
__device__ __forceinline__ void tc_mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred P1;\n\t"
        "setp.ne.b32 P1, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], P1;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// Each thread of the warp reads 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): K-major operand in the
// 128-byte swizzle layout, 8-row groups 1024 bytes apart.  The tile base must
// be 1024-byte aligned; advancing along K inside the 128-byte row is done by
// adding the byte offset to the start address.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);          // bits 0-13  start address >> 4
    d |= static_cast<uint64_t>(16u >> 4) << 16;                    // bits 16-29 leading byte offset (unused)
    d |= static_cast<uint64_t>(1024u >> 4) << 32;                  // bits 32-45 stride byte offset
    d |= static_cast<uint64_t>(1u) << 46;                          // bits 46-48 fixed 0b001
    d |= static_cast<uint64_t>(2u) << 61;                          // bits 61-63 swizzle: 128B
    return d;
}

// Descriptor of one 512-byte scale-factor block: 32 rows x 16 bytes, rows
// contiguous, no swizzle (four 8-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t sdesc_sf_block(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(16u >> 4) << 16;
    d |= static_cast<uint64_t>(128u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;
}

// Instruction descriptor of kind::mxf8f6f4 with A = e2m1, B = e4m3, fp32
// accumulate, e8m0 scales, both operands K-major, M = 128 and N = n
// (16 <= n <= 256, n % 16 == 0).  sf_id picks the byte of the 32-bit scale
// column (the 32-element block inside the 128-element K step).
__device__ __forceinline__ uint32_t idesc_mx_e2m1_e4m3(int n, uint32_t sf_id) {
    return (sf_id << 4)                             // bits 4-5   scale-factor B id
           | (5u << 7)                              // bits 7-9   A format: E2M1
           | (0u << 10)                             // bits 10-12 B format: E4M3
           | (static_cast<uint32_t>(n >> 3) << 17)  // bits 17-22 N >> 3
           | (1u << 23)                             // bit 23     scale type: UE8M0
           | ((128u >> 7) << 27)                    // bits 27-28 M >> 7
           | (sf_id << 29);                         // bits 29-30 scale-factor A id
}

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ uint8_t f32_to_e4m3_satfinite(float x) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
    return static_cast<uint8_t>(r & 0xFFu);
}

// Two floats -> two e4m3 codes packed as (lo = a, hi = b).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2_satfinite(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// MXFP8 shared exponent X of a block from the bit pattern of its (non-
// negative) amax: floor(log2 amax) - 8 clamped to [-127, 127]; a zero or
// subnormal amax gives -127.  Returns X; the scale byte is X + 127.
__device__ __forceinline__ int mx_e4m3_block_exponent(uint32_t amax_bits) {
    const int ef = static_cast<int>(amax_bits >> 23);
    if (ef == 0) return -127;
    const int x = ef - 127 - 8;
    return x < -127 ? -127 : x;   // ef <= 254 keeps x <= 119
}

// 2^-X as a float for X in [-127, 119] (always a normal number).
__device__ __forceinline__ float exp2_neg(int X) {
    return __uint_as_float(static_cast<uint32_t>(127 - X) << 23);
}

__device__ __forceinline__ void set_error(int* err, int bits) {
    if (err) atomicOr(err, bits);
}

}  // namespace kt
