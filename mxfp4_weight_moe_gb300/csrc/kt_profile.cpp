// kt_profile.cpp -- measurement hooks: a process-wide kernel launch counter
// and optional per-stage CUDA event records on the caller's stream.
#include <atomic>
#include <vector>

#include <cuda_runtime.h>

#include "kt_internal.h"

namespace kt {

static std::atomic<uint64_t> g_launches{0};
static std::atomic<uint64_t> g_wait_limit_ns{0};
static std::atomic<int> g_debug_flags{0};

DebugSettings debug_settings() {
    const uint64_t lim = g_wait_limit_ns.load();
    return {lim ? lim : 2000000000ull, g_debug_flags.load()};
}

void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

struct StageRecord {
    int stage;
    cudaEvent_t begin, end;
};

static bool g_prof_on = false;
static uint32_t g_prof_mask = 0;   // bit s: record stage s
static std::vector<StageRecord> g_records;
static std::vector<cudaEvent_t> g_pool;
static size_t g_pool_used = 0;

static cudaEvent_t take_event() {
    if (g_pool_used == g_pool.size()) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_pool.push_back(e);
    }
    return g_pool[g_pool_used++];
}

StageTimer::StageTimer(int stage, cudaStream_t s) : stage_(stage), s_(s), end_(nullptr) {
    if (!g_prof_on || !((g_prof_mask >> stage) & 1u)) return;
    cudaEvent_t b = take_event();
    end_ = take_event();
    if (!b || !end_) {
        end_ = nullptr;
        return;
    }
    cudaEventRecord(b, s_);
    g_records.push_back({stage_, b, end_});
}

StageTimer::~StageTimer() {
    if (end_) cudaEventRecord(end_, s_);
}

}  // namespace kt

extern "C" {

uint64_t kt_moe_kernel_launches(void) { return kt::g_launches.load(); }

kt_status kt_moe_debug_configure(uint64_t wait_limit_us, int flags) {
    if (flags & ~KT_DEBUG_WITHHOLD_STAGE) return KT_ERR_INVALID_ARG;
    kt::g_wait_limit_ns.store(wait_limit_us * 1000ull);
    kt::g_debug_flags.store(flags);
    return KT_OK;
}

kt_status kt_moe_profile_enable_stages(uint32_t stage_mask) {
    if (stage_mask >> KT_NUM_STAGES) return KT_ERR_INVALID_ARG;
    kt::g_prof_on = stage_mask != 0;
    kt::g_prof_mask = stage_mask;
    kt::g_records.clear();
    kt::g_pool_used = 0;
    return KT_OK;
}

kt_status kt_moe_profile_enable(int enable) {
    return kt_moe_profile_enable_stages(enable ? (1u << KT_NUM_STAGES) - 1u : 0u);
}

kt_status kt_moe_profile_read(double* stage_ms, int* calls) {
    if (!stage_ms || !calls) return KT_ERR_INVALID_ARG;
    for (int i = 0; i < KT_NUM_STAGES; ++i) {
        stage_ms[i] = 0.0;
        calls[i] = 0;
    }
    for (const auto& r : kt::g_records) {
        const cudaError_t e = cudaEventSynchronize(r.end);
        if (e != cudaSuccess) return kt::cuda_status(e);
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.begin, r.end) != cudaSuccess) continue;
        stage_ms[r.stage] += ms;
        calls[r.stage] += 1;
    }
    return KT_OK;
}

}  // extern "C"
