// Per-kernel timing: when enabled for a kernel kind, every launch of that kind
// is bracketed by CUDA events on its own stream, and the launch's algorithmic
// work (bytes for the memory-bound kernels, flops for the contractions) is
// summed, so a caller can report achieved bandwidth or throughput of the kernel
// inside a longer timed region.
#include <atomic>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "internal.h"
#include "prof.cuh"

namespace wb {
namespace {

struct ProfState {
    std::mutex mu;
    int kind = 0;                       // 0: off, -1: every kind
    std::vector<cudaEvent_t> pool;      // start/stop pairs
    std::vector<int> slot_kind;
    size_t used = 0;
    double units[WB_KERNEL_MAX + 1] = {};
    int64_t launches[WB_KERNEL_MAX + 1] = {};
    double res_ms[WB_KERNEL_MAX + 1] = {};
    double res_units[WB_KERNEL_MAX + 1] = {};
    int64_t res_launches[WB_KERNEL_MAX + 1] = {};
};
ProfState g_prof;
std::atomic<int64_t> g_launches{0};

}  // namespace

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool pdl_enabled() {
    static const bool on = [] {
        const char* e = getenv("WB_NO_PDL");
        return !(e && e[0] == '1');
    }();
    return on;
}

bool prof_active(int kind) { return g_prof.kind != 0 && (g_prof.kind == kind || g_prof.kind == -1); }
bool prof_any_active() { return g_prof.kind != 0; }

namespace {
thread_local double t_row_share = 1.0;
thread_local double t_cached_rows = -1.0;
}
void prof_set_rows(double share, double cached_rows) {
    t_row_share = share;
    t_cached_rows = cached_rows;
}
double prof_row_share() { return t_row_share; }
double prof_cached_rows() { return t_cached_rows; }

int prof_begin(int kind, cudaStream_t s) {
    if (!prof_active(kind)) return -1;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (g_prof.used + 2 > g_prof.pool.size()) return -1;
    const int slot = (int)g_prof.used;
    g_prof.used += 2;
    g_prof.slot_kind[slot / 2] = kind;
    cudaEventRecord(g_prof.pool[slot], s);
    return slot;
}

void prof_end(int slot, cudaStream_t s, double units) {
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    cudaEventRecord(g_prof.pool[slot + 1], s);
    const int k = g_prof.slot_kind[slot / 2];
    g_prof.units[k] += units;
    g_prof.launches[k] += 1;
}

}  // namespace wb

using namespace wb;

extern "C" {

wb_status wb_prof_start(int32_t kind, int32_t max_launches) {
    if (kind < 0 || kind > WB_KERNEL_MAX) return fail(WB_ERR_INVALID_ARG, "wb_prof_start: bad kind");
    if (kind == 0) kind = -1;   // every kind
    if (max_launches < 1 || max_launches > (1 << 20)) return fail(WB_ERR_SHAPE, "wb_prof_start: bad max_launches");
    std::lock_guard<std::mutex> lk(g_prof.mu);
    for (cudaEvent_t e : g_prof.pool) cudaEventDestroy(e);
    g_prof.pool.assign((size_t)max_launches * 2, nullptr);
    for (auto& e : g_prof.pool) WB_CUDA(cudaEventCreate(&e));
    g_prof.slot_kind.assign((size_t)max_launches, 0);
    g_prof.used = 0;
    for (int k = 0; k <= WB_KERNEL_MAX; ++k) { g_prof.units[k] = 0.0; g_prof.launches[k] = 0; }
    g_prof.kind = kind;
    return WB_OK;
}

int64_t wb_launch_count(void) { return g_launches.load(); }

wb_status wb_prof_result(int32_t kind, int64_t* launches, double* total_ms, double* units) {
    if (kind < 1 || kind > WB_KERNEL_MAX || !launches || !total_ms || !units)
        return fail(WB_ERR_INVALID_ARG, "wb_prof_result: bad argument");
    std::lock_guard<std::mutex> lk(g_prof.mu);
    *launches = g_prof.res_launches[kind];
    *total_ms = g_prof.res_ms[kind];
    *units = g_prof.res_units[kind];
    return WB_OK;
}

wb_status wb_prof_stop(int64_t* launches, double* total_ms, double* units) {
    if (!launches || !total_ms || !units) return fail(WB_ERR_INVALID_ARG, "wb_prof_stop: null argument");
    std::lock_guard<std::mutex> lk(g_prof.mu);
    double ms[WB_KERNEL_MAX + 1] = {};
    for (size_t i = 0; i + 1 < g_prof.used; i += 2) {
        WB_CUDA(cudaEventSynchronize(g_prof.pool[i + 1]));
        float t = 0.f;
        WB_CUDA(cudaEventElapsedTime(&t, g_prof.pool[i], g_prof.pool[i + 1]));
        ms[g_prof.slot_kind[i / 2]] += t;
    }
    *launches = 0;
    *total_ms = 0.0;
    *units = 0.0;
    for (int k = 0; k <= WB_KERNEL_MAX; ++k) {
        g_prof.res_ms[k] = ms[k];
        g_prof.res_units[k] = g_prof.units[k];
        g_prof.res_launches[k] = g_prof.launches[k];
        *launches += g_prof.launches[k];
        *total_ms += ms[k];
        *units += g_prof.units[k];
    }
    g_prof.kind = 0;
    for (cudaEvent_t e : g_prof.pool) cudaEventDestroy(e);
    g_prof.pool.clear();
    g_prof.used = 0;
    return WB_OK;
}

}  // extern "C"
