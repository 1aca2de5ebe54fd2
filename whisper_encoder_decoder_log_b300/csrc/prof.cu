// Per-kernel timing: when enabled for a kernel kind, every launch of that kind
// is bracketed by CUDA events on its own stream, and the launch's algorithmic
// work (bytes for the memory-bound kernels, flops for the contractions) is
// summed, so a caller can report achieved bandwidth or throughput of the kernel
// inside a longer timed region.
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"
#include "prof.cuh"

namespace wb {
namespace {

struct ProfState {
    std::mutex mu;
    int kind = 0;
    std::vector<cudaEvent_t> pool;      // start/stop pairs
    size_t used = 0;
    double units = 0.0;
    int64_t launches = 0;
};
ProfState g_prof;
std::atomic<int64_t> g_launches{0};

}  // namespace

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool prof_active(int kind) { return g_prof.kind != 0 && g_prof.kind == kind; }
bool prof_any_active() { return g_prof.kind != 0; }

int prof_begin(int kind, cudaStream_t s) {
    if (!prof_active(kind)) return -1;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (g_prof.used + 2 > g_prof.pool.size()) return -1;
    const int slot = (int)g_prof.used;
    g_prof.used += 2;
    cudaEventRecord(g_prof.pool[slot], s);
    return slot;
}

void prof_end(int slot, cudaStream_t s, double units) {
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    cudaEventRecord(g_prof.pool[slot + 1], s);
    g_prof.units += units;
    g_prof.launches += 1;
}

}  // namespace wb

using namespace wb;

extern "C" {

wb_status wb_prof_start(int32_t kind, int32_t max_launches) {
    if (kind < 0 || kind > WB_KERNEL_MAX) return fail(WB_ERR_INVALID_ARG, "wb_prof_start: bad kind");
    if (max_launches < 1 || max_launches > (1 << 20)) return fail(WB_ERR_SHAPE, "wb_prof_start: bad max_launches");
    std::lock_guard<std::mutex> lk(g_prof.mu);
    for (cudaEvent_t e : g_prof.pool) cudaEventDestroy(e);
    g_prof.pool.assign((size_t)max_launches * 2, nullptr);
    for (auto& e : g_prof.pool) WB_CUDA(cudaEventCreate(&e));
    g_prof.used = 0;
    g_prof.units = 0.0;
    g_prof.launches = 0;
    g_prof.kind = kind;
    return WB_OK;
}

int64_t wb_launch_count(void) { return g_launches.load(); }

wb_status wb_prof_stop(int64_t* launches, double* total_ms, double* units) {
    if (!launches || !total_ms || !units) return fail(WB_ERR_INVALID_ARG, "wb_prof_stop: null argument");
    std::lock_guard<std::mutex> lk(g_prof.mu);
    double ms = 0.0;
    for (size_t i = 0; i + 1 < g_prof.used; i += 2) {
        WB_CUDA(cudaEventSynchronize(g_prof.pool[i + 1]));
        float t = 0.f;
        WB_CUDA(cudaEventElapsedTime(&t, g_prof.pool[i], g_prof.pool[i + 1]));
        ms += t;
    }
    *launches = g_prof.launches;
    *total_ms = ms;
    *units = g_prof.units;
    g_prof.kind = 0;
    for (cudaEvent_t e : g_prof.pool) cudaEventDestroy(e);
    g_prof.pool.clear();
    g_prof.used = 0;
    return WB_OK;
}

}  // extern "C"
