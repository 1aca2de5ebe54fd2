// Per-kernel timing hooks (prof.cu).
#pragma once

#include <cuda_runtime.h>

#include <utility>

#include "internal.h"

namespace wb {

bool prof_active(int kind);
bool prof_any_active();
// Returns a slot (>= 0) when launches of `kind` are being timed.
int prof_begin(int kind, cudaStream_t s);
// Closes the slot; `units` is the launch's algorithmic bytes or flops.
void prof_end(int slot, cudaStream_t s, double units);
// The attention work of a continuous-batching decode step: the share of its
// rows that hold an active chunk (the others read nothing) and the cache rows
// those attend, summed over the rows (each row has its own position); set
// by the caller around such a step, (1, -1: one position for all) otherwise.
void prof_set_rows(double share, double cached_rows);
double prof_row_share();
double prof_cached_rows();
// Counts kernel launches (wb_launch_count).
void count_launch(int n = 1);

// Programmatic dependent launch: every kernel of the library begins with
// griddep_wait() before it reads what an earlier kernel wrote, so the next
// kernel's launch and prologue may overlap the tail of the previous one.
// Off when the environment sets WB_NO_PDL=1.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    count_launch();
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same with a cluster of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_k_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             int cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    count_launch();
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace wb
