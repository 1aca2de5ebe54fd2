// Per-kernel timing hooks (prof.cu).
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace wb {

bool prof_active(int kind);
bool prof_any_active();
// Returns a slot (>= 0) when launches of `kind` are being timed.
int prof_begin(int kind, cudaStream_t s);
// Closes the slot; `units` is the launch's algorithmic bytes or flops.
void prof_end(int slot, cudaStream_t s, double units);
// Counts kernel launches (wb_launch_count).
void count_launch(int n = 1);

}  // namespace wb
