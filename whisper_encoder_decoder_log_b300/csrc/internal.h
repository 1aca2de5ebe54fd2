// Internal host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/wb.h"

namespace wb {

// Thread-local error text, set by every failing entry point.
void set_error(const std::string& msg);
wb_status fail(wb_status code, const std::string& msg);
wb_status cuda_fail(cudaError_t e, const char* what);

#define WB_CUDA(call)                                              \
    do {                                                           \
        cudaError_t e_ = (call);                                   \
        if (e_ != cudaSuccess) return ::wb::cuda_fail(e_, #call);  \
    } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device error word of the library (mel kernels, quantiser) on the current
// device.
unsigned* lib_error_word();

// ------------------------------------------------------------------ mel
constexpr int kChunkSamples = 480000;
constexpr int kFrames = 3000;
constexpr int kNFFT = 400;
constexpr int kHop = 160;
constexpr int kBins = 201;
constexpr int kCtx = 1500;
constexpr int kMaxPos = 448;

wb_status mel_launch(const float* audio, int64_t B, int n_mels, float* mel, cudaStream_t s);

// mel [B, C, 3000] fp32 -> [B, 3002, C] fp32, or [B, 3002, 2C] bf16 pairs
// (hi | lo per row), with a zero row at both ends of each chunk: the conv1
// implicit-GEMM operand.
wb_status mel_transpose_pad(const float* mel, int64_t B, int C, void* out, bool bf16,
                            cudaStream_t s);

}  // namespace wb
