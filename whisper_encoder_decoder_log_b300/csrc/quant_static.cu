// E4M3 per-tensor quantisation for callers that cannot allocate device memory.
//
// wb_quantise_e4m3 keeps its amax accumulator in a small buffer the library
// allocates with cudaMalloc on first use.  Some callers cannot tolerate any
// allocation inside the library: code running under a custom or pooled
// allocator that owns all device memory, code that must not trigger an
// implicit device synchronisation (cudaMalloc/cudaFree can synchronise), or
// hosts that forbid allocation after start-up.  This variant computes the same
// codes and scale, but its reduction scratch is a fixed array in the library's
// own device image: one partial maximum per thread block, at most
// kMaxBlocks blocks of kPerBlock elements, so n is limited to
// kMaxBlocks * kPerBlock = 2^26 elements.
//
// The array is static device memory of the library: every GPU that loads the
// library holds it (4160 floats, 16.6 KB) until the process exits.  All calls
// share it, so calls whose kernels overlap on the GPU (different streams
// without ordering) race on it; calls on one stream, or otherwise ordered, are
// safe.  The first call in a CUDA context looks up the array's device address
// (cudaGetSymbolAddress) with that context current and keeps it for that
// context; a new context on the device (after cudaDeviceReset, say) is looked
// up again on its first call.  Make that first call before any stream
// capture.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "prof.cuh"

namespace wb {
namespace {

constexpr int kMaxBlocks = 4096;
constexpr int kThreads = 256;
constexpr int kPerBlock = 16384;            // elements reduced by one block
constexpr int64_t kMaxN = (int64_t)kMaxBlocks * kPerBlock;

// Scratch: per-block maxima, then the final scale in slot kMaxBlocks.
static __device__ __align__(256) float g_quant_scratch[kMaxBlocks + 64];

template <typename T>
__global__ void __launch_bounds__(kThreads)
block_amax_kernel(const T* __restrict__ x, int64_t n, float* __restrict__ partial) {
    const int64_t base = (int64_t)blockIdx.x * kPerBlock;
    const int64_t end = min(n, base + kPerBlock);
    float m = 0.f;
    for (int64_t i = base + threadIdx.x; i < end; i += kThreads) m = fmaxf(m, fabsf((float)x[i]));
    m = warp_max(m);
    __shared__ float red[kThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = red[0];
        for (int i = 1; i < kThreads / 32; ++i) a = fmaxf(a, red[i]);
        partial[blockIdx.x] = a;   // every block writes its slot: nothing needs clearing
    }
}

// One block: maximum over the used partials -> scale (amax / 448, 1 when 0).
__global__ void __launch_bounds__(kThreads)
final_scale_kernel(float* __restrict__ partial, int nblocks, float* __restrict__ scale_out) {
    float m = 0.f;
    for (int i = threadIdx.x; i < nblocks; i += kThreads) m = fmaxf(m, partial[i]);
    m = warp_max(m);
    __shared__ float red[kThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = red[0];
        for (int i = 1; i < kThreads / 32; ++i) a = fmaxf(a, red[i]);
        const float s = a > 0.f ? a / 448.0f : 1.0f;
        partial[kMaxBlocks] = s;
        *scale_out = s;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
quant_codes_kernel(const T* __restrict__ x, int64_t n, const float* __restrict__ scale, uint8_t* __restrict__ q) {
    const float inv = 1.0f / *scale;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads)
        q[i] = (uint8_t)(f2e4m3x2((float)x[i] * inv, 0.f) & 0xFF);
}

std::mutex g_mu;
// Per device: the context the address was looked up in, and the address.
CUcontext g_scratch_ctx[64] = {};
float* g_scratch_ptr[64] = {};
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_ctx_once;

// Device address of the static scratch in the current context (looked up
// with that context current, again whenever the device's context changes).
wb_status scratch_ptr(float** out) {
    int dev = 0;
    WB_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(WB_ERR_UNSUPPORTED, "device index out of range");
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    });
    if (!g_ctx_current) return fail(WB_ERR_CUDA, "cuCtxGetCurrent unavailable");
    // null before the runtime has made a context current on this thread
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return fail(WB_ERR_CUDA, "cuCtxGetCurrent failed");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;   // the lookup also brings up the device's primary context
        const cudaError_t e = cudaGetSymbolAddress(&p, g_quant_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(quantiser scratch)");
        if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return fail(WB_ERR_CUDA, "no current CUDA context");
        g_scratch_ptr[dev] = reinterpret_cast<float*>(p);
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return WB_OK;
}

}  // namespace
}  // namespace wb

using namespace wb;

extern "C" wb_status wb_quantise_e4m3_static(const void* x, int32_t x_is_bf16, int64_t n, uint8_t* codes,
                                             float* scale, wb_stream stream) {
    if (!scale || (n > 0 && (!x || !codes)))
        return fail(WB_ERR_INVALID_ARG, "wb_quantise_e4m3_static: null argument");
    if (n < 0) return fail(WB_ERR_SHAPE, "wb_quantise_e4m3_static: n < 0");
    if (n > kMaxN)
        return fail(WB_ERR_SHAPE, "wb_quantise_e4m3_static: n exceeds the static scratch limit of 2^26 elements");
    float* scratch = nullptr;
    if (wb_status st = scratch_ptr(&scratch)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int nblocks = (int)((n + kPerBlock - 1) / kPerBlock);
    if (nblocks > 0) {
        if (x_is_bf16)
            block_amax_kernel<__nv_bfloat16><<<nblocks, kThreads, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x), n,
                                                                          scratch);
        else
            block_amax_kernel<float><<<nblocks, kThreads, 0, s>>>(reinterpret_cast<const float*>(x), n, scratch);
        count_launch();
    }
    final_scale_kernel<<<1, kThreads, 0, s>>>(scratch, nblocks, scale);
    count_launch();
    if (n > 0) {
        const int grid = (int)std::min<int64_t>((n + kThreads - 1) / kThreads, 148 * 16);
        if (x_is_bf16)
            quant_codes_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x), n,
                                                                        scale, codes);
        else
            quant_codes_kernel<float><<<grid, kThreads, 0, s>>>(reinterpret_cast<const float*>(x), n, scale, codes);
        count_launch();
    }
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}
