// Memory-bound kernels around the GEMMs and attention: LayerNorm (fused with
// the FP8 per-row quantiser when the next GEMM runs in E4M3), token + position
// embedding, the E4M3 KV-cache scale and append, the per-tensor quantiser,
// greedy argmax with token bookkeeping, and weight re-layouts done once at
// model creation.
//
// LayerNorm follows "whisper-blaze 0.1.8", "Direct Kernel API"
// (layernorm_fused, eps 1e-5); FP8 quantisation follows the same page's
// quantise_e4m3 (per-tensor scale, amax / 448) and the float8 KV cache of
// "Blazingly fast whisper transcriptions with Inference Endpoints",
// "Inference Stack"; greedy choice follows the "thewhisper-large-v3-turbo"
// model card, "NVIDIA Usage" (no sampling, one beam).
#include <algorithm>

#include "common.cuh"
#include "prof.cuh"
#include "layers.cuh"

namespace wb {
namespace {

constexpr int kMaxPerLane = 40;   // d <= 1280

// Vector form for d % 128 == 0: one warp per row, VPL float4 per lane, the
// gain and shift fetched together with the row so that one memory round trip
// covers all three.  Optionally zeroes `zero` (n4 float4) on the side: the
// next GEMM's split-K output, which would otherwise need a launch of its own.
// LN_AMAX / LN_E4M3_GROUP: amax of every group of group_rows rows (one
// chunk's GEMM input) in amax_bits; the first pass takes it, the second
// quantises with it, both from the same arithmetic on the same row.
template <int OUT, int VPL>
__global__ void __launch_bounds__(128)
layernorm_vec_kernel(const float* __restrict__ x, int64_t ld_x, int64_t rows, const float* __restrict__ g,
                     const float* __restrict__ b, void* __restrict__ out, int64_t ld_o, float* __restrict__ row_scale,
                     float4* __restrict__ zero, int64_t zero_n4, unsigned* __restrict__ amax_bits,
                     int64_t group_rows) {
    griddep_wait();
    griddep_launch();
    if (zero) {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < zero_n4; i += (int64_t)gridDim.x * blockDim.x)
            zero[i] = z;
    }
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    constexpr int d = VPL * 128;
    const float4* xr = reinterpret_cast<const float4*>(x + row * ld_x);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    const float4* b4 = reinterpret_cast<const float4*>(b);
    float4 v[VPL], gv[VPL], bv[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        v[i] = xr[i * 32 + lane];
        gv[i] = g4[i * 32 + lane];
        bv[i] = b4[i * 32 + lane];
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    const float mean = warp_sum(s) / (float)d;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const float a = v[i].x - mean, c = v[i].y - mean, e = v[i].z - mean, f = v[i].w - mean;
        q = fmaf(a, a, q); q = fmaf(c, c, q); q = fmaf(e, e, q); q = fmaf(f, f, q);
    }
    const float rstd = rsqrtf(warp_sum(q) / (float)d + 1e-5f);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        v[i].x = (v[i].x - mean) * rstd * gv[i].x + bv[i].x;
        v[i].y = (v[i].y - mean) * rstd * gv[i].y + bv[i].y;
        v[i].z = (v[i].z - mean) * rstd * gv[i].z + bv[i].z;
        v[i].w = (v[i].w - mean) * rstd * gv[i].w + bv[i].w;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
    if (OUT == LN_F32) {
        float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + row * ld_o);
#pragma unroll
        for (int i = 0; i < VPL; ++i) o[i * 32 + lane] = v[i];
    } else if (OUT == LN_BF16 || OUT == LN_BF16X2) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out) + row * ld_o;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int c = (i * 32 + lane) * 4;
            const uint32_t h0 = pack_bf16x2(v[i].x, v[i].y), h1 = pack_bf16x2(v[i].z, v[i].w);
            *reinterpret_cast<uint2*>(o + c) = make_uint2(h0, h1);
            if (OUT == LN_BF16X2) {
                const float r0 = v[i].x - __uint_as_float(h0 << 16), r1 = v[i].y - __uint_as_float(h0 & 0xFFFF0000u);
                const float r2 = v[i].z - __uint_as_float(h1 << 16), r3 = v[i].w - __uint_as_float(h1 & 0xFFFF0000u);
                *reinterpret_cast<uint2*>(o + d + c) = make_uint2(pack_bf16x2(r0, r1), pack_bf16x2(r2, r3));
            }
        }
    } else if (OUT == LN_AMAX) {
        amax = warp_max(amax);
        if (lane == 0) atomicMax(amax_bits + row / group_rows, __float_as_uint(amax));
    } else {   // LN_E4M3: per-row scale amax / 448; LN_E4M3_GROUP: the group's
        float sc;
        if (OUT == LN_E4M3_GROUP) {
            const float a = __uint_as_float(amax_bits[row / group_rows]);
            sc = a > 0.f ? a / 448.0f : 1.0f;
        } else {
            amax = warp_max(amax);
            sc = amax > 0.f ? amax / 448.0f : 1.0f;
        }
        const float inv = 1.0f / sc;
        uint8_t* o = reinterpret_cast<uint8_t*>(out) + row * ld_o;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const uint32_t lo = f2e4m3x2(v[i].x * inv, v[i].y * inv) & 0xFFFFu;
            const uint32_t hi = f2e4m3x2(v[i].z * inv, v[i].w * inv) & 0xFFFFu;
            *reinterpret_cast<uint32_t*>(o + (i * 32 + lane) * 4) = lo | (hi << 16);
        }
        if (lane == 0) row_scale[row] = sc;
    }
}

// One warp per row; the row lives in registers for the two-pass moments.
template <int OUT>
__global__ void __launch_bounds__(256)
layernorm_kernel(const float* __restrict__ x, int64_t ld_x, int64_t rows, int d, const float* __restrict__ g,
                 const float* __restrict__ b, void* __restrict__ out, int64_t ld_o, float* __restrict__ row_scale) {
    griddep_wait();
    griddep_launch();
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float* xr = x + row * ld_x;
    const int per = d / 32;
    float v[kMaxPerLane];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
        if (i < per) { v[i] = xr[i * 32 + lane]; s += v[i]; }
    s = warp_sum(s);
    const float mean = s / (float)d;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
        if (i < per) { const float t = v[i] - mean; q = fmaf(t, t, q); }
    q = warp_sum(q);
    const float rstd = rsqrtf(q / (float)d + 1e-5f);
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
        if (i < per) {
            const int c = i * 32 + lane;
            v[i] = (v[i] - mean) * rstd * g[c] + b[c];
            amax = fmaxf(amax, fabsf(v[i]));
        }
    if (OUT == LN_F32) {
        float* o = reinterpret_cast<float*>(out) + row * ld_o;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i)
            if (i < per) o[i * 32 + lane] = v[i];
    } else if (OUT == LN_BF16) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out) + row * ld_o;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i)
            if (i < per) o[i * 32 + lane] = f2bf(v[i]);
    } else if (OUT == LN_BF16X2) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out) + row * ld_o;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i)
            if (i < per) {
                const __nv_bfloat16 hi = f2bf(v[i]);
                o[i * 32 + lane] = hi;
                o[d + i * 32 + lane] = f2bf(v[i] - bf2f(hi));
            }
    } else {   // LN_E4M3: per-row scale amax / 448
        amax = warp_max(amax);
        const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
        const float inv = 1.0f / sc;
        uint8_t* o = reinterpret_cast<uint8_t*>(out) + row * ld_o;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i)
            if (i < per) o[i * 32 + lane] = (uint8_t)(f2e4m3x2(v[i] * inv, 0.f) & 0xFF);
        if (lane == 0) row_scale[row] = sc;
    }
}

// x[r] = E[token] + P[pos] in fp32.  Row r is (chunk c = r / P, position
// p0 + r % P); the token is tokens[c * 448 + pos].
template <typename TW>
__global__ void embed_kernel(const int32_t* __restrict__ tokens, int64_t rows, int P, int p0, int d,
                             const TW* __restrict__ E, const TW* __restrict__ Pos, int vocab,
                             float* __restrict__ x, unsigned* err, const int* __restrict__ pos_dev, int pos_stride,
                             const int32_t* __restrict__ len) {
    griddep_wait();
    griddep_launch();
    const int64_t r = blockIdx.x;
    if (r >= rows) return;
    const int64_t c = r / P;
    const int pos = (pos_dev ? pos_dev[c * pos_stride] : p0) + (int)(r % P);
    if (pos >= kMaxPos || (len && pos >= len[c])) {   // a finished chunk's row: nothing to embed
        for (int i = threadIdx.x; i < d; i += blockDim.x) x[r * d + i] = 0.f;
        return;
    }
    int tok = tokens[c * kMaxPos + pos];
    if (tok < 0 || tok >= vocab) {
        if (threadIdx.x == 0) wb_set_error(err, WB_DEVERR_BOUNDS);
        tok = 0;
    }
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        x[r * d + i] = (float)E[(int64_t)tok * d + i] + (float)Pos[(int64_t)pos * d + i];
}

// Per (chunk, K|V): s = 2 * max(amax over the chunk's P rows, 1e-12) / 448.
__global__ void kv_scale_kernel(const float* __restrict__ qkv, int P, int d, float* __restrict__ k_scale,
                                float* __restrict__ v_scale) {
    griddep_wait();
    griddep_launch();
    const int64_t c = blockIdx.x;
    const int which = blockIdx.y;   // 0: K, 1: V
    float m = 0.f;
    for (int i = threadIdx.x; i < P * d; i += blockDim.x) {
        const int p = i / d, col = i % d;
        m = fmaxf(m, fabsf(qkv[(c * P + p) * 3 * (int64_t)d + (1 + which) * d + col]));
    }
    m = warp_max(m);
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = red[0];
        for (int i = 1; i < (int)(blockDim.x >> 5); ++i) a = fmaxf(a, red[i]);
        a = fmaxf(a, 1e-12f);
        const float s = (2.0f * a) / 448.0f;
        (which ? v_scale : k_scale)[c] = s;
    }
}

// Append K/V rows (fp32 inputs from the QKV GEMM) into the cache at
// positions p0 .. p0+P-1 of each chunk: E4M3 with the chunk's frozen scale,
// or fp32.  Cache of chunk c, layer l: base + off[c] + ((2l + kv) H + h) L_c 64 + pos 64.
template <bool FP8>
__global__ void kv_append_kernel(const float* __restrict__ qkv, int64_t n_chunks, int P, int p0, int d, int H,
                                 int layer, void* __restrict__ cache, const int64_t* __restrict__ off,
                                 const int32_t* __restrict__ len, const float* __restrict__ k_scale,
                                 const float* __restrict__ v_scale, unsigned* err, const int* __restrict__ pos_dev) {
    griddep_wait();
    griddep_launch();
    const int64_t r = blockIdx.x;   // row = c * P + p
    const int64_t c = r / P;
    const int pos = (pos_dev ? *pos_dev : p0) + (int)(r % P);
    if (c >= n_chunks) return;
    const int L = len[c];
    if (pos >= L) return;   // a chunk past its length keeps no more rows
    for (int i = threadIdx.x; i < 2 * d; i += blockDim.x) {
        const int kv = i / d, col = i % d, h = col / 64, e = col % 64;
        const float x = qkv[r * 3 * (int64_t)d + d + i];
        const int64_t idx = off[c] + ((int64_t)(2 * layer + kv) * H + h) * L * 64 + (int64_t)pos * 64 + e;
        if (FP8) {
            const float s = kv ? v_scale[c] : k_scale[c];
            const float inv = 1.0f / s;
            reinterpret_cast<uint8_t*>(cache)[idx] = (uint8_t)(f2e4m3x2(x * inv, 0.f) & 0xFF);
        } else {
            reinterpret_cast<float*>(cache)[idx] = x;
        }
    }
}

// Per-row E4M3 quantisation of an fp32 matrix; with GELU, of GELU(x).  One
// CTA per row: each thread keeps its (at most kQuantRowVec) float4 pieces in
// registers between the row's amax and the codes, so GELU runs once per
// element and the row is read once.
constexpr int kQuantRowThreads = 256;
constexpr int kQuantRowVec = 8;            // K <= 4 * 256 * 8 = 8192

template <bool GELU>
__global__ void __launch_bounds__(kQuantRowThreads)
quant_rows_f32_kernel(const float* __restrict__ x, int64_t rows, int K, uint8_t* __restrict__ q,
                      float* __restrict__ row_scale) {
    griddep_wait();
    griddep_launch();
    __shared__ float red[kQuantRowThreads / 32];
    const int64_t r = blockIdx.x;
    if (r >= rows) return;
    const float* xr = x + r * K;
    float4 v[kQuantRowVec];
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < kQuantRowVec; ++j) {
        const int i = (threadIdx.x + j * kQuantRowThreads) * 4;
        if (i < K) {
            float4 a = *reinterpret_cast<const float4*>(xr + i);
            if (GELU) { a.x = gelu_f(a.x); a.y = gelu_f(a.y); a.z = gelu_f(a.z); a.w = gelu_f(a.w); }
            v[j] = a;
            m = fmaxf(m, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
        }
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < kQuantRowThreads / 32; ++w) m = fmaxf(m, red[w]);
    const float sc = m > 0.f ? m / 448.0f : 1.0f;
    const float inv = 1.0f / sc;
#pragma unroll
    for (int j = 0; j < kQuantRowVec; ++j) {
        const int i = (threadIdx.x + j * kQuantRowThreads) * 4;
        if (i < K) {
            const float4 a = v[j];
            const uint32_t o = (uint32_t)f2e4m3x2(a.x * inv, a.y * inv) | ((uint32_t)f2e4m3x2(a.z * inv, a.w * inv) << 16);
            *reinterpret_cast<uint32_t*>(q + r * K + i) = o;
        }
    }
    if (threadIdx.x == 0) row_scale[r] = sc;
}

// amax of each group of group_elems consecutive fp32 values: grid (slices,
// groups), one atomic max per block.
__global__ void __launch_bounds__(256)
group_amax_kernel(const float* __restrict__ x, int64_t group_elems, unsigned* __restrict__ amax_bits) {
    griddep_wait();
    griddep_launch();
    const int64_t grp = blockIdx.y;
    const float4* p = reinterpret_cast<const float4*>(x + grp * group_elems);
    const int64_t n4 = group_elems / 4;
    float m = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = p[i];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
    }
    m = warp_max(m);
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = red[0];
        for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
        atomicMax(amax_bits + grp, __float_as_uint(a));
    }
}

// E4M3 codes of fp32 rows with one scale per group of rows: one warp per row.
__global__ void __launch_bounds__(256)
quant_groups_kernel(const float* __restrict__ x, int64_t rows, int64_t K, int64_t group_rows,
                    const unsigned* __restrict__ amax_bits, uint8_t* __restrict__ q, float* __restrict__ row_scale) {
    griddep_wait();
    griddep_launch();
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const float a = __uint_as_float(amax_bits[r / group_rows]);
    const float sc = a > 0.f ? a / 448.0f : 1.0f;
    const float inv = 1.0f / sc;
    const float4* xr = reinterpret_cast<const float4*>(x + r * K);
    uint32_t* qr = reinterpret_cast<uint32_t*>(q + r * K);
    for (int64_t i = lane; i < K / 4; i += 32) {
        const float4 v = xr[i];
        qr[i] = (uint32_t)f2e4m3x2(v.x * inv, v.y * inv) | ((uint32_t)f2e4m3x2(v.z * inv, v.w * inv) << 16);
    }
    if (row_scale && lane == 0) row_scale[r] = sc;
}

__global__ void scales_from_amax_kernel(float* __restrict__ a, int64_t n) {
    griddep_wait();
    griddep_launch();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float m = a[i];
        a[i] = m > 0.f ? m / 448.0f : 1.0f;
    }
}

// amax of a tensor (non-negative floats order like their bit patterns).
template <typename T>
__global__ void amax_kernel(const T* __restrict__ x, int64_t n, unsigned* __restrict__ out_bits) {
    griddep_wait();
    griddep_launch();
    float m = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        m = fmaxf(m, fabsf((float)x[i]));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) atomicMax(out_bits, __float_as_uint(m));
}

__global__ void scale_from_amax_kernel(const unsigned* __restrict__ amax_bits, float* __restrict__ scale) {
    griddep_wait();
    griddep_launch();
    const float a = __uint_as_float(*amax_bits);
    *scale = a > 0.f ? a / 448.0f : 1.0f;
}

template <typename T>
__global__ void quant_tensor_kernel(const T* __restrict__ x, int64_t n, const float* __restrict__ scale,
                                    uint8_t* __restrict__ q) {
    griddep_wait();
    griddep_launch();
    const float inv = 1.0f / *scale;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        q[i] = (uint8_t)(f2e4m3x2((float)x[i] * inv, 0.f) & 0xFF);
}

__global__ void dequant_kernel(const uint8_t* __restrict__ q, const float* __restrict__ scale, int64_t n,
                               float* __restrict__ out) {
    griddep_wait();
    griddep_launch();
    const float s = *scale;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = e4m3_to_f(q[i]) * s;
}

__global__ void fill_kernel(float* __restrict__ x, int64_t n, float v) {
    griddep_wait();
    griddep_launch();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        x[i] = v;
}

// Greedy token: lowest index of the row maximum.  Row r belongs to chunk
// r (one row per chunk); the token goes to column pos+1 when pos+1 < len[c].
__global__ void __launch_bounds__(256)
argmax_kernel(const float* __restrict__ logits, int64_t ld, int64_t rows, int V, int32_t* __restrict__ tokens,
              const int32_t* __restrict__ len, const int* __restrict__ pos_dev, int pos_host, int pos_stride) {
    griddep_wait();
    griddep_launch();
    const int64_t r = blockIdx.x;
    if (r >= rows) return;
    const float* lr = logits + r * ld;
    float best = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int i = threadIdx.x; i < V; i += 256) {
        const float v = lr[i];
        if (v > best) { best = v; bi = i; }
    }
    __shared__ float sv[256];
    __shared__ int si[256];
    sv[threadIdx.x] = best;
    si[threadIdx.x] = bi;
    __syncthreads();
    for (int s = 128; s > 0; s >>= 1) {
        if (threadIdx.x < s) {
            const float a = sv[threadIdx.x], b = sv[threadIdx.x + s];
            const int ia = si[threadIdx.x], ib = si[threadIdx.x + s];
            if (b > a || (b == a && ib < ia)) { sv[threadIdx.x] = b; si[threadIdx.x] = ib; }
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int pos = pos_dev ? pos_dev[r * pos_stride] : pos_host;
        if (pos + 1 < len[r] && pos + 1 < kMaxPos) tokens[r * kMaxPos + pos + 1] = si[0] == 0x7FFFFFFF ? 0 : si[0];
    }
}

// ------------------------------------------------------------------ beam search
// One beam-search step for one chunk (K rows r0 .. r0+K-1, one hypothesis
// each; "thewhisper-large-v3-turbo", "NVIDIA Usage": num_beams): every
// continuation (b, v) scores scores[b] + (logit[b][v] - logZ_b), logZ_b the
// log-sum-exp of row b; the K best (ties: lower beam, then lower token) become
// the new hypotheses: their token rows and cache histories are the parents'
// up to position pos, the chosen token goes to column pos + 1 and the cache
// row the next step appends (pos + 1) is the new row's own.
constexpr int kSelThreads = 512;

__device__ __forceinline__ bool cand_better(float s1, int b1, int v1, float s2, int b2, int v2) {
    return s1 > s2 || (s1 == s2 && (b1 < b2 || (b1 == b2 && v1 < v2)));
}

__global__ void __launch_bounds__(kSelThreads)
beam_select_kernel(const float* __restrict__ logits, int64_t ld, int K, int V, float* __restrict__ scores,
                   int32_t* __restrict__ tokens, int32_t* __restrict__ hist, const int32_t* __restrict__ len,
                   const int* __restrict__ pos_dev, int pos_host, int32_t* __restrict__ parents_out,
                   float* __restrict__ scores_out) {
    griddep_wait();
    griddep_launch();
    __shared__ float logz[kBeamMax];
    __shared__ float rf[kSelThreads / 32];
    __shared__ int rb[kSelThreads / 32], rv[kSelThreads / 32], rt[kSelThreads / 32];
    __shared__ float sel_s[kBeamMax];
    __shared__ int sel_b[kBeamMax], sel_v[kBeamMax];
    __shared__ int32_t stok[kBeamMax][kMaxPos], shis[kBeamMax][kMaxPos];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r0 = (int64_t)blockIdx.x * K;
    const int pos = pos_dev ? *pos_dev : pos_host;
    if (len[r0] <= pos + 1) return;                 // this chunk has reached its length (uniform)
    // log-sum-exp of every hypothesis's logits
    for (int b = 0; b < K; ++b) {
        const float* x = logits + (r0 + b) * ld;
        float m = -INFINITY;
        for (int v = tid; v < V; v += kSelThreads) m = fmaxf(m, x[v]);
        m = warp_max(m);
        if (lane == 0) rf[warp] = m;
        __syncthreads();
        m = rf[0];
        for (int w = 1; w < kSelThreads / 32; ++w) m = fmaxf(m, rf[w]);
        __syncthreads();
        float sum = 0.f;
        for (int v = tid; v < V; v += kSelThreads) sum += expf(x[v] - m);
        sum = warp_sum(sum);
        if (lane == 0) rf[warp] = sum;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < kSelThreads / 32; ++w) t += rf[w];
            logz[b] = m + logf(t);
        }
        __syncthreads();
    }
    // each thread's K best continuations, sorted
    float ls[kBeamMax];
    int lb[kBeamMax], lv[kBeamMax];
    int n = 0;
    for (int b = 0; b < K; ++b) {
        const float base = scores[r0 + b], lz = logz[b];
        const float* x = logits + (r0 + b) * ld;
        for (int v = tid; v < V; v += kSelThreads) {
            const float sc = base + (x[v] - lz);
            if (n == K && !cand_better(sc, b, v, ls[K - 1], lb[K - 1], lv[K - 1])) continue;
            int i = n < K ? n++ : K - 1;
            while (i > 0 && cand_better(sc, b, v, ls[i - 1], lb[i - 1], lv[i - 1])) {
                ls[i] = ls[i - 1]; lb[i] = lb[i - 1]; lv[i] = lv[i - 1];
                --i;
            }
            ls[i] = sc; lb[i] = b; lv[i] = v;
        }
    }
    // K rounds: the best head among all threads' lists wins and is popped
    int head = 0;
    for (int k = 0; k < K; ++k) {
        float s = head < n ? ls[head] : -INFINITY;
        int b = head < n ? lb[head] : 0x7FFFFFFF, v = head < n ? lv[head] : 0x7FFFFFFF, t = tid;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            const int b2 = __shfl_xor_sync(0xffffffffu, b, o), v2 = __shfl_xor_sync(0xffffffffu, v, o);
            const int t2 = __shfl_xor_sync(0xffffffffu, t, o);
            if (cand_better(s2, b2, v2, s, b, v) || (s2 == s && b2 == b && v2 == v && t2 < t)) {
                s = s2; b = b2; v = v2; t = t2;
            }
        }
        if (lane == 0) { rf[warp] = s; rb[warp] = b; rv[warp] = v; rt[warp] = t; }
        __syncthreads();
        if (tid == 0) {
            int w0 = 0;
            for (int w = 1; w < kSelThreads / 32; ++w)
                if (cand_better(rf[w], rb[w], rv[w], rf[w0], rb[w0], rv[w0])) w0 = w;
            sel_s[k] = rf[w0]; sel_b[k] = rb[w0]; sel_v[k] = rv[w0];
            rt[0] = rt[w0];
        }
        __syncthreads();
        if (tid == rt[0]) ++head;
        __syncthreads();
    }
    // gather the parents' token rows and cache histories (positions 0 .. pos)
    for (int i = tid; i < K * (pos + 1); i += kSelThreads) {
        const int b = i / (pos + 1), q = i % (pos + 1);
        stok[b][q] = tokens[(r0 + b) * kMaxPos + q];
        shis[b][q] = hist[(r0 + b) * kMaxPos + q];
    }
    __syncthreads();
    for (int i = tid; i < K * (pos + 1); i += kSelThreads) {
        const int j = i / (pos + 1), q = i % (pos + 1);
        const int p = sel_b[j];
        tokens[(r0 + j) * kMaxPos + q] = stok[p][q];
        hist[(r0 + j) * kMaxPos + q] = shis[p][q];
    }
    if (tid < K) {
        const int j = tid;
        if (pos + 1 < kMaxPos) {
            tokens[(r0 + j) * kMaxPos + pos + 1] = sel_v[j];
            hist[(r0 + j) * kMaxPos + pos + 1] = (int32_t)(r0 + j);
        }
        scores[r0 + j] = sel_s[j];
        if (parents_out) parents_out[r0 + j] = sel_b[j];
        if (scores_out) scores_out[r0 + j] = sel_s[j];
    }
}

// The best hypothesis of each chunk (lowest beam index among the maximal
// scores): its token row (positions 0 .. len - 1) into out[c].
__global__ void beam_best_kernel(const float* __restrict__ scores, const int32_t* __restrict__ tokens, int K,
                                 const int32_t* __restrict__ len, int32_t* __restrict__ out,
                                 float* __restrict__ score_out) {
    griddep_wait();
    griddep_launch();
    const int64_t c = blockIdx.x, r0 = c * K;
    int best = 0;
    for (int b = 1; b < K; ++b)
        if (scores[r0 + b] > scores[r0 + best]) best = b;
    const int L = len[r0];
    for (int q = threadIdx.x; q < L; q += blockDim.x) out[c * kMaxPos + q] = tokens[(r0 + best) * kMaxPos + q];
    if (threadIdx.x == 0 && score_out) score_out[c] = scores[r0 + best];
}

// hist[r][q] = r (every row starts with its own cache rows); scores: 0 for
// the first row of each chunk, -inf for the others (one live hypothesis).
__global__ void beam_init_kernel(int32_t* __restrict__ hist, float* __restrict__ scores, int64_t rows, int K) {
    griddep_wait();
    griddep_launch();
    const int64_t r = blockIdx.x;
    if (r >= rows) return;
    for (int q = threadIdx.x; q < kMaxPos; q += blockDim.x) hist[r * kMaxPos + q] = (int32_t)r;
    if (threadIdx.x == 0) scores[r] = (r % K == 0) ? 0.f : -INFINITY;
}

// ------------------------------------------------------------------ continuous batching
// The cross K/V of n new chunks, computed into a staging decoder ([layer][R]
// blocks of blk16 16-byte words), copied into the blocks of their slots
// ([layer][S] blocks).  grid (x, n, layers).
__global__ void slot_cross_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                       const int32_t* __restrict__ slot_of, int64_t R, int64_t S, int64_t blk16,
                                       const float* __restrict__ cs_src, float* __restrict__ cs_dst) {
    griddep_wait();
    griddep_launch();
    const int64_t i = blockIdx.y, l = blockIdx.z;
    const uint4* a = src + (l * R + i) * blk16;
    uint4* b = dst + (l * S + slot_of[i]) * blk16;
    if (cs_src && blockIdx.x == 0 && threadIdx.x < 2)     // E4M3 cross K/V: scales [layer][K|V][rows]
        cs_dst[(2 * l + threadIdx.x) * S + slot_of[i]] = cs_src[(2 * l + threadIdx.x) * R + i];
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < blk16; k += (int64_t)gridDim.x * blockDim.x)
        b[k] = a[k];
}

// The rest of a new chunk's decode state into its slot (one CTA per chunk):
// the first P rows of every (layer, K|V, head) cache block (E4M3, blocks of
// lay x 64 bytes in both decoders), the per-layer cache scales ([layer][rows]),
// the token row up to position P (the prefix and the first generated token),
// the slot's position (P) and decode length.
__global__ void slot_state_kernel(const uint8_t* __restrict__ st_cache, uint8_t* __restrict__ sl_cache,
                                  const float* __restrict__ st_ks, const float* __restrict__ st_vs,
                                  float* __restrict__ sl_ks, float* __restrict__ sl_vs,
                                  const int32_t* __restrict__ st_tok, int32_t* __restrict__ sl_tok,
                                  int* __restrict__ pos, int32_t* __restrict__ len, const int32_t* __restrict__ slot_of,
                                  const int32_t* __restrict__ new_len, int R, int S, int layers, int heads, int lay,
                                  int P) {
    griddep_wait();
    griddep_launch();
    const int i = blockIdx.x, sl = slot_of[i];
    const int64_t per_row = (int64_t)layers * 2 * heads * lay * 64;
    const uint8_t* a = st_cache + (int64_t)i * per_row;
    uint8_t* b = sl_cache + (int64_t)sl * per_row;
    const int nblk = layers * 2 * heads, w16 = P * 4;      // 16-byte words per block prefix
    for (int k = threadIdx.x; k < nblk * w16; k += blockDim.x) {
        const int64_t blk = k / w16, w = k % w16;
        reinterpret_cast<uint4*>(b + blk * lay * 64)[w] = reinterpret_cast<const uint4*>(a + blk * lay * 64)[w];
    }
    for (int l = threadIdx.x; l < layers; l += blockDim.x) {
        sl_ks[(int64_t)l * S + sl] = st_ks[(int64_t)l * R + i];
        sl_vs[(int64_t)l * S + sl] = st_vs[(int64_t)l * R + i];
    }
    for (int q = threadIdx.x; q <= P; q += blockDim.x) sl_tok[(int64_t)sl * kMaxPos + q] = st_tok[(int64_t)i * kMaxPos + q];
    if (threadIdx.x == 0) {
        pos[sl] = P;
        len[sl] = new_len[i];
    }
}

// Finished chunks: out[chunk][0 .. len) = slot token row (one CTA per pair).
__global__ void slot_out_kernel(const int32_t* __restrict__ sl_tok, const int32_t* __restrict__ slot, const int32_t* __restrict__ chunk,
                                const int32_t* __restrict__ n_len, int32_t* __restrict__ out) {
    griddep_wait();
    griddep_launch();
    const int i = blockIdx.x;
    for (int q = threadIdx.x; q < n_len[i]; q += blockDim.x)
        out[(int64_t)chunk[i] * kMaxPos + q] = sl_tok[(int64_t)slot[i] * kMaxPos + q];
}

// conv weight [O][C][3] -> GEMM operand [O][3][C] (k index = j * C + c).
// With dup, every tap j is stored twice ([o][j][hi | lo][c], k index
// (2 j + half) C + c): the weights of a stem GEMM whose input rows carry each
// frame as a bf16 pair (hi | lo).
template <typename T>
__global__ void conv_reorder_kernel(const T* __restrict__ w, int O, int C, int dup, T* __restrict__ out) {
    griddep_wait();
    griddep_launch();
    const int reps = dup ? 2 : 1;
    const int64_t kk = (int64_t)3 * reps * C;
    const int64_t n = (int64_t)O * kk;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t o = i / kk;
        const int rem = (int)(i % kk);
        const int j = rem / (reps * C), c = rem % C;
        out[i] = w[(o * C + c) * 3 + j];
    }
}

__global__ void gather_rows_kernel(const float* __restrict__ x, int64_t rows, int d, int64_t stride_rows,
                                   int64_t first, float* __restrict__ out) {
    griddep_wait();
    griddep_launch();
    const int64_t r = blockIdx.x;
    if (r >= rows) return;
    for (int i = threadIdx.x; i < d; i += blockDim.x) out[r * d + i] = x[(r * stride_rows + first) * d + i];
}

__global__ void set_pos_kernel(int* pos, int value, int add, int n) {
    griddep_wait();
    griddep_launch();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        pos[i] = add ? pos[i] + value : value;
}

// GELU after a linear GEMM: fp32 [rows, N] -> bf16 pair [rows, 2N] (hi | lo)
// or fp32 in place.
__global__ void gelu_post_kernel(float* __restrict__ x, int64_t rows, int N, __nv_bfloat16* __restrict__ out2) {
    griddep_wait();
    griddep_launch();
    const int64_t total = rows * (int64_t)N;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = gelu_f(x[i]);
        if (out2) {
            const int64_t r = i / N, c = i % N;
            const __nv_bfloat16 hi = f2bf(v);
            out2[r * 2 * N + c] = hi;
            out2[r * 2 * N + N + c] = f2bf(v - bf2f(hi));
        } else {
            x[i] = v;
        }
    }
}

// E4M3 cross-attention K/V: one CTA per (chunk of the group, K|V, layer)
// tensor of n fp32 values (contiguous in both layouts): amax over the tensor,
// scale = amax / 448 (1 for an all-zero tensor), then codes of x * (1 / scale).
__global__ void __launch_bounds__(512)
cross_kv_quant_kernel(const float* __restrict__ tmp, int64_t n, int gB, int64_t B, int64_t g0,
                      uint8_t* __restrict__ out, float* __restrict__ scale) {
    griddep_wait();
    griddep_launch();
    __shared__ float red[16];
    const int64_t c = blockIdx.x, kv = blockIdx.y, l = blockIdx.z;
    const float4* src = reinterpret_cast<const float4*>(tmp + ((l * gB + c) * 2 + kv) * n);
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + ((l * B + g0 + c) * 2 + kv) * n);
    const int64_t n4 = n / 4;
    float m = 0.f;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 w = src[i];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(w.x), fabsf(w.y)), fmaxf(fabsf(w.z), fabsf(w.w))));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
    const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
    const float inv = 1.0f / sc;
    if (threadIdx.x == 0) scale[(l * 2 + kv) * B + g0 + c] = sc;
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 w = src[i];
        dst[i] = (uint32_t)f2e4m3x2(w.x * inv, w.y * inv) | ((uint32_t)f2e4m3x2(w.z * inv, w.w * inv) << 16);
    }
}

int grid_for(int64_t n, int threads) {
    int64_t g = (n + threads - 1) / threads;
    if (g > 148 * 16) g = 148 * 16;
    return (int)(g < 1 ? 1 : g);
}

template <int OUT>
wb_status launch_ln_vec(int vpl, const float* x, int64_t ld_x, int64_t rows, const float* g, const float* b, void* out,
                        int64_t ld_o, float* row_scale, float* zero, int64_t zero_n, cudaStream_t s,
                        unsigned* amax_bits = nullptr, int64_t group_rows = 1) {
    const dim3 grid((unsigned)((rows + 3) / 4)), block(128);
    float4* z = reinterpret_cast<float4*>(zero);
    const int64_t z4 = zero ? zero_n / 4 : 0;
#define WB_LN_ARGS x, ld_x, rows, g, b, out, ld_o, row_scale, z, z4, amax_bits, group_rows
    switch (vpl) {
    case 1: return launch_k(layernorm_vec_kernel<OUT, 1>, grid, block, 0, s, WB_LN_ARGS) ? WB_ERR_CUDA : WB_OK;
    case 2: return launch_k(layernorm_vec_kernel<OUT, 2>, grid, block, 0, s, WB_LN_ARGS) ? WB_ERR_CUDA : WB_OK;
    case 3: return launch_k(layernorm_vec_kernel<OUT, 3>, grid, block, 0, s, WB_LN_ARGS) ? WB_ERR_CUDA : WB_OK;
    case 4: return launch_k(layernorm_vec_kernel<OUT, 4>, grid, block, 0, s, WB_LN_ARGS) ? WB_ERR_CUDA : WB_OK;
    case 5: return launch_k(layernorm_vec_kernel<OUT, 5>, grid, block, 0, s, WB_LN_ARGS) ? WB_ERR_CUDA : WB_OK;
    case 6: return launch_k(layernorm_vec_kernel<OUT, 6>, grid, block, 0, s, WB_LN_ARGS) ? WB_ERR_CUDA : WB_OK;
    case 8: return launch_k(layernorm_vec_kernel<OUT, 8>, grid, block, 0, s, WB_LN_ARGS) ? WB_ERR_CUDA : WB_OK;
    case 10: return launch_k(layernorm_vec_kernel<OUT, 10>, grid, block, 0, s, WB_LN_ARGS) ? WB_ERR_CUDA : WB_OK;
    default: return WB_ERR_UNSUPPORTED;
    }
#undef WB_LN_ARGS
}

bool ln_vec_ok(int d) { return d % 128 == 0 && (d / 128 <= 6 || d / 128 == 8 || d / 128 == 10); }

}  // namespace

wb_status layernorm(const float* x, int64_t ld_x, int64_t rows, int d, const float* g, const float* b, LnOut mode,
                    void* out, int64_t ld_o, float* row_scale, cudaStream_t s, float* zero, int64_t zero_n) {
    if (rows <= 0) {
        if (zero && zero_n > 0) return fill(zero, zero_n, 0.f, s);
        return WB_OK;
    }
    if (d % 32 || d > 32 * kMaxPerLane) return fail(WB_ERR_SHAPE, "LayerNorm width must be a multiple of 32, <= 1280");
    const int osz = mode == LN_F32 ? 4 : (mode == LN_E4M3 ? 1 : 2);
    const bool vec = ln_vec_ok(d) && aligned16(x) && aligned16(g) && aligned16(b) && aligned16(out) && ld_x % 4 == 0 &&
                     (ld_o * osz) % 16 == 0 && (!zero || (aligned16(zero) && zero_n % 4 == 0));
    if (vec) {
        wb_status st;
        const int vpl = d / 128;
        if (mode == LN_F32) st = launch_ln_vec<LN_F32>(vpl, x, ld_x, rows, g, b, out, ld_o, row_scale, zero, zero_n, s);
        else if (mode == LN_BF16) st = launch_ln_vec<LN_BF16>(vpl, x, ld_x, rows, g, b, out, ld_o, row_scale, zero, zero_n, s);
        else if (mode == LN_BF16X2) st = launch_ln_vec<LN_BF16X2>(vpl, x, ld_x, rows, g, b, out, ld_o, row_scale, zero, zero_n, s);
        else st = launch_ln_vec<LN_E4M3>(vpl, x, ld_x, rows, g, b, out, ld_o, row_scale, zero, zero_n, s);
        if (st) return fail(st, "LayerNorm launch failed");
        WB_CUDA(cudaGetLastError());
        return WB_OK;
    }
    if (zero && zero_n > 0)
        if (wb_status st = fill(zero, zero_n, 0.f, s)) return st;
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (mode == LN_F32) WB_CUDA(launch_k(layernorm_kernel<LN_F32>, dim3(grid), dim3(256), 0, s, x, ld_x, rows, d, g, b, out, ld_o, row_scale));
    else if (mode == LN_BF16) WB_CUDA(launch_k(layernorm_kernel<LN_BF16>, dim3(grid), dim3(256), 0, s, x, ld_x, rows, d, g, b, out, ld_o, row_scale));
    else if (mode == LN_BF16X2) WB_CUDA(launch_k(layernorm_kernel<LN_BF16X2>, dim3(grid), dim3(256), 0, s, x, ld_x, rows, d, g, b, out, ld_o, row_scale));
    else WB_CUDA(launch_k(layernorm_kernel<LN_E4M3>, dim3(grid), dim3(256), 0, s, x, ld_x, rows, d, g, b, out, ld_o, row_scale));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status layernorm_group_e4m3(const float* x, int64_t ld_x, int64_t rows, int d, const float* g, const float* b,
                               int64_t group_rows, unsigned* amax_bits, uint8_t* out, int64_t ld_o, float* row_scale,
                               cudaStream_t s) {
    if (rows <= 0) return WB_OK;
    if (!ln_vec_ok(d) || !aligned16(x) || !aligned16(g) || !aligned16(b) || !aligned16(out) || ld_x % 4 || ld_o % 16)
        return fail(WB_ERR_UNSUPPORTED, "grouped E4M3 LayerNorm needs d % 128 == 0 and 16-byte aligned rows");
    if (group_rows < 1) return fail(WB_ERR_SHAPE, "grouped E4M3 LayerNorm: group_rows < 1");
    const int vpl = d / 128;
    wb_status st = launch_ln_vec<LN_AMAX>(vpl, x, ld_x, rows, g, b, nullptr, 0, nullptr, nullptr, 0, s, amax_bits,
                                          group_rows);
    if (!st)
        st = launch_ln_vec<LN_E4M3_GROUP>(vpl, x, ld_x, rows, g, b, out, ld_o, row_scale, nullptr, 0, s, amax_bits,
                                          group_rows);
    if (st) return fail(st, "grouped LayerNorm launch failed");
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status group_amax(const float* x, int64_t n_groups, int64_t group_elems, unsigned* amax_bits, cudaStream_t s) {
    if (n_groups <= 0 || group_elems <= 0) return WB_OK;
    if (group_elems % 4 || !aligned16(x)) return fail(WB_ERR_ALIGN, "group amax: groups of whole 16-byte vectors");
    if (n_groups > 65535) return fail(WB_ERR_SHAPE, "group amax: at most 65535 groups");
    // enough blocks to fill the SMs, at most one per 256 vectors of a group
    const int64_t want = std::max<int64_t>(1, (148 * 8 + n_groups - 1) / n_groups);
    const int64_t slices = std::max<int64_t>(1, std::min<int64_t>(want, (group_elems / 4 + 255) / 256));
    WB_CUDA(launch_k(group_amax_kernel, dim3((unsigned)slices, (unsigned)n_groups), dim3(256), 0, s, x, group_elems,
                     amax_bits));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status quant_groups(const float* x, int64_t rows, int64_t K, int64_t group_rows, const unsigned* amax_bits,
                       uint8_t* q, float* row_scale, cudaStream_t s) {
    if (rows <= 0 || K <= 0) return WB_OK;
    if (K % 4 || !aligned16(x) || !aligned16(q)) return fail(WB_ERR_ALIGN, "group quantiser: rows of 16-byte vectors");
    if (group_rows < 1) return fail(WB_ERR_SHAPE, "group quantiser: group_rows < 1");
    WB_CUDA(launch_k(quant_groups_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, s, x, rows, K, group_rows,
                     amax_bits, q, row_scale));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status scales_from_amax(float* a, int64_t n, cudaStream_t s) {
    if (n <= 0) return WB_OK;
    WB_CUDA(launch_k(scales_from_amax_kernel, dim3(grid_for(n, 256)), dim3(256), 0, s, a, n));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status cross_kv_quant(const void* tmp, int64_t gB, int64_t B, int64_t g0, int layers, int64_t n, uint8_t* out,
                         float* scale, cudaStream_t s) {
    if (gB <= 0 || layers <= 0) return WB_OK;
    if (n % 16 || !aligned16(tmp) || !aligned16(out)) return fail(WB_ERR_ALIGN, "cross K/V quantiser layout");
    if (gB > 65535 || layers > 65535) return fail(WB_ERR_SHAPE, "cross K/V quantiser grid");
    WB_CUDA(launch_k(cross_kv_quant_kernel, dim3((unsigned)gB, 2, (unsigned)layers), dim3(512), 0, s,
                     reinterpret_cast<const float*>(tmp), n, (int)gB, B, g0, out, scale));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status embed(const int32_t* tokens, int64_t rows, int P, int p0, int d, const void* E, const void* Pos,
                bool bf16, int vocab, float* x, unsigned* err, cudaStream_t s, const int* pos_dev,
                const int32_t* len, int pos_stride) {
    if (rows <= 0) return WB_OK;
    if (bf16)
        WB_CUDA(launch_k(embed_kernel<__nv_bfloat16>, dim3((unsigned)rows), dim3(256), 0, s, tokens, rows, P, p0, d,
            reinterpret_cast<const __nv_bfloat16*>(E), reinterpret_cast<const __nv_bfloat16*>(Pos), vocab, x, err,
            pos_dev, pos_stride, len));
    else
        WB_CUDA(launch_k(embed_kernel<float>, dim3((unsigned)rows), dim3(256), 0, s, tokens, rows, P, p0, d, reinterpret_cast<const float*>(E),
                                                           reinterpret_cast<const float*>(Pos), vocab, x, err, pos_dev, pos_stride, len));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status kv_scales(const float* qkv, int64_t n_chunks, int P, int d, float* k_scale, float* v_scale, cudaStream_t s) {
    if (n_chunks <= 0) return WB_OK;
    WB_CUDA(launch_k(kv_scale_kernel, dim3(dim3((unsigned)n_chunks, 2)), dim3(256), 0, s, qkv, P, d, k_scale, v_scale));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status kv_append(const float* qkv, int64_t n_chunks, int P, int p0, int d, int H, int layer, bool fp8, void* cache,
                    const int64_t* off, const int32_t* len, const float* k_scale, const float* v_scale, unsigned* err,
                    cudaStream_t s, const int* pos_dev) {
    if (n_chunks <= 0) return WB_OK;
    const unsigned grid = (unsigned)(n_chunks * P);
    if (fp8) WB_CUDA(launch_k(kv_append_kernel<true>, dim3(grid), dim3(256), 0, s, qkv, n_chunks, P, p0, d, H, layer, cache, off, len, k_scale, v_scale, err, pos_dev));
    else WB_CUDA(launch_k(kv_append_kernel<false>, dim3(grid), dim3(256), 0, s, qkv, n_chunks, P, p0, d, H, layer, cache, off, len, k_scale, v_scale, err, pos_dev));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status quant_rows_f32(const float* x, int64_t rows, int K, uint8_t* q, float* row_scale, cudaStream_t s,
                         bool gelu) {
    if (rows <= 0) return WB_OK;
    if (K % 128 || K > 4 * kQuantRowThreads * kQuantRowVec)
        return fail(WB_ERR_SHAPE, "row quantiser needs K % 128 == 0 and K <= 8192");
    if (gelu)
        WB_CUDA(launch_k(quant_rows_f32_kernel<true>, dim3((unsigned)rows), dim3(kQuantRowThreads), 0, s, x, rows, K,
                         q, row_scale));
    else
        WB_CUDA(launch_k(quant_rows_f32_kernel<false>, dim3((unsigned)rows), dim3(kQuantRowThreads), 0, s, x, rows, K,
                         q, row_scale));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status quant_tensor(const void* x, bool bf16, int64_t n, uint8_t* q, float* scale, unsigned* scratch_bits,
                       cudaStream_t s) {
    WB_CUDA(cudaMemsetAsync(scratch_bits, 0, sizeof(unsigned), s));
    if (n > 0) {
        if (bf16) WB_CUDA(launch_k(amax_kernel<__nv_bfloat16>, dim3(grid_for(n, 256)), dim3(256), 0, s, reinterpret_cast<const __nv_bfloat16*>(x), n, scratch_bits));
        else WB_CUDA(launch_k(amax_kernel<float>, dim3(grid_for(n, 256)), dim3(256), 0, s, reinterpret_cast<const float*>(x), n, scratch_bits));
    }
    WB_CUDA(launch_k(scale_from_amax_kernel, dim3(1), dim3(1), 0, s, scratch_bits, scale));
    if (n > 0) {
        if (bf16) WB_CUDA(launch_k(quant_tensor_kernel<__nv_bfloat16>, dim3(grid_for(n, 256)), dim3(256), 0, s, reinterpret_cast<const __nv_bfloat16*>(x), n, scale, q));
        else WB_CUDA(launch_k(quant_tensor_kernel<float>, dim3(grid_for(n, 256)), dim3(256), 0, s, reinterpret_cast<const float*>(x), n, scale, q));
    }
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status dequant_tensor(const uint8_t* q, const float* scale, int64_t n, float* out, cudaStream_t s) {
    if (n <= 0) return WB_OK;
    WB_CUDA(launch_k(dequant_kernel, dim3(grid_for(n, 256)), dim3(256), 0, s, q, scale, n, out));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status gelu_post(float* x, int64_t rows, int N, void* out_bf16x2, cudaStream_t s) {
    const int64_t n = rows * (int64_t)N;
    if (n <= 0) return WB_OK;
    WB_CUDA(launch_k(gelu_post_kernel, dim3(grid_for(n, 256)), dim3(256), 0, s, x, rows, N, reinterpret_cast<__nv_bfloat16*>(out_bf16x2)));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status set_pos(int* pos_dev, int value, bool add, cudaStream_t s, int n) {
    WB_CUDA(launch_k(set_pos_kernel, dim3((unsigned)std::max(1, std::min((n + 255) / 256, 148))), dim3(256), 0, s,
                     pos_dev, value, add ? 1 : 0, n));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status fill(float* x, int64_t n, float v, cudaStream_t s) {
    if (n <= 0) return WB_OK;
    WB_CUDA(launch_k(fill_kernel, dim3(grid_for(n, 256)), dim3(256), 0, s, x, n, v));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status argmax_tokens(const float* logits, int64_t ld, int64_t rows, int V, int32_t* tokens, const int32_t* len,
                        const int* pos_dev, int pos_host, cudaStream_t s, int pos_stride) {
    if (rows <= 0) return WB_OK;
    WB_CUDA(launch_k(argmax_kernel, dim3((unsigned)rows), dim3(256), 0, s, logits, ld, rows, V, tokens, len, pos_dev, pos_host, pos_stride));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status beam_select(const float* logits, int64_t ld, int64_t n_chunks, int K, int V, float* scores, int32_t* tokens,
                      int32_t* hist, const int32_t* len, const int* pos_dev, int pos_host, int32_t* parents_out,
                      float* scores_out, cudaStream_t s) {
    if (n_chunks <= 0) return WB_OK;
    if (K < 1 || K > kBeamMax) return fail(WB_ERR_SHAPE, "beam search: 1 <= beams <= 8");
    WB_CUDA(launch_k(beam_select_kernel, dim3((unsigned)n_chunks), dim3(kSelThreads), 0, s, logits, ld, K, V, scores,
                     tokens, hist, len, pos_dev, pos_host, parents_out, scores_out));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status beam_best(const float* scores, const int32_t* tokens, int64_t n_chunks, int K, const int32_t* len,
                    int32_t* out, float* score_out, cudaStream_t s) {
    if (n_chunks <= 0) return WB_OK;
    WB_CUDA(launch_k(beam_best_kernel, dim3((unsigned)n_chunks), dim3(128), 0, s, scores, tokens, K, len, out,
                     score_out));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status beam_init(int32_t* hist, float* scores, int64_t rows, int K, cudaStream_t s) {
    if (rows <= 0) return WB_OK;
    WB_CUDA(launch_k(beam_init_kernel, dim3((unsigned)rows), dim3(128), 0, s, hist, scores, rows, K));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status slot_cross_copy(const void* src, void* dst, const int32_t* slot_of, int n, int64_t R, int64_t S, int layers,
                          int64_t blk_bytes, cudaStream_t s, const float* cs_src, float* cs_dst) {
    if (n <= 0 || layers <= 0) return WB_OK;
    if (blk_bytes % 16) return fail(WB_ERR_ALIGN, "slot cross copy: blocks of whole 16-byte words");
    const int64_t blk16 = blk_bytes / 16;
    const unsigned gx = (unsigned)std::max<int64_t>(1, std::min<int64_t>(64, (blk16 + 1023) / 1024));
    WB_CUDA(launch_k(slot_cross_copy_kernel, dim3(gx, (unsigned)n, (unsigned)layers), dim3(256), 0, s,
                     reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), slot_of, R, S, blk16, cs_src,
                     cs_dst));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status slot_state(const uint8_t* st_cache, uint8_t* sl_cache, const float* st_ks, const float* st_vs, float* sl_ks,
                     float* sl_vs, const int32_t* st_tok, int32_t* sl_tok, int* pos, int32_t* len, const int32_t* slot_of,
                     const int32_t* new_len, int n, int R, int S, int layers, int heads, int lay, int P, cudaStream_t s) {
    if (n <= 0) return WB_OK;
    WB_CUDA(launch_k(slot_state_kernel, dim3((unsigned)n), dim3(256), 0, s, st_cache, sl_cache, st_ks, st_vs, sl_ks,
                     sl_vs, st_tok, sl_tok, pos, len, slot_of, new_len, R, S, layers, heads, lay, P));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status slot_out(const int32_t* sl_tok, const int32_t* slot, const int32_t* chunk, const int32_t* n_len, int n,
                   int32_t* out, cudaStream_t s) {
    if (n <= 0) return WB_OK;
    WB_CUDA(launch_k(slot_out_kernel, dim3((unsigned)n), dim3(128), 0, s, sl_tok, slot, chunk, n_len, out));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status conv_reorder(const void* w, int O, int C, bool bf16, void* out, cudaStream_t s, bool dup) {
    const int64_t n = (int64_t)O * C * 3 * (dup ? 2 : 1);
    if (bf16) WB_CUDA(launch_k(conv_reorder_kernel<__nv_bfloat16>, dim3(grid_for(n, 256)), dim3(256), 0, s, reinterpret_cast<const __nv_bfloat16*>(w), O, C, dup ? 1 : 0, reinterpret_cast<__nv_bfloat16*>(out)));
    else WB_CUDA(launch_k(conv_reorder_kernel<float>, dim3(grid_for(n, 256)), dim3(256), 0, s, reinterpret_cast<const float*>(w), O, C, dup ? 1 : 0, reinterpret_cast<float*>(out)));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status gather_rows(const float* x, int64_t rows, int d, int64_t stride_rows, int64_t first, float* out,
                      cudaStream_t s) {
    if (rows <= 0) return WB_OK;
    WB_CUDA(launch_k(gather_rows_kernel, dim3((unsigned)rows), dim3(256), 0, s, x, rows, d, stride_rows, first, out));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

}  // namespace wb
