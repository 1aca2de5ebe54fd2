// Log-Mel front end: one fused kernel from float32 audio to the normalised
// [B, n_mels, 3000] log-Mel array ("whisper-blaze 0.1.8", "GPU Mel
// Spectrogram"; "Unlocking the power of OpenAI's Whisper", section 2).
//
// Work split.  A cluster of kCluster CTAs owns one 30 s chunk; CTA r computes
// frames [376 r, min(376 r + 376, 3000)) (a multiple of 4 frames, so rows of
// its output tile start on 16-byte boundaries).  Frames are processed 32 at a
// time: the audio segment they cover (5360 samples, reflect-padded at the
// chunk edges) is staged in shared memory -- the next sub-block's segment is
// copied asynchronously (cp.async) while the current one is transformed --
// and two real frames are packed into one complex
// 400-point FFT (z = x_a + i x_b), split as 400 = 16 x 25:
//   stage 1: per (pair, n2) a 16-point DFT over n1 of z[25 n1 + n2], times
//            the twiddle W400^(n2 k1);
//   stage 2: per (pair, k1) a 25-point DFT (as 5 x 5) over n2 in registers,
//            giving Z[k1 + 16 k2] for k2 = 0..24;
// then X_a, X_b are separated from Z[k] and Z[400-k] (exchanged between the
// threads that hold them by warp shuffles), the power of bins 0..200 goes
// through the sparse mel filterbank (each bin feeds at most two filters;
// one thread takes a filter over four frames), and log10 is taken.  The
// unfloored value (l + 4) / 4 is written
// to HBM right away, and the CTA keeps its maximum and each sub-block's
// minimum; the cluster then reduces the chunk maximum through distributed
// shared memory, and each CTA re-reads (from L2, 16 bytes at a time) only
// the sub-blocks whose minimum lies below the max - 8 floor, writing back the
// values that change.
#include <cooperative_groups.h>

#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "prof.cuh"

namespace cg = cooperative_groups;

namespace wb {
namespace {

constexpr int kCluster = 8;
constexpr int kFramesPerCta = 376;                     // the last CTA of a chunk: 368
constexpr int kSub = 32;                               // frames per sub-block
constexpr int kPairs = kSub / 2;
constexpr int kSeg = kSub * kHop + (kNFFT - kHop);     // 5360 samples
constexpr int kZStride = 425;                          // 400 slots + 25 pads
constexpr int kPStride = kBins;                        // odd stride: no bank conflicts
constexpr int kThreads = 256;
constexpr int kMaxMels = 128;
constexpr int kMaxFbNnz = 512;
constexpr int kSubBlocks = (kFramesPerCta + kSub - 1) / kSub;   // 12
// stage 2 runs one (pair, k1) per thread, all threads at once (its power
// step exchanges values between threads with warp shuffles)
static_assert(kPairs * 16 == kThreads, "stage 2 needs one thread per (pair, k1)");

// float -> unsigned key with the same order (for atomicMin on shared memory)
__device__ __forceinline__ unsigned order_key(float f) {
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct MelTables {
    float2 tw1[16 * 25];       // stage-1 twiddles W400^(n2 k1) at [k1][n2]
    float win[kNFFT];          // periodic Hann
    int4 meta[kMaxMels];       // filter m: first bin, bin count, weight offset
    float w[kMaxFbNnz];
};

struct MelSmem {
    MelTables t;
    float seg[kSeg];
    float2 z[kPairs * kZStride];
    float p[kSub * kPStride];
    float red[kThreads / 32];
    float cmax;
    unsigned smin[kSubBlocks];   // per sub-block minimum of log10(mel), order-preserving keys
};

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
// -i * a
__device__ __forceinline__ float2 cmi(float2 a) { return make_float2(a.y, -a.x); }

// Inner twiddles of the 16-point (W16^k = W400^(25 k), k = b c <= 9) and
// 25-point (W25^k = W400^(16 k), k <= 16) transforms: constants once the
// loops over b and c are unrolled (fp32 roundings of cos and -sin).
__device__ __forceinline__ float2 w16c(int k) {
    constexpr float c[10] = {1.0f, 0.9238795042037964f, 0.7071067690849304f, 0.3826834261417389f, 0.0f,
                             -0.3826834261417389f, -0.7071067690849304f, -0.9238795042037964f, -1.0f,
                             -0.9238795042037964f};
    constexpr float s[10] = {-0.0f, -0.3826834261417389f, -0.7071067690849304f, -0.9238795042037964f, -1.0f,
                             -0.9238795042037964f, -0.7071067690849304f, -0.3826834261417389f, 0.0f,
                             0.3826834261417389f};
    return make_float2(c[k], s[k]);
}
__device__ __forceinline__ float2 w25c(int k) {
    constexpr float c[17] = {1.0f, 0.9685831665992737f, 0.8763066530227661f, 0.728968620300293f, 0.5358268022537231f,
                             0.30901700258255005f, 0.06279052048921585f, -0.187381312251091f, -0.4257792830467224f,
                             -0.6374239921569824f, -0.80901700258255f, -0.9297764897346497f, -0.9921147227287292f,
                             -0.9921147227287292f, -0.9297764897346497f, -0.80901700258255f, -0.6374239921569824f};
    constexpr float s[17] = {-0.0f, -0.24868988990783691f, -0.4817536771297455f, -0.6845471262931824f,
                             -0.8443279266357422f, -0.9510565400123596f, -0.9980267286300659f, -0.9822872281074524f,
                             -0.9048270583152771f, -0.7705132365226746f, -0.5877852439880371f, -0.3681245446205139f,
                             -0.12533323466777802f, 0.12533323466777802f, 0.3681245446205139f, 0.5877852439880371f,
                             0.7705132365226746f};
    return make_float2(c[k], s[k]);
}

// Packed fp32 pair arithmetic (add/sub/mul/fma .f32x2: one instruction for
// both halves of a complex value); the butterflies below use it.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long r, x, y;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    unsigned long long r, x, y;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
// a * (c, c) + b
__device__ __forceinline__ float2 fma2s(float2 a, float c, float2 b) {
    unsigned long long r, x, y, cc;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(x), "l"(cc), "l"(y));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}
__device__ __forceinline__ float2 mul2s(float2 a, float c) {
    unsigned long long r, x, cc;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(cc));
    float2 o;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
    return o;
}

// 4-point DFT with W4 = -i, in place.
__device__ __forceinline__ void dft4(float2& x0, float2& x1, float2& x2, float2& x3) {
    float2 a = add2(x0, x2), b = sub2(x0, x2), c = add2(x1, x3), d = cmi(sub2(x1, x3));
    x0 = add2(a, c);
    x2 = sub2(a, c);
    x1 = add2(b, d);
    x3 = sub2(b, d);
}

// 5-point DFT with W5 = exp(-2 pi i / 5), in place.
__device__ __forceinline__ void dft5(float2& x0, float2& x1, float2& x2, float2& x3, float2& x4) {
    const float c1 = 0.30901699437494742f, c2 = -0.80901699437494742f;
    const float s1 = 0.95105651629515357f, s2 = 0.58778525229247313f;
    float2 t1 = add2(x1, x4), t2 = add2(x2, x3), t3 = sub2(x1, x4), t4 = sub2(x2, x3);
    float2 a1 = fma2s(t2, c2, fma2s(t1, c1, x0));
    float2 a2 = fma2s(t2, c1, fma2s(t1, c2, x0));
    float2 b1 = fma2s(t4, s2, mul2s(t3, s1));
    float2 b2 = fma2s(t4, -s1, mul2s(t3, s2));
    x0 = add2(x0, add2(t1, t2));
    float2 ib1 = cmi(b1), ib2 = cmi(b2);                // -i b
    x1 = add2(a1, ib1);
    x4 = sub2(a1, ib1);
    x2 = add2(a2, ib2);
    x3 = sub2(a2, ib2);
}

__global__ void __launch_bounds__(kThreads, 2)
mel_kernel(const float* __restrict__ audio, const MelTables* __restrict__ tables, int n_mels,
           float* __restrict__ out) {
    griddep_wait();
    griddep_launch();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    MelSmem& S = *reinterpret_cast<MelSmem*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    const int rank = blockIdx.x % kCluster;
    const int64_t chunk = blockIdx.x / kCluster;
    const float* x = audio + chunk * (int64_t)kChunkSamples;
    float* o = out + chunk * (int64_t)n_mels * kFrames;

    {   // tables -> shared memory
        const int4* src = reinterpret_cast<const int4*>(tables);
        int4* dst = reinterpret_cast<int4*>(&S.t);
        for (int i = tid; i < (int)(sizeof(MelTables) / 16); i += kThreads) dst[i] = src[i];
    }

    const int fbeg = rank * kFramesPerCta;
    const int fend = min(kFrames, fbeg + kFramesPerCta);
    const int nsb = (fend - fbeg + kSub - 1) / kSub;
    if (tid < kSubBlocks) S.smin[tid] = 0xFFFFFFFFu;
    float tmax = -1e30f;

    // audio segment of the sub-block at frame f0: padded index 160 f0 + i is
    // sample 160 f0 + i - 200 (a multiple of 4 samples, so 16-byte aligned)
    auto interior = [](int f0) {
        const int q0 = kHop * f0 - kNFFT / 2;
        return q0 >= 0 && q0 + kSeg <= kChunkSamples;
    };
    auto load_async = [&](int f0) {
        const float* src = x + (kHop * f0 - kNFFT / 2);
        for (int i = tid; i < kSeg / 4; i += kThreads) cp_async16(S.seg + 4 * i, src + 4 * i);
        cp_async_commit();
    };
    if (interior(fbeg)) load_async(fbeg);

    for (int sb = 0; sb < nsb; ++sb) {
        const int f0 = fbeg + sb * kSub;
        const int nf = min(kSub, fend - f0);
        if (!interior(f0)) {   // chunk edges: reflect (the segment buffer is free here)
            const int q0 = kHop * f0 - kNFFT / 2;
            for (int i = tid; i < kSeg; i += kThreads) {
                int q = q0 + i;
                if (q < 0) q = -q;
                if (q >= kChunkSamples) q = 2 * (kChunkSamples - 1) - q;
                q = max(0, min(q, kChunkSamples - 1));
                S.seg[i] = __ldg(x + q);
            }
        }
        cp_async_wait<0>();
        __syncthreads();   // segment (and, the first time, tables) ready; previous sub-block consumed
        // ---- stage 1: 16-point DFTs over n1, twiddle W400^(n2 k1)
        for (int it = tid; it < kPairs * 25; it += kThreads) {
            const int pr = it / 25, n2 = it % 25;
            const float* fa = S.seg + kHop * (2 * pr);
            const float* fb = fa + kHop;
            float2 v[16];
#pragma unroll
            for (int n1 = 0; n1 < 16; ++n1) {
                const int n = 25 * n1 + n2;
                const float w = S.t.win[n];
                v[n1] = make_float2(fa[n] * w, fb[n] * w);
            }
            // 16 = 4 x 4: n1 = 4 a + b, k1 = c + 4 d
#pragma unroll
            for (int b = 0; b < 4; ++b) dft4(v[b], v[4 + b], v[8 + b], v[12 + b]);   // over a -> c
#pragma unroll
            for (int b = 1; b < 4; ++b)
#pragma unroll
                for (int c = 1; c < 4; ++c)
                    v[4 * c + b] = (b * c == 4) ? cmi(v[4 * c + b]) : cmul(v[4 * c + b], w16c(b * c));
#pragma unroll
            for (int c = 0; c < 4; ++c) dft4(v[4 * c + 0], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            // v[4 c + d] now holds Y[k1 = c + 4 d]
            float2* zp = S.z + pr * kZStride + n2 * 17;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int d = 0; d < 4; ++d) {
                    const int k1 = c + 4 * d;
                    zp[k1] = (k1 == 0) ? v[4 * c + d] : cmul(v[4 * c + d], S.t.tw1[k1 * 25 + n2]);
                }
        }
        __syncthreads();
        // the segment is consumed: the next sub-block's copy overlaps the rest
        if (sb + 1 < nsb && interior(f0 + kSub)) load_async(f0 + kSub);
        // ---- stage 2: 25-point DFTs over n2 (5 x 5), in place
        for (int it = tid; it < kPairs * 16; it += kThreads) {
            const int pr = it / 16, k1 = it % 16;
            float2* zp = S.z + pr * kZStride + k1;
            float2 v[25];
#pragma unroll
            for (int n2 = 0; n2 < 25; ++n2) v[n2] = zp[17 * n2];
            // n2 = 5 a + b; k2 = c + 5 d
#pragma unroll
            for (int b = 0; b < 5; ++b) dft5(v[b], v[5 + b], v[10 + b], v[15 + b], v[20 + b]);
#pragma unroll
            for (int b = 1; b < 5; ++b)
#pragma unroll
                for (int c = 1; c < 5; ++c) v[5 * c + b] = cmul(v[5 * c + b], w25c(b * c));
#pragma unroll
            for (int c = 0; c < 5; ++c)
                dft5(v[5 * c + 0], v[5 * c + 1], v[5 * c + 2], v[5 * c + 3], v[5 * c + 4]);
            // v[5 c + d] holds Z[k1 + 16 k2], k2 = c + 5 d.
            // ---- separate the two real frames and take the power of the bins
            // k = k1 + 16 k2 <= 200 held here: Z[400 - k] is held by the
            // thread (16 - k1, 24 - k2) of the same pair, in the same half-warp
            // (k1 = 0: by this thread, as Z[16 (25 - k2) mod 400])
            const int partner = (tid & 16) | ((16 - k1) & 15);
            float* pa = S.p + (2 * pr) * kPStride;
            float* pb = pa + kPStride;
#pragma unroll
            for (int k2 = 0; k2 <= 12; ++k2) {
                const int sk = 24 - k2;                  // the value the partner takes from this thread
                const float2 mine = v[5 * (sk % 5) + sk / 5];
                float2 zn;
                zn.x = __shfl_sync(0xffffffffu, mine.x, partner);
                zn.y = __shfl_sync(0xffffffffu, mine.y, partner);
                if (k1 == 0) {
                    const int q = (25 - k2) % 25;
                    zn = v[5 * (q % 5) + q / 5];
                }
                const int k = k1 + 16 * k2;
                if (k < kBins) {
                    const float2 zk = v[5 * (k2 % 5) + k2 / 5];
                    const float ar = zk.x + zn.x, ai = zk.y - zn.y;     // 2 X_a
                    const float br = zk.y + zn.y, bi = zn.x - zk.x;     // 2 X_b
                    pa[k] = 0.25f * (ar * ar + ai * ai);
                    pb[k] = 0.25f * (br * br + bi * bi);
                }
            }
        }
        __syncthreads();
        // ---- mel filterbank, log10, unfloored output: one item = filter m
        // over frames f, f + 8, f + 16, f + 24 (each weight read once for 4)
        float smin = 1e30f;
        for (int it = tid; it < n_mels * (kSub / 4); it += kThreads) {
            const int m = it / (kSub / 4), f = it % (kSub / 4);
            const int4 mt = S.t.meta[m];
            const float* pf = S.p + f * kPStride + mt.x;
            float e[4] = {0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < mt.y; ++j) {
                const float w = S.t.w[mt.z + j];
#pragma unroll
                for (int i = 0; i < 4; ++i) e[i] = fmaf(w, pf[i * 8 * kPStride + j], e[i]);
            }
            float* orow = o + (int64_t)m * kFrames + f0 + f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (f + 8 * i >= nf) break;
                const float ell = __log2f(fmaxf(e[i], 1e-10f)) * 0.30102999566398120f;
                tmax = fmaxf(tmax, ell);
                smin = fminf(smin, ell);
                orow[8 * i] = (ell + 4.0f) * 0.25f;
            }
        }
        smin = warp_min(smin);
        if ((tid & 31) == 0) atomicMin(&S.smin[sb], order_key(smin));
    }
    // ---- chunk maximum across the cluster
    tmax = warp_max(tmax);
    if ((tid & 31) == 0) S.red[tid >> 5] = tmax;
    __syncthreads();
    if (tid == 0) {
        float m = S.red[0];
        for (int i = 1; i < kThreads / 32; ++i) m = fmaxf(m, S.red[i]);
        S.cmax = m;
    }
    cluster.sync();   // releases this CTA's global writes and its cmax
    float cm = -1e30f;
#pragma unroll
    for (int r = 0; r < kCluster; ++r) cm = fmaxf(cm, *cluster.map_shared_rank(&S.cmax, r));
    const float floor_log = cm - 8.0f;
    const float floor_v = (floor_log + 4.0f) * 0.25f;
    // ---- the floor, on the sub-blocks that hold a value below it; a value
    // at or above floor_log maps to an output at or above floor_v, so the
    // skipped sub-blocks are unchanged
    for (int sb = 0; sb < nsb; ++sb) {
        if (!(key_value(S.smin[sb]) < floor_log)) continue;
        const int f0 = fbeg + sb * kSub;
        const int q4 = min(kSub, fend - f0) / 4;       // 16-byte pieces per mel row
        for (int it = tid; it < n_mels * q4; it += kThreads) {
            const int m = it / q4, q = it % q4;
            float4* p = reinterpret_cast<float4*>(o + (int64_t)m * kFrames + f0) + q;
            float4 v = *p;
            if (v.x < floor_v || v.y < floor_v || v.z < floor_v || v.w < floor_v) {
                v.x = fmaxf(v.x, floor_v); v.y = fmaxf(v.y, floor_v);
                v.z = fmaxf(v.z, floor_v); v.w = fmaxf(v.w, floor_v);
                *p = v;
            }
        }
    }
    cluster.sync();   // no CTA leaves while another may still read its cmax
}

// ------------------------------------------------------------------ host tables
double hz_to_mel_slaney(double f) {
    const double f_sp = 200.0 / 3.0, min_log_hz = 1000.0, min_log_mel = min_log_hz / f_sp;
    const double logstep = std::log(6.4) / 27.0;
    return f >= min_log_hz ? min_log_mel + std::log(f / min_log_hz) / logstep : f / f_sp;
}
double mel_to_hz_slaney(double m) {
    const double f_sp = 200.0 / 3.0, min_log_hz = 1000.0, min_log_mel = min_log_hz / f_sp;
    const double logstep = std::log(6.4) / 27.0;
    return m >= min_log_mel ? min_log_hz * std::exp(logstep * (m - min_log_mel)) : f_sp * m;
}

bool build_tables(int n_mels, MelTables* t) {
    const double pi = 3.14159265358979323846;
    for (int j = 0; j < kNFFT; ++j) t->win[j] = (float)(0.5 - 0.5 * std::cos(2 * pi * j / kNFFT));
    for (int k1 = 0; k1 < 16; ++k1)
        for (int n2 = 0; n2 < 25; ++n2) {
            const int j = (k1 * n2) % kNFFT;
            t->tw1[k1 * 25 + n2] = make_float2((float)std::cos(2 * pi * j / kNFFT), (float)-std::sin(2 * pi * j / kNFFT));
        }
    const double mlo = hz_to_mel_slaney(0.0), mhi = hz_to_mel_slaney(8000.0);
    std::vector<double> pts(n_mels + 2);
    for (int i = 0; i < n_mels + 2; ++i)
        pts[i] = mel_to_hz_slaney(mlo + (mhi - mlo) * i / (n_mels + 1));
    int nnz = 0;
    for (int m = 0; m < n_mels; ++m) {
        const double lo = pts[m], c = pts[m + 1], hi = pts[m + 2];
        int first = -1, last = -1;
        std::vector<float> ws;
        for (int k = 0; k < kBins; ++k) {
            const double f = 40.0 * k;
            const double wv = std::fmax(0.0, std::fmin((f - lo) / (c - lo), (hi - f) / (hi - c))) *
                              (2.0 / (hi - lo));
            if (wv > 0) {
                if (first < 0) first = k;
                last = k;
            }
        }
        if (first < 0) first = last = 0;
        t->meta[m] = make_int4(first, last - first + 1, nnz, 0);
        for (int k = first; k <= last; ++k) {
            const double f = 40.0 * k;
            const double wv = std::fmax(0.0, std::fmin((f - lo) / (c - lo), (hi - f) / (hi - c))) *
                              (2.0 / (hi - lo));
            if (nnz >= kMaxFbNnz) return false;
            t->w[nnz++] = (float)wv;
        }
    }
    return true;
}

struct DeviceTables {
    MelTables* d80 = nullptr;
    MelTables* d128 = nullptr;
};
std::mutex g_tab_mu;
DeviceTables g_tabs[64];

// bf16 output rows carry each value as a pair: [hi (C) | lo (C)] with
// hi = bf16(x), lo = bf16(x - hi), so the stem GEMM keeps ~16 bits of the
// fp32 mel.
__global__ void transpose_pad_kernel(const float* __restrict__ mel, int C, void* __restrict__ out,
                                     bool bf16) {
    griddep_wait();
    griddep_launch();
    // grid: (ceil(3002 / 32), B); block 32 x 8.  Row r of the output is frame r - 1.
    __shared__ float tile[32][129];
    const int64_t b = blockIdx.y;
    const int r0 = blockIdx.x * 32;
    const float* src = mel + b * (int64_t)C * kFrames;
    for (int c = threadIdx.y; c < C; c += 8) {
        const int r = r0 + threadIdx.x;
        const int f = r - 1;
        tile[threadIdx.x][c] = (f >= 0 && f < kFrames) ? src[(int64_t)c * kFrames + f] : 0.f;
    }
    __syncthreads();
    for (int rr = threadIdx.y; rr < 32; rr += 8) {
        const int r = r0 + rr;
        if (r >= kFrames + 2) break;
        for (int c = threadIdx.x; c < C; c += 32) {
            if (bf16) {
                const int64_t idx = (b * (kFrames + 2) + r) * (int64_t)(2 * C) + c;
                const float x = tile[rr][c];
                const __nv_bfloat16 hi = __float2bfloat16_rn(x);
                reinterpret_cast<__nv_bfloat16*>(out)[idx] = hi;
                reinterpret_cast<__nv_bfloat16*>(out)[idx + C] = __float2bfloat16_rn(x - __bfloat162float(hi));
            } else {
                reinterpret_cast<float*>(out)[(b * (kFrames + 2) + r) * (int64_t)C + c] = tile[rr][c];
            }
        }
    }
}

}  // namespace

wb_status mel_launch(const float* audio, int64_t B, int n_mels, float* mel, cudaStream_t s) {
    int dev = 0;
    WB_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return fail(WB_ERR_UNSUPPORTED, "device index out of range");
    MelTables* tab = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_tab_mu);
        MelTables*& slot = n_mels == 80 ? g_tabs[dev].d80 : g_tabs[dev].d128;
        if (!slot) {
            MelTables h;
            memset(&h, 0, sizeof(h));
            if (!build_tables(n_mels, &h)) return fail(WB_ERR_SHAPE, "mel filterbank too large");
            WB_CUDA(cudaMalloc(&slot, sizeof(MelTables)));
            WB_CUDA(cudaMemcpy(slot, &h, sizeof(MelTables), cudaMemcpyHostToDevice));
            WB_CUDA(cudaFuncSetAttribute(mel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(MelSmem)));
        }
        tab = slot;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * kCluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(MelSmem);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    count_launch();
    const int slot = prof_begin(WB_KERNEL_MEL, s);
    WB_CUDA(cudaLaunchKernelEx(&cfg, mel_kernel, audio, (const MelTables*)tab, n_mels, mel));
    prof_end(slot, s, (double)B * ((double)kChunkSamples * 4.0 + (double)n_mels * kFrames * 4.0));
    return WB_OK;
}

wb_status mel_transpose_pad(const float* mel, int64_t B, int C, void* out, bool bf16,
                            cudaStream_t s) {
    if (C > 128) return fail(WB_ERR_SHAPE, "n_mels > 128");
    dim3 grid((kFrames + 2 + 31) / 32, (unsigned)B);
    WB_CUDA(launch_k(transpose_pad_kernel, dim3(grid), dim3(dim3(32, 8)), 0, s, mel, C, out, bf16));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

}  // namespace wb
