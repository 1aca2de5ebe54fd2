// Attention kernels ("whisper-blaze 0.1.8", "Direct Kernel API":
// encoder_self_attn without mask, decoder_self_attn with a causal mask,
// decoder_cross_attn without mask; "Unlocking the power of OpenAI's Whisper",
// section 3).  Every head has width 64 and computes softmax(q k^T / 8) v.
//
//  * The bf16 encoder self-attention runs on tcgen05 (flash_tc.cu).
//  * attn_rows_kernel: one CTA per (chunk, head, group of up to 4 query rows)
//    streams the chunk's keys with 16-byte loads (8 lanes per key row),
//    keeps the scores in shared memory, and reduces p . V across the CTA.  It
//    serves the fp32 model's encoder, the decoder's cross-attention over the
//    precomputed bf16 K/V, and the prefix pass's causal self-attention over
//    the (E4M3 or fp32) KV cache, where query row p sees cache rows 0..p.
//  * self_attn_step_kernel: one warp per (chunk, head) for a decode step over
//    E4M3 rows -- the causal self-attention (appending the token's own K/V
//    row) and the cross-attention over E4M3 cross K/V.
#include <type_traits>

#include "attn.cuh"
#include "common.cuh"
#include "prof.cuh"

namespace wb {
namespace {

// ------------------------------------------------------------------ row attention
constexpr int kRowThreads = 256;
constexpr int kGroups = kRowThreads / 8;    // key rows handled per pass (8 lanes per row)
constexpr int kUnroll = 4;                  // independent 16-byte loads in flight per thread

// Streaming 16-byte load that does not allocate in L1 (every byte is read once).
WB_DEV uint4 ld_stream(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
WB_DEV uint2 ld_stream8(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// Raw bytes of the 8 elements a lane owns in one key/value row.
template <typename T>
struct Raw8 { uint4 a, b; };
template <typename T>
WB_DEV Raw8<T> load_raw8(const T* p);
template <>
WB_DEV Raw8<float> load_raw8<float>(const float* p) { return {ld_stream(p), ld_stream(p + 4)}; }
template <>
WB_DEV Raw8<__nv_bfloat16> load_raw8<__nv_bfloat16>(const __nv_bfloat16* p) { return {ld_stream(p), make_uint4(0, 0, 0, 0)}; }
template <>
WB_DEV Raw8<uint8_t> load_raw8<uint8_t>(const uint8_t* p) {
    const uint2 v = ld_stream8(p);
    return {make_uint4(v.x, v.y, 0, 0), make_uint4(0, 0, 0, 0)};
}

template <typename T>
WB_DEV void unpack8(const Raw8<T>& r, float (&v)[8]);
template <>
WB_DEV void unpack8<float>(const Raw8<float>& r, float (&v)[8]) {
    v[0] = __uint_as_float(r.a.x); v[1] = __uint_as_float(r.a.y); v[2] = __uint_as_float(r.a.z); v[3] = __uint_as_float(r.a.w);
    v[4] = __uint_as_float(r.b.x); v[5] = __uint_as_float(r.b.y); v[6] = __uint_as_float(r.b.z); v[7] = __uint_as_float(r.b.w);
}
template <>
WB_DEV void unpack8<__nv_bfloat16>(const Raw8<__nv_bfloat16>& r, float (&v)[8]) {
    const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
template <>
WB_DEV void unpack8<uint8_t>(const Raw8<uint8_t>& r, float (&v)[8]) {
    const uint32_t w[2] = {r.a.x, r.a.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        __nv_fp8x4_e4m3 q;
        q.__x = w[i];
        const float4 f = static_cast<float4>(q);
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
}

// One query row per CTA over 16-bit or 8-bit K/V (decode steps) keeps 6 CTAs
// resident per SM: the K/V stream needs the loads of many CTAs in flight.
template <int NQ, typename TQ, typename TKV, typename TO>
__global__ void __launch_bounds__(kRowThreads, (NQ == 1 && sizeof(TKV) < 4) ? 6 : 1)
attn_rows_kernel(const TQ* __restrict__ q, int64_t q_ld, int rows_per_chunk, int n_rows_total,
                 KVView kv, int kv_len, int causal, int q_pos0, TO* __restrict__ out, int64_t o_ld,
                 int64_t o_split) {
    griddep_wait();
    griddep_launch();
    // scores for up to NQ query rows over up to kv_len keys
    extern __shared__ float sm[];
    float* sq = sm;                              // [NQ][64], pre-scaled by 1/8
    float* ss = sq + NQ * 64;                    // [NQ][kv_len]
    float* sred = ss + NQ * kv_len;              // [kGroups][NQ][64] partial outputs
    const int64_t chunk = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int r_first = blockIdx.z * NQ;
    const int nq = min(NQ, rows_per_chunk - r_first);
    if (nq <= 0) return;
    const int64_t row0 = chunk * rows_per_chunk + r_first;
    if (row0 >= n_rows_total) return;
    if (kv.pos_dev) {
        q_pos0 = kv.pos_dev[chunk * kv.pos_stride];
        if (kv.active_len && kv.active_len[chunk] <= q_pos0 + 1) return;   // finished chunk
    }

    for (int i = tid; i < NQ * 64; i += kRowThreads) {
        const int qi = i / 64, c = i % 64;
        sq[i] = qi < nq ? (float)q[(row0 + qi) * q_ld + h * 64 + c] * 0.125f : 0.f;
    }
    const int64_t kc = kv.beam_div > 1 ? chunk / kv.beam_div : chunk;   // the chunk whose keys this row reads
    const int64_t cb = kv.chunk_off ? kv.chunk_off[kc] : kc * kv.chunk_stride;
    const int64_t hs = kv.head_stride * (kv.chunk_len ? (int64_t)kv.chunk_len[kc] : 1);
    const TKV* Kp = reinterpret_cast<const TKV*>(kv.ptr) + cb + ((int64_t)kv.k_blk * kv.heads + h) * hs;
    const TKV* Vp = reinterpret_cast<const TKV*>(kv.ptr) + cb + ((int64_t)kv.v_blk * kv.heads + h) * hs;
    const float ks = kv.k_scale ? kv.k_scale[kc] : 1.f;
    const float vs = kv.v_scale ? kv.v_scale[kc] : 1.f;
    int nk = kv_len;
    if (causal) nk = min(kv_len, q_pos0 + r_first + nq);
    __syncthreads();

    const int sub = tid & 7;
    const int grp = tid >> 3;
    float qv[NQ][8];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int c = 0; c < 8; ++c) qv[qi][c] = sq[qi * 64 + sub * 8 + c];

    // phase 1: scores.  Trip count is uniform per warp (the 8-lane shuffles
    // need full warps); kUnroll rows are loaded before any is used.
    for (int jb = 0; jb < nk; jb += kGroups * kUnroll) {
        Raw8<TKV> raw[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jb + u * kGroups + grp;
            raw[u] = j < nk ? load_raw8<TKV>(Kp + (int64_t)j * kv.row_stride + sub * 8) : Raw8<TKV>{};
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jb + u * kGroups + grp;
            float kf[8];
            unpack8<TKV>(raw[u], kf);
            float acc[NQ];
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                float a = 0.f;
#pragma unroll
                for (int c = 0; c < 8; ++c) a = fmaf(qv[qi][c], kf[c], a);
                acc[qi] = a;
            }
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                acc[qi] += __shfl_xor_sync(0xffffffffu, acc[qi], 1);
                acc[qi] += __shfl_xor_sync(0xffffffffu, acc[qi], 2);
                acc[qi] += __shfl_xor_sync(0xffffffffu, acc[qi], 4);
            }
            if (j < nk && sub < nq) {
                float v = acc[0];
#pragma unroll
                for (int qi = 1; qi < NQ; ++qi)
                    if (sub == qi) v = acc[qi];
                v *= ks;
                if (causal && j > q_pos0 + r_first + sub) v = -INFINITY;
                ss[sub * kv_len + j] = v;
            }
        }
    }
    __syncthreads();
    // softmax per query row: warp qi handles row qi
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < nq) {
        float* sr = ss + warp * kv_len;
        float m = -INFINITY;
        for (int j = lane; j < nk; j += 32) m = fmaxf(m, sr[j]);
        m = warp_max(m);
        float sum = 0.f;
        for (int j = lane; j < nk; j += 32) {
            const float e = __expf(sr[j] - m);   // inputs <= 0
            sr[j] = e;
            sum += e;
        }
        sum = warp_sum(sum);
        const float inv = 1.f / sum;
        for (int j = lane; j < nk; j += 32) sr[j] *= inv;
    }
    __syncthreads();
    // phase 2: o = p . V ; thread (group grp, dims 8*sub..) over keys j = grp mod kGroups
    float o[NQ][8];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int c = 0; c < 8; ++c) o[qi][c] = 0.f;
    for (int jb = 0; jb < nk; jb += kGroups * kUnroll) {
        Raw8<TKV> raw[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jb + u * kGroups + grp;
            raw[u] = j < nk ? load_raw8<TKV>(Vp + (int64_t)j * kv.row_stride + sub * 8) : Raw8<TKV>{};
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jb + u * kGroups + grp;
            if (j < nk) {
                float vf[8];
                unpack8<TKV>(raw[u], vf);
#pragma unroll
                for (int qi = 0; qi < NQ; ++qi) {
                    const float p = ss[qi * kv_len + j];
#pragma unroll
                    for (int c = 0; c < 8; ++c) o[qi][c] = fmaf(p, vf[c], o[qi][c]);
                }
            }
        }
    }
    // reduce the kGroups row groups
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int c = 0; c < 8; ++c) sred[(grp * NQ + qi) * 64 + sub * 8 + c] = o[qi][c];
    __syncthreads();
    for (int i = tid; i < nq * 64; i += kRowThreads) {
        const int qi = i / 64, c = i % 64;
        float a = 0.f;
        for (int g = 0; g < kGroups; ++g) a += sred[(g * NQ + qi) * 64 + c];
        a *= vs;
        const TO hi = (TO)a;
        out[(row0 + qi) * o_ld + h * 64 + c] = hi;
        if (o_split) out[(row0 + qi) * o_ld + o_split + h * 64 + c] = (TO)(a - (float)hi);
    }
}

// Decode step, causal self-attention over the E4M3 cache, with the cache
// append of the current token fused in.  One warp per (chunk, head), kStepHeads
// heads per CTA.  Lane = (row r of 8, sub s of 4): a pass covers 8 cache rows
// and each lane owns 16 bytes of the K row and of the V row.  Every lane
// streams its own pieces into a kStepDepth-deep shared-memory ring with
// cp.async (16 bytes, L2 only), so the data in flight costs no registers and
// a lane only ever reads back what it copied itself.  The current token's K
// and V rows (fp32 in the QKV output) are quantised here with the chunk's
// scales, exactly as the append kernel does, written to cache row pos, and
// used from registers at j = pos.
constexpr int kStepHeads = 4;
constexpr int kStepDepth = 8;

// dot(q[0..15], E4M3 codes w) and o += p * E4M3 codes v
WB_DEV float dot16_e4m3(const float (&q)[16], const uint4& w) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_fp8x4_e4m3 a;
        a.__x = u[i];
        const float4 f = static_cast<float4>(a);
        s = fmaf(q[4 * i], f.x, s); s = fmaf(q[4 * i + 1], f.y, s);
        s = fmaf(q[4 * i + 2], f.z, s); s = fmaf(q[4 * i + 3], f.w, s);
    }
    return s;
}
WB_DEV void axpy16_e4m3(float (&o)[16], float p, const uint4& w) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_fp8x4_e4m3 a;
        a.__x = u[i];
        const float4 f = static_cast<float4>(a);
        o[4 * i] = fmaf(p, f.x, o[4 * i]); o[4 * i + 1] = fmaf(p, f.y, o[4 * i + 1]);
        o[4 * i + 2] = fmaf(p, f.z, o[4 * i + 2]); o[4 * i + 3] = fmaf(p, f.w, o[4 * i + 3]);
    }
}

WB_DEV uint4 quant16(const float* x, float inv) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 t = *reinterpret_cast<const float4*>(x + 4 * i);
        const uint32_t lo = f2e4m3x2(t.x * inv, t.y * inv), hi = f2e4m3x2(t.z * inv, t.w * inv);
        w[i] = (lo & 0xFFFFu) | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// CROSS: the same stream over a chunk's 1500 precomputed E4M3 cross K/V rows
// (q is the cross-attention query row, nothing is appended).
template <typename TO, bool CROSS>
__global__ void __launch_bounds__(32 * kStepHeads, 6)
self_attn_step_kernel(const float* __restrict__ qkv, int64_t q_ld, int heads, KVView kv, int q_pos_host,
                      TO* __restrict__ out, int64_t o_ld, int64_t o_split) {
    __shared__ uint4 ring[kStepHeads][kStepDepth][2][32];   // [warp][stage][K|V][lane]
    __shared__ int64_t shist[CROSS ? 1 : kMaxPos];          // beam search: cache base of each row j
    griddep_wait();
    griddep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t chunk = blockIdx.x;
    const int h = blockIdx.y * kStepHeads + warp;
    const int pos = kv.pos_dev ? kv.pos_dev[chunk * kv.pos_stride] : q_pos_host;
    if (kv.active_len && kv.active_len[chunk] <= pos + 1) return;   // finished chunk (uniform per CTA)
    const int64_t kc = CROSS ? chunk / kv.beam_div : chunk;         // whose cross K/V / scales
    const int L = CROSS ? kCtx : kv.chunk_len[chunk];
    if (!CROSS && pos >= L) return;                                // no cache row for this position
    if (!CROSS && kv.hist) {   // hypothesis history: row j of this row's cache sits in row hist[j]'s cache
        for (int j = threadIdx.x; j < pos; j += blockDim.x) shist[j] = kv.chunk_off[kv.hist[chunk * kMaxPos + j]];
        __syncthreads();
    }
    if (h >= heads) return;
    const int r = lane >> 2, sub = lane & 3;
    const int d = heads * 64;
    const int64_t hs = kv.head_stride * (CROSS ? 1 : (int64_t)L);
    uint8_t* const kvb = const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(kv.ptr));
    uint8_t* base = kvb + (CROSS ? kc * kv.chunk_stride : kv.chunk_off[chunk]);
    const int64_t koff = ((int64_t)kv.k_blk * kv.heads + h) * hs, voff = ((int64_t)kv.v_blk * kv.heads + h) * hs;
    uint8_t* Kp = base + koff;
    uint8_t* Vp = base + voff;
    const bool hist = !CROSS && kv.hist != nullptr;
    const int nk = CROSS ? kCtx : pos + 1;                         // rows attended
    const int nmem = CROSS ? kCtx : pos;                           // rows read from memory
    const int npass = (nk + 7) >> 3;
    uint4 (*rg)[2][32] = ring[warp];
    // rows below pos stream in while the current row is quantised
    auto issue = [&](int pass) {
        const int j = pass * 8 + r;
        if (pass < npass && j < nmem) {
            const int st = pass % kStepDepth;
            const uint8_t* rb = hist ? kvb + shist[j] : base;      // the cache that holds row j
            cp_async16(&rg[st][0][lane], rb + koff + (int64_t)j * 64 + sub * 16);
            cp_async16(&rg[st][1][lane], rb + voff + (int64_t)j * 64 + sub * 16);
        }
        cp_async_commit();      // one group per pass, empty or not
    };
#pragma unroll
    for (int u = 0; u < kStepDepth; ++u) issue(u);
    const float ks = kv.k_scale[kc], vs = kv.v_scale[kc];
    const float* qr = qkv + chunk * q_ld + h * 64 + sub * 16;
    // the current token's cache rows, quantised as the append kernel does
    uint4 kcur = make_uint4(0, 0, 0, 0), vcur = kcur;
    if (!CROSS) {
        kcur = quant16(qr + d, 1.0f / ks);
        vcur = quant16(qr + 2 * d, 1.0f / vs);
        if (r == 0) {
            *reinterpret_cast<uint4*>(Kp + (int64_t)pos * 64 + sub * 16) = kcur;
            *reinterpret_cast<uint4*>(Vp + (int64_t)pos * 64 + sub * 16) = vcur;
        }
    }
    float qv[16];
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
        const float4 t = *reinterpret_cast<const float4*>(qr + i);
        // fold the 1/sqrt(64) and the K scale into q
        qv[i] = t.x * 0.125f * ks; qv[i + 1] = t.y * 0.125f * ks; qv[i + 2] = t.z * 0.125f * ks; qv[i + 3] = t.w * 0.125f * ks;
    }
    float m = -INFINITY, l = 0.f, o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = 0.f;
    for (int pass = 0; pass < npass; ++pass) {
        cp_async_wait<kStepDepth - 1>();                           // this pass's group has landed
        const int j = pass * 8 + r;
        const int st = pass % kStepDepth;
        uint4 kr = make_uint4(0, 0, 0, 0), vr = kr;
        if (j < nmem) { kr = rg[st][0][lane]; vr = rg[st][1][lane]; }
        else if (!CROSS && j == pos) { kr = kcur; vr = vcur; }
        const bool valid = j < nk;
        float sc = dot16_e4m3(qv, kr);
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        if (!valid) sc = -INFINITY;
        float pm = sc;     // max over the 8 rows of the pass
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
        pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
        // the running maximum is raised only when a pass exceeds it by more
        // than 8 (natural log): otherwise p <= e^8 and o, l keep their scale,
        // which saves the per-pass correction multiply (pm and m are the same
        // in every lane, so the branch is warp-uniform)
        if (pm > m + 8.f) {
            const float alpha = __expf(m - pm);   // 0 on the first pass (m = -inf)
            l *= alpha;
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= alpha;
            m = pm;
        }
        const float pr = valid ? __expf(sc - m) : 0.f;
        float ps = pr;
        ps += __shfl_xor_sync(0xffffffffu, ps, 4);
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 16);
        l += ps;
        axpy16_e4m3(o, pr, vr);
        issue(pass + kStepDepth);                                  // refill the stage just consumed
    }
    cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        o[i] += __shfl_xor_sync(0xffffffffu, o[i], 4);
        o[i] += __shfl_xor_sync(0xffffffffu, o[i], 8);
        o[i] += __shfl_xor_sync(0xffffffffu, o[i], 16);
    }
    if (r == 0) {
        const float sc = vs / l;
        TO* orow = out + chunk * o_ld + h * 64 + sub * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float a = o[i] * sc;
            const TO hi = (TO)a;
            orow[i] = hi;
            if (o_split) orow[o_split + i] = (TO)(a - (float)hi);
        }
    }
}

template <int NQ, typename TQ, typename TKV, typename TO>
wb_status launch_rows_nq(const void* q, int64_t q_ld, int64_t n_chunks, int rows_per_chunk, int heads,
                         const KVView& kv, int kv_len, bool causal, int q_pos0, void* out, int64_t o_ld,
                         cudaStream_t s, int64_t o_split) {
    const size_t smem = sizeof(float) * (NQ * 64 + NQ * (size_t)kv_len + (size_t)kGroups * NQ * 64);
    static bool attr[64] = {};
    int dev = 0;
    WB_CUDA(cudaGetDevice(&dev));
    if (!attr[dev & 63]) {
        WB_CUDA(cudaFuncSetAttribute(attn_rows_kernel<NQ, TQ, TKV, TO>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        attr[dev & 63] = true;
    }
    if (smem > 200 * 1024) return fail(WB_ERR_SHAPE, "attention key length too large");
    dim3 grid((unsigned)n_chunks, (unsigned)heads, (unsigned)((rows_per_chunk + NQ - 1) / NQ));
    const int kind = causal ? WB_KERNEL_SELF_ATTN : WB_KERNEL_CROSS_ATTN;
    const int slot = prof_begin(kind, s);
    WB_CUDA(launch_k(attn_rows_kernel<NQ, TQ, TKV, TO>, dim3(grid), dim3(kRowThreads), smem, s, 
        reinterpret_cast<const TQ*>(q), q_ld, rows_per_chunk, (int)(n_chunks * rows_per_chunk), kv, kv_len,
        causal ? 1 : 0, q_pos0, reinterpret_cast<TO*>(out), o_ld, o_split));
    if (slot >= 0) {
        // K and V rows attended (each read once: beams of a chunk share its
        // cross K/V), queries in, outputs out
        const double kv_rows = causal ? (double)(q_pos0 + rows_per_chunk) : (double)kv_len;
        const double kv_sets = (double)n_chunks / (causal ? 1 : std::max(1, kv.beam_div));
        const double bytes = (double)heads * (kv_sets * 2.0 * kv_rows * 64.0 * sizeof(TKV) +
                                              (double)n_chunks * rows_per_chunk * 64.0 * (sizeof(TQ) + sizeof(TO)));
        prof_end(slot, s, bytes * prof_row_share());
    }
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

template <typename TQ, typename TKV, typename TO>
wb_status launch_rows(const void* q, int64_t q_ld, int64_t n_chunks, int rows_per_chunk, int heads,
                      const KVView& kv, int kv_len, bool causal, int q_pos0, void* out, int64_t o_ld,
                      cudaStream_t s, int64_t o_split) {
    if (!causal && rows_per_chunk == 1 && kv_len == kCtx && std::is_same<TKV, uint8_t>::value &&
        std::is_same<TQ, float>::value && std::is_same<TO, __nv_bfloat16>::value && (q_ld % 4) == 0 &&
        kv.k_scale && kv.v_scale && !kv.chunk_off && kv.head_stride == (int64_t)kCtx * 64 && kv.row_stride == 64 &&
        aligned16(q) && aligned16(kv.ptr) && (kv.chunk_stride % 16) == 0) {
        // decode step over E4M3 cross K/V: one warp per (chunk, head), cp.async ring
        if (n_chunks > 0x7FFFFFFF || heads > 65535 * kStepHeads) return fail(WB_ERR_SHAPE, "attention grid too large");
        const dim3 grid((unsigned)n_chunks, (unsigned)((heads + kStepHeads - 1) / kStepHeads));
        const int slot = prof_begin(WB_KERNEL_CROSS_ATTN, s);
        WB_CUDA(launch_k(self_attn_step_kernel<__nv_bfloat16, true>, grid, dim3(32 * kStepHeads), 0, s,
                         reinterpret_cast<const float*>(q), q_ld, heads, kv, q_pos0,
                         reinterpret_cast<__nv_bfloat16*>(out), o_ld, o_split));
        prof_end(slot, s, prof_row_share() * (double)heads *
                              ((double)n_chunks / std::max(1, kv.beam_div) * 2.0 * kCtx * 64.0 +
                               (double)n_chunks * 64.0 * (4 + 2)));
        WB_CUDA(cudaGetLastError());
        return WB_OK;
    }
    if (rows_per_chunk == 1)
        return launch_rows_nq<1, TQ, TKV, TO>(q, q_ld, n_chunks, rows_per_chunk, heads, kv, kv_len, causal, q_pos0,
                                              out, o_ld, s, o_split);
    return launch_rows_nq<4, TQ, TKV, TO>(q, q_ld, n_chunks, rows_per_chunk, heads, kv, kv_len, causal, q_pos0, out,
                                          o_ld, s, o_split);
}

}  // namespace

wb_status attn_self_step_e4m3(const float* qkv, int64_t q_ld, int64_t n_chunks, int heads, const KVView& kv,
                              int q_pos, void* out, int64_t o_ld, cudaStream_t s, int64_t o_split) {
    if (n_chunks <= 0) return WB_OK;
    if (!kv.chunk_off || !kv.chunk_len || !kv.k_scale || !kv.v_scale || kv.head_stride != 64 || kv.row_stride != 64)
        return fail(WB_ERR_INVALID_ARG, "step self-attention needs a ragged E4M3 cache with scales");
    if ((q_ld % 4) || !aligned16(qkv) || !aligned16(kv.ptr)) return fail(WB_ERR_ALIGN, "step self-attention operands");
    if (n_chunks > 0x7FFFFFFF || heads > 65535 * kStepHeads) return fail(WB_ERR_SHAPE, "attention grid too large");
    const dim3 grid((unsigned)n_chunks, (unsigned)((heads + kStepHeads - 1) / kStepHeads));
    const int slot = prof_begin(WB_KERNEL_SELF_ATTN, s);
    WB_CUDA(launch_k(self_attn_step_kernel<__nv_bfloat16, false>, grid, dim3(32 * kStepHeads), 0, s, qkv, q_ld, heads,
                     kv, q_pos, reinterpret_cast<__nv_bfloat16*>(out), o_ld, o_split));
    const double cached = prof_cached_rows() >= 0 ? prof_cached_rows() : (double)n_chunks * q_pos;
    prof_end(slot, s, (double)heads * (2.0 * cached * 64.0 +
                                       prof_row_share() * (double)n_chunks * (2.0 * 64.0 * (4 + 1) + 64.0 * (4 + 2))));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

wb_status attn_rows(DType tq, DType tkv, DType to, const void* q, int64_t q_ld, int64_t n_chunks,
                    int rows_per_chunk, int heads, const KVView& kv, int kv_len, bool causal, int q_pos0,
                    void* out, int64_t o_ld, cudaStream_t s, int64_t o_split) {
    if (n_chunks <= 0 || rows_per_chunk <= 0) return WB_OK;
    if (to == DT_BF16X2) {
        if (o_split <= 0) return fail(WB_ERR_INVALID_ARG, "split attention output needs an offset");
        to = DT_BF16;
    } else {
        o_split = 0;
    }
    if (n_chunks > 0x7FFFFFFF || heads > 65535) return fail(WB_ERR_SHAPE, "attention grid too large");
#define WB_ROWS(TQ_, TKV_, TO_) \
    return launch_rows<TQ_, TKV_, TO_>(q, q_ld, n_chunks, rows_per_chunk, heads, kv, kv_len, causal, q_pos0, out, o_ld, s, o_split)
    if (tq == DT_F32 && tkv == DT_F32 && to == DT_F32) WB_ROWS(float, float, float);
    if (tq == DT_F32 && tkv == DT_BF16 && to == DT_BF16) WB_ROWS(float, __nv_bfloat16, __nv_bfloat16);
    if (tq == DT_BF16 && tkv == DT_BF16 && to == DT_BF16) WB_ROWS(__nv_bfloat16, __nv_bfloat16, __nv_bfloat16);
    if (tq == DT_F32 && tkv == DT_E4M3 && to == DT_BF16) WB_ROWS(float, uint8_t, __nv_bfloat16);
    if (tq == DT_F32 && tkv == DT_F32 && to == DT_BF16) WB_ROWS(float, float, __nv_bfloat16);
#undef WB_ROWS
    return fail(WB_ERR_UNSUPPORTED, "attention type combination not built");
}

}  // namespace wb
