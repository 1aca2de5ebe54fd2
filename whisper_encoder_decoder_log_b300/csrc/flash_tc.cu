// Encoder self-attention on the 5th-generation tensor cores ("whisper-blaze
// 0.1.8", "Direct Kernel API": encoder_self_attn, no mask; here softmax(Q K^T
// / 8) V per 64-wide head over the 1500 positions of a chunk, bf16 in, fp32
// accumulation).
//
// One CTA = 128 query rows of one (chunk, head); 192 threads, two CTAs per SM:
//   warp 0      TMA: Q once, then K and V tiles of 128 keys into a 2-deep ring
//   warp 1      TMEM owner and MMA issuer (one thread):
//                 S_j  = Q . K_j^T          M 128, N 128, K 64   -> TMEM S
//                 O   += P_j . V_j          M 128, N 64,  K 128  -> TMEM O
//               V is read MN-major straight from its [key][dim] tile.
//   warps 2-5   softmax, one query row per thread (TMEM lane = row): load the
//               S row into registers once (S is then free for S_{j+1}), take
//               its maximum, write P = exp2(S c - m) as bf16 into a
//               128-byte-swizzled shared tile.
// The output accumulates in TMEM across all key tiles.  The running maximum m
// is only raised when a tile's maximum exceeds it by more than 2^8 (the
// published "conditional rescaling" of FlashAttention-4): P stays <= 256, and
// the rare raise rescales the row of O in TMEM once the previous P V product
// has landed.  The final O / l equals softmax(S) V for any such m.
// Keys past 1500 (the last tile reads into the next chunk or past the tensor,
// where TMA fills zeros) are masked to -inf; query rows past 1500 are not
// stored.  Every mbarrier wait is bounded by wall time.
#include "attn.cuh"
#include "common.cuh"
#include "prof.cuh"

namespace wb {
namespace {

constexpr int kRows = 128;          // query rows per CTA
constexpr int kKeys = 128;          // keys per tile
constexpr int kStages = 2;
constexpr int kTmemCols = 256;      // S 0-127, O 128-191
constexpr int kOCol = 128;
constexpr float kRaise = 8.0f;      // log2 growth of a row maximum absorbed without rescaling O
constexpr int kTileBytes = 128 * 128;            // 128 rows x 64 bf16
constexpr int kSmemSlack = 256;     // alignment slack requested above sizeof(FlashSmem)
constexpr uint32_t kIdescS = UmmaIdesc<128, 128, 1>::value;
constexpr uint32_t kIdescPV = UmmaIdesc<128, 64, 1>::value | (1u << 16);   // B (V) MN-major

struct FlashSmem {
    unsigned char q[kTileBytes];
    unsigned char k[kStages][kTileBytes];
    unsigned char v[kStages][kTileBytes];
    unsigned char p[2 * kTileBytes];              // [key half]
    uint64_t q_full;
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full, s_empty;
    uint64_t p_full, p_empty;                     // p_empty completes when P_j . V_j has landed in O
    uint64_t drain;
    uint32_t tmem;
    int abort_flag;
};

// Hardware base-2 exponential (MUFU, ~2^-22 relative error).
WB_DEV float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait that also gives up when another role has aborted.
WB_DEV bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned* err, unsigned bits) {
    for (WaitClock clk; !clk.expired();) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    wb_set_error(err, bits);
    *abort_flag = 1;
    return false;
}

__global__ void __launch_bounds__(192, 2)
flash_tc_kernel(const __grid_constant__ CUtensorMap tma_qkv, int d, __nv_bfloat16* __restrict__ out, unsigned* err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // two CTAs share an SM only if the alignment slack stays small; the
    // dynamic window starts 1024-aligned when, as here, there is no static
    // shared memory -- checked, not assumed
    const uint32_t mis = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if (mis > (uint32_t)kSmemSlack) {
        if (threadIdx.x == 0) wb_set_error(err, WB_DEVERR_BOUNDS);
        return;
    }
    FlashSmem& S = *reinterpret_cast<FlashSmem*>(smem_raw + mis);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = blockIdx.x * kRows;
    const int h = blockIdx.y;
    const int chunk = blockIdx.z;
    const int row_base = chunk * kCtx;              // first row of this chunk in [B * 1500, 3d]
    const int n_tiles = (kCtx + kKeys - 1) / kKeys;
    volatile int* abort_flag = &S.abort_flag;

    if (threadIdx.x == 0) {
        mbar_init(&S.q_full, 1);
        for (int i = 0; i < kStages; ++i) { mbar_init(&S.kv_full[i], 1); mbar_init(&S.kv_empty[i], 1); }
        mbar_init(&S.s_full, 1);
        mbar_init(&S.s_empty, 128);
        mbar_init(&S.p_full, 128);
        mbar_init(&S.p_empty, 1);
        mbar_init(&S.drain, 1);
        S.abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tma_qkv);
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem;
    griddep_wait();
    griddep_launch();

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            mbar_arrive_expect_tx(&S.q_full, kTileBytes);
            tma_load_2d(S.q, &tma_qkv, &S.q_full, h * 64, row_base + q0);
            uint32_t issued_parity[kStages];
            bool issued[kStages];
            for (int st = 0; st < kStages; ++st) { issued_parity[st] = 0; issued[st] = false; }
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int st = j % kStages;
                if (!wait_or_abort(&S.kv_empty[st], ((j / kStages) & 1) ^ 1, abort_flag, err, WB_DEVERR_TIMEOUT_TMA)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&S.kv_full[st], 2 * kTileBytes);
                tma_load_2d(S.k[st], &tma_qkv, &S.kv_full[st], d + h * 64, row_base + j * kKeys);
                tma_load_2d(S.v[st], &tma_qkv, &S.kv_full[st], 2 * d + h * 64, row_base + j * kKeys);
                issued[st] = true;
                issued_parity[st] = (j / kStages) & 1;
            }
            // no TMA writes may be in flight when the CTA leaves
            mbar_wait(&S.q_full, 0, err, WB_DEVERR_TIMEOUT_TMA);
            for (int st = 0; st < kStages; ++st)
                if (issued[st]) mbar_wait(&S.kv_full[st], issued_parity[st], err, WB_DEVERR_TIMEOUT_TMA);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = wait_or_abort(&S.q_full, 0, abort_flag, err, WB_DEVERR_TIMEOUT_MMA);
            const uint32_t q_addr = smem_u32(S.q);
            bool any = false;
            for (int j = 0; j <= n_tiles && ok; ++j) {
                if (j < n_tiles) {   // S_j = Q K_j^T
                    const int st = j % kStages;
                    if (!wait_or_abort(&S.kv_full[st], (j / kStages) & 1, abort_flag, err, WB_DEVERR_TIMEOUT_MMA) ||
                        !wait_or_abort(&S.s_empty, (j & 1) ^ 1, abort_flag, err, WB_DEVERR_TIMEOUT_MMA)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k_addr = smem_u32(S.k[st]);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_bf16(tmem, umma_desc_sw128(q_addr + 32 * k), umma_desc_sw128(k_addr + 32 * k), kIdescS,
                                  k ? 1u : 0u);
                    any = true;
                    umma_commit(&S.s_full);
                }
                if (j >= 1) {        // O += P_{j-1} V_{j-1}
                    const int i = j - 1, st = i % kStages;
                    if (!wait_or_abort(&S.p_full, i & 1, abort_flag, err, WB_DEVERR_TIMEOUT_MMA)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t p_addr = smem_u32(S.p);
                    const uint32_t v_addr = smem_u32(S.v[st]);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        // A: P, K-major, 64-key halves of 16 KB; B: V rows (keys) of 128 B, MN-major
                        const uint64_t ad = umma_desc_sw128(p_addr + (k >> 2) * kTileBytes + 32 * (k & 3));
                        const uint64_t bd = umma_desc_sw128(v_addr + 2048 * k);
                        umma_bf16(tmem + kOCol, ad, bd, kIdescPV, (i | k) ? 1u : 0u);
                    }
                    umma_commit(&S.p_empty);
                    umma_commit(&S.kv_empty[st]);
                }
            }
            if (any) {
                umma_commit(&S.drain);
                mbar_wait(&S.drain, 0, err, WB_DEVERR_TIMEOUT_MMA);
            }
        }
    } else {
        // softmax: thread = query row r (TMEM lane r)
        const int g = warp & 3;
        const int r = g * 32 + lane;
        const uint32_t lane_off = (uint32_t)(g * 32) << 16;
        const float c = 0.125f * 1.4426950408889634f;   // 1/sqrt(64) * log2(e)
        const uint64_t c2 = f32x2(c, c);
        float m = -INFINITY, l = 0.f;                    // running maximum (log2 units) and sum
        bool ok = true;
        // row swizzle inside a 128-byte atom row
        const uint32_t row_off = (uint32_t)(r >> 3) * 1024 + (uint32_t)(r & 7) * 128;
        const uint32_t sa = tmem + lane_off;
        const uint32_t oa = tmem + lane_off + kOCol;
        for (int j = 0; j < n_tiles && ok; ++j) {
            if (!wait_or_abort(&S.s_full, j & 1, abort_flag, err, WB_DEVERR_TIMEOUT_EPI)) { ok = false; break; }
            tc_fence_after();
            uint32_t s0[32], s1[32], s2[32], s3[32];
            tmem_ld32(sa, s0);
            tmem_ld32(sa + 32, s1);
            tmem_ld32(sa + 64, s2);
            tmem_ld32(sa + 96, s3);
            tmem_wait_ld();
            // S is in registers: the tensor core may compute S_{j+1}
            tc_fence_before();
            mbar_arrive(&S.s_empty);
            const int valid = min(kKeys, kCtx - j * kKeys);
            if (valid < kKeys) {                       // only the last tile is ragged
                constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    if (t >= valid) s0[t] = kNegInf;
                    if (32 + t >= valid) s1[t] = kNegInf;
                    if (64 + t >= valid) s2[t] = kNegInf;
                    if (96 + t >= valid) s3[t] = kNegInf;
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int t = 0; t < 32; t += 2) {
                mx0 = fmax3(mx0, __uint_as_float(s0[t]), __uint_as_float(s0[t + 1]));
                mx1 = fmax3(mx1, __uint_as_float(s1[t]), __uint_as_float(s1[t + 1]));
                mx0 = fmax3(mx0, __uint_as_float(s2[t]), __uint_as_float(s2[t + 1]));
                mx1 = fmax3(mx1, __uint_as_float(s3[t]), __uint_as_float(s3[t + 1]));
            }
            const float mt = fmaxf(mx0, mx1) * c;
            const bool raise = mt > m + kRaise;          // always on the first tile (m = -inf)
            const float m_use = raise ? mt : m;
            const float alpha = raise ? ex2_fast(m - m_use) : 1.f;   // 0 when m = -inf
            const bool warp_raise = __any_sync(0xffffffffu, raise) && j > 0;
            // P and O may be touched once P_{j-1} V_{j-1} has landed
            if (!wait_or_abort(&S.p_empty, (j & 1) ^ 1, abort_flag, err, WB_DEVERR_TIMEOUT_EPI)) { ok = false; break; }
            tc_fence_after();
            const uint64_t nm2 = f32x2(-m_use, -m_use);
            uint64_t sum2 = f32x2(0.f, 0.f);
            unsigned char* pb = S.p;
            auto emit = [&](const uint32_t (&sv)[32], int cc) {
                uint32_t pk[16];
#pragma unroll
                for (int t = 0; t < 32; t += 2) {
                    float a0, a1;
                    f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[t]), __uint_as_float(sv[t + 1])), c2, nm2), a0, a1);
                    const float p0 = ex2_fast(a0), p1 = ex2_fast(a1);
                    sum2 = add_f32x2(sum2, f32x2(p0, p1));
                    pk[t >> 1] = pack_bf16x2(p0, p1);
                }
                // keys cc*32 .. cc*32+31: half = cc / 2, 16-byte chunks (cc % 2) * 4 .. +3
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int chunk16 = (cc & 1) * 4 + q4;
                    const uint32_t off = (uint32_t)(cc >> 1) * kTileBytes + row_off +
                                         (uint32_t)((chunk16 ^ (r & 7)) * 16);
                    *reinterpret_cast<uint4*>(pb + off) =
                        make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                }
            };
            emit(s0, 0);
            emit(s1, 1);
            emit(s2, 2);
            emit(s3, 3);
            // rescale O after P is out (the S registers are dead by now)
            if (warp_raise) {                          // warp-uniform: tcgen05.ld/st are collective
                const uint64_t a2 = f32x2(alpha, alpha);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(oa + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < 32; t += 2) {
                        float x0, x1;
                        f32x2_split(mul_f32x2(f32x2(__uint_as_float(o[t]), __uint_as_float(o[t + 1])), a2), x0, x1);
                        o[t] = __float_as_uint(x0);
                        o[t + 1] = __float_as_uint(x1);
                    }
                    tmem_st32(oa + cc * 32, o);
                }
                tmem_wait_st();
            }
            float sl, sh;
            f32x2_split(sum2, sl, sh);
            l = l * alpha + (sl + sh);
            m = m_use;
            // P_j is ready for the tensor core (and O's rescale has landed)
            tc_fence_before();
            fence_proxy_async();
            mbar_arrive(&S.p_full);
        }
        // the last P V product
        if (ok && !wait_or_abort(&S.p_empty, (n_tiles - 1) & 1, abort_flag, err, WB_DEVERR_TIMEOUT_EPI)) ok = false;
        if (ok) {
            tc_fence_after();
            uint32_t o0[32], o1[32];
            tmem_ld32(oa, o0);
            tmem_ld32(oa + 32, o1);
            tmem_wait_ld();
            if (q0 + r < kCtx) {
                const float inv = 1.f / l;
                __nv_bfloat16* dst = out + ((int64_t)row_base + q0 + r) * d + h * 64;
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) {
                    const uint32_t* v = q8 < 4 ? o0 + q8 * 8 : o1 + (q8 - 4) * 8;
                    *reinterpret_cast<uint4*>(dst + q8 * 8) = make_uint4(
                        pack_bf16x2(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                        pack_bf16x2(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                        pack_bf16x2(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                        pack_bf16x2(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

wb_status attn_flash_tc_bf16(const CUtensorMap* tma_qkv, int64_t n_chunks, int d, int heads, void* out,
                             unsigned* err, cudaStream_t s) {
    if (n_chunks > 65535) return fail(WB_ERR_SHAPE, "too many chunks for one attention launch");
    const size_t smem = sizeof(FlashSmem) + kSmemSlack;
    static bool attr[64] = {};
    int dev = 0;
    WB_CUDA(cudaGetDevice(&dev));
    if (!attr[dev & 63]) {
        WB_CUDA(cudaFuncSetAttribute(flash_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        attr[dev & 63] = true;
    }
    dim3 grid((kCtx + kRows - 1) / kRows, heads, (unsigned)n_chunks);
    const int slot = prof_begin(WB_KERNEL_ENC_ATTN, s);
    WB_CUDA(launch_k(flash_tc_kernel, grid, dim3(192), smem, s, *tma_qkv, d,
                     reinterpret_cast<__nv_bfloat16*>(out), err));
    prof_end(slot, s, 4.0 * (double)kCtx * kCtx * 64.0 * heads * (double)n_chunks);
    return WB_OK;
}

}  // namespace wb
