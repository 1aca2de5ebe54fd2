// Encoder self-attention on the 5th-generation tensor cores ("whisper-blaze
// 0.1.8", "Direct Kernel API": encoder_self_attn, no mask; here softmax(Q K^T
// / 8) V per 64-wide head over the 1500 positions of a chunk, bf16 in, fp32
// accumulation).
//
// One CTA = 128 query rows of one (chunk, head); 192 threads:
//   warp 0      TMA: Q once, then K and V tiles of 128 keys into a 3-deep ring
//   warp 1      TMEM owner and MMA issuer (one thread):
//                 S_j  = Q . K_j^T   M 128, N 128, K 64   -> TMEM S[j % 2]
//                 PV_j = P_j . V_j   M 128, N 64,  K 128  -> TMEM PV[j % 2]
//               V is read MN-major straight from its [key][dim] tile.
//   warps 2-5   softmax, one query row per thread (TMEM lane = row): read the
//               S row twice (maximum, then exp2 and sum), write P as bf16 into
//               a 128-byte-swizzled shared tile (double buffered), and keep the
//               fp32 output row in registers: O = O * exp2(m_old - m_new) + PV.
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
constexpr int kSBuf = 1;            // S buffers in TMEM
constexpr int kPBuf = 1;            // P buffers in shared memory
constexpr int kTmemCols = 256;      // S 0-127, PV[0] 128-191, PV[1] 192-255
constexpr int kTileBytes = 128 * 128;            // 128 rows x 64 bf16
constexpr int kSmemSlack = 256;     // alignment slack requested above sizeof(FlashSmem)
constexpr uint32_t kIdescS = UmmaIdesc<128, 128, 1>::value;
constexpr uint32_t kIdescPV = UmmaIdesc<128, 64, 1>::value | (1u << 16);   // B (V) MN-major

struct FlashSmem {
    unsigned char q[kTileBytes];
    unsigned char k[kStages][kTileBytes];
    unsigned char v[kStages][kTileBytes];
    unsigned char p[kPBuf][2 * kTileBytes];       // [buffer][key half]
    uint64_t q_full;
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full[kSBuf], s_empty[kSBuf];
    uint64_t p_full[kPBuf], p_empty[kPBuf];
    uint64_t pv_full[2], pv_empty[2];
    uint64_t drain;
    uint32_t tmem;
    int abort_flag;
};

// Hardware base-2 exponential (MUFU, ~2^-22 relative error; arguments here
// are <= 0 so the result never overflows).
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
        for (int i = 0; i < kSBuf; ++i) { mbar_init(&S.s_full[i], 1); mbar_init(&S.s_empty[i], 128); }
        for (int i = 0; i < kPBuf; ++i) { mbar_init(&S.p_full[i], 128); mbar_init(&S.p_empty[i], 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(&S.pv_full[i], 1); mbar_init(&S.pv_empty[i], 128); }
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
                    const int st = j % kStages, b = j % kSBuf;
                    if (!wait_or_abort(&S.kv_full[st], (j / kStages) & 1, abort_flag, err, WB_DEVERR_TIMEOUT_MMA) ||
                        !wait_or_abort(&S.s_empty[b], ((j / kSBuf) & 1) ^ 1, abort_flag, err, WB_DEVERR_TIMEOUT_MMA)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k_addr = smem_u32(S.k[st]);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_bf16(tmem + b * 128, umma_desc_sw128(q_addr + 32 * k), umma_desc_sw128(k_addr + 32 * k),
                                  kIdescS, k ? 1u : 0u);
                    any = true;
                    umma_commit(&S.s_full[b]);
                }
                if (j >= 1) {        // PV_{j-1} = P_{j-1} V_{j-1}
                    const int i = j - 1, st = i % kStages, b = i & 1, pbf = i % kPBuf;
                    if (!wait_or_abort(&S.p_full[pbf], (i / kPBuf) & 1, abort_flag, err, WB_DEVERR_TIMEOUT_MMA) ||
                        !wait_or_abort(&S.pv_empty[b], ((i >> 1) & 1) ^ 1, abort_flag, err, WB_DEVERR_TIMEOUT_MMA)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t p_addr = smem_u32(S.p[pbf]);
                    const uint32_t v_addr = smem_u32(S.v[st]);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        // A: P, K-major, 64-key halves of 16 KB; B: V rows (keys) of 128 B, MN-major
                        const uint64_t ad = umma_desc_sw128(p_addr + (k >> 2) * kTileBytes + 32 * (k & 3));
                        const uint64_t bd = umma_desc_sw128(v_addr + 2048 * k);
                        umma_bf16(tmem + 128 + b * 64, ad, bd, kIdescPV, k ? 1u : 0u);
                    }
                    umma_commit(&S.pv_full[b]);
                    umma_commit(&S.p_empty[pbf]);
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
        float m = -INFINITY, l = 0.f, o[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) o[i] = 0.f;
        float alpha_prev = 0.f;   // rescale belonging to the PV in flight
        bool ok = true;
        // row swizzle inside a 128-byte atom row
        const uint32_t row_off = (uint32_t)(r >> 3) * 1024 + (uint32_t)(r & 7) * 128;
        for (int j = 0; j <= n_tiles && ok; ++j) {
            if (j < n_tiles) {
                const int b = j % kSBuf, pbf = j % kPBuf;
                if (!wait_or_abort(&S.s_full[b], (j / kSBuf) & 1, abort_flag, err, WB_DEVERR_TIMEOUT_EPI)) { ok = false; break; }
                tc_fence_after();
                const int valid = min(kKeys, kCtx - j * kKeys);
                const bool full = valid == kKeys;          // only the last tile is ragged
                const uint32_t sa = tmem + lane_off + b * 128;
                float mx = -INFINITY;
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t raw[32];
                    tmem_ld32(sa + cc * 32, raw);
                    tmem_wait_ld();
                    if (full) {
#pragma unroll
                        for (int t = 0; t < 32; ++t) mx = fmaxf(mx, __uint_as_float(raw[t]));
                    } else {
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            if (cc * 32 + t < valid) mx = fmaxf(mx, __uint_as_float(raw[t]));
                    }
                }
                const float mn = fmaxf(m, mx * c);
                const float alpha = ex2_fast(m - mn);      // 0 on the first tile (m = -inf)
                // P may be overwritten once the previous PV has consumed it
                if (!wait_or_abort(&S.p_empty[pbf], ((j / kPBuf) & 1) ^ 1, abort_flag, err, WB_DEVERR_TIMEOUT_EPI)) { ok = false; break; }
                float sum = 0.f;
                unsigned char* pb = S.p[pbf];
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t raw[32];
                    tmem_ld32(sa + cc * 32, raw);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int t = 0; t < 32; t += 2) {
                        float p0 = ex2_fast(fmaf(__uint_as_float(raw[t]), c, -mn));
                        float p1 = ex2_fast(fmaf(__uint_as_float(raw[t + 1]), c, -mn));
                        if (!full) {
                            const int col = cc * 32 + t;
                            if (col >= valid) p0 = 0.f;
                            if (col + 1 >= valid) p1 = 0.f;
                        }
                        sum += p0 + p1;
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
                }
                // S[b] has been read; P[b] is ready for the tensor core
                tc_fence_before();
                mbar_arrive(&S.s_empty[b]);
                fence_proxy_async();
                mbar_arrive(&S.p_full[pbf]);
                l = l * alpha + sum;
                m = mn;
                // O holds sum_{i < j-1} at the maximum of tile j-1; add PV_{j-1}
                // (also at that maximum), then bring O to this tile's maximum
                const float a_here = alpha;
                if (j >= 1) {
                    const int i = j - 1, bi = i & 1;
                    if (!wait_or_abort(&S.pv_full[bi], (i >> 1) & 1, abort_flag, err, WB_DEVERR_TIMEOUT_EPI)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t pa = tmem + lane_off + 128 + bi * 64;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t raw[32];
                        tmem_ld32(pa + cc * 32, raw);
                        tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[cc * 32 + t] = o[cc * 32 + t] * alpha_prev + __uint_as_float(raw[t]);
                    }
                    tc_fence_before();
                    mbar_arrive(&S.pv_empty[bi]);
                    // bring O to this tile's maximum
#pragma unroll
                    for (int t = 0; t < 64; ++t) o[t] *= a_here;
                }
                else {
#pragma unroll
                    for (int t = 0; t < 64; ++t) o[t] *= a_here;   // first tile: O is zero
                }
                alpha_prev = 1.f;
            } else {
                // last PV
                const int i = n_tiles - 1, bi = i & 1;
                if (!wait_or_abort(&S.pv_full[bi], (i >> 1) & 1, abort_flag, err, WB_DEVERR_TIMEOUT_EPI)) { ok = false; break; }
                tc_fence_after();
                const uint32_t pa = tmem + lane_off + 128 + bi * 64;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t raw[32];
                    tmem_ld32(pa + cc * 32, raw);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < 32; ++t) o[cc * 32 + t] += __uint_as_float(raw[t]);
                }
                tc_fence_before();
                mbar_arrive(&S.pv_empty[bi]);
            }
        }
        if (ok && q0 + r < kCtx) {
            const float inv = 1.f / l;
            __nv_bfloat16* dst = out + ((int64_t)row_base + q0 + r) * d + h * 64;
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                const float* v = o + q8 * 8;
                *reinterpret_cast<uint4*>(dst + q8 * 8) =
                    make_uint4(pack_bf16x2(v[0] * inv, v[1] * inv), pack_bf16x2(v[2] * inv, v[3] * inv),
                               pack_bf16x2(v[4] * inv, v[5] * inv), pack_bf16x2(v[6] * inv, v[7] * inv));
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
