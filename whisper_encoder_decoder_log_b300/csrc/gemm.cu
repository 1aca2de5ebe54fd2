// Dense contractions of the encoder/decoder on the 5th-generation tensor
// cores ("whisper-blaze 0.1.8" lists FP16/FP8 tensor-core GEMMs fed by TMA for
// the QKV, output and FFN projections; here they are tcgen05 with TMEM
// accumulators for sm_103a).
//
// Kernel shape: persistent, 320 threads in three roles.
//   warp 0      TMA producer: 128 x 128-byte A box and BN x 128-byte B box per
//               k-block into a STAGES-deep ring (128-byte swizzle).
//   warp 1      owns TMEM (2 x BN fp32 columns: a double-buffered accumulator)
//               and, from one thread, issues tcgen05.mma (M 128, N BN, K 16
//               for bf16 / 32 for E4M3) and tcgen05.commit to release stages
//               and to hand a finished accumulator to the epilogue.
//               Large GEMMs run on CTA pairs (cta_group::2, M 256 over two
//               SMs, each SM loading half of the B tile): see gemm_tc_kernel.
//   warps 2-9   epilogue: two warps per TMEM lane quarter, alternate
//               32-column chunks: tcgen05.ld, scale, bias, GELU, positional
//               table, residual accumulate, store.
// Tiles are visited in groups of 16 M-tiles so that the A panel of a group and
// the whole B operand stay in L2.  Every mbarrier wait is bounded; a wait that
// runs out records an error bit and the CTA winds down (waiting, bounded, for
// its own TMA copies and MMAs) before releasing TMEM.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "gemm.cuh"
#include "prof.cuh"

namespace wb {

namespace {

constexpr int kBM = 128;
constexpr int kRowBytes = 128;       // one k-block row: 64 bf16 or 128 E4M3
constexpr int kGroupM = 16;

// fp32 epilogue staging: one 32 x 32 fp32 block per epilogue warp, so that
// global stores and reductions go out one 128-byte row segment at a time.
constexpr int kEpiStageBytes = 8 * 32 * 32 * 4;

// PAIR: each CTA of a pair holds half of the BN rows of B.
template <int BN, bool PAIR = false>
struct Cfg {
    static constexpr int A_BYTES = kBM * kRowBytes;
    static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * kRowBytes;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (192 * 1024) / STAGE_BYTES > 8 ? 8 : (192 * 1024) / STAGE_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int SMEM = STAGES * STAGE_BYTES + kEpiStageBytes + 1024 + 256;
};

struct GemmArgs {
    int64_t rows;            // rows per batch
    int64_t batches;
    int64_t N, K;
    int64_t mt_per_batch, mt_total, nt_total, tiles;
    int kblocks;            // k-blocks of the longest split
    int kb_all;             // k-blocks of the whole K
    int ksplit;             // K partitions; > 1 adds partial tiles atomically
    int stages;             // smem ring depth (<= the compile-time maximum)
    int w_const;            // the weight operand is constant: load it before the grid dependency wait
    int b_kwrap;
    // Failure-detection test hook: when non-zero, the MMA issuer first waits
    // this many ns on a barrier nothing arrives on, and takes the same
    // give-up path as a pipeline wait that ran out.
    uint64_t stall_ns;
    GemmEpi epi;
};

__device__ __forceinline__ void tile_coords(const GemmArgs& a, int64_t t, int64_t& mt, int64_t& nt) {
    t /= a.ksplit;
    const int64_t group = (int64_t)kGroupM * a.nt_total;
    const int64_t gid = t / group;
    const int64_t first_m = gid * kGroupM;
    const int64_t gsz = min((int64_t)kGroupM, a.mt_total - first_m);
    const int64_t local = t % group;
    mt = first_m + local % gsz;
    nt = local / gsz;
}

// Per-row epilogue arithmetic of an fp32 output (row r of batch b, columns
// n0..n0+31): scales, bias (first K partition only), GELU, added matrix.
__device__ __forceinline__ void transform_f32(const GemmArgs& a, int64_t b, int64_t r, int64_t n0, float (&v)[32],
                                              int ks) {
    const GemmEpi& e = a.epi;
    const int64_t N = a.N;
    const bool full = n0 + 32 <= N;
    // column vectors as 16-byte loads when the chunk is whole and aligned
    const bool v4 = full && (n0 & 3) == 0;
    if (e.row_scale || e.col_scale) {
        const float rs = e.row_scale ? e.row_scale[b * a.rows + r] : 1.f;
        if (e.col_scale && v4 && (reinterpret_cast<uintptr_t>(e.col_scale) & 15) == 0) {
            const float4* c4 = reinterpret_cast<const float4*>(e.col_scale + n0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 c = c4[q];
                v[4 * q] *= rs * c.x; v[4 * q + 1] *= rs * c.y; v[4 * q + 2] *= rs * c.z; v[4 * q + 3] *= rs * c.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float cs = (e.col_scale && (full || n0 + j < N)) ? e.col_scale[n0 + j] : 1.f;
                v[j] *= rs * cs;
            }
        }
    }
    if (e.bias && ks == 0) {
        if (v4 && (reinterpret_cast<uintptr_t>(e.bias) & 15) == 0) {
            const float4* b4 = reinterpret_cast<const float4*>(e.bias + n0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 c = b4[q];
                v[4 * q] += c.x; v[4 * q + 1] += c.y; v[4 * q + 2] += c.z; v[4 * q + 3] += c.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += (full || n0 + j < N) ? e.bias[n0 + j] : 0.f;
        }
    }
    if (e.gelu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_f(v[j]);
    }
    if (e.add) {
        const float* ap = e.add + r * e.ld_add + n0;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += (full || n0 + j < N) ? ap[j] : 0.f;
    }
}

__device__ __forceinline__ void store_chunk(const GemmArgs& a, int64_t b, int64_t r, int64_t n0,
                                            float (&v)[32], int ks) {
    const GemmEpi& e = a.epi;
    const int64_t N = a.N;
    const bool full = n0 + 32 <= N;
    const bool vec = full && e.vec;
    if (a.ksplit > 1) {
        // split-K partial tile: fp32 output (zeroed beforehand unless it is a
        // residual), bias from the first split only, no nonlinearity
        const float rs = e.row_scale ? e.row_scale[b * a.rows + r] : 1.f;
        const int64_t obr = e.out_batch_rows ? e.out_batch_rows : a.rows;
        float* dst = reinterpret_cast<float*>(e.out) + (b * obr + e.out_row_offset + r) * e.ldo + n0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (!full && n0 + j >= N) continue;
            float x = v[j];
            if (e.row_scale || e.col_scale) x *= rs * (e.col_scale ? e.col_scale[n0 + j] : 1.f);
            if (e.bias && ks == 0) x += e.bias[n0 + j];
            v[j] = x;
        }
        if (vec) {
            float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int q = 0; q < 8; ++q) atomicAdd(d4 + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n0 + j < N) atomicAdd(dst + j, v[j]);
        }
        return;
    }
    // scale, bias, GELU, positional table
    if (e.row_scale || e.col_scale) {
        const float rs = e.row_scale ? e.row_scale[b * a.rows + r] : 1.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float cs = (e.col_scale && (full || n0 + j < N)) ? e.col_scale[n0 + j] : 1.f;
            v[j] *= rs * cs;
        }
    }
    if (e.bias) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += (full || n0 + j < N) ? e.bias[n0 + j] : 0.f;
    }
    if (e.gelu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_f(v[j]);
    }
    if (e.add) {
        const float* ap = e.add + r * e.ld_add + n0;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += (full || n0 + j < N) ? ap[j] : 0.f;
    }
    int64_t orow;
    void* base;
    if (e.mode == MODE_CROSS_KV) {
        const int64_t m = b * a.rows + r;
        const int64_t ch = m / kCtx, s = m % kCtx;
        const int64_t two_d = 2 * (int64_t)e.ckv_d;
        const int64_t l = n0 / two_d, rem = n0 % two_d;
        const int64_t kv = rem / e.ckv_d, h = (rem % e.ckv_d) / 64, c0 = n0 % 64;
        const int64_t off = ((((l * e.ckv_chunks + ch) * 2 + kv) * e.ckv_heads + h) * kCtx + s) * 64 + c0;
        if (e.out_type == OUT_F32) {
            float4* d4 = reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + off);
#pragma unroll
            for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            return;
        }
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(e.out) + off;
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        return;
    }
    const int64_t obr = e.out_batch_rows ? e.out_batch_rows : a.rows;
    orow = b * obr + e.out_row_offset + r;
    base = e.out;
    if (e.out_type == OUT_BF16X2) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(base) + orow * e.ldo + n0;
        float lo[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) lo[j] = v[j] - __bfloat162float(__float2bfloat16_rn(v[j]));
        if (vec) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            uint4* l4 = reinterpret_cast<uint4*>(dst + N);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                d4[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                   pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
                l4[q] = make_uint4(pack_bf16x2(lo[8 * q + 0], lo[8 * q + 1]), pack_bf16x2(lo[8 * q + 2], lo[8 * q + 3]),
                                   pack_bf16x2(lo[8 * q + 4], lo[8 * q + 5]), pack_bf16x2(lo[8 * q + 6], lo[8 * q + 7]));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n0 + j < N) { dst[j] = f2bf(v[j]); dst[N + j] = f2bf(lo[j]); }
        }
    } else if (e.out_type == OUT_BF16) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(base) + orow * e.ldo + n0;
        if (vec) {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                d4[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]),
                                   pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                   pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                                   pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n0 + j < N) dst[j] = f2bf(v[j]);
        }
    } else {
        float* dst = reinterpret_cast<float*>(base) + orow * e.ldo + n0;
        const bool acc = e.out_type == OUT_F32_ACC;
        if (vec) {
            float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float4 w = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                if (acc) {
                    const float4 o = d4[q];
                    w.x += o.x; w.y += o.y; w.z += o.z; w.w += o.w;
                }
                d4[q] = w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n0 + j < N) dst[j] = acc ? dst[j] + v[j] : v[j];
        }
    }
}

// Swapped operands (small M): TMEM lane = output feature n, column = row m.
// One call stores 32 rows m0 .. m0+31 of feature n; lanes of a warp hold
// consecutive n, so every store instruction is coalesced.
// Swapped form: lane = output feature n (cs, bias: its column scale and bias,
// the bias only on the first K partition), the 32 values = rows m0..m0+31.
// rs_lane is row m0 + lane's scale, loaded before the accumulator was ready
// and broadcast by shuffles, so no store waits on a load.
__device__ __forceinline__ void store_swap(const GemmArgs& a, int64_t n, int64_t m0, const uint32_t (&raw)[32],
                                           float cs, float bias, float rs_lane) {
    const GemmEpi& e = a.epi;
    const int64_t left = a.rows - m0;
    const int nrow = left < 32 ? (int)left : 32;
    const bool nok = n < a.N;
    const bool red = a.ksplit > 1 || e.out_type == OUT_F32_ACC;
    float* dst = reinterpret_cast<float*>(e.out) + m0 * e.ldo + n;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float rs = __shfl_sync(0xffffffffu, rs_lane, j);
        if (nok && j < nrow) {
            const float v = __uint_as_float(raw[j]) * rs * cs + bias;
            if (red) atomicAdd(dst + j * e.ldo, v);    // result unused: a reduction
            else dst[j * e.ldo] = v;
        }
    }
}

// K partition of tile t: k-blocks [kb0, kb1).  Partitions differ by at most
// one k-block, so any ksplit <= kb_all spreads K evenly.
__device__ __forceinline__ void split_range(const GemmArgs& a, int64_t t, int& kb0, int& kb1) {
    const int ks = (int)(t % a.ksplit);
    kb0 = (int)((int64_t)ks * a.kb_all / a.ksplit);
    kb1 = (int)((int64_t)(ks + 1) * a.kb_all / a.ksplit);
}

// One CTA's work: tiles c, c + G, c + 2 G, ... (G CTAs or CTA pairs), each
// with its K partition [kb0, kb1) (split_range); kb0 == 0 marks the part
// that adds the bias.
struct WorkIter {
    int64_t cur, end, step;
};
__device__ __forceinline__ WorkIter work_begin(const GemmArgs& a, int64_t c, int64_t g) {
    WorkIter w;
    w.cur = c;
    w.end = a.tiles;
    w.step = g;
    return w;
}
__device__ __forceinline__ bool work_next(const GemmArgs& a, WorkIter& w, int64_t& mt, int64_t& nt, int& kb0,
                                          int& kb1) {
    if (w.cur >= w.end) return false;
    tile_coords(a, w.cur, mt, nt);
    split_range(a, w.cur, kb0, kb1);
    w.cur += w.step;
    return true;
}

// Fold the per-thread maxima of one warp's 32 consecutive rows into the
// group maxima: the rows span at most two groups (amax_rows >= 32), so two
// warp reductions and at most two atomics per warp and tile.
__device__ __forceinline__ void epi_group_amax(unsigned* amax, int64_t group_rows, int64_t row, bool row_ok, float m) {
    const int64_t grp = row_ok ? row / group_rows : -1;
    const long long g0 = __shfl_sync(0xffffffffu, (long long)grp, 0);
    if (g0 < 0) return;                       // lane 0 holds the warp's first row
    const float m0 = warp_max(grp == g0 ? m : 0.f);
    const float m1 = warp_max(grp == g0 + 1 ? m : 0.f);
    if ((threadIdx.x & 31) == 0) {
        atomicMax(amax + g0, __float_as_uint(m0));
        if (m1 > 0.f) atomicMax(amax + g0 + 1, __float_as_uint(m1));
    }
}

constexpr int kEpiWarps = 8;                       // two per TMEM lane quarter
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;  // producer + MMA + epilogue

// PAIR: a cluster of two CTAs computes a 256 x BN tile with cta_group::2 MMAs:
// CTA r of the pair holds rows [128 r, 128 r + 128) of A and rows
// [BN/2 r, BN/2 r + BN/2) of B in its shared memory (each CTA's own TMA
// copies, not shared with the other) and the accumulator of its 128 rows in
// its TMEM.  One thread of the leader CTA (rank 0) issues the MMAs, which
// read both CTAs' shared memory, so a k-block costs each SM's L2 feed
// A + B/2 instead of A + B.  Hand-offs across the pair:
//   stage loaded   both CTAs' copies of a stage count their bytes on the
//                  leader's full barrier (cta_group::2 copies), which the
//                  leader arms for both halves;
//   stage free     the leader's MMA commit arrives on both CTAs' empty
//                  barriers (one commit per barrier);
//   tile ready     likewise on both CTAs' accumulator-full barriers;
//   tile drained   each peer epilogue warp arrives on the leader's
//                  accumulator-empty barrier.
// Every wait stays bounded; a CTA that gives up leaves its peer to time out
// in turn, and both meet at the final cluster barrier before TMEM is released.
template <int BN, bool FP8, bool SWAP, bool PAIR = false>
__global__ void __launch_bounds__(kGemmThreads, SWAP ? 2 : 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
               const GemmArgs args, unsigned* err) {
    using C = Cfg<BN, PAIR>;
    const int STAGES = args.stages;
    constexpr uint32_t IDESC = UmmaIdesc<PAIR ? 2 * kBM : kBM, BN, FP8 ? 0 : 1>::value;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* epi_stage = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + kEpiStageBytes);
    uint64_t* empty_bar = full_bar + STAGES;
    uint64_t* tfull_bar = empty_bar + STAGES;     // [2]
    uint64_t* tempty_bar = tfull_bar + 2;         // [2]
    uint64_t* drain_bar = tempty_bar + 2;         // [1]
    uint64_t* stall_bar = drain_bar + 1;          // [1] never arrived on (stall_ns)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stall_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = PAIR ? (int)cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int64_t cta_id = PAIR ? blockIdx.x / 2 : blockIdx.x;      // CTA (pair) index: 256-row tiles when PAIR
    const int64_t n_ctas = PAIR ? gridDim.x / 2 : gridDim.x;
    // M tile (128 rows) of this CTA within tile index mt
    auto my_mt = [&](int64_t mt) { return PAIR ? 2 * mt + rank : mt; };
    // try_wait at cluster scope where the peer (or its tensor core) arrives
    auto try_wait = [&](uint64_t* bar, uint32_t parity) {
        return PAIR ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull_bar[i], 1);
            // local epilogue threads, plus one arrival per peer epilogue warp
            mbar_init(&tempty_bar[i], 32 * kEpiWarps + (PAIR ? kEpiWarps : 0));
        }
        mbar_init(drain_bar, 1);
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tma_a);
        tma_prefetch_desc(&tma_b);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();    // both CTAs' barriers exist before either arrives on the other's
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const bool producer = warp == 0 && lane == 0;
    if (!producer) {
        griddep_wait();
        griddep_launch();   // barriers and TMEM are set up; now wait for the producer kernels
    }

    if (warp == 0) {
        if (lane == 0) {
            // PAIR: every copy of the pair counts on the leader's full barrier
            const uint32_t full_leader = PAIR ? mapa_shared(full_bar, 0) : 0u;
            // Arm a stage: the leader expects both CTAs' bytes.
            auto arm = [&](int stage) {
                if (!PAIR || leader) mbar_arrive_expect_tx(&full_bar[stage], (PAIR ? 2 : 1) * C::STAGE_BYTES);
            };
            // Weight half of one stage (swapped: A holds the weights, else B).
            auto load_w = [&](int stage, int64_t mt, int n0, int kx) {
                unsigned char* sa = smem + stage * C::STAGE_BYTES;
                const int kw = args.b_kwrap ? kx % args.b_kwrap : kx;
                if (SWAP) tma_load_3d(sa, &tma_a, &full_bar[stage], kw, (int)(mt * kBM), 0);
                else if (PAIR) tma_load_2d_pair(sa + C::A_BYTES, &tma_b, full_leader + 8u * (uint32_t)stage, kw,
                                                n0 + rank * (BN / 2));
                else tma_load_2d(sa + C::A_BYTES, &tma_b, &full_bar[stage], kw, n0);
            };
            // Constant weights do not depend on the kernels this one waits
            // for: the first ring stages fetch them before the wait, which
            // overlaps the previous kernel's tail (programmatic launch).
            int pre = 0;
            if (args.w_const) {
                WorkIter wi = work_begin(args, cta_id, n_ctas);
                int64_t mt, nt;
                int kb0, kb1;
                while (pre < STAGES && work_next(args, wi, mt, nt, kb0, kb1)) {
                    for (int kb = kb0; kb < kb1 && pre < STAGES; ++kb, ++pre) {
                        arm(pre);
                        load_w(pre, mt, (int)(nt * BN), kb * (FP8 ? 128 : 64));
                    }
                }
            }
            griddep_wait();
            griddep_launch();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_parity = 0;      // bit s: stage s was loaded / its last phase
            bool ok = true;
            int it = 0;
            WorkIter wi = work_begin(args, cta_id, n_ctas);
            int64_t mt, nt;
            int kb0, kb1;
            while (ok && work_next(args, wi, mt, nt, kb0, kb1)) {
                const int b = PAIR ? 0 : (int)(mt / args.mt_per_batch);
                const int r0 = PAIR ? (int)(my_mt(mt) * kBM) : (int)((mt % args.mt_per_batch) * kBM);
                const int n0 = (int)(nt * BN);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int kx = kb * (FP8 ? 128 : 64);
                    if (it >= pre) {
                        bool got = false;
                        for (WaitClock clk; !clk.expired();) {
                            if (try_wait(&empty_bar[stage], phase ^ 1)) { got = true; break; }
                            if (*abort_flag) break;
                        }
                        if (!got) {
                            wb_set_error(err, WB_DEVERR_TIMEOUT_TMA);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        arm(stage);
                        load_w(stage, mt, n0, kx);
                    }
                    // activation half: swapped -> B (BN activation rows), else A
                    unsigned char* sa = smem + stage * C::STAGE_BYTES;
                    if (SWAP) tma_load_2d(sa + C::A_BYTES, &tma_b, &full_bar[stage], kx, n0);
                    else if (PAIR) tma_load_3d_pair(sa, &tma_a, full_leader + 8u * (uint32_t)stage, kx, r0, b);
                    else tma_load_3d(sa, &tma_a, &full_bar[stage], kx, r0, b);
                    issued |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }

            // never leave TMA writes in flight into shared memory: the leader's
            // full barriers count both CTAs' copies (the peer leaves only
            // after the leader, at the final cluster barrier)
            if (!PAIR || leader)
                for (int s = 0; s < STAGES; ++s)
                    if ((issued >> s) & 1u)
                        mbar_wait(&full_bar[s], (last_parity >> s) & 1u, err, WB_DEVERR_TIMEOUT_TMA);
        }
    } else if (warp == 1) {
        if (lane == 0 && (!PAIR || leader)) {
            // shared::cluster addresses of both CTAs' barriers (PAIR)
            const uint32_t empty_c[2] = {PAIR ? mapa_shared(empty_bar, 0) : 0u, PAIR ? mapa_shared(empty_bar, 1) : 0u};
            const uint32_t tfull_c[2] = {PAIR ? mapa_shared(tfull_bar, 0) : 0u, PAIR ? mapa_shared(tfull_bar, 1) : 0u};
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            bool any = false;
            if (args.stall_ns) {
                bool got = false;
                for (WaitClock clk(args.stall_ns); !clk.expired();)
                    if (mbar_try_wait(stall_bar, 0)) { got = true; break; }
                if (!got) { wb_set_error(err, WB_DEVERR_TIMEOUT_MMA); *abort_flag = 1; ok = false; }
            }
            WorkIter wi = work_begin(args, cta_id, n_ctas);
            int64_t mt_w, nt_w;
            int kb0, kb1;
            for (; ok && work_next(args, wi, mt_w, nt_w, kb0, kb1); ++local) {
                const int acc = local & 1;
                const uint32_t aphase = (local >> 1) & 1;
                bool got = false;
                for (WaitClock clk; !clk.expired();) {
                    if (try_wait(&tempty_bar[acc], aphase ^ 1)) { got = true; break; }
                    if (*abort_flag) break;
                }
                if (!got) { wb_set_error(err, WB_DEVERR_TIMEOUT_MMA); *abort_flag = 1; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < kb1 - kb0; ++kb) {
                    got = false;
                    for (WaitClock clk; !clk.expired();) {
                        if (try_wait(&full_bar[stage], phase)) { got = true; break; }
                        if (*abort_flag) break;
                    }
                    if (!got) { wb_set_error(err, WB_DEVERR_TIMEOUT_MMA); *abort_flag = 1; ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = umma_desc_sw128(a_addr + 32 * k);
                        const uint64_t bd = umma_desc_sw128(b_addr + 32 * k);
                        const uint32_t accum = (kb | k) ? 1u : 0u;
                        if (PAIR) {
                            if (FP8) umma_fp8_pair(d_tmem, ad, bd, IDESC, accum);
                            else umma_bf16_pair(d_tmem, ad, bd, IDESC, accum);
                        } else {
                            if (FP8) umma_fp8(d_tmem, ad, bd, IDESC, accum);
                            else umma_bf16(d_tmem, ad, bd, IDESC, accum);
                        }
                    }
                    any = true;
                    if (PAIR) {   // both CTAs' copies of the stage are free
                        umma_commit_pair(empty_c[0] + 8u * (uint32_t)stage);
                        umma_commit_pair(empty_c[1] + 8u * (uint32_t)stage);
                    } else {
                        umma_commit(&empty_bar[stage]);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if (PAIR) {
                    umma_commit_pair(tfull_c[0] + 8u * (uint32_t)acc);
                    umma_commit_pair(tfull_c[1] + 8u * (uint32_t)acc);
                } else {
                    umma_commit(&tfull_bar[acc]);
                }
            }
            // all issued MMAs complete before TMEM can be released
            if (any) {
                if (PAIR) umma_commit_pair(mapa_shared(drain_bar, 0));
                else umma_commit(drain_bar);
                mbar_wait(drain_bar, 0, err, WB_DEVERR_TIMEOUT_MMA);
            }
        }
    } else {
        // epilogue warps 2..9: lane quarter g = warp % 4 (each quarter twice),
        // the two warps of a quarter take alternate 32-column chunks
        const int g = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t tempty_leader = PAIR ? mapa_shared(tempty_bar, 0) : 0u;
        int local = 0;
        WorkIter wi = work_begin(args, cta_id, n_ctas);
        int64_t mt, nt;
        int kb0, kb1;
        for (; work_next(args, wi, mt, nt, kb0, kb1); ++local) {
            const int acc = local & 1;
            const uint32_t aphase = (local >> 1) & 1;
            const int ks = kb0 == 0 ? 0 : 1;     // 0: the tile's first K part (bias, plain stores)
            // swapped form: this lane's column scale and bias and its rows'
            // scales (chunks c = half, half + 2, ...) go out before the wait
            constexpr int kSwapChunks = (BN / 32 + 1) / 2;
            float sw_cs = 1.f, sw_bias = 0.f, sw_rs[kSwapChunks];
            if (SWAP) {
                const int64_t n = mt * kBM + g * 32 + lane;
                const bool nok = n < args.N;
                if (args.epi.col_scale && nok) sw_cs = args.epi.col_scale[n];
                if (args.epi.bias && nok && ks == 0) sw_bias = args.epi.bias[n];
#pragma unroll
                for (int i = 0; i < kSwapChunks; ++i) {
                    const int64_t m = nt * BN + (half + 2 * i) * 32 + lane;
                    sw_rs[i] = (args.epi.row_scale && m < args.rows) ? args.epi.row_scale[m] : 1.f;
                }
            }
            bool got = false;
            for (WaitClock clk; !clk.expired();) {
                if (try_wait(&tfull_bar[acc], aphase)) { got = true; break; }
                if (*abort_flag) break;
            }
            if (!got) { wb_set_error(err, WB_DEVERR_TIMEOUT_EPI); *abort_flag = 1; break; }
            tc_fence_after();
            if (PAIR) mt = my_mt(mt);     // one batch: M tile index = row tile
            const int64_t b = PAIR ? 0 : mt / args.mt_per_batch;
            const int64_t r = (PAIR ? mt : mt % args.mt_per_batch) * kBM + g * 32 + lane;
            const bool row_ok = r < args.rows;
            const uint32_t taddr = tmem_base + ((uint32_t)(g * 32) << 16) + acc * BN;
            if (SWAP) {
                const int64_t n = mt * kBM + g * 32 + lane;      // output feature of this lane
#pragma unroll
                for (int i = 0; i < kSwapChunks; ++i) {
                    const int c = half + 2 * i;
                    if (c >= BN / 32 || nt * BN + c * 32 >= args.rows) break;   // warp-uniform
                    uint32_t raw[32];
                    tmem_ld32(taddr + c * 32, raw);
                    tmem_wait_ld();
                    store_swap(args, n, nt * BN + c * 32, raw, sw_cs, sw_bias, sw_rs[i]);
                }
                tc_fence_before();
                mbar_arrive(&tempty_bar[acc]);
                continue;
            }
            const GemmEpi& e = args.epi;
            // fp32 stores and split-K reductions are staged; a residual update
            // without split-K reads its destination: it stays in the thread's
            // row, where 8 float4 loads go out at once
            const bool staged = e.mode == MODE_PLAIN &&
                                (e.out_type == OUT_F32 || (e.out_type == OUT_F32_ACC && args.ksplit > 1));
            // bf16 rows go out as full 64-byte segments (8 rows per instruction)
            const bool staged16 = e.mode == MODE_PLAIN && e.out_type == OUT_BF16 && e.vec && args.ksplit == 1 &&
                                  (args.N & 7) == 0;
            float* stg = epi_stage + (warp - 2) * 32 * 32;
            float tmax = 0.f;     // largest |v| of this thread's row in the tile (e.amax)
#pragma unroll 1
            for (int c = half; c < BN / 32; c += 2) {
                uint32_t raw[32];
                tmem_ld32(taddr + c * 32, raw);
                tmem_wait_ld();
                const int64_t n0 = nt * BN + c * 32;
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(raw[j]);
                if (staged16) {
                    if (row_ok && n0 < args.N) transform_f32(args, b, r, n0, v, 0);
                    uint4* s4 = reinterpret_cast<uint4*>(stg);        // [32 rows][4 x 16 B]
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        s4[lane * 4 + (q ^ ((lane >> 1) & 3))] =
                            make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                       pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
                    __syncwarp();
                    const int pq = lane & 3;                          // 16-byte piece of the row segment
                    const int64_t col = n0 + pq * 8;
                    const int64_t rq = (PAIR ? mt : mt % args.mt_per_batch) * kBM + g * 32;
                    const int64_t obr = e.out_batch_rows ? e.out_batch_rows : args.rows;
                    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(e.out) + (b * obr + e.out_row_offset) * e.ldo + col;
                    if (col < args.N) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int rr = (lane >> 2) + 8 * i;
                            if (rq + rr < args.rows)
                                *reinterpret_cast<uint4*>(ob + (rq + rr) * e.ldo) = s4[rr * 4 + (pq ^ ((rr >> 1) & 3))];
                        }
                    }
                    __syncwarp();
                    continue;
                }
                if (!staged) {
                    if (row_ok && n0 < args.N) store_chunk(args, b, r, n0, v, ks);
                    continue;
                }
                // fp32 output: transform in the thread's row, then transpose the
                // 32 x 32 block through shared memory (16-byte chunks XOR-swizzled
                // by row) and write one 128-byte row segment per instruction
                if (row_ok && n0 < args.N) {
                    transform_f32(args, b, r, n0, v, ks);
                    if (e.amax) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (n0 + j < args.N) tmax = fmaxf(tmax, fabsf(v[j]));
                    }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4*>(stg + lane * 32 + ((q ^ (lane & 7)) << 2)) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                __syncwarp();
                const int64_t rq = (PAIR ? mt : mt % args.mt_per_batch) * kBM + g * 32;   // first row of the quarter
                const int64_t obr = e.out_batch_rows ? e.out_batch_rows : args.rows;
                const bool reduce = args.ksplit > 1;             // partial tiles of one output
                float* obase = reinterpret_cast<float*>(e.out) + (b * obr + e.out_row_offset) * e.ldo;
                if (e.vec) {
                    // lane = (row i4 of 4, 16-byte piece q of 8): one instruction
                    // writes 4 rows x 128 bytes
                    const int i4 = lane >> 3, q = lane & 7;
                    const int64_t col = n0 + 4 * q;
#pragma unroll 2
                    for (int pp = 0; pp < 8; ++pp) {
                        const int rr = 4 * pp + i4;
                        if (rq + rr >= args.rows) break;
                        const float4 x = *reinterpret_cast<const float4*>(stg + rr * 32 + ((q ^ (rr & 7)) << 2));
                        float* dst = obase + (rq + rr) * e.ldo + col;
                        if (col + 3 < args.N) {
                            if (reduce) atomicAdd(reinterpret_cast<float4*>(dst), x);   // a reduction
                            else *reinterpret_cast<float4*>(dst) = x;
                        } else {
                            const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                if (col + j < args.N) {
                                    if (reduce) atomicAdd(dst + j, xs[j]);
                                    else dst[j] = xs[j];
                                }
                        }
                    }
                } else {
                    const int64_t col = n0 + lane;
                    if (col < args.N) {
#pragma unroll 4
                        for (int rr = 0; rr < 32; ++rr) {
                            if (rq + rr >= args.rows) break;
                            const float x = stg[rr * 32 + ((((lane >> 2) ^ (rr & 7))) << 2) + (lane & 3)];
                            float* dst = obase + (rq + rr) * e.ldo + col;
                            if (reduce) atomicAdd(dst, x);   // result unused: a reduction
                            else *dst = x;
                        }
                    }
                }
                __syncwarp();
            }
            if (e.amax) epi_group_amax(e.amax, e.amax_rows, b * args.rows + r, row_ok, tmax);
            tc_fence_before();
            if (!PAIR || leader) {
                mbar_arrive(&tempty_bar[acc]);
            } else {   // one arrival per peer warp on the leader's barrier, after all its lanes' loads
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * (uint32_t)acc);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    // neither CTA of a pair releases TMEM (or leaves) while the leader's MMAs
    // may still write the peer's TMEM or either CTA may arrive on the other's
    // barriers
    if (PAIR) cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        if (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
        else tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host: TMA
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

wb_status get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return fail(WB_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    return WB_OK;
}

wb_status encode_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box, bool fp8) {
    uint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          rank, const_cast<void*>(ptr), dims, strides_bytes, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(WB_ERR_SHAPE, "cuTensorMapEncodeTiled rejected an operand");
    return WB_OK;
}

int g_num_sms = 0;

// One-shot failure-detection hook (wb_debug_stall_next_gemm).
std::atomic<uint64_t> g_stall_next{0};

}  // namespace

wb_status make_tma_2d_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                           uint32_t box_inner, uint32_t box_outer) {
    if (wb_status st = get_encoder()) return st;
    if (!aligned16(ptr) || row_stride_bytes % 16) return fail(WB_ERR_ALIGN, "TMA operand alignment");
    uint64_t dims[2] = {inner, outer};
    uint64_t strides[1] = {row_stride_bytes};
    uint32_t box[2] = {box_inner, box_outer};
    return encode_map(m, ptr, 2, dims, strides, box, false);
}

namespace {

template <int BN, bool FP8, bool SWAP>
wb_status launch_tc(const GemmPlan& p, GemmArgs a, unsigned* err, cudaStream_t s, int max_ctas) {
    using C = Cfg<BN>;
    static bool attr_set[64] = {};
    int dev = 0;
    WB_CUDA(cudaGetDevice(&dev));
    if (!attr_set[dev & 63]) {
        WB_CUDA(cudaFuncSetAttribute(gemm_tc_kernel<BN, FP8, SWAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::SMEM));
        attr_set[dev & 63] = true;
    }
    // A CTA that sees few k-blocks needs a shallow ring; the smaller footprint
    // lets several CTAs share an SM (bounded by shared memory and TMEM).
    const int64_t kb_per_cta = (int64_t)a.kblocks * ((a.tiles + num_sms() - 1) / num_sms());
    a.stages = (int)std::max<int64_t>(2, std::min<int64_t>(C::STAGES, kb_per_cta));
    const int smem = a.stages * C::STAGE_BYTES + kEpiStageBytes + 1024 + 256;
    int occ = 1;
    WB_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemm_tc_kernel<BN, FP8, SWAP>, kGemmThreads, smem));
    const int per_sm = std::max(1, std::min({occ, 512 / C::TMEM_COLS, 4}));
    int grid = num_sms() * per_sm;
    if (max_ctas > 0) grid = std::min(grid, max_ctas);
    grid = (int)std::min<int64_t>(grid, a.tiles);
    if (grid <= 0) return WB_OK;
    WB_CUDA(launch_k(gemm_tc_kernel<BN, FP8, SWAP>, dim3(grid), dim3(kGemmThreads), smem, s, p.tma_a, p.tma_b, a, err));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

// CTA pairs (clusters of two, cta_group::2 MMAs over 256-row tiles); a.tiles
// counts 256-row tiles.
template <int BN, bool FP8>
wb_status launch_tc_pair(const GemmPlan& p, GemmArgs a, unsigned* err, cudaStream_t s) {
    using C = Cfg<BN, true>;
    auto kern = gemm_tc_kernel<BN, FP8, false, true>;
    static bool attr_set[64] = {};
    int dev = 0;
    WB_CUDA(cudaGetDevice(&dev));
    if (!attr_set[dev & 63]) {
        WB_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
        attr_set[dev & 63] = true;
    }
    const int64_t pairs_per_wave = num_sms() / 2;
    const int64_t kb_per_cta = (int64_t)a.kblocks * ((a.tiles + pairs_per_wave - 1) / pairs_per_wave);
    a.stages = (int)std::max<int64_t>(2, std::min<int64_t>(C::STAGES, kb_per_cta));
    const int smem = a.stages * C::STAGE_BYTES + kEpiStageBytes + 1024 + 256;
    // as many clusters as can be resident at once (persistent)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs_per_wave));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    WB_CUDA(cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg));
    if (clusters <= 0) return fail(WB_ERR_CUDA, "no resident CTA pair for the paired GEMM");
    clusters = (int)std::min<int64_t>(clusters, a.tiles);
    WB_CUDA(launch_k_cluster(kern, dim3(2 * clusters), dim3(kGemmThreads), smem, s, 2, p.tma_a, p.tma_b, a, err));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

}  // namespace

int num_sms() {
    if (!g_num_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    return g_num_sms;
}

wb_status gemm_plan(GemmPlan* plan, const GemmOperand& A, const GemmOperand& B, int64_t N, int64_t K,
                    bool fp8, int bn, int64_t b_kwrap, bool pair) {
    if (wb_status st = get_encoder()) return st;
    const int esz = fp8 ? 1 : 2;
    const int bk = fp8 ? 128 : 64;
    if (K % bk != 0) return fail(WB_ERR_SHAPE, "GEMM K must be a multiple of the k-block");
    if (bn != 32 && bn != 64 && bn != 128 && bn != 256) return fail(WB_ERR_SHAPE, "GEMM BN must be 32/64/128/256");
    if (!aligned16(A.ptr) || !aligned16(B.ptr)) return fail(WB_ERR_ALIGN, "GEMM operand not 16-byte aligned");
    if ((A.row_stride * esz) % 16 || (B.row_stride * esz) % 16 || (A.batch_stride * esz) % 16)
        return fail(WB_ERR_ALIGN, "GEMM operand stride not a multiple of 16 bytes");
    {
        uint64_t dims[3] = {(uint64_t)K, (uint64_t)A.rows, (uint64_t)A.batches};
        uint64_t bstride = A.batches > 1 ? A.batch_stride : A.rows * A.row_stride;
        uint64_t strides[2] = {(uint64_t)(A.row_stride * esz), (uint64_t)(bstride * esz)};
        uint32_t box[3] = {(uint32_t)bk, (uint32_t)kBM, 1};
        if (wb_status st = encode_map(&plan->tma_a, A.ptr, 3, dims, strides, box, fp8)) return st;
    }
    if (b_kwrap && (b_kwrap % bk || K % b_kwrap)) return fail(WB_ERR_SHAPE, "GEMM k-wrap must divide K");
    {
        uint64_t dims[2] = {(uint64_t)(b_kwrap ? b_kwrap : K), (uint64_t)N};
        uint64_t strides[1] = {(uint64_t)(B.row_stride * esz)};
        // a CTA pair loads the B tile as two halves, one per CTA
        uint32_t box[2] = {(uint32_t)bk, (uint32_t)(pair ? bn / 2 : bn)};
        if (wb_status st = encode_map(&plan->tma_b, B.ptr, 2, dims, strides, box, fp8)) return st;
    }
    if (pair && (A.batches != 1 || bn != 256)) return fail(WB_ERR_INVALID_ARG, "paired GEMM: one batch, 256-wide tiles");
    plan->pair = pair;
    plan->M_rows = A.rows;
    plan->batches = A.batches;
    plan->N = N;
    plan->K = K;
    plan->bn = bn;
    plan->b_kwrap = b_kwrap;
    plan->fp8 = fp8;
    plan->ok = true;
    return WB_OK;
}

wb_status gemm_plan_swap(GemmPlan* plan, const GemmOperand& X, const GemmOperand& W, int64_t N, int64_t K, bool fp8,
                         int bn, int64_t w_kwrap) {
    if (wb_status st = get_encoder()) return st;
    const int esz = fp8 ? 1 : 2;
    const int bk = fp8 ? 128 : 64;
    if (K % bk != 0) return fail(WB_ERR_SHAPE, "GEMM K must be a multiple of the k-block");
    if (bn != 32 && bn != 64 && bn != 128) return fail(WB_ERR_SHAPE, "swapped GEMM: activation tile 32/64/128");
    if (X.batches != 1) return fail(WB_ERR_SHAPE, "swapped GEMM: no batched activations");
    if (!aligned16(X.ptr) || !aligned16(W.ptr)) return fail(WB_ERR_ALIGN, "GEMM operand not 16-byte aligned");
    if ((X.row_stride * esz) % 16 || (W.row_stride * esz) % 16) return fail(WB_ERR_ALIGN, "GEMM stride % 16 bytes");
    if (w_kwrap && (w_kwrap % bk || K % w_kwrap)) return fail(WB_ERR_SHAPE, "GEMM k-wrap must divide K");
    const int64_t kw = w_kwrap ? w_kwrap : K;
    {   // A = weights [N, kw], 128-row boxes
        uint64_t dims[3] = {(uint64_t)kw, (uint64_t)N, 1};
        uint64_t strides[2] = {(uint64_t)(W.row_stride * esz), (uint64_t)(N * W.row_stride * esz)};
        uint32_t box[3] = {(uint32_t)bk, (uint32_t)kBM, 1};
        if (wb_status st = encode_map(&plan->tma_a, W.ptr, 3, dims, strides, box, fp8)) return st;
    }
    {   // B = activations [M, K], bn-row boxes
        uint64_t dims[2] = {(uint64_t)K, (uint64_t)X.rows};
        uint64_t strides[1] = {(uint64_t)(X.row_stride * esz)};
        uint32_t box[2] = {(uint32_t)bk, (uint32_t)bn};
        if (wb_status st = encode_map(&plan->tma_b, X.ptr, 2, dims, strides, box, fp8)) return st;
    }
    plan->M_rows = X.rows;
    plan->batches = 1;
    plan->N = N;
    plan->K = K;
    plan->bn = bn;
    plan->b_kwrap = w_kwrap;
    plan->fp8 = fp8;
    plan->swap = true;
    plan->ok = true;
    return WB_OK;
}

wb_status gemm_run(const GemmPlan& p, const GemmEpi& epi, unsigned* err, cudaStream_t s, int max_ctas, int ksplit,
                   int64_t rows_override) {
    if (!p.ok) return fail(WB_ERR_INVALID_ARG, "GEMM plan not built");
    GemmArgs a;
    a.rows = rows_override > 0 ? std::min<int64_t>(rows_override, p.M_rows) : p.M_rows;
    a.batches = p.batches;
    a.N = p.N;
    a.K = p.K;
    if (p.swap) {
        if (epi.out_type != OUT_F32 && epi.out_type != OUT_F32_ACC) return fail(WB_ERR_INVALID_ARG, "swapped GEMM: fp32 output only");
        if (epi.gelu || epi.add || epi.mode != MODE_PLAIN) return fail(WB_ERR_INVALID_ARG, "swapped GEMM: linear epilogue only");
        a.mt_per_batch = (p.N + kBM - 1) / kBM;        // weight-row tiles
        a.mt_total = a.mt_per_batch;
        a.nt_total = (a.rows + p.bn - 1) / p.bn;        // activation-row tiles
    } else if (p.pair) {
        a.mt_per_batch = ((a.rows + kBM - 1) / kBM + 1) / 2;   // 256-row tiles
        a.mt_total = a.mt_per_batch;
        a.nt_total = (p.N + p.bn - 1) / p.bn;
    } else {
        a.mt_per_batch = (a.rows + kBM - 1) / kBM;
        a.mt_total = a.mt_per_batch * p.batches;
        a.nt_total = (p.N + p.bn - 1) / p.bn;
    }
    const int kb_all = (int)(p.K / (p.fp8 ? 128 : 64));
    if (ksplit < 1) ksplit = 1;
    if (ksplit > 1) {
        if (epi.out_type != OUT_F32 && epi.out_type != OUT_F32_ACC) return fail(WB_ERR_INVALID_ARG, "split-K needs fp32 output");
        if (epi.gelu || epi.add || epi.mode != MODE_PLAIN) return fail(WB_ERR_INVALID_ARG, "split-K: linear epilogue only");
        if (ksplit > kb_all) ksplit = kb_all;
    }
    a.ksplit = ksplit;
    a.tiles = a.mt_total * a.nt_total * ksplit;
    a.kb_all = kb_all;
    a.kblocks = (kb_all + ksplit - 1) / ksplit;
    a.b_kwrap = (int)p.b_kwrap;
    a.w_const = p.w_const ? 1 : 0;
    a.stall_ns = g_stall_next.exchange(0);
    a.epi = epi;
    const bool half = epi.out_type == OUT_BF16 || epi.out_type == OUT_BF16X2;
    a.epi.vec = aligned16(epi.out) && (epi.mode == MODE_CROSS_KV || (epi.ldo * (half ? 2 : 4)) % 16 == 0) &&
                (epi.out_type != OUT_BF16X2 || (p.N * 2) % 16 == 0);
    if (epi.mode == MODE_CROSS_KV && !a.epi.vec) return fail(WB_ERR_ALIGN, "cross K/V output not 16-byte aligned");
    if (epi.amax && (p.swap || epi.out_type != OUT_F32 || ksplit != 1 || epi.mode != MODE_PLAIN || epi.amax_rows < 32))
        return fail(WB_ERR_INVALID_ARG, "GEMM group amax: fp32 output, no split-K, groups of >= 32 rows");
    if (a.tiles == 0 || a.kblocks == 0) return WB_OK;
    const bool small = a.rows * p.batches < 1024;
    const int slot = prof_begin(small ? WB_KERNEL_GEMM_SMALL : WB_KERNEL_GEMM, s);
    wb_status st;
    if (p.swap) {
        if (p.fp8) {
            if (p.bn == 128) st = launch_tc<128, true, true>(p, a, err, s, max_ctas);
            else if (p.bn == 64) st = launch_tc<64, true, true>(p, a, err, s, max_ctas);
            else st = launch_tc<32, true, true>(p, a, err, s, max_ctas);
        } else {
            if (p.bn == 128) st = launch_tc<128, false, true>(p, a, err, s, max_ctas);
            else if (p.bn == 64) st = launch_tc<64, false, true>(p, a, err, s, max_ctas);
            else st = launch_tc<32, false, true>(p, a, err, s, max_ctas);
        }
    } else if (p.pair) {
        if (a.ksplit != 1) return fail(WB_ERR_INVALID_ARG, "paired GEMM: no split-K");
        st = p.fp8 ? launch_tc_pair<256, true>(p, a, err, s) : launch_tc_pair<256, false>(p, a, err, s);
    } else if (p.fp8) {
        if (p.bn == 256) st = launch_tc<256, true, false>(p, a, err, s, max_ctas);
        else if (p.bn == 128) st = launch_tc<128, true, false>(p, a, err, s, max_ctas);
        else if (p.bn == 64) st = launch_tc<64, true, false>(p, a, err, s, max_ctas);
        else st = launch_tc<32, true, false>(p, a, err, s, max_ctas);
    } else {
        if (p.bn == 256) st = launch_tc<256, false, false>(p, a, err, s, max_ctas);
        else if (p.bn == 128) st = launch_tc<128, false, false>(p, a, err, s, max_ctas);
        else if (p.bn == 64) st = launch_tc<64, false, false>(p, a, err, s, max_ctas);
        else st = launch_tc<32, false, false>(p, a, err, s, max_ctas);
    }
    const double k_alg = (double)(p.b_kwrap ? p.b_kwrap : p.K);
    const double M = (double)(a.rows * p.batches), esz = p.fp8 ? 1.0 : 2.0;
    (void)M;
    const double osz = (epi.out_type == OUT_BF16) ? 2.0 : (epi.out_type == OUT_F32_ACC ? 8.0 : 4.0);
    if (small) prof_end(slot, s, (double)p.N * k_alg * esz + M * (double)p.K * esz + M * (double)p.N * osz);
    else prof_end(slot, s, 2.0 * M * (double)p.N * k_alg);
    return st;
}

// ------------------------------------------------------------------ SIMT GEMM
namespace {

template <bool ABF, bool BBF>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const void* __restrict__ Ap, GemmOperand A, const void* __restrict__ Bp, int64_t ldb,
                 GemmArgs args) {
    griddep_wait();
    griddep_launch();
    // 64 x 64 output tile, 16-deep k-steps, 4 x 4 per thread.
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int64_t mt = blockIdx.y, nt = blockIdx.x;
    const int64_t b = mt / args.mt_per_batch;
    const int64_t r0 = (mt % args.mt_per_batch) * 64;
    const int64_t n0 = nt * 64;
    float acc[4][4] = {};
    for (int64_t k0 = 0; k0 < args.K; k0 += 16) {
        for (int i = threadIdx.x; i < 16 * 64; i += 256) {
            const int kk = i % 16, rr = i / 16;
            const int64_t r = r0 + rr, k = k0 + kk;
            float va = 0.f;
            if (r < args.rows && k < args.K) {
                const int64_t idx = b * A.batch_stride + r * A.row_stride + k;
                va = ABF ? bf2f(reinterpret_cast<const __nv_bfloat16*>(Ap)[idx])
                         : reinterpret_cast<const float*>(Ap)[idx];
            }
            As[kk][rr] = va;
            const int64_t n = n0 + rr;
            float vb = 0.f;
            if (n < args.N && k < args.K) {
                const int64_t idx = n * ldb + k;
                vb = BBF ? bf2f(reinterpret_cast<const __nv_bfloat16*>(Bp)[idx])
                         : reinterpret_cast<const float*>(Bp)[idx];
            }
            Bs[kk][rr] = vb;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a4[4], b4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a4[i] = As[kk][ty * 4 + i]; b4[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a4[i], b4[j], acc[i][j]);
        }
        __syncthreads();
    }
    const GemmEpi& e = args.epi;
    for (int i = 0; i < 4; ++i) {
        const int64_t r = r0 + ty * 4 + i;
        if (r >= args.rows) continue;
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tx * 4 + j;
            if (n >= args.N) continue;
            float v = acc[i][j];
            if (e.row_scale) v *= e.row_scale[b * args.rows + r];
            if (e.col_scale) v *= e.col_scale[n];
            if (e.bias) v += e.bias[n];
            if (e.gelu) v = gelu_f(v);
            if (e.add) v += e.add[r * e.ld_add + n];
            if (e.mode == MODE_CROSS_KV) {
                const int64_t m = b * args.rows + r;
                const int64_t ch = m / kCtx, s = m % kCtx;
                const int64_t two_d = 2 * (int64_t)e.ckv_d;
                const int64_t l = n / two_d, rem = n % two_d;
                const int64_t kv = rem / e.ckv_d, h = (rem % e.ckv_d) / 64, c = n % 64;
                const int64_t off = ((((l * e.ckv_chunks + ch) * 2 + kv) * e.ckv_heads + h) * kCtx + s) * 64 + c;
                if (e.out_type == OUT_BF16) reinterpret_cast<__nv_bfloat16*>(e.out)[off] = f2bf(v);
                else reinterpret_cast<float*>(e.out)[off] = v;
                continue;
            }
            const int64_t obr = e.out_batch_rows ? e.out_batch_rows : args.rows;
            const int64_t orow = b * obr + e.out_row_offset + r;
            if (e.out_type == OUT_BF16) reinterpret_cast<__nv_bfloat16*>(e.out)[orow * e.ldo + n] = f2bf(v);
            else if (e.out_type == OUT_F32) reinterpret_cast<float*>(e.out)[orow * e.ldo + n] = v;
            else reinterpret_cast<float*>(e.out)[orow * e.ldo + n] += v;
        }
    }
}

}  // namespace

wb_status gemm_simt(const GemmOperand& A, bool a_bf16, const GemmOperand& B, bool b_bf16, int64_t N,
                    int64_t K, const GemmEpi& epi, cudaStream_t s) {
    GemmArgs a;
    a.rows = A.rows;
    a.batches = A.batches;
    a.N = N;
    a.K = K;
    a.mt_per_batch = (A.rows + 63) / 64;
    a.mt_total = a.mt_per_batch * A.batches;
    a.nt_total = (N + 63) / 64;
    a.tiles = a.mt_total * a.nt_total;
    a.kblocks = 0;
    a.kb_all = 0;
    a.b_kwrap = 0;
    a.epi = epi;
    if (epi.out_type == OUT_BF16X2) return fail(WB_ERR_UNSUPPORTED, "SIMT GEMM: no split output");
    if (a.tiles == 0) return WB_OK;
    if (a.mt_total > 65535) return fail(WB_ERR_SHAPE, "SIMT GEMM: too many row tiles");
    dim3 grid((unsigned)a.nt_total, (unsigned)a.mt_total);
    if (a_bf16 && b_bf16) WB_CUDA(launch_k(gemm_simt_kernel<true, true>, dim3(grid), dim3(256), 0, s, A.ptr, A, B.ptr, B.row_stride, a));
    else if (!a_bf16 && b_bf16) WB_CUDA(launch_k(gemm_simt_kernel<false, true>, dim3(grid), dim3(256), 0, s, A.ptr, A, B.ptr, B.row_stride, a));
    else if (a_bf16 && !b_bf16) WB_CUDA(launch_k(gemm_simt_kernel<true, false>, dim3(grid), dim3(256), 0, s, A.ptr, A, B.ptr, B.row_stride, a));
    else WB_CUDA(launch_k(gemm_simt_kernel<false, false>, dim3(grid), dim3(256), 0, s, A.ptr, A, B.ptr, B.row_stride, a));
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

}  // namespace wb

extern "C" wb_status wb_debug_stall_next_gemm(uint64_t limit_ns) {
    if (limit_ns == 0 || limit_ns > 1000000000ull)
        return wb::fail(WB_ERR_INVALID_ARG, "wb_debug_stall_next_gemm: limit must be in (0, 1e9] ns");
    wb::g_stall_next.store(limit_ns);
    return WB_OK;
}
