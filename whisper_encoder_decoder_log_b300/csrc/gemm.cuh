// GEMM interface shared by the encoder, decoder and conv stem.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "internal.h"

namespace wb {

enum GemmOut : int { OUT_BF16 = 0, OUT_F32 = 1, OUT_F32_ACC = 2, OUT_BF16X2 = 3 };
// OUT_BF16X2 writes v as a bf16 pair: hi = bf16(v) at column n and
// lo = bf16(v - hi) at column N + n of the same row (ldo >= 2N).
enum GemmMode : int { MODE_PLAIN = 0, MODE_CROSS_KV = 1 };

// C = epilogue(A[M, K] . B[N, K]^T)
//   v = acc * row_scale[m] * col_scale[n] + bias[n];  v = GELU(v) if gelu;
//   v += add[r, n] (r = row within its batch);  out = v (or out += v)
// Rows are grouped in batches of rows_per_batch (the conv stem reads an
// overlapping-window view of each chunk); output row of (batch b, row r) is
// b * out_batch_rows + out_row_offset + r.
struct GemmEpi {
    void* out = nullptr;
    int64_t ldo = 0;                 // elements
    int out_type = OUT_BF16;
    const float* bias = nullptr;     // [N]
    int gelu = 0;
    const float* add = nullptr;      // [rows_per_batch, N] fp32, ld = ld_add
    int64_t ld_add = 0;
    const float* row_scale = nullptr;
    const float* col_scale = nullptr;
    int mode = MODE_PLAIN;
    // MODE_CROSS_KV: column n -> (layer, K|V, head, c); row -> (chunk, s)
    int ckv_d = 0, ckv_heads = 0;
    int64_t ckv_chunks = 0;
    int64_t out_batch_rows = 0;      // 0: = rows_per_batch
    int out_row_offset = 0;
    // With amax set (fp32 output, no split-K, tcgen05 path): the largest |v|
    // of every group of amax_rows output rows (>= 32) is folded into
    // amax[group] by atomic max over the bit patterns (zero it beforehand).
    unsigned* amax = nullptr;
    int64_t amax_rows = 0;
    int vec = 1;                     // set by the launcher: 16-byte stores allowed
};

// Operand description.  A is either a plain [M, K] matrix (batches = 1,
// rows = M) or `batches` stacked views of `rows` rows each, where row r of
// batch b starts at ptr + b * batch_stride + r * row_stride (elements).
struct GemmOperand {
    const void* ptr = nullptr;
    int64_t rows = 0;
    int64_t batches = 1;
    int64_t row_stride = 0;          // elements
    int64_t batch_stride = 0;        // elements
};

struct GemmPlan {
    CUtensorMap tma_a;
    CUtensorMap tma_b;
    int64_t M_rows = 0, batches = 1;
    int64_t N = 0, K = 0;
    int64_t b_kwrap = 0;   // A has K columns, B has b_kwrap: B is read at k mod b_kwrap
    int bn = 256;
    bool fp8 = false;
    bool swap = false;     // small-M form: weights are the 128-row MMA operand
    bool w_const = false;  // the weight operand is not written by kernels this GEMM may overlap
    bool pair = false;     // CTA pairs: cta_group::2 MMAs over 256-row tiles, each CTA loads half of B
    bool ok = false;
};

// Build the TMA descriptors (host only, no launch).  Element type bf16, or
// E4M3 when fp8.  Returns WB_OK or an error code with the message set.
wb_status gemm_plan(GemmPlan* plan, const GemmOperand& A, const GemmOperand& B, int64_t N,
                    int64_t K, bool fp8, int bn, int64_t b_kwrap = 0, bool pair = false);
// Small-M form: C[M, N] = X[M, K] . W[N, K]^T computed as W . X^T, with the
// weights as the 128-row MMA operand and bn (32/64/128) activation rows as the
// MMA N dimension; fp32 output, linear epilogue; w_kwrap as b_kwrap above.
wb_status gemm_plan_swap(GemmPlan* plan, const GemmOperand& X, const GemmOperand& W, int64_t N, int64_t K,
                         bool fp8, int bn, int64_t w_kwrap = 0);
// ksplit > 1 partitions K across CTAs and adds partial tiles with fp32
// atomics (fp32 outputs only; the caller zeroes a non-residual output first).
// rows_override < M_rows restricts the launch to the first rows.
wb_status gemm_run(const GemmPlan& plan, const GemmEpi& epi, unsigned* err, cudaStream_t s,
                   int max_ctas = 0, int ksplit = 1, int64_t rows_override = 0);

// fp32 / bf16 CUDA-core GEMM with the same semantics (used by the fp32 model
// and for small problems).  a_bf16 / b_bf16 select the operand types.
wb_status gemm_simt(const GemmOperand& A, bool a_bf16, const GemmOperand& B, bool b_bf16,
                    int64_t N, int64_t K, const GemmEpi& epi, cudaStream_t s);

int num_sms();

// 2-D bf16 TMA descriptor with the 128-byte swizzle: `outer` rows of
// `inner` elements, rows `row_stride_bytes` apart, box box_inner x box_outer.
wb_status make_tma_2d_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t row_stride_bytes,
                           uint32_t box_inner, uint32_t box_outer);

}  // namespace wb
