// Launchers of the memory-bound kernels (layers.cu).
#pragma once

#include <stdint.h>

#include "internal.h"

namespace wb {

// LN_BF16X2 writes hi = bf16(y) at column c and lo = bf16(y - hi) at d + c.
// LN_AMAX writes nothing but the amax of every group of rows (see
// layernorm_group_e4m3); LN_E4M3_GROUP quantises with that group's scale.
enum LnOut : int { LN_F32 = 0, LN_BF16 = 1, LN_E4M3 = 2, LN_BF16X2 = 3, LN_AMAX = 4, LN_E4M3_GROUP = 5 };

// With zero set, zero[0 .. zero_n) is cleared by the same launch (the next
// GEMM's split-K output).
wb_status layernorm(const float* x, int64_t ld_x, int64_t rows, int d, const float* g, const float* b, LnOut mode,
                    void* out, int64_t ld_o, float* row_scale, cudaStream_t s, float* zero = nullptr,
                    int64_t zero_n = 0);
// LayerNorm into E4M3 with one scale per group of group_rows consecutive rows
// (one chunk's GEMM input): a first pass takes each group's amax of the
// normalised values into amax_bits[group] (zero beforehand; non-negative
// floats as their bit patterns), a second recomputes the rows and writes
// codes of y * fp32(1 / s), s = amax / 448 (1 when amax is 0), and
// row_scale[row] = s.  Needs d % 128 == 0.
wb_status layernorm_group_e4m3(const float* x, int64_t ld_x, int64_t rows, int d, const float* g, const float* b,
                               int64_t group_rows, unsigned* amax_bits, uint8_t* out, int64_t ld_o, float* row_scale,
                               cudaStream_t s);
// amax of each group of group_elems consecutive fp32 values (group_elems % 4
// == 0, x 16-byte aligned) into amax_bits[group] (atomic max: zero before).
wb_status group_amax(const float* x, int64_t n_groups, int64_t group_elems, unsigned* amax_bits, cudaStream_t s);
// E4M3 codes of fp32 rows x [rows, K] (K % 4 == 0) with one scale per group of
// group_rows rows, s = amax_bits[group] / 448 (1 when 0); row_scale[row] = s
// when row_scale is non-null.
wb_status quant_groups(const float* x, int64_t rows, int64_t K, int64_t group_rows, const unsigned* amax_bits,
                       uint8_t* q, float* row_scale, cudaStream_t s);
// scale[g] = amax / 448 (1 when 0) in place over an array that holds amax bits.
wb_status scales_from_amax(float* amax_then_scale, int64_t n, cudaStream_t s);
// Positions come from pos_dev[c * pos_stride] when pos_dev is non-null (graph
// replay; pos_stride 0: one position for all, 1: one per chunk), else p0.
wb_status embed(const int32_t* tokens, int64_t rows, int P, int p0, int d, const void* E, const void* Pos, bool bf16,
                int vocab, float* x, unsigned* err, cudaStream_t s, const int* pos_dev = nullptr,
                const int32_t* len = nullptr, int pos_stride = 0);
wb_status kv_scales(const float* qkv, int64_t n_chunks, int P, int d, float* k_scale, float* v_scale, cudaStream_t s);
wb_status kv_append(const float* qkv, int64_t n_chunks, int P, int p0, int d, int H, int layer, bool fp8, void* cache,
                    const int64_t* off, const int32_t* len, const float* k_scale, const float* v_scale, unsigned* err,
                    cudaStream_t s, const int* pos_dev = nullptr);
// x = GELU(x) in place, or GELU(x) as a bf16 (hi | lo) pair into out_bf16x2 [rows, 2N].
wb_status gelu_post(float* x, int64_t rows, int N, void* out_bf16x2, cudaStream_t s);
// pos_dev[0 .. n) = value, or += value when add.
wb_status set_pos(int* pos_dev, int value, bool add, cudaStream_t s, int n = 1);
// E4M3 codes of an fp32 matrix with one scale amax / 448 per row.
wb_status quant_rows_f32(const float* x, int64_t rows, int K, uint8_t* q, float* row_scale, cudaStream_t s,
                         bool gelu = false);
wb_status quant_tensor(const void* x, bool bf16, int64_t n, uint8_t* q, float* scale, unsigned* scratch_bits,
                       cudaStream_t s);
wb_status dequant_tensor(const uint8_t* q, const float* scale, int64_t n, float* out, cudaStream_t s);
wb_status fill(float* x, int64_t n, float v, cudaStream_t s);
// E4M3 cross K/V of chunks g0 .. g0+gB-1 from their fp32 projection tmp
// [layers][gB][K|V][n] into out [layers][B][K|V][n], scale [layers][K|V][B].
wb_status cross_kv_quant(const void* tmp, int64_t gB, int64_t B, int64_t g0, int layers, int64_t n, uint8_t* out,
                         float* scale, cudaStream_t s);
// Beam search (at most kBeamMax hypotheses per chunk; rows r0 = c K .. c K +
// K - 1 are chunk c's): one selection step over the logits of the first
// n_chunks chunks' rows at position pos (= *pos_dev when set), updating
// scores, token rows and cache histories [rows][448]; the best hypothesis
// per chunk; the initial histories and scores.
constexpr int kBeamMax = 8;
wb_status beam_select(const float* logits, int64_t ld, int64_t n_chunks, int K, int V, float* scores, int32_t* tokens,
                      int32_t* hist, const int32_t* len, const int* pos_dev, int pos_host, int32_t* parents_out,
                      float* scores_out, cudaStream_t s);
wb_status beam_best(const float* scores, const int32_t* tokens, int64_t n_chunks, int K, const int32_t* len,
                    int32_t* out, float* score_out, cudaStream_t s);
wb_status beam_init(int32_t* hist, float* scores, int64_t rows, int K, cudaStream_t s);
// Continuous batching: move the decode state of n chunks prepared in a
// staging decoder of R rows into their slots of an S-row decoder (cross K/V
// blocks of blk_bytes per layer and chunk, with their [layer][K|V][rows]
// scales when cs_src is given; the first P cache rows of each (layer, K|V,
// head) block of lay rows, cache scales, token rows, position P, decode
// length), and copy finished slots' token rows to the output.
wb_status slot_cross_copy(const void* src, void* dst, const int32_t* slot_of, int n, int64_t R, int64_t S, int layers,
                          int64_t blk_bytes, cudaStream_t s, const float* cs_src = nullptr, float* cs_dst = nullptr);
wb_status slot_state(const uint8_t* st_cache, uint8_t* sl_cache, const float* st_ks, const float* st_vs, float* sl_ks,
                     float* sl_vs, const int32_t* st_tok, int32_t* sl_tok, int* pos, int32_t* len, const int32_t* slot_of,
                     const int32_t* new_len, int n, int R, int S, int layers, int heads, int lay, int P, cudaStream_t s);
wb_status slot_out(const int32_t* sl_tok, const int32_t* slot, const int32_t* chunk, const int32_t* n_len, int n,
                   int32_t* out, cudaStream_t s);
wb_status argmax_tokens(const float* logits, int64_t ld, int64_t rows, int V, int32_t* tokens, const int32_t* len,
                        const int* pos_dev, int pos_host, cudaStream_t s, int pos_stride = 0);
// conv weight [O][C][3] -> [O][3][C]; dup: [O][3][2][C] (each tap twice, for
// stem inputs that carry a bf16 pair per value)
wb_status conv_reorder(const void* w, int O, int C, bool bf16, void* out, cudaStream_t s, bool dup = false);
wb_status gather_rows(const float* x, int64_t rows, int d, int64_t stride_rows, int64_t first, float* out,
                      cudaStream_t s);

}  // namespace wb
