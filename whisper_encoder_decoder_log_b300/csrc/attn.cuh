// Attention launch interface.
#pragma once

#include <stdint.h>

#include <cuda.h>

#include "internal.h"

namespace wb {

// DT_BF16X2 (outputs only): hi = bf16(o) at column c, lo = bf16(o - hi) at c + o_split.
enum DType : int { DT_F32 = 0, DT_BF16 = 1, DT_E4M3 = 2, DT_BF16X2 = 3 };

// Where the keys/values of (chunk c, head h, key j) live (element offsets):
//   hs(c)   = head_stride * (chunk_len ? chunk_len[c] : 1)
//   base(c) = chunk_off ? chunk_off[c] : c * chunk_stride
//   K[c,h,j] = ptr + base(c) + (k_blk * heads + h) * hs(c) + j * row_stride
//   V[c,h,j] = ptr + base(c) + (v_blk * heads + h) * hs(c) + j * row_stride
// E4M3 keys/values are multiplied by k_scale[c] / v_scale[c].
struct KVView {
    const void* ptr = nullptr;
    int64_t chunk_stride = 0;
    const int64_t* chunk_off = nullptr;
    int64_t head_stride = 0;
    const int32_t* chunk_len = nullptr;
    int heads = 0;
    int k_blk = 0, v_blk = 1;
    int64_t row_stride = 64;
    const float* k_scale = nullptr;
    const float* v_scale = nullptr;
    // Graph replay: when pos_dev is set, the first query row of each chunk
    // sits at position *pos_dev (overrides q_pos0), and a chunk c with
    // active_len[c] <= *pos_dev + 1 has finished and is skipped.
    const int* pos_dev = nullptr;
    const int32_t* active_len = nullptr;
    // Beam search: query row c reads the cross K/V (and their scales) of
    // chunk c / beam_div; and, when hist is set, cache row j of row c (j <
    // the current position) lives in the cache of row hist[c * 448 + j] (the
    // row whose hypothesis wrote it).
    int beam_div = 1;
    const int32_t* hist = nullptr;
    // with pos_dev: row c's position is pos_dev[c * pos_stride] (0: one for all)
    int pos_stride = 0;
};

// Encoder self-attention, bf16, on tcgen05 (TMEM accumulators, TMA-fed tiles):
// qkv [n_chunks*1500, 3d] -> out [n_chunks*1500, d]; tma_qkv is a 2-D map over
// the qkv buffer with 64 x 128 boxes.
wb_status attn_flash_tc_bf16(const CUtensorMap* tma_qkv, int64_t n_chunks, int d, int heads, void* out,
                             unsigned* err, cudaStream_t s);

// Row attention: query row r of chunk c is q[(c*rows_per_chunk + r) * q_ld + h*64 ..]
// (pre-scaling by 1/8 inside); it attends over keys 0..kv_len-1, or, when
// causal, over keys 0..q_pos0 + r.  Output row likewise with o_ld.
wb_status attn_rows(DType tq, DType tkv, DType to, const void* q, int64_t q_ld, int64_t n_chunks,
                    int rows_per_chunk, int heads, const KVView& kv, int kv_len, bool causal, int q_pos0,
                    void* out, int64_t o_ld, cudaStream_t s, int64_t o_split = 0);

// Decode step (one query row per chunk at position pos = *kv.pos_dev, else
// q_pos): quantises the token's K and V rows of qkv [n_chunks, 3d] (fp32) to
// E4M3 with the chunk's scales, writes them to cache row pos, and attends over
// cache rows 0..pos; output bf16 (plus the bf16 remainder at o_split when
// o_split > 0).  Needs a ragged cache view (chunk_off, chunk_len, scales).
wb_status attn_self_step_e4m3(const float* qkv, int64_t q_ld, int64_t n_chunks, int heads, const KVView& kv,
                              int q_pos, void* out, int64_t o_ld, cudaStream_t s, int64_t o_split);

}  // namespace wb
