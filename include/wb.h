/*
 * wb.h -- C ABI of the B300 (sm_103a) Whisper transcription hot path.
 *
 * Whisper turns 16 kHz mono audio into text in three stages: a log-Mel
 * spectrogram, a transformer encoder, and an autoregressive decoder with
 * self-attention over the tokens so far and cross-attention over the encoder
 * output ("Unlocking the power of OpenAI's Whisper", sections 1-3).  This
 * library runs those stages on one GPU for a batch of independent 30-second
 * chunks ("whisper-blaze 0.1.8", "Batch Transcription"), with bf16 arithmetic
 * and a float8 E4M3 self-attention KV cache ("Blazingly fast whisper
 * transcriptions with Inference Endpoints", "Inference Stack"), or FP8 GEMMs for
 * the QKV and FFN projections ("whisper-blaze 0.1.8", "Precision Presets",
 * mixed_fp8).
 *
 * Conventions shared by every entry point
 *   - Pointers marked [dev] are device pointers, [host] host pointers.  The
 *     caller owns every buffer it passes; the library never frees them and
 *     keeps no reference after the call returns, except where stated (a
 *     model keeps its weight pointer, a decoder its workspace pointer).
 *   - Device buffers must be 16-byte aligned (TMA requirement) and
 *     contiguous in the layout stated.  Violations return WB_ERR_ALIGN or
 *     WB_ERR_SHAPE before anything is launched.
 *   - Every call that takes a stream is asynchronous on that stream and does
 *     not synchronise, except where stated.  A null stream is the legacy
 *     default stream.
 *   - No call throws or aborts; failures return a negative wb_status and set a
 *     thread-local message readable with wb_last_error().
 *   - Device-side errors (a bounded wait on the GPU that ran out, a bounds
 *     check) are recorded in a device error word; wb_sync_status() waits for
 *     the stream and reports them.
 */
#ifndef WB_H
#define WB_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define WB_API __attribute__((visibility("default")))
#else
#define WB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int wb_status;
#define WB_OK               0
#define WB_ERR_INVALID_ARG -1   /* null pointer, bad enum, negative size        */
#define WB_ERR_SHAPE       -2   /* size outside what the entry point supports   */
#define WB_ERR_ALIGN       -3   /* device pointer not 16-byte aligned           */
#define WB_ERR_OOM         -4   /* the library could not allocate what it owns  */
#define WB_ERR_CUDA        -5   /* a CUDA runtime/driver call failed            */
#define WB_ERR_TIMEOUT     -6   /* a bounded device-side wait expired           */
#define WB_ERR_UNSUPPORTED -7   /* no GPU of compute capability 10.3            */

typedef struct CUstream_st* wb_stream;   /* == cudaStream_t */

/* Thread-local text of the last failure on this thread ("" if none). */
WB_API const char* wb_last_error(void);

/* Library version, 100 * major + minor. */
WB_API int wb_version(void);

/* ------------------------------------------------------------------ front end */

/*
 * Log-Mel spectrogram of a batch of 30 s chunks.
 * "whisper-blaze 0.1.8", "GPU Mel Spectrogram" / "Direct Kernel API"
 * (mel_spectrogram); "Unlocking the power of OpenAI's Whisper", section 2.
 *
 *   audio [dev] float32 [B, 480000]  16 kHz mono samples in [-1, 1]
 *   B           number of chunks, 1 <= B <= 2^20
 *   n_mels      80 or 128
 *   mel   [dev] float32 [B, n_mels, 3000] output
 *
 * Per chunk: reflect-pad 200 samples each side, frame t = padded samples
 * [160 t, 160 t + 400) times a periodic Hann window, |rFFT|^2 (201 bins),
 * Slaney-scale area-normalised triangular filters 0..8 kHz, log10 of the
 * energy clamped at 1e-10, floored at (the chunk's maximum - 8), mapped by
 * (x + 4) / 4.  Frames 0..2999 are returned.  The first call on a device
 * uploads constant tables synchronously; make it before any stream capture.
 */
WB_API wb_status wb_mel(const float* audio, int64_t B, int32_t n_mels, float* mel,
                 wb_stream stream);

/* ------------------------------------------------------------------ model */

#define WB_PREC_FP32      0   /* all arithmetic and storage in fp32           */
#define WB_PREC_BF16      1   /* bf16 weights/activations, fp32 accumulation  */
#define WB_PREC_MIXED_FP8 2   /* as BF16, QKV and FFN GEMMs in E4M3           */

typedef struct wb_model_desc {
    int32_t n_mels;       /* 80 or 128                                      */
    int32_t d_model;      /* multiple of 64, <= 1280; heads of width 64     */
    int32_t n_heads;      /* d_model / 64                                   */
    int32_t d_ffn;        /* multiple of 64                                 */
    int32_t enc_layers;   /* >= 0                                           */
    int32_t dec_layers;   /* >= 0                                           */
    int32_t vocab;        /* >= 1                                           */
    int32_t precision;    /* WB_PREC_*                                      */
    int32_t kv_fp8;       /* WB_KV_*: 0 none; 1 self-attention cache in E4M3;
                             2 also the cross-attention K/V (not with FP32)  */
} wb_model_desc;

/*
 * kv_fp8 values.  WB_KV_FP8_CROSS additionally stores each chunk's
 * precomputed cross-attention K and V in E4M3 with one scale per (chunk,
 * decoder layer, K or V): amax / 448 over that 1500 x d tensor (the float8
 * KV cache of "Blazingly fast whisper transcriptions with Inference
 * Endpoints", "Inference Stack", applied to the cross-attention as
 * "whisper-blaze 0.1.8", "Precision Presets" does for attention under
 * aggressive_fp8).  It halves the bytes the decode step streams per chunk.
 */
#define WB_KV_NONE 0
#define WB_KV_FP8_SELF 1
#define WB_KV_FP8_CROSS 2

typedef struct wb_model wb_model;

/*
 * Weight layout.  The model reads one flat device buffer of
 * wb_weights_bytes() bytes that the caller fills; each named tensor sits at
 * the byte offset wb_weight_offset() reports.  Matrices (projections, conv
 * kernels, embeddings) are stored in the model's weight type (fp32 for
 * WB_PREC_FP32, bf16 otherwise), row-major in the shapes below; vectors
 * (biases, LayerNorm gains and shifts) are always fp32.
 *
 *   enc.conv1.w [d, n_mels, 3]   enc.conv1.b [d]
 *   enc.conv2.w [d, d, 3]        enc.conv2.b [d]
 *   enc.<l>.{ln1,ln2}.{g,b} [d]
 *   enc.<l>.{q,k,v,o}.w [d, d]   enc.<l>.{q,k,v,o}.b [d]
 *   enc.<l>.fc1.w [d_ffn, d]     enc.<l>.fc1.b [d_ffn]
 *   enc.<l>.fc2.w [d, d_ffn]     enc.<l>.fc2.b [d]
 *   enc.lnp.{g,b} [d]
 *   dec.tok [vocab, d]  dec.pos [448, d]
 *   dec.<l>.{ln1,ln2,ln3}.{g,b} [d]
 *   dec.<l>.{sq,sk,sv,so,cq,ck,cv,co}.w [d, d]  (.b [d])
 *   dec.<l>.fc1.w [d_ffn, d] fc1.b [d_ffn]  dec.<l>.fc2.w [d, d_ffn] fc2.b [d]
 *   dec.lnf.{g,b} [d]
 *
 * A projection computes y = x W^T + b.  Returns 0 and sets *offset / *numel,
 * or WB_ERR_INVALID_ARG for an unknown name.
 */
WB_API size_t wb_weights_bytes(const wb_model_desc* desc);
WB_API wb_status wb_weight_offset(const wb_model_desc* desc, const char* name,
                           size_t* offset, int64_t* numel);

/*
 * Create a model over a filled weight buffer [dev] (kept by reference: it must
 * outlive the model).  The model allocates what it derives (conv kernels in
 * GEMM order, E4M3 weight copies and scales for WB_PREC_MIXED_FP8, position
 * tables, TMA descriptors) and frees it in wb_model_destroy.  Synchronises
 * the device once at the end.
 */
WB_API wb_status wb_model_create(const wb_model_desc* desc, const void* weights,
                          wb_model** out);
WB_API wb_status wb_model_destroy(wb_model* model);

/* Bytes of scratch wb_encode needs for B chunks. */
WB_API size_t wb_encode_workspace_size(const wb_model* model, int64_t B);

/*
 * Encoder forward: conv1(k3)+GELU, conv2(k3, stride 2)+GELU, + sinusoids, then
 * enc_layers pre-LN layers h += Wo MHA(LN1 h); h += W2 GELU(W1 LN2 h), and a
 * final LayerNorm ("Unlocking the power of OpenAI's Whisper", section 3;
 * "whisper-blaze 0.1.8", "Direct Kernel API", encoder_self_attn without mask,
 * layernorm_fused with eps 1e-5).
 *
 *   mel [dev] float32 [B, n_mels, 3000]  (wb_mel's output)
 *   enc [dev] [B, 1500, d] output, fp32 for WB_PREC_FP32, bf16 otherwise
 *   workspace [dev] >= wb_encode_workspace_size(model, B) bytes
 */
WB_API wb_status wb_encode(wb_model* model, const float* mel, int64_t B, void* enc,
                    void* workspace, size_t workspace_bytes, wb_stream stream);

/* ------------------------------------------------------------------ decoder */

typedef struct wb_decoder wb_decoder;

/*
 * Bytes of device memory a decoder over B chunks needs.  chunk_len [host]
 * int32 [B] gives each chunk's total decode length in positions (forced
 * prefix included), 1 <= chunk_len <= 448, and must be non-increasing: the
 * chunks still decoding at any step are then a prefix of the batch.  The
 * memory holds the cross-attention K/V of every layer (bf16), the ragged
 * self-attention cache (E4M3 or the activation type) sized by each chunk's
 * own length, and per-step scratch.
 */
WB_API size_t wb_decoder_workspace_size(const wb_model* model, int64_t B,
                                 const int32_t* chunk_len);

/*
 * Set up a decoder over B chunks: computes cross-attention K and V of every
 * decoder layer from enc ([dev] [B, 1500, d], wb_encode's output) into the
 * workspace ("whisper-blaze 0.1.8", "Direct Kernel API", decoder_cross_attn:
 * K/V come from the encoder and are computed once per chunk).  With
 * kv_fp8 = WB_KV_FP8_CROSS they are computed 16 chunks at a time into an
 * fp32 scratch area of the workspace and stored as E4M3 with one scale per
 * (chunk, layer, K|V), each value rounded once from fp32;
 * wb_decoder_workspace_size includes that scratch.
 *   tokens [dev] int32 [B, 448]  token matrix the decoder reads and writes
 *     (kept by reference).  Row c receives chunk c's tokens, position p in
 *     column p.
 * The handle lives in host memory allocated here; device memory is only the
 * caller's workspace.  wb_decoder_destroy frees the handle.
 */
WB_API wb_status wb_decoder_init(wb_model* model, int64_t B, const int32_t* chunk_len,
                          const void* enc, int32_t* tokens, void* workspace,
                          size_t workspace_bytes, wb_stream stream,
                          wb_decoder** out);

/*
 * Forced-prefix (or teacher-forced) pass: tokens[:, 0:P] must hold the prefix
 * ids.  Runs all P positions through every decoder layer with a causal mask
 * ("whisper-blaze 0.1.8", decoder_self_attn with causal mask), fixes the E4M3
 * cache scale of each (chunk, layer, K|V) from these rows as
 * 2 * max(amax, 1e-12) / 448, stores their K/V rows, and writes the greedy
 * token (lowest index of the maximal logit) of position P-1 into column P for
 * every chunk whose length exceeds P.  logits [dev] float32 [B, P, vocab] or
 * null.  1 <= P <= min(chunk_len).
 */
WB_API wb_status wb_decode_prefix(wb_decoder* dec, int32_t P, float* logits,
                           wb_stream stream);

/*
 * One greedy decode step at the decoder's current position t (t = P after the
 * prefix, +1 per step): chunks c < n_active must have chunk_len[c] > t + 1;
 * each reads token t, appends its self-attention K/V row t to the cache
 * (E4M3 with the chunk's frozen scale when kv_fp8), attends over rows 0..t
 * and over its 1500 cross-attention rows, and writes the greedy token into
 * column t + 1.  logits [dev] float32 [n_active, vocab] or null.
 * ("Thewhisper-large-v3-turbo" model card, "NVIDIA Usage": greedy, one beam,
 * KV cache; "Blazingly fast whisper transcriptions", "Inference Stack":
 * float8 KV cache.)
 */
WB_API wb_status wb_decode_step(wb_decoder* dec, int64_t n_active, float* logits,
                         wb_stream stream);

/*
 * Beam search ("thewhisper-large-v3-turbo" model card, "NVIDIA Usage":
 * generate_kwargs with num_beams; "Blazingly fast whisper transcriptions",
 * "Benchmarks": a fixed beam size).  A beam decoder over B chunks keeps
 * `beams` (2..8) hypotheses per chunk: token rows c*beams .. c*beams+beams-1
 * of `tokens` ([dev] int32 [B*beams, 448], every row holding the forced
 * prefix) belong to chunk c; the cross-attention K/V are computed once per
 * chunk and shared by its hypotheses.  wb_decode_prefix runs the prefix and
 * the first selection.  A hypothesis scores the sum of its generated tokens'
 * log-probabilities (log-softmax of its logits); every step ranks all
 * beams x vocab continuations of a chunk by that sum (ties: the lower beam,
 * then the lower token id) and keeps the best `beams`; their token rows and
 * cache histories are their parents' (a hypothesis reads the cached K/V rows
 * its ancestors wrote; no cache row is copied), with the chosen token in
 * column t + 1.  No length penalty, no end token: every chunk decodes to its
 * chunk_len.
 *   wb_decode_step_beams: one step for the first n_active chunks (launched
 *     directly, not through a captured graph); scores_out [dev] float32
 *     [B*beams] and parents_out [dev] int32 [B*beams] (beam index within its
 *     chunk) receive the new hypotheses' scores and parents, or are null.
 *   wb_decoder_best_beams: each chunk's best hypothesis (lowest beam among
 *     the maximal scores) into out_tokens [dev] int32 [B, 448] (columns 0 ..
 *     chunk_len - 1) and its score into out_scores [dev] float32 [B] or null.
 */
WB_API size_t wb_decoder_workspace_size_beams(const wb_model* model, int64_t B, const int32_t* chunk_len,
                                              int32_t beams);
WB_API wb_status wb_decoder_init_beams(wb_model* model, int64_t B, const int32_t* chunk_len, int32_t beams,
                                       const void* enc, int32_t* tokens, void* workspace, size_t workspace_bytes,
                                       wb_stream stream, wb_decoder** out);
WB_API wb_status wb_decode_step_beams(wb_decoder* dec, int64_t n_active, float* scores_out, int32_t* parents_out,
                                      wb_stream stream);
WB_API wb_status wb_decoder_best_beams(wb_decoder* dec, int32_t* out_tokens, float* out_scores, wb_stream stream);
/* The current running scores of every hypothesis into out [dev] float32 [B*beams]. */
WB_API wb_status wb_decoder_beam_scores(wb_decoder* dec, float* out, wb_stream stream);

/* Position the next wb_decode_step will process. */
WB_API int32_t wb_decoder_position(const wb_decoder* dec);
WB_API wb_status wb_decoder_destroy(wb_decoder* dec);

/* ------------------------------------------------------------------ batch */

/*
 * Transcribe a batch of requests end to end ("whisper-blaze 0.1.8",
 * "Batch Transcription" and "VRAM usage guide").  Each request is cut into
 * 30 s chunks (the last zero-padded); chunks are ordered by decode length,
 * longest first (ties by chunk index), and packed greedily into waves whose
 * decoder state stays within wave_budget_bytes; each wave runs mel, encoder,
 * cross-K/V, the forced prefix and greedy steps until every chunk reaches its
 * length.
 *
 *   audio       [dev] float32, requests back to back
 *   req_offset  [host] int64 [n_req] first sample of each request in audio
 *               (>= 0, else WB_ERR_SHAPE; offset + samples must lie inside
 *               audio, whose length the library does not see)
 *   req_samples [host] int64 [n_req] samples of each request (>= 1)
 *   prefix      [host] int32 [4] forced prefix token ids (< vocab)
 *   chunk_len   [host] int32 [n_chunks] decode length of each chunk in
 *               request order, 5 <= len <= 448 (prefix included)
 *   tokens      [dev] int32 [n_chunks, 448] output, request order; columns
 *               >= chunk_len are left untouched
 *   workspace   [dev] scratch of workspace_bytes; wb_transcribe_workspace_size
 *               tells how much a given batch needs
 *   n_waves_out [host] optional: number of waves used
 * With several waves, the next wave's mel and encoder run on a stream of the
 * library's own (lower priority, ordered after the caller's stream's earlier
 * work) while the current wave decodes; the encoder states are
 * double-buffered in the workspace.
 * Synchronises the stream before returning (it reads nothing back per step,
 * but checks the device error word at the end).
 */
WB_API size_t wb_transcribe_workspace_size(const wb_model* model, int32_t n_req,
                                    const int64_t* req_samples,
                                    const int32_t* chunk_len,
                                    uint64_t wave_budget_bytes);
WB_API wb_status wb_transcribe_batch(wb_model* model, const float* audio,
                              const int64_t* req_offset,
                              const int64_t* req_samples, int32_t n_req,
                              const int32_t* prefix, const int32_t* chunk_len,
                              int32_t* tokens, uint64_t wave_budget_bytes,
                              void* workspace, size_t workspace_bytes,
                              int32_t* n_waves_out, wb_stream stream);

/*
 * Overlapping windows ("whisper-blaze 0.1.8", "GPU Mel Spectrogram":
 * process_chunks(..., overlap_s); "thewhisper-large-v3-turbo": overlap_seconds
 * when long audio is split into windows).  With overlap_samples in
 * [0, 480000), chunk k of a request starts k * (480000 - overlap_samples)
 * samples in and holds the next 480000 samples (zero past the request's
 * end); a request of s samples has 1 + ceil(max(0, s - 480000) / stride)
 * chunks.  overlap_samples = 0 is the plain chunking of wb_transcribe_batch.
 *
 * wb_chunk_count: number of chunks of the batch (host only), -1 on bad input.
 * wb_transcribe_workspace_size_overlap / wb_transcribe_batch_overlap: as the
 *   calls without _overlap, on that chunking (chunk_len and the token rows
 *   follow the same chunk order).
 */
WB_API int64_t wb_chunk_count(int32_t n_req, const int64_t* req_samples, int64_t overlap_samples);
WB_API size_t wb_transcribe_workspace_size_overlap(const wb_model* model, int32_t n_req,
                                                   const int64_t* req_samples, const int32_t* chunk_len,
                                                   uint64_t wave_budget_bytes, int64_t overlap_samples);
WB_API wb_status wb_transcribe_batch_overlap(wb_model* model, const float* audio, const int64_t* req_offset,
                                             const int64_t* req_samples, int32_t n_req, int64_t overlap_samples,
                                             const int32_t* prefix, const int32_t* chunk_len, int32_t* tokens,
                                             uint64_t wave_budget_bytes, void* workspace, size_t workspace_bytes,
                                             int32_t* n_waves_out, wb_stream stream);

/*
 * One transcript per request from its chunks' token rows (host only).
 * Overlapping windows transcribe their shared audio twice, so each chunk's
 * generated tokens (columns prefix_len .. chunk_len - 1 of its row) are joined
 * to the request's text after dropping the longest prefix of them that
 * repeats the end of the text so far; with no such prefix they are appended
 * whole.  Token ids only: there are no timestamps to align on.
 *   tokens [host] int32 [n_chunks, 448] (wb_transcribe_batch_overlap's rows,
 *          copied to the host), chunk_len [host] int32 [n_chunks]
 *   out [host] int32 [out_cap]: request r's text is
 *          out[out_offset[r] .. out_offset[r + 1]); out_offset [host] int64
 *          [n_req + 1].  WB_ERR_SHAPE when out_cap is too small.
 */
WB_API wb_status wb_stitch_tokens(int32_t n_req, const int64_t* req_samples, int64_t overlap_samples,
                                  const int32_t* tokens, const int32_t* chunk_len, int32_t prefix_len,
                                  int32_t* out, int64_t out_cap, int64_t* out_offset);

/*
 * Continuous batching ("whisper-blaze 0.1.8", "Serving at Scale": requests of
 * mixed lengths batched together).  The same transcription as
 * wb_transcribe_batch, but instead of fixed waves the decoder keeps S slots
 * busy: S = min(n_chunks, wave_budget_bytes / per-slot bytes), a slot holding
 * one chunk's cross-attention K/V, a 448-row E4M3 cache and a token row.
 * Every chunk first goes through the mel and the encoder; then chunks,
 * longest first, enter free slots in groups of up to R = clamp(S / 8, 1, 32)
 * (their cross K/V and forced prefix are computed in a staging decoder and
 * moved into the slots), and each step -- one CUDA graph over all S slots --
 * advances every slot at its own position; a slot whose chunk has reached its
 * length is masked until it is refilled.  A chunk's tokens do not depend on
 * the slot it ran in or on the other chunks.  Needs a bf16 or mixed_fp8
 * model with kv_fp8 != 0.  n_slots_out [host] optional: S.
 */
WB_API size_t wb_transcribe_workspace_size_continuous(const wb_model* model, int32_t n_req,
                                                      const int64_t* req_samples, uint64_t wave_budget_bytes);
WB_API wb_status wb_transcribe_batch_continuous(wb_model* model, const float* audio, const int64_t* req_offset,
                                                const int64_t* req_samples, int32_t n_req, const int32_t* prefix,
                                                const int32_t* chunk_len, int32_t* tokens,
                                                uint64_t wave_budget_bytes, void* workspace,
                                                size_t workspace_bytes, int32_t* n_slots_out, wb_stream stream);

/* Wave plan alone (host only): wave_of_chunk[host] int32 [n_chunks],
 * order[host] int32 [n_chunks] chunk indices in decode order. */
WB_API wb_status wb_plan_waves(const wb_model_desc* desc, int32_t n_chunks,
                        const int32_t* chunk_len, uint64_t wave_budget_bytes,
                        int32_t* wave_of_chunk, int32_t* order,
                        int32_t* n_waves_out);

/*
 * One batch over several GPUs (host only; one process per GPU, each calling
 * wb_transcribe_batch on its share).  Chunks are independent from the mel to
 * the last decode step ("whisper-blaze 0.1.8", "Batch Transcription": every
 * 30 s chunk of every request is its own unit of the batch), so the split
 * needs no data from other GPUs.  The chunks, in request order, are cut into
 * `world` contiguous ranges balanced on their work: chunk c weighs
 * chunk_len[c] + 48 (its decode positions, plus the mel and encoder, which
 * cost about as much as 48 positions of the large-v3 decoder); range r begins
 * at the first chunk whose preceding work w satisfies w * world >= r * total.
 * For rank `rank` this returns its range as a request list -- every request
 * that overlaps the range, cut at chunk boundaries, with offsets into the
 * same audio buffer -- so that
 *   wb_transcribe_batch(model, audio, out_req_offset, out_req_samples,
 *                       *out_n_req, prefix, chunk_len + *out_chunk_first, ...)
 * transcribes exactly chunks [*out_chunk_first, *out_chunk_first +
 * *out_chunk_count) and writes their token rows in the same order.  A rank
 * may get no chunk (*out_chunk_count == 0, *out_n_req == 0).
 *   req_offset, req_samples [host] int64 [n_req]; chunk_len [host] int32 [n_chunks]
 *   out_req_offset, out_req_samples [host] int64 [n_req] (the first *out_n_req used)
 */
WB_API wb_status wb_shard_batch(int32_t n_req, const int64_t* req_offset, const int64_t* req_samples,
                                const int32_t* chunk_len, int32_t world, int32_t rank,
                                int64_t* out_req_offset, int64_t* out_req_samples, int32_t* out_n_req,
                                int32_t* out_chunk_first, int32_t* out_chunk_count);

/* ------------------------------------------------------------------ FP8 */

/*
 * E4M3 quantisation with a per-tensor scale ("whisper-blaze 0.1.8",
 * "Direct Kernel API": quantise_e4m3 / dequantise_e4m3).
 *   x      [dev] bf16 [n] or float32 [n] (x_is_bf16 selects)
 *   codes  [dev] uint8 [n] output
 *   scale  [dev] float32 [1] output: amax / 448 (1 when amax is 0)
 * Each code is round-to-nearest-even with saturation to +-448 of the fp32
 * product x * fp32(1 / scale).  Scratch: none.
 */
WB_API wb_status wb_quantise_e4m3(const void* x, int32_t x_is_bf16, int64_t n,
                           uint8_t* codes, float* scale, wb_stream stream);
/*
 * Same result as wb_quantise_e4m3 (identical codes and scale) for callers that
 * cannot allocate device memory: applications whose allocator owns every byte
 * of device memory, code paths where an implicit synchronisation from
 * cudaMalloc/cudaFree is not acceptable, or hosts that forbid allocation after
 * start-up.  The pages have no counterpart to this entry point.
 * It allocates nothing: its reduction scratch (one partial maximum per block
 * of 16384 elements) is a fixed array of 4160 floats (16.6 KB) in the
 * library's device image, held by every GPU that loads the library until the
 * process exits.
 *   n <= 2^26 (67108864) elements; larger n returns WB_ERR_SHAPE; n == 0
 *   writes scale 1 (x and codes may then be null).
 * All calls share that array: calls whose kernels overlap on the GPU (e.g. on
 * two unordered streams) race; calls ordered on one stream are safe.  The
 * first call in a CUDA context looks the array's address up
 * (cudaGetSymbolAddress) and keeps it for that context; make that first call
 * before any stream capture.  After cudaDeviceReset (a new context on the
 * device) the next call looks it up again, so the same rule applies to it.
 */
WB_API wb_status wb_quantise_e4m3_static(const void* x, int32_t x_is_bf16, int64_t n,
                                         uint8_t* codes, float* scale, wb_stream stream);

/*
 * The same quantisation over n_groups tensors at once, one scale each: group
 * g is x[g * group_elems .. (g + 1) * group_elems).  This is how the
 * WB_PREC_MIXED_FP8 encoder rounds each chunk's E4M3 GEMM input (one
 * 1500 x K tensor per chunk, "whisper-blaze 0.1.8", "Direct Kernel API",
 * quantise_e4m3: one scale per tensor).
 *   x      [dev] float32 [n_groups * group_elems], 16-byte aligned
 *   codes  [dev] uint8 [n_groups * group_elems] output, 16-byte aligned
 *   scales [dev] float32 [n_groups] output: amax_g / 448 (1 when amax_g is 0)
 * 1 <= n_groups <= 65535; group_elems a positive multiple of 4.  Codes are as
 * in wb_quantise_e4m3 with the group's scale.  Scratch: none (scales doubles
 * as the amax accumulator).
 */
WB_API wb_status wb_quantise_e4m3_groups(const float* x, int64_t n_groups, int64_t group_elems,
                                         uint8_t* codes, float* scales, wb_stream stream);

/* out [dev] float32 [n] = value(codes) * scale[0]. */
WB_API wb_status wb_dequantise_e4m3(const uint8_t* codes, const float* scale,
                             int64_t n, float* out, wb_stream stream);

/* ------------------------------------------------------------------ GEMM */

/*
 * The dense contraction every projection of the path runs on ("whisper-blaze
 * 0.1.8" lists FP16 and FP8 tensor-core GEMMs; here tcgen05 with TMEM
 * accumulators):  C[M, N] = epi(A[M, K] . B[N, K]^T)
 *   ab_type 0: A, B bf16 [dev]; 1: A, B E4M3 [dev], then the accumulator is
 *              multiplied by row_scale[m] * col_scale[n] ([dev] fp32, required)
 *   bias [dev] fp32 [N] or null;  gelu != 0 applies exact GELU after the bias
 *   C [dev] fp32 (c_bf16 = 0) or bf16 (c_bf16 = 1), row-major [M, N]
 * K must be a multiple of 64 (bf16) or 128 (E4M3); N a multiple of 8.
 * Device-side failures go to the library error word (wb_sync_status(NULL)).
 */
WB_API wb_status wb_gemm(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                         int32_t ab_type, const float* row_scale, const float* col_scale,
                         const float* bias, int32_t gelu, void* C, int32_t c_bf16,
                         wb_stream stream);

/* ------------------------------------------------------------------ timing */

/*
 * Per-kernel timing for roofline reports (diagnostics; no counterpart on the
 * pages).  After wb_prof_start(kind, max_launches), the library brackets every
 * launch of that kernel kind with CUDA events recorded on the launch's own
 * stream (up to max_launches launches; later ones are not timed) and sums
 * each launch's algorithmic work: flops for WB_KERNEL_GEMM and
 * WB_KERNEL_ENC_ATTN (2 M N K; 4 S^2 64 per chunk-head), bytes read and
 * written once for the memory-bound kinds (mel: audio in + mel out; decoder
 * attention: the K/V rows attended).  wb_prof_stop waits for the events and
 * returns launches, their summed duration in ms, and the summed work; it ends
 * the timing.  kind 0 times every kind at once; wb_prof_result then returns
 * one kind's share of the last timing.  Not thread-safe against concurrent
 * wb_prof_start calls.
 */
#define WB_KERNEL_GEMM        1
#define WB_KERNEL_ENC_ATTN    2
#define WB_KERNEL_CROSS_ATTN  3
#define WB_KERNEL_SELF_ATTN   4
#define WB_KERNEL_MEL         5
#define WB_KERNEL_GEMM_SMALL  6   /* GEMMs with < 1024 rows: bytes of A, B, C */
#define WB_KERNEL_MAX         6
WB_API wb_status wb_prof_start(int32_t kind, int32_t max_launches);
WB_API wb_status wb_prof_stop(int64_t* launches, double* total_ms, double* units);
WB_API wb_status wb_prof_result(int32_t kind, int64_t* launches, double* total_ms, double* units);

/* Number of kernels this library has launched in this process so far. */
WB_API int64_t wb_launch_count(void);

/* ------------------------------------------------------------------ status */

/* Waits for the stream, then reports (and clears) the device error word of
 * the model (or of the library's mel kernels when model is null). */
WB_API wb_status wb_sync_status(wb_model* model, wb_stream stream);

/*
 * Failure-detection test hook (no counterpart on the pages).  The next
 * tensor-core GEMM the library launches in this process (any entry point)
 * first waits limit_ns on a device barrier that nothing arrives on, then takes
 * the path of a pipeline wait that ran out: it records a timeout in the error
 * word it was given, stops issuing copies and MMAs, waits for the copies it
 * already issued, releases its tensor memory and exits.  That call's output
 * is unspecified; wb_sync_status reports WB_ERR_TIMEOUT and clears the word,
 * and later calls run normally.  0 < limit_ns <= 1e9, else WB_ERR_INVALID_ARG.
 */
WB_API wb_status wb_debug_stall_next_gemm(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* WB_H */
