// C ABI and host orchestration (include/wb.h).  The host issues kernels on
// the caller's stream and never reads device data inside a step: per-chunk
// decode lengths are host-known, and the chunks still decoding at a step are
// a prefix of the (length-sorted) batch.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "attn.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "internal.h"
#include "prof.cuh"
#include "layers.cuh"

namespace wb {

static thread_local std::string t_last_error;
static std::mutex g_err_mu;
static unsigned* g_lib_err[64] = {};

void set_error(const std::string& msg) { t_last_error = msg; }
wb_status fail(wb_status code, const std::string& msg) {
    t_last_error = msg;
    return code;
}
wb_status cuda_fail(cudaError_t e, const char* what) {
    t_last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return WB_ERR_CUDA;
}
unsigned* lib_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_lib_err[dev]) {
        if (cudaMalloc(&g_lib_err[dev], sizeof(unsigned)) != cudaSuccess) return nullptr;
        cudaMemset(g_lib_err[dev], 0, sizeof(unsigned));
    }
    return g_lib_err[dev];
}

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ weight layout
struct Entry {
    size_t offset;
    int64_t numel;
    bool matrix;
};
struct Layout {
    std::unordered_map<std::string, Entry> map;
    size_t total = 0;
};
struct LayoutBuilder {
    Layout* L;
    size_t wsz;
    size_t cur = 0;
    void group() { cur = align_up(cur, 256); }
    void add(const std::string& n, int64_t numel, bool matrix) {
        L->map[n] = Entry{cur, numel, matrix};
        cur += (size_t)numel * (matrix ? wsz : 4);
    }
};

bool valid_desc(const wb_model_desc* d, std::string* why) {
    if (!d) { *why = "null descriptor"; return false; }
    if (d->n_mels != 80 && d->n_mels != 128) { *why = "n_mels must be 80 or 128"; return false; }
    if (d->d_model <= 0 || d->d_model % 64 || d->d_model > 1280) { *why = "d_model must be a multiple of 64, <= 1280"; return false; }
    if (d->n_heads * 64 != d->d_model) { *why = "n_heads must be d_model / 64"; return false; }
    if (d->d_ffn <= 0 || d->d_ffn % 256) { *why = "d_ffn must be a positive multiple of 256"; return false; }
    if (d->enc_layers < 0 || d->dec_layers < 0 || d->enc_layers > 256 || d->dec_layers > 256) { *why = "bad layer count"; return false; }
    if (d->vocab <= 0) { *why = "vocab must be positive"; return false; }
    if (d->precision < WB_PREC_FP32 || d->precision > WB_PREC_MIXED_FP8) { *why = "bad precision"; return false; }
    if (d->kv_fp8 && d->precision == WB_PREC_FP32) { *why = "kv_fp8 needs a bf16 precision"; return false; }
    if (d->kv_fp8 < WB_KV_NONE || d->kv_fp8 > WB_KV_FP8_CROSS) { *why = "kv_fp8 must be 0, 1 or 2"; return false; }
    return true;
}

std::string nm(const char* pre, int l, const char* name) { return std::string(pre) + std::to_string(l) + "." + name; }

void build_layout(const wb_model_desc& d, Layout* L) {
    LayoutBuilder b{L, (size_t)(d.precision == WB_PREC_FP32 ? 4 : 2)};
    const int64_t D = d.d_model, F = d.d_ffn, C = d.n_mels;
    b.group(); b.add("enc.conv1.w", D * C * 3, true);
    b.group(); b.add("enc.conv1.b", D, false);
    b.group(); b.add("enc.conv2.w", D * D * 3, true);
    b.group(); b.add("enc.conv2.b", D, false);
    for (int l = 0; l < d.enc_layers; ++l) {
        b.group(); b.add(nm("enc.", l, "ln1.g"), D, false); b.add(nm("enc.", l, "ln1.b"), D, false);
        b.group(); b.add(nm("enc.", l, "q.w"), D * D, true); b.add(nm("enc.", l, "k.w"), D * D, true); b.add(nm("enc.", l, "v.w"), D * D, true);
        b.group(); b.add(nm("enc.", l, "q.b"), D, false); b.add(nm("enc.", l, "k.b"), D, false); b.add(nm("enc.", l, "v.b"), D, false);
        b.group(); b.add(nm("enc.", l, "o.w"), D * D, true);
        b.group(); b.add(nm("enc.", l, "o.b"), D, false);
        b.group(); b.add(nm("enc.", l, "ln2.g"), D, false); b.add(nm("enc.", l, "ln2.b"), D, false);
        b.group(); b.add(nm("enc.", l, "fc1.w"), F * D, true);
        b.group(); b.add(nm("enc.", l, "fc1.b"), F, false);
        b.group(); b.add(nm("enc.", l, "fc2.w"), D * F, true);
        b.group(); b.add(nm("enc.", l, "fc2.b"), D, false);
    }
    b.group(); b.add("enc.lnp.g", D, false); b.add("enc.lnp.b", D, false);
    b.group(); b.add("dec.tok", (int64_t)d.vocab * D, true);
    b.group(); b.add("dec.pos", (int64_t)kMaxPos * D, true);
    for (int l = 0; l < d.dec_layers; ++l) {
        b.group(); b.add(nm("dec.", l, "ln1.g"), D, false); b.add(nm("dec.", l, "ln1.b"), D, false);
        b.group(); b.add(nm("dec.", l, "sq.w"), D * D, true); b.add(nm("dec.", l, "sk.w"), D * D, true); b.add(nm("dec.", l, "sv.w"), D * D, true);
        b.group(); b.add(nm("dec.", l, "sq.b"), D, false); b.add(nm("dec.", l, "sk.b"), D, false); b.add(nm("dec.", l, "sv.b"), D, false);
        b.group(); b.add(nm("dec.", l, "so.w"), D * D, true);
        b.group(); b.add(nm("dec.", l, "so.b"), D, false);
        b.group(); b.add(nm("dec.", l, "ln2.g"), D, false); b.add(nm("dec.", l, "ln2.b"), D, false);
        b.group(); b.add(nm("dec.", l, "cq.w"), D * D, true);
        b.group(); b.add(nm("dec.", l, "cq.b"), D, false);
        b.group(); b.add(nm("dec.", l, "co.w"), D * D, true);
        b.group(); b.add(nm("dec.", l, "co.b"), D, false);
        b.group(); b.add(nm("dec.", l, "ln3.g"), D, false); b.add(nm("dec.", l, "ln3.b"), D, false);
        b.group(); b.add(nm("dec.", l, "fc1.w"), F * D, true);
        b.group(); b.add(nm("dec.", l, "fc1.b"), F, false);
        b.group(); b.add(nm("dec.", l, "fc2.w"), D * F, true);
        b.group(); b.add(nm("dec.", l, "fc2.b"), D, false);
    }
    // cross-attention K and V of every decoder layer form one [L * 2d, d] operand
    b.group();
    for (int l = 0; l < d.dec_layers; ++l) { b.add(nm("dec.", l, "ck.w"), D * D, true); b.add(nm("dec.", l, "cv.w"), D * D, true); }
    b.group();
    for (int l = 0; l < d.dec_layers; ++l) { b.add(nm("dec.", l, "ck.b"), D, false); b.add(nm("dec.", l, "cv.b"), D, false); }
    b.group(); b.add("dec.lnf.g", D, false); b.add("dec.lnf.b", D, false);
    b.group();
    L->total = b.cur;
}

void sinusoids(int n_ctx, int d, std::vector<float>& out) {
    out.resize((size_t)n_ctx * d);
    const int half = d / 2;
    const double inc = std::log(10000.0) / (half - 1);
    for (int s = 0; s < n_ctx; ++s)
        for (int i = 0; i < half; ++i) {
            const double a = s * std::exp(-i * inc);
            out[(size_t)s * d + i] = (float)std::sin(a);
            out[(size_t)s * d + half + i] = (float)std::cos(a);
        }
}

__global__ void expand_scale_kernel(float* col_scale, int64_t rows_each) {
    griddep_wait();
    griddep_launch();
    const float s = col_scale[0];
    for (int64_t r = 1 + threadIdx.x; r < rows_each; r += blockDim.x) col_scale[r] = s;
}

// Bump allocator over a caller-provided workspace.
struct Carve {
    uint8_t* base;
    size_t cap;
    size_t cur = 0;
    bool overflow = false;
    template <typename T>
    T* take(size_t count) {
        cur = align_up(cur, 256);
        T* p = reinterpret_cast<T*>(base ? base + cur : nullptr);
        cur += count * sizeof(T);
        if (base && cur > cap) overflow = true;
        return p;
    }
};

}  // namespace
}  // namespace wb

using namespace wb;

struct FP8Weight {
    uint8_t* w = nullptr;
    float* col_scale = nullptr;
};

struct wb_model {
    wb_model_desc desc{};
    int device = 0;
    const uint8_t* w = nullptr;
    Layout layout;
    void* conv1_w = nullptr;
    void* conv2_w = nullptr;
    float* pe = nullptr;
    unsigned* err = nullptr;
    unsigned* scratch_bits = nullptr;
    std::vector<FP8Weight> enc_qkv, enc_fc1, enc_fc2, dec_qkv, dec_fc1, dec_fc2;
    std::vector<void*> allocs;

    const void* W(const std::string& n) const { return w + layout.map.at(n).offset; }
    const float* V(const std::string& n) const { return reinterpret_cast<const float*>(w + layout.map.at(n).offset); }
    bool fp32() const { return desc.precision == WB_PREC_FP32; }
    bool fp8() const { return desc.precision == WB_PREC_MIXED_FP8; }
    int d() const { return desc.d_model; }
    int H() const { return desc.n_heads; }
    int F() const { return desc.d_ffn; }
    size_t wsz() const { return fp32() ? 4 : 2; }
};

namespace wb {
namespace {

wb_status dev_alloc(wb_model* m, void** p, size_t bytes) {
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) return fail(WB_ERR_OOM, std::string("cudaMalloc: ") + cudaGetErrorString(e));
    m->allocs.push_back(*p);
    return WB_OK;
}

// E4M3 copy of a fused weight block: member i (rows_each x K) gets its own
// per-tensor scale amax / 448, expanded to that member's output columns.
wb_status make_fp8(wb_model* m, const std::vector<std::string>& names, int64_t rows_each, int64_t K, FP8Weight* out,
                   cudaStream_t s) {
    const int64_t n = (int64_t)names.size();
    if (wb_status st = dev_alloc(m, (void**)&out->w, (size_t)(n * rows_each * K))) return st;
    if (wb_status st = dev_alloc(m, (void**)&out->col_scale, (size_t)(n * rows_each) * 4)) return st;
    for (int64_t i = 0; i < n; ++i) {
        float* sc = out->col_scale + i * rows_each;
        if (wb_status st = quant_tensor(m->W(names[i]), true, rows_each * K, out->w + i * rows_each * K, sc,
                                        m->scratch_bits, s))
            return st;
        WB_CUDA(launch_k(expand_scale_kernel, dim3(1), dim3(256), 0, s, sc, rows_each));
    }
    WB_CUDA(cudaGetLastError());
    return WB_OK;
}

// ------------------------------------------------------------------ GEMM helper
// y = x W^T (+ epilogue) with the model's arithmetic: SIMT fp32 for the fp32
// model, tcgen05 otherwise (E4M3 when fp8 is given).
#ifndef WB_SWAP_ROWS
#define WB_SWAP_ROWS 1024
#endif
constexpr int64_t kSwapRows = WB_SWAP_ROWS;   // GEMMs with at most this many rows use the swapped form

struct Lin {
    const void* a = nullptr;      // activations
    int64_t rows = 0, lda = 0;
    int64_t batches = 1, batch_stride = 0;
    const void* w = nullptr;      // [N, K]
    int64_t N = 0, K = 0;
    const FP8Weight* f8 = nullptr;
    const float* a_scale = nullptr;
    bool split = false;           // a holds [hi | lo] bf16 halves: 2K columns, lda >= 2K
    bool out_zeroed = false;      // the caller has zeroed a plain fp32 output already
    bool w_const = false;         // w is model data, written by no kernel this GEMM can overlap
};

// How linear_impl runs a GEMM: SIMT, swapped (few rows) or plain tcgen05, the
// activation tile width and the K partitions.  Split-K adds fp32 partials
// atomically, so a plain fp32 output must be zero before the launch.
struct LinChoice {
    bool simt = false, swap = false;
    int bn = 0, ksplit = 1;
    bool pair = false;            // CTA pairs share B tiles (large plain GEMMs)
    bool needs_zero = false;
};

LinChoice linear_choose(const Lin& L, const GemmEpi& e, bool simt_fp32) {
    LinChoice c;
    const bool f8 = L.f8 != nullptr;
    if (simt_fp32 || L.K % (f8 ? 128 : 64) != 0) {
        c.simt = true;
        return c;
    }
    const int sms = num_sms();
    const bool linear_f32 = (e.out_type == OUT_F32 || e.out_type == OUT_F32_ACC) && !e.gelu && !e.add &&
                            e.mode == MODE_PLAIN;
    const int64_t kb_all = (L.split ? 2 * L.K : L.K) / (f8 ? 128 : 64);
    // a wide GEMM (the logits) over at least 256 rows has enough 256 x 256
    // CTA-pair tiles to fill the GPU; the pair form reads each operand tile
    // for twice the outputs of the swapped form
    const bool wide_pair = L.rows >= 256 && ((L.rows + 255) / 256) * ((L.N + 255) / 256) >= 2 * sms;
    if (linear_f32 && L.batches == 1 && L.rows <= kSwapRows && !wide_pair && !e.out_batch_rows &&
        !e.out_row_offset) {
        // few rows: weights as the 128-row MMA operand, rows as the MMA N
        c.swap = true;
        c.bn = L.rows <= 32 ? 32 : (L.rows <= 64 ? 64 : 128);
        const int64_t tiles = ((L.N + 127) / 128) * ((L.rows + c.bn - 1) / c.bn);
        // one CTA per SM, down to a single k-block per partition
        const int64_t want = sms / tiles;
        c.ksplit = (int)std::max<int64_t>(1, std::min<int64_t>(want, kb_all));
    } else {
        const int64_t tiles_m = ((L.rows + 127) / 128) * L.batches;
        auto tiles = [&](int bn) { return tiles_m * ((L.N + bn - 1) / bn); };
        c.bn = 256;
        if (tiles(256) < sms) c.bn = 128;
        if (tiles(128) < sms) c.bn = 64;
        // split-K applies to linear fp32 epilogues; otherwise narrow the tiles
        if (tiles(c.bn) < 2 * sms) {
            if (linear_f32) {
                c.ksplit = (int)std::min<int64_t>((2 * sms + tiles(c.bn) - 1) / tiles(c.bn),
                                                  std::max<int64_t>(1, kb_all / 4));
            } else if (tiles(32) <= 4 * sms) {
                c.bn = 32;
            }
        }
    }
    // enough M-tile pairs x N tiles for every SM pair: share B across a CTA pair
    if (!c.swap && c.ksplit == 1 && c.bn == 256 && L.batches == 1 &&
        ((L.rows + 255) / 256) * ((L.N + 255) / 256) >= sms)
        c.pair = true;
    c.needs_zero = c.ksplit > 1 && e.out_type == OUT_F32;
    return c;
}

// Elements of the output that linear_impl zeroes (or that a caller zeroes
// for it and flags with Lin::out_zeroed).
int64_t linear_out_elems(const Lin& L, const GemmEpi& e) {
    const int64_t obr = e.out_batch_rows ? e.out_batch_rows : L.rows;
    return L.batches * obr * e.ldo;
}

wb_status linear_impl(const Lin& L, GemmEpi e, bool simt_fp32, unsigned* err, cudaStream_t s) {
    GemmOperand A;
    A.ptr = L.a;
    A.rows = L.rows;
    A.batches = L.batches;
    A.row_stride = L.lda;
    A.batch_stride = L.batch_stride;
    GemmOperand B;
    B.ptr = L.f8 ? (const void*)L.f8->w : L.w;
    B.rows = L.N;
    B.row_stride = L.K;
    if (L.rows <= 0 || L.N <= 0) return WB_OK;
    const LinChoice c = linear_choose(L, e, simt_fp32);
    if (c.simt) {
        if (simt_fp32) return gemm_simt(A, false, B, false, L.N, L.K, e, s);
        if (L.f8) return fail(WB_ERR_UNSUPPORTED, "E4M3 GEMM needs K % 128 == 0");
        if (L.split) return fail(WB_ERR_UNSUPPORTED, "split GEMM needs K % 64 == 0");
        return gemm_simt(A, true, B, true, L.N, L.K, e, s);
    }
    const bool f8 = L.f8 != nullptr;
    if (f8) {
        e.row_scale = L.a_scale;
        e.col_scale = L.f8->col_scale;
    }
    if (c.needs_zero && !L.out_zeroed)
        if (wb_status st = fill(reinterpret_cast<float*>(e.out), linear_out_elems(L, e), 0.f, s)) return st;
    GemmPlan p;
    if (c.swap) {
        if (wb_status st = gemm_plan_swap(&p, A, B, L.N, L.split ? 2 * L.K : L.K, f8, c.bn, L.split ? L.K : 0))
            return st;
    } else {
        if (wb_status st = gemm_plan(&p, A, B, L.N, L.split ? 2 * L.K : L.K, f8, c.bn, L.split ? L.K : 0, c.pair))
            return st;
    }
    p.w_const = L.w_const;
    return gemm_run(p, e, err, s, 0, c.ksplit);
}

wb_status linear(const wb_model* m, const Lin& L0, GemmEpi e, cudaStream_t s) {
    Lin L = L0;
    L.w_const = true;   // every model GEMM multiplies by model weights
    return linear_impl(L, e, m->fp32(), m->err, s);
}

GemmEpi epi_out(void* out, int64_t ldo, int type, const float* bias, int gelu = 0) {
    GemmEpi e;
    e.out = out;
    e.ldo = ldo;
    e.out_type = type;
    e.bias = bias;
    e.gelu = gelu;
    return e;
}

// LayerNorm of the residual into the GEMM input, then the GEMM; when the GEMM
// splits K into an fp32 output, the LayerNorm launch zeroes that output too.
wb_status ln_then_linear(const wb_model* m, const float* h, int64_t R, const std::string& ln, LnOut mode, void* a,
                         int64_t lda, float* a_scale, Lin L, const GemmEpi& e, cudaStream_t s) {
    const int d = m->d();
    float* zero = nullptr;
    int64_t zn = 0;
    if (L.rows > 0 && L.N > 0) {
        const LinChoice c = linear_choose(L, e, m->fp32());
        if (c.needs_zero) {
            zero = reinterpret_cast<float*>(e.out);
            zn = linear_out_elems(L, e);
            L.out_zeroed = true;
        }
    }
    if (wb_status st = layernorm(h, d, R, d, m->V(ln + "g"), m->V(ln + "b"), mode, a, lda, a_scale, s, zero, zn))
        return st;
    return linear(m, L, e, s);
}

}  // namespace
}  // namespace wb

// ------------------------------------------------------------------ decoder state
struct StepGraph {
    int64_t rows = 0;
    cudaGraphExec_t exec = nullptr;
    int64_t kernels = 0;
};

struct wb_decoder {
    wb_model* m = nullptr;
    int64_t B = 0;
    std::vector<int32_t> len;
    int32_t* tokens = nullptr;
    int pos = 0;
    int P = 0;
    int max_len = 0;
    int* pos_dev = nullptr;            // position of the next step, on the device
    std::vector<StepGraph> graphs;     // one captured step per active-row bucket
    cudaStream_t cap_stream = nullptr; // graphs are captured here (capture runs nothing)
    // device buffers carved from the workspace
    void* crosskv = nullptr;
    void* ckv_tmp = nullptr;           // fp32 cross K/V of one chunk group before E4M3 rounding
    float* cscale = nullptr;           // E4M3 cross K/V scales [layer][K|V][chunk]
    void* cache = nullptr;
    float* kscale = nullptr;
    float* vscale = nullptr;
    int64_t* off = nullptr;
    int32_t* len_dev = nullptr;
    float* h = nullptr;
    void* a = nullptr;
    float* a_scale = nullptr;
    float* qkv = nullptr;
    void* attn = nullptr;
    float* cq = nullptr;
    void* f = nullptr;
    void* f2 = nullptr;
    uint8_t* fq = nullptr;
    float* f_scale = nullptr;
    float* logits = nullptr;
    // beam search: rows = chunks x beams (chunk c owns rows c*beams ..);
    // cross K/V are held once per chunk (n_cross chunks)
    int beams = 1;
    int64_t n_cross = 0;
    int32_t* hist = nullptr;           // [rows][448] row whose cache holds each position
    float* scores = nullptr;           // [rows] running log-probability sums
    int32_t* step_parents = nullptr;   // caller buffers of the current step (or null)
    float* step_scores = nullptr;
    // continuous batching: one position per row (pos_dev[row]) and cache
    // layout lengths (448 per slot) apart from the rows' decode lengths
    int pos_stride = 0;
    int32_t* lay_dev = nullptr;
    int32_t* lay_buf = nullptr;
};

namespace wb {
namespace {

constexpr int kMaxPrefix = 32;
constexpr int64_t kCrossGroup = 16;   // chunks per E4M3 cross K/V precompute group

struct DecLayout {
    size_t total = 0;
};

// Carve (or size, with base == nullptr) the decoder workspace.
// B rows (chunks x beams); the cross K/V are held once per chunk.
size_t carve_decoder(const wb_model* m, int64_t B, const int32_t* len, wb_decoder* dec, uint8_t* base, size_t cap,
                     bool* overflow, int beams = 1) {
    Carve c{base, cap};
    const int Ld = m->desc.dec_layers, d = m->d(), H = m->H(), F = m->F();
    const size_t act = m->fp32() ? 4 : 2;
    const int64_t R = B * kMaxPrefix;
    const int64_t NC = B / beams;
    const bool c8 = m->desc.kv_fp8 == WB_KV_FP8_CROSS;
    void* crosskv = c.take<uint8_t>((size_t)Ld * NC * 2 * kCtx * d * (c8 ? 1 : act));
    void* ckv_tmp = c8 ? c.take<float>((size_t)Ld * std::min<int64_t>(NC, kCrossGroup) * 2 * kCtx * d) : nullptr;
    float* cscale = c8 ? c.take<float>((size_t)std::max(1, Ld) * 2 * NC) : nullptr;
    int32_t* hist = beams > 1 ? c.take<int32_t>((size_t)B * kMaxPos) : nullptr;
    float* scores = beams > 1 ? c.take<float>(B) : nullptr;
    int64_t cache_elems = 0;
    for (int64_t i = 0; i < B; ++i) cache_elems += (int64_t)Ld * 2 * H * len[i] * 64;
    void* cache = c.take<uint8_t>((size_t)cache_elems * (m->desc.kv_fp8 ? 1 : 4));
    float* kscale = c.take<float>((size_t)std::max(1, Ld) * B);
    float* vscale = c.take<float>((size_t)std::max(1, Ld) * B);
    int64_t* off = c.take<int64_t>(B);
    int32_t* lend = c.take<int32_t>(B);
    float* h = c.take<float>((size_t)R * d);
    void* a = c.take<uint8_t>((size_t)R * d * 4);
    float* a_scale = c.take<float>(R);
    float* qkv = c.take<float>((size_t)R * 3 * d);
    void* attn = c.take<uint8_t>((size_t)R * d * 4);
    float* cq = c.take<float>((size_t)R * d);
    void* f = c.take<uint8_t>((size_t)R * F * 4);
    void* f2 = c.take<uint8_t>((size_t)R * F * 4);
    uint8_t* fq = c.take<uint8_t>((size_t)R * F);
    float* f_scale = c.take<float>(R);
    float* logits = c.take<float>((size_t)B * ((m->desc.vocab + 7) / 8 * 8));
    int* pos_dev = c.take<int>((size_t)std::max<int64_t>(64, B));   // one per row with per-row positions
    int32_t* lay = c.take<int32_t>(B);
    if (dec) {
        dec->beams = beams;
        dec->n_cross = NC;
        dec->hist = hist;
        dec->scores = scores;
        dec->pos_dev = pos_dev;
        dec->lay_dev = nullptr;     // set (to lay_buf) by decoders whose layout differs from their lengths
        dec->lay_buf = lay;
        dec->crosskv = crosskv; dec->ckv_tmp = ckv_tmp; dec->cscale = cscale;
        dec->cache = cache; dec->kscale = kscale; dec->vscale = vscale;
        dec->off = off; dec->len_dev = lend; dec->h = h; dec->a = a; dec->a_scale = a_scale; dec->qkv = qkv;
        dec->attn = attn; dec->cq = cq; dec->f = f; dec->f2 = f2; dec->fq = fq; dec->f_scale = f_scale; dec->logits = logits;
    }
    if (overflow) *overflow = c.overflow;
    return align_up(c.cur, 256);
}

struct EncBufs {
    void* melT;
    void* x1;
    float* h;
    void* a;
    float* a_scale;
    void* qkv;
    void* attn;
    void* f;
    uint8_t* fq;
    float* f_scale;
    unsigned* amax;     // mixed_fp8: [layer][LN1 | LN2 | GELU][chunk] E4M3 tensor amax
};

size_t carve_encoder(const wb_model* m, int64_t B, EncBufs* eb, uint8_t* base, size_t cap, bool* overflow) {
    Carve c{base, cap};
    const int d = m->d(), C = m->desc.n_mels, F = m->F();
    const size_t act = m->fp32() ? 4 : 2;
    const int64_t M = B * kCtx;
    EncBufs e;
    // bf16 models: stem rows hold (hi | lo) bf16 pairs, the size of fp32
    e.melT = c.take<uint8_t>((size_t)B * (kFrames + 2) * C * 4);
    e.x1 = c.take<uint8_t>((size_t)B * (kFrames + 2) * d * 4);
    e.h = c.take<float>((size_t)M * d);
    e.a = c.take<uint8_t>((size_t)M * d * act);
    e.a_scale = c.take<float>(M);
    e.qkv = c.take<uint8_t>((size_t)M * 3 * d * act);
    e.attn = c.take<uint8_t>((size_t)M * d * act);
    // mixed_fp8 keeps the GELU output in fp32: FC2's E4M3 input is rounded
    // once, from fp32, with the chunk's scale
    e.f = c.take<uint8_t>((size_t)M * F * (m->fp8() ? 4 : act));
    e.fq = m->fp8() ? c.take<uint8_t>((size_t)M * F) : nullptr;
    e.f_scale = c.take<float>(M);
    e.amax = m->fp8() ? c.take<unsigned>((size_t)std::max(1, m->desc.enc_layers) * 3 * B) : nullptr;
    if (eb) *eb = e;
    if (overflow) *overflow = c.overflow;
    return align_up(c.cur, 256);
}

// All decoder layers over R = n_chunks * rows_per_chunk rows (first position
// p0).  With bf16 weights every activation that feeds a GEMM is carried as a
// bf16 pair (hi, lo = bf16(x - hi)) and the GEMM runs over both halves against
// the same weights: the step is bound by weight bandwidth, so the second half
// costs no extra HBM traffic and the products keep ~16 mantissa bits of the
// fp32 activation.  FP8 GEMMs quantise from fp32.
wb_status decoder_layers(wb_decoder* dec, int64_t n_chunks, int rows_per_chunk, int p0, bool set_scales,
                         cudaStream_t s, const int* pos_dev) {
    wb_model* m = dec->m;
    const int d = m->d(), H = m->H(), F = m->F();
    const int64_t R = n_chunks * rows_per_chunk;
    const bool f32 = m->fp32(), f8 = m->fp8();
    // split bf16 activations for every bf16 GEMM input (mixed_fp8 included:
    // there the E4M3 codes of the next QKV/FFN inputs depend on these values,
    // and a bf16 rounding upstream would move some of them to the next code)
    const bool sp = !f32;
    const LnOut ln_act = f32 ? LN_F32 : (sp ? LN_BF16X2 : LN_BF16);
    const DType attn_dt = f32 ? DT_F32 : (sp ? DT_BF16X2 : DT_BF16);
    const int64_t lda = sp ? 2 * d : d;                // row stride of LN / attention outputs
    for (int l = 0; l < m->desc.dec_layers; ++l) {
        // ---- self-attention
        {
            Lin L;
            L.a = dec->a; L.rows = R; L.w = m->W(nm("dec.", l, "sq.w")); L.N = 3 * d; L.K = d;
            if (f8) { L.f8 = &m->dec_qkv[l]; L.a_scale = dec->a_scale; L.lda = d; }
            else { L.lda = lda; L.split = sp; }
            const GemmEpi e = epi_out(dec->qkv, 3 * d, OUT_F32, m->V(nm("dec.", l, "sq.b")));
            if (wb_status st = ln_then_linear(m, dec->h, R, nm("dec.", l, "ln1."), f8 ? LN_E4M3 : ln_act, dec->a,
                                              f8 ? d : lda, dec->a_scale, L, e, s))
                return st;
        }
        const bool kv8 = m->desc.kv_fp8 != 0;
        float* ks = dec->kscale + (int64_t)l * dec->B;
        float* vs = dec->vscale + (int64_t)l * dec->B;
        if (kv8 && set_scales)
            if (wb_status st = kv_scales(dec->qkv, n_chunks, rows_per_chunk, d, ks, vs, s)) return st;
        // a decode step over the E4M3 cache appends inside the attention kernel
        const bool fused_step = kv8 && rows_per_chunk == 1 && !f32;
        if (!fused_step)
            if (wb_status st = kv_append(dec->qkv, n_chunks, rows_per_chunk, p0, d, H, l, kv8, dec->cache, dec->off,
                                         dec->len_dev, ks, vs, m->err, s, pos_dev))
                return st;
        {
            KVView kv;
            kv.ptr = dec->cache; kv.chunk_off = dec->off; kv.head_stride = 64; kv.chunk_len = dec->len_dev;
            kv.heads = H; kv.k_blk = 2 * l; kv.v_blk = 2 * l + 1; kv.row_stride = 64;
            if (kv8) { kv.k_scale = ks; kv.v_scale = vs; }
            if (pos_dev) { kv.pos_dev = pos_dev; kv.active_len = dec->len_dev; kv.pos_stride = dec->pos_stride; }
            if (dec->lay_dev) kv.chunk_len = dec->lay_dev;
            if (dec->beams > 1 && rows_per_chunk == 1) kv.hist = dec->hist;
            if (fused_step) {
                if (wb_status st = attn_self_step_e4m3(dec->qkv, 3 * d, n_chunks, H, kv, p0, dec->attn, lda, s,
                                                       sp ? d : 0))
                    return st;
            } else {
            // with a device-side position the score buffer is sized for the longest chunk
            const int kv_len = pos_dev ? dec->max_len : p0 + rows_per_chunk;
            if (wb_status st = attn_rows(DT_F32, kv8 ? DT_E4M3 : DT_F32, attn_dt, dec->qkv, 3 * d, n_chunks,
                                         rows_per_chunk, H, kv, kv_len, true, p0, dec->attn, lda, s, sp ? d : 0))
                return st;
            }
        }
        {
            Lin L;
            L.a = dec->attn; L.rows = R; L.lda = lda; L.split = sp; L.w = m->W(nm("dec.", l, "so.w")); L.N = d; L.K = d;
            if (wb_status st = linear(m, L, epi_out(dec->h, d, OUT_F32_ACC, m->V(nm("dec.", l, "so.b"))), s)) return st;
        }
        // ---- cross-attention
        {
            Lin L;
            L.a = dec->a; L.rows = R; L.lda = lda; L.split = sp; L.w = m->W(nm("dec.", l, "cq.w")); L.N = d; L.K = d;
            const GemmEpi e = epi_out(dec->cq, d, OUT_F32, m->V(nm("dec.", l, "cq.b")));
            if (wb_status st = ln_then_linear(m, dec->h, R, nm("dec.", l, "ln2."), ln_act, dec->a, lda, nullptr, L, e, s))
                return st;
        }
        {
            const bool c8 = m->desc.kv_fp8 == WB_KV_FP8_CROSS;
            const size_t act = c8 ? 1 : (f32 ? 4 : 2);
            KVView kv;
            kv.ptr = reinterpret_cast<uint8_t*>(dec->crosskv) + (size_t)l * dec->n_cross * 2 * H * kCtx * 64 * act;
            kv.chunk_stride = (int64_t)2 * H * kCtx * 64; kv.head_stride = (int64_t)kCtx * 64; kv.heads = H;
            kv.k_blk = 0; kv.v_blk = 1; kv.row_stride = 64;
            kv.beam_div = dec->beams;
            kv.pos_stride = dec->pos_stride;
            if (c8) {
                kv.k_scale = dec->cscale + (size_t)(2 * l) * dec->n_cross;
                kv.v_scale = dec->cscale + (size_t)(2 * l + 1) * dec->n_cross;
            }
            if (pos_dev) { kv.pos_dev = pos_dev; kv.active_len = dec->len_dev; }
            if (wb_status st = attn_rows(DT_F32, c8 ? DT_E4M3 : (f32 ? DT_F32 : DT_BF16), attn_dt, dec->cq, d, n_chunks,
                                         rows_per_chunk, H, kv, kCtx, false, 0, dec->attn, lda, s, sp ? d : 0))
                return st;
        }
        {
            Lin L;
            L.a = dec->attn; L.rows = R; L.lda = lda; L.split = sp; L.w = m->W(nm("dec.", l, "co.w")); L.N = d; L.K = d;
            if (wb_status st = linear(m, L, epi_out(dec->h, d, OUT_F32_ACC, m->V(nm("dec.", l, "co.b"))), s)) return st;
        }
        // ---- FFN
        // FC1 (+GELU): with few rows the swapped GEMM writes fp32 and a
        // post-pass applies GELU (and the bf16 split); otherwise GELU is fused
        const bool few = R <= kSwapRows && !f32;
        Lin L1;
        L1.a = dec->a; L1.rows = R; L1.w = m->W(nm("dec.", l, "fc1.w")); L1.N = F; L1.K = d;
        if (f8) { L1.lda = d; L1.f8 = &m->dec_fc1[l]; L1.a_scale = dec->a_scale; }
        else { L1.lda = lda; L1.split = sp; }
        const int64_t ldf = sp ? 2 * F : F;
        void* fin = f32 ? dec->f : dec->f2;          // FC2 input (bf16 models)
        float* f32buf = reinterpret_cast<float*>(dec->f);
        const float* b1 = m->V(nm("dec.", l, "fc1.b"));
        const GemmEpi e1 = (few || f8) ? epi_out(f32buf, F, OUT_F32, b1, few ? 0 : 1)
                                       : epi_out(fin, ldf, f32 ? OUT_F32 : OUT_BF16X2, b1, 1);
        if (wb_status st = ln_then_linear(m, dec->h, R, nm("dec.", l, "ln3."), f8 ? LN_E4M3 : ln_act, dec->a,
                                          f8 ? d : lda, dec->a_scale, L1, e1, s))
            return st;
        // few rows, E4M3: GELU goes into the FC2 input quantiser
        if (few && !f8)
            if (wb_status st = gelu_post(f32buf, R, F, dec->f2, s)) return st;
        Lin L2;
        L2.rows = R; L2.w = m->W(nm("dec.", l, "fc2.w")); L2.N = d; L2.K = F;
        if (f8) {
            if (wb_status st = quant_rows_f32(f32buf, R, F, dec->fq, dec->f_scale, s, few)) return st;
            L2.a = dec->fq; L2.lda = F; L2.f8 = &m->dec_fc2[l]; L2.a_scale = dec->f_scale;
        } else {
            L2.a = fin; L2.lda = ldf; L2.split = sp;
        }
        if (wb_status st = linear(m, L2, epi_out(dec->h, d, OUT_F32_ACC, m->V(nm("dec.", l, "fc2.b"))), s)) return st;
    }
    return WB_OK;
}

// Final LayerNorm, logits = LN(h) E^T, greedy token into column pos+1.
wb_status decoder_head(wb_decoder* dec, int64_t n_chunks, int rows_per_chunk, int pos_last, float* logits_all,
                       cudaStream_t s, const int* pos_dev) {
    wb_model* m = dec->m;
    const int d = m->d(), V = m->desc.vocab;
    const bool sp = !m->fp32();
    const LnOut ln_act = m->fp32() ? LN_F32 : (sp ? LN_BF16X2 : LN_BF16);
    const int64_t lda = sp ? 2 * d : d;
    const int64_t R = n_chunks * rows_per_chunk;
    Lin L;
    L.w = m->W("dec.tok"); L.N = V; L.K = d; L.lda = lda; L.split = sp;
    if (logits_all) {
        if (wb_status st = layernorm(dec->h, d, R, d, m->V("dec.lnf.g"), m->V("dec.lnf.b"), ln_act, dec->a, lda,
                                     nullptr, s))
            return st;
        L.a = dec->a; L.rows = R;
        if (wb_status st = linear(m, L, epi_out(logits_all, V, OUT_F32, nullptr), s)) return st;
        if (dec->beams > 1)
            return beam_select(logits_all + (int64_t)(rows_per_chunk - 1) * V, (int64_t)rows_per_chunk * V,
                               n_chunks / dec->beams, dec->beams, V, dec->scores, dec->tokens, dec->hist, dec->len_dev,
                               pos_dev, pos_last, dec->step_parents, dec->step_scores, s);
        return argmax_tokens(logits_all + (int64_t)(rows_per_chunk - 1) * V, (int64_t)rows_per_chunk * V, n_chunks, V,
                             dec->tokens, dec->len_dev, pos_dev, pos_last, s);
    }
    // only the last row of each chunk matters
    if (wb_status st = layernorm(dec->h + (int64_t)(rows_per_chunk - 1) * d, (int64_t)rows_per_chunk * d, n_chunks, d,
                                 m->V("dec.lnf.g"), m->V("dec.lnf.b"), ln_act, dec->a, lda, nullptr, s))
        return st;
    L.a = dec->a; L.rows = n_chunks;
    const int64_t ldl = (V + 7) / 8 * 8;
    if (wb_status st = linear(m, L, epi_out(dec->logits, ldl, OUT_F32, nullptr), s)) return st;
    if (dec->beams > 1)
        return beam_select(dec->logits, ldl, n_chunks / dec->beams, dec->beams, V, dec->scores, dec->tokens, dec->hist,
                           dec->len_dev, pos_dev, pos_last, dec->step_parents, dec->step_scores, s);
    return argmax_tokens(dec->logits, ldl, n_chunks, V, dec->tokens, dec->len_dev, pos_dev, pos_last, s,
                         dec->pos_stride);
}

__global__ void gather_chunks_kernel(const float* __restrict__ audio, const int64_t* __restrict__ src,
                                     const int32_t* __restrict__ valid, float* __restrict__ out) {
    griddep_wait();
    griddep_launch();
    const int64_t c = blockIdx.y;
    const int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i0 >= kChunkSamples) return;
    const int v = valid[c];
    float4 o;
    float* op = reinterpret_cast<float*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) op[j] = (i0 + j < v) ? audio[src[c] + i0 + j] : 0.f;
    *reinterpret_cast<float4*>(out + c * kChunkSamples + i0) = o;
}

__global__ void fill_prefix_kernel(int32_t* tokens, int64_t n, int32_t p0, int32_t p1, int32_t p2, int32_t p3) {
    griddep_wait();
    griddep_launch();
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= n) return;
    tokens[c * kMaxPos + 0] = p0;
    tokens[c * kMaxPos + 1] = p1;
    tokens[c * kMaxPos + 2] = p2;
    tokens[c * kMaxPos + 3] = p3;
}

__global__ void scatter_tokens_kernel(const int32_t* __restrict__ wave_tok, const int32_t* __restrict__ dst_row,
                                      const int32_t* __restrict__ len, int32_t* __restrict__ out) {
    griddep_wait();
    griddep_launch();
    const int64_t c = blockIdx.x;
    const int64_t r = dst_row[c];
    for (int i = threadIdx.x; i < len[c]; i += blockDim.x) out[r * kMaxPos + i] = wave_tok[c * kMaxPos + i];
}

void plan_waves_host(const wb_model_desc& d, int32_t n, const int32_t* len, uint64_t budget,
                     std::vector<std::vector<int32_t>>& waves, bool* too_big) {
    std::vector<int32_t> order(n);
    for (int32_t i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return len[a] > len[b]; });
    const uint64_t cross_elt = d.kv_fp8 == WB_KV_FP8_CROSS ? 1 : 2;
    auto bytes = [&](int32_t L) {
        return (uint64_t)d.dec_layers * 2 * kCtx * d.d_model * cross_elt + (uint64_t)d.dec_layers * 2 * L * d.d_model +
               (uint64_t)kMaxPos * 4;
    };
    *too_big = false;
    waves.clear();
    std::vector<int32_t> cur;
    uint64_t used = 0;
    for (int32_t c : order) {
        const uint64_t b = bytes(len[c]);
        if (b > budget) { *too_big = true; return; }
        if (!cur.empty() && used + b > budget) { waves.push_back(cur); cur.clear(); used = 0; }
        cur.push_back(c);
        used += b;
    }
    if (!cur.empty()) waves.push_back(cur);
}

constexpr int64_t kEncSubBatch = 32;

}  // namespace
}  // namespace wb

extern "C" {

const char* wb_last_error(void) { return t_last_error.c_str(); }
int wb_version(void) { return 100; }

wb_status wb_mel(const float* audio, int64_t B, int32_t n_mels, float* mel, wb_stream stream) {
    if (!audio || !mel) return fail(WB_ERR_INVALID_ARG, "wb_mel: null pointer");
    if (B < 1 || B > (1 << 20)) return fail(WB_ERR_SHAPE, "wb_mel: B must be in [1, 2^20]");
    if (n_mels != 80 && n_mels != 128) return fail(WB_ERR_SHAPE, "wb_mel: n_mels must be 80 or 128");
    if (!aligned16(audio) || !aligned16(mel)) return fail(WB_ERR_ALIGN, "wb_mel: pointers must be 16-byte aligned");
    return mel_launch(audio, B, n_mels, mel, reinterpret_cast<cudaStream_t>(stream));
}

size_t wb_weights_bytes(const wb_model_desc* desc) {
    std::string why;
    if (!valid_desc(desc, &why)) return 0;
    Layout L;
    build_layout(*desc, &L);
    return L.total;
}

wb_status wb_weight_offset(const wb_model_desc* desc, const char* name, size_t* offset, int64_t* numel) {
    std::string why;
    if (!valid_desc(desc, &why)) return fail(WB_ERR_INVALID_ARG, "wb_weight_offset: " + why);
    if (!name || !offset || !numel) return fail(WB_ERR_INVALID_ARG, "wb_weight_offset: null argument");
    Layout L;
    build_layout(*desc, &L);
    auto it = L.map.find(name);
    if (it == L.map.end()) return fail(WB_ERR_INVALID_ARG, std::string("unknown weight ") + name);
    *offset = it->second.offset;
    *numel = it->second.numel;
    return WB_OK;
}

wb_status wb_model_create(const wb_model_desc* desc, const void* weights, wb_model** out) {
    std::string why;
    if (!out) return fail(WB_ERR_INVALID_ARG, "wb_model_create: null out");
    *out = nullptr;
    if (!valid_desc(desc, &why)) return fail(WB_ERR_INVALID_ARG, "wb_model_create: " + why);
    if (!weights) return fail(WB_ERR_INVALID_ARG, "wb_model_create: null weights");
    if (!aligned16(weights)) return fail(WB_ERR_ALIGN, "wb_model_create: weights not 16-byte aligned");
    int dev = 0;
    WB_CUDA(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    WB_CUDA(cudaGetDeviceProperties(&prop, dev));
    if (prop.major != 10 || prop.minor != 3)
        return fail(WB_ERR_UNSUPPORTED, "wb_model_create: needs a compute capability 10.3 GPU");
    wb_model* m = new wb_model();
    m->desc = *desc;
    m->device = dev;
    m->w = reinterpret_cast<const uint8_t*>(weights);
    build_layout(*desc, &m->layout);
    cudaStream_t s = nullptr;
    auto bail = [&](wb_status st) {
        for (void* p : m->allocs) cudaFree(p);
        delete m;
        return st;
    };
    const int d = m->d(), C = desc->n_mels, F = m->F();
    const bool bf = !m->fp32();
    if (wb_status st = dev_alloc(m, (void**)&m->err, 16)) return bail(st);
    m->scratch_bits = m->err + 1;
    if (cudaMemset(m->err, 0, 16) != cudaSuccess) return bail(fail(WB_ERR_CUDA, "memset"));
    // bf16 models feed the stem GEMMs bf16 pairs (hi | lo) of every value:
    // each conv tap is stored twice to multiply both halves
    const size_t taps = bf ? 6 : 3;
    if (wb_status st = dev_alloc(m, &m->conv1_w, (size_t)d * C * taps * m->wsz())) return bail(st);
    if (wb_status st = dev_alloc(m, &m->conv2_w, (size_t)d * d * taps * m->wsz())) return bail(st);
    if (wb_status st = conv_reorder(m->W("enc.conv1.w"), d, C, bf, m->conv1_w, s, bf)) return bail(st);
    if (wb_status st = conv_reorder(m->W("enc.conv2.w"), d, d, bf, m->conv2_w, s, bf)) return bail(st);
    {
        std::vector<float> pe;
        sinusoids(kCtx, d, pe);
        if (wb_status st = dev_alloc(m, (void**)&m->pe, pe.size() * 4)) return bail(st);
        if (cudaMemcpy(m->pe, pe.data(), pe.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
            return bail(fail(WB_ERR_CUDA, "upload positions"));
    }
    if (m->fp8()) {
        for (int l = 0; l < desc->enc_layers; ++l) {
            FP8Weight q, f1, f2;
            wb_status st = make_fp8(m, {nm("enc.", l, "q.w"), nm("enc.", l, "k.w"), nm("enc.", l, "v.w")}, d, d, &q, s);
            if (!st) st = make_fp8(m, {nm("enc.", l, "fc1.w")}, F, d, &f1, s);
            if (!st) st = make_fp8(m, {nm("enc.", l, "fc2.w")}, d, F, &f2, s);
            if (st) return bail(st);
            m->enc_qkv.push_back(q); m->enc_fc1.push_back(f1); m->enc_fc2.push_back(f2);
        }
        for (int l = 0; l < desc->dec_layers; ++l) {
            FP8Weight q, f1, f2;
            wb_status st = make_fp8(m, {nm("dec.", l, "sq.w"), nm("dec.", l, "sk.w"), nm("dec.", l, "sv.w")}, d, d, &q, s);
            if (!st) st = make_fp8(m, {nm("dec.", l, "fc1.w")}, F, d, &f1, s);
            if (!st) st = make_fp8(m, {nm("dec.", l, "fc2.w")}, d, F, &f2, s);
            if (st) return bail(st);
            m->dec_qkv.push_back(q); m->dec_fc1.push_back(f1); m->dec_fc2.push_back(f2);
        }
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return bail(fail(WB_ERR_CUDA, "model setup failed"));
    *out = m;
    return WB_OK;
}

wb_status wb_model_destroy(wb_model* m) {
    if (!m) return fail(WB_ERR_INVALID_ARG, "wb_model_destroy: null model");
    for (void* p : m->allocs) cudaFree(p);
    delete m;
    return WB_OK;
}

size_t wb_encode_workspace_size(const wb_model* m, int64_t B) {
    if (!m || B < 1) return 0;
    return carve_encoder(m, B, nullptr, nullptr, 0, nullptr);
}

wb_status wb_encode(wb_model* m, const float* mel, int64_t B, void* enc, void* workspace, size_t ws_bytes,
                    wb_stream stream) {
    if (!m || !mel || !enc || !workspace) return fail(WB_ERR_INVALID_ARG, "wb_encode: null argument");
    if (B < 1 || B > 65535) return fail(WB_ERR_SHAPE, "wb_encode: B must be in [1, 65535]");
    if (!aligned16(mel) || !aligned16(enc) || !aligned16(workspace)) return fail(WB_ERR_ALIGN, "wb_encode: alignment");
    EncBufs e;
    bool over = false;
    carve_encoder(m, B, &e, reinterpret_cast<uint8_t*>(workspace), ws_bytes, &over);
    if (over) return fail(WB_ERR_SHAPE, "wb_encode: workspace too small");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int d = m->d(), C = m->desc.n_mels, H = m->H(), F = m->F();
    const int64_t M = B * kCtx;
    const bool f32 = m->fp32(), f8 = m->fp8();
    const size_t act = f32 ? 4 : 2;
    const int act_out = f32 ? OUT_F32 : OUT_BF16;
    const LnOut ln_plain = f32 ? LN_F32 : LN_BF16;
    // ---- stem: mel -> [B, 3002, C] -> conv1 (+GELU) -> padded [B, 3002, d] -> conv2 (+GELU, +PE)
    // bf16 models carry every stem value as a bf16 pair (hi | lo) and multiply
    // both halves by the same (duplicated) conv taps: the stem output enters
    // the fp32 residual with ~16 bits instead of bf16's 8
    const int64_t pw = f32 ? 1 : 2;    // stored values per mel / conv1 value
    if (wb_status st = mel_transpose_pad(mel, B, C, e.melT, !f32, s)) return st;
    WB_CUDA(cudaMemset2DAsync(e.x1, (size_t)(kFrames + 2) * pw * d * act, 0, (size_t)pw * d * act, (size_t)B, s));
    WB_CUDA(cudaMemset2DAsync(reinterpret_cast<uint8_t*>(e.x1) + (size_t)(kFrames + 1) * pw * d * act,
                              (size_t)(kFrames + 2) * pw * d * act, 0, (size_t)pw * d * act, (size_t)B, s));
    {
        Lin L;
        L.a = e.melT; L.rows = kFrames; L.lda = pw * C; L.batches = B;
        L.batch_stride = (int64_t)(kFrames + 2) * pw * C;
        L.w = m->conv1_w; L.N = d; L.K = 3 * pw * C;
        GemmEpi ep = epi_out(e.x1, pw * d, f32 ? OUT_F32 : OUT_BF16X2, m->V("enc.conv1.b"), 1);
        ep.out_batch_rows = kFrames + 2;
        ep.out_row_offset = 1;
        if (wb_status st = linear(m, L, ep, s)) return st;
    }
    {
        Lin L;
        L.a = e.x1; L.rows = kCtx; L.lda = 2 * pw * d; L.batches = B;
        L.batch_stride = (int64_t)(kFrames + 2) * pw * d;
        L.w = m->conv2_w; L.N = d; L.K = 3 * pw * d;
        GemmEpi ep = epi_out(e.h, d, OUT_F32, m->V("enc.conv2.b"), 1);
        ep.add = m->pe;
        ep.ld_add = d;
        ep.out_batch_rows = kCtx;
        if (wb_status st = linear(m, L, ep, s)) return st;
    }
    // ---- layers
    // mixed_fp8: every E4M3 GEMM input is one tensor per chunk (1500 rows)
    // with one scale amax / 448 ("whisper-blaze 0.1.8", "Direct Kernel API",
    // quantise_e4m3 returns one scale per tensor)
    if (f8 && m->desc.enc_layers > 0)
        WB_CUDA(cudaMemsetAsync(e.amax, 0, sizeof(unsigned) * (size_t)m->desc.enc_layers * 3 * B, s));
    auto amax_of = [&](int l, int which) { return e.amax + ((int64_t)l * 3 + which) * B; };
    for (int l = 0; l < m->desc.enc_layers; ++l) {
        if (f8) {
            if (wb_status st = layernorm_group_e4m3(e.h, d, M, d, m->V(nm("enc.", l, "ln1.g")),
                                                    m->V(nm("enc.", l, "ln1.b")), kCtx, amax_of(l, 0),
                                                    reinterpret_cast<uint8_t*>(e.a), d, e.a_scale, s))
                return st;
        } else if (wb_status st = layernorm(e.h, d, M, d, m->V(nm("enc.", l, "ln1.g")), m->V(nm("enc.", l, "ln1.b")),
                                            ln_plain, e.a, d, e.a_scale, s)) {
            return st;
        }
        {
            Lin L;
            L.a = e.a; L.rows = M; L.lda = d; L.w = m->W(nm("enc.", l, "q.w")); L.N = 3 * d; L.K = d;
            if (f8) { L.f8 = &m->enc_qkv[l]; L.a_scale = e.a_scale; }
            if (wb_status st = linear(m, L, epi_out(e.qkv, 3 * d, act_out, m->V(nm("enc.", l, "q.b"))), s)) return st;
        }
        if (f32) {
            KVView kv;
            kv.ptr = e.qkv; kv.chunk_stride = (int64_t)kCtx * 3 * d; kv.head_stride = 64; kv.heads = H;
            kv.k_blk = 1; kv.v_blk = 2; kv.row_stride = 3 * d;
            if (wb_status st = attn_rows(DT_F32, DT_F32, DT_F32, e.qkv, 3 * d, B, kCtx, H, kv, kCtx, false, 0, e.attn,
                                         d, s))
                return st;
        } else {
            CUtensorMap tq;
            if (wb_status st = make_tma_2d_bf16(&tq, e.qkv, 3 * (uint64_t)d, (uint64_t)M, 3 * (uint64_t)d * 2, 64, 128))
                return st;
            if (wb_status st = attn_flash_tc_bf16(&tq, B, d, H, e.attn, m->err, s)) return st;
        }
        {
            Lin L;
            L.a = e.attn; L.rows = M; L.lda = d; L.w = m->W(nm("enc.", l, "o.w")); L.N = d; L.K = d;
            if (wb_status st = linear(m, L, epi_out(e.h, d, OUT_F32_ACC, m->V(nm("enc.", l, "o.b"))), s)) return st;
        }
        if (f8) {
            if (wb_status st = layernorm_group_e4m3(e.h, d, M, d, m->V(nm("enc.", l, "ln2.g")),
                                                    m->V(nm("enc.", l, "ln2.b")), kCtx, amax_of(l, 1),
                                                    reinterpret_cast<uint8_t*>(e.a), d, e.a_scale, s))
                return st;
        } else if (wb_status st = layernorm(e.h, d, M, d, m->V(nm("enc.", l, "ln2.g")), m->V(nm("enc.", l, "ln2.b")),
                                            ln_plain, e.a, d, e.a_scale, s)) {
            return st;
        }
        {
            Lin L;
            L.a = e.a; L.rows = M; L.lda = d; L.w = m->W(nm("enc.", l, "fc1.w")); L.N = F; L.K = d;
            GemmEpi ep = epi_out(e.f, F, act_out, m->V(nm("enc.", l, "fc1.b")), 1);
            if (f8) {
                // fp32 GELU output and each chunk's amax of it, taken in the epilogue
                L.f8 = &m->enc_fc1[l]; L.a_scale = e.a_scale;
                ep.out_type = OUT_F32;
                ep.amax = amax_of(l, 2);
                ep.amax_rows = kCtx;
            }
            if (wb_status st = linear(m, L, ep, s)) return st;
        }
        {
            Lin L;
            L.rows = M; L.w = m->W(nm("enc.", l, "fc2.w")); L.N = d; L.K = F;
            if (f8) {
                if (wb_status st = quant_groups(reinterpret_cast<const float*>(e.f), M, F, kCtx, amax_of(l, 2), e.fq,
                                                e.f_scale, s))
                    return st;
                L.a = e.fq; L.lda = F; L.f8 = &m->enc_fc2[l]; L.a_scale = e.f_scale;
            } else {
                L.a = e.f; L.lda = F;
            }
            if (wb_status st = linear(m, L, epi_out(e.h, d, OUT_F32_ACC, m->V(nm("enc.", l, "fc2.b"))), s)) return st;
        }
    }
    return layernorm(e.h, d, M, d, m->V("enc.lnp.g"), m->V("enc.lnp.b"), ln_plain, enc, d, nullptr, s);
}

size_t wb_decoder_workspace_size(const wb_model* m, int64_t B, const int32_t* len) {
    if (!m || B < 1 || !len) return 0;
    return carve_decoder(m, B, len, nullptr, nullptr, 0, nullptr);
}

// A decoder over n_chunks chunks with `beams` hypotheses each (rows c*beams
// .. c*beams + beams - 1 belong to chunk c), without its cross K/V yet.
static wb_status decoder_setup(wb_model* m, int64_t n_chunks, const int32_t* chunk_len, int beams, int32_t* tokens,
                               void* workspace, size_t ws_bytes, wb_stream stream, wb_decoder** out) {
    if (!out) return fail(WB_ERR_INVALID_ARG, "wb_decoder_init: null out");
    *out = nullptr;
    if (!m || !chunk_len || !tokens || !workspace) return fail(WB_ERR_INVALID_ARG, "wb_decoder_init: null argument");
    if (n_chunks < 1 || n_chunks * beams > 65535) return fail(WB_ERR_SHAPE, "wb_decoder_init: B * beams must be in [1, 65535]");
    if (!aligned16(tokens) || !aligned16(workspace)) return fail(WB_ERR_ALIGN, "wb_decoder_init: alignment");
    for (int64_t i = 0; i < n_chunks; ++i) {
        if (chunk_len[i] < 1 || chunk_len[i] > kMaxPos) return fail(WB_ERR_SHAPE, "wb_decoder_init: chunk_len must be in [1, 448]");
        if (i && chunk_len[i] > chunk_len[i - 1]) return fail(WB_ERR_SHAPE, "wb_decoder_init: chunk_len must be non-increasing");
    }
    const int64_t B = n_chunks * beams;          // rows
    std::vector<int32_t> len(B);
    for (int64_t r = 0; r < B; ++r) len[r] = chunk_len[r / beams];
    wb_decoder* dec = new wb_decoder();
    dec->m = m;
    dec->B = B;
    dec->len = len;
    dec->tokens = tokens;
    dec->max_len = len[0];
    bool over = false;
    carve_decoder(m, B, len.data(), dec, reinterpret_cast<uint8_t*>(workspace), ws_bytes, &over, beams);
    if (over) {
        delete dec;
        return fail(WB_ERR_SHAPE, "wb_decoder_init: workspace too small");
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int H = m->H(), Ld = m->desc.dec_layers;
    // per-row cache offsets (elements) and lengths
    std::vector<int64_t> off(B);
    int64_t acc = 0;
    for (int64_t i = 0; i < B; ++i) {
        off[i] = acc;
        acc += (int64_t)Ld * 2 * H * len[i] * 64;
    }
    auto fail_free = [&](wb_status st) { delete dec; return st; };
    if (cudaMemcpyAsync(dec->off, off.data(), B * 8, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dec->len_dev, len.data(), B * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return fail_free(fail(WB_ERR_CUDA, "wb_decoder_init: upload"));
    if (beams > 1)
        if (wb_status st = beam_init(dec->hist, dec->scores, B, beams, s)) return fail_free(st);
    *out = dec;
    return WB_OK;
}

// Cross-attention K/V of every decoder layer for the first NC chunks of the
// decoder from their encoder states enc [NC, 1500, d].
static wb_status compute_cross_kv(wb_decoder* dec, const void* enc, int64_t NC, cudaStream_t s) {
    wb_model* m = dec->m;
    const int d = m->d(), H = m->H(), Ld = m->desc.dec_layers;
    if (Ld <= 0 || NC <= 0) return WB_OK;
    if (m->desc.kv_fp8 != WB_KV_FP8_CROSS) {
        Lin L;
        L.a = enc; L.rows = NC * kCtx; L.lda = d; L.w = m->W("dec.0.ck.w"); L.N = (int64_t)Ld * 2 * d; L.K = d;
        GemmEpi ep = epi_out(dec->crosskv, 0, m->fp32() ? OUT_F32 : OUT_BF16, m->V("dec.0.ck.b"));
        ep.mode = MODE_CROSS_KV;
        ep.ckv_d = d;
        ep.ckv_heads = H;
        ep.ckv_chunks = dec->n_cross;
        return linear(m, L, ep, s);
    }
    // E4M3 cross K/V: per group of chunks, the fp32 projection into a scratch
    // area, then one amax / 448 scale and the codes per (chunk, layer, K|V)
    // tensor, rounded once from fp32
    for (int64_t g0 = 0; g0 < NC; g0 += kCrossGroup) {
        const int64_t gB = std::min<int64_t>(kCrossGroup, NC - g0);
        Lin L;
        L.a = reinterpret_cast<const __nv_bfloat16*>(enc) + g0 * kCtx * d;
        L.rows = gB * kCtx; L.lda = d; L.w = m->W("dec.0.ck.w"); L.N = (int64_t)Ld * 2 * d; L.K = d;
        GemmEpi ep = epi_out(dec->ckv_tmp, 0, OUT_F32, m->V("dec.0.ck.b"));
        ep.mode = MODE_CROSS_KV;
        ep.ckv_d = d;
        ep.ckv_heads = H;
        ep.ckv_chunks = gB;
        if (wb_status st = linear(m, L, ep, s)) return st;
        if (wb_status st = cross_kv_quant(dec->ckv_tmp, gB, dec->n_cross, g0, Ld, (int64_t)H * kCtx * 64,
                                          reinterpret_cast<uint8_t*>(dec->crosskv), dec->cscale, s))
            return st;
    }
    return WB_OK;
}

static wb_status decoder_init(wb_model* m, int64_t n_chunks, const int32_t* chunk_len, int beams, const void* enc,
                              int32_t* tokens, void* workspace, size_t ws_bytes, wb_stream stream, wb_decoder** out) {
    if (!enc) return fail(WB_ERR_INVALID_ARG, "wb_decoder_init: null argument");
    if (!aligned16(enc)) return fail(WB_ERR_ALIGN, "wb_decoder_init: alignment");
    wb_decoder* dec = nullptr;
    if (wb_status st = decoder_setup(m, n_chunks, chunk_len, beams, tokens, workspace, ws_bytes, stream, &dec))
        return st;
    if (wb_status st = compute_cross_kv(dec, enc, n_chunks, reinterpret_cast<cudaStream_t>(stream))) {
        delete dec;
        return st;
    }
    *out = dec;
    return WB_OK;
}

wb_status wb_decoder_init(wb_model* m, int64_t B, const int32_t* len, const void* enc, int32_t* tokens,
                          void* workspace, size_t ws_bytes, wb_stream stream, wb_decoder** out) {
    return decoder_init(m, B, len, 1, enc, tokens, workspace, ws_bytes, stream, out);
}

size_t wb_decoder_workspace_size_beams(const wb_model* m, int64_t B, const int32_t* chunk_len, int32_t beams) {
    if (!m || B < 1 || !chunk_len || beams < 1 || beams > kBeamMax) return 0;
    std::vector<int32_t> len((size_t)(B * beams));
    for (int64_t r = 0; r < B * beams; ++r) len[r] = chunk_len[r / beams];
    return carve_decoder(m, B * beams, len.data(), nullptr, nullptr, 0, nullptr, beams);
}

wb_status wb_decoder_init_beams(wb_model* m, int64_t B, const int32_t* chunk_len, int32_t beams, const void* enc,
                                int32_t* tokens, void* workspace, size_t ws_bytes, wb_stream stream, wb_decoder** out) {
    if (beams < 2 || beams > kBeamMax) return fail(WB_ERR_SHAPE, "wb_decoder_init_beams: beams must be in [2, 8]");
    return decoder_init(m, B, chunk_len, beams, enc, tokens, workspace, ws_bytes, stream, out);
}

wb_status wb_decode_prefix(wb_decoder* dec, int32_t P, float* logits, wb_stream stream) {
    if (!dec) return fail(WB_ERR_INVALID_ARG, "wb_decode_prefix: null decoder");
    if (P < 1 || P > kMaxPrefix || P > dec->len.back()) return fail(WB_ERR_SHAPE, "wb_decode_prefix: bad P");
    if (logits && !aligned16(logits)) return fail(WB_ERR_ALIGN, "wb_decode_prefix: logits alignment");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    wb_model* m = dec->m;
    const int64_t R = dec->B * P;
    if (wb_status st = embed(dec->tokens, R, P, 0, m->d(), m->W("dec.tok"), m->W("dec.pos"), !m->fp32(),
                             m->desc.vocab, dec->h, m->err, s))
        return st;
    if (wb_status st = decoder_layers(dec, dec->B, P, 0, true, s, nullptr)) return st;
    if (wb_status st = decoder_head(dec, dec->B, P, P - 1, logits, s, nullptr)) return st;
    if (wb_status st = set_pos(dec->pos_dev, P, false, s)) return st;
    dec->P = P;
    dec->pos = P;
    return WB_OK;
}

// One decode step over the first `rows` chunks; every position-dependent
// kernel reads the position from dec->pos_dev, and chunks that have finished
// are skipped on the device, so the same launch sequence serves every step.
static wb_status run_step(wb_decoder* dec, int64_t rows, float* logits, cudaStream_t s) {
    wb_model* m = dec->m;
    if (wb_status st = embed(dec->tokens, rows, 1, dec->pos, m->d(), m->W("dec.tok"), m->W("dec.pos"), !m->fp32(),
                             m->desc.vocab, dec->h, m->err, s, dec->pos_dev, dec->len_dev, dec->pos_stride))
        return st;
    if (wb_status st = decoder_layers(dec, rows, 1, dec->pos, false, s, dec->pos_dev)) return st;
    if (wb_status st = decoder_head(dec, rows, 1, dec->pos, logits, s, dec->pos_dev)) return st;
    return set_pos(dec->pos_dev, 1, true, s, dec->pos_stride ? (int)rows : 1);
}

static bool graphs_enabled() {
    const char* e = getenv("WB_NO_GRAPHS");
    return !(e && e[0] == '1');
}

// One decode step over `rows` rows, replayed from a CUDA graph captured the
// first time this row count is used (the step reads its positions from the
// device, so the same graph serves every step).
static wb_status replay_step(wb_decoder* dec, int64_t rows, cudaStream_t s) {
    StepGraph* g = nullptr;
    for (auto& x : dec->graphs)
        if (x.rows == rows) g = &x;
    if (!g) {
        StepGraph ng;
        ng.rows = rows;
        const int64_t k0 = wb_launch_count();
        // the caller's stream may be the legacy default stream, which cannot be
        // captured: record on a private stream, replay on the caller's
        if (!dec->cap_stream) WB_CUDA(cudaStreamCreateWithFlags(&dec->cap_stream, cudaStreamNonBlocking));
        WB_CUDA(cudaStreamBeginCapture(dec->cap_stream, cudaStreamCaptureModeThreadLocal));
        wb_status st = run_step(dec, rows, nullptr, dec->cap_stream);
        cudaGraph_t graph = nullptr;
        const cudaError_t ce = cudaStreamEndCapture(dec->cap_stream, &graph);
        if (st) {
            if (graph) cudaGraphDestroy(graph);
            return st;
        }
        if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamEndCapture(decode step)");
        const cudaError_t ie = cudaGraphInstantiate(&ng.exec, graph, 0);
        cudaGraphDestroy(graph);
        if (ie != cudaSuccess) return cuda_fail(ie, "cudaGraphInstantiate(decode step)");
        ng.kernels = wb_launch_count() - k0;
        count_launch((int)-ng.kernels);    // captured, not launched
        dec->graphs.push_back(ng);
        g = &dec->graphs.back();
    }
    WB_CUDA(cudaGraphLaunch(g->exec, s));
    count_launch((int)g->kernels);
    return WB_OK;
}

wb_status wb_decode_step(wb_decoder* dec, int64_t n_active, float* logits, wb_stream stream) {
    if (!dec) return fail(WB_ERR_INVALID_ARG, "wb_decode_step: null decoder");
    if (dec->beams > 1) return fail(WB_ERR_INVALID_ARG, "wb_decode_step: a beam decoder steps with wb_decode_step_beams");
    if (dec->P == 0) return fail(WB_ERR_INVALID_ARG, "wb_decode_step: run wb_decode_prefix first");
    if (n_active < 1 || n_active > dec->B) return fail(WB_ERR_SHAPE, "wb_decode_step: bad n_active");
    if (dec->len[n_active - 1] <= dec->pos + 1)
        return fail(WB_ERR_SHAPE, "wb_decode_step: an active chunk has reached its length");
    if (logits && !aligned16(logits)) return fail(WB_ERR_ALIGN, "wb_decode_step: logits alignment");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // logits for the caller, or per-kernel timing: launch directly with exactly n_active rows
    if (logits || !graphs_enabled() || prof_any_active()) {
        if (wb_status st = run_step(dec, n_active, logits, s)) return st;
        dec->pos += 1;
        return WB_OK;
    }
    // graph replay: rows rounded up to a 128-row bucket (finished chunks are masked)
    const int64_t rows = std::min<int64_t>(dec->B, (n_active + 127) / 128 * 128);
    if (wb_status st = replay_step(dec, rows, s)) return st;
    dec->pos += 1;
    return WB_OK;
}

wb_status wb_decode_step_beams(wb_decoder* dec, int64_t n_active, float* scores_out, int32_t* parents_out,
                               wb_stream stream) {
    if (!dec) return fail(WB_ERR_INVALID_ARG, "wb_decode_step_beams: null decoder");
    if (dec->beams < 2) return fail(WB_ERR_INVALID_ARG, "wb_decode_step_beams: not a beam decoder");
    if (dec->P == 0) return fail(WB_ERR_INVALID_ARG, "wb_decode_step_beams: run wb_decode_prefix first");
    const int64_t rows = n_active * dec->beams;
    if (n_active < 1 || rows > dec->B) return fail(WB_ERR_SHAPE, "wb_decode_step_beams: bad n_active");
    if (dec->len[rows - 1] <= dec->pos + 1)
        return fail(WB_ERR_SHAPE, "wb_decode_step_beams: an active chunk has reached its length");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dec->step_scores = scores_out;
    dec->step_parents = parents_out;
    const wb_status st = run_step(dec, rows, nullptr, s);
    dec->step_scores = nullptr;
    dec->step_parents = nullptr;
    if (st) return st;
    dec->pos += 1;
    return WB_OK;
}

wb_status wb_decoder_beam_scores(wb_decoder* dec, float* out, wb_stream stream) {
    if (!dec || !out) return fail(WB_ERR_INVALID_ARG, "wb_decoder_beam_scores: null argument");
    if (dec->beams < 2) return fail(WB_ERR_INVALID_ARG, "wb_decoder_beam_scores: not a beam decoder");
    WB_CUDA(cudaMemcpyAsync(out, dec->scores, sizeof(float) * (size_t)dec->B, cudaMemcpyDeviceToDevice,
                            reinterpret_cast<cudaStream_t>(stream)));
    return WB_OK;
}

wb_status wb_decoder_best_beams(wb_decoder* dec, int32_t* out_tokens, float* out_scores, wb_stream stream) {
    if (!dec || !out_tokens) return fail(WB_ERR_INVALID_ARG, "wb_decoder_best_beams: null argument");
    if (dec->beams < 2) return fail(WB_ERR_INVALID_ARG, "wb_decoder_best_beams: not a beam decoder");
    return beam_best(dec->scores, dec->tokens, dec->B / dec->beams, dec->beams, dec->len_dev, out_tokens, out_scores,
                     reinterpret_cast<cudaStream_t>(stream));
}

int32_t wb_decoder_position(const wb_decoder* dec) { return dec ? dec->pos : -1; }

wb_status wb_decoder_destroy(wb_decoder* dec) {
    if (!dec) return fail(WB_ERR_INVALID_ARG, "wb_decoder_destroy: null decoder");
    for (auto& g : dec->graphs)
        if (g.exec) cudaGraphExecDestroy(g.exec);
    if (dec->cap_stream) cudaStreamDestroy(dec->cap_stream);
    delete dec;
    return WB_OK;
}

wb_status wb_plan_waves(const wb_model_desc* desc, int32_t n, const int32_t* len, uint64_t budget,
                        int32_t* wave_of_chunk, int32_t* order, int32_t* n_waves_out) {
    std::string why;
    if (!valid_desc(desc, &why)) return fail(WB_ERR_INVALID_ARG, "wb_plan_waves: " + why);
    if (n < 0 || (n > 0 && (!len || !wave_of_chunk || !order))) return fail(WB_ERR_INVALID_ARG, "wb_plan_waves: args");
    std::vector<std::vector<int32_t>> waves;
    bool too_big = false;
    plan_waves_host(*desc, n, len, budget, waves, &too_big);
    if (too_big) return fail(WB_ERR_SHAPE, "wb_plan_waves: one chunk exceeds the wave budget");
    int32_t k = 0;
    for (size_t w = 0; w < waves.size(); ++w)
        for (int32_t c : waves[w]) {
            wave_of_chunk[c] = (int32_t)w;
            order[k++] = c;
        }
    if (n_waves_out) *n_waves_out = (int32_t)waves.size();
    return WB_OK;
}

// Work of one chunk for the split across GPUs, in decode positions: its own
// decode length plus the mel and encoder, which cost about as much as 48
// decode positions of the 32-layer large-v3 decoder.
constexpr int64_t kShardChunkBase = 48;

wb_status wb_shard_batch(int32_t n_req, const int64_t* req_offset, const int64_t* req_samples,
                         const int32_t* chunk_len, int32_t world, int32_t rank, int64_t* out_req_offset,
                         int64_t* out_req_samples, int32_t* out_n_req, int32_t* out_chunk_first,
                         int32_t* out_chunk_count) {
    if (n_req < 1 || !req_offset || !req_samples || !chunk_len || !out_req_offset || !out_req_samples || !out_n_req ||
        !out_chunk_first || !out_chunk_count)
        return fail(WB_ERR_INVALID_ARG, "wb_shard_batch: null argument or n_req < 1");
    if (world < 1 || rank < 0 || rank >= world) return fail(WB_ERR_INVALID_ARG, "wb_shard_batch: bad world/rank");
    // chunks in request order: (request, index), as the chunk table of wb_transcribe_batch
    std::vector<int32_t> creq;
    std::vector<int64_t> cidx;
    for (int32_t r = 0; r < n_req; ++r) {
        if (req_samples[r] < 1) return fail(WB_ERR_SHAPE, "wb_shard_batch: empty request");
        const int64_t n = (req_samples[r] + kChunkSamples - 1) / kChunkSamples;
        for (int64_t k = 0; k < n; ++k) {
            creq.push_back(r);
            cidx.push_back(k);
        }
    }
    const int64_t n = (int64_t)creq.size();
    if (n > INT32_MAX) return fail(WB_ERR_SHAPE, "wb_shard_batch: too many chunks");
    int64_t total = 0;
    for (int64_t c = 0; c < n; ++c) {
        if (chunk_len[c] < 1) return fail(WB_ERR_SHAPE, "wb_shard_batch: chunk_len < 1");
        total += chunk_len[c] + kShardChunkBase;
    }
    // range r = [first(r), first(r + 1)), first(r) = the first chunk whose
    // preceding work w satisfies w * world >= r * total
    auto first_of = [&](int64_t r) -> int64_t {
        if (r <= 0) return 0;
        if (r >= world) return n;
        int64_t w = 0;
        for (int64_t c = 0; c < n; ++c) {
            if (w * world >= r * total) return c;
            w += chunk_len[c] + kShardChunkBase;
        }
        return n;
    };
    const int64_t c0 = first_of(rank), c1 = first_of((int64_t)rank + 1);
    *out_chunk_first = (int32_t)c0;
    *out_chunk_count = (int32_t)(c1 - c0);
    int32_t k = 0;
    for (int64_t c = c0; c < c1;) {
        const int32_t r = creq[c];
        int64_t e = c;   // chunks of request r inside the range
        while (e < c1 && creq[e] == r) ++e;
        const int64_t s0 = cidx[c] * kChunkSamples;
        const int64_t s1 = std::min<int64_t>(req_samples[r], (cidx[e - 1] + 1) * kChunkSamples);
        out_req_offset[k] = req_offset[r] + s0;
        out_req_samples[k] = s1 - s0;
        ++k;
        c = e;
    }
    *out_n_req = k;
    return WB_OK;
}

struct TranscribeBufs {
    float* chunk_audio = nullptr;
    float* mel = nullptr;
    uint8_t* enc = nullptr;          // encoder states of one wave
    uint8_t* enc2 = nullptr;         // the next wave's, encoded while this one decodes (several waves)
    int32_t* wave_tok = nullptr;
    int64_t* src = nullptr;
    int32_t* valid = nullptr;
    int32_t* dst_row = nullptr;
    int32_t* wlen = nullptr;
    uint8_t* enc_ws = nullptr;
    size_t enc_ws_bytes = 0;
    uint8_t* dec_ws = nullptr;
    size_t dec_ws_bytes = 0;
};

static size_t transcribe_ws(const wb_model* m, int64_t max_wave, const std::vector<std::vector<int32_t>>& waves,
                            const std::vector<int32_t>& lens, uint8_t* base, size_t cap, TranscribeBufs* tb,
                            bool* overflow) {
    Carve c{base, cap};
    const int d = m->d();
    const size_t act = m->fp32() ? 4 : 2;
    const int64_t EB = std::min<int64_t>(kEncSubBatch, std::max<int64_t>(1, max_wave));
    TranscribeBufs t;
    t.chunk_audio = c.take<float>((size_t)max_wave * kChunkSamples);
    t.mel = c.take<float>((size_t)max_wave * m->desc.n_mels * kFrames);
    t.enc = c.take<uint8_t>((size_t)max_wave * kCtx * d * act);
    if (waves.size() > 1) t.enc2 = c.take<uint8_t>((size_t)max_wave * kCtx * d * act);
    t.wave_tok = c.take<int32_t>((size_t)max_wave * kMaxPos);
    // per-chunk tables of all waves, in wave order
    const int64_t n_all = (int64_t)lens.size();
    t.src = c.take<int64_t>(n_all);
    t.valid = c.take<int32_t>(n_all);
    t.dst_row = c.take<int32_t>(n_all);
    t.wlen = c.take<int32_t>(n_all);
    t.enc_ws_bytes = carve_encoder(m, EB, nullptr, nullptr, 0, nullptr);
    t.enc_ws = c.take<uint8_t>(t.enc_ws_bytes);
    for (const auto& w : waves) {
        std::vector<int32_t> l;
        for (int32_t ci : w) l.push_back(lens[ci]);
        t.dec_ws_bytes = std::max(t.dec_ws_bytes, carve_decoder(m, (int64_t)w.size(), l.data(), nullptr, nullptr, 0, nullptr));
    }
    t.dec_ws = c.take<uint8_t>(t.dec_ws_bytes);
    if (tb) *tb = t;
    if (overflow) *overflow = c.overflow;
    return align_up(c.cur, 256);
}

// Chunk k of request r starts k * stride samples in (stride = 480000 -
// overlap) and holds min(480000, samples_r - k * stride) real samples; a
// request has 1 + ceil(max(0, samples_r - 480000) / stride) chunks.
static bool chunk_table(int32_t n_req, const int64_t* req_samples, std::vector<int32_t>& req, std::vector<int64_t>& idx,
                        std::vector<int32_t>& valid, int64_t overlap = 0) {
    const int64_t stride = kChunkSamples - overlap;
    if (overlap < 0 || stride < 1) return false;
    for (int32_t r = 0; r < n_req; ++r) {
        if (req_samples[r] < 1) return false;
        const int64_t n = 1 + (std::max<int64_t>(0, req_samples[r] - kChunkSamples) + stride - 1) / stride;
        for (int64_t k = 0; k < n; ++k) {
            req.push_back(r);
            idx.push_back(k);
            valid.push_back((int32_t)std::min<int64_t>(kChunkSamples, req_samples[r] - k * stride));
        }
    }
    return true;
}

int64_t wb_chunk_count(int32_t n_req, const int64_t* req_samples, int64_t overlap_samples) {
    if (n_req < 1 || !req_samples) return -1;
    std::vector<int32_t> req, valid;
    std::vector<int64_t> idx;
    if (!chunk_table(n_req, req_samples, req, idx, valid, overlap_samples)) return -1;
    return (int64_t)req.size();
}

static size_t transcribe_ws_size(const wb_model* m, int32_t n_req, const int64_t* req_samples, const int32_t* chunk_len,
                                 uint64_t budget, int64_t overlap);

size_t wb_transcribe_workspace_size(const wb_model* m, int32_t n_req, const int64_t* req_samples,
                                    const int32_t* chunk_len, uint64_t budget) {
    return transcribe_ws_size(m, n_req, req_samples, chunk_len, budget, 0);
}

size_t wb_transcribe_workspace_size_overlap(const wb_model* m, int32_t n_req, const int64_t* req_samples,
                                            const int32_t* chunk_len, uint64_t budget, int64_t overlap_samples) {
    return transcribe_ws_size(m, n_req, req_samples, chunk_len, budget, overlap_samples);
}

static size_t transcribe_ws_size(const wb_model* m, int32_t n_req, const int64_t* req_samples, const int32_t* chunk_len,
                                 uint64_t budget, int64_t overlap) {
    if (!m || n_req < 1 || !req_samples || !chunk_len) return 0;
    std::vector<int32_t> req, valid;
    std::vector<int64_t> idx;
    if (!chunk_table(n_req, req_samples, req, idx, valid, overlap)) return 0;
    std::vector<int32_t> lens(chunk_len, chunk_len + req.size());
    std::vector<std::vector<int32_t>> waves;
    bool too_big = false;
    plan_waves_host(m->desc, (int32_t)req.size(), lens.data(), budget, waves, &too_big);
    if (too_big) return 0;
    int64_t mw = 0;
    for (auto& w : waves) mw = std::max<int64_t>(mw, (int64_t)w.size());
    return transcribe_ws(m, mw, waves, lens, nullptr, 0, nullptr, nullptr);
}

static wb_status transcribe_impl(wb_model* m, const float* audio, const int64_t* req_offset, const int64_t* req_samples,
                                 int32_t n_req, const int32_t* prefix, const int32_t* chunk_len, int32_t* tokens,
                                 uint64_t budget, void* workspace, size_t ws_bytes, int32_t* n_waves_out,
                                 wb_stream stream, int64_t overlap);

wb_status wb_transcribe_batch(wb_model* m, const float* audio, const int64_t* req_offset, const int64_t* req_samples,
                              int32_t n_req, const int32_t* prefix, const int32_t* chunk_len, int32_t* tokens,
                              uint64_t budget, void* workspace, size_t ws_bytes, int32_t* n_waves_out,
                              wb_stream stream) {
    return transcribe_impl(m, audio, req_offset, req_samples, n_req, prefix, chunk_len, tokens, budget, workspace,
                           ws_bytes, n_waves_out, stream, 0);
}

wb_status wb_transcribe_batch_overlap(wb_model* m, const float* audio, const int64_t* req_offset,
                                      const int64_t* req_samples, int32_t n_req, int64_t overlap_samples,
                                      const int32_t* prefix, const int32_t* chunk_len, int32_t* tokens, uint64_t budget,
                                      void* workspace, size_t ws_bytes, int32_t* n_waves_out, wb_stream stream) {
    if (overlap_samples < 0 || overlap_samples >= kChunkSamples)
        return fail(WB_ERR_SHAPE, "wb_transcribe_batch_overlap: overlap must be in [0, 480000)");
    return transcribe_impl(m, audio, req_offset, req_samples, n_req, prefix, chunk_len, tokens, budget, workspace,
                           ws_bytes, n_waves_out, stream, overlap_samples);
}

static wb_status transcribe_impl(wb_model* m, const float* audio, const int64_t* req_offset, const int64_t* req_samples,
                                 int32_t n_req, const int32_t* prefix, const int32_t* chunk_len, int32_t* tokens,
                                 uint64_t budget, void* workspace, size_t ws_bytes, int32_t* n_waves_out,
                                 wb_stream stream, int64_t overlap) {
    if (!m || !audio || !req_offset || !req_samples || !prefix || !chunk_len || !tokens || !workspace)
        return fail(WB_ERR_INVALID_ARG, "wb_transcribe_batch: null argument");
    if (n_req < 1) return fail(WB_ERR_SHAPE, "wb_transcribe_batch: n_req < 1");
    if (!aligned16(audio) || !aligned16(tokens) || !aligned16(workspace))
        return fail(WB_ERR_ALIGN, "wb_transcribe_batch: alignment");
    for (int32_t r = 0; r < n_req; ++r)
        if (req_offset[r] < 0) return fail(WB_ERR_SHAPE, "wb_transcribe_batch: negative request offset");
    for (int i = 0; i < 4; ++i)
        if (prefix[i] < 0 || prefix[i] >= m->desc.vocab) return fail(WB_ERR_SHAPE, "wb_transcribe_batch: prefix id");
    std::vector<int32_t> req, valid;
    std::vector<int64_t> idx;
    if (!chunk_table(n_req, req_samples, req, idx, valid, overlap))
        return fail(WB_ERR_SHAPE, "wb_transcribe_batch: empty request");
    const int64_t stride = kChunkSamples - overlap;
    const int32_t n = (int32_t)req.size();
    std::vector<int32_t> lens(chunk_len, chunk_len + n);
    for (int32_t c = 0; c < n; ++c)
        if (lens[c] < 5 || lens[c] > kMaxPos) return fail(WB_ERR_SHAPE, "wb_transcribe_batch: chunk_len must be in [5, 448]");
    std::vector<std::vector<int32_t>> waves;
    bool too_big = false;
    plan_waves_host(m->desc, n, lens.data(), budget, waves, &too_big);
    if (too_big) return fail(WB_ERR_SHAPE, "wb_transcribe_batch: one chunk exceeds the wave budget");
    int64_t mw = 0;
    for (auto& w : waves) mw = std::max<int64_t>(mw, (int64_t)w.size());
    TranscribeBufs tb;
    bool over = false;
    transcribe_ws(m, mw, waves, lens, reinterpret_cast<uint8_t*>(workspace), ws_bytes, &tb, &over);
    if (over) return fail(WB_ERR_SHAPE, "wb_transcribe_batch: workspace too small");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int d = m->d();
    const size_t act = m->fp32() ? 4 : 2;
    // chunk tables of all waves, wave after wave
    const size_t nwav = waves.size();
    std::vector<int64_t> wave_off(nwav + 1, 0), hsrc((size_t)n);
    std::vector<int32_t> hvalid((size_t)n), hdst((size_t)n), hlen((size_t)n);
    for (size_t wi = 0; wi < nwav; ++wi) {
        wave_off[wi + 1] = wave_off[wi] + (int64_t)waves[wi].size();
        for (size_t i = 0; i < waves[wi].size(); ++i) {
            const int32_t c = waves[wi][i];
            const int64_t k = wave_off[wi] + (int64_t)i;
            hsrc[k] = req_offset[req[c]] + idx[c] * stride;
            hvalid[k] = valid[c];
            hdst[k] = c;
            hlen[k] = lens[c];
        }
    }
    WB_CUDA(cudaMemcpyAsync(tb.src, hsrc.data(), (size_t)n * 8, cudaMemcpyHostToDevice, s));
    WB_CUDA(cudaMemcpyAsync(tb.valid, hvalid.data(), (size_t)n * 4, cudaMemcpyHostToDevice, s));
    WB_CUDA(cudaMemcpyAsync(tb.dst_row, hdst.data(), (size_t)n * 4, cudaMemcpyHostToDevice, s));
    WB_CUDA(cudaMemcpyAsync(tb.wlen, hlen.data(), (size_t)n * 4, cudaMemcpyHostToDevice, s));
    WB_CUDA(cudaStreamSynchronize(s));        // pageable sources are consumed before the vectors go away
    // The next wave's mel and encoder run on a second, lower-priority stream
    // while this wave decodes: the decode steps are bound by HBM (the
    // cross-attention stream), the encoder by the tensor cores.
    cudaStream_t es = nullptr;
    cudaEvent_t ev_enc[2] = {nullptr, nullptr}, ev_init[2] = {nullptr, nullptr};
    auto release = [&](wb_status st) {
        for (int b = 0; b < 2; ++b) {
            if (ev_enc[b]) cudaEventDestroy(ev_enc[b]);
            if (ev_init[b]) cudaEventDestroy(ev_init[b]);
        }
        if (es) cudaStreamDestroy(es);
        return st;
    };
    {
        int lo = 0, hi = 0;
        if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess ||
            cudaStreamCreateWithPriority(&es, cudaStreamNonBlocking, lo) != cudaSuccess)
            return release(fail(WB_ERR_CUDA, "wb_transcribe_batch: encoder stream"));
        for (int b = 0; b < 2; ++b)
            if (cudaEventCreateWithFlags(&ev_enc[b], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&ev_init[b], cudaEventDisableTiming) != cudaSuccess)
                return release(fail(WB_ERR_CUDA, "wb_transcribe_batch: events"));
    }
    // the ordering of the caller's stream so far (the tables above) precedes the encoder stream's work
    if (cudaEventRecord(ev_init[1], s) != cudaSuccess || cudaStreamWaitEvent(es, ev_init[1], 0) != cudaSuccess)
        return release(fail(WB_ERR_CUDA, "wb_transcribe_batch: stream order"));
    uint8_t* enc_buf[2] = {tb.enc, tb.enc2 ? tb.enc2 : tb.enc};
    auto encode_wave = [&](size_t wi) -> wb_status {
        const int64_t nw = (int64_t)waves[wi].size(), off = wave_off[wi];
        uint8_t* enc = enc_buf[wi & 1];
        WB_CUDA(launch_k(gather_chunks_kernel, dim3((kChunkSamples / 4 + 255) / 256, (unsigned)nw), dim3(256), 0, es,
                         audio, tb.src + off, tb.valid + off, tb.chunk_audio));
        WB_CUDA(cudaGetLastError());
        if (wb_status st = wb_mel(tb.chunk_audio, nw, m->desc.n_mels, tb.mel, reinterpret_cast<wb_stream>(es)))
            return st;
        for (int64_t i0 = 0; i0 < nw; i0 += kEncSubBatch) {
            const int64_t nb = std::min<int64_t>(kEncSubBatch, nw - i0);
            if (wb_status st = wb_encode(m, tb.mel + i0 * m->desc.n_mels * kFrames, nb, enc + (size_t)i0 * kCtx * d * act,
                                         tb.enc_ws, tb.enc_ws_bytes, reinterpret_cast<wb_stream>(es)))
                return st;
        }
        WB_CUDA(cudaEventRecord(ev_enc[wi & 1], es));
        return WB_OK;
    };
    auto run = [&]() -> wb_status {
        if (wb_status st = encode_wave(0)) return st;
        for (size_t wi = 0; wi < nwav; ++wi) {
            const int64_t nw = (int64_t)waves[wi].size(), off = wave_off[wi];
            const int32_t* wl = hlen.data() + off;
            WB_CUDA(cudaStreamWaitEvent(s, ev_enc[wi & 1], 0));
            WB_CUDA(launch_k(fill_prefix_kernel, dim3((unsigned)((nw + 255) / 256)), dim3(256), 0, s, tb.wave_tok, nw,
                             prefix[0], prefix[1], prefix[2], prefix[3]));
            WB_CUDA(cudaGetLastError());
            wb_decoder* dec = nullptr;
            if (wb_status st = wb_decoder_init(m, nw, wl, enc_buf[wi & 1], tb.wave_tok, tb.dec_ws, tb.dec_ws_bytes, stream,
                                               &dec))
                return st;
            // this wave's encoder states are consumed (cross K/V computed): the
            // buffer takes wave wi + 2
            WB_CUDA(cudaEventRecord(ev_init[wi & 1], s));
            if (wi + 1 < nwav) {
                WB_CUDA(cudaStreamWaitEvent(es, ev_init[(wi + 1) & 1], 0));
                if (wb_status st = encode_wave(wi + 1)) {
                    wb_decoder_destroy(dec);
                    return st;
                }
            }
            wb_status st = wb_decode_prefix(dec, 4, nullptr, stream);
            for (int t = 4; !st && t + 1 < wl[0]; ++t) {
                int64_t na = 0;
                while (na < nw && wl[na] > t + 1) ++na;
                st = wb_decode_step(dec, na, nullptr, stream);
            }
            wb_decoder_destroy(dec);
            if (st) return st;
            WB_CUDA(launch_k(scatter_tokens_kernel, dim3((unsigned)nw), dim3(128), 0, s, tb.wave_tok, tb.dst_row + off,
                             tb.wlen + off, tokens));
            WB_CUDA(cudaGetLastError());
        }
        return WB_OK;
    };
    if (wb_status st = release(run())) return st;
    if (n_waves_out) *n_waves_out = (int32_t)waves.size();
    return wb_sync_status(m, stream);
}

// ------------------------------------------------------------------ continuous batching
// Slots of a decoder that stays full: chunks (longest first) enter free
// slots in groups of up to R as earlier chunks finish, every slot at its own
// position ("whisper-blaze 0.1.8", "Serving at Scale": requests of mixed
// lengths are batched together).  Per-slot state: cross K/V, an E4M3 cache of
// 448 rows, the token row.
struct ContPlan {
    int64_t S = 0, R = 0;
};

static uint64_t slot_bytes(const wb_model_desc& d) {
    const uint64_t cross_elt = d.kv_fp8 == WB_KV_FP8_CROSS ? 1 : 2;
    return (uint64_t)d.dec_layers * 2 * kCtx * d.d_model * cross_elt + (uint64_t)d.dec_layers * 2 * kMaxPos * d.d_model +
           (uint64_t)kMaxPos * 4;
}

static ContPlan cont_plan(const wb_model_desc& d, int64_t n_chunks, uint64_t budget) {
    ContPlan p;
    p.S = std::min<int64_t>(n_chunks, (int64_t)(budget / std::max<uint64_t>(1, slot_bytes(d))));
    p.S = std::min<int64_t>(p.S, 65535);
    p.R = std::max<int64_t>(1, std::min<int64_t>({p.S, 32, p.S / 8}));
    return p;
}

struct ContBufs {
    float* chunk_audio = nullptr;
    float* mel = nullptr;
    uint8_t* enc_ws = nullptr;
    size_t enc_ws_bytes = 0;
    uint8_t* enc_all = nullptr;      // [n_chunks, 1500, d] encoder states
    uint8_t* st_enc = nullptr;       // [R, 1500, d] states of the chunks entering slots
    int32_t* st_tok = nullptr;       // [R, 448]
    int32_t* sl_tok = nullptr;       // [S, 448]
    int64_t* src = nullptr;
    int32_t* valid = nullptr;
    int32_t* slot_of = nullptr;      // [R]
    int32_t* new_len = nullptr;      // [R]
    int32_t* out_slot = nullptr;     // [S]
    int32_t* out_chunk = nullptr;    // [S]
    int32_t* out_len = nullptr;      // [S]
    uint8_t* sl_ws = nullptr;
    size_t sl_ws_bytes = 0;
    uint8_t* st_ws = nullptr;
    size_t st_ws_bytes = 0;
};

static size_t cont_ws(const wb_model* m, int64_t n_chunks, const ContPlan& p, uint8_t* base, size_t cap, ContBufs* cb,
                      bool* overflow) {
    Carve c{base, cap};
    const int d = m->d();
    const size_t act = m->fp32() ? 4 : 2;
    const int64_t EB = std::min<int64_t>(kEncSubBatch, n_chunks);
    ContBufs b;
    b.chunk_audio = c.take<float>((size_t)EB * kChunkSamples);
    b.mel = c.take<float>((size_t)EB * m->desc.n_mels * kFrames);
    b.enc_ws_bytes = carve_encoder(m, EB, nullptr, nullptr, 0, nullptr);
    b.enc_ws = c.take<uint8_t>(b.enc_ws_bytes);
    b.enc_all = c.take<uint8_t>((size_t)n_chunks * kCtx * d * act);
    b.st_enc = c.take<uint8_t>((size_t)p.R * kCtx * d * act);
    b.st_tok = c.take<int32_t>((size_t)p.R * kMaxPos);
    b.sl_tok = c.take<int32_t>((size_t)p.S * kMaxPos);
    b.src = c.take<int64_t>(EB);
    b.valid = c.take<int32_t>(EB);
    b.slot_of = c.take<int32_t>(p.R);
    b.new_len = c.take<int32_t>(p.R);
    b.out_slot = c.take<int32_t>(p.S);
    b.out_chunk = c.take<int32_t>(p.S);
    b.out_len = c.take<int32_t>(p.S);
    std::vector<int32_t> lay_s((size_t)p.S, kMaxPos), lay_r((size_t)p.R, kMaxPos);
    b.sl_ws_bytes = carve_decoder(m, p.S, lay_s.data(), nullptr, nullptr, 0, nullptr);
    b.sl_ws = c.take<uint8_t>(b.sl_ws_bytes);
    b.st_ws_bytes = carve_decoder(m, p.R, lay_r.data(), nullptr, nullptr, 0, nullptr);
    b.st_ws = c.take<uint8_t>(b.st_ws_bytes);
    if (cb) *cb = b;
    if (overflow) *overflow = c.overflow;
    return align_up(c.cur, 256);
}

size_t wb_transcribe_workspace_size_continuous(const wb_model* m, int32_t n_req, const int64_t* req_samples,
                                               uint64_t budget) {
    if (!m || n_req < 1 || !req_samples) return 0;
    std::vector<int32_t> req, valid;
    std::vector<int64_t> idx;
    if (!chunk_table(n_req, req_samples, req, idx, valid)) return 0;
    const ContPlan p = cont_plan(m->desc, (int64_t)req.size(), budget);
    if (p.S < 1) return 0;
    return cont_ws(m, (int64_t)req.size(), p, nullptr, 0, nullptr, nullptr);
}

wb_status wb_transcribe_batch_continuous(wb_model* m, const float* audio, const int64_t* req_offset,
                                         const int64_t* req_samples, int32_t n_req, const int32_t* prefix,
                                         const int32_t* chunk_len, int32_t* tokens, uint64_t budget, void* workspace,
                                         size_t ws_bytes, int32_t* n_slots_out, wb_stream stream) {
    if (!m || !audio || !req_offset || !req_samples || !prefix || !chunk_len || !tokens || !workspace)
        return fail(WB_ERR_INVALID_ARG, "wb_transcribe_batch_continuous: null argument");
    if (n_req < 1) return fail(WB_ERR_SHAPE, "wb_transcribe_batch_continuous: n_req < 1");
    if (!aligned16(audio) || !aligned16(tokens) || !aligned16(workspace))
        return fail(WB_ERR_ALIGN, "wb_transcribe_batch_continuous: alignment");
    for (int32_t r = 0; r < n_req; ++r)
        if (req_offset[r] < 0) return fail(WB_ERR_SHAPE, "wb_transcribe_batch_continuous: negative request offset");
    if (m->fp32() || !m->desc.kv_fp8)
        return fail(WB_ERR_UNSUPPORTED, "wb_transcribe_batch_continuous: needs a bf16 model with the E4M3 cache");
    for (int i = 0; i < 4; ++i)
        if (prefix[i] < 0 || prefix[i] >= m->desc.vocab)
            return fail(WB_ERR_SHAPE, "wb_transcribe_batch_continuous: prefix id");
    std::vector<int32_t> req, valid;
    std::vector<int64_t> idx;
    if (!chunk_table(n_req, req_samples, req, idx, valid))
        return fail(WB_ERR_SHAPE, "wb_transcribe_batch_continuous: empty request");
    const int64_t n = (int64_t)req.size();
    for (int64_t c = 0; c < n; ++c)
        if (chunk_len[c] < 5 || chunk_len[c] > kMaxPos)
            return fail(WB_ERR_SHAPE, "wb_transcribe_batch_continuous: chunk_len must be in [5, 448]");
    const ContPlan p = cont_plan(m->desc, n, budget);
    if (p.S < 1) return fail(WB_ERR_SHAPE, "wb_transcribe_batch_continuous: the budget holds no slot");
    ContBufs cb;
    bool over = false;
    cont_ws(m, n, p, reinterpret_cast<uint8_t*>(workspace), ws_bytes, &cb, &over);
    if (over) return fail(WB_ERR_SHAPE, "wb_transcribe_batch_continuous: workspace too small");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int d = m->d(), H = m->H(), Ld = m->desc.dec_layers;
    const size_t act = 2;
    const size_t enc_bytes = (size_t)kCtx * d * act;
    // ---- every chunk through mel and the encoder, in groups
    for (int64_t c0 = 0; c0 < n; c0 += kEncSubBatch) {
        const int64_t nb = std::min<int64_t>(kEncSubBatch, n - c0);
        std::vector<int64_t> hsrc(nb);
        std::vector<int32_t> hval(nb);
        for (int64_t i = 0; i < nb; ++i) {
            hsrc[i] = req_offset[req[c0 + i]] + idx[c0 + i] * kChunkSamples;
            hval[i] = valid[c0 + i];
        }
        WB_CUDA(cudaMemcpyAsync(cb.src, hsrc.data(), nb * 8, cudaMemcpyHostToDevice, s));
        WB_CUDA(cudaMemcpyAsync(cb.valid, hval.data(), nb * 4, cudaMemcpyHostToDevice, s));
        WB_CUDA(cudaStreamSynchronize(s));    // pageable sources are consumed before the vectors go away
        WB_CUDA(launch_k(gather_chunks_kernel, dim3((kChunkSamples / 4 + 255) / 256, (unsigned)nb), dim3(256), 0, s,
                         audio, cb.src, cb.valid, cb.chunk_audio));
        WB_CUDA(cudaGetLastError());
        if (wb_status st = wb_mel(cb.chunk_audio, nb, m->desc.n_mels, cb.mel, stream)) return st;
        if (wb_status st = wb_encode(m, cb.mel, nb, cb.enc_all + (size_t)c0 * enc_bytes, cb.enc_ws, cb.enc_ws_bytes,
                                     stream))
            return st;
    }
    // ---- the slot decoder (S rows, one position each) and the staging decoder (R rows)
    std::vector<int32_t> lay_s((size_t)p.S, kMaxPos), lay_r((size_t)p.R, kMaxPos);
    wb_decoder* sl = nullptr;
    wb_decoder* stg = nullptr;
    if (wb_status st = decoder_setup(m, p.S, lay_s.data(), 1, cb.sl_tok, cb.sl_ws, cb.sl_ws_bytes, stream, &sl)) return st;
    auto done = [&](wb_status st) {
        if (sl) wb_decoder_destroy(sl);
        if (stg) wb_decoder_destroy(stg);
        return st;
    };
    if (wb_status st = decoder_setup(m, p.R, lay_r.data(), 1, cb.st_tok, cb.st_ws, cb.st_ws_bytes, stream, &stg))
        return done(st);
    sl->pos_stride = 1;
    sl->lay_dev = sl->lay_buf;
    sl->P = 4;
    WB_CUDA(cudaMemcpyAsync(sl->lay_dev, lay_s.data(), p.S * 4, cudaMemcpyHostToDevice, s));
    WB_CUDA(cudaMemsetAsync(sl->len_dev, 0, p.S * 4, s));       // every slot starts empty (masked)
    WB_CUDA(cudaMemsetAsync(sl->pos_dev, 0, p.S * 4, s));
    WB_CUDA(cudaMemsetAsync(sl->attn, 0, (size_t)p.S * kMaxPrefix * d * 4, s));
    WB_CUDA(cudaStreamSynchronize(s));                          // lay_s is pageable
    // ---- schedule: longest chunks first, refills of up to R slots
    std::vector<int32_t> order((size_t)n);
    for (int64_t i = 0; i < n; ++i) order[i] = (int32_t)i;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return chunk_len[a] > chunk_len[b]; });
    std::vector<int32_t> slot_chunk((size_t)p.S, -1);     // chunk held (finished or not), -1: empty
    std::vector<int32_t> remaining((size_t)p.S, 0);       // steps the slot's chunk still needs
    const int64_t cross_blk = (int64_t)2 * H * kCtx * 64 * (m->desc.kv_fp8 == WB_KV_FP8_CROSS ? 1 : 2);
    // finished chunks' token rows to the output (the listed slots)
    auto flush = [&](const std::vector<int32_t>& slots) -> wb_status {
        std::vector<int32_t> os, oc, ol;
        for (int32_t q : slots)
            if (slot_chunk[q] >= 0) {
                os.push_back(q);
                oc.push_back(slot_chunk[q]);
                ol.push_back(chunk_len[slot_chunk[q]]);
                slot_chunk[q] = -1;
            }
        if (os.empty()) return WB_OK;
        const size_t k = os.size();
        WB_CUDA(cudaMemcpyAsync(cb.out_slot, os.data(), k * 4, cudaMemcpyHostToDevice, s));
        WB_CUDA(cudaMemcpyAsync(cb.out_chunk, oc.data(), k * 4, cudaMemcpyHostToDevice, s));
        WB_CUDA(cudaMemcpyAsync(cb.out_len, ol.data(), k * 4, cudaMemcpyHostToDevice, s));
        return slot_out(cb.sl_tok, cb.out_slot, cb.out_chunk, cb.out_len, (int)k, tokens, s);
    };
    size_t qi = 0;
    while (true) {
        std::vector<int32_t> free_slots;
        int64_t active = 0;
        for (int64_t q = 0; q < p.S; ++q) {
            if (remaining[q] > 0) ++active;
            else free_slots.push_back((int32_t)q);
        }
        if (qi < order.size() && ((int64_t)free_slots.size() >= p.R || active == 0)) {
            const int64_t k = std::min<int64_t>({(int64_t)free_slots.size(), p.R, (int64_t)(order.size() - qi)});
            std::vector<int32_t> slots(free_slots.begin(), free_slots.begin() + k), chunks(k), lens(k);
            if (wb_status st = flush(slots)) return done(st);
            for (int64_t i = 0; i < k; ++i) {
                chunks[i] = order[qi + i];
                lens[i] = chunk_len[chunks[i]];
                WB_CUDA(cudaMemcpyAsync(cb.st_enc + (size_t)i * enc_bytes, cb.enc_all + (size_t)chunks[i] * enc_bytes,
                                        enc_bytes, cudaMemcpyDeviceToDevice, s));
            }
            qi += (size_t)k;
            // the entering chunks' prefix pass in the staging decoder
            WB_CUDA(launch_k(fill_prefix_kernel, dim3((unsigned)((p.R + 255) / 256)), dim3(256), 0, s, cb.st_tok,
                             (int64_t)p.R, prefix[0], prefix[1], prefix[2], prefix[3]));
            if (wb_status st = compute_cross_kv(stg, cb.st_enc, k, s)) return done(st);
            if (wb_status st = wb_decode_prefix(stg, 4, nullptr, stream)) return done(st);
            WB_CUDA(cudaMemcpyAsync(cb.slot_of, slots.data(), k * 4, cudaMemcpyHostToDevice, s));
            WB_CUDA(cudaMemcpyAsync(cb.new_len, lens.data(), k * 4, cudaMemcpyHostToDevice, s));
            const bool c8 = m->desc.kv_fp8 == WB_KV_FP8_CROSS;
            if (wb_status st = slot_cross_copy(stg->crosskv, sl->crosskv, cb.slot_of, (int)k, p.R, p.S, Ld, cross_blk, s,
                                               c8 ? stg->cscale : nullptr, c8 ? sl->cscale : nullptr))
                return done(st);
            if (wb_status st = slot_state(reinterpret_cast<const uint8_t*>(stg->cache), reinterpret_cast<uint8_t*>(sl->cache),
                                          stg->kscale, stg->vscale, sl->kscale, sl->vscale, cb.st_tok, cb.sl_tok,
                                          sl->pos_dev, sl->len_dev, cb.slot_of, cb.new_len, (int)k, (int)p.R,
                                          (int)p.S, Ld, H, kMaxPos, 4, s))
                return done(st);
            for (int64_t i = 0; i < k; ++i) {
                slot_chunk[slots[i]] = chunks[i];
                remaining[slots[i]] = lens[i] - 5;       // steps at positions 4 .. len - 2
            }
            continue;
        }
        if (active == 0) break;
        if (graphs_enabled() && !prof_any_active()) {
            if (wb_status st = replay_step(sl, p.S, s)) return done(st);
        } else {
            // per-kernel timing cannot bracket kernels inside a graph: launch
            // directly, with the attention work of the active slots only (a
            // slot at position pos attends pos earlier cache rows)
            double cached = 0;
            for (int64_t q = 0; q < p.S; ++q)
                if (remaining[q] > 0) cached += chunk_len[slot_chunk[q]] - 1 - remaining[q];
            prof_set_rows((double)active / (double)p.S, cached);
            const wb_status st = run_step(sl, p.S, nullptr, s);
            prof_set_rows(1.0, -1.0);
            if (st) return done(st);
        }
        for (int64_t q = 0; q < p.S; ++q)
            if (remaining[q] > 0) --remaining[q];
    }
    std::vector<int32_t> all((size_t)p.S);
    for (int64_t q = 0; q < p.S; ++q) all[q] = (int32_t)q;
    if (wb_status st = flush(all)) return done(st);
    if (n_slots_out) *n_slots_out = (int32_t)p.S;
    done(WB_OK);
    return wb_sync_status(m, stream);
}

wb_status wb_stitch_tokens(int32_t n_req, const int64_t* req_samples, int64_t overlap_samples, const int32_t* tokens,
                           const int32_t* chunk_len, int32_t prefix_len, int32_t* out, int64_t out_cap,
                           int64_t* out_offset) {
    if (n_req < 1 || !req_samples || !tokens || !chunk_len || !out || !out_offset)
        return fail(WB_ERR_INVALID_ARG, "wb_stitch_tokens: null argument");
    if (prefix_len < 0 || prefix_len > kMaxPos) return fail(WB_ERR_SHAPE, "wb_stitch_tokens: bad prefix_len");
    std::vector<int32_t> req, valid;
    std::vector<int64_t> idx;
    if (!chunk_table(n_req, req_samples, req, idx, valid, overlap_samples))
        return fail(WB_ERR_SHAPE, "wb_stitch_tokens: bad requests or overlap");
    int64_t pos = 0;
    size_t c = 0;
    for (int32_t r = 0; r < n_req; ++r) {
        out_offset[r] = pos;
        const int64_t start = pos;
        for (; c < req.size() && req[c] == r; ++c) {
            const int32_t L = chunk_len[c];
            if (L < prefix_len || L > kMaxPos) return fail(WB_ERR_SHAPE, "wb_stitch_tokens: chunk_len out of range");
            const int32_t* row = tokens + (int64_t)c * kMaxPos + prefix_len;
            const int64_t n = L - prefix_len;
            // longest prefix of this row that repeats the end of the text so far
            int64_t k = std::min<int64_t>(pos - start, n);
            for (; k > 0; --k)
                if (std::equal(row, row + k, out + pos - k)) break;
            if (pos + (n - k) > out_cap) return fail(WB_ERR_SHAPE, "wb_stitch_tokens: out_cap too small");
            std::copy(row + k, row + n, out + pos);
            pos += n - k;
        }
    }
    out_offset[n_req] = pos;
    return WB_OK;
}

wb_status wb_quantise_e4m3(const void* x, int32_t x_is_bf16, int64_t n, uint8_t* codes, float* scale, wb_stream stream) {
    if (!x || !codes || !scale) return fail(WB_ERR_INVALID_ARG, "wb_quantise_e4m3: null argument");
    if (n < 0) return fail(WB_ERR_SHAPE, "wb_quantise_e4m3: n < 0");
    unsigned* err = lib_error_word();
    if (!err) return fail(WB_ERR_CUDA, "wb_quantise_e4m3: no device error word");
    static unsigned* bits[64] = {};
    int dev = 0;
    WB_CUDA(cudaGetDevice(&dev));
    {
        std::lock_guard<std::mutex> lk(g_err_mu);
        if (!bits[dev & 63]) WB_CUDA(cudaMalloc(&bits[dev & 63], 16));
    }
    return quant_tensor(x, x_is_bf16 != 0, n, codes, scale, bits[dev & 63], reinterpret_cast<cudaStream_t>(stream));
}

wb_status wb_quantise_e4m3_groups(const float* x, int64_t n_groups, int64_t group_elems, uint8_t* codes,
                                  float* scales, wb_stream stream) {
    if (!x || !codes || !scales) return fail(WB_ERR_INVALID_ARG, "wb_quantise_e4m3_groups: null argument");
    if (n_groups < 1 || n_groups > 65535 || group_elems < 4 || group_elems % 4 || group_elems > ((int64_t)1 << 34))
        return fail(WB_ERR_SHAPE, "wb_quantise_e4m3_groups: 1 <= n_groups <= 65535, group_elems a positive multiple of 4");
    if (!aligned16(x) || !aligned16(codes)) return fail(WB_ERR_ALIGN, "wb_quantise_e4m3_groups: x and codes 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // scales[] first accumulates each group's amax (as bit patterns)
    WB_CUDA(cudaMemsetAsync(scales, 0, sizeof(float) * (size_t)n_groups, s));
    unsigned* amax = reinterpret_cast<unsigned*>(scales);
    if (wb_status st = group_amax(x, n_groups, group_elems, amax, s)) return st;
    // codes row by row, a group split into rows of at most 8192 values
    int64_t R = group_elems;
    if (R > 8192) {
        R = 8192;
        while (group_elems % R) R -= 4;
    }
    if (wb_status st = quant_groups(x, n_groups * (group_elems / R), R, group_elems / R, amax, codes, nullptr, s))
        return st;
    return scales_from_amax(scales, n_groups, s);
}

wb_status wb_dequantise_e4m3(const uint8_t* codes, const float* scale, int64_t n, float* out, wb_stream stream) {
    if (!codes || !scale || !out) return fail(WB_ERR_INVALID_ARG, "wb_dequantise_e4m3: null argument");
    if (n < 0) return fail(WB_ERR_SHAPE, "wb_dequantise_e4m3: n < 0");
    return dequant_tensor(codes, scale, n, out, reinterpret_cast<cudaStream_t>(stream));
}

wb_status wb_gemm(const void* A, const void* Bw, int64_t M, int64_t N, int64_t K, int32_t ab_type,
                  const float* row_scale, const float* col_scale, const float* bias, int32_t gelu, void* C,
                  int32_t c_bf16, wb_stream stream) {
    if (!A || !Bw || !C) return fail(WB_ERR_INVALID_ARG, "wb_gemm: null pointer");
    if (ab_type != 0 && ab_type != 1) return fail(WB_ERR_INVALID_ARG, "wb_gemm: ab_type must be 0 or 1");
    if (ab_type == 1 && (!row_scale || !col_scale)) return fail(WB_ERR_INVALID_ARG, "wb_gemm: E4M3 needs scales");
    if (M < 1 || N < 1 || K < 1 || N % 8) return fail(WB_ERR_SHAPE, "wb_gemm: bad M/N/K");
    if (K % (ab_type ? 128 : 64)) return fail(WB_ERR_SHAPE, "wb_gemm: K must be a multiple of 64 (bf16) / 128 (E4M3)");
    unsigned* err = lib_error_word();
    if (!err) return fail(WB_ERR_CUDA, "wb_gemm: no error word");
    Lin L;
    L.a = A; L.rows = M; L.lda = K; L.w = Bw; L.N = N; L.K = K;
    FP8Weight f8w;
    if (ab_type == 1) {
        f8w.w = reinterpret_cast<uint8_t*>(const_cast<void*>(Bw));
        f8w.col_scale = const_cast<float*>(col_scale);
        L.f8 = &f8w;
        L.a_scale = row_scale;
    }
    GemmEpi e;
    e.out = C;
    e.ldo = N;
    e.out_type = c_bf16 ? OUT_BF16 : OUT_F32;
    e.bias = bias;
    e.gelu = gelu;
    return linear_impl(L, e, false, err, reinterpret_cast<cudaStream_t>(stream));
}

wb_status wb_sync_status(wb_model* m, wb_stream stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    WB_CUDA(cudaStreamSynchronize(s));
    unsigned* err = m ? m->err : lib_error_word();
    if (!err) return fail(WB_ERR_CUDA, "wb_sync_status: no error word");
    unsigned v = 0;
    WB_CUDA(cudaMemcpy(&v, err, sizeof(unsigned), cudaMemcpyDeviceToHost));
    if (v) {
        WB_CUDA(cudaMemset(err, 0, sizeof(unsigned)));
        char buf[96];
        snprintf(buf, sizeof(buf), "device error word 0x%x", v);
        return fail((v & (WB_DEVERR_TIMEOUT_TMA | WB_DEVERR_TIMEOUT_MMA | WB_DEVERR_TIMEOUT_EPI)) ? WB_ERR_TIMEOUT
                                                                                                     : WB_ERR_SHAPE,
                    buf);
    }
    return WB_OK;
}

}  // extern "C"
