"""Oracle: conv stem, pre-LN transformer encoder, teacher-forced decoder.

[UOW] section 1: log-Mel spectrogram -> transformer encoder -> autoregressive
decoder that produces tokens one at a time.  Section 3: the encoder applies
multi-head self-attention over all time steps; the decoder applies causal
self-attention over the tokens so far and cross-attention over the encoder
output; the encoder opens with two conv1d layers over the mel channels and adds
a positional encoding.  [WB] "Direct Kernel API": encoder self-attention has no
mask, decoder self-attention a causal mask, cross-attention no mask; the
residual is fused into a LayerNorm with eps 1e-5.  [TWT] "NVIDIA Usage": greedy
decoding with a KV cache (no sampling, one beam).  [BFW] "Inference Stack":
arithmetic in bfloat16, KV cache stored as float8.  [WB] "Precision Presets":
``mixed_fp8`` runs the QKV and FFN GEMMs in FP8 and attention in 16-bit.

Readings taken where the pages are silent or contradict one another:
  * the snippet in [UOW] section 3 shows ReLU and no stride; the workloads
    checked here use GELU after both convs and stride 2 on the second, which
    halves 3000 mel frames to 1500 encoder positions;
  * GELU is the exact form x * Phi(x) = x/2 (1 + erf(x / sqrt 2));
  * LayerNorm: (x - mean) / sqrt(biased var + 1e-5) * gain + shift;
  * every projection has a bias; attention is softmax(Q K^T / sqrt(64)) V per
    head of width 64, heads being consecutive 64-column slices;
  * encoder positions: sinusoids [sin(s tau_i) | cos(s tau_i)],
    tau_i = exp(-i ln(10000) / (d/2 - 1)), i < d/2, added after the stem;
  * the decoder input is token embedding + a learned position row (448 rows);
    the output projection is tied to the token embedding and has no bias; a
    final LayerNorm precedes it; the encoder ends with its own LayerNorm;
  * greedy choice = lowest index among the maximal logits; no token is
    suppressed and decoding runs to the requested length (no end token);
  * beam search (the beam size of [TWT] / [BFW]): hypotheses ranked by the
    sum of their tokens' log-softmax probabilities, ties to the lower beam
    then the lower token id, no length penalty (see beam_search);
  * FP8 GEMMs (``mixed_fp8``): every E4M3 operand is a tensor with one scale
    amax / 448 ([WB] "Direct Kernel API": ``quantise_e4m3(x) -> (fp8,
    scale)``, one scale per call).  Weights: one scale per weight matrix.
    Activations: one scale per (chunk, GEMM input) -- in the encoder the
    1500 x K input one chunk feeds a GEMM; in the decoder the one-token input
    a decode step feeds per chunk, so a teacher-forced pass quantises each
    position as its own step would (the forced prefix counts as one step per
    token) and incremental decoding equals the full pass.  Scales are per
    chunk, never per batch, so a chunk's result does not depend on what it is
    batched with.  The product of the two scales multiplies the exact product
    of the decoded codes;
  * 16-bit storage ([BFW] "Inference Stack": the arithmetic is bfloat16;
    [WB] "Precision Presets": mixed_fp8 keeps attention in 16 bits): with
    ``act16`` the tensors the method holds in bf16 between its steps are
    rounded to bf16 (nearest, ties to even) where it holds them -- the
    encoder's attention operands Q, K, V and its attention output, the
    encoder states handed to the decoder, and the cross-attention K/V cache
    -- and every other value stays float64.  Under FP8 this matters: a bf16
    rounding upstream of an E4M3 quantiser moves some codes to a neighbour,
    and those moves compound through the layers;
  * FP8 self-attention cache: one scale per (layer, K or V) of each chunk,
    taken from the forced-prefix rows (oracle.e4m3.kv_scale_of); attention
    reads the dequantised cache, the current token's own row included;
  * FP8 cross-attention K/V (the float8 KV cache of [BFW] "Inference Stack"
    extended to the cross-attention, as [WB] "Precision Presets" does for
    attention under aggressive_fp8): one scale per (layer, K or V) of each
    chunk, amax / 448 over all 1500 x d values of that tensor (all of them
    are known when it is precomputed, so no headroom factor), applied to the
    fp32 projection before rounding; attention reads the dequantised values.
"""
from __future__ import annotations

import math
import weakref

import numpy as np
from scipy.special import erf

from . import e4m3

EPS = 1e-5
HEAD_DIM = 64


# ------------------------------------------------------------------ elementwise

def gelu(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def layer_norm(x, g, b, eps=EPS):
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(g, np.float64) + np.asarray(b, np.float64)


def bf16(x) -> np.ndarray:
    """Nearest bfloat16 value of each entry (8 significant bits, ties to
    even), returned as float64: inside binade [2^e, 2^(e+1)) the bf16 values
    are 2^(e-7) apart, so the nearest is rint(x / 2^(e-7)) * 2^(e-7) (rint
    rounds ties to even, the even significand)."""
    x = np.asarray(x, dtype=np.float64)
    _, ex = np.frexp(x)                        # |x| = f 2^ex, f in [0.5, 1)
    step = np.ldexp(1.0, ex - 8)
    return np.where(x == 0, x, np.rint(x / step) * step)


def sinusoids(n_ctx: int, d: int) -> np.ndarray:
    half = d // 2
    tau = np.exp(-np.arange(half, dtype=np.float64) * (math.log(10000.0) / (half - 1)))
    ang = np.arange(n_ctx, dtype=np.float64)[:, None] * tau[None, :]
    return np.concatenate([np.sin(ang), np.cos(ang)], axis=1)


# ------------------------------------------------------------------ GEMM forms

_W8_CACHE = {}


def _fp8_weight(w):
    """(scale, fp32 products w * fp32(1/scale), their E4M3 values) of one weight
    matrix, one scale amax / 448 over it; memoised per array object (the
    weights of a model are quantised once, as a deployed model would be)."""
    key = id(w)
    hit = _W8_CACHE.get(key)
    if hit is not None and hit[0]() is w:
        return hit[1]
    w32 = np.asarray(w, np.float32)
    s = e4m3.scale_of(float(np.max(np.abs(w32))) if w32.size else 0.0)
    q = (w32 * np.float32(np.float32(1.0) / s)).astype(np.float32)
    res = (s, q, e4m3.round_values(q))
    try:
        _W8_CACHE[key] = (weakref.ref(w), res)
    except TypeError:          # not weak-referenceable (a list): no memo
        pass
    return res


class Linear:
    """y = x W^T + b, optionally through E4M3 codes (``mixed_fp8``).

    ``act_scale`` says what one activation scale covers: ``"tensor"`` -- the
    whole input x (the encoder calls this once per chunk), ``"row"`` -- each
    row of x on its own (a decoder row is one decode step's input).
    """

    def __init__(self, w, b, fp8: bool = False, act_scale: str = "row"):
        if act_scale not in ("row", "tensor"):
            raise ValueError(act_scale)
        self.w = np.asarray(w, dtype=np.float64)
        self.b = np.asarray(b, dtype=np.float64)
        self.fp8 = fp8
        self.act_scale = act_scale
        if fp8:
            self.w_scale, self._w_q, self.w_deq = _fp8_weight(w)

    @property
    def w_codes(self):
        """E4M3 codes of the weights (the values w_deq holds)."""
        return e4m3.encode(self._w_q)

    def __call__(self, x):
        x = np.asarray(x, dtype=np.float64)
        if not self.fp8:
            return x @ self.w.T + self.b
        x32 = x.astype(np.float32).reshape(-1, x.shape[-1])
        if self.act_scale == "tensor":   # one scale amax / 448 over the whole input
            s_t = e4m3.scale_of(float(np.max(np.abs(x32))) if x32.size else 0.0)
            s_x = np.full(x32.shape[0], s_t, dtype=np.float32)
        else:                            # every row (one step's token) has its own
            amax = np.max(np.abs(x32), axis=-1)
            s_x = np.array([e4m3.scale_of(a) for a in amax], dtype=np.float32)
        inv = (np.float32(1.0) / s_x).astype(np.float32)
        qx = e4m3.round_values((x32 * inv[:, None]).astype(np.float32))
        acc = qx @ self.w_deq.T
        out = acc * (s_x.astype(np.float64)[:, None] * np.float64(self.w_scale))
        return out.reshape(x.shape[:-1] + (self.w.shape[0],)) + self.b


def conv1d_k3(x, w, b, stride: int):
    """y[o, s] = b[o] + sum_{c, j} w[o, c, j] x[c, stride s + j - 1], zero padded.

    x: [C, T]; w: [O, C, 3]; returns [O, T // stride].
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    C, T = x.shape
    T_out = (T + 2 - 3) // stride + 1
    xp = np.zeros((C, T + 2), dtype=np.float64)
    xp[:, 1:T + 1] = x
    y = np.zeros((w.shape[0], T_out), dtype=np.float64)
    for j in range(3):
        cols = xp[:, j: j + stride * (T_out - 1) + 1: stride]
        y += w[:, :, j] @ cols
    return y + np.asarray(b, np.float64)[:, None]


# ------------------------------------------------------------------ attention

def attention(q, k, v, causal: bool = False, q_offset: int = 0):
    """softmax(q k^T / sqrt(hd)) v for one head; q [Tq,hd], k,v [Tk,hd].

    With ``causal`` query i (absolute position q_offset + i) sees keys j <= it.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    s = q @ k.T / math.sqrt(q.shape[-1])
    if causal:
        qi = q_offset + np.arange(q.shape[0])[:, None]
        kj = np.arange(k.shape[0])[None, :]
        s = np.where(kj <= qi, s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ v


def multi_head(q, k, v, n_heads: int, causal: bool = False):
    out = np.empty((q.shape[0], n_heads * HEAD_DIM), dtype=np.float64)
    for h in range(n_heads):
        sl = slice(h * HEAD_DIM, (h + 1) * HEAD_DIM)
        out[:, sl] = attention(q[:, sl], k[:, sl], v[:, sl], causal=causal)
    return out


# ------------------------------------------------------------------ encoder

def conv_stem(mel, W):
    """[n_mels, 3000] -> [1500, d]: GELU(conv1), GELU(conv2 stride 2), + sinusoids."""
    x = gelu(conv1d_k3(mel, W["enc.conv1.w"], W["enc.conv1.b"], 1))
    x = gelu(conv1d_k3(x, W["enc.conv2.w"], W["enc.conv2.b"], 2))
    x = x.T
    return x + sinusoids(x.shape[0], x.shape[1])


def encoder_layer(h, W, l: int, n_heads: int, fp8: bool = False, act16: bool = False):
    """One pre-LN layer over one chunk's [1500, d] states; under ``mixed_fp8``
    each E4M3 GEMM input (LN1 output, LN2 output, GELU output) is one tensor
    with one scale; with ``act16`` attention reads bf16 Q, K, V and hands on a
    bf16 result."""
    p = f"enc.{l}."
    a = layer_norm(h, W[p + "ln1.g"], W[p + "ln1.b"])
    q = Linear(W[p + "q.w"], W[p + "q.b"], fp8, "tensor")(a)
    k = Linear(W[p + "k.w"], W[p + "k.b"], fp8, "tensor")(a)
    v = Linear(W[p + "v.w"], W[p + "v.b"], fp8, "tensor")(a)
    if act16:
        q, k, v = bf16(q), bf16(k), bf16(v)
    att = multi_head(q, k, v, n_heads)
    if act16:
        att = bf16(att)
    h = h + Linear(W[p + "o.w"], W[p + "o.b"])(att)
    a = layer_norm(h, W[p + "ln2.g"], W[p + "ln2.b"])
    f = gelu(Linear(W[p + "fc1.w"], W[p + "fc1.b"], fp8, "tensor")(a))
    return h + Linear(W[p + "fc2.w"], W[p + "fc2.b"], fp8, "tensor")(f)


def encode(mel, W, dims, fp8: bool = False, layers=None, act16: bool = False):
    """[n_mels, 3000] -> [1500, d] encoder states (after the final LayerNorm;
    bf16 values with ``act16``, the form the decoder receives them in)."""
    h = conv_stem(mel, W)
    for l in range(dims.enc_layers if layers is None else layers):
        h = encoder_layer(h, W, l, dims.n_heads, fp8, act16)
    out = layer_norm(h, W["enc.lnp.g"], W["enc.lnp.b"])
    return bf16(out) if act16 else out


# ------------------------------------------------------------------ decoder

def cross_kv(enc, W, l: int):
    p = f"dec.{l}."
    return (Linear(W[p + "ck.w"], W[p + "ck.b"])(enc),
            Linear(W[p + "cv.w"], W[p + "cv.b"])(enc))


def cross_kv_fp8(k, v):
    """E4M3 round trip of one chunk's cross K and V of one layer, each with its
    own per-tensor scale amax / 448 (returned with the dequantised values)."""
    out = []
    for x in (k, v):
        x32 = np.asarray(x, np.float32)
        s = e4m3.scale_of(float(np.max(np.abs(x32))))
        out.append((e4m3.dequantise(e4m3.quantise(x32, s), s), s))
    return out


def _kv_fp8(x, prefix_len: int):
    s = e4m3.kv_scale_of(np.max(np.abs(np.asarray(x[:prefix_len], np.float32))))
    return e4m3.dequantise(e4m3.quantise(x, s), s), s


def decode_teacher_forced(tokens, enc, W, dims, kv_fp8: bool = False,
                          prefix_len: int = 4, fp8: bool = False,
                          return_hidden: bool = False, cross_fp8: bool = False, act16: bool = False):
    """Logits [T, V] for a token sequence run through the decoder in one causal pass.

    Equivalent to stepping token by token with a KV cache: every position only
    sees earlier positions, and the FP8 cache scale depends on the prefix rows
    alone.  With ``act16`` the cross-attention K/V cache holds bf16 values
    (E4M3 ones with ``cross_fp8``, rounded from the float64 projection).
    Returns (logits, info) with the per-layer KV scales in ``info``.
    """
    tokens = np.asarray(tokens)
    T = tokens.shape[0]
    h = W["dec.tok"][tokens].astype(np.float64) + W["dec.pos"][:T].astype(np.float64)
    info = {"kv_scales": []}
    for l in range(dims.dec_layers):
        p = f"dec.{l}."
        a = layer_norm(h, W[p + "ln1.g"], W[p + "ln1.b"])
        q = Linear(W[p + "sq.w"], W[p + "sq.b"], fp8)(a)
        k = Linear(W[p + "sk.w"], W[p + "sk.b"], fp8)(a)
        v = Linear(W[p + "sv.w"], W[p + "sv.b"], fp8)(a)
        if kv_fp8:
            k, sk = _kv_fp8(k, prefix_len)
            v, sv = _kv_fp8(v, prefix_len)
            info["kv_scales"].append((sk, sv))
        h = h + Linear(W[p + "so.w"], W[p + "so.b"])(multi_head(q, k, v, dims.n_heads, causal=True))
        a = layer_norm(h, W[p + "ln2.g"], W[p + "ln2.b"])
        q = Linear(W[p + "cq.w"], W[p + "cq.b"])(a)
        ck, cv = cross_kv(enc, W, l)
        if cross_fp8:
            (ck, sck), (cv, scv) = cross_kv_fp8(ck, cv)
            info.setdefault("cross_scales", []).append((sck, scv))
        elif act16:
            ck, cv = bf16(ck), bf16(cv)
        h = h + Linear(W[p + "co.w"], W[p + "co.b"])(multi_head(q, ck, cv, dims.n_heads))
        a = layer_norm(h, W[p + "ln3.g"], W[p + "ln3.b"])
        f = gelu(Linear(W[p + "fc1.w"], W[p + "fc1.b"], fp8)(a))
        h = h + Linear(W[p + "fc2.w"], W[p + "fc2.b"], fp8)(f)
    hf = layer_norm(h, W["dec.lnf.g"], W["dec.lnf.b"])
    logits = hf @ W["dec.tok"].astype(np.float64).T
    if return_hidden:
        info["hidden"] = hf
    return logits, info


def greedy(logits) -> np.ndarray:
    """Lowest index of the maximum of each row."""
    return np.argmax(np.asarray(logits), axis=-1).astype(np.int32)


# ------------------------------------------------------------------ beam search

def log_softmax(x):
    """log p_v = x_v - max - log sum_u exp(x_u - max), float64."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=-1, keepdims=True)
    return x - m - np.log(np.exp(x - m).sum(axis=-1, keepdims=True))


def beam_candidates(scores, logits, beams: int):
    """One beam-search step.  ``scores`` [n] are the running sums of the live
    hypotheses' token log-probabilities, ``logits`` [n, V] their next-token
    logits.  Every continuation (b, v) scores scores[b] + log_softmax(logits[b])[v];
    the ``beams`` best continue, ranked by score, ties to the lower beam then
    the lower token id.  Returns (new scores, parent beams, tokens)."""
    lp = log_softmax(logits)
    cand = np.asarray(scores, np.float64)[:, None] + lp
    n, V = cand.shape
    b_idx = np.repeat(np.arange(n), V)
    v_idx = np.tile(np.arange(V), n)
    order = np.lexsort((v_idx, b_idx, -cand.reshape(-1)))[:beams]
    return cand.reshape(-1)[order], b_idx[order].astype(np.int32), v_idx[order].astype(np.int32)


def beam_search(prefix, length: int, beams: int, enc, W, dims, **decode_kw):
    """Beam search over one chunk ([TWT] "NVIDIA Usage": ``num_beams``; [BFW]
    "Benchmarks": a fixed beam size).  Readings: a hypothesis is scored by the
    sum of its generated tokens' log-probabilities; there is no length penalty
    and no end token, so every hypothesis reaches ``length`` positions
    (prefix included) and the answer is the best-scoring one (ties: the lower
    beam); the first step expands the forced prefix alone.  Each hypothesis's
    logits come from the teacher-forced decoder over its own tokens.
    Returns (tokens [length] of the best hypothesis, its score, the per-step
    list of (scores, parents, tokens))."""
    hyps = [list(np.asarray(prefix, np.int64))]
    scores = np.zeros(1)
    trace = []
    P = len(hyps[0])
    for t in range(P - 1, length - 1):
        logits = np.stack([decode_teacher_forced(np.array(h), enc, W, dims, prefix_len=P, **decode_kw)[0][-1]
                           for h in hyps])
        scores, parents, toks = beam_candidates(scores, logits, beams)
        hyps = [hyps[p] + [int(v)] for p, v in zip(parents, toks)]
        trace.append((scores.copy(), parents, toks))
    best = int(np.argmax(scores))          # lowest index among the maxima
    return np.array(hyps[best], np.int32), float(scores[best]), trace
