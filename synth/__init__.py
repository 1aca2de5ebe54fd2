"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This module holds no arithmetic of the transcription method itself: it only
draws audio, token ids, request lengths and random-init weights from seeded
generators, and describes the model shapes.  Both the CPU oracle (``oracle/``)
and the GPU library consume what it produces; neither side's arithmetic lives
here.

Workload recipes (all seeded through ``numpy.random.default_rng``):

* ``sine_chunk_audio``: one 30 s chunk at 16 kHz = 480000 float32 samples, the
  sum of three sines at frequencies drawn U[100, 4000] Hz with amplitude 0.2 and
  a random phase, plus N(0, 0.01) noise, clipped to [-1, 1].  This is the
  synthetic stand-in for speech used by the tiny, encoder and transcription
  workloads (the pages measure on long-form recordings that are not available
  here).
* ``pink_chunk_audio``: the mel workload's audio, a 1-pole low-pass
  y[n] = 0.95 y[n-1] + N(0, 0.1) with about 10 % of the samples zeroed in
  seeded silent spans of 0.2-1 s, clipped to [-1, 1].
* ``serving_requests``: the mixed-length serving batch -- 48 requests with
  durations U[120, 900] s, each a sine+noise recording, plus a decode length
  per 30 s chunk drawn uniformly from 64..448 token positions (prefix included).
* ``make_weights``: every matrix, conv kernel, bias and embedding is
  N(0, 0.02); LayerNorm gains are 1 + N(0, 0.02) and shifts N(0, 0.02).  Each
  tensor has its own seed derived from (seed, tensor name), so any one tensor
  can be regenerated alone.  For bf16 models every tensor is rounded to the
  nearest bf16 value (ties to even) here, so that both sides read identical
  weights.
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np

SAMPLE_RATE = 16000
CHUNK_SAMPLES = 480000          # 30 s at 16 kHz
N_FRAMES = 3000                 # mel frames per chunk
N_CTX = 1500                    # encoder positions per chunk
MAX_POS = 448                   # decoder position table size
HEAD_DIM = 64


@dataclasses.dataclass(frozen=True)
class ModelDims:
    """Shapes of one Whisper-style encoder-decoder."""
    name: str
    n_mels: int
    d_model: int
    n_heads: int
    d_ffn: int
    enc_layers: int
    dec_layers: int
    vocab: int

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_heads


TINY = ModelDims("tiny", 80, 384, 6, 1536, 4, 4, 51865)
LARGE_V3 = ModelDims("large-v3", 128, 1280, 20, 5120, 32, 32, 51866)
TURBO = ModelDims("large-v3-turbo", 128, 1280, 20, 5120, 32, 4, 51866)


def _rng(seed: int, tag: str) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed) & 0xFFFFFFFF,
                                                         zlib.crc32(tag.encode())]))


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value of each float32 (ties to even), returned as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------- audio

def sine_chunk_audio(seed: int, n_samples: int = CHUNK_SAMPLES) -> np.ndarray:
    rng = _rng(seed, "sine-audio")
    freqs = rng.uniform(100.0, 4000.0, size=3)
    phases = rng.uniform(0.0, 2 * np.pi, size=3)
    n = np.arange(n_samples, dtype=np.float64) / SAMPLE_RATE
    y = np.zeros(n_samples, dtype=np.float64)
    for f, p in zip(freqs, phases):
        y += 0.2 * np.sin(2 * np.pi * f * n + p)
    y += rng.normal(0.0, 0.01, size=n_samples)
    return np.clip(y, -1.0, 1.0).astype(np.float32)


def pink_chunk_audio(seed: int, n_samples: int = CHUNK_SAMPLES) -> np.ndarray:
    from scipy.signal import lfilter
    rng = _rng(seed, "pink-audio")
    w = rng.normal(0.0, 0.1, size=n_samples)
    y = lfilter([1.0], [1.0, -0.95], w)
    silent = 0
    target = n_samples // 10
    while silent < target:
        span = int(rng.uniform(0.2, 1.0) * SAMPLE_RATE)
        span = min(span, target - silent)
        start = int(rng.integers(0, n_samples - span + 1))
        y[start:start + span] = 0.0
        silent += span
    return np.clip(y, -1.0, 1.0).astype(np.float32)


def batch_audio(kind: str, n_chunks: int, seed: int) -> np.ndarray:
    """[n_chunks, 480000] float32; chunk i uses seed (seed*1000003 + i)."""
    fn = {"sine": sine_chunk_audio, "pink": pink_chunk_audio}[kind]
    out = np.empty((n_chunks, CHUNK_SAMPLES), dtype=np.float32)
    for i in range(n_chunks):
        out[i] = fn(seed * 1000003 + i)
    return out


def random_tokens(seed: int, shape, vocab: int) -> np.ndarray:
    return _rng(seed, "tokens").integers(0, vocab, size=shape).astype(np.int32)


def forced_prefix(seed: int, vocab: int) -> np.ndarray:
    """Four fixed seeded token ids standing in for <start><lang><task><notimestamps>."""
    return _rng(seed, "prefix").integers(0, vocab, size=4).astype(np.int32)


@dataclasses.dataclass
class ServingBatch:
    audio: np.ndarray            # float32 [total_samples], requests back to back
    req_offsets: np.ndarray      # int64 [n_req] start sample of each request
    req_samples: np.ndarray      # int64 [n_req] samples of each request
    chunk_len: np.ndarray        # int32 [n_chunks] decode length (prefix included)


def serving_requests(seed: int, n_req: int = 48, min_s: float = 120.0,
                     max_s: float = 900.0, min_len: int = 64,
                     max_len: int = 448, with_audio: bool = True) -> ServingBatch:
    rng = _rng(seed, "serving")
    durs = rng.uniform(min_s, max_s, size=n_req)
    samples = np.round(durs * SAMPLE_RATE).astype(np.int64)
    offsets = np.zeros(n_req, dtype=np.int64)
    offsets[1:] = np.cumsum(samples)[:-1]
    audio = np.empty(int(samples.sum()) if with_audio else 0, dtype=np.float32)
    for r in range(n_req if with_audio else 0):
        audio[offsets[r]:offsets[r] + samples[r]] = sine_chunk_audio(
            seed * 7919 + r, int(samples[r]))
    n_chunks = int(sum((s + CHUNK_SAMPLES - 1) // CHUNK_SAMPLES for s in samples))
    lens = rng.integers(min_len, max_len + 1, size=n_chunks).astype(np.int32)
    return ServingBatch(audio, offsets, samples, lens)


# ----------------------------------------------------------------------------- weights

def encoder_tensor_specs(m: ModelDims):
    """(name, shape, kind) for every encoder tensor; kind in {w, b, g, beta}."""
    d, f = m.d_model, m.d_ffn
    specs = [("enc.conv1.w", (d, m.n_mels, 3), "w"), ("enc.conv1.b", (d,), "b"),
             ("enc.conv2.w", (d, d, 3), "w"), ("enc.conv2.b", (d,), "b")]
    for l in range(m.enc_layers):
        p = f"enc.{l}."
        specs += [(p + "ln1.g", (d,), "g"), (p + "ln1.b", (d,), "b"),
                  (p + "q.w", (d, d), "w"), (p + "q.b", (d,), "b"),
                  (p + "k.w", (d, d), "w"), (p + "k.b", (d,), "b"),
                  (p + "v.w", (d, d), "w"), (p + "v.b", (d,), "b"),
                  (p + "o.w", (d, d), "w"), (p + "o.b", (d,), "b"),
                  (p + "ln2.g", (d,), "g"), (p + "ln2.b", (d,), "b"),
                  (p + "fc1.w", (f, d), "w"), (p + "fc1.b", (f,), "b"),
                  (p + "fc2.w", (d, f), "w"), (p + "fc2.b", (d,), "b")]
    specs += [("enc.lnp.g", (d,), "g"), ("enc.lnp.b", (d,), "b")]
    return specs


def decoder_tensor_specs(m: ModelDims):
    d, f = m.d_model, m.d_ffn
    specs = [("dec.tok", (m.vocab, d), "w"), ("dec.pos", (MAX_POS, d), "w")]
    for l in range(m.dec_layers):
        p = f"dec.{l}."
        specs += [(p + "ln1.g", (d,), "g"), (p + "ln1.b", (d,), "b")]
        for nm in ("sq", "sk", "sv", "so"):
            specs += [(p + nm + ".w", (d, d), "w"), (p + nm + ".b", (d,), "b")]
        specs += [(p + "ln2.g", (d,), "g"), (p + "ln2.b", (d,), "b")]
        for nm in ("cq", "ck", "cv", "co"):
            specs += [(p + nm + ".w", (d, d), "w"), (p + nm + ".b", (d,), "b")]
        specs += [(p + "ln3.g", (d,), "g"), (p + "ln3.b", (d,), "b"),
                  (p + "fc1.w", (f, d), "w"), (p + "fc1.b", (f,), "b"),
                  (p + "fc2.w", (d, f), "w"), (p + "fc2.b", (d,), "b")]
    specs += [("dec.lnf.g", (d,), "g"), ("dec.lnf.b", (d,), "b")]
    return specs


def make_tensor(seed: int, name: str, shape, kind: str, bf16: bool) -> np.ndarray:
    rng = _rng(seed, "w:" + name)
    x = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(0.02)
    if kind == "g":
        x = x + np.float32(1.0)
    x = x.astype(np.float32)
    return round_to_bf16(x) if bf16 else x


def make_weights(m: ModelDims, seed: int, bf16: bool, encoder: bool = True,
                 decoder: bool = True, enc_layers=None, dec_layers=None) -> dict:
    """Dict name -> float32 array (bf16-exact when ``bf16``).

    ``enc_layers`` / ``dec_layers`` optionally restrict which layer indices are
    generated (the others are simply absent), for oracle runs on a subset.
    """
    out = {}
    specs = []
    if encoder:
        specs += encoder_tensor_specs(m)
    if decoder:
        specs += decoder_tensor_specs(m)
    for name, shape, kind in specs:
        parts = name.split(".")
        if parts[1].isdigit():
            l = int(parts[1])
            sel = enc_layers if parts[0] == "enc" else dec_layers
            if sel is not None and l not in sel:
                continue
        out[name] = make_tensor(seed, name, shape, kind, bf16)
    return out
