"""Benchmark of the Whisper transcription hot path on B300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c5] [--impl ours|reference]

One step is one pass of the whole hot path over one batch of seeded synthetic
audio, through the library's public C ABI.  Workloads (random-init weights of
the named shapes; synthetic audio standing in for the long-form recordings the
pages measure on):

  c1  tiny fp32: 1 chunk, mel + encoder + 32 teacher-forced decoder tokens
  c2  mel front end: 64 chunks of 30 s, 128 mels
  c3  large-v3 encoder, bf16: 16 chunks (mel + encoder)
  c4  large-v3-turbo transcription: one 16-min recording = 32 chunks,
      mel, encoder, cross-K/V, 4-token forced prefix + 224 greedy tokens with
      the E4M3 self-attention cache
  c5  large-v3 mixed serving batch (default, the largest workload and the one
      that runs every step of the path): 48 requests of 2-15 min, FP8 QKV/FFN
      GEMMs (one E4M3 scale per chunk and GEMM input), E4M3 cache, 32-layer
      decoder, decode lengths 64-448, waves within 180 GB
  c5x c5 with the cross-attention K/V stored in E4M3 as well

The metric is RTFx = audio seconds processed / wall seconds.  `value` is the
device-resident throughput (audio already in HBM); `e2e` repeats the same work
through the same C-ABI call with the audio copied from pinned host memory and
the tokens copied back inside each timed step.  With N GPUs the batch grows
with N (N recordings for c4, 48 N requests for c5) and is split across the
GPUs by contiguous chunk ranges (wb_shard_batch); every GPU transcribes its
share with no collective on the data path (weak scaling).  `--impl reference`
times the CPU oracle instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import LARGE_V3, TINY, TURBO  # noqa: E402

AUDIO_S_PER_CHUNK = 30.0
CHUNK = 480000
L2_BYTES = 126 * 2 ** 20
KERNEL_NAMES = {1: "gemm_tc", 2: "flash_enc", 3: "cross_attn", 4: "self_attn", 5: "mel", 6: "gemm_tc_small"}
KIND = {v: k for k, v in KERNEL_NAMES.items()}
PREC_FP32, PREC_BF16, PREC_MIXED_FP8 = 0, 1, 2
KV_FP8_SELF, KV_FP8_CROSS = 1, 2


# ----------------------------------------------------------------- workloads

class Workload:
    name = ""
    dims = None
    precision = None
    kv_fp8 = False
    audio_s = 0.0
    bound_kernel = None   # dominant kernel kind for the roofline object

    def describe(self) -> dict:
        return {"workload": self.name}


def _local_requests(g_offsets, g_samples, offs, samples, gen):
    """Audio of a rank's (cut) requests in a buffer of its own: the global
    request each piece belongs to is generated (gen(r)) and the piece copied;
    returns (audio, local offsets)."""
    audio = np.empty(int(np.sum(samples)), np.float32)
    local = np.zeros(len(offs), np.int64)
    pos, cache = 0, {}
    for i, (o, s) in enumerate(zip(offs, samples)):
        r = int(np.searchsorted(g_offsets, o, side="right") - 1)
        if r not in cache:
            cache = {r: gen(r)}
        a = cache[r]
        start = int(o - g_offsets[r])
        audio[pos:pos + s] = a[start:start + s]
        local[i] = pos
        pos += int(s)
    return audio, local


def make_workload(cfg: str, seed: int, world: int = 1, rank: int = 0, with_audio: bool = True):
    if cfg == "c1":
        w = Workload()
        w.name = "tiny-fp32 1x30s chunk, mel+encoder+32 teacher-forced tokens"
        w.dims, w.precision, w.kv_fp8 = TINY, PREC_FP32, False
        w.audio = synth.batch_audio("sine", 1, seed + rank) if with_audio else None
        w.tokens = synth.random_tokens(seed + rank, (1, 32), TINY.vocab)
        w.audio_s = 30.0
        w.kind = "teacher"
        w.bound_kernel = KIND["flash_enc"]
    elif cfg == "c2":
        w = Workload()
        w.name = "mel 64x30s chunks, 128 mels"
        w.dims, w.precision, w.kv_fp8 = LARGE_V3, None, False
        w.audio = synth.batch_audio("pink", 64, seed + rank) if with_audio else None
        w.audio_s = 64 * 30.0
        w.kind = "mel"
        w.bound_kernel = KIND["mel"]
    elif cfg == "c3":
        w = Workload()
        w.name = "large-v3 encoder bf16, 16x30s chunks"
        w.dims = synth.ModelDims("large-v3-enc", 128, 1280, 20, 5120, 32, 0, 51866)
        w.precision, w.kv_fp8 = PREC_BF16, False
        w.audio = synth.batch_audio("sine", 16, seed + rank) if with_audio else None
        w.audio_s = 16 * 30.0
        w.kind = "encode"
        w.bound_kernel = KIND["gemm_tc"]
    elif cfg in ("c4", "c4o", "c4b", "c5", "c5x", "c5c"):
        w = Workload()
        w.kind = {"c4o": "overlap", "c4b": "beam", "c5c": "cont"}.get(cfg, "batch")
        w.budget = 180 * 10 ** 9
        w.overlap = 16000 if cfg == "c4o" else 0
        w.beams = 4 if cfg == "c4b" else 1
        if cfg in ("c4", "c4o", "c4b"):
            w.name = {"c4": "large-v3-turbo transcription, 16-min recording = 32x30s chunks, prefix 4 + 224 greedy "
                            "tokens",
                      "c4o": "large-v3-turbo transcription of the c4 recording in overlapping 30 s windows (1 s "
                             "shared between neighbours: 34 windows), prefix 4 + 224 greedy tokens, stitched",
                      "c4b": "large-v3-turbo, the c4 recording's 32 chunks decoded by beam search with 4 beams, "
                             "prefix 4 + 224 tokens"}[cfg]
            w.dims, w.precision, w.kv_fp8 = TURBO, PREC_BF16, True
            n = 32                                    # one 16-minute recording per GPU
            g_samples = np.full(world, n * CHUNK, np.int64)
            g_offsets = np.arange(world, dtype=np.int64) * n * CHUNK
            n_chunks = 1 + (n * CHUNK - CHUNK + (CHUNK - w.overlap) - 1) // (CHUNK - w.overlap)
            g_len = np.full(n_chunks * world, 228, np.int32)
            gen = lambda r: synth.batch_audio("sine", n, seed + r).reshape(-1)  # noqa: E731
            w.bound_kernel = KIND["gemm_tc"]
        else:
            if cfg == "c5":
                w.name = ("large-v3 mixed serving: 48 requests 2-15 min, mixed_fp8 (one E4M3 scale per chunk and "
                          "GEMM input), E4M3 KV, lengths 64-448, waves <= 180 GB")
                w.dims, w.precision, w.kv_fp8 = LARGE_V3, PREC_MIXED_FP8, True
            elif cfg == "c5c":
                w.name = ("large-v3 mixed serving as c5 by continuous batching: decode slots for <= 180 GB, "
                          "refilled as chunks finish")
                w.dims, w.precision, w.kv_fp8 = LARGE_V3, PREC_MIXED_FP8, True
            else:
                w.name = ("large-v3 mixed serving as c5, with E4M3 cross-attention K/V as well: 48 requests 2-15 min, "
                          "mixed_fp8, lengths 64-448, waves <= 180 GB")
                w.dims, w.precision, w.kv_fp8 = LARGE_V3, PREC_MIXED_FP8, KV_FP8_CROSS
            sb = synth.serving_requests(seed, n_req=48 * world, with_audio=False)
            g_offsets, g_samples, g_len = sb.req_offsets, sb.req_samples, sb.chunk_len
            gen = lambda r: synth.sine_chunk_audio(seed * 7919 + r, int(g_samples[r]))  # noqa: E731
            w.bound_kernel = KIND["cross_attn"]
        w.global_chunk_len = g_len
        if world > 1:
            import whisper_encoder_decoder_log_b300 as wb
            if w.overlap:
                raise SystemExit("overlapping windows are measured on one GPU")
            offs, samples, c0, cn = wb.wb_shard_batch(g_offsets, g_samples, g_len, world, rank)
        else:
            offs, samples, c0, cn = g_offsets, g_samples, 0, int(g_len.size)
        w.chunk_first, w.chunk_count = c0, cn
        w.chunk_len = np.ascontiguousarray(g_len[c0:c0 + cn])
        w.req_samples = np.ascontiguousarray(samples, np.int64)
        w.audio_s = float(np.sum(samples)) / 16000.0
        if with_audio:
            w.audio_flat, w.req_offsets = _local_requests(g_offsets, g_samples, offs, samples, gen)
        else:
            w.audio_flat, w.req_offsets = None, None
    else:
        raise SystemExit(f"unknown config {cfg}")
    w.cfg = cfg
    return w

# ----------------------------------------------------------------- GPU runner

class GpuRunner:
    def __init__(self, w: Workload, seed: int):
        import torch
        import whisper_encoder_decoder_log_b300 as wb
        self.torch, self.wb, self.w = torch, wb, w
        self.model = None
        self.idle = w.kind in ("batch", "overlap", "cont", "beam") and w.chunk_count == 0   # an empty share
        if w.precision is not None:
            desc = wb.make_desc(w.dims, w.precision, w.kv_fp8)
            W = synth.make_weights(w.dims, seed, bf16=w.precision != PREC_FP32)
            self.wbuf = wb.pack_weights(desc, W)
            del W
            torch.cuda.synchronize()
            self.model = wb.wb_model_create(desc, self.wbuf)
        dev = "cuda"
        self.h2d = self.d2h = 0
        if w.kind in ("batch", "overlap", "cont", "beam"):
            if self.idle:
                return
            self.audio_host = torch.from_numpy(w.audio_flat).pin_memory()
            self.audio = self.audio_host.to(dev)
            n_chunks = w.chunk_len.size
            rows = n_chunks * w.beams
            self.tokens = torch.zeros(rows, 448, dtype=torch.int32, device=dev)
            self.tokens_host = torch.empty(rows, 448, dtype=torch.int32).pin_memory()
            self.prefix = synth.forced_prefix(seed, w.dims.vocab)
            if w.kind == "cont":
                nbytes = wb.wb_transcribe_workspace_size_continuous(self.model, w.req_samples, w.budget)
            elif w.kind == "overlap":
                nbytes = wb.wb_transcribe_workspace_size_overlap(self.model, w.req_samples, w.chunk_len, w.budget,
                                                                 w.overlap)
            elif w.kind == "batch":
                nbytes = wb.wb_transcribe_workspace_size(self.model, w.req_samples, w.chunk_len, w.budget)
            else:
                # beam search through the decoder API: mel, encoder in groups of 16, K beams per chunk
                self.chunk_audio = torch.empty(n_chunks, CHUNK, device=dev)
                self.mel = torch.empty(n_chunks, w.dims.n_mels, 3000, device=dev)
                self.enc = torch.empty(n_chunks, 1500, w.dims.d_model, dtype=torch.bfloat16, device=dev)
                self.ews = torch.empty(wb.wb_encode_workspace_size(self.model, min(16, n_chunks)), dtype=torch.uint8,
                                       device=dev)
                self.best = torch.empty(n_chunks, 448, dtype=torch.int32, device=dev)
                self.best_host = torch.empty(n_chunks, 448, dtype=torch.int32).pin_memory()
                self.best_scores = torch.empty(n_chunks, device=dev)
                nbytes = wb.wb_decoder_workspace_size_beams(self.model, w.chunk_len, w.beams)
            self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            self.h2d = int(w.audio_flat.nbytes)
            self.d2h = int((self.best if w.kind == "beam" else self.tokens).numel() * 4)
        else:
            self.audio_host = torch.from_numpy(np.ascontiguousarray(w.audio)).pin_memory()
            self.audio = self.audio_host.to(dev)
            B = w.audio.shape[0]
            self.mel = torch.empty(B, w.dims.n_mels, 3000, device=dev)
            self.h2d = int(w.audio.nbytes)
            if w.kind in ("encode", "teacher"):
                act = torch.float32 if w.precision == PREC_FP32 else torch.bfloat16
                self.enc = torch.empty(B, 1500, w.dims.d_model, dtype=act, device=dev)
                self.enc_host = torch.empty(self.enc.shape, dtype=act).pin_memory()
                self.ews = torch.empty(wb.wb_encode_workspace_size(self.model, B), dtype=torch.uint8, device=dev)
            if w.kind == "teacher":
                P = w.tokens.shape[1]
                self.chunk_len = np.full(B, P + 1, np.int32)
                self.tok = torch.zeros(B, 448, dtype=torch.int32, device=dev)
                self.tok[:, :P] = torch.from_numpy(w.tokens).to(dev)
                self.logits = torch.empty(B, P, w.dims.vocab, device=dev)
                self.logits_host = torch.empty(self.logits.shape).pin_memory()
                self.dws = torch.empty(wb.wb_decoder_workspace_size(self.model, self.chunk_len), dtype=torch.uint8,
                                       device=dev)
                self.d2h = int(self.logits.numel() * 4)
            elif w.kind == "encode":
                self.d2h = int(self.enc.numel() * self.enc.element_size())
            else:
                self.mel_host = torch.empty(self.mel.shape).pin_memory()
                self.d2h = int(self.mel.numel() * 4)
        self.flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(self):
        if not self.idle:
            self.flush_buf.fill_(1.0)

    def step(self, host_io: bool = False):
        wb, w = self.wb, self.w
        if self.idle:
            return
        if w.kind in ("batch", "overlap", "cont", "beam"):
            if host_io:
                self.audio.copy_(self.audio_host, non_blocking=True)
            if w.kind == "batch":
                wb.wb_transcribe_batch(self.model, self.audio, w.req_offsets, w.req_samples, self.prefix, w.chunk_len,
                                       self.tokens, w.budget, self.ws)
            elif w.kind == "overlap":
                wb.wb_transcribe_batch_overlap(self.model, self.audio, w.req_offsets, w.req_samples, w.overlap,
                                               self.prefix, w.chunk_len, self.tokens, w.budget, self.ws)
            elif w.kind == "cont":
                wb.wb_transcribe_batch_continuous(self.model, self.audio, w.req_offsets, w.req_samples, self.prefix,
                                                  w.chunk_len, self.tokens, w.budget, self.ws)
            else:
                self._beam_step()
            if host_io:
                (self.best_host if w.kind == "beam" else self.tokens_host).copy_(
                    self.best if w.kind == "beam" else self.tokens, non_blocking=True)
            return
        if host_io:
            self.audio.copy_(self.audio_host, non_blocking=True)
        wb.wb_mel(self.audio, w.dims.n_mels, self.mel)
        if w.kind == "mel":
            if host_io:
                self.mel_host.copy_(self.mel, non_blocking=True)
            return
        wb.wb_encode(self.model, self.mel, self.enc, self.ews)
        if w.kind == "encode":
            if host_io:
                self.enc_host.copy_(self.enc, non_blocking=True)
            return
        dec = wb.wb_decoder_init(self.model, self.chunk_len, self.enc, self.tok, self.dws)
        wb.wb_decode_prefix(dec, w.tokens.shape[1], self.logits)
        wb.wb_decoder_destroy(dec)
        if host_io:
            self.logits_host.copy_(self.logits, non_blocking=True)

    def _beam_step(self):
        """Mel and encoder of the recording's chunks, then K-beam decoding of
        every chunk to its length (one chunk = consecutive 30 s of the
        recording), and the best hypothesis per chunk."""
        wb, w, torch = self.wb, self.w, self.torch
        n = w.chunk_len.size
        self.chunk_audio.copy_(self.audio.view(-1)[:n * CHUNK].view(n, CHUNK))
        wb.wb_mel(self.chunk_audio, w.dims.n_mels, self.mel)
        for i0 in range(0, n, 16):
            i1 = min(n, i0 + 16)
            wb.wb_encode(self.model, self.mel[i0:i1], self.enc[i0:i1], self.ews)
        self.tokens[:, :4] = torch.from_numpy(np.tile(self.prefix, (n * w.beams, 1))).to(self.tokens.device)
        dec = wb.wb_decoder_init_beams(self.model, w.chunk_len, w.beams, self.enc, self.tokens, self.ws)
        wb.wb_decode_prefix(dec, 4)
        L = int(w.chunk_len.max())
        for t in range(4, L - 1):
            wb.wb_decode_step_beams(dec, int((w.chunk_len > t + 1).sum()))
        wb.wb_decoder_best_beams(dec, self.best, self.best_scores)
        wb.wb_decoder_destroy(dec)

    def sync_check(self):
        self.torch.cuda.synchronize()
        if self.model is not None or self.w.kind == "mel":
            self.wb.wb_sync_status(self.model)


# ----------------------------------------------------------------- multi-rank

def _reduce(x: float, op: str) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def max_over_ranks(x: float) -> float:
    """Maximum of a per-rank float over all ranks (identity without a process
    group).  Ranks share nothing on the data path; this timing reduction is
    the only collective."""
    return _reduce(x, "max")


def sum_over_ranks(x: float) -> float:
    return _reduce(x, "sum")


def whole_job_rate(audio_s_per_rank: float, world: int, max_ms: float) -> float:
    """Audio seconds of all ranks over the slowest rank's wall seconds (equal
    shares)."""
    return audio_s_per_rank * world / (max_ms / 1000.0)


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- CPU oracle sample

class OracleSample:
    """The oracle, as it stands, timed on a bounded piece of one 30 s chunk of
    the workload and scaled to the chunk's whole work: the log-Mel and the
    conv stem in full, ``n_enc`` encoder layers (scaled to all of them), and
    ``n_dec`` decoder layers teacher-forced over two lengths (the decoder's
    cost is linear in the positions: a per-chunk part, the cross-attention
    K/V, and a per-position part), plus the output head timed on its own.
    One run takes a few seconds; RTFx = 30 s / the estimated chunk time."""

    def __init__(self, w: Workload, seed: int):
        from oracle import model as omodel
        self.w, self.om = w, omodel
        dims = w.dims
        self.audio = (synth.pink_chunk_audio(seed) if w.cfg == "c2" else synth.sine_chunk_audio(seed)).astype(
            np.float64)
        if w.cfg == "c2":
            return
        whole = w.cfg == "c1"                        # the tiny model runs in full
        self.n_enc = dims.enc_layers if whole else min(1, dims.enc_layers)
        self.n_dec = dims.dec_layers if whole else min(1, dims.dec_layers)
        self.sub = synth.ModelDims(dims.name, dims.n_mels, dims.d_model, dims.n_heads, dims.d_ffn, self.n_enc,
                                   self.n_dec, dims.vocab)
        self.W = synth.make_weights(dims, seed, bf16=w.precision != PREC_FP32, enc_layers=range(self.n_enc),
                                    dec_layers=range(self.n_dec))
        self.fp8 = w.precision == PREC_MIXED_FP8
        self.act16 = w.precision != PREC_FP32
        self.cross8 = w.kv_fp8 == KV_FP8_CROSS
        if w.kind == "teacher":
            self.L = int(w.tokens.shape[1])
        elif w.kind in ("batch", "overlap", "cont", "beam"):
            self.L = int(round(float(np.mean(w.global_chunk_len))))
        else:
            self.L = 0
        self.tokens = synth.random_tokens(seed, 64, dims.vocab)

    def threads(self) -> int:
        try:
            from threadpoolctl import threadpool_info
            return max([t.get("num_threads", 1) for t in threadpool_info()] + [1])
        except Exception:
            return os.cpu_count() or 1

    def run(self):
        """(RTFx estimate, seconds spent, description)."""
        from oracle import mel as omel
        w, om = self.w, self.om
        t0 = time.perf_counter()
        mel = omel.log_mel(self.audio, w.dims.n_mels)
        t_mel = time.perf_counter() - t0
        if w.cfg == "c2":
            return 30.0 / t_mel, t_mel, "oracle log-Mel of one 30 s chunk of the workload; RTFx = 30 s / its time"
        dims, W = w.dims, self.W
        t1 = time.perf_counter()
        h = om.conv_stem(mel, W)
        t_stem = time.perf_counter() - t1
        t1 = time.perf_counter()
        for l in range(self.n_enc):
            h = om.encoder_layer(h, W, l, dims.n_heads, self.fp8, self.act16)
        t_enc = time.perf_counter() - t1
        est = t_mel + t_stem + t_enc * dims.enc_layers / max(1, self.n_enc)
        desc = (f"oracle on one 30 s chunk: log-Mel, conv stem, {self.n_enc} of {dims.enc_layers} encoder layers "
                f"timed and scaled")
        if self.n_dec and w.kind != "encode":
            enc = om.layer_norm(h, W["enc.lnp.g"], W["enc.lnp.b"])
            if w.cfg == "c1":                         # the whole teacher-forced pass
                t1 = time.perf_counter()
                om.decode_teacher_forced(w.tokens[0], enc, W, self.sub)
                est += time.perf_counter() - t1
                desc += ", the decoder teacher-forced over all 32 tokens"
            else:
                T1, T2 = 16, 32
                tt = {}
                for T in (T1, T2):
                    t1 = time.perf_counter()
                    om.decode_teacher_forced(self.tokens[:T], enc, W, self.sub, kv_fp8=bool(w.kv_fp8), fp8=self.fp8,
                                             cross_fp8=self.cross8, act16=self.act16)
                    tt[T] = time.perf_counter() - t1
                # the output head (final LayerNorm, tied-embedding logits) on its own
                hh = np.random.default_rng(0).normal(size=(T2, dims.d_model))
                t1 = time.perf_counter()
                om.layer_norm(hh, W["dec.lnf.g"], W["dec.lnf.b"]) @ W["dec.tok"].astype(np.float64).T
                head_pos = (time.perf_counter() - t1) / T2
                per_layer = {T: max(0.0, tt[T] - head_pos * T) / self.n_dec for T in (T1, T2)}
                slope = max(0.0, per_layer[T2] - per_layer[T1]) / (T2 - T1)
                L = self.L
                K = getattr(w, "beams", 1)            # beam search: K hypotheses decoded per chunk
                est += K * (dims.dec_layers * (per_layer[T1] + slope * (L - T1)) + head_pos * L)
                desc += (f", {self.n_dec} of {dims.dec_layers} decoder layers teacher-forced over {T1} and {T2} "
                         f"positions extrapolated linearly to {L} positions and scaled, output head timed alone"
                         + (f", times {K} hypotheses" if K > 1 else ""))
        spent = time.perf_counter() - t0
        if w.kind in ("batch", "overlap", "cont", "beam"):
            # audio per chunk of the workload: partial last chunks, windows that overlap
            per_chunk = w.audio_s / max(1, w.chunk_len.size)
            return (per_chunk / est, spent,
                    desc + f"; RTFx = {per_chunk:.2f} s of audio per chunk / the estimated time of one chunk")
        return 30.0 / est, spent, desc + "; RTFx = 30 s / the estimated time of one 30 s chunk"


# ----------------------------------------------------------------- main

def reference_arm(args, metric, unit):
    """The oracle on the host cores (rank 0 only), each step one bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = make_workload(args.config, args.seed, with_audio=False)
    sampler = OracleSample(w, args.seed)
    vals, spent, desc = [], 0.0, ""
    for i in range(args.warmup + args.steps):
        v, s, desc = sampler.run()
        if i >= args.warmup:
            vals.append(v)
            spent += s
    value = float(np.mean(vals))
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * spent / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": w.describe(),
            "cpu_baseline": {"value": value, "unit": unit, "cores": sampler.threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="c5", choices=["c1", "c2", "c3", "c4", "c4o", "c4b", "c5", "c5x", "c5c"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    metric, unit = "RTFx", "audio_s/wall_s"
    if args.impl == "reference":
        return reference_arm(args, metric, unit)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    import whisper_encoder_decoder_log_b300 as wb
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    w = make_workload(args.config, args.seed, world, rank)
    run = GpuRunner(w, args.seed)
    audio_total = sum_over_ranks(w.audio_s)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    warmup = max(3, args.warmup)
    for _ in range(warmup):
        run.step()
    run.sync_check()

    # which kernel kind dominates: one step with every kind timed (launched
    # directly, since events cannot bracket single kernels inside a replayed
    # graph); this also counts each kind's launches per step
    wb.wb_prof_start(0, 1 << 20)
    run.step()
    torch.cuda.synchronize()
    wb.wb_prof_stop()
    shares, per_step = {}, {}
    for k in KERNEL_NAMES:
        n, ms, units = wb.wb_prof_result(k)
        if n:
            shares[k], per_step[k] = ms, n
    dom = max(shares, key=shares.get) if shares else w.bound_kernel

    # ---- timed region: device-resident inputs (decode steps replay CUDA graphs)
    clocks = ClockSampler(local_rank)
    barrier()
    clocks.start()
    launches0 = wb.wb_launch_count()
    times = []
    for i in range(args.steps):
        run.flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run.step()
        e1.record()
        times.append((e0, e1))
    torch.cuda.synchronize()
    launches = (wb.wb_launch_count() - launches0) // max(1, args.steps)
    barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in times] or [0.0]
    max_ms = max_over_ranks(float(np.mean(step_ms)))
    value = audio_total / (max_ms / 1000.0)

    # ---- kernel timing: one more step with every launch of the dominant kind
    # bracketed by CUDA events on its own stream (event pool sized to the step)
    n_dom_step = per_step.get(dom, 0)
    wb.wb_prof_start(dom, min(1 << 20, max(1024, 2 * n_dom_step + 64)))
    run.flush_l2()
    run.step()
    torch.cuda.synchronize()
    n_dom, ms_dom, units_dom = wb.wb_prof_stop()
    run.sync_check()

    # ---- end to end through the same C-ABI call with host buffers
    e2e_steps = min(args.steps, 5)
    barrier()
    e2e_times = []
    for i in range(e2e_steps):
        run.flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run.step(host_io=True)
        e1.record()
        e2e_times.append((e0, e1))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in e2e_times] or [0.0])))
    e2e = {"value": audio_total / (e2e_ms / 1000.0), "unit": unit, "h2d_bytes_per_step": run.h2d,
           "d2h_bytes_per_step": run.d2h, "steps": e2e_steps}

    # ---- roofline of the dominant kernel: algorithmic work per launch over
    # the mean launch duration, against the measured peak
    peaks, src = {}, "fallback"
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        src = "measured"
    except Exception:
        pass
    mean_ms = ms_dom / n_dom if n_dom else 0.0
    units_launch = units_dom / n_dom if n_dom else 0.0
    if dom in (KIND["gemm_tc"], KIND["flash_enc"]):
        achieved = units_launch / (mean_ms / 1000.0) / 1e12 if mean_ms > 0 else 0.0
        # a kernel inside a long step: the sustained bf16 rate; E4M3 GEMMs at
        # the nominal 2x of bf16
        peak = float(peaks.get("bf16_tflops_sustained", 1400.0))
        if w.precision == PREC_MIXED_FP8 and dom == KIND["gemm_tc"]:
            peak *= 2.0
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        achieved = units_launch / (mean_ms / 1000.0) / 1e9 if mean_ms > 0 else 0.0
        peak = float(peaks.get("hbm_gbs", 6400.0))
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"] if roof["peak"] else None
    # DRAM read + write bytes per launch from the committed ncu captures
    # (profiles/) of kernels unchanged since, as a ratio to the capture's
    # algorithmic bytes, applied to this launch's algorithmic bytes
    traffic_ratio = {
        # three launches over 128 chunks x 20 heads (cross_attn_decode_turbo.md)
        KIND["cross_attn"]: ((983.745e6 + 3.027e6) + (983.727e6 + 0.506e6) + (983.804e6 + 0.812e6)) / 3
                            / (128 * 20 * (2 * 1500 * 64 * 2 + 64 * 4 + 64 * 2)),
        KIND["mel"]: (126.83e6 + 62.09e6) / (64 * (480000 * 4 + 128 * 3000 * 4)),
    }
    if w.kv_fp8 == KV_FP8_CROSS or getattr(w, "beams", 1) > 1:
        # no capture of their own: the E4M3 cross-attention; beams re-reading their chunk's K/V from L2
        traffic_ratio.pop(KIND["cross_attn"])
    if w.cfg != "c2":
        # the mel capture is of the 64-chunk batch; a single chunk's output
        # stays in L2, so its DRAM bytes do not scale from that capture
        traffic_ratio.pop(KIND["mel"])
    roof["traffic"] = units_launch * traffic_ratio[dom] if (dom in traffic_ratio and roof["bound"] == "hbm") else None
    roof["traffic_unit"] = "DRAM bytes per launch"
    if roof["bound"] == "hbm" and roof["frac"] and roof["frac"] > 1.0:
        roof["note"] = ("a read-mostly stream measured against the copy (read + write) peak can exceed 1.0; "
                        "traffic / algorithmic bytes shows whether bytes are re-read")
    roof.update({"kernel": KERNEL_NAMES.get(dom, str(dom)), "launches_per_step": n_dom_step,
                 "launches_timed": n_dom, "mean_launch_ms": mean_ms, "units_per_launch": units_launch,
                 "peak_source": src + (" bf16 sustained" if roof["bound"] == "tensor" else " copy bandwidth"),
                 "kernel_ms_per_step": {KERNEL_NAMES[k]: v for k, v in shares.items()}})

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        sampler = OracleSample(w, args.seed)
        v, spent, desc = sampler.run()
        cpu = {"value": v, "unit": unit, "cores": sampler.threads(), "kind": "oracle", "sample": desc}
    dtype = {PREC_FP32: "f32", PREC_BF16: "bf16", PREC_MIXED_FP8: "bf16+e4m3"}.get(w.precision, "f32")
    cfg = w.describe()
    cfg.update({"config": args.config, "audio_s": audio_total, "audio_s_rank0": w.audio_s,
                "l2": "flushed between timed steps",
                "parallelism": (f"dp{world}: one batch split over the GPUs by chunk ranges, no collective on the "
                                f"data path" if world > 1 else "1 GPU")})
    if w.precision == PREC_MIXED_FP8:
        cfg["fp8_scales"] = ("weights: one per matrix; activations: one per (chunk, GEMM input) tensor -- the "
                             "1500-row encoder input of a chunk, the one-token decoder input of a step")
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": warmup, "ms_per_step": max_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": cfg, "roofline": roof,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "gpu_launches": int(launches)}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
