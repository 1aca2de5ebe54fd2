"""Python binding of libwb.so, the B300 Whisper transcription hot path.

Argument marshalling only: every function below forwards device pointers,
sizes and the current CUDA stream to the C ABI declared in include/wb.h and
raises WBError on a negative status.  There is no Python or CPU fallback: if
the shared library is missing, the first call raises.  PyTorch supplies device
memory and streams.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwb.so")

PREC_FP32, PREC_BF16, PREC_MIXED_FP8 = 0, 1, 2
CHUNK_SAMPLES, N_FRAMES, N_CTX, MAX_POS = 480000, 3000, 1500, 448

_lib = None


class WBError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libwb status {status}: {msg}")
        self.status = status


class ModelDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_mels", "d_model", "n_heads", "d_ffn", "enc_layers",
                                               "dec_layers", "vocab", "precision", "kv_fp8")]


_VP, _I64, _I32, _SZ, _U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_uint64
_SIGS = {
    "wb_last_error": (ctypes.c_char_p, []),
    "wb_version": (ctypes.c_int, []),
    "wb_mel": (ctypes.c_int, [_VP, _I64, _I32, _VP, _VP]),
    "wb_weights_bytes": (_SZ, [ctypes.POINTER(ModelDesc)]),
    "wb_weight_offset": (ctypes.c_int, [ctypes.POINTER(ModelDesc), ctypes.c_char_p, ctypes.POINTER(_SZ),
                                        ctypes.POINTER(_I64)]),
    "wb_model_create": (ctypes.c_int, [ctypes.POINTER(ModelDesc), _VP, ctypes.POINTER(_VP)]),
    "wb_model_destroy": (ctypes.c_int, [_VP]),
    "wb_encode_workspace_size": (_SZ, [_VP, _I64]),
    "wb_encode": (ctypes.c_int, [_VP, _VP, _I64, _VP, _VP, _SZ, _VP]),
    "wb_decoder_workspace_size": (_SZ, [_VP, _I64, _VP]),
    "wb_decoder_init": (ctypes.c_int, [_VP, _I64, _VP, _VP, _VP, _VP, _SZ, _VP, ctypes.POINTER(_VP)]),
    "wb_decode_prefix": (ctypes.c_int, [_VP, _I32, _VP, _VP]),
    "wb_decode_step": (ctypes.c_int, [_VP, _I64, _VP, _VP]),
    "wb_decoder_position": (_I32, [_VP]),
    "wb_decoder_workspace_size_beams": (_SZ, [_VP, _I64, _VP, _I32]),
    "wb_decoder_init_beams": (ctypes.c_int, [_VP, _I64, _VP, _I32, _VP, _VP, _VP, _SZ, _VP, ctypes.POINTER(_VP)]),
    "wb_decode_step_beams": (ctypes.c_int, [_VP, _I64, _VP, _VP, _VP]),
    "wb_decoder_best_beams": (ctypes.c_int, [_VP, _VP, _VP, _VP]),
    "wb_decoder_beam_scores": (ctypes.c_int, [_VP, _VP, _VP]),
    "wb_decoder_destroy": (ctypes.c_int, [_VP]),
    "wb_transcribe_workspace_size": (_SZ, [_VP, _I32, _VP, _VP, _U64]),
    "wb_transcribe_batch": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _VP, _VP, _VP, _U64, _VP, _SZ, _VP, _VP]),
    "wb_plan_waves": (ctypes.c_int, [ctypes.POINTER(ModelDesc), _I32, _VP, _U64, _VP, _VP, _VP]),
    "wb_chunk_count": (_I64, [_I32, _VP, _I64]),
    "wb_transcribe_workspace_size_continuous": (_SZ, [_VP, _I32, _VP, _U64]),
    "wb_transcribe_batch_continuous": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _VP, _VP, _VP, _U64, _VP, _SZ, _VP,
                                                      _VP]),
    "wb_transcribe_workspace_size_overlap": (_SZ, [_VP, _I32, _VP, _VP, _U64, _I64]),
    "wb_transcribe_batch_overlap": (ctypes.c_int, [_VP, _VP, _VP, _VP, _I32, _I64, _VP, _VP, _VP, _U64, _VP, _SZ,
                                                   _VP, _VP]),
    "wb_stitch_tokens": (ctypes.c_int, [_I32, _VP, _I64, _VP, _VP, _I32, _VP, _I64, _VP]),
    "wb_shard_batch": (ctypes.c_int, [_I32, _VP, _VP, _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP]),
    "wb_quantise_e4m3": (ctypes.c_int, [_VP, _I32, _I64, _VP, _VP, _VP]),
    "wb_dequantise_e4m3": (ctypes.c_int, [_VP, _VP, _I64, _VP, _VP]),
    "wb_quantise_e4m3_static": (ctypes.c_int, [_VP, _I32, _I64, _VP, _VP, _VP]),
    "wb_quantise_e4m3_groups": (ctypes.c_int, [_VP, _I64, _I64, _VP, _VP, _VP]),
    "wb_sync_status": (ctypes.c_int, [_VP, _VP]),
    "wb_debug_stall_next_gemm": (ctypes.c_int, [_U64]),
    "wb_gemm": (ctypes.c_int, [_VP, _VP, _I64, _I64, _I64, _I32, _VP, _VP, _VP, _I32, _VP, _I32, _VP]),
    "wb_prof_start": (ctypes.c_int, [_I32, _I32]),
    "wb_launch_count": (_I64, []),
    "wb_prof_result": (ctypes.c_int, [_I32, ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_double)]),
    "wb_prof_stop": (ctypes.c_int, [ctypes.POINTER(_I64), ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double)]),
}

KERNEL_GEMM, KERNEL_ENC_ATTN, KERNEL_CROSS_ATTN, KERNEL_SELF_ATTN, KERNEL_MEL, KERNEL_GEMM_SMALL = 1, 2, 3, 4, 5, 6
KERNEL_NAMES = {1: "gemm_tc", 2: "flash_enc", 3: "cross_attn", 4: "self_attn", 5: "mel", 6: "gemm_tc_small"}


def lib():
    """Load libwb.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m whisper_encoder_decoder_log_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _check(st: int):
    if st != 0:
        raise WBError(st, lib().wb_last_error().decode())


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t, dtype_name: str, what: str):
    """Reject a tensor whose element type is not the one the C ABI expects."""
    if t is not None and str(t.dtype) != "torch." + dtype_name:
        raise TypeError(f"{what} must be torch.{dtype_name}, got {t.dtype}")
    if t is not None and not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")


def _host_arr(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def _room(t, n: int, what: str):
    """Reject a buffer smaller than the n elements the call will touch: the C
    ABI takes every size from the other arguments, so a short buffer would be
    read or written past its end on the device."""
    if t is not None and t.numel() < n:
        raise ValueError(f"{what} holds {t.numel()} elements; the call touches {n}")


def _batch_args(audio, ro, rs, pf, cl, tokens, overlap: int = 0, rows_per_chunk: int = 1) -> int:
    """Host-side size checks shared by the batch entry points: one offset per
    request, one decode length per chunk, a 4-token prefix, audio covering
    every request and a token row per chunk.  Returns the chunk count."""
    if ro.size != rs.size:
        raise ValueError(f"{ro.size} request offsets for {rs.size} requests")
    n_chunks = wb_chunk_count(rs, overlap)
    if cl.size != n_chunks:
        raise ValueError(f"chunk_len has {cl.size} entries; the requests make {n_chunks} chunks")
    if pf.size != 4:
        raise ValueError(f"the forced prefix has {pf.size} ids, not 4")
    if rs.size and (ro < 0).any():
        raise ValueError("negative request offset")
    _room(audio, int((ro + rs).max()) if rs.size else 0, "audio")
    _room(tokens, n_chunks * rows_per_chunk * MAX_POS, "tokens")
    return n_chunks


# ----------------------------------------------------------------- thin wrappers

def wb_version() -> int:
    return lib().wb_version()


def wb_mel(audio, n_mels: int, mel, stream=None):
    _need(audio, "float32", "audio")
    _need(mel, "float32", "mel")
    _room(audio, audio.shape[0] * CHUNK_SAMPLES, "audio")
    _room(mel, audio.shape[0] * n_mels * N_FRAMES, "mel")
    _check(lib().wb_mel(_p(audio), audio.shape[0], n_mels, _p(mel), _stream(stream)))


def wb_weights_bytes(desc: ModelDesc) -> int:
    return lib().wb_weights_bytes(ctypes.byref(desc))


def wb_weight_offset(desc: ModelDesc, name: str):
    off, n = _SZ(0), _I64(0)
    _check(lib().wb_weight_offset(ctypes.byref(desc), name.encode(), ctypes.byref(off), ctypes.byref(n)))
    return off.value, n.value


def wb_model_create(desc: ModelDesc, weights) -> int:
    h = _VP(0)
    _check(lib().wb_model_create(ctypes.byref(desc), _p(weights), ctypes.byref(h)))
    return h.value


def wb_model_destroy(model: int):
    _check(lib().wb_model_destroy(model))


def wb_encode_workspace_size(model: int, B: int) -> int:
    return lib().wb_encode_workspace_size(model, B)


def wb_encode(model: int, mel, enc, workspace, stream=None):
    _need(mel, "float32", "mel")
    if str(enc.dtype) not in ("torch.float32", "torch.bfloat16"):
        raise TypeError("enc must be float32 (fp32 model) or bfloat16")
    _check(lib().wb_encode(model, _p(mel), mel.shape[0], _p(enc), _p(workspace), workspace.numel() *
                           workspace.element_size(), _stream(stream)))


def wb_decoder_workspace_size(model: int, chunk_len) -> int:
    arr, ptr = _host_arr(chunk_len, np.int32)
    return lib().wb_decoder_workspace_size(model, arr.size, ptr)


def wb_decoder_init(model: int, chunk_len, enc, tokens, workspace, stream=None) -> int:
    arr, ptr = _host_arr(chunk_len, np.int32)
    _need(tokens, "int32", "tokens")
    _room(tokens, arr.size * MAX_POS, "tokens")
    h = _VP(0)
    _check(lib().wb_decoder_init(model, arr.size, ptr, _p(enc), _p(tokens), _p(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream), ctypes.byref(h)))
    return h.value


def wb_decode_prefix(dec: int, P: int, logits=None, stream=None):
    _need(logits, "float32", "logits")
    _check(lib().wb_decode_prefix(dec, P, _p(logits), _stream(stream)))


def wb_decode_step(dec: int, n_active: int, logits=None, stream=None):
    _need(logits, "float32", "logits")
    _check(lib().wb_decode_step(dec, n_active, _p(logits), _stream(stream)))


def wb_decoder_workspace_size_beams(model: int, chunk_len, beams: int) -> int:
    arr, ptr = _host_arr(chunk_len, np.int32)
    return lib().wb_decoder_workspace_size_beams(model, arr.size, ptr, beams)


def wb_decoder_init_beams(model: int, chunk_len, beams: int, enc, tokens, workspace, stream=None) -> int:
    arr, ptr = _host_arr(chunk_len, np.int32)
    _need(tokens, "int32", "tokens")
    _room(tokens, arr.size * max(int(beams), 1) * MAX_POS, "tokens")
    h = _VP(0)
    _check(lib().wb_decoder_init_beams(model, arr.size, ptr, beams, _p(enc), _p(tokens), _p(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream), ctypes.byref(h)))
    return h.value


def wb_decode_step_beams(dec: int, n_active: int, scores_out=None, parents_out=None, stream=None):
    _need(scores_out, "float32", "scores_out")
    _need(parents_out, "int32", "parents_out")
    _check(lib().wb_decode_step_beams(dec, n_active, _p(scores_out), _p(parents_out), _stream(stream)))


def wb_decoder_best_beams(dec: int, out_tokens, out_scores=None, stream=None):
    _need(out_tokens, "int32", "out_tokens")
    _need(out_scores, "float32", "out_scores")
    _check(lib().wb_decoder_best_beams(dec, _p(out_tokens), _p(out_scores), _stream(stream)))


def wb_decoder_beam_scores(dec: int, out, stream=None):
    _need(out, "float32", "out")
    _check(lib().wb_decoder_beam_scores(dec, _p(out), _stream(stream)))


def wb_decoder_position(dec: int) -> int:
    return lib().wb_decoder_position(dec)


def wb_decoder_destroy(dec: int):
    _check(lib().wb_decoder_destroy(dec))


def wb_transcribe_workspace_size(model: int, req_samples, chunk_len, budget: int) -> int:
    rs, rsp = _host_arr(req_samples, np.int64)
    cl, clp = _host_arr(chunk_len, np.int32)
    return lib().wb_transcribe_workspace_size(model, rs.size, rsp, clp, budget)


def wb_transcribe_batch(model: int, audio, req_offset, req_samples, prefix, chunk_len, tokens, budget: int,
                        workspace, stream=None) -> int:
    ro, rop = _host_arr(req_offset, np.int64)
    rs, rsp = _host_arr(req_samples, np.int64)
    pf, pfp = _host_arr(prefix, np.int32)
    cl, clp = _host_arr(chunk_len, np.int32)
    _need(audio, "float32", "audio")
    _need(tokens, "int32", "tokens")
    _batch_args(audio, ro, rs, pf, cl, tokens)
    nw = _I32(0)
    _check(lib().wb_transcribe_batch(model, _p(audio), rop, rsp, rs.size, pfp, clp, _p(tokens), budget,
                                     _p(workspace), workspace.numel() * workspace.element_size(),
                                     ctypes.addressof(nw), _stream(stream)))
    return nw.value


def wb_transcribe_workspace_size_continuous(model: int, req_samples, budget: int) -> int:
    rs, rsp = _host_arr(req_samples, np.int64)
    return lib().wb_transcribe_workspace_size_continuous(model, rs.size, rsp, budget)


def wb_transcribe_batch_continuous(model: int, audio, req_offset, req_samples, prefix, chunk_len, tokens, budget: int,
                                   workspace, stream=None) -> int:
    """Transcribe with continuous batching; returns the number of slots."""
    ro, rop = _host_arr(req_offset, np.int64)
    rs, rsp = _host_arr(req_samples, np.int64)
    pf, pfp = _host_arr(prefix, np.int32)
    cl, clp = _host_arr(chunk_len, np.int32)
    _need(audio, "float32", "audio")
    _need(tokens, "int32", "tokens")
    _batch_args(audio, ro, rs, pf, cl, tokens)
    ns = _I32(0)
    _check(lib().wb_transcribe_batch_continuous(model, _p(audio), rop, rsp, rs.size, pfp, clp, _p(tokens), budget,
                                                _p(workspace), workspace.numel() * workspace.element_size(),
                                                ctypes.addressof(ns), _stream(stream)))
    return ns.value


def wb_chunk_count(req_samples, overlap: int = 0) -> int:
    rs, rsp = _host_arr(req_samples, np.int64)
    n = lib().wb_chunk_count(rs.size, rsp, overlap)
    if n < 0:
        raise WBError(-2, "bad requests or overlap")
    return n


def wb_transcribe_workspace_size_overlap(model: int, req_samples, chunk_len, budget: int, overlap: int) -> int:
    rs, rsp = _host_arr(req_samples, np.int64)
    cl, clp = _host_arr(chunk_len, np.int32)
    return lib().wb_transcribe_workspace_size_overlap(model, rs.size, rsp, clp, budget, overlap)


def wb_transcribe_batch_overlap(model: int, audio, req_offset, req_samples, overlap: int, prefix, chunk_len, tokens,
                                budget: int, workspace, stream=None) -> int:
    ro, rop = _host_arr(req_offset, np.int64)
    rs, rsp = _host_arr(req_samples, np.int64)
    pf, pfp = _host_arr(prefix, np.int32)
    cl, clp = _host_arr(chunk_len, np.int32)
    _need(audio, "float32", "audio")
    _need(tokens, "int32", "tokens")
    _batch_args(audio, ro, rs, pf, cl, tokens, overlap)
    nw = _I32(0)
    _check(lib().wb_transcribe_batch_overlap(model, _p(audio), rop, rsp, rs.size, overlap, pfp, clp, _p(tokens), budget,
                                             _p(workspace), workspace.numel() * workspace.element_size(),
                                             ctypes.addressof(nw), _stream(stream)))
    return nw.value


def wb_stitch_tokens(req_samples, overlap: int, tokens, chunk_len, prefix_len: int = 4):
    """Per-request transcripts (list of int32 arrays) from host token rows [n_chunks, 448]."""
    rs, rsp = _host_arr(req_samples, np.int64)
    tk, tkp = _host_arr(tokens, np.int32)
    cl, clp = _host_arr(chunk_len, np.int32)
    n_chunks = wb_chunk_count(rs, overlap)
    if cl.size != n_chunks or tk.size < n_chunks * MAX_POS:
        raise ValueError(f"{n_chunks} chunks need {n_chunks} decode lengths and [{n_chunks}, 448] tokens")
    cap = int(np.maximum(cl - prefix_len, 0).sum())
    out = np.zeros(max(cap, 1), np.int32)
    off = np.zeros(rs.size + 1, np.int64)
    _check(lib().wb_stitch_tokens(rs.size, rsp, overlap, tkp, clp, prefix_len, out.ctypes.data, cap, off.ctypes.data))
    return [out[off[r]:off[r + 1]].copy() for r in range(rs.size)]


def wb_plan_waves(desc: ModelDesc, chunk_len, budget: int):
    cl, clp = _host_arr(chunk_len, np.int32)
    wave = np.zeros(cl.size, np.int32)
    order = np.zeros(cl.size, np.int32)
    nw = _I32(0)
    _check(lib().wb_plan_waves(ctypes.byref(desc), cl.size, clp, budget, wave.ctypes.data, order.ctypes.data,
                               ctypes.addressof(nw)))
    return wave, order, nw.value


def wb_shard_batch(req_offset, req_samples, chunk_len, world: int, rank: int):
    """This rank's share of one batch: (req_offset, req_samples, chunk_first,
    chunk_count), the requests cut at chunk boundaries (host only)."""
    ro, rop = _host_arr(req_offset, np.int64)
    rs, rsp = _host_arr(req_samples, np.int64)
    cl, clp = _host_arr(chunk_len, np.int32)
    if ro.size != rs.size or cl.size != wb_chunk_count(rs):
        raise ValueError("one offset per request and one decode length per chunk are needed")
    oo = np.zeros(rs.size, np.int64)
    os_ = np.zeros(rs.size, np.int64)
    nr, c0, cn = _I32(0), _I32(0), _I32(0)
    _check(lib().wb_shard_batch(rs.size, rop, rsp, clp, world, rank, oo.ctypes.data, os_.ctypes.data,
                                ctypes.addressof(nr), ctypes.addressof(c0), ctypes.addressof(cn)))
    return oo[:nr.value].copy(), os_[:nr.value].copy(), c0.value, cn.value


def _quant_args(x, codes, scale, n_scales: int = 1):
    if str(x.dtype) not in ("torch.float32", "torch.bfloat16"):
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    _need(x, str(x.dtype)[6:], "x")
    _need(codes, "uint8", "codes")
    _need(scale, "float32", "scale")
    _room(codes, x.numel(), "codes")
    _room(scale, n_scales, "scale")


def wb_quantise_e4m3(x, codes, scale, stream=None):
    import torch
    _quant_args(x, codes, scale)
    _check(lib().wb_quantise_e4m3(_p(x), 1 if x.dtype == torch.bfloat16 else 0, x.numel(), _p(codes), _p(scale),
                                  _stream(stream)))


def wb_quantise_e4m3_static(x, codes, scale, stream=None):
    """wb_quantise_e4m3 without any device allocation (n <= 2^26)."""
    import torch
    _quant_args(x, codes, scale)
    _check(lib().wb_quantise_e4m3_static(_p(x), 1 if x.dtype == torch.bfloat16 else 0, x.numel(), _p(codes),
                                         _p(scale), _stream(stream)))


def wb_quantise_e4m3_groups(x, n_groups: int, codes, scales, stream=None):
    """One E4M3 scale per group of x.numel() // n_groups consecutive fp32 values."""
    _need(x, "float32", "x")
    _need(codes, "uint8", "codes")
    _need(scales, "float32", "scales")
    if n_groups < 1 or x.numel() % n_groups:
        raise ValueError("x.numel() must be a multiple of n_groups")
    _room(codes, x.numel(), "codes")
    _room(scales, n_groups, "scales")
    _check(lib().wb_quantise_e4m3_groups(_p(x), n_groups, x.numel() // n_groups, _p(codes), _p(scales),
                                         _stream(stream)))


def wb_dequantise_e4m3(codes, scale, out, stream=None):
    _need(codes, "uint8", "codes")
    _need(scale, "float32", "scale")
    _need(out, "float32", "out")
    _room(scale, 1, "scale")
    _room(out, codes.numel(), "out")
    _check(lib().wb_dequantise_e4m3(_p(codes), _p(scale), codes.numel(), _p(out), _stream(stream)))


def wb_gemm(A, B, C, bias=None, gelu=False, row_scale=None, col_scale=None, stream=None):
    import torch
    fp8 = A.dtype == torch.uint8
    if A.dtype not in (torch.bfloat16, torch.uint8) or B.dtype != A.dtype:
        raise TypeError(f"A and B must both be bfloat16 or both E4M3 codes (uint8), got {A.dtype} and {B.dtype}")
    if C.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"C must be float32 or bfloat16, got {C.dtype}")
    for t, what in ((A, "A"), (B, "B"), (C, "C"), (bias, "bias"), (row_scale, "row_scale"), (col_scale, "col_scale")):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{what} must be contiguous")
    M, K = A.shape
    N = B.shape[0]
    if B.dim() != 2 or B.shape[1] != K:
        raise ValueError(f"B must be [N, {K}], got {tuple(B.shape)}")
    _room(C, M * N, "C")
    for t, n, what in ((bias, N, "bias"), (row_scale, M, "row_scale"), (col_scale, N, "col_scale")):
        _need(t, "float32", what)
        _room(t, n, what)
    _check(lib().wb_gemm(_p(A), _p(B), M, N, K, 1 if fp8 else 0, _p(row_scale), _p(col_scale), _p(bias),
                         1 if gelu else 0, _p(C), 1 if C.dtype == torch.bfloat16 else 0, _stream(stream)))


def wb_launch_count() -> int:
    return lib().wb_launch_count()


def wb_prof_start(kind: int, max_launches: int = 1 << 16):
    _check(lib().wb_prof_start(kind, max_launches))


def wb_prof_stop():
    n, ms, u = _I64(0), ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().wb_prof_stop(ctypes.byref(n), ctypes.byref(ms), ctypes.byref(u)))
    return n.value, ms.value, u.value


def wb_prof_result(kind: int):
    n, ms, u = _I64(0), ctypes.c_double(0), ctypes.c_double(0)
    _check(lib().wb_prof_result(kind, ctypes.byref(n), ctypes.byref(ms), ctypes.byref(u)))
    return n.value, ms.value, u.value


def wb_sync_status(model: Optional[int] = None, stream=None):
    _check(lib().wb_sync_status(model, _stream(stream)))


def wb_debug_stall_next_gemm(limit_ns: int):
    """Make the next tensor-core GEMM give up after a bounded wait (test hook)."""
    _check(lib().wb_debug_stall_next_gemm(limit_ns))


# ----------------------------------------------------------------- marshalling helpers

KV_NONE, KV_FP8_SELF, KV_FP8_CROSS = 0, 1, 2


def make_desc(dims, precision: int, kv_fp8) -> ModelDesc:
    """kv_fp8: False/True (E4M3 self-attention cache) or one of KV_* (KV_FP8_CROSS
    also stores the cross-attention K/V in E4M3)."""
    kv = int(kv_fp8) if not isinstance(kv_fp8, bool) else (KV_FP8_SELF if kv_fp8 else KV_NONE)
    return ModelDesc(dims.n_mels, dims.d_model, dims.n_heads, dims.d_ffn, dims.enc_layers, dims.dec_layers,
                     dims.vocab, precision, kv)


def pack_weights(desc: ModelDesc, tensors: Dict[str, np.ndarray], device="cuda"):
    """Copy named tensors into one device buffer at the offsets libwb reports.

    Matrices are stored as bf16 (values must already be bf16-exact) unless the
    model is fp32; vectors as fp32.  Returns a uint8 CUDA tensor.
    """
    import torch
    total = wb_weights_bytes(desc)
    if total == 0:
        raise WBError(-1, "invalid model descriptor")
    host = torch.zeros(total, dtype=torch.uint8, pin_memory=torch.cuda.is_available())
    hnp = host.numpy()
    bf = desc.precision != PREC_FP32
    for name, arr in tensors.items():
        off, n = wb_weight_offset(desc, name)
        a = np.ascontiguousarray(arr, dtype=np.float32).reshape(-1)
        if a.size != n:
            raise ValueError(f"{name}: {a.size} elements, layout expects {n}")
        is_matrix = name.endswith(".w") or name in ("dec.tok", "dec.pos")
        if bf and is_matrix:
            bits = (a.view(np.uint32) >> 16).astype(np.uint16)
            hnp[off:off + 2 * n] = bits.view(np.uint8)
        else:
            hnp[off:off + 4 * n] = a.view(np.uint8)
    return host.to(device, non_blocking=True)
