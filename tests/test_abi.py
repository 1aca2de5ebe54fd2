"""The C-ABI library loads, exports every declared symbol, and its host-only
logic (weight layout, wave plan, argument checks) behaves -- no GPU needed."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import whisper_encoder_decoder_log_b300 as wb
from oracle import plan as oplan
from synth import LARGE_V3, TINY, TURBO, decoder_tensor_specs, encoder_tensor_specs, serving_requests

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from whisper_encoder_decoder_log_b300 import build
    build.build()
    yield


def header_functions():
    text = open(os.path.join(ROOT, "include", "wb.h")).read()
    return sorted(set(re.findall(r"WB_API\s+[\w\s\*]+?\b(wb_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", wb.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (wb_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    L = ctypes.CDLL(wb.LIB_PATH)
    for n in names:
        assert getattr(L, n) is not None
    assert sorted(wb.exported_symbols()) == names


def test_version_and_error_text():
    assert wb.wb_version() == 100
    assert isinstance(wb.lib().wb_last_error(), bytes)


@pytest.mark.parametrize("dims,prec", [(TINY, wb.PREC_FP32), (LARGE_V3, wb.PREC_BF16), (TURBO, wb.PREC_MIXED_FP8)])
def test_weight_layout_is_complete_and_disjoint(dims, prec):
    desc = wb.make_desc(dims, prec, prec != wb.PREC_FP32)
    total = wb.wb_weights_bytes(desc)
    wsz = 4 if prec == wb.PREC_FP32 else 2
    spans = []
    for name, shape, kind in encoder_tensor_specs(dims) + decoder_tensor_specs(dims):
        off, n = wb.wb_weight_offset(desc, name)
        assert n == int(np.prod(shape)), name
        assert off % 16 == 0, name
        size = n * (wsz if (name.endswith(".w") or name in ("dec.tok", "dec.pos")) else 4)
        spans.append((off, off + size, name))
    spans.sort()
    for (a0, a1, na), (b0, b1, nb) in zip(spans, spans[1:]):
        assert a1 <= b0, (na, nb)
    assert spans[-1][1] <= total
    # fused operands are contiguous
    q, _ = wb.wb_weight_offset(desc, "enc.0.q.w")
    k, _ = wb.wb_weight_offset(desc, "enc.0.k.w")
    v, _ = wb.wb_weight_offset(desc, "enc.0.v.w")
    d = dims.d_model
    assert k == q + d * d * wsz and v == k + d * d * wsz
    ck0, _ = wb.wb_weight_offset(desc, "dec.0.ck.w")
    cv_last, _ = wb.wb_weight_offset(desc, f"dec.{dims.dec_layers - 1}.cv.w")
    assert cv_last == ck0 + (2 * dims.dec_layers - 1) * d * d * wsz


def test_unknown_weight_name_is_an_error():
    desc = wb.make_desc(TINY, wb.PREC_FP32, False)
    with pytest.raises(wb.WBError) as e:
        wb.wb_weight_offset(desc, "enc.99.q.w")
    assert e.value.status == -1


@pytest.mark.parametrize("kv", [1, 2])
@pytest.mark.parametrize("budget", [2 * 10**9, 50 * 10**9, 180 * 10**9])
def test_wave_plan_matches_oracle_bit_exact(budget, kv):
    sb = serving_requests(0, n_req=48, with_audio=False)
    desc = wb.make_desc(LARGE_V3, wb.PREC_MIXED_FP8, kv)
    wave, order, nw = wb.wb_plan_waves(desc, sb.chunk_len, budget)
    # float8 cross K/V (kv = 2) halve the per-chunk cross bytes
    ref = oplan.plan_waves(sb.chunk_len, LARGE_V3.d_model, LARGE_V3.dec_layers, budget, 1 if kv == 2 else 2)
    assert nw == len(ref)
    assert np.array_equal(order, np.concatenate(ref))
    for w, chunks in enumerate(ref):
        assert (wave[chunks] == w).all()


def test_wave_plan_rejects_oversize_chunk():
    desc = wb.make_desc(LARGE_V3, wb.PREC_BF16, True)
    with pytest.raises(wb.WBError) as e:
        wb.wb_plan_waves(desc, np.array([448], np.int32), 10**6)
    assert e.value.status == -2


def test_host_side_argument_checks_need_no_gpu():
    L = wb.lib()
    assert L.wb_mel(None, 1, 128, None, None) == -1
    assert L.wb_mel(16, 0, 128, 16, None) == -2
    assert L.wb_mel(16, 1, 64, 16, None) == -2
    assert L.wb_mel(8, 1, 128, 16, None) == -3
    bad = wb.ModelDesc(128, 1000, 20, 5120, 1, 1, 10, 1, 0)
    h = ctypes.c_void_p(0)
    assert L.wb_model_create(ctypes.byref(bad), 16, ctypes.byref(h)) == -1
    assert L.wb_gemm(None, None, 1, 8, 64, 0, None, None, None, 0, None, 0, None) == -1
    assert L.wb_gemm(16, 16, 1, 8, 63, 0, None, None, None, 0, 16, 0, None) == -2
    assert L.wb_decode_step(None, 1, None, None) == -1
    assert L.wb_weights_bytes(ctypes.byref(bad)) == 0
    # grouped quantiser: group count, group size and alignment are checked first
    assert L.wb_quantise_e4m3_groups(None, 1, 4, 16, 16, None) == -1
    assert L.wb_quantise_e4m3_groups(16, 0, 4, 16, 16, None) == -2
    assert L.wb_quantise_e4m3_groups(16, 1, 6, 16, 16, None) == -2
    assert L.wb_quantise_e4m3_groups(16, 65536, 4, 16, 16, None) == -2
    assert L.wb_quantise_e4m3_groups(8, 1, 4, 16, 16, None) == -3
    # the failure-detection hook rejects limits outside (0, 1 s] without arming
    assert L.wb_debug_stall_next_gemm(0) == -1
    assert L.wb_debug_stall_next_gemm(2 * 10**9) == -1
    # continuous batching: null arguments and an empty request list
    assert L.wb_transcribe_batch_continuous(None, 16, 16, 16, 1, 16, 16, 16, 1 << 30, 16, 1 << 30, None, None) == -1
    assert L.wb_transcribe_workspace_size_continuous(None, 1, None, 1 << 30) == 0


def test_negative_request_offsets_are_rejected_before_any_launch():
    """A negative request offset would make the chunk gather read before the
    audio buffer; every batch entry point refuses it on the host, before it
    touches the model (a dummy non-null handle is enough to reach the check)."""
    L = wb.lib()
    offs = np.array([0, -480000], np.int64)
    samples = np.array([480000, 480000], np.int64)
    prefix = np.zeros(4, np.int32)
    lens = np.full(2, 10, np.int32)
    nw = ctypes.c_int32(0)
    args = (16, 16, offs.ctypes.data, samples.ctypes.data, 2)
    tail = (prefix.ctypes.data, lens.ctypes.data, 16, 1 << 30, 16, 1 << 30, ctypes.addressof(nw), None)
    assert L.wb_transcribe_batch(*args, *tail) == -2
    assert b"negative request offset" in L.wb_last_error()
    assert L.wb_transcribe_batch_continuous(*args, *tail) == -2
    assert b"negative request offset" in L.wb_last_error()
    assert L.wb_transcribe_batch_overlap(*args, 16000, *tail) == -2
    assert b"negative request offset" in L.wb_last_error()


def test_kv_modes_are_validated_on_the_host():
    L = wb.lib()
    from synth import TURBO
    for prec, kv, ok in [(wb.PREC_BF16, wb.KV_NONE, True), (wb.PREC_BF16, wb.KV_FP8_SELF, True),
                         (wb.PREC_MIXED_FP8, wb.KV_FP8_CROSS, True), (wb.PREC_FP32, wb.KV_FP8_CROSS, False),
                         (wb.PREC_BF16, 3, False), (wb.PREC_BF16, -1, False)]:
        desc = wb.make_desc(TURBO, prec, kv)
        assert (L.wb_weights_bytes(ctypes.byref(desc)) > 0) == ok, (prec, kv)
    # the E4M3 cross K/V do not change the weight layout
    a = L.wb_weights_bytes(ctypes.byref(wb.make_desc(TURBO, wb.PREC_MIXED_FP8, wb.KV_FP8_SELF)))
    b = L.wb_weights_bytes(ctypes.byref(wb.make_desc(TURBO, wb.PREC_MIXED_FP8, wb.KV_FP8_CROSS)))
    assert a == b


@pytest.mark.parametrize("world", [1, 2, 3, 8, 2000])
def test_shard_batch_matches_oracle_bit_exact(world):
    sb = serving_requests(0, n_req=48, with_audio=False)
    first = oplan.shard_ranges(sb.chunk_len, world)
    seen = 0
    for rank in range(min(world, 9)):
        offs, samples, c0, cn = wb.wb_shard_batch(sb.req_offsets, sb.req_samples, sb.chunk_len, world, rank)
        assert (c0, cn) == (first[rank], first[rank + 1] - first[rank])
        ro, rs = oplan.shard_requests(sb.req_offsets, sb.req_samples, c0, c0 + cn)
        assert np.array_equal(offs, ro) and np.array_equal(samples, rs)
        seen += cn
    if world <= 9:
        assert seen == sb.chunk_len.size


def test_shard_batch_rejects_bad_rank():
    with pytest.raises(wb.WBError):
        wb.wb_shard_batch(np.zeros(1, np.int64), np.ones(1, np.int64), np.ones(1, np.int32), 2, 2)


@pytest.mark.parametrize("overlap", [0, 16000, 320000])
def test_overlap_chunk_count_and_stitching_match_oracle(overlap):
    rng = np.random.default_rng(overlap % 97)
    samples = np.array([1, 480000, 480001, 1_234_567, 5_000_000], np.int64)
    req, idx, valid = oplan.chunk_table(samples, overlap)
    assert wb.wb_chunk_count(samples, overlap) == req.size
    n = req.size
    lens = rng.integers(5, 40, size=n).astype(np.int32)
    tok = rng.integers(0, 4, size=(n, 448)).astype(np.int32)   # a small alphabet makes overlaps common
    got = wb.wb_stitch_tokens(samples, overlap, tok, lens, 4)
    for r in range(samples.size):
        rows = [tok[c, 4:lens[c]] for c in range(n) if req[c] == r]
        assert np.array_equal(got[r], oplan.stitch(rows)), r
    assert wb.lib().wb_chunk_count(1, samples.ctypes.data, 480000) == -1
