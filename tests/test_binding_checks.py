"""The Python binding rejects buffers too small for the sizes the C ABI takes
from its other arguments, and mismatched element types, before anything is
launched: a short token matrix or output would otherwise be written past its
end on the device.  CPU tensors stand in for device buffers (the checks run
first, so no GPU is needed)."""
import numpy as np
import pytest
import torch

import whisper_encoder_decoder_log_b300 as wb


@pytest.fixture(scope="module", autouse=True)
def built():
    from whisper_encoder_decoder_log_b300 import build
    build.build()
    yield


def _batch(samples=(800000, 100000)):
    samples = np.array(samples, np.int64)
    offs = np.zeros_like(samples)
    offs[1:] = np.cumsum(samples)[:-1]
    n = wb.wb_chunk_count(samples)
    audio = torch.zeros(int(samples.sum()), dtype=torch.float32)
    tokens = torch.zeros(n, 448, dtype=torch.int32)
    lens = np.full(n, 10, np.int32)
    prefix = np.arange(4, dtype=np.int32)
    return audio, offs, samples, prefix, lens, tokens


@pytest.mark.parametrize("fn", ["wb_transcribe_batch", "wb_transcribe_batch_continuous"])
def test_batch_entry_points_check_sizes_on_the_host(fn):
    call = getattr(wb, fn)
    audio, offs, samples, prefix, lens, tokens = _batch()
    ws = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="tokens"):
        call(0, audio, offs, samples, prefix, lens, tokens[:-1], 1 << 30, ws)
    with pytest.raises(ValueError, match="audio"):
        call(0, audio[:-1], offs, samples, prefix, lens, tokens, 1 << 30, ws)
    with pytest.raises(ValueError, match="chunk_len"):
        call(0, audio, offs, samples, prefix, lens[:-1], tokens, 1 << 30, ws)
    with pytest.raises(ValueError, match="offsets"):
        call(0, audio, offs[:1], samples, prefix, lens, tokens, 1 << 30, ws)
    with pytest.raises(ValueError, match="prefix"):
        call(0, audio, offs, samples, prefix[:3], lens, tokens, 1 << 30, ws)
    with pytest.raises(wb.WBError):          # an empty request: rejected by the chunk count
        call(0, audio, offs, np.array([800000, 0], np.int64), prefix, lens, tokens, 1 << 30, ws)


def test_overlap_entry_point_counts_overlapping_chunks():
    audio, offs, samples, prefix, _, _ = _batch((950000, 100000))
    overlap = 160000
    n = wb.wb_chunk_count(samples, overlap)
    assert n > wb.wb_chunk_count(samples)
    lens = np.full(n, 10, np.int32)
    tokens = torch.zeros(n, 448, dtype=torch.int32)
    ws = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="chunk_len"):      # one length per non-overlapping chunk is too few
        wb.wb_transcribe_batch_overlap(0, audio, offs, samples, overlap, prefix, lens[:wb.wb_chunk_count(samples)],
                                       tokens, 1 << 30, ws)
    with pytest.raises(ValueError, match="tokens"):
        wb.wb_transcribe_batch_overlap(0, audio, offs, samples, overlap, prefix, lens, tokens[:-1], 1 << 30, ws)


def test_mel_and_decoder_buffers_are_checked():
    audio = torch.zeros(2, 480000)
    with pytest.raises(ValueError, match="mel"):
        wb.wb_mel(audio, 128, torch.zeros(2, 128, 2999))
    with pytest.raises(ValueError, match="audio"):           # one flat row read as 480000 chunks
        wb.wb_mel(torch.zeros(480000), 128, torch.zeros(1, 128, 3000))
    lens = np.array([10, 12], np.int32)
    with pytest.raises(ValueError, match="tokens"):
        wb.wb_decoder_init(0, lens, None, torch.zeros(1, 448, dtype=torch.int32), torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="tokens"):           # beams x chunks token rows
        wb.wb_decoder_init_beams(0, lens, 4, None, torch.zeros(7, 448, dtype=torch.int32),
                                 torch.zeros(16, dtype=torch.uint8))


def test_gemm_shapes_and_types_are_checked():
    M, N, K = 8, 16, 32
    A = torch.zeros(M, K, dtype=torch.bfloat16)
    B = torch.zeros(N, K, dtype=torch.bfloat16)
    C = torch.zeros(M, N)
    with pytest.raises(ValueError, match="C"):
        wb.wb_gemm(A, B, C[:-1])
    with pytest.raises(ValueError, match="B must be"):
        wb.wb_gemm(A, torch.zeros(N, K + 8, dtype=torch.bfloat16), C)
    with pytest.raises(TypeError):                           # operands of two types
        wb.wb_gemm(A, B.to(torch.float16), C)
    with pytest.raises(TypeError):                           # E4M3 codes against bf16 weights
        wb.wb_gemm(torch.zeros(M, K, dtype=torch.uint8), B, C)
    with pytest.raises(TypeError):                           # a 2-byte output the kernel would write as fp32
        wb.wb_gemm(A, B, C.to(torch.float16))
    with pytest.raises(ValueError, match="bias"):
        wb.wb_gemm(A, B, C, bias=torch.zeros(N - 1))
    with pytest.raises(TypeError):
        wb.wb_gemm(A, B, C, bias=torch.zeros(N, dtype=torch.float64))
    qa, qb = torch.zeros(M, K, dtype=torch.uint8), torch.zeros(N, K, dtype=torch.uint8)
    with pytest.raises(ValueError, match="row_scale"):
        wb.wb_gemm(qa, qb, C, row_scale=torch.ones(M - 1), col_scale=torch.ones(N))
    with pytest.raises(ValueError, match="col_scale"):
        wb.wb_gemm(qa, qb, C, row_scale=torch.ones(M), col_scale=torch.ones(1))


def test_quantiser_buffers_are_checked():
    x = torch.zeros(100)
    with pytest.raises(ValueError, match="codes"):
        wb.wb_quantise_e4m3(x, torch.zeros(99, dtype=torch.uint8), torch.zeros(1))
    with pytest.raises(ValueError, match="scale"):
        wb.wb_quantise_e4m3(x, torch.zeros(100, dtype=torch.uint8), torch.zeros(0))
    with pytest.raises(TypeError):                           # fp16 input would be read as fp32
        wb.wb_quantise_e4m3(x.half(), torch.zeros(100, dtype=torch.uint8), torch.zeros(1))
    with pytest.raises(ValueError, match="codes"):
        wb.wb_quantise_e4m3_static(x, torch.zeros(50, dtype=torch.uint8), torch.zeros(1))
    with pytest.raises(ValueError, match="scales"):
        wb.wb_quantise_e4m3_groups(x, 4, torch.zeros(100, dtype=torch.uint8), torch.zeros(3))
    with pytest.raises(ValueError):
        wb.wb_quantise_e4m3_groups(x, 0, torch.zeros(100, dtype=torch.uint8), torch.zeros(1))
    with pytest.raises(ValueError, match="out"):
        wb.wb_dequantise_e4m3(torch.zeros(100, dtype=torch.uint8), torch.ones(1), torch.zeros(99))


def test_host_bookkeeping_checks_its_arrays():
    samples = np.array([800000, 100000], np.int64)
    offs = np.array([0, 800000], np.int64)
    n = wb.wb_chunk_count(samples)
    with pytest.raises(ValueError):
        wb.wb_shard_batch(offs, samples, np.full(n - 1, 10, np.int32), 2, 0)
    with pytest.raises(ValueError):
        wb.wb_shard_batch(offs[:1], samples, np.full(n, 10, np.int32), 2, 0)
    with pytest.raises(ValueError):
        wb.wb_stitch_tokens(samples, 0, np.zeros((n - 1, 448), np.int32), np.full(n, 10, np.int32))
    with pytest.raises(ValueError):
        wb.wb_stitch_tokens(samples, 0, np.zeros((n, 448), np.int32), np.full(n + 1, 10, np.int32))
