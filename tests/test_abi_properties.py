"""Randomised agreement of the library's host-side bookkeeping with the
oracle ("whisper-blaze 0.1.8": Batch Transcription, VRAM usage guide, GPU Mel
Spectrogram's overlapping windows): wave plans, the split of one batch over
several GPUs, overlapping chunk counts and token stitching, bit for bit on
seeded random batches that include the edge cases (one-sample requests,
requests of exactly one chunk, a budget that holds exactly one chunk, more
GPUs than chunks).  No GPU is needed."""
import numpy as np
import pytest
from hypothesis import assume, given, settings, strategies as st

import whisper_encoder_decoder_log_b300 as wb
from oracle import plan as oplan
from synth import LARGE_V3, TURBO

CHUNK = 480000


@pytest.fixture(scope="module", autouse=True)
def built():
    from whisper_encoder_decoder_log_b300 import build
    build.build()
    yield


# request lengths: the edges (1 sample, one chunk exactly, one sample past it)
# mixed with random lengths of up to 7 chunks
_samples = st.lists(st.one_of(st.sampled_from([1, CHUNK - 1, CHUNK, CHUNK + 1, 2 * CHUNK]),
                              st.integers(1, 7 * CHUNK)), min_size=1, max_size=12)


@settings(max_examples=60, deadline=None, derandomize=True)
@given(lens=st.lists(st.integers(5, 448), min_size=1, max_size=160), slack=st.floats(1.0, 40.0),
       kv=st.sampled_from([wb.KV_FP8_SELF, wb.KV_FP8_CROSS]), turbo=st.booleans())
def test_wave_plan_equals_the_oracle(lens, slack, kv, turbo):
    dims = TURBO if turbo else LARGE_V3
    lens = np.array(lens, np.int32)
    cb = 1 if kv == wb.KV_FP8_CROSS else 2
    biggest = oplan.chunk_state_bytes(dims.d_model, dims.dec_layers, int(lens.max()), cb)
    budget = int(biggest * slack)
    desc = wb.make_desc(dims, wb.PREC_MIXED_FP8, kv)
    wave, order, nw = wb.wb_plan_waves(desc, lens, budget)
    ref = oplan.plan_waves(lens, dims.d_model, dims.dec_layers, budget, cb)
    assert nw == len(ref)
    assert np.array_equal(order, np.concatenate(ref))
    for w, chunks in enumerate(ref):
        assert (wave[chunks] == w).all()
    # one byte less than the largest chunk needs: both sides refuse
    with pytest.raises(wb.WBError):
        wb.wb_plan_waves(desc, lens, biggest - 1)
    with pytest.raises(ValueError):
        oplan.plan_waves(lens, dims.d_model, dims.dec_layers, biggest - 1, cb)


@settings(max_examples=60, deadline=None, derandomize=True)
@given(samples=_samples, world=st.integers(1, 12), seed=st.integers(0, 10**6))
def test_shard_split_equals_the_oracle_and_covers_each_chunk_once(samples, world, seed):
    samples = np.array(samples, np.int64)
    offs = np.zeros_like(samples)
    offs[1:] = np.cumsum(samples)[:-1]
    n = wb.wb_chunk_count(samples)
    assert n == oplan.chunk_table(samples)[0].size
    lens = np.random.default_rng(seed).integers(5, 449, size=n).astype(np.int32)
    first = oplan.shard_ranges(lens, world)
    covered = np.zeros(n, np.int32)
    for rank in range(world):
        ro, rs, c0, cn = wb.wb_shard_batch(offs, samples, lens, world, rank)
        assert (c0, cn) == (first[rank], first[rank + 1] - first[rank])
        eo, es = oplan.shard_requests(offs, samples, c0, c0 + cn)
        assert np.array_equal(ro, eo) and np.array_equal(rs, es)
        covered[c0:c0 + cn] += 1
        # the rank's requests re-chunk to exactly its chunks, with the same valid samples
        if cn:
            assert wb.wb_chunk_count(rs) == cn
            assert np.array_equal(oplan.chunk_table(rs)[2], oplan.chunk_table(samples)[2][c0:c0 + cn])
    assert (covered == 1).all()


@settings(max_examples=60, deadline=None, derandomize=True)
@given(samples=_samples, overlap=st.one_of(st.sampled_from([0, 1, 16000, CHUNK // 2, CHUNK - 1]),
                                           st.integers(0, CHUNK - 1)),
       seed=st.integers(0, 10**6))
def test_overlap_count_and_stitching_equal_the_oracle(samples, overlap, seed):
    samples = np.array(samples, np.int64)
    stride = CHUNK - overlap
    assume(int(sum(1 + (max(0, int(s) - CHUNK) + stride - 1) // stride for s in samples)) <= 3000)
    req, idx, valid = oplan.chunk_table(samples, overlap)
    n = req.size
    assert wb.wb_chunk_count(samples, overlap) == n
    # the chunks of a request start `CHUNK - overlap` apart and together reach its end
    for r in range(samples.size):
        k = idx[req == r]
        assert k.max() * (CHUNK - overlap) + valid[req == r][-1] == samples[r]
    rng = np.random.default_rng(seed)
    lens = rng.integers(4, 40, size=n).astype(np.int32)        # 4: a chunk with no generated token
    tok = rng.integers(0, 3, size=(n, 448)).astype(np.int32)   # a 3-token alphabet: overlaps are common
    got = wb.wb_stitch_tokens(samples, overlap, tok, lens, 4)
    for r in range(samples.size):
        rows = [tok[c, 4:lens[c]] for c in range(n) if req[c] == r]
        assert np.array_equal(got[r], oplan.stitch(rows)), r
