"""Pins for the oracle's chunk table and wave packing."""
import numpy as np
import pytest

from oracle import plan
from synth import serving_requests


def test_chunk_table_counts():
    req, idx, valid = plan.chunk_table([480000, 480001, 1, 1_000_000])
    assert list(req) == [0, 1, 1, 2, 3, 3, 3]
    assert list(idx) == [0, 0, 1, 0, 0, 1, 2]
    assert list(valid) == [480000, 480000, 1, 1, 480000, 480000, 40000]


def test_chunk_state_bytes_closed_form():
    # large-v3 decoder: 32 layers x (2 x 1500 x 1280 x 2 + 2 x L x 1280) + 448 x 4
    assert plan.chunk_state_bytes(1280, 32, 448) == 32 * (7_680_000 + 1_146_880) + 1792


@pytest.mark.parametrize("budget", [10**9, 5 * 10**9, 180 * 10**9])
def test_waves_cover_each_chunk_once_within_budget(budget):
    rng = np.random.default_rng(0)
    lens = rng.integers(64, 449, size=300)
    waves = plan.plan_waves(lens, 1280, 4, budget)
    allc = np.concatenate(waves)
    assert sorted(allc.tolist()) == list(range(300))
    prev_min = None
    for w in waves:
        assert sum(plan.chunk_state_bytes(1280, 4, lens[c]) for c in w) <= budget
        wl = lens[w]
        assert (np.diff(wl) <= 0).all()                       # longest first
        if prev_min is not None:
            assert wl[0] <= prev_min
        prev_min = wl[-1]
    # greedy: each wave but the last could not take the next chunk
    for a, b in zip(waves[:-1], waves[1:]):
        used = sum(plan.chunk_state_bytes(1280, 4, lens[c]) for c in a)
        assert used + plan.chunk_state_bytes(1280, 4, lens[b[0]]) > budget


def test_serving_batch_waves():
    sb = serving_requests(0, n_req=48, with_audio=False)
    req, idx, valid = plan.chunk_table(sb.req_samples)
    assert req.size == sb.chunk_len.size
    assert 600 <= req.size <= 1100
    waves = plan.plan_waves(sb.chunk_len, 1280, 32, 180 * 10**9)
    assert len(waves) == 2
    assert int(valid.sum()) == int(sb.req_samples.sum())


def test_oversize_chunk_rejected():
    with pytest.raises(ValueError):
        plan.plan_waves([448], 1280, 32, 10**6)


def test_fp8_cross_kv_halves_the_cross_bytes_and_fits_more_per_wave():
    d, L, n = 1280, 32, 200
    bf = plan.chunk_state_bytes(d, L, n)
    f8 = plan.chunk_state_bytes(d, L, n, cross_bytes=1)
    assert bf - f8 == L * 2 * 1500 * d                      # exactly half of the bf16 cross K/V
    lens = np.full(900, 448, np.int32)
    budget = 180 * 10 ** 9
    w_bf = plan.plan_waves(lens, d, L, budget)
    w_f8 = plan.plan_waves(lens, d, L, budget, cross_bytes=1)
    assert len(w_f8) < len(w_bf)
    assert sorted(np.concatenate(w_f8).tolist()) == list(range(900))


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_ranges_cover_every_chunk_once_and_balance(world):
    sb = serving_requests(3, n_req=20, with_audio=False)
    lens = sb.chunk_len
    first = plan.shard_ranges(lens, world)
    assert first[0] == 0 and first[-1] == lens.size and len(first) == world + 1
    assert all(a <= b for a, b in zip(first, first[1:]))
    owner = np.concatenate([np.full(b - a, r) for r, (a, b) in enumerate(zip(first, first[1:]))])
    assert owner.size == lens.size                      # each chunk on exactly one rank, in order
    w = lens.astype(np.int64) + plan.SHARD_CHUNK_BASE
    total = int(w.sum())
    for r in range(world):                               # greedy prefix cut: within one chunk of the mean
        got = int(w[first[r]:first[r + 1]].sum())
        assert abs(got - total / world) <= w.max(), (r, got, total / world)


def test_shard_ranges_more_ranks_than_chunks():
    first = plan.shard_ranges(np.array([100, 200], np.int32), 5)
    assert first[0] == 0 and first[-1] == 2
    sizes = np.diff(first)
    assert sizes.sum() == 2 and (sizes >= 0).all()


def test_shard_requests_rechunk_to_the_same_chunks():
    """A rank's trimmed requests, cut into chunks again, are exactly its chunk
    range: same audio start and same valid samples, in the same order."""
    sb = serving_requests(4, n_req=12, with_audio=False)
    req, idx, valid = plan.chunk_table(sb.req_samples)
    start = sb.req_offsets[req] + idx.astype(np.int64) * plan.CHUNK
    first = plan.shard_ranges(sb.chunk_len, 3)
    for r in range(3):
        c0, c1 = first[r], first[r + 1]
        offs, samples = plan.shard_requests(sb.req_offsets, sb.req_samples, c0, c1)
        rreq, ridx, rvalid = plan.chunk_table(samples)
        assert rreq.size == c1 - c0
        assert np.array_equal(rvalid, valid[c0:c1])
        assert np.array_equal(offs[rreq] + ridx.astype(np.int64) * plan.CHUNK, start[c0:c1])


@pytest.mark.parametrize("overlap", [0, 16000, 160000, 479999])
def test_overlapping_chunk_table_covers_each_request(overlap):
    samples = np.array([1, 480000, 480001, 960000 - overlap, 2_345_678, 31 * 16000], np.int64)
    req, idx, valid = plan.chunk_table(samples, overlap)
    stride = plan.CHUNK - overlap
    for r, s in enumerate(samples):
        ks = idx[req == r]
        n = ks.size
        assert np.array_equal(ks, np.arange(n))
        # brute force: the fewest windows of 480000 samples, stride apart, reaching the end
        m = 1
        while (m - 1) * stride + plan.CHUNK < s:
            m += 1
        assert n == m
        v = valid[req == r]
        assert np.array_equal(v, np.minimum(plan.CHUNK, s - stride * ks))
        assert (v > 0).all()


def test_overlapping_chunks_share_their_samples():
    from oracle import mel as omel
    rng = np.random.default_rng(8)
    samples = np.array([1_000_000, 700_000], np.int64)
    offs = np.array([0, 1_000_000], np.int64)
    audio = rng.normal(size=int(samples.sum()))
    ov = 16000
    chunks, req, idx, valid = omel.split_into_chunks(audio, offs, samples, overlap=ov)
    for c in range(len(req) - 1):
        if req[c] == req[c + 1]:
            assert np.array_equal(chunks[c][plan.CHUNK - ov:], chunks[c + 1][:ov])
    assert np.array_equal(chunks[0], audio[:plan.CHUNK])


def test_stitch_removes_the_repeated_overlap_once():
    a, b, c = [5, 6, 7, 8], [7, 8, 9, 10], [1, 2]
    assert plan.stitch([a, b]).tolist() == [5, 6, 7, 8, 9, 10]       # suffix [7, 8] = prefix of b
    assert plan.stitch([a, c]).tolist() == a + c                     # no overlap: concatenation
    assert plan.stitch([a, [6, 7, 8]]).tolist() == a                 # fully repeated: nothing new
    assert plan.stitch([[], a, []]).tolist() == a
    assert plan.stitch([[3, 3, 3], [3, 3, 4]]).tolist() == [3, 3, 3, 4]   # the longest overlap wins
    rng = np.random.default_rng(9)
    for _ in range(200):                     # planted overlaps on random rows
        x = rng.integers(0, 5, size=rng.integers(0, 12)).tolist()
        k = int(rng.integers(0, len(x) + 1))
        y = x[len(x) - k:] + rng.integers(0, 5, size=rng.integers(0, 6)).tolist()
        out = plan.stitch([x, y]).tolist()
        best = max(j for j in range(min(len(x), len(y)) + 1) if x[len(x) - j:] == y[:j])
        assert out == x + y[best:]
