"""The seeded synthetic inputs follow their stated recipe: the sine + noise
speech stand-in, the mel workload's low-passed noise with silent spans, the
mixed-length serving batch (48 requests of 2-15 min, decode lengths 64-448)
and the N(0, 0.02) random-init weights.  Seeds make every input reproducible
and independent of the order it is drawn in."""
import numpy as np
import pytest

import synth
from synth import CHUNK_SAMPLES, SAMPLE_RATE


def test_sine_audio_is_three_sines_plus_small_noise():
    x = synth.sine_chunk_audio(5).astype(np.float64)
    assert x.shape == (CHUNK_SAMPLES,) and x.dtype == np.float64
    assert np.abs(x).max() <= 1.0
    spec = np.abs(np.fft.rfft(x)) / (CHUNK_SAMPLES / 2)       # sine amplitude per bin (2 bins per Hz)
    top = np.argsort(spec)[-3:]
    freqs = top * SAMPLE_RATE / CHUNK_SAMPLES
    assert ((freqs >= 100) & (freqs <= 4000)).all(), freqs
    # a sine between bins spreads its energy: sum the peak's neighbourhood
    amps = [np.sqrt((spec[max(0, k - 3):k + 4] ** 2).sum()) for k in top]
    assert all(0.17 < a < 0.21 for a in amps), amps
    # above 6 kHz, 2 kHz clear of every line, only the N(0, 0.01) noise is
    # left: white noise puts N sigma^2 of power in each bin on average
    X = np.fft.rfft(x)
    band = X[int(6000 * CHUNK_SAMPLES / SAMPLE_RATE):]
    sigma = np.sqrt(np.mean(np.abs(band) ** 2) / CHUNK_SAMPLES)
    assert 0.0095 < sigma < 0.0105, sigma


def test_pink_audio_is_low_passed_noise_with_tenth_silent():
    x = synth.pink_chunk_audio(3).astype(np.float64)
    assert x.shape == (CHUNK_SAMPLES,) and np.abs(x).max() <= 1.0
    zero = x == 0.0
    assert 0.08 <= zero.mean() <= 0.105, zero.mean()      # about 10 %: spans may overlap
    # silent spans are runs of zeros of 0.2-1 s (shorter only where spans meet or the quota ends)
    edges = np.flatnonzero(np.diff(np.concatenate([[0], zero.astype(np.int8), [0]])))
    runs = edges[1::2] - edges[::2]
    assert (runs >= 0.2 * SAMPLE_RATE).mean() > 0.6
    # y[n] = 0.95 y[n-1] + w[n]: lag-1 autocorrelation 0.95 on the voiced part
    v = x[~zero]
    r1 = np.corrcoef(v[:-1], v[1:])[0, 1]
    assert 0.93 < r1 < 0.97, r1


def test_serving_batch_matches_its_stated_size():
    sb = synth.serving_requests(0, n_req=48, with_audio=False)
    assert sb.req_samples.size == 48
    dur = sb.req_samples / SAMPLE_RATE
    assert dur.min() >= 120 and dur.max() <= 900
    assert round(float(dur.sum())) == 25647
    assert sb.chunk_len.size == 875 == int(np.ceil(sb.req_samples / CHUNK_SAMPLES).sum())
    assert sb.chunk_len.min() >= 64 and sb.chunk_len.max() <= 448
    assert 200 < sb.chunk_len.mean() < 310                  # uniform on 64..448: mean 256
    assert np.array_equal(sb.req_offsets[1:], np.cumsum(sb.req_samples)[:-1])
    # with audio (a smaller batch): requests back to back, each its own seeded recording
    small = synth.serving_requests(1, n_req=3)
    assert small.audio.size == small.req_samples.sum()
    for r in range(3):
        seg = small.audio[small.req_offsets[r]:small.req_offsets[r] + small.req_samples[r]]
        assert np.array_equal(seg, synth.sine_chunk_audio(1 * 7919 + r, int(small.req_samples[r])))
    nb = synth.serving_requests(1, n_req=3, with_audio=False)
    assert np.array_equal(nb.chunk_len, small.chunk_len) and np.array_equal(nb.req_samples, small.req_samples)


@pytest.mark.parametrize("bf16", [False, True])
def test_weights_are_small_normals_with_unit_gains(bf16):
    W = synth.make_weights(synth.TINY, 4, bf16=bf16)
    w = W["enc.0.fc1.w"].astype(np.float64)
    assert abs(w.mean()) < 1e-3 and 0.0195 < w.std() < 0.0205
    g = W["enc.0.ln1.g"].astype(np.float64)
    assert abs(g.mean() - 1.0) < 5e-3 and 0.015 < g.std() < 0.025
    b = W["enc.0.ln1.b"].astype(np.float64)
    assert abs(b.mean()) < 5e-3 and 0.015 < b.std() < 0.025
    if bf16:
        for v in (w, g, b):
            assert np.array_equal(synth.round_to_bf16(v.astype(np.float32)), v.astype(np.float32))
    # one tensor regenerates alone, and layer subsets draw the same values
    sub = synth.make_weights(synth.TINY, 4, bf16=bf16, decoder=False, enc_layers=[0])
    assert np.array_equal(sub["enc.0.fc1.w"], W["enc.0.fc1.w"]) and "enc.1.fc1.w" not in sub


def test_seeds_are_reproducible_and_distinct():
    a = synth.batch_audio("sine", 2, 11)
    assert np.array_equal(a, synth.batch_audio("sine", 2, 11))
    assert not np.array_equal(a[0], a[1])
    assert not np.array_equal(a[0], synth.batch_audio("sine", 1, 12)[0])
    p = synth.forced_prefix(0, 51866)
    assert p.shape == (4,) and np.array_equal(p, synth.forced_prefix(0, 51866))
    t = synth.random_tokens(3, (5, 7), 51866)
    assert t.shape == (5, 7) and t.min() >= 0 and t.max() < 51866
