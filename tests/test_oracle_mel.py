"""Pins for the oracle's front end: chunking, window, DFT, mel scale, log-Mel."""
import os

import numpy as np
import pytest

from oracle import mel

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_hann_periodic_matches_scipy_and_closed_forms():
    from scipy.signal import get_window
    w = mel.hann_periodic()
    np.testing.assert_allclose(w, get_window("hann", 400, fftbins=True), atol=1e-15)
    assert w[0] == 0.0 and abs(w[200] - 1.0) < 1e-15
    assert abs(w.sum() - 200.0) < 1e-9 and abs((w ** 2).sum() - 150.0) < 1e-9


def test_reflect_pad_matches_numpy():
    x = np.random.default_rng(0).normal(size=1000)
    np.testing.assert_array_equal(mel.reflect_pad(x), np.pad(x, 200, mode="reflect"))


def test_power_spectrum_direct_sum_dft():
    rng = np.random.default_rng(1)
    chunk = rng.uniform(-1, 1, size=mel.CHUNK)
    P = mel.power_spectrum(chunk)
    assert P.shape == (3000, 201)
    xp = np.pad(chunk, 200, mode="reflect")
    w = 0.5 - 0.5 * np.cos(2 * np.pi * np.arange(400) / 400)
    for t in (0, 1, 1500, 2999):
        fr = xp[160 * t:160 * t + 400] * w
        for k in (0, 1, 37, 100, 199, 200):
            re = sum(fr[n] * np.cos(2 * np.pi * k * n / 400) for n in range(400))
            im = -sum(fr[n] * np.sin(2 * np.pi * k * n / 400) for n in range(400))
            assert abs(P[t, k] - (re * re + im * im)) <= 1e-9 * max(1.0, P[t, k])


def test_power_spectrum_matches_numpy_rfft():
    chunk = np.random.default_rng(2).normal(0, 0.3, size=mel.CHUNK)
    P = mel.power_spectrum(chunk)
    ref = np.abs(np.fft.rfft(mel.frames(chunk), axis=1)) ** 2
    np.testing.assert_allclose(P, ref, rtol=1e-9, atol=1e-9)


def test_parseval_per_frame():
    chunk = np.random.default_rng(3).normal(0, 0.3, size=mel.CHUNK)
    F = mel.frames(chunk)
    P = mel.power_spectrum(chunk)
    lhs = (F ** 2).sum(axis=1)
    rhs = (P[:, 0] + 2 * P[:, 1:200].sum(axis=1) + P[:, 200]) / 400.0
    np.testing.assert_allclose(lhs, rhs, rtol=1e-10)


@pytest.mark.parametrize("k0", [2, 25, 101, 198])
def test_pure_sine_three_bins(k0):
    A = 0.5
    n = np.arange(mel.CHUNK)
    chunk = A * np.sin(2 * np.pi * 40.0 * k0 * n / 16000.0 + 0.3)
    P = mel.power_spectrum(chunk)
    inner = P[5:2990]           # frames clear of the reflect padding
    np.testing.assert_allclose(inner[:, k0], (100 * A) ** 2, rtol=1e-9)
    np.testing.assert_allclose(inner[:, k0 - 1], (50 * A) ** 2, rtol=1e-9)
    np.testing.assert_allclose(inner[:, k0 + 1], (50 * A) ** 2, rtol=1e-9)
    others = np.delete(inner, [k0 - 1, k0, k0 + 1], axis=1)
    assert np.abs(others).max() < 1e-12 * (100 * A) ** 2


def test_slaney_mel_golden():
    rows = [l.split() for l in open(os.path.join(GOLD, "slaney_mel.txt"))
            if l.strip() and not l.startswith("#")]
    for hz, m in rows:
        assert abs(float(mel.hz_to_mel(float(hz))) - float(m)) < 1e-9
        assert abs(float(mel.mel_to_hz(float(m))) - float(hz)) < 1e-6


@pytest.mark.parametrize("n_mels", [80, 128])
def test_filterbank_properties(n_mels):
    fb = mel.mel_filterbank(n_mels)
    assert fb.shape == (n_mels, 201)
    assert (fb >= 0).all() and (fb.sum(axis=1) > 0).all()
    pts = mel.mel_to_hz(np.linspace(0, mel.hz_to_mel(8000.0), n_mels + 2))
    bins = np.arange(201) * 40.0
    for m in range(n_mels):
        # the maximum sits on the FFT bin nearest the filter centre
        lo, c, hi = pts[m:m + 3]
        near = np.argmin(np.abs(bins - c))
        assert abs(bins[np.argmax(fb[m])] - c) <= abs(bins[near] - c) + 40.0
        # continuous area 1: the Riemann sum converges for filters much wider than a bin
        if hi - lo > 400.0:
            assert abs(fb[m].sum() * 40.0 - 1.0) < 0.02
    # every FFT bin below 8 kHz feeds at most two filters
    assert ((fb > 0).sum(axis=0) <= 2).all()


@pytest.mark.parametrize("n_mels", [80, 128])
def test_silence_is_minus_one_and_a_half(n_mels):
    out = mel.log_mel(np.zeros(mel.CHUNK), n_mels)
    assert out.shape == (n_mels, 3000)
    assert (out == -1.5).all()


def test_sine_lands_in_expected_mel_band():
    k0 = 30                                      # 1200 Hz
    n = np.arange(mel.CHUNK)
    chunk = 0.3 * np.sin(2 * np.pi * 40.0 * k0 * n / 16000.0)
    out = mel.log_mel(chunk, 128)
    fb = mel.mel_filterbank(128)
    expect = np.argmax(fb[:, k0 - 1] / 4 + fb[:, k0] + fb[:, k0 + 1] / 4)
    assert (np.argmax(out[:, 100:2900], axis=0) == expect).all()
    assert out.max() == pytest.approx(out[expect, 1500], abs=1e-6)


def test_floor_is_chunk_max_minus_eight():
    rng = np.random.default_rng(4)
    chunk = rng.normal(0, 0.1, size=mel.CHUNK)
    chunk[100000:200000] = 0.0                   # a silent span
    out = mel.log_mel(chunk, 128)
    floor = (out.max() * 4 - 4 - 8 + 4) / 4      # (max_ell - 8 + 4) / 4
    assert abs(out.min() - floor) < 1e-12
    assert np.all(out[:, 700:1200] == out.min())


def test_chunks_zero_pad_and_table():
    audio = np.arange(1_200_000, dtype=np.float32) / 1e6
    ch, req, idx, valid = mel.split_into_chunks(audio, [0, 500_000], [500_000, 700_000])
    assert ch.shape == (4, 480000)
    assert list(req) == [0, 0, 1, 1] and list(idx) == [0, 1, 0, 1]
    assert list(valid) == [480000, 20000, 480000, 220000]
    assert (ch[1, 20000:] == 0).all() and ch[1, 0] == audio[480000]
    assert ch[3, 219999] == audio[500000 + 480000 + 219999]
