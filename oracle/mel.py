"""Oracle: audio chunking and the log-Mel spectrogram, in float64.

[WB] "GPU Mel Spectrogram" and "Direct Kernel API": the front end maps float32
16 kHz audio to a [n_mels, T] log-Mel array on the GPU, replacing the CPU
librosa / Hugging Face preprocessor.  [UOW] section 2: the signal is cut into
short overlapping frames, each frame is Fourier transformed, and the spectrum is
mapped onto the mel scale; window, hop and band count are the key parameters.
[WB] "Batch Transcription": long audio is processed as 30-second chunks.

Readings taken where the pages are silent (the preprocessor being replaced is
the librosa-style Whisper front end, so its conventions are used):
  * n_fft 400 (25 ms), hop 160 (10 ms), periodic Hann window;
  * the frame is centred: reflect padding of n_fft/2 samples on both sides of
    the chunk (mirror without repeating the edge sample), which yields 3001
    frames of which the last is dropped, leaving 3000;
  * power spectrum |X_k|^2, k = 0..200;
  * Slaney mel scale with area-normalised triangles, 0 Hz .. 8 kHz;
  * log10 of the mel energy clamped below at 1e-10, then floored at
    (maximum over the whole chunk) - 8, then mapped by (x + 4) / 4.
"""
from __future__ import annotations

import numpy as np

SR = 16000
N_FFT = 400
HOP = 160
N_BINS = N_FFT // 2 + 1
CHUNK = 480000
N_FRAMES = 3000


# ------------------------------------------------------------------ chunking

def split_into_chunks(audio: np.ndarray, offsets, samples, overlap: int = 0):
    """Cut each request into 30 s chunks, zero-padding its last chunk.

    [WB] "Batch Transcription": every input is split into 30-second chunks and
    all chunks go through one generate pass.  With ``overlap`` samples
    ([WB] "GPU Mel Spectrogram", ``process_chunks(..., overlap_s)``;
    [TWT] ``overlap_seconds``), consecutive chunks of a request start
    480000 - overlap samples apart and share ``overlap`` samples; the last
    chunk is the first that reaches the request's end.  Chunk k holds samples
    [k stride, k stride + 480000) of its request; samples past the end are
    zero.  Returns (chunks [n,480000] float64, req_of_chunk int32,
    index_in_req int32, valid_samples int32).
    """
    stride = CHUNK - int(overlap)
    if not 0 <= int(overlap) < CHUNK:
        raise ValueError("overlap must be in [0, 480000)")
    chunks, req, idx, valid = [], [], [], []
    for r, (o, s) in enumerate(zip(offsets, samples)):
        s = int(s)
        n = 1 + (max(0, s - CHUNK) + stride - 1) // stride
        for k in range(n):
            lo = k * stride
            hi = min(s, lo + CHUNK)
            c = np.zeros(CHUNK, dtype=np.float64)
            c[: hi - lo] = audio[int(o) + lo: int(o) + hi]
            chunks.append(c)
            req.append(r)
            idx.append(k)
            valid.append(hi - lo)
    return (np.array(chunks).reshape(-1, CHUNK), np.array(req, np.int32),
            np.array(idx, np.int32), np.array(valid, np.int32))


# ------------------------------------------------------------------ window, DFT

def hann_periodic(n: int = N_FFT) -> np.ndarray:
    """w[i] = 0.5 - 0.5 cos(2 pi i / n), i = 0..n-1 (periodic form)."""
    i = np.arange(n, dtype=np.float64)
    return 0.5 - 0.5 * np.cos(2.0 * np.pi * i / n)


def reflect_pad(x: np.ndarray, p: int = N_FFT // 2) -> np.ndarray:
    """Mirror p samples onto each side, not repeating the edge sample."""
    left = x[p:0:-1]
    right = x[-2:-p - 2:-1]
    return np.concatenate([left, x, right])


def frames(chunk: np.ndarray) -> np.ndarray:
    """[3000, 400] windowed frames; frame t covers padded[160 t : 160 t + 400]."""
    xp = reflect_pad(np.asarray(chunk, dtype=np.float64))
    idx = HOP * np.arange(N_FRAMES)[:, None] + np.arange(N_FFT)[None, :]
    return xp[idx] * hann_periodic()[None, :]


def dft_matrix(n: int = N_FFT) -> np.ndarray:
    """[n, n//2+1] complex, M[i, k] = exp(-2 pi i k j / n)."""
    i = np.arange(n)[:, None]
    k = np.arange(n // 2 + 1)[None, :]
    return np.exp(-2j * np.pi * ((i * k) % n) / n)


def power_spectrum(chunk: np.ndarray) -> np.ndarray:
    """[3000, 201] |X_k|^2 of every frame (one-sided)."""
    X = frames(chunk) @ dft_matrix()
    return X.real ** 2 + X.imag ** 2


# ------------------------------------------------------------------ mel scale

_F_SP = 200.0 / 3.0                 # Hz per mel below 1 kHz
_MIN_LOG_HZ = 1000.0
_MIN_LOG_MEL = _MIN_LOG_HZ / _F_SP  # 15
_LOGSTEP = np.log(6.4) / 27.0


def hz_to_mel(f):
    """Slaney mel: linear below 1 kHz, logarithmic above."""
    f = np.asarray(f, dtype=np.float64)
    lin = f / _F_SP
    log = _MIN_LOG_MEL + np.log(np.maximum(f, 1e-300) / _MIN_LOG_HZ) / _LOGSTEP
    return np.where(f >= _MIN_LOG_HZ, log, lin)


def mel_to_hz(m):
    m = np.asarray(m, dtype=np.float64)
    lin = _F_SP * m
    log = _MIN_LOG_HZ * np.exp(_LOGSTEP * (m - _MIN_LOG_MEL))
    return np.where(m >= _MIN_LOG_MEL, log, lin)


def mel_filterbank(n_mels: int, sr: int = SR, n_fft: int = N_FFT,
                   fmin: float = 0.0, fmax: float = 8000.0) -> np.ndarray:
    """[n_mels, n_fft//2+1] area-normalised triangular filters on the Slaney scale.

    Filter m rises linearly from f_m to f_{m+1} and falls to f_{m+2}, where the
    f's are n_mels+2 points equally spaced in mel between fmin and fmax; it is
    scaled by 2 / (f_{m+2} - f_m) so that its continuous area is 1.
    """
    bin_hz = np.arange(n_fft // 2 + 1, dtype=np.float64) * sr / n_fft
    pts = mel_to_hz(np.linspace(hz_to_mel(fmin), hz_to_mel(fmax), n_mels + 2))
    fb = np.zeros((n_mels, bin_hz.size), dtype=np.float64)
    for m in range(n_mels):
        lo, c, hi = pts[m], pts[m + 1], pts[m + 2]
        up = (bin_hz - lo) / (c - lo)
        down = (hi - bin_hz) / (hi - c)
        fb[m] = np.maximum(0.0, np.minimum(up, down)) * (2.0 / (hi - lo))
    return fb


# ------------------------------------------------------------------ log-Mel

def log_mel(chunk: np.ndarray, n_mels: int) -> np.ndarray:
    """[n_mels, 3000] normalised log-Mel of one 30 s chunk (float64)."""
    mel = mel_filterbank(n_mels) @ power_spectrum(chunk).T
    ell = np.log10(np.maximum(mel, 1e-10))
    ell = np.maximum(ell, ell.max() - 8.0)
    return (ell + 4.0) / 4.0


def log_mel_batch(audio: np.ndarray, n_mels: int) -> np.ndarray:
    """[B, n_mels, 3000]; each chunk is normalised on its own maximum."""
    return np.stack([log_mel(a, n_mels) for a in np.asarray(audio)])
