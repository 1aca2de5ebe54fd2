"""Oracle: float8 E4M3 quantisation with a per-tensor scale.

[WB] "Direct Kernel API": ``quantise_e4m3(x) -> (fp8, scale)`` and
``dequantise_e4m3(fp8, scale, shape)``; "Precision Presets": ``mixed_fp8``
runs FFN and QKV in FP8.  [BFW] "Inference Stack": activations are dynamically
quantised so the KV cache holds 1-byte float8 values while the arithmetic is
done in bfloat16.

Format (OCP FP8 E4M3, the ``e4m3fn`` variant): 1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits; exponent field 0 encodes subnormals m/8 * 2^-6; the
largest finite magnitude is 1.75 * 2^8 = 448 (code 0x7E); codes 0x7F / 0xFF are
NaN; there is no infinity.

Readings (the pages name the scaling but give no rule):
  * quantisation of an fp32 value x with scale s: q = RNE_satfinite(x * inv_s)
    where inv_s = fp32(1 / s) and x * inv_s is one fp32 product; ties go to the
    even code, magnitudes beyond 448 clamp to 448, the sign of zero is kept;
  * dequantisation: value(q) * s;
  * weights and GEMM activations: s = amax / 448 (fp32 division);
  * self-attention KV cache: one scale per (chunk, layer, K or V), fixed from
    the forced-prefix rows as s = 2 * max(amax, 1e-12) / 448 (a 2x headroom)
    and kept for every later position; later values beyond 448 * s saturate.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def decode_table() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for 0x7F and 0xFF)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_TABLE = decode_table()
_POS_VALUES = _TABLE[:0x7F]          # codes 0x00..0x7E, increasing magnitude


def decode(codes: np.ndarray) -> np.ndarray:
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x) -> np.ndarray:
    """Round float values to E4M3 codes: nearest, ties to even code, satfinite."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    hi = np.searchsorted(_POS_VALUES, mag, side="left")   # first value >= mag
    hi = np.clip(hi, 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo = mag - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= E4M3_MAX, 0x7E, code)           # satfinite
    code = code.astype(np.uint8)
    code |= np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    code = np.where(np.isnan(x), 0x7F, code).astype(np.uint8)
    return code


def round_values(x) -> np.ndarray:
    """E4M3 rounding as values: the same result as decode(encode(x)) for
    finite x, written as rounding onto the format's grid.  Inside binade
    [2^e, 2^(e+1)) E4M3 has 8 values 2^(e-3) apart (e >= -6; below 2^-6 the
    subnormals keep the spacing 2^-9), so the nearest value is rint(|x| /
    2^(e-3)) * 2^(e-3), rint rounding ties to even, which is the even code
    (the code's last bit is the last mantissa bit); magnitudes above 448 take
    448 (satfinite); the sign is kept."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    _, ex = np.frexp(mag)                      # mag = f 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)
    step = np.ldexp(1.0, e - 3)
    q = np.minimum(np.rint(mag / step) * step, E4M3_MAX)
    return np.copysign(q, x)


def scale_of(amax: float) -> np.float32:
    """Per-tensor scale of a weight or GEMM activation: amax / 448 in fp32.

    An all-zero tensor (amax 0) takes scale 1 so that the inverse exists.
    """
    a = np.float32(amax)
    if a == 0:
        return np.float32(1.0)
    return np.float32(a / np.float32(E4M3_MAX))


def kv_scale_of(amax: float) -> np.float32:
    """KV-cache scale: 2 * max(amax, 1e-12) / 448 in fp32."""
    a = np.maximum(np.float32(amax), np.float32(1e-12))
    return np.float32(np.float32(2.0) * a / np.float32(E4M3_MAX))


def quantise(x, s: np.float32) -> np.ndarray:
    """Codes of fp32(x) * fp32(1/s), one fp32 product per element."""
    inv = np.float32(np.float32(1.0) / np.float32(s))
    return encode(np.asarray(x, dtype=np.float32) * inv)


def dequantise(codes, s) -> np.ndarray:
    return decode(codes) * np.float64(np.float32(s))


def quantise_tensor(x):
    """[WB] ``quantise_e4m3``: (codes, scale) with scale = amax / 448."""
    x32 = np.asarray(x, dtype=np.float32)
    s = scale_of(np.max(np.abs(x32)) if x32.size else 0.0)
    return quantise(x32, s), s
