"""Pins for the oracle's E4M3 quantiser against the format and torch's float8."""
import os

import numpy as np
import pytest
import torch

from oracle import e4m3

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_decode_table_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.decode_table()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_golden_codes():
    for line in open(os.path.join(GOLD, "e4m3_codes.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        v, c = line.split()
        assert int(e4m3.encode(float(v))) == int(c, 16), v
        assert e4m3.decode(np.uint8(int(c, 16))) == float(v)


def test_round_trip_all_finite_codes():
    for code in range(256):
        if code in (0x7F, 0xFF):
            continue
        assert int(e4m3.encode(e4m3.decode(np.uint8(code)))) == code


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 50, 200000), rng.normal(0, 0.01, 100000),
                        rng.uniform(-440, 440, 100000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode(x), ref)


def test_ties_to_even_and_saturation():
    vals = e4m3.decode_table()[:0x7F]
    mids = (vals[:-1] + vals[1:]) / 2
    codes = e4m3.encode(mids)
    lo = np.arange(0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(codes, expect.astype(np.uint8))
    assert int(e4m3.encode(449.0)) == 0x7E and int(e4m3.encode(1e30)) == 0x7E
    assert int(e4m3.encode(-np.inf)) == 0xFE and int(e4m3.encode(np.nan)) == 0x7F
    assert int(e4m3.encode(-0.0)) == 0x80 and int(e4m3.encode(-1e-30)) == 0x80


def test_scale_rules():
    assert e4m3.scale_of(448.0) == np.float32(1.0)
    assert e4m3.scale_of(0.0) == np.float32(1.0)
    assert e4m3.kv_scale_of(224.0) == np.float32(1.0)
    assert e4m3.kv_scale_of(0.0) == np.float32(np.float32(2e-12) / np.float32(448))
    x = np.random.default_rng(1).normal(size=(64, 64)).astype(np.float32)
    q, s = e4m3.quantise_tensor(x)
    assert int(np.max(q & 0x7F)) == 0x7E       # the amax lands on the top code
    err = np.abs(e4m3.dequantise(q, s) - x)
    assert (err <= np.abs(x) * 2.0 ** -4 + s * 2.0 ** -10).all()


@pytest.mark.parametrize("s", [0.37, 1.0, 3e-3])
def test_quantise_is_one_fp32_product(s):
    s = np.float32(s)
    x = np.random.default_rng(2).normal(size=5000).astype(np.float32)
    inv = np.float32(1) / s
    ref = torch.from_numpy(np.clip(x * inv, -448, 448)).to(torch.float8_e4m3fn)
    assert np.array_equal(e4m3.quantise(x, s), ref.view(torch.uint8).numpy())


def test_grid_rounding_equals_code_rounding():
    """round_values (rounding onto the 2^(e-3) grid) is the same map as
    decode(encode(x)) (nearest of the 253 finite values, ties to the even
    code): on every value, every tie between neighbours, just either side of
    each tie, past the top, and over random magnitudes 2^-14 .. 2^10."""
    vals = e4m3.decode_table()[:0x7F]
    mids = (vals[:-1] + vals[1:]) / 2
    near = np.concatenate([np.nextafter(mids, 0), np.nextafter(mids, np.inf)])
    rng = np.random.default_rng(5)
    rand = np.ldexp(rng.uniform(1, 2, 400000), rng.integers(-14, 11, 400000))
    x = np.concatenate([vals, mids, near, [0.0, 448.0, 449.0, 463.9, 464.0, 465.0, 1e9, np.inf], rand])
    x = np.concatenate([x, -x])
    assert np.array_equal(e4m3.round_values(x), e4m3.decode(e4m3.encode(x)))
    assert np.array_equal(np.signbit(e4m3.round_values(np.array([-0.0, -1e-30]))), [True, True])
