"""The allocation-free quantiser entry point gives the same result as the
regular one.

wb_quantise_e4m3_static serves callers that cannot allocate device memory
(an application allocator that owns all device memory, or code that must not
risk the implicit synchronisation of cudaMalloc/cudaFree).  Its scratch is a
fixed array inside the library, shared by all calls, so this test calls it
twice in a row on different inputs: the second call must not see anything
left over from the first.  It is called through the C ABI with ctypes and
compared with wb_quantise_e4m3 on the same inputs; E4M3 codes and scales are
integer-exact results, so the comparison is bit-exact.  This file is named to
be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import whisper_encoder_decoder_log_b300 as wb

pytestmark = pytest.mark.gpu


def _regular(x):
    codes = torch.empty(x.numel(), dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, device="cuda")
    wb.wb_quantise_e4m3(x, codes, scale)
    return codes, scale


def _static_via_cabi(x):
    L = wb.lib()
    codes = torch.full((x.numel(),), 0xAA, dtype=torch.uint8, device="cuda")
    scale = torch.full((1,), -1.0, device="cuda")
    st = L.wb_quantise_e4m3_static(ctypes.c_void_p(x.data_ptr()), 1 if x.dtype == torch.bfloat16 else 0,
                                   x.numel(), ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scale.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.wb_last_error()
    return codes, scale


def test_static_quantiser_matches_regular_twice_in_a_row():
    rng = np.random.default_rng(123)
    big = torch.from_numpy(rng.normal(0, 40.0, size=3_000_001).astype(np.float32)).cuda()
    small = torch.from_numpy(rng.normal(0, 0.5, size=70_000).astype(np.float32)).cuda().to(torch.bfloat16)
    for x in (big, small):           # the second call follows a larger, larger-valued one
        c_ref, s_ref = _regular(x)
        c_got, s_got = _static_via_cabi(x)
        torch.cuda.synchronize()
        assert s_got.item() == s_ref.item()
        assert torch.equal(c_got, c_ref)
    wb.wb_sync_status()


def test_static_quantiser_at_its_limit_matches_the_oracle():
    """n = 2^26, the largest size the fixed scratch covers: codes and scale
    bit-exact against the oracle's per-tensor quantiser (scale amax / 448,
    codes of x * fp32(1 / scale)), compared piecewise; and n = 0 writes scale 1."""
    from oracle import e4m3 as oe4m3
    n = 1 << 26
    rng = np.random.default_rng(321)
    x = rng.normal(0, 3.0, size=n).astype(np.float32)
    x[n - 5] = -1234.5                       # the amax sits in the last block
    c_got, s_got = _static_via_cabi(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    s_ref = oe4m3.scale_of(float(np.max(np.abs(x))))
    assert np.float32(s_got.item()) == s_ref
    got = c_got.cpu().numpy()
    step = 1 << 23
    for i in range(0, n, step):
        assert np.array_equal(got[i:i + step], oe4m3.quantise(x[i:i + step], s_ref)), i
    empty = torch.empty(0, device="cuda")
    c0, s0 = _static_via_cabi(empty)
    torch.cuda.synchronize()
    assert s0.item() == 1.0 and c0.numel() == 0
    wb.wb_sync_status()


def test_static_quantiser_rejects_oversize_input():
    L = wb.lib()
    n = (1 << 26) + 1
    st = L.wb_quantise_e4m3_static(ctypes.c_void_p(16), 0, n, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                   ctypes.c_void_p(0))
    assert st == -2
    assert b"2^26" in L.wb_last_error()
