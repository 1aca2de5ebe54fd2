"""GPU parity of the single kernels reachable through the C ABI: the log-Mel
front end, the tcgen05 GEMM (bf16 and E4M3) and the E4M3 quantiser, against
the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import whisper_encoder_decoder_log_b300 as wb
from oracle import e4m3 as oe4m3
from oracle import mel as omel
from oracle import model as omodel
from synth import batch_audio, round_to_bf16

pytestmark = pytest.mark.gpu

MEL_TOL = 1e-4      # absolute, normalised log domain


def run_mel(audio, n_mels):
    a = torch.from_numpy(audio).cuda()
    out = torch.empty(audio.shape[0], n_mels, 3000, device="cuda")
    wb.wb_mel(a, n_mels, out)
    wb.wb_sync_status()
    return out.cpu().numpy()


@pytest.mark.parametrize("n_mels,kind", [(128, "pink"), (80, "sine"), (128, "sine")])
def test_mel_matches_oracle(n_mels, kind):
    audio = batch_audio(kind, 3, seed=11)
    got = run_mel(audio, n_mels)
    for i in range(3):
        ref = omel.log_mel(audio[i].astype(np.float64), n_mels)
        err = np.abs(got[i] - ref).max()
        assert err <= MEL_TOL, (i, err)


def test_mel_silence_and_edge_cases():
    audio = np.zeros((2, 480000), np.float32)
    audio[1, 240000] = 1.0          # a single click: energy in ~3 frames only
    got = run_mel(audio, 128)
    assert (got[0] == -1.5).all()
    ref = omel.log_mel(audio[1].astype(np.float64), 128)
    assert np.abs(got[1] - ref).max() <= MEL_TOL


def test_mel_full_batch_sampled():
    """The 64-chunk mel workload; the oracle checks a sample of whole chunks."""
    audio = batch_audio("pink", 64, seed=2)
    got = run_mel(audio, 128)
    for i in (0, 17, 63):
        ref = omel.log_mel(audio[i].astype(np.float64), 128)
        assert np.abs(got[i] - ref).max() <= MEL_TOL, i
    # chunk independence: chunk 17 alone gives the same bits
    alone = run_mel(audio[17:18].copy(), 128)
    assert np.array_equal(alone[0], got[17])


def _bf16(x):
    return round_to_bf16(np.asarray(x, np.float32))


@pytest.mark.parametrize("M,N,K", [(300, 320, 640), (128, 256, 64), (3000, 1280, 1280), (37, 3840, 1280),
                                   (1, 64, 128), (5, 51866 - 51866 % 8, 384)])
def test_gemm_bf16_matches_oracle(M, N, K):
    rng = np.random.default_rng(M * 7 + N)
    a = _bf16(rng.normal(size=(M, K)))
    b = _bf16(rng.normal(size=(N, K)) * 0.05)
    bias = rng.normal(size=N).astype(np.float32)
    A = torch.from_numpy(a).to(torch.bfloat16).cuda()
    B = torch.from_numpy(b).to(torch.bfloat16).cuda()
    C = torch.empty(M, N, device="cuda")
    wb.wb_gemm(A, B, C, bias=torch.from_numpy(bias).cuda())
    wb.wb_sync_status()
    ref = omodel.Linear(b, bias)(a)
    got = C.cpu().numpy()
    scale = np.abs(a).max() * np.abs(b).max() * np.sqrt(K)
    assert np.abs(got - ref).max() <= 1e-5 * scale + 1e-6


def test_gemm_bf16_gelu_bf16_out():
    rng = np.random.default_rng(3)
    M, N, K = 500, 512, 256
    a, b = _bf16(rng.normal(size=(M, K))), _bf16(rng.normal(size=(N, K)) * 0.05)
    bias = rng.normal(size=N).astype(np.float32)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    wb.wb_gemm(torch.from_numpy(a).to(torch.bfloat16).cuda(), torch.from_numpy(b).to(torch.bfloat16).cuda(), C,
               bias=torch.from_numpy(bias).cuda(), gelu=True)
    wb.wb_sync_status()
    ref = omodel.gelu(omodel.Linear(b, bias)(a))
    got = C.float().cpu().numpy()
    assert np.abs(got - ref).max() <= 2 ** -8 * np.abs(ref).max() + 1e-3


@pytest.mark.parametrize("M,N,K", [(200, 256, 256), (1500, 1280, 1280), (3, 5120, 1280)])
def test_gemm_e4m3_matches_oracle(M, N, K):
    rng = np.random.default_rng(N + K)
    x = rng.normal(size=(M, K)).astype(np.float32)
    w = (rng.normal(size=(N, K)) * 0.02).astype(np.float32)
    lin = omodel.Linear(w, np.zeros(N), fp8=True)
    ref = lin(x)
    # identical codes and scales on both sides: the oracle's own quantisation
    amax = np.abs(x).max(axis=1)
    sx = np.array([oe4m3.scale_of(a) for a in amax], np.float32)
    qx = np.stack([oe4m3.quantise(x[i], sx[i]) for i in range(M)])
    A = torch.from_numpy(qx).cuda()
    B = torch.from_numpy(lin.w_codes).cuda()
    C = torch.empty(M, N, device="cuda")
    wb.wb_gemm(A, B, C, row_scale=torch.from_numpy(sx).cuda(),
               col_scale=torch.full((N,), float(lin.w_scale), device="cuda"))
    wb.wb_sync_status()
    got = C.cpu().numpy()
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max() * np.sqrt(K / 64) + 1e-7


def _sample_rows(M, seed):
    rng = np.random.default_rng(seed)
    # both ends of every 256-row pair, the ragged last tile, and random rows
    rows = {0, 127, 128, 255, M - 1, M - 2, (M // 128) * 128, max(0, (M // 128) * 128 - 1)}
    rows.update(rng.integers(0, M, 40).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < M))


@pytest.mark.parametrize("M,N,K", [(9000, 5120, 1280), (4100, 3840, 640)])
def test_gemm_pair_bf16_matches_oracle(M, N, K):
    """Large plain GEMMs run on CTA pairs (cta_group::2 MMAs over 256-row
    tiles, each CTA loading its own half of A and of B): an odd number of
    128-row tiles leaves the last pair's second half empty."""
    rng = np.random.default_rng(M + N)
    a = _bf16(rng.normal(size=(M, K)))
    b = _bf16(rng.normal(size=(N, K)) * 0.05)
    bias = rng.normal(size=N).astype(np.float32)
    C = torch.empty(M, N, device="cuda")
    wb.wb_gemm(torch.from_numpy(a).to(torch.bfloat16).cuda(), torch.from_numpy(b).to(torch.bfloat16).cuda(), C,
               bias=torch.from_numpy(bias).cuda())
    wb.wb_sync_status()
    rows = _sample_rows(M, 1)
    ref = omodel.Linear(b, bias)(a[rows])
    got = C.cpu().numpy()[rows]
    scale = np.abs(a).max() * np.abs(b).max() * np.sqrt(K)
    assert np.abs(got - ref).max() <= 1e-5 * scale + 1e-6


def test_gemm_pair_e4m3_matches_oracle():
    M, N, K = 9000, 3840, 1280
    rng = np.random.default_rng(11)
    x = rng.normal(size=(M, K)).astype(np.float32)
    w = (rng.normal(size=(N, K)) * 0.02).astype(np.float32)
    lin = omodel.Linear(w, np.zeros(N), fp8=True)
    rows = _sample_rows(M, 2)
    ref = lin(x[rows])
    amax = np.abs(x).max(axis=1)
    sx = np.array([oe4m3.scale_of(v) for v in amax], np.float32)
    qx = oe4m3.encode((x * (np.float32(1.0) / sx)[:, None]).astype(np.float32))
    C = torch.empty(M, N, device="cuda")
    wb.wb_gemm(torch.from_numpy(qx).cuda(), torch.from_numpy(lin.w_codes).cuda(), C,
               row_scale=torch.from_numpy(sx).cuda(), col_scale=torch.full((N,), float(lin.w_scale), device="cuda"))
    wb.wb_sync_status()
    got = C.cpu().numpy()[rows]
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max() * np.sqrt(K / 64) + 1e-7


def test_gemm_pair_gelu_bf16_out_ragged_n():
    M, N, K = 12000, 1000, 256
    rng = np.random.default_rng(5)
    a, b = _bf16(rng.normal(size=(M, K))), _bf16(rng.normal(size=(N, K)) * 0.05)
    bias = rng.normal(size=N).astype(np.float32)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    wb.wb_gemm(torch.from_numpy(a).to(torch.bfloat16).cuda(), torch.from_numpy(b).to(torch.bfloat16).cuda(), C,
               bias=torch.from_numpy(bias).cuda(), gelu=True)
    wb.wb_sync_status()
    rows = _sample_rows(M, 3)
    ref = omodel.gelu(omodel.Linear(b, bias)(a[rows]))
    got = C.float().cpu().numpy()[rows]
    assert np.abs(got - ref).max() <= 2 ** -8 * np.abs(ref).max() + 1e-3


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("n", [1, 1000, 1 << 20])
def test_quantiser_codes_bit_exact(bf16, n):
    rng = np.random.default_rng(n)
    x = rng.normal(0, 3, size=n).astype(np.float32)
    if bf16:
        x = _bf16(x)
    X = torch.from_numpy(x).cuda()
    if bf16:
        X = X.to(torch.bfloat16)
    codes = torch.empty(n, dtype=torch.uint8, device="cuda")
    scale = torch.empty(1, device="cuda")
    wb.wb_quantise_e4m3(X, codes, scale)
    out = torch.empty(n, device="cuda")
    wb.wb_dequantise_e4m3(codes, scale, out)
    wb.wb_sync_status()
    ref_codes, ref_scale = oe4m3.quantise_tensor(x)
    assert np.float32(scale.item()) == ref_scale
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    assert np.array_equal(out.cpu().numpy(), (oe4m3.decode(ref_codes) * np.float64(ref_scale)).astype(np.float32))


@pytest.mark.parametrize("n_groups,group_elems", [(5, 1500 * 64), (3, 4), (2, 1500 * 1284), (1, 1 << 20)])
def test_group_quantiser_bit_exact(n_groups, group_elems):
    """One E4M3 scale per group (the mixed_fp8 encoder's per-chunk tensors):
    codes and scales bit-exact against the oracle's per-tensor quantiser on
    each group, including an all-zero group and a group whose amax is one
    outlier."""
    rng = np.random.default_rng(n_groups * 31 + group_elems % 997)
    x = rng.normal(0, 2.0, size=(n_groups, group_elems)).astype(np.float32)
    if n_groups > 1:
        x[1] = 0.0
    if n_groups > 2:
        x[2] *= 1e-3
        x[2, group_elems // 2] = -300.0
    X = torch.from_numpy(x.reshape(-1)).cuda()
    codes = torch.full((x.size,), 0xAA, dtype=torch.uint8, device="cuda")
    scales = torch.full((n_groups,), -1.0, device="cuda")
    wb.wb_quantise_e4m3_groups(X, n_groups, codes, scales)
    wb.wb_sync_status()
    got_c = codes.cpu().numpy().reshape(n_groups, group_elems)
    got_s = scales.cpu().numpy()
    for g in range(n_groups):
        ref_c, ref_s = oe4m3.quantise_tensor(x[g])
        assert np.float32(got_s[g]) == ref_s, g
        assert np.array_equal(got_c[g], ref_c), g


def test_gemm_bounded_wait_runs_out_and_recovers():
    """Failure detection without a fault: the GEMM's first pipeline wait is
    made to run out (a 1 ms wait on a barrier nothing arrives on).  The kernel
    records a timeout, drains its own copies, frees its tensor memory and
    exits; wb_sync_status reports WB_ERR_TIMEOUT, and the next call on the
    same context computes the right product."""
    rng = np.random.default_rng(77)
    M, N, K = 256, 512, 256
    a, b = _bf16(rng.normal(size=(M, K))), _bf16(rng.normal(size=(N, K)) * 0.05)
    A = torch.from_numpy(a).to(torch.bfloat16).cuda()
    B = torch.from_numpy(b).to(torch.bfloat16).cuda()
    C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    wb.wb_sync_status()
    wb.wb_debug_stall_next_gemm(1_000_000)
    wb.wb_gemm(A, B, C, gelu=True)
    with pytest.raises(wb.WBError) as err:
        wb.wb_sync_status()
    assert err.value.status == -6, err.value
    wb.wb_sync_status()                     # the error word was cleared
    wb.wb_gemm(A, B, C, gelu=True)
    wb.wb_sync_status()
    ref = omodel.gelu(omodel.Linear(b, np.zeros(N))(a))
    assert np.abs(C.float().cpu().numpy() - ref).max() <= 2 ** -8 * np.abs(ref).max() + 1e-3
