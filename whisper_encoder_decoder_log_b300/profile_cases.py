"""Small, self-contained runs of single kernel kinds for profiling.

    python -m whisper_encoder_decoder_log_b300.profile_cases <case> [--iters N]

Each case builds its inputs (seeded, synthetic), runs the kernel kind a few
times through the C ABI and exits; a profiler can then select one launch of
the kernel of interest.  Sizes are the workloads' own per-launch shapes with a
small batch, so a capture holds well under a few GB of device memory.

  mel     wb_mel on 64 chunks (the mel workload itself, 221 MB in + out)
  gemm    encoder FC1-shaped bf16 GEMM, 24000 x 5120 x 1280 (16 chunks)
  gemm8   the same GEMM in E4M3
  decode  large-v3-turbo decoder over 32 chunks: prefix + 8 greedy steps
          (cross-attention over 1500 bf16 rows per chunk and head, causal
          self-attention over the E4M3 cache, few-row GEMMs)
  decode8 large-v3 decoder layers in mixed_fp8 (4 of the 32) over --chunks
          chunks (default 512): prefix + --steps greedy steps through the
          captured step graphs, the launch pattern of the serving batch's
          decode; the encoder states are random; --kv 2 stores the cross
          K/V in E4M3 as well
  flash   encoder self-attention over 16 chunks x 20 heads
  small   decode-step GEMMs of the serving batch (swapped form): --rows
          activation rows (default 440) through the E4M3 QKV (3840 x 1280),
          FC1 (5120 x 1280) and FC2 (1280 x 5120) shapes

--time prints the mean CUDA-event time per iteration (after one untimed
iteration) and the achieved rate of the case's algorithmic work.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import synth
    import whisper_encoder_decoder_log_b300 as wb

    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["mel", "gemm", "gemm8", "decode", "decode8", "flash", "small"])
    ap.add_argument("--time", action="store_true")
    ap.add_argument("--rows", type=int, default=440)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--chunks", type=int, default=512)
    ap.add_argument("--steps", type=int, default=8)
    ap.add_argument("--kv", type=int, default=1, choices=[1, 2])
    a = ap.parse_args()
    dev = "cuda"

    def timed(fn, work, unit):
        """Run fn a.iters times; with --time, report the mean of all but the first."""
        fn()
        if not a.time:
            for _ in range(a.iters - 1):
                fn()
            return
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(1, a.iters - 1)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        scale = 1e12 if unit == "TFLOP/s" else 1e9
        print(f"profile case {a.case}: {ms:.4f} ms per iteration, {work / (ms / 1e3) / scale:.1f} {unit}")

    if a.case == "mel":
        audio = torch.from_numpy(synth.batch_audio("pink", 64, 0)).to(dev)
        mel = torch.empty(64, 128, 3000, device=dev)
        timed(lambda: wb.wb_mel(audio, 128, mel), 64 * (480000 * 4 + 128 * 3000 * 4), "GB/s")
    elif a.case in ("gemm", "gemm8"):
        M, N, K = 24000, 5120, 1280
        A = torch.randn(M, K, device=dev)
        B = torch.randn(N, K, device=dev) * 0.02
        C = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        if a.case == "gemm":
            A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
            timed(lambda: wb.wb_gemm(A, B, C), 2.0 * M * N * K, "TFLOP/s")
        else:
            qa = torch.empty(M * K, dtype=torch.uint8, device=dev)
            qb = torch.empty(N * K, dtype=torch.uint8, device=dev)
            sa = torch.empty(1, device=dev)
            sb = torch.empty(1, device=dev)
            wb.wb_quantise_e4m3(A.reshape(-1), qa, sa)
            wb.wb_quantise_e4m3(B.reshape(-1), qb, sb)
            rs = sa.expand(M).contiguous()
            cs = sb.expand(N).contiguous()
            timed(lambda: wb.wb_gemm(qa.view(M, K), qb.view(N, K), C, row_scale=rs, col_scale=cs), 2.0 * M * N * K,
                  "TFLOP/s")
    elif a.case == "small":
        R = a.rows
        X = torch.randn(R, 5120, device=dev)
        qx = torch.empty(R * 5120, dtype=torch.uint8, device=dev)
        sx = torch.empty(1, device=dev)
        wb.wb_quantise_e4m3(X.reshape(-1), qx, sx)
        rs = sx.expand(R).contiguous()
        shapes = [(3840, 1280), (5120, 1280), (1280, 5120)]
        ws, outs, css = [], [], []
        for N, K in shapes:
            Wt = torch.randn(N, K, device=dev) * 0.02
            qw = torch.empty(N * K, dtype=torch.uint8, device=dev)
            sw = torch.empty(1, device=dev)
            wb.wb_quantise_e4m3(Wt.reshape(-1), qw, sw)
            ws.append(qw.view(N, K))
            css.append(sw.expand(N).contiguous())
            outs.append(torch.empty(R, N, device=dev))

        def run():
            for (N, K), qw, cs, out in zip(shapes, ws, css, outs):
                wb.wb_gemm(qx[:R * K].view(R, K), qw, out, row_scale=rs, col_scale=cs)
        # bytes: E4M3 weights + E4M3 activations + fp32 outputs
        work = sum(N * K + R * K + 4 * R * N for N, K in shapes)
        timed(run, work, "GB/s")
    elif a.case == "decode8":
        dims = synth.ModelDims("large-v3-dec4", 128, 1280, 20, 5120, 1, 4, 51866)
        desc = wb.make_desc(dims, wb.PREC_MIXED_FP8, a.kv)
        buf = wb.pack_weights(desc, synth.make_weights(dims, 0, bf16=True))
        torch.cuda.synchronize()
        model = wb.wb_model_create(desc, buf)
        B = a.chunks
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        enc = torch.randn(B, 1500, 1280, device=dev, generator=g).to(torch.bfloat16)
        lens = np.full(B, 4 + a.steps + 1, np.int32)
        tok = torch.zeros(B, 448, dtype=torch.int32, device=dev)
        tok[:, :4] = torch.from_numpy(synth.forced_prefix(0, dims.vocab)).to(dev)
        dws = torch.empty(wb.wb_decoder_workspace_size(model, lens), dtype=torch.uint8, device=dev)
        for _ in range(a.iters):
            d = wb.wb_decoder_init(model, lens, enc, tok, dws)
            wb.wb_decode_prefix(d, 4)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for i in range(a.steps):
                if i == min(2, a.steps - 1):
                    e0.record()
                wb.wb_decode_step(d, B)
            e1.record()
            torch.cuda.synchronize()
            if a.time and a.steps > 2:
                print(f"profile case decode8: {e0.elapsed_time(e1) * 1e3 / (a.steps - 2):.1f} us per decode step "
                      f"({B} chunks, graph replay)")
            wb.wb_decoder_destroy(d)
        wb.wb_sync_status(model)
        wb.wb_model_destroy(model)
    else:
        layers = (1, 4) if a.case == "decode" else (1, 0)
        dims = synth.ModelDims("turbo", 128, 1280, 20, 5120, layers[0], layers[1], 51866)
        desc = wb.make_desc(dims, wb.PREC_BF16, True)
        buf = wb.pack_weights(desc, synth.make_weights(dims, 0, bf16=True))
        torch.cuda.synchronize()
        model = wb.wb_model_create(desc, buf)
        B = 32 if a.case == "decode" else 16
        audio = torch.from_numpy(synth.batch_audio("sine", B, 0)).to(dev)
        mel = torch.empty(B, 128, 3000, device=dev)
        wb.wb_mel(audio, 128, mel)
        ws = torch.empty(wb.wb_encode_workspace_size(model, B), dtype=torch.uint8, device=dev)
        enc = torch.empty(B, 1500, 1280, dtype=torch.bfloat16, device=dev)
        for _ in range(a.iters if a.case == "flash" else 1):
            wb.wb_encode(model, mel, enc, ws)
        if a.case == "decode":
            lens = np.full(B, 16, np.int32)
            tok = torch.zeros(B, 448, dtype=torch.int32, device=dev)
            tok[:, :4] = torch.from_numpy(synth.forced_prefix(0, dims.vocab)).to(dev)
            dws = torch.empty(wb.wb_decoder_workspace_size(model, lens), dtype=torch.uint8, device=dev)
            for _ in range(a.iters):
                d = wb.wb_decoder_init(model, lens, enc, tok, dws)
                wb.wb_decode_prefix(d, 4)
                for _ in range(8):
                    wb.wb_decode_step(d, B)
                wb.wb_decoder_destroy(d)
        wb.wb_sync_status(model)
        wb.wb_model_destroy(model)
    torch.cuda.synchronize()
    wb.wb_sync_status()
    print(f"profile case {a.case}: ok")


if __name__ == "__main__":
    main()
