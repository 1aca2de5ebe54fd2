"""Helpers shared by the GPU parity tests: model construction from the seeded
weights and end-to-end calls through the C ABI."""
import numpy as np
import torch

import whisper_encoder_decoder_log_b300 as wb
from synth import make_weights


class GpuModel:
    def __init__(self, dims, precision, kv_fp8, seed, weights=None):
        self.dims = dims
        self.precision = precision
        self.desc = wb.make_desc(dims, precision, kv_fp8)
        bf16 = precision != wb.PREC_FP32
        self.W = weights if weights is not None else make_weights(dims, seed, bf16=bf16)
        self.buf = wb.pack_weights(self.desc, self.W)
        torch.cuda.synchronize()
        self.h = wb.wb_model_create(self.desc, self.buf)

    @property
    def act_dtype(self):
        return torch.float32 if self.precision == wb.PREC_FP32 else torch.bfloat16

    def mel(self, audio_np):
        a = torch.from_numpy(np.ascontiguousarray(audio_np, np.float32)).cuda()
        out = torch.empty(a.shape[0], self.dims.n_mels, 3000, device="cuda")
        wb.wb_mel(a, self.dims.n_mels, out)
        return out

    def encode(self, mel):
        B = mel.shape[0]
        ws = torch.empty(wb.wb_encode_workspace_size(self.h, B), dtype=torch.uint8, device="cuda")
        enc = torch.empty(B, 1500, self.dims.d_model, dtype=self.act_dtype, device="cuda")
        wb.wb_encode(self.h, mel, enc, ws)
        return enc

    def decode(self, enc, prefix_tokens, chunk_len, steps=0, want_logits=True):
        """Prefix pass with P = prefix_tokens.shape[1], then `steps` greedy steps.

        Returns (tokens [B,448] int32 numpy, list of logits arrays: the prefix
        logits [B,P,V] then one [n_active,V] per step)."""
        B, P = prefix_tokens.shape
        tok = torch.zeros(B, 448, dtype=torch.int32, device="cuda")
        tok[:, :P] = torch.from_numpy(np.ascontiguousarray(prefix_tokens, np.int32)).cuda()
        ws = torch.empty(wb.wb_decoder_workspace_size(self.h, chunk_len), dtype=torch.uint8, device="cuda")
        dec = wb.wb_decoder_init(self.h, chunk_len, enc, tok, ws)
        outs = []
        V = self.dims.vocab
        lg = torch.empty(B, P, V, device="cuda") if want_logits else None
        wb.wb_decode_prefix(dec, P, lg)
        if want_logits:
            outs.append(lg.cpu().numpy())
        for i in range(steps):
            t = P + i
            n_act = int((np.asarray(chunk_len) > t + 1).sum())
            if n_act == 0:
                break
            lg = torch.empty(n_act, V, device="cuda") if want_logits else None
            wb.wb_decode_step(dec, n_act, lg)
            if want_logits:
                outs.append(lg.cpu().numpy())
        wb.wb_sync_status(self.h)
        wb.wb_decoder_destroy(dec)
        return tok.cpu().numpy(), outs

    def close(self):
        wb.wb_model_destroy(self.h)


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def greedy_choice_check(ref, chosen, tol=2e-2):
    """Greedy decisions against the oracle's logits (several correct results:
    compare what is unique, check that the rest is valid).

    ref [n, V] oracle logits, chosen [n] the GPU's token ids.  A position
    whose oracle top-2 gap is at least tol (the logit bound) has one valid
    greedy token, the oracle's argmax; at a near-tie any token within tol of
    the oracle's maximum is a valid choice.  Returns (agreeing unique
    positions, unique positions, near-ties, near-ties outside tol)."""
    ref = np.asarray(ref, np.float64)
    chosen = np.asarray(chosen).astype(np.int64)
    top2 = np.sort(ref, axis=1)[:, -2:]
    unique = (top2[:, 1] - top2[:, 0]) >= tol
    agree = int((chosen[unique] == np.argmax(ref[unique], axis=1)).sum())
    picked = ref[np.arange(ref.shape[0]), chosen]
    bad = int(((ref.max(axis=1) - picked) > tol)[~unique].sum())
    return agree, int(unique.sum()), int((~unique).sum()), bad
