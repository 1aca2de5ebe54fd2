"""Beam search on the GPU against the oracle.

A beam step is a discrete choice, and the GPU's logits differ from the
oracle's in the last bits, so the GPU is checked step by step on its own
hypotheses (the unique part of the result given them): before each
selection the oracle recomputes every hypothesis's running score and its
next-token log-probabilities by teacher forcing; the GPU's running scores
must agree within the logit tolerance, the continuations it keeps must be a
best-`beams` set of the oracle's candidates up to that tolerance, and its
token rows must be the parents' rows plus the chosen tokens (exact).
"""
import numpy as np
import pytest
import torch

import whisper_encoder_decoder_log_b300 as wb
from oracle import mel as omel
from oracle import model as omodel
from synth import ModelDims, batch_audio, forced_prefix
from tests.gpu_util import GpuModel

pytestmark = pytest.mark.gpu

DIMS = ModelDims("beam-384", 128, 384, 6, 1536, 1, 2, 51865)


def _oracle_state(hist, P, enc, W):
    """Running score of a token history and the log-probabilities of its next token."""
    logits, _ = omodel.decode_teacher_forced(np.asarray(hist), enc, W, DIMS, kv_fp8=True, act16=True)
    lp = omodel.log_softmax(logits)
    score = sum(lp[q, hist[q + 1]] for q in range(P - 1, len(hist) - 1))
    return score, lp[-1]


def _check_selection(before_rows, before_scores, after_rows, after_scores, parents, t, K, P, enc, W, tol):
    """One chunk's selection at position t (the token for t + 1)."""
    live = np.isfinite(before_scores)
    cand = np.full((K, DIMS.vocab), -np.inf)
    for b in range(K):
        if not live[b]:
            continue
        sc, lp = _oracle_state(before_rows[b, :t + 1], P, enc, W)
        assert abs(sc - before_scores[b]) <= tol, (t, b, sc, before_scores[b])
        cand[b] = sc + lp
    flat = np.sort(cand.reshape(-1))[::-1]
    kth = flat[K - 1]
    chosen = set()
    for j in range(K):
        p, v = int(parents[j]), int(after_rows[j, t + 1])
        assert np.array_equal(after_rows[j, :t + 1], before_rows[p, :t + 1])     # parent's row, exact
        assert cand[p, v] >= kth - 2 * tol, (t, j, cand[p, v], kth)             # a best-K continuation
        assert abs(after_scores[j] - cand[p, v]) <= tol, (t, j, after_scores[j], cand[p, v])
        chosen.add((p, v))
    worst_kept = min(cand[p, v] for p, v in chosen)
    better = np.argwhere(cand > worst_kept + 2 * tol)
    assert all((int(b), int(v)) in chosen for b, v in better)                  # nothing clearly better left out


def test_beam_search_steps_match_oracle():
    K, P = 4, 4
    m = GpuModel(DIMS, wb.PREC_BF16, wb.KV_FP8_SELF, seed=17)
    audio = batch_audio("sine", 3, seed=91)
    enc = m.encode(m.mel(audio))
    lens = np.array([18, 13, 9], np.int32)
    B = lens.size
    prefix = forced_prefix(7, DIMS.vocab)
    tok = torch.zeros(B * K, 448, dtype=torch.int32, device="cuda")
    tok[:, :P] = torch.from_numpy(np.tile(prefix, (B * K, 1))).cuda()
    ws = torch.empty(wb.wb_decoder_workspace_size_beams(m.h, lens, K), dtype=torch.uint8, device="cuda")
    dec = wb.wb_decoder_init_beams(m.h, lens, K, enc, tok, ws)
    scores = torch.empty(B * K, device="cuda")
    parents = torch.empty(B * K, dtype=torch.int32, device="cuda")
    ref_enc = [omodel.encode(omel.log_mel(audio[c].astype(np.float64), 128), m.W, DIMS, act16=True) for c in range(B)]
    # the prefix pass makes the first selection (position P - 1) from the prefix alone
    before_rows = tok.cpu().numpy().copy()
    before_scores = np.tile(np.array([0.0] + [-np.inf] * (K - 1)), B)
    wb.wb_decode_prefix(dec, P)
    wb.wb_decoder_beam_scores(dec, scores)
    rows = tok.cpu().numpy().copy()
    sc = scores.cpu().numpy().astype(np.float64)
    first = True
    steps = 0
    for t in range(P - 1, int(lens.max()) - 1):
        n_act = int((lens > t + 1).sum())
        if not first:
            before_rows, before_scores = rows, sc
            wb.wb_decode_step_beams(dec, n_act, scores, parents)
            rows = tok.cpu().numpy().copy()
            sc = scores.cpu().numpy().astype(np.float64)
        par = parents.cpu().numpy() if not first else np.zeros(B * K, np.int32)
        steps += 1
        tol = 2e-2 + 2e-3 * steps
        for c in range(n_act):
            r = slice(c * K, (c + 1) * K)
            if first:   # every new hypothesis continues the prefix (parent 0)
                assert (rows[r, :P] == prefix).all()
                cand0 = _oracle_state(before_rows[c * K, :P], P, ref_enc[c], m.W)[1]
                top = np.sort(cand0)[::-1]
                for j in range(K):
                    v = int(rows[c * K + j, P])
                    assert cand0[v] >= top[K - 1] - 2 * tol and abs(sc[c * K + j] - cand0[v]) <= tol
            else:
                _check_selection(before_rows[r], before_scores[r], rows[r], sc[r], par[r], t, K, P, ref_enc[c], m.W, tol)
        first = False
    best = torch.full((B, 448), -1, dtype=torch.int32, device="cuda")
    best_sc = torch.empty(B, device="cuda")
    wb.wb_decoder_best_beams(dec, best, best_sc)
    wb.wb_sync_status(m.h)
    wb.wb_decoder_destroy(dec)
    best, best_sc = best.cpu().numpy(), best_sc.cpu().numpy()
    for c in range(B):
        L = int(lens[c])
        j = int(np.argmax(sc[c * K:(c + 1) * K]))
        assert np.array_equal(best[c, :L], rows[c * K + j, :L]) and (best[c, L:] == -1).all()
        ref_score, _ = _oracle_state(best[c, :L], P, ref_enc[c], m.W)
        assert abs(best_sc[c] - ref_score) <= 2e-2 + 2e-3 * (L - P)
    m.close()
