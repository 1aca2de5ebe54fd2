"""Oracle: chunk table and wave packing (integer bookkeeping only).

[WB] "Batch Transcription": all 30-second chunks of several requests are fused
into one generate pass to fill the GPU's memory; "VRAM usage guide": memory
grows linearly with the number of chunks in flight (a fixed per-chunk cost plus
the weights); "Serving at Scale": concurrent requests are grouped into GPU
batches.

Readings:
  * chunk c of the batch is (request r, index k) in request order, then index
    order; it holds min(480000, samples_r - 480000 k) real samples;
  * a chunk's decode state costs, per decoder layer, the cross-attention K
    and V over 1500 encoder positions (bf16, or float8 when the cross K/V are
    stored as E4M3) plus its float8 self-attention K and V over its own decode
    length L_c, plus its token row (448 int32);
  * overlapping windows: chunk k of a request starts k (480000 - overlap)
    samples in; a request's transcript joins its chunks' tokens, dropping the
    longest prefix of each chunk that repeats the end of the text so far;
  * several GPUs: contiguous ranges of chunks in request order, balanced on
    decode length plus a fixed per-chunk share for the mel and encoder (each
    chunk is transcribed on exactly one GPU; no step needs another GPU's data);
  * waves: chunks sorted by decode length, longest first (ties by chunk
    index), are packed greedily in that order; a new wave opens when the next
    chunk would push the running total of per-chunk bytes past the budget.
    Within a wave the chunks keep that order, so the chunks still decoding at
    any step form a prefix of the wave.
"""
from __future__ import annotations

import numpy as np

CHUNK = 480000
N_CTX = 1500
MAX_POS = 448


def chunk_table(req_samples, overlap: int = 0):
    """(req_of_chunk, index_in_req, valid_samples) as int32 arrays; chunk k of
    a request starts at k (480000 - overlap) (see oracle.mel.split_into_chunks)."""
    stride = CHUNK - int(overlap)
    req, idx, valid = [], [], []
    for r, s in enumerate(np.asarray(req_samples, dtype=np.int64)):
        n = 1 + (max(0, int(s) - CHUNK) + stride - 1) // stride
        for k in range(n):
            req.append(r)
            idx.append(k)
            valid.append(int(min(CHUNK, s - stride * k)))
    return (np.array(req, np.int32), np.array(idx, np.int32), np.array(valid, np.int32))


def stitch(rows):
    """One request's transcript (token ids) from its chunks' generated tokens,
    in chunk order.  Overlapping windows transcribe the shared audio twice, so
    the next chunk's tokens are joined after removing the longest prefix of
    them that equals a suffix of the transcript so far; with no such prefix
    the tokens are simply appended (token ids only: no timestamps)."""
    out = []
    for row in rows:
        row = [int(t) for t in row]
        k = min(len(out), len(row))
        while k > 0 and out[len(out) - k:] != row[:k]:
            k -= 1
        out.extend(row[k:])
    return np.array(out, np.int32)


def chunk_state_bytes(d_model: int, dec_layers: int, length: int, cross_bytes: int = 2) -> int:
    cross = dec_layers * 2 * N_CTX * d_model * cross_bytes
    self_kv = dec_layers * 2 * int(length) * d_model
    return cross + self_kv + MAX_POS * 4


def plan_waves(chunk_len, d_model: int, dec_layers: int, budget_bytes: int, cross_bytes: int = 2):
    """List of waves, each an int32 array of chunk indices in decode order."""
    chunk_len = np.asarray(chunk_len, dtype=np.int64)
    order = sorted(range(chunk_len.size), key=lambda c: (-int(chunk_len[c]), c))
    waves, cur, used = [], [], 0
    for c in order:
        b = chunk_state_bytes(d_model, dec_layers, int(chunk_len[c]), cross_bytes)
        if b > budget_bytes:
            raise ValueError("one chunk exceeds the wave budget")
        if cur and used + b > budget_bytes:
            waves.append(np.array(cur, np.int32))
            cur, used = [], 0
        cur.append(c)
        used += b
    if cur:
        waves.append(np.array(cur, np.int32))
    return waves


SHARD_CHUNK_BASE = 48


def shard_ranges(chunk_len, world: int):
    """Contiguous chunk ranges of one batch for ``world`` GPUs, balanced on
    work: chunk c weighs chunk_len[c] + 48 (its decode positions plus the mel
    and encoder, about 48 positions' worth); range r starts at the first chunk
    whose preceding work w has w * world >= r * total.  Returns first[0..world]
    with first[0] = 0 and first[world] = n_chunks."""
    w = [int(x) + SHARD_CHUNK_BASE for x in np.asarray(chunk_len)]
    total = sum(w)
    first = [0]
    for r in range(1, world):
        acc, pick = 0, len(w)
        for c in range(len(w)):
            if acc * world >= r * total:
                pick = c
                break
            acc += w[c]
        first.append(pick)
    first.append(len(w))
    return first


def shard_requests(req_offsets, req_samples, c0: int, c1: int):
    """The requests overlapping chunks [c0, c1), cut at chunk boundaries:
    (offsets, samples) into the same audio buffer."""
    req, idx, valid = chunk_table(req_samples)
    offs, samples = [], []
    c = c0
    while c < c1:
        r, e = int(req[c]), c
        while e < c1 and req[e] == r:
            e += 1
        s0 = int(idx[c]) * CHUNK
        s1 = s0 + sum(int(v) for v in valid[c:e])
        offs.append(int(req_offsets[r]) + s0)
        samples.append(s1 - s0)
        c = e
    return np.array(offs, np.int64), np.array(samples, np.int64)
