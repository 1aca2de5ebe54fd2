"""The N > 1 path on CPU, two gloo ranks.

One batch is split across the ranks by contiguous chunk ranges
(wb_shard_batch, host only); every rank transcribes its share with no
collective on the data path, the token rows are gathered on the host
afterwards, and the whole-job rate counts the audio of all ranks over the
slowest rank's time (the only collective of the timed region is the
max-over-ranks of the step time).  Here the ranks are CPU processes with the
gloo backend and the per-rank transcriber is a host stub.
"""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 180.0][rank]                       # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms)
    rate = bench.whole_job_rate(960.0, world, m)
    q.put((rank, m, rate))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_reduce_to_the_slowest():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, rate in res:
        assert m == 180.0
        assert rate == pytest.approx(960.0 * 2 / 0.180)


def test_single_process_needs_no_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(42.0) == 42.0
    assert bench.whole_job_rate(30.0, 1, 1000.0) == 30.0


# ----------------------------------------------------------------- one batch over two ranks

def _stub_transcribe(audio, req_offsets, req_samples, chunk_len, vocab=51866):
    """Stands in for wb_transcribe_batch on the host: each chunk's token row is
    a deterministic function of its own samples and length (the one property
    of the real path the split relies on: a chunk's result depends on that
    chunk alone)."""
    from oracle import plan as oplan
    req, idx, valid = oplan.chunk_table(req_samples)
    tok = np.full((req.size, 448), -1, np.int32)
    for c in range(req.size):
        s0 = int(req_offsets[req[c]]) + int(idx[c]) * oplan.CHUNK
        x = audio[s0:s0 + int(valid[c])].astype(np.float64)
        h = int(abs(x.sum()) * 1e6 + (x * x).sum() * 1e3 + valid[c]) % vocab
        L = int(chunk_len[c])
        tok[c, :L] = (h + np.arange(L)) % vocab
    return tok


def _shard_worker(rank, world, port, q):
    import whisper_encoder_decoder_log_b300 as wb
    from synth import serving_requests
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sb = serving_requests(9, n_req=6, min_s=40.0, max_s=150.0)      # one global batch, the same on every rank
    offs, samples, c0, cn = wb.wb_shard_batch(sb.req_offsets, sb.req_samples, sb.chunk_len, world, rank)
    mine = _stub_transcribe(sb.audio, offs, samples, sb.chunk_len[c0:c0 + cn]) if cn else np.zeros((0, 448), np.int32)
    parts = [None] * world
    dist.all_gather_object(parts, (c0, cn, mine))                    # host-side gather of token rows
    if rank == 0:
        n = sb.chunk_len.size
        owner = np.full(n, -1)
        full = np.full((n, 448), -7, np.int32)
        for r, (a, k, rows) in enumerate(parts):
            assert (owner[a:a + k] == -1).all()                      # no chunk on two ranks
            owner[a:a + k] = r
            full[a:a + k] = rows
        ref = _stub_transcribe(sb.audio, sb.req_offsets, sb.req_samples, sb.chunk_len)
        q.put(((owner >= 0).all(), bool(np.array_equal(full, ref)), [p[1] for p in parts]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_one_batch_split_over_two_gloo_ranks_gathers_to_the_single_rank_result():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30500 + os.getpid() % 1000
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(150)
        assert p.exitcode == 0
    covered, same, counts = q.get(timeout=10)
    assert covered and same
    assert all(c > 0 for c in counts)
