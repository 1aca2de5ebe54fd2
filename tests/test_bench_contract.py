"""bench.py's reference arm (the oracle on the host cores) prints one JSON
line with the keys of the benchmark contract; it needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = dict(os.environ)
    env.setdefault("OMP_NUM_THREADS", "4")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "c1",
                          "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_reference_arm_finishes_the_serving_workload_at_driver_step_counts():
    """The serving-batch reference arm with 20 timed and 5 warm-up steps ends
    well inside the driver's limit: every step is one bounded oracle sample of
    a few seconds, and only the sampled chunk's weights are generated."""
    env = dict(os.environ)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "c5",
                          "--steps", "20", "--warmup", "5"], capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    d = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][0])
    assert d["impl"] == "reference" and d["steps"] == 20 and d["warmup"] == 5 and d["value"] > 0
    assert "extrapolated" in d["cpu_baseline"]["sample"]


def test_row_workloads_match_the_oracle_tables():
    """The continuous (c5c), overlapping-window (c4o) and beam (c4b) bench
    workloads are the c5 / c4 inputs: the same requests, and for c4o the
    oracle's chunk table with 1 s of overlap."""
    import importlib.util

    import numpy as np

    from oracle import plan as oplan
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    c5 = bench.make_workload("c5", 0, with_audio=False)
    c5c = bench.make_workload("c5c", 0, with_audio=False)
    assert np.array_equal(c5.req_samples, c5c.req_samples) and np.array_equal(c5.chunk_len, c5c.chunk_len)
    assert c5c.kind == "cont" and c5c.budget == c5.budget
    c4 = bench.make_workload("c4", 0, with_audio=False)
    c4o = bench.make_workload("c4o", 0, with_audio=False)
    req, idx, valid = oplan.chunk_table(c4o.req_samples, c4o.overlap)
    assert c4o.overlap == 16000 and c4o.chunk_len.size == req.size == 34
    assert np.array_equal(c4.req_samples, c4o.req_samples) and c4o.audio_s == c4.audio_s
    c4b = bench.make_workload("c4b", 0, with_audio=False)
    assert c4b.beams == 4 and np.array_equal(c4b.chunk_len, c4.chunk_len)
