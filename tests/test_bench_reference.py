"""The benchmark's reference arm (the CPU oracle), run on the host.

`bench.py --impl reference` must print one JSON line in the same metric,
unit and direction as the GPU arm, with the CPU-baseline and end-to-end
objects the line contract asks for (no host/device copies: it runs on the
host).  It needs no GPU, so it runs with the CPU tests.
"""
import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_prints_one_contract_line():
    import bench
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--steps", "1",
                        "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == (os.cpu_count() or 1)
    assert cb["sample"]
    assert cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_row_split_oracle_equals_one_call():
    """The all-core baseline splits a GEMV's output rows over threads, each
    slice an unmodified oracle call with its own weight-scale segments: the
    result is the single call's, bit for bit (the wqkv segments are cut)."""
    import numpy as np

    import bench
    import oracle
    import synth
    N, K, bounds = synth.DECODE_SHAPES["wqkv"]
    case = synth.gemv_case(1, N, K, synth.base_seed(1, 9), bounds=bounds)
    q, s = oracle.quant_act(case["xf"])
    want = oracle.gemv(q, case["canon"], s, case["ws"], case["bounds"], N, K)
    for threads in (1, 3, 7, 16):
        got = bench.oracle_gemv_threads(oracle, q, case["canon"], s,
                                        case["ws"], case["bounds"], N, K,
                                        threads)
        assert (got == want).all(), threads
