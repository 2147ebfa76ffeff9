"""Host-side logic of bench.py, on the CPU: the CPU baseline's extrapolation.

The oracle's calls have a fixed part that does not grow with the sample (the
projection decodes all of W; the KV call copies the caches).  The bench times
two sample sizes and extrapolates fixed + per-unit cost; these tests check that
the fit recovers both parts from exact linear timings and falls back to the
linear upper bound when noise makes a part negative.
"""
import math
import os
import sys
import time

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


@pytest.mark.parametrize("fixed,per_unit", [(1.25, 3e-4), (0.0, 2e-3), (7.0, 1e-6)])
def test_fit_recovers_fixed_and_per_unit_cost(fixed, per_unit):
    n1, n2, n_full = 128, 4096, 75600
    t = lambda n: fixed + per_unit * n
    full, how, f, u = bench.fit_full_time(n1, t(n1), n2, t(n2), n_full)
    assert how == "fit"
    assert math.isclose(f, fixed, rel_tol=1e-9, abs_tol=1e-12)
    assert math.isclose(u, per_unit, rel_tol=1e-9)
    assert math.isclose(full, t(n_full), rel_tol=1e-9)
    # the old single-sample linear scaling charges the fixed part n_full / n1 times
    assert full <= t(n1) * n_full / n1 + 1e-12


def test_fit_falls_back_to_the_linear_upper_bound():
    # the larger sample timed faster than the smaller one: no meaningful per-unit cost
    full, how, f, u = bench.fit_full_time(128, 1.3, 4096, 1.2, 75600)
    assert how == "linear" and f == 0.0
    assert math.isclose(full, 1.2 * 75600 / 4096)
    # a negative fixed part
    full, how, _, _ = bench.fit_full_time(1, 0.1, 2, 1.0, 8)
    assert how == "linear" and math.isclose(full, 4.0)
    # one sample size only
    full, how, _, _ = bench.fit_full_time(8, 2.0, 8, 2.0, 8)
    assert how == "linear" and math.isclose(full, 2.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`bench.py --impl reference` launched as two ranks: rank 0 times the oracle
    and prints the one JSON line; the other rank exits 0 without work."""
    import json
    import socket
    import subprocess

    with socket.socket() as sk:  # a free port for the rendezvous
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(root, "bench.py"),
           "--impl", "reference", "--workload", "small", "--gpus", "2", "--steps", "1", "--warmup", "1",
           "--oracle-rows", "64"]
    t0 = time.perf_counter()
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    wall_s = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # what was timed is what is reported: the steps the line claims fit inside the run's
    # own wall time (each is one bounded sample; the full step is only extrapolated),
    # and the config is the repo arm's own
    assert d["ms_per_step"] > 0 and d["extrapolated_step_s"] > 0
    assert d["steps"] * d["ms_per_step"] / 1e3 < wall_s
    from bench import bench_config, workload
    q, k = workload("small")
    assert d["config"] == bench_config(q, k, 2)
