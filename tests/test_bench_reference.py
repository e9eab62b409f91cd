"""bench.py's reference arm on CPU: the fp64 oracle timed on the host cores.

Its line carries the same `config` as the GPU arm's (so the two compare), says
plainly that its steps are extrapolated from a bounded sample, and scales each
sampled step by the oracle's own iteration count for that step of its
trajectory when the committed table has it."""
import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_linear_solve_gb300 import workloads as W  # noqa: E402


def _args(**kw):
    a = dict(gpus=1, steps=2, warmup=1, impl="reference", config="C1", oracle_iters=4)
    a.update(kw)
    return argparse.Namespace(**a)


def test_reference_line_matches_the_gpu_arms_config_and_is_labelled():
    line = bench.run_reference(_args())
    assert line["impl"] == "reference"
    assert line["config"] == bench.bench_config(W.make("C1"))
    assert line["extrapolated"] is True
    assert "EXTRAPOLATED" in line["cpu_baseline"]["sample"]
    assert line["value"] == line["cpu_baseline"]["value"] == line["e2e"]["value"]
    assert abs(line["ms_per_step"] - 1e3 / line["value"]) < 1e-6 * line["ms_per_step"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_steps_use_the_oracle_trajectory_counts(monkeypatch):
    table = [100, 200, 300, 400]
    monkeypatch.setattr(bench, "oracle_step_iterations", lambda config: table)
    line = bench.run_reference(_args(steps=2, warmup=1))
    # the timed steps are steps 1 and 2 of the trajectory
    assert line["pcg_iterations_mean"] == 250.0
    line = bench.run_reference(_args(steps=3, warmup=2))
    # steps 2, 3 and 4: the last is past the table and takes its mean
    assert line["pcg_iterations_mean"] == (300 + 400 + 250) / 3
