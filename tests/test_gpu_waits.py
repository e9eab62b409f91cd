"""The device-side bounded waits give up and report instead of hanging.

Every wait of the library's kernels (the SpMV pipeline's mbarriers, the PCG
kernel's grid barrier) is bounded in time and records a status bit when it
gives up, so that a lost arrival can never hang the GPU.  These tests run
each kind of wait on something that never completes -- an mbarrier phase
without arrivals, a barrier counter that gets one of the two arrivals it
waits for -- with a short limit, and check that the call returns the same
error a real timeout reports, after about that limit, and that the GPU
context is still usable afterwards.  No fault, trap or endless loop is
involved.
"""
import time

import numpy as np
import pytest

from sparse_linear_solve_gb300 import pcloth as pc
from sparse_linear_solve_gb300 import workloads as W

from gpu_helpers import DEV, to_dev

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT_BIT = 1 << 4


@pytest.mark.parametrize("which", [0, 1], ids=["mbarrier", "grid_counter"])
def test_bounded_wait_gives_up_and_reports(which):
    limit = 0.05
    pc.pcloth_selftest_bounded_wait(which, limit)          # warm-up: module load
    t0 = time.perf_counter()
    rc, status, msg = pc.pcloth_selftest_bounded_wait(which, limit)
    elapsed = time.perf_counter() - t0
    assert rc == pc.ERR_CUDA and "timed out" in msg
    assert status & WAIT_TIMEOUT_BIT
    assert limit <= elapsed < limit + 2.0
    # the context is still usable: a small solve right afterwards is correct
    w = W.tiny_cloth(n=16)
    cl = pc.PCloth.from_workload(w, device=DEV)
    cl.assemble(to_dev(w.x0), to_dev(w.v0), None, w.h)
    dv, it, rr, code = cl.solve(w.tol, w.maxit)
    assert code == pc.OK and rr <= w.tol
    assert np.isfinite(dv.cpu().numpy()).all()


def test_poisoned_grid_barrier_stops_every_cta():
    """One CTA of two arrives at the PCG kernel's grid barrier marked as
    having timed out; both leave at once with the timeout verdict."""
    t0 = time.perf_counter()
    rc, status, msg = pc.pcloth_selftest_bounded_wait(2, 1.0)
    elapsed = time.perf_counter() - t0
    assert rc == pc.ERR_CUDA and "timed out" in msg
    assert status & WAIT_TIMEOUT_BIT
    assert (status >> 8) & 0xFF == 2
    assert elapsed < 1.5          # no CTA waited for the 2 s limit


def test_selftest_rejects_bad_arguments():
    for which, limit in ((3, 0.05), (-1, 0.05), (0, 0.0), (1, 11.0)):
        rc, _, _ = pc.pcloth_selftest_bounded_wait(which, limit)
        assert rc == pc.ERR_INVALID_ARG
