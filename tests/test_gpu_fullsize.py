"""Full-size configurations (the benchmark's launch configuration) against the
fp64 oracle.  P-Cloth (arXiv 2008.00409) Sec. 2.5 Eq. (3), Sec. 3.1, 3.2.2.

Assembly (pattern bit-exact, every block) and SpMV are compared in full at
every size; the oracle assembles a 10.9M-block system in seconds.  The fp64
PCG of the two largest systems would take minutes on one host core, so there
the solve is checked through properties that hold at any size: the recursive
residual meets the tolerance, the true residual |b - A dv| / |b| of the
GPU's dv, recomputed in fp64 with the oracle's own A and b, stays within the
accuracy that fp32 storage allows, and the iteration count matches the one
the oracle's own solve of the same system recorded (oracle/iteration_table.py).  The two smaller full configurations also
compare dv with the oracle's PCG directly.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_linear_solve_gb300 import pcloth as pc
from sparse_linear_solve_gb300 import workloads as W

from gpu_helpers import compare_assembly, rel_l2, to_dev

pytestmark = pytest.mark.gpu

# |b - A dv| / |b| in fp64 for an fp32 solve stopped at |r|/|b| <= 1e-6: the
# recursion's fp32 rounding leaves the true residual above the recursive one
# (up to ~1e-4 has been seen on the 32x32 grid); 1e-3 bounds it with margin.
TRUE_RESIDUAL_BOUND = 1e-3


def oracle_iterations(name):
    """PCG iterations of the fp64 oracle on the first step of a configuration,
    as oracle/iteration_table.py recorded them (same seeded inputs)."""
    import json
    import os
    path = os.path.join(os.path.dirname(oracle.__file__), "iteration_table.json")
    with open(path) as f:
        return int(json.load(f)[name]["iterations"][0])


@pytest.mark.parametrize("name", ["C2", "C3"])
def test_fullsize_pcg_against_oracle(name):
    w = W.make(name)
    c = w.contacts(0)
    pcl, ref, _, _ = compare_assembly(w, w.x0, w.v0, c if c.n else None)
    x = np.random.default_rng(4).normal(size=(w.n_verts, 3)).astype(np.float32)
    xd = to_dev(x)
    y = pcl.spmv(xd)
    assert rel_l2(y.cpu().numpy(), ref.spmv(x)) <= 1e-5
    # the block-ELL layout of the pages gives the same bits at full size
    pcl.bell_build()
    assert torch.equal(pcl.spmv_bell(xd), y)
    dv, it, rr, code = pcl.solve(w.tol, w.maxit)
    assert code == pc.OK and rr <= w.tol
    dv_ref, it_ref, rr_ref, st = ref.pcg(w.tol, w.maxit)
    assert st == oracle.OK
    assert rel_l2(dv.cpu().numpy(), dv_ref) <= 1e-4
    assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)


@pytest.mark.parametrize("name", ["C4", "C5"])
def test_fullsize_assembly_spmv_and_residual(name):
    w = W.make(name)
    c = w.contacts(0)
    pcl, ref, _, _ = compare_assembly(w, w.x0, w.v0, c)
    x = np.random.default_rng(4).normal(size=(w.n_verts, 3)).astype(np.float32)
    xd = to_dev(x)
    y = pcl.spmv(xd)
    assert rel_l2(y.cpu().numpy(), ref.spmv(x)) <= 1e-5
    # the block-ELL layout of the pages gives the same bits at full size
    pcl.bell_build()
    assert torch.equal(pcl.spmv_bell(xd), y)
    dv, it, rr, code = pcl.solve(w.tol, w.maxit)
    assert code == pc.OK and rr <= w.tol
    d = dv.cpu().numpy().astype(np.float64)
    true = np.linalg.norm(ref.b - ref.spmv(d)) / np.linalg.norm(ref.b)
    assert true <= TRUE_RESIDUAL_BOUND, true
    # the same PCG on the same system as the fp64 oracle's solve of this first
    # step, whose iteration count oracle/iteration_table.py recorded
    it_ref = oracle_iterations(name)
    assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)
