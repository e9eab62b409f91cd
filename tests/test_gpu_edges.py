"""Edge sizes of the GPU path against the fp64 oracle.

A chain of n vertices (springs between neighbours and weaker ones between
second neighbours, perturbed positions so that the springs are stretched
and compressed) for n = 1 (a single vertex with no spring: A = m I), 2, and
values on both sides of the row-tile sizes of the streaming SpMV (32 and 64
rows), up to a few tiles with a ragged tail.  Every case checks the
assembled system (pattern bit-exact, blocks 1e-5), the SpMV (1e-5 relative
L2) and the PCG solution (1e-4 relative L2 at relative residual <= 1e-6) --
the same bars as the other parity tests.

The stiffnesses give kappa(P A) ~ 400.  Iteration counts are compared
(within max(3, 3%)) from 64 rows up only: on smaller chains (under 200
unknowns) fp64 CG nearly terminates within the Krylov dimension, which fp32
arithmetic cannot reproduce.  A plain float32 restatement of the same PCG
in numpy needs 10-15% more iterations there, as the GPU does, while from 63
rows up the counts agree exactly.
"""
import numpy as np
import pytest

from oracle import oracle
from sparse_linear_solve_gb300 import pcloth as pc

from gpu_helpers import DEV, block_rel_err, rel_l2, to_dev

pytestmark = pytest.mark.gpu

H = 1e-2
GRAVITY = np.array([0.0, 0.0, -9.8], np.float32)


def chain(n, seed):
    rng = np.random.default_rng(seed)
    x = np.zeros((n, 3), np.float32)
    x[:, 0] = np.arange(n, dtype=np.float32) * 0.01
    x += rng.normal(0.0, 1e-3, size=(n, 3)).astype(np.float32)
    v = rng.normal(0.0, 0.1, size=(n, 3)).astype(np.float32)
    i1 = np.arange(max(n - 1, 0), dtype=np.int32)
    i2 = np.arange(max(n - 2, 0), dtype=np.int32)
    si = np.concatenate([i1, i2]).astype(np.int32)
    sj = np.concatenate([i1 + 1, i2 + 2]).astype(np.int32)
    k = np.concatenate([np.full(len(i1), 1e2), np.full(len(i2), 1e-1)]).astype(np.float32)
    rest = np.concatenate([np.full(len(i1), 0.01), np.full(len(i2), 0.02)]).astype(np.float32)
    mass = np.full(n, 1e-4, np.float32)
    return mass, x, v, (si, sj, k, rest)


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 63, 64, 65, 129, 1000])
def test_chain_sizes_match_oracle(n):
    mass, x, v, springs = chain(n, 3000 + n)
    cl = pc.PCloth(mass, GRAVITY, springs if len(springs[0]) else None, device=DEV)
    cl.assemble(to_dev(x), to_dev(v), None, H)
    ref = oracle.assemble(n, mass, GRAVITY, springs, None, x, v, H)
    g = cl.export()
    assert np.array_equal(g["rowptr"].cpu().numpy().astype(np.int64), ref.rowptr)
    assert np.array_equal(g["colind"].cpu().numpy(), ref.colind)
    assert block_rel_err(g["vals"].cpu().numpy(), ref.vals) <= 1e-5
    xin = np.random.default_rng(n).normal(size=(n, 3)).astype(np.float32)
    y = cl.spmv(to_dev(xin)).cpu().numpy()
    assert rel_l2(y, ref.spmv(xin)) <= 1e-5
    dv, it, rr, code = cl.solve(1e-6, 20000)
    dv_ref, it_ref, rr_ref, _ = ref.pcg(1e-6, 20000)
    assert code == pc.OK and rr <= 1e-6
    assert rel_l2(dv.cpu().numpy(), dv_ref) <= 1e-4
    if n >= 64:
        assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)


def test_single_vertex_falls_freely():
    """No spring: A = m I and b = h m g, so one iteration gives dv = h g."""
    mass = np.array([2e-4], np.float32)
    cl = pc.PCloth(mass, GRAVITY, None, device=DEV)
    x = np.array([[0.1, -0.2, 0.3]], np.float32)
    v = np.array([[1.0, 0.0, -0.5]], np.float32)
    cl.assemble(to_dev(x), to_dev(v), None, H)
    dv, it, rr, code = cl.solve(1e-6, 10)
    assert code == pc.OK and it == 1
    np.testing.assert_allclose(dv.cpu().numpy(), (H * GRAVITY)[None, :], rtol=1e-6)
