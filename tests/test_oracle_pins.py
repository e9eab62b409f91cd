"""Pins of the fp64 oracle against hand values, closed forms, invariants and
brute force (no GPU).  Every check here is independent of the oracle's own
formulas: hand-derived fixtures, a dense LAPACK solve, eigenvalues, finite
differences, brute-force pattern sets, exact special cases.

P-Cloth (arXiv 2008.00409): Sec. 2.5 Eq. (1)-(3) define the system, Sec. 3.2.2
the pattern and value filling, Sec. 3.1 the PCG solve.
"""
import json
import os

import numpy as np
import pytest

from oracle import oracle
from sparse_linear_solve_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- element --

@pytest.mark.parametrize("case", load("single_spring.json")["cases"], ids=lambda c: c["name"])
def test_single_spring_hand_values(case):
    K, F, ok = oracle.element(case["xa"], case["xb"], case["va"], case["vb"],
                              case["k"], case["rest"], case["h"])
    assert ok
    np.testing.assert_allclose(K, np.array(case["K"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(F, np.array(case["F"]), rtol=0, atol=1e-12)


def test_jacobian_is_force_derivative_in_tension():
    """K = -dF_a/dx_a by central differences when every spring is stretched."""
    rng = np.random.default_rng(7)
    for _ in range(20):
        xa = rng.normal(size=3)
        xb = xa + rng.normal(size=3)
        l = np.linalg.norm(xb - xa)
        rest = 0.5 * l
        k = rng.uniform(0.5, 5.0)
        K, _, _ = oracle.element(xa, xb, np.zeros(3), np.zeros(3), k, rest, 0.0)
        eps = 1e-6
        J = np.zeros((3, 3))
        for c in range(3):
            dp = xa.copy(); dp[c] += eps
            dm = xa.copy(); dm[c] -= eps
            Fp = oracle.element(dp, xb, np.zeros(3), np.zeros(3), k, rest, 0.0)[1]
            Fm = oracle.element(dm, xb, np.zeros(3), np.zeros(3), k, rest, 0.0)[1]
            J[:, c] = (Fp - Fm) / (2 * eps)
        np.testing.assert_allclose(K, -J, rtol=1e-6, atol=1e-7 * k)


def test_jacobian_clamp_in_compression_is_axial_only():
    """Compressed spring: the clamp drops the transverse term, K = k d d^T."""
    rng = np.random.default_rng(8)
    for _ in range(10):
        xa = rng.normal(size=3)
        xb = xa + rng.normal(size=3)
        e = xb - xa
        l = np.linalg.norm(e)
        d = e / l
        K, _, _ = oracle.element(xa, xb, np.zeros(3), np.zeros(3), 3.0, 2.0 * l, 0.0)
        np.testing.assert_allclose(K, 3.0 * np.outer(d, d), atol=1e-12)
        # and it is positive semidefinite with the axis as its only mode
        w = np.linalg.eigvalsh(K)
        assert w.min() > -1e-12 and abs(w.max() - 3.0) < 1e-12


def test_zero_length_is_reported():
    _, _, ok = oracle.element([1, 2, 3], [1, 2, 3], [0, 0, 0], [0, 0, 0], 1.0, 1.0, 0.0)
    assert not ok


# ------------------------------------------------------------- assembly --

def test_two_vertex_closed_form_and_solve():
    g = load("two_vertex.json")
    x = np.array(g["x"], np.float32)
    s = oracle.assemble(2, np.array(g["mass"], np.float32), np.array(g["gravity"], np.float32),
                        (np.array([0], np.int32), np.array([1], np.int32),
                         np.array([g["k"]], np.float32), np.array([g["rest"]], np.float32)),
                        None, x, np.zeros_like(x), g["h"])
    assert s.status == oracle.OK
    A = np.array(g["A"])
    b = np.array(g["b"])
    np.testing.assert_allclose(s.dense(), A, atol=1e-12)
    # b: gravity is float32-rounded on the way in (9.8 is not exact in fp32)
    np.testing.assert_allclose(s.b.reshape(-1), b, atol=1e-7)
    dv, it, rr, st = s.pcg(1e-14, 100)
    assert st == oracle.OK
    ref = np.linalg.solve(A, s.b.reshape(-1))
    np.testing.assert_allclose(dv.reshape(-1), ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv[:, 2], np.array(g["dv_z"]), atol=1e-6)
    # block-Jacobi inverse is the inverse of the diagonal blocks
    for i in range(2):
        np.testing.assert_allclose(s.pinv[i] @ A[3 * i:3 * i + 3, 3 * i:3 * i + 3], np.eye(3),
                                   atol=1e-12)


def test_two_vertex_moving_rhs_at_advanced_positions():
    """b = h f(x_t + h v_t) with both velocities nonzero (Eq. (3)), and A
    unchanged by v (K at x_t).  Forces taken at x_t, at x_t + 2 h v_t, or
    with either vertex's velocity dropped all give other values."""
    g = load("two_vertex_moving.json")
    x = np.array(g["x"], np.float32)
    v = np.array(g["v"], np.float32)
    s = oracle.assemble(2, np.array(g["mass"], np.float32), np.array(g["gravity"], np.float32),
                        (np.array([0], np.int32), np.array([1], np.int32),
                         np.array([g["k"]], np.float32), np.array([g["rest"]], np.float32)),
                        None, x, v, g["h"])
    assert s.status == oracle.OK
    np.testing.assert_allclose(s.b.reshape(-1), np.array(g["b"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(s.dense(), np.array(g["A"]), rtol=0, atol=1e-12)
    dv, it, rr, st = s.pcg(1e-14, 100)
    assert st == oracle.OK
    ref = np.linalg.solve(np.array(g["A"]), np.array(g["b"]))
    np.testing.assert_allclose(dv.reshape(-1), ref, rtol=1e-10, atol=1e-12)


def _tiny(n, rest_from_grid=False):
    return W.tiny_cloth(n=n, seed=1000 + n, rest_from_grid=rest_from_grid)


def brute_pattern(n, pairs):
    keys = {(i, i) for i in range(n)}
    for a, b in pairs:
        keys.add((a, b))
        keys.add((b, a))
    return sorted(keys)


@pytest.mark.parametrize("n", [2, 4, 8, 32])
def test_pattern_matches_brute_force_and_count(n):
    w = _tiny(n)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    assert s.status == oracle.OK
    pat = brute_pattern(w.n_verts, zip(w.spring_i.tolist(), w.spring_j.tolist()))
    got = [(i, int(c)) for i in range(w.n_verts)
           for c in s.colind[s.rowptr[i]:s.rowptr[i + 1]]]
    assert got == pat
    # grid springs never repeat a pair: nnzb = N + 2 * #springs
    assert s.nnzb == w.n_verts + 2 * w.n_springs
    if n >= 5:
        # an interior vertex has 6 stretch + 6 bend neighbours + itself
        i = (n // 2) * n + n // 2
        assert s.rowptr[i + 1] - s.rowptr[i] == 13


def test_grid_spring_counts():
    # stretch: 2 n (n-1) + (n-1)^2 ; bend: 2 (n-1)(n-2) + (n-1)^2
    for n in (3, 4, 32, 256):
        w = W.tiny_cloth(n=n)
        stretch = 2 * n * (n - 1) + (n - 1) ** 2
        bend = 2 * (n - 1) * (n - 2) + (n - 1) ** 2
        assert w.n_springs == stretch + bend
        assert (w.spring_k == W.K_STRETCH).sum() == stretch


@pytest.mark.parametrize("n,rest_from_grid", [(4, False), (8, False), (8, True), (32, False), (32, True)])
def test_invariants_symmetry_rowsum_definiteness_solve(n, rest_from_grid):
    w = _tiny(n, rest_from_grid)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    A = s.dense()
    scale = np.abs(A).max()
    # symmetric
    assert np.abs(A - A.T).max() <= 1e-12 * scale
    # the springs are translation invariant: A (1 (x) c) = M (1 (x) c)
    M = np.kron(np.diag(w.mass.astype(np.float64)), np.eye(3))
    for c in np.eye(3):
        one = np.tile(c, w.n_verts)
        np.testing.assert_allclose(A @ one, M @ one, rtol=0, atol=1e-12 * scale)
    # A - M is positive semidefinite, A positive definite
    ev = np.linalg.eigvalsh(A - M)
    assert ev.min() >= -1e-12 * scale
    assert np.linalg.eigvalsh(A).min() > 0
    # PCG at a tight tolerance reproduces the dense LU solve
    dv, it, rr, st = s.pcg(1e-13, 20000)
    assert st == oracle.OK and rr <= 1e-13
    ref = np.linalg.solve(A, s.b.reshape(-1))
    err = np.linalg.norm(dv.reshape(-1) - ref) / np.linalg.norm(ref)
    assert err < 1e-10, err


def test_translation_invariance_of_assembly():
    w = _tiny(8, rest_from_grid=True)
    # positions on a 2^-20 lattice so that the shifted copy is exact in fp32
    x = (np.round(w.x0.astype(np.float64) * 2**20) / 2**20).astype(np.float32)
    v = (np.round(w.v0.astype(np.float64) * 2**10) / 2**10).astype(np.float32)
    s0 = oracle.assemble_workload(w, x, v)
    shift = np.array([0.25, -0.5, 0.125], np.float32)
    xs = x + shift
    assert np.array_equal(xs.astype(np.float64) - shift.astype(np.float64), x.astype(np.float64))
    s1 = oracle.assemble_workload(w, xs, v)
    np.testing.assert_allclose(s1.vals, s0.vals, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s1.b, s0.b, rtol=1e-9, atol=1e-12)


def test_zero_stiffness_reduces_to_mass_matrix():
    """k = 0: A = M, P = M^-1, PCG converges in one iteration to dv = h g."""
    w = _tiny(8)
    w.spring_k[:] = 0.0
    mass = np.linspace(1e-4, 3e-4, w.n_verts).astype(np.float32)
    w.mass = mass
    s = oracle.assemble_workload(w, w.x0, w.v0)
    M = np.kron(np.diag(mass.astype(np.float64)), np.eye(3))
    np.testing.assert_array_equal(s.dense(), M)
    for i in range(w.n_verts):
        np.testing.assert_allclose(s.pinv[i], np.eye(3) / float(mass[i]), rtol=1e-15)
    dv, it, rr, st = s.pcg(1e-12, 10)
    assert st == oracle.OK and it == 1
    np.testing.assert_allclose(dv, np.tile(w.h * w.gravity.astype(np.float64), (w.n_verts, 1)),
                               rtol=1e-15, atol=1e-18)


def test_contacts_merge_and_sum():
    """A contact on a spring's pair and a repeated contact land in one block
    each, with their contributions summed (filling step 3: duplicates removed)."""
    w = _tiny(4, rest_from_grid=True)
    x, v = w.x0, w.v0
    a, b = int(w.spring_i[0]), int(w.spring_j[0])   # an existing spring pair
    c, d = 0, 15                                    # a new pair, given twice
    ci = np.array([a, c, d], np.int32)
    cj = np.array([b, d, c], np.int32)
    ck = np.array([1e3, 1e3, 5e2], np.float32)
    cr = np.array([0.002, 0.003, 0.004], np.float32)
    s0 = oracle.assemble_workload(w, x, v)
    s1 = oracle.assemble(w.n_verts, w.mass, w.gravity,
                         (w.spring_i, w.spring_j, w.spring_k, w.spring_rest),
                         (ci, cj, ck, cr), x, v, w.h)
    assert s1.nnzb == s0.nnzb + 2
    h2 = w.h * w.h

    def blk(s, i, j):
        p = s.rowptr[i] + np.searchsorted(s.colind[s.rowptr[i]:s.rowptr[i + 1]], j)
        assert s.colind[p] == j
        return s.vals[p]

    x64 = x.astype(np.float64)
    Ka, _, _ = oracle.element(x64[a], x64[b], np.zeros(3), np.zeros(3), ck[0], cr[0], 0)
    np.testing.assert_allclose(blk(s1, a, b), blk(s0, a, b) - h2 * Ka, rtol=1e-12, atol=1e-15)
    K1, _, _ = oracle.element(x64[c], x64[d], np.zeros(3), np.zeros(3), ck[1], cr[1], 0)
    K2, _, _ = oracle.element(x64[d], x64[c], np.zeros(3), np.zeros(3), ck[2], cr[2], 0)
    np.testing.assert_allclose(blk(s1, c, d), -h2 * (K1 + K2), rtol=1e-12)
    np.testing.assert_allclose(blk(s1, d, c), -h2 * (K1 + K2), rtol=1e-12)


def test_bad_inputs_are_rejected():
    w = _tiny(4)
    for ci, cj in ((0, 16), (-1, 2), (3, 3)):
        s = oracle.assemble(w.n_verts, w.mass, w.gravity,
                            (w.spring_i, w.spring_j, w.spring_k, w.spring_rest),
                            (np.array([ci], np.int32), np.array([cj], np.int32),
                             np.array([1.0], np.float32), np.array([0.1], np.float32)),
                            w.x0, w.v0, w.h)
        assert s.status == oracle.BAD_INDEX
    v = w.v0.copy()
    v[3, 1] = np.nan
    s = oracle.assemble_workload(w, w.x0, v)
    assert s.status == oracle.NONFINITE


def test_maxit_reports_not_converged():
    w = _tiny(8, rest_from_grid=True)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    dv, it, rr, st = s.pcg(1e-12, 1)
    assert st == oracle.NOT_CONVERGED and it == 1 and rr > 1e-12


def test_state_update_by_hand():
    x = np.array([[1.0, 2.0, 3.0]], np.float32)
    v = np.array([[0.5, -0.5, 0.25]], np.float32)
    dv = np.array([[0.25, 0.5, -1.25]])
    xn, vn = oracle.update(x, v, dv, 0.5)
    np.testing.assert_array_equal(vn, [[0.75, 0.0, -1.0]])
    np.testing.assert_array_equal(xn, [[1.375, 2.0, 2.5]])


def test_pcg_residual_definition():
    """The reported residual is |b - A dv| / |b| of the returned dv (up to the
    recursion's drift), and it meets the tolerance."""
    w = _tiny(16, rest_from_grid=True)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    dv, it, rr, st = s.pcg(1e-8, 10000)
    assert st == oracle.OK and rr <= 1e-8
    true = np.linalg.norm(s.b - s.spmv(dv)) / np.linalg.norm(s.b)
    assert true <= 2e-8
    # CG on an SPD system of m unknowns needs at most m iterations in exact
    # arithmetic; well-conditioned blocks need far fewer
    assert it < 3 * w.n_verts


def test_spmv_against_dense():
    w = _tiny(8, rest_from_grid=True)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    x = np.random.default_rng(3).normal(size=(w.n_verts, 3))
    np.testing.assert_allclose(s.spmv(x).reshape(-1), s.dense() @ x.reshape(-1),
                               rtol=1e-13, atol=1e-13)


# ---- PCG from an initial guess (warm start) -----------------------------

def _solution_lu(s):
    return np.linalg.solve(s.dense(), s.b.reshape(-1)).reshape(-1, 3)


def test_guess_at_the_solution_takes_no_iteration():
    w = _tiny(8, rest_from_grid=True)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    x = _solution_lu(s)
    dv, it, rr, st = s.pcg(1e-8, 100, x0=x)
    assert st == oracle.OK and it == 0
    np.testing.assert_array_equal(dv, x)
    # both residuals are rounding noise of an exact solution
    true = np.linalg.norm(s.b.reshape(-1) - s.dense() @ x.reshape(-1)) / np.linalg.norm(s.b)
    assert rr <= 1e-13 and true <= 1e-13


def test_guess_with_no_iteration_reports_its_own_residual():
    """maxit = 0: the returned residual is |b - A x0| / |b| (numpy, dense)."""
    w = _tiny(8, rest_from_grid=True)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    x0 = np.random.default_rng(5).normal(size=(w.n_verts, 3)) * 1e-3
    dv, it, rr, st = s.pcg(1e-8, 0, x0=x0)
    assert st == oracle.NOT_CONVERGED and it == 0
    np.testing.assert_array_equal(dv, x0)
    true = np.linalg.norm(s.b.reshape(-1) - s.dense() @ x0.reshape(-1)) / np.linalg.norm(s.b)
    assert rr == pytest.approx(true, rel=1e-12)


def test_any_guess_converges_to_the_dense_solution():
    w = _tiny(8, rest_from_grid=True)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    x = _solution_lu(s)
    x0 = np.random.default_rng(6).normal(size=x.shape) * np.abs(x).max()
    dv, it, rr, st = s.pcg(1e-12, 10000, x0=x0)
    assert st == oracle.OK and rr <= 1e-12 and it > 0
    assert np.linalg.norm(dv - x) <= 1e-10 * np.linalg.norm(x)


def test_zero_guess_is_the_cold_start_bit_for_bit():
    """b - A 0 = b exactly, so a zero guess must follow the cold iteration."""
    w = _tiny(16, rest_from_grid=True)
    s = oracle.assemble_workload(w, w.x0, w.v0)
    cold = s.pcg(1e-8, 10000)
    warm = s.pcg(1e-8, 10000, x0=np.zeros((w.n_verts, 3)))
    np.testing.assert_array_equal(cold[0], warm[0])
    assert cold[1:] == warm[1:]


# ---- vertex-vertex proximity contacts ------------------------------------

def _numpy_pairs(x, radius, springs):
    """Independent restatement: all pairs in float32 numpy arithmetic."""
    x = np.asarray(x, np.float32)
    n = x.shape[0]
    excl = {(min(a, b), max(a, b)) for a, b in zip(springs[0], springs[1])}
    r2 = np.float32(radius) * np.float32(radius)
    out = []
    for i in range(n):
        d = x[i + 1:] - x[i]
        d2 = (d[:, 0] * d[:, 0] + d[:, 1] * d[:, 1]) + d[:, 2] * d[:, 2]
        for j in (np.nonzero(d2 < r2)[0] + i + 1):
            if (i, int(j)) not in excl:
                out.append((i, int(j)))
    return out


def test_contacts_hand_case():
    # A-B 1.5 mm, B-D 1.9 mm, A-C 2.1 mm, A-D sqrt(1.5^2 + 1.9^2) = 2.42 mm
    x = np.array([[0, 0, 0], [0.0015, 0, 0], [0, 0.0021, 0], [0.0015, 0, 0.0019]], np.float32)
    none = (np.zeros(0, np.int32), np.zeros(0, np.int32))
    i, j, total = oracle.find_contacts(x, 2e-3, none)
    assert total == 2 and list(zip(i, j)) == [(0, 1), (1, 3)]
    # a spring between A and B (given as B-A) removes that pair
    i, j, total = oracle.find_contacts(x, 2e-3, (np.array([1], np.int32), np.array([0], np.int32)))
    assert total == 1 and list(zip(i, j)) == [(1, 3)]


def test_contacts_radius_is_strict():
    r = 0.25   # r and r^2 exact in float32
    none = (np.zeros(0, np.int32), np.zeros(0, np.int32))
    at = np.array([[0, 0, 0], [r, 0, 0]], np.float32)
    assert oracle.find_contacts(at, r, none)[2] == 0
    inside = np.array([[0, 0, 0], [np.nextafter(np.float32(r), np.float32(0)), 0, 0]], np.float32)
    assert oracle.find_contacts(inside, r, none)[2] == 1


def test_contacts_match_a_numpy_float32_restatement():
    rng = np.random.default_rng(21)
    x = rng.uniform(0, 0.03, size=(400, 3)).astype(np.float32)
    springs = (rng.integers(0, 400, 300).astype(np.int32), rng.integers(0, 400, 300).astype(np.int32))
    i, j, total = oracle.find_contacts(x, 4e-3, springs)
    ref = _numpy_pairs(x, 4e-3, springs)
    assert total == len(ref) > 50
    assert list(zip(i.tolist(), j.tolist())) == ref


def test_contacts_beyond_capacity_are_counted():
    x = np.zeros((10, 3), np.float32)   # every pair at distance 0
    none = (np.zeros(0, np.int32), np.zeros(0, np.int32))
    i, j, total = oracle.find_contacts(x, 1e-3, none, capacity=7)
    assert total == 45 and len(i) == 7
    assert list(zip(i, j)) == [(0, 1), (0, 2), (0, 3), (0, 4), (0, 5), (0, 6), (0, 7)]
