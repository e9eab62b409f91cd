"""GPU path (through the C ABI) against the fp64 oracle on identical seeded
inputs.  P-Cloth (arXiv 2008.00409): Sec. 2.5 Eq. (3) (system), Sec. 3.2.2
(pattern and value filling), Sec. 3.1 (SpMV and PCG).

Tolerances (fp32 storage and arithmetic against fp64):
  * pattern (rowptr, colind): bit-exact;
  * assembled blocks: max per-block relative Frobenius error <= 1e-5;
  * b: <= 1e-5 relative to the summed magnitude of its terms per vertex;
  * block-Jacobi inverses: per block within the perturbation bound
    kappa(D) (|dD|/|D| + 16 eps32) of a matrix inverse, and P D = I to
    16 kappa(D) eps32 against the GPU's own diagonal block;
  * SpMV: relative L2 <= 1e-5;
  * PCG: same algorithm and tolerance on both sides, relative L2 of dv
    <= 1e-4 and iteration counts within max(3, 3%).
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_linear_solve_gb300 import pcloth as pc
from sparse_linear_solve_gb300 import workloads as W

from gpu_helpers import DEV, compare_assembly, make, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def small_configs():
    return {
        "tiny32": W.tiny_cloth(),
        "tiny32_tension": W.tiny_cloth(rest_from_grid=True),
        "droop37": W.drooped_cloth(n=37, steps=2),          # ragged tiles
        "jitter64": W.jittered_cloth(n=64, steps=2),
        "twolayer33": W.two_layer_cloth(n=33, steps=2),
        "folded4x29": W.folded_stack(n=29, steps=2),
    }


@pytest.mark.parametrize("name", list(small_configs()))
def test_assembly_matches_oracle(name):
    w = small_configs()[name]
    c = w.contacts(0)
    compare_assembly(w, w.x0, w.v0, c if c.n else None)


@pytest.mark.parametrize("name", list(small_configs()))
def test_spmv_matches_oracle(name):
    w = small_configs()[name]
    c = w.contacts(0)
    pcl, ref, _, _ = compare_assembly(w, w.x0, w.v0, c if c.n else None)
    rng = np.random.default_rng(11)
    for _ in range(2):
        x = rng.normal(size=(w.n_verts, 3)).astype(np.float32)
        y = pcl.spmv(to_dev(x)).cpu().numpy()
        e = rel_l2(y, ref.spmv(x))
        assert e <= 1e-5, e


@pytest.mark.parametrize("name", list(small_configs()))
def test_pcg_matches_oracle(name):
    w = small_configs()[name]
    c = w.contacts(0)
    pcl, ref, _, _ = compare_assembly(w, w.x0, w.v0, c if c.n else None)
    dv_ref, it_ref, rr_ref, st_ref = ref.pcg(w.tol, w.maxit)
    assert st_ref == oracle.OK
    dv, it, rr, code = pcl.solve(w.tol, w.maxit)
    assert code == pc.OK and rr <= w.tol
    e = rel_l2(dv.cpu().numpy(), dv_ref)
    assert e <= 1e-4, (e, it, it_ref)
    assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)


def test_multistep_per_step_parity():
    """Per-step parity on identical inputs over several steps with changing
    contacts: each step both sides start from the oracle's state."""
    w = W.jittered_cloth(n=48, steps=3)
    pcl = make(w)
    x, v = w.x0, w.v0
    for step in range(3):
        c = w.contacts(step)
        res = oracle.step(w, x, v, c)
        assert res["status"] == oracle.OK
        xd, vd = to_dev(x), to_dev(v)
        dv = torch.empty_like(xd)
        it, rr, code = pcl.step(xd, vd, c, w.h, w.tol, w.maxit, dv)
        assert code == pc.OK
        assert rel_l2(dv.cpu().numpy(), res["dv"]) <= 1e-4
        # v' = v + dv, x' = x + h v': the dv tolerance carries over, plus one
        # fp32 rounding of each update
        dvn = np.linalg.norm(res["dv"])
        vn, xn = np.linalg.norm(res["v"]), np.linalg.norm(res["x"])
        assert rel_l2(vd.cpu().numpy(), res["v"]) <= (1e-4 * dvn) / vn + 4 * 2.0**-24
        assert rel_l2(xd.cpu().numpy(), res["x"]) <= (w.h * 1e-4 * dvn + w.h * 4 * 2.0**-24 * vn) / xn \
            + 4 * 2.0**-24
        x, v = res["x"].astype(np.float32), res["v"].astype(np.float32)


def test_contacts_duplicates_and_spring_pairs():
    """Contacts repeated, reversed and on existing spring pairs merge into
    one block each (filling step 3) with summed values."""
    w = W.tiny_cloth(n=16, rest_from_grid=True)
    a, b = int(w.spring_i[5]), int(w.spring_j[5])
    ci = np.array([a, 3, 40, 3, b, 7], np.int32)
    cj = np.array([b, 40, 3, 40, a, 200], np.int32)
    ck = np.array([1e3, 1e3, 5e2, 2e2, 1e3, 1e3], np.float32)
    cr = np.array([2e-3, 3e-3, 4e-3, 5e-3, 1e-3, 2e-3], np.float32)
    c = W.Contacts(ci, cj, ck, cr)
    w.max_contacts = 16
    compare_assembly(w, w.x0, w.v0, c)


def test_rows_with_new_blocks_on_both_sides_of_the_diagonal():
    """Rows whose new (contact) columns interleave with their spring columns
    below and above the diagonal, with several contacts on one block, on
    spring blocks and on new blocks: the assembly's lanes find every block's
    column and contact run by walking the row (filling steps 1-3), so each
    row's pattern must still come out bit-exact and its values match."""
    w = W.tiny_cloth(n=16, rest_from_grid=True)
    rng = np.random.default_rng(7)
    nv = w.n_verts
    ci, cj = [], []
    for hub in (17, 60, 119, 120, 201, 254):
        springs = np.concatenate([w.spring_j[w.spring_i == hub], w.spring_i[w.spring_j == hub]])
        others = rng.choice(nv, size=10, replace=False)
        partners = [int(o) for o in others if o != hub] + [int(springs[0]), int(springs[-1])]
        partners += partners[:3]   # repeated contacts on the same block
        for q, j in enumerate(partners):
            # both orientations of the pair, as callers may list either
            ci.append(hub if q % 2 == 0 else j)
            cj.append(j if q % 2 == 0 else hub)
    ci, cj = np.array(ci, np.int32), np.array(cj, np.int32)
    nc = len(ci)
    ck = rng.uniform(1e2, 1e3, nc).astype(np.float32)
    cr = rng.uniform(1e-3, 5e-3, nc).astype(np.float32)
    c = W.Contacts(ci, cj, ck, cr)
    w.max_contacts = nc
    compare_assembly(w, w.x0, w.v0, c)


def test_long_rows_exercise_chunked_paths():
    """One vertex in contact with 1500 others: its row is longer than the
    assembly staging and the SpMV chunk, and a tile exceeds both.  Soft
    contacts (k in [1, 10]) near their rest lengths; test_stiff_long_row is
    the same row at contact stiffness."""
    w = W.tiny_cloth(n=48, rest_from_grid=True)
    N = w.n_verts
    hub = N // 2 + 7
    others = np.array([j for j in range(N) if j != hub][:1500], np.int32)
    rng = np.random.default_rng(5)
    dist = np.linalg.norm(w.x0[others].astype(np.float64) - w.x0[hub], axis=1)
    c = W.Contacts(np.full(len(others), hub, np.int32), others,
                   rng.uniform(1.0, 10.0, len(others)).astype(np.float32),
                   (dist * rng.uniform(0.9, 1.1, len(others))).astype(np.float32))
    w.max_contacts = len(others)
    pcl, ref, g, _ = compare_assembly(w, w.x0, w.v0, c)
    assert int(g["rowptr"][hub + 1] - g["rowptr"][hub]) > 1024
    x = np.random.default_rng(2).normal(size=(N, 3)).astype(np.float32)
    assert rel_l2(pcl.spmv(to_dev(x)).cpu().numpy(), ref.spmv(x)) <= 1e-5
    dv_ref, it_ref, _, _ = ref.pcg(w.tol, w.maxit)
    dv, it, rr, code = pcl.solve(w.tol, w.maxit)
    assert code == pc.OK
    assert rel_l2(dv.cpu().numpy(), dv_ref) <= 1e-4


def fp32_storage_floor(ref):
    """Distance between the exact solutions of the oracle's system and of the
    same system rounded to fp32 (A and b), both by a direct fp64 solve: what
    fp32 storage alone moves the solution by, measured from the oracle."""
    sp = pytest.importorskip("scipy.sparse")
    spl = pytest.importorskip("scipy.sparse.linalg")
    n3 = 3 * ref.n
    a64 = sp.bsr_matrix((ref.vals, ref.colind, ref.rowptr), shape=(n3, n3)).tocsc()
    a32 = sp.bsr_matrix((ref.vals.astype(np.float32).astype(np.float64), ref.colind, ref.rowptr),
                        shape=(n3, n3)).tocsc()
    b = ref.b.reshape(-1)
    x64 = spl.spsolve(a64, b)
    x32 = spl.spsolve(a32, b.astype(np.float32).astype(np.float64))
    return float(np.linalg.norm(x32 - x64) / np.linalg.norm(x64))


def test_stiff_long_row():
    """The long-row case at contact stiffness: one vertex joined to 1500
    others by contacts of k in [1e2, 1e3] and rest lengths in [1 mm, 5 cm].
    The hub's diagonal block reaches ~8e5 times its mass, and the hub row of
    every product A p sums 1500 terms that cancel to a small fraction of
    their size; rows that long are summed with compensation in the SpMV.
    This system sits at the fp32 limit: the solve is compared with the
    oracle's PCG at the 1e-4 bar plus the fp32 storage floor measured from
    the oracle itself (about 2.5e-5 here)."""
    w = W.tiny_cloth(n=48, rest_from_grid=True)
    N = w.n_verts
    hub = N // 2 + 7
    others = np.array([j for j in range(N) if j != hub][:1500], np.int32)
    rng = np.random.default_rng(5)
    c = W.Contacts(np.full(len(others), hub, np.int32), others,
                   rng.uniform(1e2, 1e3, len(others)).astype(np.float32),
                   rng.uniform(1e-3, 5e-2, len(others)).astype(np.float32))
    w.max_contacts = len(others)
    pcl, ref, g, _ = compare_assembly(w, w.x0, w.v0, c)
    assert int(g["rowptr"][hub + 1] - g["rowptr"][hub]) > 1024
    x = np.random.default_rng(2).normal(size=(N, 3)).astype(np.float32)
    assert rel_l2(pcl.spmv(to_dev(x)).cpu().numpy(), ref.spmv(x)) <= 1e-5
    dv_ref, it_ref, _, st = ref.pcg(w.tol, w.maxit)
    assert st == oracle.OK
    dv, it, rr, code = pcl.solve(w.tol, w.maxit)
    assert code == pc.OK
    floor = fp32_storage_floor(ref)
    assert floor < 1e-4
    e = rel_l2(dv.cpu().numpy(), dv_ref)
    assert e <= 1e-4 + floor, (e, floor, it, it_ref)
    assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)


def test_pattern_rebuilt_in_place_across_steps():
    """The pattern grows and shrinks with the contacts, always matching the
    oracle, inside the buffers allocated at create."""
    w = W.jittered_cloth(n=40)
    pcl = make(w)
    for step in range(4):
        c = w.contacts(step) if step != 2 else None
        compare_assembly(w, w.x0, w.v0, c, pcl=pcl)
    # back to no contacts: the static pattern
    _, ref, _, _ = compare_assembly(w, w.x0, w.v0, None, pcl=pcl)
    assert ref.nnzb == w.n_verts + 2 * w.n_springs


def test_deterministic_bitwise():
    w = W.folded_stack(n=24)
    c = w.contacts(1)
    outs = []
    for _ in range(2):
        pcl = make(w)
        xd, vd = to_dev(w.x0), to_dev(w.v0)
        pcl.assemble(xd, vd, c, w.h)
        g = pcl.export()
        dv, it, rr, _ = pcl.solve(w.tol, w.maxit)
        outs.append((g["vals"].cpu().numpy(), g["b"].cpu().numpy(), dv.cpu().numpy(), it, rr))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(np.asarray(a), np.asarray(b))


@pytest.mark.parametrize("make_w", [lambda: W.folded_stack(n=29, steps=2),
                                    lambda: W.jittered_cloth(n=48),
                                    lambda: W.tiny_cloth(rest_from_grid=True)],
                         ids=["folded4x29", "jitter48", "tiny32_tension"])
def test_blocks_bitwise_symmetric_and_rows_sum_to_the_mass(make_w):
    """Two properties of Eq. (3)'s matrix that the assembly keeps exactly.
    A_ji = A_ij^T = A_ij: the block (j, i) is computed from the negated edge
    and must carry the bits of the block (i, j).  And the rows of A sum to
    M (every element stiffness is subtracted from the diagonal it adds to):
    the diagonal is formed from the row's stored off-diagonal blocks with a
    compensated sum, so sum_j A_ij - m_i I, taken in fp64 from the stored
    fp32 blocks, stays within the rounding of the diagonal entry (2 ulp) plus
    the compensated sum's own second-order error (2^-40 of the row's sum of
    magnitudes; a plain fp32 sum would leave about 2^-24 of it)."""
    w = make_w()
    c = w.contacts(1)
    pcl = make(w)
    pcl.assemble(to_dev(w.x0), to_dev(w.v0), c if c.n else None, w.h)
    g = pcl.export()
    rowptr = g["rowptr"].cpu().numpy().astype(np.int64)
    colind = g["colind"].cpu().numpy()
    vals = g["vals"].cpu().numpy()
    n = w.n_verts
    rows = np.repeat(np.arange(n), np.diff(rowptr))
    where = {(int(i), int(j)): q for q, (i, j) in enumerate(zip(rows, colind))}
    mirror = np.array([where[(int(j), int(i))] for i, j in zip(rows, colind)])
    bits = vals.view(np.uint32)
    assert np.array_equal(bits, bits[mirror]), "A_ij and A_ji differ in their bits"
    assert np.array_equal(bits, np.transpose(bits, (0, 2, 1))), "a block is not symmetric"
    sums = np.zeros((n, 3, 3))
    np.add.at(sums, rows, vals.astype(np.float64))
    resid = sums - w.mass.astype(np.float64)[:, None, None] * np.eye(3)
    absum = np.zeros((n, 3, 3))
    np.add.at(absum, rows, np.abs(vals.astype(np.float64)))
    diag = vals[rows == colind].astype(np.float64)
    ulp = np.spacing(np.abs(diag).astype(np.float32)).astype(np.float64)
    tol = 2.0 * ulp + 2.0**-40 * absum
    assert np.all(np.abs(resid) <= tol), float(np.max(np.abs(resid) / tol))


def test_zero_stiffness_one_iteration():
    w = W.tiny_cloth(n=12)
    w.spring_k[:] = 0.0
    pcl = make(w)
    xd, vd = to_dev(w.x0), to_dev(w.v0)
    pcl.assemble(xd, vd, None, w.h)
    dv, it, rr, code = pcl.solve(1e-6, 100)
    assert code == pc.OK and it == 1
    np.testing.assert_allclose(dv.cpu().numpy(), np.tile(w.h * w.gravity, (w.n_verts, 1)),
                               rtol=1e-6)


def test_zero_rhs_returns_zero_iterations():
    """b = 0 exactly (no stiffness, no gravity): dv = 0 after 0 iterations."""
    w = W.tiny_cloth(n=10)
    w.gravity[:] = 0.0
    w.spring_k[:] = 0.0
    pcl = make(w)
    xd, vd = to_dev(w.x0), to_dev(w.v0)
    pcl.assemble(xd, vd, None, w.h)
    dv, it, rr, code = pcl.solve(1e-6, 100)
    assert code == pc.OK and it == 0 and rr == 0.0
    assert float(dv.abs().max()) == 0.0


def test_maxit_and_error_codes():
    w = W.tiny_cloth(n=20, rest_from_grid=True)
    w.max_contacts = 2
    pcl = make(w)
    xd, vd = to_dev(w.x0), to_dev(w.v0)
    pcl.assemble(xd, vd, None, w.h)
    dv, it, rr, code = pcl.solve(1e-12, 1)
    assert code == pc.NOT_CONVERGED and it == 1 and rr > 1e-12
    dv, it, rr, code = pcl.solve(1e-6, 0)
    assert code == pc.NOT_CONVERGED and it == 0 and abs(rr - 1.0) < 1e-12
    # out-of-range, self contact
    for ci, cj in ((0, w.n_verts), (-1, 3), (4, 4)):
        bad = W.Contacts(np.array([ci], np.int32), np.array([cj], np.int32),
                         np.array([1.0], np.float32), np.array([0.1], np.float32))
        pcl.assemble(xd, vd, bad, w.h)
        with pytest.raises(pc.PClothError) as ei:
            pcl.nnzb()
        assert ei.value.code == pc.ERR_BAD_INDEX
    # more contacts than max_contacts
    many = W.Contacts(np.zeros(3, np.int32), np.ones(3, np.int32),
                      np.ones(3, np.float32), np.ones(3, np.float32))
    with pytest.raises(pc.PClothError) as ei:
        pcl.assemble(xd, vd, many, w.h)
    assert ei.value.code == pc.ERR_CAPACITY
    # NaN velocity
    vbad = vd.clone()
    vbad[3, 1] = float("nan")
    pcl.assemble(xd, vbad, None, w.h)
    with pytest.raises(pc.PClothError) as ei:
        pcl.solve(1e-6, 100)
    assert ei.value.code == pc.ERR_NONFINITE
    # the handle is usable again afterwards
    pcl.assemble(xd, vd, None, w.h)
    dv, it, rr, code = pcl.solve(1e-6, 10000)
    assert code == pc.OK


def test_solve_before_assemble_is_rejected():
    w = W.tiny_cloth(n=8)
    pcl = make(w)
    with pytest.raises(pc.PClothError) as ei:
        pcl.solve(1e-6, 10)
    assert ei.value.code == pc.ERR_STATE


def test_step_host_matches_device_step():
    w = W.jittered_cloth(n=40)
    c = w.contacts(0)
    pcl = make(w)
    xd, vd = to_dev(w.x0), to_dev(w.v0)
    it_d, rr_d, _ = pcl.step(xd, vd, c, w.h, w.tol, w.maxit)
    xh = torch.from_numpy(w.x0.copy()).pin_memory()
    vh = torch.from_numpy(w.v0.copy()).pin_memory()
    it_h, rr_h, _ = pcl.step_host(xh, vh, c, w.h, w.tol, w.maxit)
    assert it_h == it_d and rr_h == rr_d
    assert torch.equal(xh, xd.cpu()) and torch.equal(vh, vd.cpu())


def test_repeated_and_interleaved_solves_are_bitwise_identical():
    """Each solve is one persistent kernel with its own barrier counter:
    solving again on the same handle, and interleaving solves of two handles
    on one stream, gives the same bits every time."""
    w = W.drooped_cloth(n=30)
    pcls = [make(w), make(w)]
    for pcl in pcls:
        pcl.assemble(to_dev(w.x0), to_dev(w.v0), None, w.h)
    res = []
    for rep in range(3):
        for pcl in pcls:
            dv, it, rr, code = pcl.solve(w.tol, w.maxit)
            assert code == pc.OK
            res.append((dv.cpu().numpy(), it, rr))
    for r in res[1:]:
        assert np.array_equal(r[0], res[0][0]) and r[1] == res[0][1] and r[2] == res[0][2]


def test_profiling_times_every_iteration_and_changes_nothing():
    """With profiling on, the PCG kernel times its SpMV phase once per
    iteration (its vector phases too) and the results keep their bits;
    resetting the counters keeps profiling on."""
    w = W.drooped_cloth(n=30)
    ref_pcl = make(w)
    xr, vr = to_dev(w.x0), to_dev(w.v0)
    it_ref, rr_ref, _ = ref_pcl.step(xr, vr, None, w.h, w.tol, w.maxit)
    for mode in (2, 1):
        pcl = make(w)
        pcl.profile(mode)
        pcl.profile_read(reset=True)
        xd, vd = to_dev(w.x0), to_dev(w.v0)
        it, rr, _ = pcl.step(xd, vd, None, w.h, w.tol, w.maxit)
        p = pcl.profile_read(reset=True)
        assert it == it_ref and rr == rr_ref
        assert torch.equal(xd, xr) and torch.equal(vd, vr)
        assert p["iterations"] == it and p["samples"] == it, (mode, p, it)
        assert p["spmv_ms"] > 0 and p["update_ms"] > 0 and p["assemble_calls"] == 1
        assert p["solve_ms"] >= p["spmv_ms"]


@pytest.mark.parametrize("name", ["droop37", "twolayer33", "folded4x29"])
def test_block_ell_spmv_matches_oracle_and_bsr3(name):
    """The pages' block-ELL layout (P-Cloth Sec. 3.2.2 tables) gives the same
    product as the oracle (1e-5) and the same bits as the BSR3 kernel (same
    products in the same order)."""
    w = small_configs()[name]
    c = w.contacts(0)
    pcl, ref, _, _ = compare_assembly(w, w.x0, w.v0, c if c.n else None)
    W = pcl.bell_build()
    g = pcl.export()
    lengths = np.diff(g["rowptr"].cpu().numpy())
    assert W == int(lengths.max())
    x = np.random.default_rng(12).normal(size=(w.n_verts, 3)).astype(np.float32)
    xd = to_dev(x)
    y_bell = pcl.spmv_bell(xd)
    y_bsr = pcl.spmv(xd)
    assert rel_l2(y_bell.cpu().numpy(), ref.spmv(x)) <= 1e-5
    assert torch.equal(y_bell, y_bsr)


def test_block_ell_copy_is_invalid_after_the_next_assembly():
    w = W.jittered_cloth(n=40, steps=2)
    pcl = make(w)
    xd, vd = to_dev(w.x0), to_dev(w.v0)
    pcl.assemble(xd, vd, w.contacts(0), w.h)
    pcl.bell_build()
    pcl.spmv_bell(xd)
    pcl.assemble(xd, vd, w.contacts(1), w.h)
    with pytest.raises(pc.PClothError) as ei:
        pcl.spmv_bell(xd)
    assert ei.value.code == pc.ERR_STATE
    pcl.bell_build()
    assert torch.equal(pcl.spmv_bell(xd), pcl.spmv(xd))
