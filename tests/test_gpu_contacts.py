"""Vertex-vertex proximity contacts on the GPU (spatial hashing) against the
brute-force oracle: the (i, j) lists are compared exactly (integer output;
the distance test is float32 on both sides).  P-Cloth Sec. 4.2-4.3,
restricted to vertex pairs."""
import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_linear_solve_gb300 import pcloth as pc
from sparse_linear_solve_gb300 import workloads as W

from gpu_helpers import DEV, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def springs_of(w):
    return (w.spring_i, w.spring_j)


def cloud(n, box, seed, clusters=0):
    rng = np.random.default_rng(seed)
    x = rng.uniform(-box, box, size=(n, 3))
    if clusters:   # a few tight clumps with many close pairs
        c = rng.uniform(-box, box, size=(clusters, 3))
        idx = rng.integers(0, clusters, size=n // 4)
        x[: n // 4] = c[idx] + rng.normal(0, box * 1e-3, size=(n // 4, 3))
    return x.astype(np.float32)


def gpu_pairs(pcl, x, radius, capacity=None):
    (i, j, k, rest), found = pcl.find_contacts(to_dev(x), radius, 1e3, capacity)
    return i.cpu().numpy(), j.cpu().numpy(), k.cpu().numpy(), rest.cpu().numpy(), found


@pytest.mark.parametrize("name", ["folded", "twolayer", "cloud", "cloud_clusters", "far"])
def test_contacts_match_oracle(name):
    if name == "folded":
        w = W.folded_stack(n=29, steps=1)
        x, radius = w.x0, 2e-3
    elif name == "twolayer":
        # the top layer sits half a cell off, 2 mm up: nearest pairs 7.35 mm
        w = W.two_layer_cloth(n=33, steps=1)
        x, radius = w.x0, 8e-3
    else:
        w = W.tiny_cloth(n=24)      # springs among the first 576 vertices only
        n = 3000
        box = {"cloud": 0.05, "cloud_clusters": 0.05, "far": 0.05}[name]
        x = cloud(n, box, 7, clusters=8 if name == "cloud_clusters" else 0)
        if name == "far":
            x = x + np.float32(37.5)   # far from the origin: cells still neighbour
        x[: w.n_verts] = w.x0
        w.mass = np.concatenate([w.mass, np.full(n - w.n_verts, 1e-4, np.float32)])
        w.n_verts = n
        radius = 3e-3
    w.max_contacts = 200000
    pcl = pc.PCloth.from_workload(w, device=DEV)
    oi, oj, total = oracle.find_contacts(x, radius, springs_of(w))
    gi, gj, gk, gr, found = gpu_pairs(pcl, x, radius)
    assert found == total and total > 0
    assert np.array_equal(gi, oi) and np.array_equal(gj, oj)
    assert np.all(gk == np.float32(1e3)) and np.all(gr == np.float32(radius))


def test_contacts_capacity_and_empty():
    w = W.tiny_cloth(n=8)
    w.max_contacts = 100
    pcl = pc.PCloth.from_workload(w, device=DEV)
    x = np.zeros((w.n_verts, 3), np.float32)   # every pair at distance 0
    _, _, total = oracle.find_contacts(x, 1e-3, springs_of(w))
    with pytest.raises(pc.PClothError) as ei:
        pcl.find_contacts(to_dev(x), 1e-3, 1e3)
    assert ei.value.code == pc.ERR_CAPACITY and ei.value.found == total
    # nothing closer than the radius: an empty list
    gi, gj, gk, gr, found = gpu_pairs(pcl, w.x0, 1e-4)
    assert found == 0 and len(gi) == 0


def test_contacts_at_exactly_the_capacity():
    """As many pairs as the capacity allows: all are written; one more pair
    than the capacity: nothing is written and the count is reported."""
    w = W.tiny_cloth(n=24)
    n = 3000
    x = cloud(n, 0.05, 11, clusters=4)
    x[: w.n_verts] = w.x0
    w.mass = np.concatenate([w.mass, np.full(n - w.n_verts, 1e-4, np.float32)])
    w.n_verts = n
    w.max_contacts = 200000
    pcl = pc.PCloth.from_workload(w, device=DEV)
    oi, oj, total = oracle.find_contacts(x, 3e-3, springs_of(w))
    assert total > 1
    gi, gj, _, _, found = gpu_pairs(pcl, x, 3e-3, capacity=total)
    assert found == total and np.array_equal(gi, oi) and np.array_equal(gj, oj)
    with pytest.raises(pc.PClothError) as ei:
        pcl.find_contacts(to_dev(x), 3e-3, 1e3, total - 1)
    assert ei.value.code == pc.ERR_CAPACITY and ei.value.found == total


def test_contacts_with_colliding_cells():
    """Two of the cells a vertex searches that share a bucket of the spatial
    hash table (of 1,024 buckets for a cloud this small): the partner in one
    of them must be found once, not once per cell that hashes to its bucket.
    Cells have edge 2 r (1 + 2^-7); a vertex a quarter of the way into its
    cell searches it and the cells below it.  The cells were found by a
    search with the hash written out in numpy: at r = 3 mm the searched
    cells (828, 826, 826) and (827, 827, 826) share bucket 444."""
    w = W.tiny_cloth(n=8)
    r = np.float32(3e-3)
    edge = np.float32(np.float32(2) * r * np.float32(1 + 1 / 128))
    ca = np.array([828, 827, 826], np.float32)
    xa = ((ca + np.float32(0.25)) * edge).astype(np.float32)
    xb = xa - np.array([0, 0.3, 0], np.float32) * edge   # in cell (828, 826, 826)
    inv = np.float32(1) / edge
    assert np.array_equal(np.floor(xa * inv), ca)
    assert np.array_equal(np.floor(xb * inv), ca - np.array([0, 1, 0], np.float32))
    x = np.concatenate([w.x0, xa[None], xb[None]]).astype(np.float32)
    w.mass = np.concatenate([w.mass, np.full(2, 1e-4, np.float32)])
    w.n_verts = len(x)
    w.max_contacts = 1000
    pcl = pc.PCloth.from_workload(w, device=DEV)
    oi, oj, total = oracle.find_contacts(x, float(r), springs_of(w))
    gi, gj, gk, gr, found = gpu_pairs(pcl, x, float(r))
    assert found == total and np.array_equal(gi, oi) and np.array_equal(gj, oj)
    assert (w.n_verts - 2, w.n_verts - 1) in set(zip(gi.tolist(), gj.tolist()))


def test_contacts_count_past_int32():
    """65,600 vertices at one point: 2,151,647,200 pairs, past 2^31 - 1 less
    the springs.  The count must still exceed the capacity (not wrap), the
    call must write nothing, and the reported count saturates at 2^31 - 1."""
    w = W.tiny_cloth(n=8)
    n = 65600
    w.mass = np.concatenate([w.mass, np.full(n - w.n_verts, 1e-4, np.float32)])
    w.n_verts = n
    w.max_contacts = 100
    pcl = pc.PCloth.from_workload(w, device=DEV)
    x = np.zeros((n, 3), np.float32)
    pairs = n * (n - 1) // 2 - len(w.spring_i)
    assert pairs > 2**31 - 1
    with pytest.raises(pc.PClothError) as ei:
        pcl.find_contacts(to_dev(x), 1e-3, 1e3)
    assert ei.value.code == pc.ERR_CAPACITY and ei.value.found == 2**31 - 1


def test_found_contacts_drive_a_step_like_the_oracle():
    """The found list, fed to the step, gives the oracle's step with the
    oracle's own list."""
    w = W.folded_stack(n=24, steps=1)
    w.max_contacts = 200000
    pcl = pc.PCloth.from_workload(w, device=DEV)
    (ci, cj, ck, cr), found = pcl.find_contacts(to_dev(w.x0), 2e-3, 1e3)
    assert found > 0
    oi, oj, _ = oracle.find_contacts(w.x0, 2e-3, springs_of(w))
    contacts = W.Contacts(oi, oj, np.full(len(oi), 1e3, np.float32), np.full(len(oi), 2e-3, np.float32))
    ref = oracle.assemble_workload(w, w.x0, w.v0, contacts)
    dv_ref, it_ref, _, _ = ref.pcg(w.tol, w.maxit)
    xd, vd = to_dev(w.x0), to_dev(w.v0)
    dv = torch.empty_like(xd)
    it, rr, code = pcl.step(xd, vd, (ci, cj, ck, cr), w.h, w.tol, w.maxit, dv)
    assert code == pc.OK and rr <= w.tol
    assert abs(it - it_ref) <= max(3, 0.03 * it_ref)
    assert rel_l2(dv.cpu().numpy(), dv_ref) <= 1e-4


def test_contacts_at_full_size_sampled():
    """The 1.65M-triangle folded stack: every returned pair passes the test
    and is no spring; for 1500 sampled vertices, brute force over all
    vertices finds exactly the returned partners."""
    w = W.make("C5")
    w.max_contacts = 4000000
    pcl = pc.PCloth.from_workload(w, device=DEV)
    radius = 2e-3
    gi, gj, _, _, found = gpu_pairs(pcl, w.x0, radius)
    assert found == len(gi) > 0
    x = w.x0.astype(np.float32)
    d = x[gj] - x[gi]
    d2 = (d[:, 0] * d[:, 0] + d[:, 1] * d[:, 1]) + d[:, 2] * d[:, 2]
    assert np.all(gi < gj) and np.all(d2 < np.float32(radius) * np.float32(radius))
    assert np.all(np.diff(gi.astype(np.int64) * w.n_verts + gj) > 0)   # (i, j) order, unique
    springs = set(zip(np.minimum(w.spring_i, w.spring_j).tolist(),
                      np.maximum(w.spring_i, w.spring_j).tolist()))
    assert not any((a, b) in springs for a, b in zip(gi[:20000].tolist(), gj[:20000].tolist()))
    rng = np.random.default_rng(9)
    r2 = np.float32(radius) * np.float32(radius)
    partners = {}
    for a, b in zip(gi.tolist(), gj.tolist()):
        partners.setdefault(a, set()).add(b)
        partners.setdefault(b, set()).add(a)
    for v in rng.choice(w.n_verts, 1500, replace=False):
        dv = x - x[v]
        dd = (dv[:, 0] * dv[:, 0] + dv[:, 1] * dv[:, 1]) + dv[:, 2] * dv[:, 2]
        near = set(np.nonzero(dd < r2)[0].tolist()) - {int(v)}
        near = {u for u in near if (min(u, v), max(u, v)) not in springs}
        assert near == partners.get(int(v), set()), v
