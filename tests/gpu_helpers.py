"""Helpers shared by the GPU parity tests: run one step on both sides from
identical seeded inputs and compare (P-Cloth, arXiv 2008.00409, Sec. 2.5
Eq. (3) and Sec. 3.2.2)."""
import numpy as np
import torch

from oracle import oracle
from sparse_linear_solve_gb300 import pcloth as pc

DEV = torch.device("cuda", 0)


def to_dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=DEV, dtype=dtype)


def make(w):
    return pc.PCloth.from_workload(w, device=DEV)


def block_rel_err(vals_gpu, vals_ref):
    """Max over blocks of |B_gpu - B_ref|_F / |B_ref|_F (floored at 1e-30)."""
    d = np.linalg.norm((vals_gpu.astype(np.float64) - vals_ref).reshape(len(vals_ref), -1), axis=1)
    r = np.linalg.norm(vals_ref.reshape(len(vals_ref), -1), axis=1)
    return float((d / np.maximum(r, 1e-30)).max()) if len(r) else 0.0


def rhs_scale(w, contacts, x, v):
    """Per-vertex magnitude of the terms summed into b_i = h (sum F_e + m g):
    h (sum_e k_e (|x~_j - x~_i| + L0_e) + m |g|).  A floating-point sum is
    accurate relative to the sum of the magnitudes of its terms, not to its
    (possibly cancelling) total; this is the scale of the b check."""
    h = w.h
    xt = x.astype(np.float64) + h * v.astype(np.float64)
    s = np.full(w.n_verts, float(np.linalg.norm(w.gravity.astype(np.float64))))
    s *= w.mass.astype(np.float64)
    els = [(w.spring_i, w.spring_j, w.spring_k, w.spring_rest)]
    if contacts is not None and contacts.n:
        els.append((contacts.i, contacts.j, contacts.k, contacts.rest))
    for i, j, k, r in els:
        lt = np.linalg.norm(xt[j] - xt[i], axis=1)
        mag = k.astype(np.float64) * (lt + r.astype(np.float64))
        np.add.at(s, i, mag)
        np.add.at(s, j, mag)
    return h * s


def compare_assembly(w, x, v, contacts, pcl=None, tol_block=1e-5, tol_b=1e-5):
    """Assemble on both sides and check pattern (bit-exact), blocks, b, P."""
    ref = oracle.assemble_workload(w, x, v, contacts)
    assert ref.status == oracle.OK
    if pcl is None:
        pcl = make(w)
    xd, vd = to_dev(x), to_dev(v)
    pcl.assemble(xd, vd, contacts, w.h)
    g = pcl.export()
    rowptr = g["rowptr"].cpu().numpy()
    colind = g["colind"].cpu().numpy()
    assert np.array_equal(rowptr, ref.rowptr.astype(np.int32)), "rowptr differs"
    assert np.array_equal(colind, ref.colind), "colind differs"
    vals = g["vals"].cpu().numpy()
    e_blk = block_rel_err(vals, ref.vals)
    assert e_blk <= tol_block, "block rel err %.3g" % e_blk
    b = g["b"].cpu().numpy().astype(np.float64)
    scale = rhs_scale(w, contacts, x, v)
    e_b = float((np.abs(b - ref.b).max(axis=1) / scale).max())
    assert e_b <= tol_b, "rhs err %.3g (relative to the summed magnitudes)" % e_b
    pinv = g["pinv"].cpu().numpy().astype(np.float64)
    e_p = check_pinv(pinv, vals, ref, rowptr, colind)
    return pcl, ref, g, dict(block=e_blk, b=e_b, pinv=e_p)


EPS32 = 2.0 ** -24


def diag_blocks(vals, rowptr, colind):
    n = len(rowptr) - 1
    rows = np.repeat(np.arange(n), np.diff(rowptr))
    return vals[np.nonzero(colind == rows)[0]]


def check_pinv(pinv, vals_gpu, ref, rowptr, colind):
    """Block-Jacobi inverses.  The GPU inverts its own fp32 diagonal block
    D_gpu, which differs from the oracle's D by rounding; the perturbation
    bound of a matrix inverse gives, per block,
        |P_gpu - P_ref| / |P_ref| <= kappa(D) (|D_gpu - D_ref| / |D_ref| + c eps)
    and the fp32 adjugate itself leaves |P_gpu D_gpu - I| <= c kappa(D) eps."""
    Dg = diag_blocks(vals_gpu.astype(np.float64), rowptr, colind)
    Dr = diag_blocks(ref.vals, rowptr, colind)
    kappa = np.linalg.cond(Dr)
    dD = np.linalg.norm((Dg - Dr).reshape(len(Dr), -1), axis=1) / \
        np.linalg.norm(Dr.reshape(len(Dr), -1), axis=1)
    err = np.linalg.norm((pinv - ref.pinv).reshape(len(Dr), -1), axis=1) / \
        np.linalg.norm(ref.pinv.reshape(len(Dr), -1), axis=1)
    bound = 4.0 * kappa * (dD + 16 * EPS32)
    worst = int(np.argmax(err / bound))
    assert np.all(err <= bound), "P block %d: err %.3g > bound %.3g (kappa %.3g)" % (
        worst, err[worst], bound[worst], kappa[worst])
    resid = np.abs(np.einsum("nij,njk->nik", pinv, Dg) - np.eye(3)).max(axis=(1, 2))
    assert np.all(resid <= 16 * kappa * EPS32 + 1e-6), float((resid / kappa).max())
    return float(err.max())


def rel_l2(a, b):
    a = np.asarray(a, np.float64).reshape(-1)
    b = np.asarray(b, np.float64).reshape(-1)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
