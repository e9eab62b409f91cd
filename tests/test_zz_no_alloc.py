"""The allocation-free solve entry point (pcloth_solve_bsr3_static).

It exists for callers that cannot allocate GPU memory when they need a
solve -- a host application that reserves the GPU's memory for itself and
forbids plug-ins to allocate, or a real-time loop where an allocation's
latency or failure mid-frame is unacceptable.  It keeps all of its scratch
in one fixed array inside the library, shared by every call on a device.

These tests call it through the C ABI on a system assembled by the regular
path and check it against the regular solve (pcloth_solve) with the same
tolerances the other PCG parity tests use: relative L2 of dv <= 1e-4 and
iteration counts within max(3, 3%).  Two calls in a row must both agree --
the second call finds the first call's leftovers in the shared array.  The
file is collected last so that a failure here does not hide the others.
"""
import numpy as np
import pytest
import torch

from sparse_linear_solve_gb300 import pcloth as pc
from sparse_linear_solve_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


def rel_l2(a, b):
    a = np.asarray(a, np.float64).reshape(-1)
    b = np.asarray(b, np.float64).reshape(-1)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def assembled(w, step=0):
    cloth = pc.PCloth.from_workload(w, device=DEV)
    x = torch.from_numpy(w.x0).to(DEV)
    v = torch.from_numpy(w.v0).to(DEV)
    c = w.contacts(step)
    cloth.assemble(x, v, c if c.n else None, w.h)
    return cloth, cloth.export()


@pytest.mark.parametrize("make", [lambda: W.jittered_cloth(n=64), lambda: W.tiny_cloth(n=40)],
                         ids=["jittered64_contacts", "tiny40"])
def test_static_solve_matches_regular_solve_twice(make):
    w = make()
    assert w.n_verts <= pc.STATIC_MAX_VERTS
    cloth, g = assembled(w)
    dv_ref, it_ref, rr_ref, code_ref = cloth.solve(w.tol, w.maxit)
    assert code_ref == pc.OK
    for _ in range(2):
        dv = torch.full((w.n_verts, 3), float("nan"), dtype=torch.float32, device=DEV)
        it, rr, code = pc.pcloth_solve_bsr3_static(w.n_verts, g["rowptr"], g["colind"],
                                                   g["vals"], g["b"], w.tol, w.maxit, dv)
        torch.cuda.synchronize()
        assert code == pc.OK and rr <= w.tol
        assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)
        assert rel_l2(dv.cpu().numpy(), dv_ref.cpu().numpy()) <= 1e-4


def test_static_solve_after_a_larger_call_and_not_converged():
    """A small system after a larger one (stale data in the shared array),
    and maxit = 1 reports NOT_CONVERGED with one iteration."""
    big, gb = assembled(W.jittered_cloth(n=96))
    dvb = torch.empty((big.n, 3), dtype=torch.float32, device=DEV)
    pc.pcloth_solve_bsr3_static(big.n, gb["rowptr"], gb["colind"], gb["vals"], gb["b"],
                                1e-6, 20000, dvb)
    w = W.tiny_cloth(n=24, rest_from_grid=True)
    cloth, g = assembled(w)
    dv_ref, it_ref, _, _ = cloth.solve(w.tol, w.maxit)
    dv = torch.empty_like(dv_ref)
    it, rr, code = pc.pcloth_solve_bsr3_static(w.n_verts, g["rowptr"], g["colind"], g["vals"],
                                               g["b"], w.tol, w.maxit, dv)
    assert code == pc.OK and abs(it - it_ref) <= max(3, 0.03 * it_ref)
    assert rel_l2(dv.cpu().numpy(), dv_ref.cpu().numpy()) <= 1e-4
    it, rr, code = pc.pcloth_solve_bsr3_static(w.n_verts, g["rowptr"], g["colind"], g["vals"],
                                               g["b"], 1e-12, 1, dv)
    assert code == pc.NOT_CONVERGED and it == 1


def test_static_solve_rejects_sizes_beyond_the_maximum():
    n = pc.STATIC_MAX_VERTS + 1
    dummy = torch.zeros(8, dtype=torch.float32, device=DEV)
    with pytest.raises(pc.PClothError) as ei:
        pc.pcloth_solve_bsr3_static(n, dummy, dummy, dummy, dummy, 1e-6, 10, dummy)
    assert ei.value.code == pc.ERR_CAPACITY
    assert "PCLOTH_STATIC_MAX_VERTS" in str(ei.value)
