"""The allocation-free solve entry point (pcloth_solve_bsr3_static).

It exists for callers that cannot allocate GPU memory when they need a
solve -- a host application that reserves the GPU's memory for itself and
forbids plug-ins to allocate, or a real-time loop where an allocation's
latency or failure mid-frame is unacceptable.  It keeps all of its scratch
in one fixed array inside the library, shared by every call on a device.

These tests call it through the C ABI on a system assembled by the regular
path and check it against the regular solve (pcloth_solve) and against the
fp64 oracle's PCG of the same system, with the tolerances the other PCG
parity tests use: relative L2 of dv <= 1e-4 and iteration counts within
max(3, 3%).  Two calls in a row must both agree -- the second call finds the
first call's leftovers in the shared array.  A warm call must change no
device allocation.  Misaligned arrays and malformed patterns are rejected
before the solve runs.  The file is collected last so that a failure here
does not hide the others.
"""
import gc

import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_linear_solve_gb300 import pcloth as pc
from sparse_linear_solve_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
SLACK = 64   # elements of readable memory after every array the solve streams


def rel_l2(a, b):
    a = np.asarray(a, np.float64).reshape(-1)
    b = np.asarray(b, np.float64).reshape(-1)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def padded(t):
    """A copy of t at the start of a larger buffer: 16-byte aligned, with the
    readable slack after its end that the entry point asks for."""
    flat = torch.zeros(t.numel() + SLACK, dtype=t.dtype, device=DEV)
    flat[:t.numel()].copy_(t.reshape(-1))
    return flat[:t.numel()].view(t.shape)


def assembled(w, step=0):
    cloth = pc.PCloth.from_workload(w, device=DEV)
    x = torch.from_numpy(w.x0).to(DEV)
    v = torch.from_numpy(w.v0).to(DEV)
    c = w.contacts(step)
    cloth.assemble(x, v, c if c.n else None, w.h)
    g = cloth.export()
    for key in ("rowptr", "colind", "vals"):
        g[key] = padded(g[key])
    return cloth, g


def static_solve(n, g, tol, maxit, dv):
    return pc.pcloth_solve_bsr3_static(n, g["rowptr"], g["colind"], g["vals"], g["b"], tol,
                                       maxit, dv)


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
        it, rr, code = static_solve(w.n_verts, g, w.tol, w.maxit, dv)
        torch.cuda.synchronize()
        assert code == pc.OK and rr <= w.tol
        assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)
        assert rel_l2(dv.cpu().numpy(), dv_ref.cpu().numpy()) <= 1e-4


@pytest.mark.parametrize("make", [lambda: W.jittered_cloth(n=64), lambda: W.folded_stack(n=29)],
                         ids=["jittered64_contacts", "folded4x29"])
def test_static_solve_matches_the_oracle(make):
    """The same PCG on the same system as the fp64 oracle (P-Cloth Sec. 2.5
    Eq. (3), Sec. 3.1), from the oracle's own assembly of the inputs."""
    w = make()
    c = w.contacts(0)
    ref = oracle.assemble_workload(w, w.x0, w.v0, c if c.n else None)
    dv_ref, it_ref, _, st = ref.pcg(w.tol, w.maxit)
    assert st == oracle.OK
    _, g = assembled(w)
    dv = torch.empty((w.n_verts, 3), dtype=torch.float32, device=DEV)
    it, rr, code = static_solve(w.n_verts, g, w.tol, w.maxit, dv)
    assert code == pc.OK and rr <= w.tol
    assert rel_l2(dv.cpu().numpy(), dv_ref) <= 1e-4
    assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)


def test_static_solve_after_a_larger_call_and_not_converged():
    """A small system after a larger one (stale data in the shared array),
    and maxit = 1 reports NOT_CONVERGED with one iteration."""
    big, gb = assembled(W.jittered_cloth(n=96))
    dvb = torch.empty((big.n, 3), dtype=torch.float32, device=DEV)
    static_solve(big.n, gb, 1e-6, 20000, dvb)
    w = W.tiny_cloth(n=24, rest_from_grid=True)
    cloth, g = assembled(w)
    dv_ref, it_ref, _, _ = cloth.solve(w.tol, w.maxit)
    dv = torch.empty_like(dv_ref)
    it, rr, code = static_solve(w.n_verts, g, w.tol, w.maxit, dv)
    assert code == pc.OK and abs(it - it_ref) <= max(3, 0.03 * it_ref)
    assert rel_l2(dv.cpu().numpy(), dv_ref.cpu().numpy()) <= 1e-4
    it, rr, code = static_solve(w.n_verts, g, 1e-12, 1, dv)
    assert code == pc.NOT_CONVERGED and it == 1


def test_warm_call_changes_no_device_allocation():
    """After one warm-up call (which may load the library's device code),
    further calls leave the device's free memory and torch's pool as they
    were: the entry point allocates nothing."""
    w = W.jittered_cloth(n=48)
    cloth, g = assembled(w)
    dv = torch.empty((w.n_verts, 3), dtype=torch.float32, device=DEV)
    static_solve(w.n_verts, g, w.tol, w.maxit, dv)
    gc.collect()   # handles of earlier tests are freed now, not in between
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(DEV)
    alloc0, res0 = torch.cuda.memory_allocated(DEV), torch.cuda.memory_reserved(DEV)
    for _ in range(3):
        it, rr, code = static_solve(w.n_verts, g, w.tol, w.maxit, dv)
        assert code == pc.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(DEV)
    # nothing was allocated, so the device's free memory cannot have fallen
    # (it may rise if something else in the process releases memory)
    assert free1 >= free0, (free0, free1)
    assert torch.cuda.memory_allocated(DEV) == alloc0
    assert torch.cuda.memory_reserved(DEV) == res0
    del cloth


def test_tiny_but_well_conditioned_system():
    """A scaled by 1e-13 (b kept, so dv grows by 1e13 and every PCG scalar
    stays in fp32 range): the diagonal blocks' determinants, about 1e-39,
    would underflow fp32 unscaled; the solution is unchanged."""
    w = W.tiny_cloth(n=24, rest_from_grid=True)
    cloth, g = assembled(w)
    dv_ref, it_ref, _, _ = cloth.solve(w.tol, w.maxit)
    gs = dict(g)
    gs["vals"] = padded(g["vals"] * 1e-13)
    dv = torch.empty_like(dv_ref)
    it, rr, code = static_solve(w.n_verts, gs, w.tol, w.maxit, dv)
    assert code == pc.OK and abs(it - it_ref) <= max(3, 0.03 * it_ref), (code, it, it_ref)
    assert rel_l2(dv.cpu().numpy() * 1e-13, dv_ref.cpu().numpy()) <= 1e-4


def test_misaligned_arrays_are_rejected_before_any_launch():
    w = W.tiny_cloth(n=12)
    _, g = assembled(w)
    dv = torch.empty((w.n_verts, 3), dtype=torch.float32, device=DEV)
    for key in ("rowptr", "colind", "vals"):
        t = g[key]
        flat = torch.zeros(t.numel() + SLACK, dtype=t.dtype, device=DEV)
        view = flat[1:1 + t.numel()].view(t.shape)   # 4 bytes past a 16-byte boundary
        view.copy_(t)
        bad = dict(g)
        bad[key] = view
        with pytest.raises(pc.PClothError) as ei:
            static_solve(w.n_verts, bad, w.tol, w.maxit, dv)
        assert ei.value.code == pc.ERR_INVALID_ARG
        assert "16-byte aligned" in str(ei.value)


def _malformed_cases(g, n):
    """Host-made malformed patterns; every array keeps rowptr[n] readable
    column entries, so the check that rejects them never reads out of range."""
    rp = g["rowptr"].cpu().numpy().copy()
    ci = g["colind"].cpu().numpy().copy()
    cases = {}
    c = ci.copy()
    c[rp[3]] = n                                  # a column equal to n
    cases["column_n"] = (rp.copy(), c)
    c = ci.copy()
    c[rp[4]] = -1                                 # a negative column
    cases["column_negative"] = (rp.copy(), c)
    r = rp.copy()
    r[6] = r[7] + 1                               # rowptr decreasing
    cases["rowptr_decreasing"] = (r, ci.copy())
    r = rp.copy()
    r[0] = 1                                      # rowptr[0] != 0
    cases["rowptr_start"] = (r, ci.copy())
    c = ci.copy()
    c[rp[5]], c[rp[5] + 1] = c[rp[5] + 1], c[rp[5]]   # unsorted row
    cases["unsorted_row"] = (rp.copy(), c)
    c = ci.copy()
    c[rp[8] + 1] = c[rp[8]]                       # duplicate column
    cases["duplicate_column"] = (rp.copy(), c)
    return cases


def test_malformed_patterns_are_rejected_and_the_device_stays_usable():
    w = W.tiny_cloth(n=12)
    cloth, g = assembled(w)
    n = w.n_verts
    dv = torch.empty((n, 3), dtype=torch.float32, device=DEV)
    for name, (r, c) in _malformed_cases(g, n).items():
        bad = dict(g)
        bad["rowptr"] = padded(torch.from_numpy(r).to(DEV))
        bad["colind"] = padded(torch.from_numpy(c).to(DEV))
        with pytest.raises(pc.PClothError) as ei:
            static_solve(n, bad, w.tol, w.maxit, dv)
        assert ei.value.code == pc.ERR_BAD_INDEX, name
    # a 2-vertex matrix of off-diagonal blocks only: no diagonal
    rp2 = padded(torch.tensor([0, 1, 2], dtype=torch.int32, device=DEV))
    ci2 = padded(torch.tensor([1, 0], dtype=torch.int32, device=DEV))
    v2 = padded(torch.eye(3, device=DEV).repeat(2, 1, 1))
    b2 = torch.ones((2, 3), device=DEV)
    with pytest.raises(pc.PClothError) as ei:
        pc.pcloth_solve_bsr3_static(2, rp2, ci2, v2, b2, 1e-6, 10, dv[:2])
    assert ei.value.code == pc.ERR_BAD_INDEX
    # the device and the shared array are fine afterwards
    dv_ref, it_ref, _, _ = cloth.solve(w.tol, w.maxit)
    it, rr, code = static_solve(n, g, w.tol, w.maxit, dv)
    assert code == pc.OK and rel_l2(dv.cpu().numpy(), dv_ref.cpu().numpy()) <= 1e-4


def test_static_solve_rejects_sizes_beyond_the_maximum():
    n = pc.STATIC_MAX_VERTS + 1
    dummy = torch.zeros(8, dtype=torch.float32, device=DEV)
    with pytest.raises(pc.PClothError) as ei:
        pc.pcloth_solve_bsr3_static(n, dummy, dummy, dummy, dummy, 1e-6, 10, dummy)
    assert ei.value.code == pc.ERR_CAPACITY
    assert "PCLOTH_STATIC_MAX_VERTS" in str(ei.value)
