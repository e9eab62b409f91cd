"""The PCG solve from an initial iterate and the asynchronous step that a CUDA
graph can capture, through the C ABI.

P-Cloth (arXiv 2008.00409) solves Eq. (3) by PCG every step (Sec. 3.1); the
textbook PCG from a nonzero first iterate x0 starts from r = b - A x0.  The
GPU's solve from a guess is compared with the fp64 oracle's PCG from the same
guess (dv to 1e-4, iteration counts within max(3, 3%)), with a zero guess it
must give the bits of the plain solve, and a guess that already meets the
tolerance returns after 0 iterations.  The asynchronous step must give the
bits of pcloth_step, eagerly and replayed from a captured CUDA graph.
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from sparse_linear_solve_gb300 import pcloth as pc
from sparse_linear_solve_gb300 import workloads as W

from gpu_helpers import DEV, make, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _assembled(w, step=0):
    c = w.contacts(step)
    pcl = make(w)
    pcl.assemble(to_dev(w.x0), to_dev(w.v0), c if c.n else None, w.h)
    ref = oracle.assemble_workload(w, w.x0, w.v0, c if c.n else None)
    return pcl, ref


@pytest.mark.parametrize("make_w", [lambda: W.jittered_cloth(n=64, steps=2),
                                    lambda: W.folded_stack(n=29, steps=2),
                                    lambda: W.tiny_cloth(rest_from_grid=True)],
                         ids=["jitter64", "folded4x29", "tiny32_tension"])
def test_solve_from_guess_matches_oracle(make_w):
    w = make_w()
    pcl, ref = _assembled(w)
    dv_exact, _, _, st = ref.pcg(w.tol, w.maxit)
    assert st == oracle.OK
    # a partial guess: half the solution, with a perturbation of its own size
    rng = np.random.default_rng(21)
    x0 = (0.5 * dv_exact + 0.25 * np.abs(dv_exact).mean() *
          rng.normal(size=dv_exact.shape)).astype(np.float32)
    dv_ref, it_ref, rr_ref, st = ref.pcg(w.tol, w.maxit, x0=x0)
    assert st == oracle.OK
    dv = to_dev(x0)
    _, it, rr, code = pcl.solve_guess(dv, w.tol, w.maxit)
    assert code == pc.OK and rr <= w.tol
    e = rel_l2(dv.cpu().numpy(), dv_ref)
    assert e <= 1e-4, (e, it, it_ref)
    assert abs(it - it_ref) <= max(3, 0.03 * it_ref), (it, it_ref)


def test_zero_guess_gives_the_plain_solve_bit_for_bit():
    w = W.jittered_cloth(n=48)
    pcl, _ = _assembled(w)
    dv_plain, it_plain, rr_plain, _ = pcl.solve(w.tol, w.maxit)
    dv = torch.zeros_like(dv_plain)
    _, it, rr, code = pcl.solve_guess(dv, w.tol, w.maxit)
    assert code == pc.OK and it == it_plain and rr == rr_plain
    assert torch.equal(dv, dv_plain)


def test_guess_that_meets_the_tolerance_returns_at_once():
    w = W.jittered_cloth(n=48)
    pcl, ref = _assembled(w)
    dv_plain, _, _, _ = pcl.solve(w.tol, w.maxit)
    dv = dv_plain.clone()
    _, it, rr, code = pcl.solve_guess(dv, 1e-3, w.maxit)
    assert code == pc.OK and it == 0
    assert torch.equal(dv, dv_plain)
    # the reported residual is the GPU's fp32 |b - A dv| / |b|; against the
    # fp64 one of the same dv it differs by the fp32 rounding of b - A dv
    true = np.linalg.norm(ref.b - ref.spmv(dv_plain.cpu().numpy())) / np.linalg.norm(ref.b)
    assert rr <= 1e-3 and abs(rr - true) <= 0.5 * true + 1e-6, (rr, true)
    # maxit = 0 from a guess that does not meet the tolerance
    _, it, rr, code = pcl.solve_guess(torch.zeros_like(dv), 1e-6, 0)
    assert code == pc.NOT_CONVERGED and it == 0 and abs(rr - 1.0) < 1e-6


def _contacts_dev(c):
    return tuple(to_dev(a, dtype) for a, dtype in ((c.i, torch.int32), (c.j, torch.int32),
                                                  (c.k, torch.float32), (c.rest, torch.float32)))


def test_async_step_gives_the_bits_of_the_step():
    w = W.jittered_cloth(n=48, steps=3)
    a, b = make(w), make(w)
    xa, va = to_dev(w.x0), to_dev(w.v0)
    xb, vb = xa.clone(), va.clone()
    for t in range(3):
        c = w.contacts(t)
        it, rr, code = a.step(xa, va, c, w.h, w.tol, w.maxit)
        b.step_async(xb, vb, _contacts_dev(c), w.h, w.tol, w.maxit)
        it_b, rr_b, code_b = b.step_result()
        assert (it_b, rr_b, code_b) == (it, rr, code)
        assert torch.equal(xa, xb) and torch.equal(va, vb)


def test_async_step_replayed_from_a_cuda_graph():
    """One step captured in a CUDA graph on a side stream, replayed for three
    steps with each step's contacts written into the captured arrays: the
    same bits and results as the plain steps."""
    w = W.jittered_cloth(n=48, steps=3)
    ref = make(w)
    xr, vr = to_dev(w.x0), to_dev(w.v0)
    expect = []
    for t in range(3):
        it, rr, code = ref.step(xr, vr, w.contacts(t), w.h, w.tol, w.maxit)
        expect.append((it, rr, code, xr.clone(), vr.clone()))

    s = torch.cuda.Stream(device=DEV)
    g_cl = make(w)
    g_cl.set_stream(s.cuda_stream)
    x, v = to_dev(w.x0), to_dev(w.v0)
    bufs = tuple(t.clone() for t in _contacts_dev(w.contacts(0)))
    dv = torch.empty_like(x)
    with torch.cuda.stream(s):   # one eager step on scratch state, so that
        xs, vs = x.clone(), v.clone()   # the capture records a warmed-up library
        g_cl.step_async(xs, vs, bufs, w.h, w.tol, w.maxit, dv)
    g_cl.step_result()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s, capture_error_mode="thread_local"):
        g_cl.step_async(x, v, bufs, w.h, w.tol, w.maxit, dv)
    for t in range(3):
        with torch.cuda.stream(s):
            for dst, src in zip(bufs, _contacts_dev(w.contacts(t))):
                dst.copy_(src)
            graph.replay()
        it, rr, code = g_cl.step_result()
        e_it, e_rr, e_code, e_x, e_v = expect[t]
        assert (it, rr, code) == (e_it, e_rr, e_code), t
        assert torch.equal(x, e_x) and torch.equal(v, e_v), t
