"""ctypes front end of the fp64 C++ oracle (test infrastructure only).

Each function names the passage of P-Cloth (arXiv 2008.00409) that it
follows; the arithmetic itself lives in pcloth_oracle.cpp.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional

import numpy as np

from . import build as _build

_LIB = None

OK, NOT_CONVERGED = 0, 1
INVALID_ARG, BAD_INDEX, NONFINITE, BREAKDOWN = -1, -3, -4, -5

_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_element.argtypes = [_f64p, _f64p, _f64p, _f64p, ctypes.c_double,
                                     ctypes.c_double, ctypes.c_double, _f64p, _f64p]
        L.oracle_element.restype = ctypes.c_int
        L.oracle_assemble.argtypes = [
            ctypes.c_int32, _f32p, _f32p,
            ctypes.c_int32, _i32p, _i32p, _f32p, _f32p,
            ctypes.c_int32, _i32p, _i32p, _f32p, _f32p,
            _f32p, _f32p, ctypes.c_double]
        L.oracle_assemble.restype = ctypes.c_void_p
        L.oracle_status.argtypes = [ctypes.c_void_p]
        L.oracle_status.restype = ctypes.c_int
        L.oracle_nnzb.argtypes = [ctypes.c_void_p]
        L.oracle_nnzb.restype = ctypes.c_int64
        L.oracle_export.argtypes = [ctypes.c_void_p, _i64p, _i32p, _f64p, _f64p, _f64p]
        L.oracle_export.restype = None
        L.oracle_spmv.argtypes = [ctypes.c_void_p, _f64p, _f64p]
        L.oracle_spmv.restype = None
        L.oracle_pcg.argtypes = [ctypes.c_void_p, ctypes.c_double, ctypes.c_int32, _f64p,
                                 ctypes.POINTER(ctypes.c_int32),
                                 ctypes.POINTER(ctypes.c_double)]
        L.oracle_pcg.restype = ctypes.c_int
        L.oracle_pcg_x0.argtypes = [ctypes.c_void_p, ctypes.c_double, ctypes.c_int32, _f64p,
                                    _f64p, ctypes.POINTER(ctypes.c_int32),
                                    ctypes.POINTER(ctypes.c_double)]
        L.oracle_pcg_x0.restype = ctypes.c_int
        L.oracle_update.argtypes = [ctypes.c_int32, _f32p, _f32p, _f64p, ctypes.c_double,
                                    _f64p, _f64p]
        L.oracle_update.restype = None
        L.oracle_find_contacts.argtypes = [ctypes.c_int32, _f32p, ctypes.c_float, ctypes.c_int32,
                                           _i32p, _i32p, _i32p, _i32p, ctypes.c_int64]
        L.oracle_find_contacts.restype = ctypes.c_int64
        L.oracle_free.argtypes = [ctypes.c_void_p]
        L.oracle_free.restype = None
        _LIB = L
    return _LIB


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def element(xa, xb, va, vb, k, rest, h):
    """Stiffness block K (3x3) and force on vertex a of one spring element.

    P-Cloth Sec. 2.5, Eq. (2)-(3): K is taken at x_t, the force at x_t + h v_t;
    spring law K = k[max(0, 1 - L0/l)(I - dd^T) + dd^T], F = k(l - L0)d.
    Returns (K, F, ok) with ok False when a length is zero.
    """
    K = np.zeros(9, np.float64)
    F = np.zeros(3, np.float64)
    ok = lib().oracle_element(_c(xa, np.float64), _c(xb, np.float64), _c(va, np.float64),
                              _c(vb, np.float64), float(k), float(rest), float(h), K, F)
    return K.reshape(3, 3), F, bool(ok)


@dataclasses.dataclass
class System:
    """An assembled fp64 system A dv = b (BSR, 3x3 row-major blocks)."""
    n: int
    rowptr: np.ndarray   # int64 [n+1]
    colind: np.ndarray   # int32 [nnzb]
    vals: np.ndarray     # float64 [nnzb, 3, 3]
    b: np.ndarray        # float64 [n, 3]
    pinv: np.ndarray     # float64 [n, 3, 3]
    status: int
    _handle: Optional[int] = None

    @property
    def nnzb(self) -> int:
        return int(self.colind.shape[0])

    def __del__(self):
        if self._handle is not None and _LIB is not None:
            _LIB.oracle_free(self._handle)
            self._handle = None

    def spmv(self, x: np.ndarray) -> np.ndarray:
        """y = A x in fp64 (the block definition of the product, Eq. (4) for one GPU)."""
        xin = _c(x, np.float64).reshape(-1)
        y = np.zeros(self.n * 3, np.float64)
        lib().oracle_spmv(self._handle, xin, y)
        return y.reshape(self.n, 3)

    def pcg(self, tol: float, maxit: int, x0=None):
        """Block-Jacobi PCG on A dv = b (Eq. (3) text): (dv, iterations, relres, status).

        x0: optional initial guess (n x 3); the residual then starts as
        b - A x0 and a guess that already meets |r| <= tol |b| is returned
        after 0 iterations."""
        dv = np.zeros(self.n * 3, np.float64)
        it = ctypes.c_int32(0)
        rr = ctypes.c_double(0.0)
        if x0 is None:
            st = lib().oracle_pcg(self._handle, float(tol), int(maxit), dv,
                                  ctypes.byref(it), ctypes.byref(rr))
        else:
            g = _c(x0, np.float64).reshape(-1)
            assert g.shape[0] == self.n * 3
            st = lib().oracle_pcg_x0(self._handle, float(tol), int(maxit), g, dv,
                                     ctypes.byref(it), ctypes.byref(rr))
        return dv.reshape(self.n, 3), int(it.value), float(rr.value), int(st)

    def dense(self) -> np.ndarray:
        """Dense 3n x 3n copy (tiny systems only)."""
        A = np.zeros((3 * self.n, 3 * self.n))
        for i in range(self.n):
            for p in range(self.rowptr[i], self.rowptr[i + 1]):
                j = self.colind[p]
                A[3 * i:3 * i + 3, 3 * j:3 * j + 3] = self.vals[p]
        return A


def assemble(n, mass, gravity, springs, contacts, x, v, h) -> System:
    """Assemble A = M + h^2 sum K_e, b = h f(x + h v), P = blockdiag(A)^-1.

    P-Cloth Sec. 2.5 Eq. (3) for the system; Sec. 3.2.2 steps 1-5 for the
    pattern (diagonal plus both directions of every element, sorted, unique)
    and the summed block values.  `springs` and `contacts` are (i, j, k, rest)
    tuples of arrays; contacts may be None.
    """
    si, sj, sk, sr = springs
    if contacts is None:
        ci = cj = np.zeros(0, np.int32)
        ck = cr = np.zeros(0, np.float32)
    else:
        ci, cj, ck, cr = contacts
    ns, nc = len(si), len(ci)
    h_ = lib().oracle_assemble(
        int(n), _c(mass, np.float32), _c(gravity, np.float32),
        ns, _c(si, np.int32), _c(sj, np.int32), _c(sk, np.float32), _c(sr, np.float32),
        nc, _c(ci, np.int32), _c(cj, np.int32), _c(ck, np.float32), _c(cr, np.float32),
        _c(x, np.float32).reshape(-1), _c(v, np.float32).reshape(-1), float(h))
    if not h_:
        raise MemoryError("oracle_assemble: out of host memory")
    st = lib().oracle_status(h_)
    if st in (INVALID_ARG, BAD_INDEX):
        lib().oracle_free(h_)
        return System(int(n), np.zeros(0, np.int64), np.zeros(0, np.int32),
                      np.zeros((0, 3, 3)), np.zeros((0, 3)), np.zeros((0, 3, 3)), st)
    nnzb = lib().oracle_nnzb(h_)
    rowptr = np.zeros(n + 1, np.int64)
    colind = np.zeros(nnzb, np.int32)
    vals = np.zeros(nnzb * 9, np.float64)
    b = np.zeros(n * 3, np.float64)
    pinv = np.zeros(n * 9, np.float64)
    lib().oracle_export(h_, rowptr, colind, vals, b, pinv)
    return System(int(n), rowptr, colind, vals.reshape(nnzb, 3, 3), b.reshape(n, 3),
                  pinv.reshape(n, 3, 3), st, h_)


def assemble_workload(w, x, v, contacts=None) -> System:
    """Assemble one step of a `workloads.Workload` at state (x, v)."""
    c = None
    if contacts is not None and contacts.n > 0:
        c = (contacts.i, contacts.j, contacts.k, contacts.rest)
    return assemble(w.n_verts, w.mass, w.gravity,
                    (w.spring_i, w.spring_j, w.spring_k, w.spring_rest), c, x, v, w.h)


def find_contacts(x, radius, springs, capacity=None):
    """Vertex pairs i < j closer than `radius` that are not springs, in (i, j)
    order (P-Cloth Sec. 4.2-4.3, vertex-vertex proximity), by brute force
    over all pairs with the distance test in float32 (the GPU's precision).
    Returns (i, j, total); i and j hold min(total, capacity) pairs."""
    x = _c(x, np.float32).reshape(-1, 3)
    n = x.shape[0]
    si = _c(springs[0], np.int32)
    sj = _c(springs[1], np.int32)
    cap = n * (n - 1) // 2 if capacity is None else int(capacity)
    cap = max(cap, 1)
    oi = np.zeros(cap, np.int32)
    oj = np.zeros(cap, np.int32)
    total = int(lib().oracle_find_contacts(n, x.reshape(-1), float(radius), si.shape[0], si, sj,
                                           oi, oj, cap))
    k = min(total, cap)
    return oi[:k], oj[:k], total


def update(x, v, dv, h):
    """Backward-Euler state update (Eq. (3)): v' = v + dv, x' = x + h v'. fp64 out."""
    x32 = _c(x, np.float32).reshape(-1)
    v32 = _c(v, np.float32).reshape(-1)
    n = x32.shape[0] // 3
    xo = np.zeros(n * 3, np.float64)
    vo = np.zeros(n * 3, np.float64)
    lib().oracle_update(n, x32, v32, _c(dv, np.float64).reshape(-1), float(h), xo, vo)
    return xo.reshape(n, 3), vo.reshape(n, 3)


def step(w, x, v, contacts=None, tol=None, maxit=None):
    """One implicit step: assemble, PCG, update.  Returns a dict of results."""
    sysm = assemble_workload(w, x, v, contacts)
    if sysm.status not in (OK,):
        return dict(status=sysm.status, system=sysm)
    dv, it, rr, st = sysm.pcg(w.tol if tol is None else tol,
                              w.maxit if maxit is None else maxit)
    xn, vn = update(x, v, dv, w.h)
    return dict(status=st, system=sysm, dv=dv, iterations=it, relres=rr, x=xn, v=vn)
