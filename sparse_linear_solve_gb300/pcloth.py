"""Thin ctypes binding of libpcloth (include/pcloth.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch supplies the device memory (tensors) and the stream.
The module-level functions carry the C names; `PCloth` wraps a handle.

If libpcloth.so is missing it is built (nvcc required); if that fails the
import of this module fails -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

from . import build as _build

OK, NOT_CONVERGED = 0, 1
ERR_INVALID_ARG, ERR_CAPACITY, ERR_BAD_INDEX = -1, -2, -3
ERR_NONFINITE, ERR_BREAKDOWN, ERR_CUDA, ERR_STATE = -4, -5, -6, -7
CODE_NAMES = {OK: "OK", NOT_CONVERGED: "NOT_CONVERGED", ERR_INVALID_ARG: "INVALID_ARG",
              ERR_CAPACITY: "CAPACITY", ERR_BAD_INDEX: "BAD_INDEX",
              ERR_NONFINITE: "NONFINITE", ERR_BREAKDOWN: "BREAKDOWN", ERR_CUDA: "CUDA",
              ERR_STATE: "STATE"}

# Every symbol declared in include/pcloth.h.
EXPORTS = ("pcloth_create", "pcloth_assemble", "pcloth_spmv", "pcloth_solve", "pcloth_step",
           "pcloth_step_host", "pcloth_nnzb", "pcloth_export", "pcloth_set_stream",
           "pcloth_sync", "pcloth_last_error", "pcloth_destroy", "pcloth_profile_enable",
           "pcloth_profile_read", "pcloth_solve_bsr3_static", "pcloth_bell_build",
           "pcloth_spmv_bell", "pcloth_find_contacts", "pcloth_selftest_bounded_wait",
           "pcloth_solve_guess", "pcloth_step_async", "pcloth_step_result")

STATIC_MAX_VERTS = 16384   # PCLOTH_STATIC_MAX_VERTS


class PClothError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("%s (%d): %s" % (CODE_NAMES.get(code, "?"), code, msg))
        self.code = code


class Mesh(ctypes.Structure):
    _fields_ = [("n_verts", ctypes.c_int32), ("mass", ctypes.c_void_p),
                ("gravity", ctypes.c_float * 3)]


class Springs(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("i", ctypes.c_void_p), ("j", ctypes.c_void_p),
                ("k", ctypes.c_void_p), ("rest", ctypes.c_void_p)]


class Opts(ctypes.Structure):
    _fields_ = [("max_contacts", ctypes.c_int32), ("device", ctypes.c_int),
                ("stream", ctypes.c_void_p)]


_LIB = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libpcloth.so (building it first if it is missing or stale)."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        P = ctypes.POINTER
        L.pcloth_create.argtypes = [P(Mesh), P(Springs), P(Opts), P(vp)]
        L.pcloth_assemble.argtypes = [vp, vp, vp, P(Springs), ctypes.c_float]
        L.pcloth_spmv.argtypes = [vp, vp, vp]
        L.pcloth_bell_build.argtypes = [vp, P(i32)]
        L.pcloth_find_contacts.argtypes = [vp, vp, ctypes.c_float, ctypes.c_float, P(Springs),
                                           i32, P(i32)]
        L.pcloth_spmv_bell.argtypes = [vp, vp, vp]
        L.pcloth_solve.argtypes = [vp, dbl, i32, vp, P(i32), P(dbl)]
        L.pcloth_step.argtypes = [vp, vp, vp, P(Springs), ctypes.c_float, dbl, i32, vp,
                                  P(i32), P(dbl)]
        L.pcloth_step_host.argtypes = [vp, vp, vp, P(Springs), ctypes.c_float, dbl, i32,
                                       P(i32), P(dbl)]
        L.pcloth_solve_guess.argtypes = [vp, dbl, i32, vp, P(i32), P(dbl)]
        L.pcloth_step_async.argtypes = [vp, vp, vp, P(Springs), ctypes.c_float, dbl, i32, vp]
        L.pcloth_step_result.argtypes = [vp, P(i32), P(dbl)]
        L.pcloth_nnzb.argtypes = [vp, P(i64)]
        L.pcloth_export.argtypes = [vp, vp, vp, vp, vp, vp]
        L.pcloth_set_stream.argtypes = [vp, vp]
        L.pcloth_sync.argtypes = [vp]
        L.pcloth_last_error.argtypes = [vp]
        L.pcloth_last_error.restype = ctypes.c_char_p
        L.pcloth_destroy.argtypes = [vp]
        L.pcloth_destroy.restype = None
        L.pcloth_profile_enable.argtypes = [vp, ctypes.c_int]
        L.pcloth_profile_read.argtypes = [vp, P(dbl), P(i64), ctypes.c_int]
        L.pcloth_solve_bsr3_static.argtypes = [i32, vp, vp, vp, vp, dbl, i32, vp, P(i32), P(dbl),
                                               vp]
        L.pcloth_selftest_bounded_wait.argtypes = [ctypes.c_int, dbl, P(ctypes.c_uint32)]
        for name in EXPORTS:
            f = getattr(L, name)
            if name not in ("pcloth_last_error", "pcloth_destroy"):
                f.restype = ctypes.c_int
        _LIB = L
    return _LIB


# ---------------------------------------------------------------- helpers --

def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, dtype, device, shape=None, name="tensor"):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if device is not None and t.device != device:
        raise ValueError("%s must be on %s, got %s" % (name, device, t.device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, shape, tuple(t.shape)))
    return t


def _raise(handle, code: int):
    msg = lib().pcloth_last_error(handle)
    raise PClothError(code, msg.decode() if msg else "")


def _elements(el, device, name) -> Springs:
    """(i, j, k, rest) tensors -> Springs struct (pointers kept alive by caller)."""
    if el is None:
        return Springs(0, None, None, None, None)
    i, j, k, rest = el
    n = int(i.shape[0])
    for t, dt, nm in ((i, torch.int32, "i"), (j, torch.int32, "j"),
                      (k, torch.float32, "k"), (rest, torch.float32, "rest")):
        _check(t, dt, device, (n,), "%s.%s" % (name, nm))
    return Springs(n, _ptr(i), _ptr(j), _ptr(k), _ptr(rest))


# ------------------------------------------------------ C-named functions --

def pcloth_create(mass: torch.Tensor, gravity, springs, max_contacts: int = 0,
                  stream: Optional[int] = None) -> int:
    """Create a handle (int).  mass: cuda float32[N]; springs: (i, j, k, rest)."""
    _check(mass, torch.float32, None, None, "mass")
    dev = mass.device
    if dev.type != "cuda":
        raise ValueError("mass must be a CUDA tensor")
    sp = _elements(springs, dev, "springs")
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    g = (ctypes.c_float * 3)(*[float(x) for x in gravity])
    mesh = Mesh(int(mass.shape[0]), _ptr(mass), g)
    opts = Opts(int(max_contacts), int(dev.index or 0), ctypes.c_void_p(stream))
    out = ctypes.c_void_p()
    rc = lib().pcloth_create(ctypes.byref(mesh), ctypes.byref(sp), ctypes.byref(opts),
                             ctypes.byref(out))
    if rc != OK:
        _raise(None, rc)
    return out.value


def pcloth_assemble(h: int, x: torch.Tensor, v: torch.Tensor, contacts, dt: float,
                    n: Optional[int] = None):
    n = x.shape[0] if n is None else n
    _check(x, torch.float32, None, (n, 3), "x")
    _check(v, torch.float32, x.device, (n, 3), "v")
    c = _elements(contacts, x.device, "contacts")
    rc = lib().pcloth_assemble(h, _ptr(x), _ptr(v), ctypes.byref(c), float(dt))
    if rc != OK:
        _raise(h, rc)


def pcloth_spmv(h: int, inp: torch.Tensor, out: torch.Tensor):
    _check(inp, torch.float32, None, None, "in")
    _check(out, torch.float32, inp.device, tuple(inp.shape), "out")
    rc = lib().pcloth_spmv(h, _ptr(inp), _ptr(out))
    if rc != OK:
        _raise(h, rc)


def pcloth_find_contacts(h: int, x: torch.Tensor, radius: float, stiffness: float,
                         capacity: int):
    """Vertex pairs closer than `radius` (not springs) as contact springs:
    returns ((i, j, k, rest) device tensors of length n_found, n_found).
    Raises PClothError (ERR_CAPACITY) if more than `capacity` exist; the
    count found is in the exception's `found` attribute."""
    _check(x, torch.float32, None, None, "x")
    dev = x.device
    cap = max(int(capacity), 0)
    oi = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    oj = torch.empty_like(oi)
    ok = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
    orest = torch.empty_like(ok)
    out = Springs(0, _ptr(oi), _ptr(oj), _ptr(ok), _ptr(orest))
    found = ctypes.c_int32(0)
    rc = lib().pcloth_find_contacts(h, _ptr(x), float(radius), float(stiffness), ctypes.byref(out),
                                    cap, ctypes.byref(found))
    if rc != OK:
        try:
            _raise(h, rc)
        except PClothError as e:
            e.found = int(found.value)
            raise
    m = int(out.n)
    return (oi[:m], oj[:m], ok[:m], orest[:m]), int(found.value)


def pcloth_bell_build(h: int) -> int:
    """Block-ELL copy of the last assembled matrix; returns its width W."""
    w = ctypes.c_int32(0)
    rc = lib().pcloth_bell_build(h, ctypes.byref(w))
    if rc != OK:
        _raise(h, rc)
    return int(w.value)


def pcloth_spmv_bell(h: int, inp: torch.Tensor, out: torch.Tensor):
    _check(inp, torch.float32, None, None, "in")
    _check(out, torch.float32, inp.device, tuple(inp.shape), "out")
    rc = lib().pcloth_spmv_bell(h, _ptr(inp), _ptr(out))
    if rc != OK:
        _raise(h, rc)


def pcloth_solve(h: int, tol: float, maxit: int, dv: torch.Tensor):
    """Returns (iterations, rel_residual, code); code is OK or NOT_CONVERGED."""
    _check(dv, torch.float32, None, None, "dv")
    it = ctypes.c_int32(0)
    rr = ctypes.c_double(0.0)
    rc = lib().pcloth_solve(h, float(tol), int(maxit), _ptr(dv), ctypes.byref(it),
                            ctypes.byref(rr))
    if rc not in (OK, NOT_CONVERGED):
        _raise(h, rc)
    return int(it.value), float(rr.value), rc


def pcloth_solve_guess(h: int, tol: float, maxit: int, dv: torch.Tensor):
    """PCG from the guess held in dv (overwritten with the solution).
    Returns (iterations, rel_residual, code) like pcloth_solve."""
    _check(dv, torch.float32, None, None, "dv")
    it = ctypes.c_int32(0)
    rr = ctypes.c_double(0.0)
    rc = lib().pcloth_solve_guess(h, float(tol), int(maxit), _ptr(dv), ctypes.byref(it),
                                  ctypes.byref(rr))
    if rc not in (OK, NOT_CONVERGED):
        _raise(h, rc)
    return int(it.value), float(rr.value), rc


def pcloth_step_async(h: int, x: torch.Tensor, v: torch.Tensor, contacts, dt: float,
                      tol: float, maxit: int, dv: Optional[torch.Tensor] = None):
    """Enqueue one whole step (no host synchronisation); contacts: device
    (i, j, k, rest) tensors kept alive by the caller, or None."""
    _check(x, torch.float32, None, None, "x")
    _check(v, torch.float32, x.device, tuple(x.shape), "v")
    c = _elements(contacts, x.device, "contacts")
    rc = lib().pcloth_step_async(h, _ptr(x), _ptr(v), ctypes.byref(c), float(dt), float(tol),
                                 int(maxit), _ptr(dv))
    if rc != OK:
        _raise(h, rc)


def pcloth_step_result(h: int):
    """(iterations, rel_residual, code) of the last asynchronous step."""
    it = ctypes.c_int32(0)
    rr = ctypes.c_double(0.0)
    rc = lib().pcloth_step_result(h, ctypes.byref(it), ctypes.byref(rr))
    if rc not in (OK, NOT_CONVERGED):
        _raise(h, rc)
    return int(it.value), float(rr.value), rc


def pcloth_step(h: int, x: torch.Tensor, v: torch.Tensor, contacts, dt: float, tol: float,
                maxit: int, dv: Optional[torch.Tensor] = None):
    _check(x, torch.float32, None, None, "x")
    _check(v, torch.float32, x.device, tuple(x.shape), "v")
    c = _elements(contacts, x.device, "contacts")
    it = ctypes.c_int32(0)
    rr = ctypes.c_double(0.0)
    rc = lib().pcloth_step(h, _ptr(x), _ptr(v), ctypes.byref(c), float(dt), float(tol),
                           int(maxit), _ptr(dv), ctypes.byref(it), ctypes.byref(rr))
    if rc not in (OK, NOT_CONVERGED):
        _raise(h, rc)
    return int(it.value), float(rr.value), rc


def pcloth_step_host(h: int, x: torch.Tensor, v: torch.Tensor, contacts, dt: float,
                     tol: float, maxit: int):
    """x, v: CPU float32 [N, 3] (pinned recommended); contacts: CPU tensors."""
    _check(x, torch.float32, torch.device("cpu"), None, "x")
    _check(v, torch.float32, torch.device("cpu"), tuple(x.shape), "v")
    c = _elements(contacts, torch.device("cpu"), "contacts")
    it = ctypes.c_int32(0)
    rr = ctypes.c_double(0.0)
    rc = lib().pcloth_step_host(h, _ptr(x), _ptr(v), ctypes.byref(c), float(dt), float(tol),
                                int(maxit), ctypes.byref(it), ctypes.byref(rr))
    if rc not in (OK, NOT_CONVERGED):
        _raise(h, rc)
    return int(it.value), float(rr.value), rc


def pcloth_nnzb(h: int) -> int:
    out = ctypes.c_int64(0)
    rc = lib().pcloth_nnzb(h, ctypes.byref(out))
    if rc != OK:
        _raise(h, rc)
    return int(out.value)


def pcloth_export(h: int, rowptr=None, colind=None, vals=None, b=None, pinv=None):
    rc = lib().pcloth_export(h, _ptr(rowptr), _ptr(colind), _ptr(vals), _ptr(b), _ptr(pinv))
    if rc != OK:
        _raise(h, rc)


def pcloth_set_stream(h: int, stream: int):
    rc = lib().pcloth_set_stream(h, ctypes.c_void_p(stream))
    if rc != OK:
        _raise(h, rc)


def pcloth_sync(h: int):
    rc = lib().pcloth_sync(h)
    if rc != OK:
        _raise(h, rc)


def pcloth_last_error(h: Optional[int]) -> str:
    m = lib().pcloth_last_error(h)
    return m.decode() if m else ""


def pcloth_destroy(h: int):
    lib().pcloth_destroy(h)


def pcloth_profile_enable(h: int, on=True):
    """on: 0/False off; any other value times assemblies, PCG launches and the
    PCG kernel's phases."""
    rc = lib().pcloth_profile_enable(h, int(on))
    if rc != OK:
        _raise(h, rc)


def pcloth_profile_read(h: int, reset: bool = False) -> dict:
    ms = (ctypes.c_double * 4)()
    cnt = (ctypes.c_int64 * 7)()
    rc = lib().pcloth_profile_read(h, ms, cnt, int(bool(reset)))
    if rc != OK:
        _raise(h, rc)
    return dict(assemble_ms=ms[0], spmv_ms=ms[1], update_ms=ms[2], solve_ms=ms[3],
                assemble_calls=cnt[0], spmv_launches=cnt[1], update_launches=cnt[2],
                solves=cnt[3], iterations=cnt[4], kernel_launches=cnt[5], samples=cnt[6])


def pcloth_solve_bsr3_static(n: int, rowptr, colind, vals, b, tol: float, maxit: int, dv,
                             stream: Optional[int] = None):
    """Allocation-free block-Jacobi PCG on a symmetric positive-definite BSR3
    system the caller holds (device tensors: rowptr int32[n+1], colind
    int32[nnzb], vals float32[nnzb,3,3], b float32[n,3]; dv float32[n,3] is
    written).  For callers that must not allocate GPU memory;
    n <= STATIC_MAX_VERTS.  rowptr, colind and vals must start 16-byte
    aligned and be followed by at least 16 readable bytes (e.g. views at the
    start of larger tensors).  Returns (iterations, rel_residual, code) like
    pcloth_solve."""
    ptrs = [None if t is None else t.data_ptr() for t in (rowptr, colind, vals, b, dv)]
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    it = ctypes.c_int32(0)
    rr = ctypes.c_double(0.0)
    rc = lib().pcloth_solve_bsr3_static(int(n), *ptrs[:4], float(tol), int(maxit), ptrs[4],
                                        ctypes.byref(it), ctypes.byref(rr),
                                        ctypes.c_void_p(stream))
    if rc not in (OK, NOT_CONVERGED):
        _raise(None, rc)
    return int(it.value), float(rr.value), rc


def pcloth_selftest_bounded_wait(which: int, limit_seconds: float):
    """Runs one of the library's bounded device waits on something that never
    completes (which = 0: the SpMV pipeline's mbarrier wait; 1: the PCG grid
    barrier's counter poll) with a limit of limit_seconds.  Returns (code,
    status word, message): a wait that gave up as designed returns ERR_CUDA,
    the device status word with bit 4 set and "device wait timed out"."""
    st = ctypes.c_uint32(0)
    rc = lib().pcloth_selftest_bounded_wait(int(which), float(limit_seconds), ctypes.byref(st))
    msg = lib().pcloth_last_error(None)
    return rc, int(st.value), (msg.decode() if msg else "")


# ------------------------------------------------------------ convenience --

def _dev_tensor(a, dtype, device):
    if isinstance(a, torch.Tensor):
        return a.to(device=device, dtype=dtype).contiguous()
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


def to_device_elements(el, device):
    """(i, j, k, rest) numpy/tensors or an object with .i/.j/.k/.rest -> cuda tensors."""
    if el is None:
        return None
    if hasattr(el, "rest"):
        el = (el.i, el.j, el.k, el.rest)
    i, j, k, rest = el
    if len(i) == 0:
        return None
    return (_dev_tensor(i, torch.int32, device), _dev_tensor(j, torch.int32, device),
            _dev_tensor(k, torch.float32, device), _dev_tensor(rest, torch.float32, device))


class PCloth:
    """One cloth on one GPU: owns a libpcloth handle and keeps inputs alive."""

    def __init__(self, mass, gravity, springs, max_contacts: int = 0,
                 device="cuda", stream: Optional[int] = None):
        device = torch.device(device)
        if device.type == "cuda" and device.index is None:
            device = torch.device("cuda", torch.cuda.current_device())
        self.device = device
        self.mass = _dev_tensor(mass, torch.float32, device)
        self.n = int(self.mass.shape[0])
        self.springs = to_device_elements(springs, device)
        self.max_contacts = int(max_contacts)
        self.h = pcloth_create(self.mass, gravity, self.springs, max_contacts, stream)
        self._contacts = None

    @classmethod
    def from_workload(cls, w, device="cuda", **kw):
        return cls(w.mass, w.gravity, (w.spring_i, w.spring_j, w.spring_k, w.spring_rest),
                   max_contacts=w.max_contacts, device=device, **kw)

    def close(self):
        if getattr(self, "h", None):
            pcloth_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def assemble(self, x, v, contacts=None, dt: float = 1e-2):
        self._contacts = to_device_elements(contacts, self.device)
        pcloth_assemble(self.h, x, v, self._contacts, dt, self.n)

    def spmv(self, inp: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        _check(inp, torch.float32, self.device, (self.n, 3), "in")
        if out is None:
            out = torch.empty_like(inp)
        pcloth_spmv(self.h, inp, out)
        return out

    def find_contacts(self, x: torch.Tensor, radius: float, stiffness: float,
                      capacity: Optional[int] = None):
        """((i, j, k, rest), n_found): the vertex pairs of x closer than radius
        that are not springs, as contact springs (rest = radius)."""
        _check(x, torch.float32, self.device, (self.n, 3), "x")
        return pcloth_find_contacts(self.h, x, radius, stiffness,
                                    self.max_contacts if capacity is None else capacity)

    def bell_build(self) -> int:
        return pcloth_bell_build(self.h)

    def spmv_bell(self, inp: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
        _check(inp, torch.float32, self.device, (self.n, 3), "in")
        if out is None:
            out = torch.empty_like(inp)
        pcloth_spmv_bell(self.h, inp, out)
        return out

    def solve(self, tol: float, maxit: int, dv: Optional[torch.Tensor] = None):
        if dv is None:
            dv = torch.empty((self.n, 3), dtype=torch.float32, device=self.device)
        _check(dv, torch.float32, self.device, (self.n, 3), "dv")
        it, rr, code = pcloth_solve(self.h, tol, maxit, dv)
        return dv, it, rr, code

    def solve_guess(self, dv: torch.Tensor, tol: float, maxit: int):
        """PCG from the guess in dv (device float32 [n, 3], overwritten)."""
        _check(dv, torch.float32, self.device, (self.n, 3), "dv")
        it, rr, code = pcloth_solve_guess(self.h, tol, maxit, dv)
        return dv, it, rr, code

    def set_stream(self, stream: int):
        pcloth_set_stream(self.h, stream)

    def step_async(self, x, v, contacts=None, dt: float = 1e-2, tol: float = 1e-6,
                   maxit: int = 20000, dv: Optional[torch.Tensor] = None):
        """Enqueue one step without synchronising (capturable in a CUDA graph);
        contacts: device (i, j, k, rest) tensors that the caller keeps alive
        (a captured graph reads the same arrays at every replay), or None."""
        _check(x, torch.float32, self.device, (self.n, 3), "x")
        pcloth_step_async(self.h, x, v, contacts, dt, tol, maxit, dv)

    def step_result(self):
        return pcloth_step_result(self.h)

    def step(self, x, v, contacts=None, dt: float = 1e-2, tol: float = 1e-6,
             maxit: int = 20000, dv: Optional[torch.Tensor] = None):
        _check(x, torch.float32, self.device, (self.n, 3), "x")
        self._contacts = to_device_elements(contacts, self.device)
        return pcloth_step(self.h, x, v, self._contacts, dt, tol, maxit, dv)

    def step_host(self, x, v, contacts=None, dt: float = 1e-2, tol: float = 1e-6,
                  maxit: int = 20000):
        c = None
        if contacts is not None:
            if hasattr(contacts, "rest"):
                contacts = (contacts.i, contacts.j, contacts.k, contacts.rest)
            if len(contacts[0]) > 0:
                c = tuple(t if isinstance(t, torch.Tensor) else torch.from_numpy(
                    np.ascontiguousarray(t)) for t in contacts)
        return pcloth_step_host(self.h, x, v, c, dt, tol, maxit)

    def nnzb(self) -> int:
        return pcloth_nnzb(self.h)

    def export(self) -> dict:
        nnzb = self.nnzb()
        d = self.device
        out = dict(rowptr=torch.empty(self.n + 1, dtype=torch.int32, device=d),
                   colind=torch.empty(nnzb, dtype=torch.int32, device=d),
                   vals=torch.empty((nnzb, 3, 3), dtype=torch.float32, device=d),
                   b=torch.empty((self.n, 3), dtype=torch.float32, device=d),
                   pinv=torch.empty((self.n, 3, 3), dtype=torch.float32, device=d))
        pcloth_export(self.h, out["rowptr"], out["colind"], out["vals"], out["b"], out["pinv"])
        return out

    def profile(self, on=True):
        pcloth_profile_enable(self.h, on)

    def profile_read(self, reset: bool = False) -> dict:
        return pcloth_profile_read(self.h, reset)
