"""Seeded synthetic cloth workloads (inputs only, no solver arithmetic).

This module builds the inputs of the implicit-integration hot path: a
triangulated square-grid cloth (one or several stacked layers), its stretch and
bending springs, per-vertex masses, the initial state (x, v) and, per time
step, a list of penalty contacts.  It computes nothing of the method itself
(no force, Jacobian, matrix or solve); both the CUDA path and the CPU oracle
receive the arrays it returns, so the two sides always see identical inputs.

The five named configurations are synthetic stand-ins for the garment scenes of
P-Cloth (arXiv 2008.00409, Sec. 6, benchmark list and Fig. 1: Kneel, 1.65M
triangles, is the largest), which are not available here.

Conventions (the pages fix none of them; the readings are listed in the design
notes):

* vertex id = layer * n^2 + i * n + j, rest position (i*s, j*s, layer*gap);
* every grid cell (i, j)-(i+1, j+1) is split into the triangles
  (i,j)(i+1,j)(i+1,j+1) and (i,j)(i+1,j+1)(i,j+1);
* stretch springs join the three edge offsets (1,0), (0,1), (1,1);
* a bending spring joins the two opposite vertices of each interior edge,
  which on this triangulation gives the offsets (1,2), (2,1), (1,-1);
* rest lengths come from the unperturbed grid unless a config says otherwise;
* contacts are (i, j, k, rest) tuples, exactly like springs.

All float arrays are float32 (the storage type of the GPU path); the oracle
promotes them to float64.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Optional

import numpy as np

SPACING = 0.01          # grid spacing s [m]
K_STRETCH = 1.0e4       # stretch spring stiffness [N/m]
K_BEND = 1.0e1          # bending spring stiffness [N/m]
K_CONTACT = 1.0e3       # penalty contact stiffness [N/m]
MASS = 1.0e-4           # per-vertex mass [kg]
GRAVITY = (0.0, 0.0, -9.8)

STRETCH_OFFSETS = ((1, 0), (0, 1), (1, 1))
BEND_OFFSETS = ((1, 2), (2, 1), (1, -1))


@dataclasses.dataclass
class Contacts:
    i: np.ndarray      # int32 [nc]
    j: np.ndarray      # int32 [nc]
    k: np.ndarray      # float32 [nc]
    rest: np.ndarray   # float32 [nc]

    @property
    def n(self) -> int:
        return int(self.i.shape[0])

    @staticmethod
    def empty() -> "Contacts":
        return Contacts(np.zeros(0, np.int32), np.zeros(0, np.int32),
                        np.zeros(0, np.float32), np.zeros(0, np.float32))


@dataclasses.dataclass
class Workload:
    name: str
    n_verts: int
    mass: np.ndarray        # float32 [N]
    gravity: np.ndarray     # float32 [3]
    spring_i: np.ndarray    # int32 [S]
    spring_j: np.ndarray    # int32 [S]
    spring_k: np.ndarray    # float32 [S]
    spring_rest: np.ndarray  # float32 [S]
    x0: np.ndarray          # float32 [N, 3]
    v0: np.ndarray          # float32 [N, 3]
    h: float
    steps: int
    tol: float
    maxit: int
    max_contacts: int
    triangles: int
    contact_fn: Optional[Callable[[int, np.ndarray], Contacts]] = None
    seed: int = 0
    description: str = ""

    @property
    def n_springs(self) -> int:
        return int(self.spring_i.shape[0])

    def contacts(self, step: int, x: Optional[np.ndarray] = None) -> Contacts:
        """Contact list of time step `step` (0-based), seeded per step."""
        if self.contact_fn is None:
            return Contacts.empty()
        return self.contact_fn(step, self.x0 if x is None else x)


# ---------------------------------------------------------------------------
# grid topology
# ---------------------------------------------------------------------------

def grid_springs(n: int, offsets) -> tuple[np.ndarray, np.ndarray]:
    """Vertex pairs (a, b) of one n x n layer for the given (di, dj) offsets."""
    ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    a_all, b_all = [], []
    for di, dj in offsets:
        i2, j2 = ii + di, jj + dj
        ok = (i2 >= 0) & (i2 < n) & (j2 >= 0) & (j2 < n)
        a_all.append((ii[ok] * n + jj[ok]).astype(np.int64))
        b_all.append((i2[ok] * n + j2[ok]).astype(np.int64))
    return np.concatenate(a_all), np.concatenate(b_all)


def grid_positions(n: int) -> np.ndarray:
    ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    p = np.zeros((n * n, 3), np.float64)
    p[:, 0] = ii.reshape(-1) * SPACING
    p[:, 1] = jj.reshape(-1) * SPACING
    return p


def layered_springs(n: int, layers: int, rest_pos: np.ndarray):
    """Stretch + bending springs of `layers` stacked n x n grids.

    Rest lengths are measured on `rest_pos` (float64 [layers*n*n, 3]).
    """
    sa, sb = grid_springs(n, STRETCH_OFFSETS)
    ba, bb = grid_springs(n, BEND_OFFSETS)
    ii, jj, kk = [], [], []
    for layer in range(layers):
        off = layer * n * n
        ii += [sa + off, ba + off]
        jj += [sb + off, bb + off]
        kk += [np.full(sa.shape, K_STRETCH), np.full(ba.shape, K_BEND)]
    si = np.concatenate(ii)
    sj = np.concatenate(jj)
    sk = np.concatenate(kk)
    rest = np.linalg.norm(rest_pos[sj] - rest_pos[si], axis=1)
    return (si.astype(np.int32), sj.astype(np.int32), sk.astype(np.float32),
            rest.astype(np.float32))


def n_triangles(n: int, layers: int = 1) -> int:
    return 2 * (n - 1) * (n - 1) * layers


def _base(name, n, layers, rest_pos, x0, v0, h, steps, max_contacts,
          contact_fn=None, seed=0, tol=1e-6, maxit=20000, description=""):
    N = n * n * layers
    si, sj, sk, rest = layered_springs(n, layers, rest_pos)
    return Workload(
        name=name, n_verts=N,
        mass=np.full(N, MASS, np.float32),
        gravity=np.asarray(GRAVITY, np.float32),
        spring_i=si, spring_j=sj, spring_k=sk, spring_rest=rest,
        x0=np.ascontiguousarray(x0, dtype=np.float32),
        v0=np.ascontiguousarray(v0, dtype=np.float32),
        h=h, steps=steps, tol=tol, maxit=maxit, max_contacts=max_contacts,
        triangles=n_triangles(n, layers), contact_fn=contact_fn, seed=seed,
        description=description)


def step_rng(seed: int, step: int) -> np.random.Generator:
    """The per-step contact generator: seeded with seed * 10007 + step."""
    return np.random.default_rng(seed * 10007 + step)


# ---------------------------------------------------------------------------
# the five configurations
# ---------------------------------------------------------------------------

def tiny_cloth(n: int = 32, seed: int = 1000, rest_from_grid: bool = False,
               velocity_sigma: float = 0.1, h: float = 1e-2) -> Workload:
    """C1: one n x n layer, rest positions perturbed by N(0, 1 mm).

    Literal reading (default): the perturbed grid is both the rest shape and
    x0, so every spring starts at rest.  With rest_from_grid=True the rest
    lengths come from the unperturbed grid instead, so the tension branch of
    the Jacobian is exercised too.  v0 ~ N(0, 0.1) per component.
    """
    rng = np.random.default_rng(seed)
    grid = grid_positions(n)
    x0 = grid + rng.normal(0.0, 1e-3, grid.shape)
    v0 = rng.normal(0.0, velocity_sigma, grid.shape)
    rest_pos = grid if rest_from_grid else x0
    return _base("tiny_cloth_%d" % n, n, 1, rest_pos, x0, v0, h, 1, 0,
                 seed=seed,
                 description="%dx%d grid, rest and x0 perturbed N(0,1e-3), "
                 "v0 N(0,0.1), h=%g, no contacts" % (n, n, h))


def drooped_cloth(n: int = 256, seed: int = 1001, steps: int = 10) -> Workload:
    """C2: one n x n layer drooped by z = 0.02 sin(6x) cos(4y) + N(0, 0.5 mm)."""
    rng = np.random.default_rng(seed)
    grid = grid_positions(n)
    x0 = grid.copy()
    x0[:, 2] = 0.02 * np.sin(6.0 * grid[:, 0]) * np.cos(4.0 * grid[:, 1])
    x0 += rng.normal(0.0, 5e-4, grid.shape)
    return _base("drooped_cloth_%d" % n, n, 1, grid, x0, np.zeros_like(x0),
                 1e-2, steps, 0, seed=seed,
                 description="%dx%d grid, sine droop + N(0,5e-4), no contacts"
                 % (n, n))


def jittered_cloth(n: int = 512, seed: int = 1002, steps: int = 10,
                   contact_frac: float = 0.01, radius_cells: int = 8) -> Workload:
    """C3: one n x n layer jittered by U(+-0.2 s), plus random contacts.

    Each step, a seeded 1% of the vertices each get one penalty contact
    (k = 1e3, rest length radius_cells * s) to a random other vertex whose
    grid-index distance is at most radius_cells.
    """
    rng = np.random.default_rng(seed)
    grid = grid_positions(n)
    x0 = grid + rng.uniform(-0.2 * SPACING, 0.2 * SPACING, grid.shape)
    N = n * n
    nc = int(contact_frac * N)
    r = radius_cells
    cand = [(di, dj) for di in range(-r, r + 1) for dj in range(-r, r + 1)
            if (di or dj) and di * di + dj * dj <= r * r]
    cand = np.asarray(cand, np.int64)

    def contact_fn(step, _x):
        g = step_rng(seed, step)
        a = g.choice(N, size=nc, replace=False)
        ai, aj = a // n, a % n
        pick = g.integers(0, len(cand), size=nc)
        bi, bj = ai + cand[pick, 0], aj + cand[pick, 1]
        # redraw partners that fall off the grid (bounded number of rounds),
        # then clip the few left over into the grid
        for _ in range(64):
            bad = (bi < 0) | (bi >= n) | (bj < 0) | (bj >= n)
            if not bad.any():
                break
            pick = g.integers(0, len(cand), size=int(bad.sum()))
            bi[bad] = ai[bad] + cand[pick, 0]
            bj[bad] = aj[bad] + cand[pick, 1]
        bi = np.clip(bi, 0, n - 1)
        bj = np.clip(bj, 0, n - 1)
        same = (bi == ai) & (bj == aj)
        bi = np.where(same, np.where(ai + 1 < n, ai + 1, ai - 1), bi)
        b = bi * n + bj
        return Contacts(a.astype(np.int32), b.astype(np.int32),
                        np.full(nc, K_CONTACT, np.float32),
                        np.full(nc, r * SPACING, np.float32))

    return _base("jittered_cloth_%d" % n, n, 1, grid, x0, np.zeros_like(x0),
                 1e-2, steps, nc, contact_fn=contact_fn, seed=seed,
                 description="%dx%d grid, jitter U(+-0.2s), %d contacts/step "
                 "within %d cells" % (n, n, nc, r))


def two_layer_cloth(n: int = 585, seed: int = 1003, steps: int = 10,
                    gap: float = 2e-3, churn: float = 0.05,
                    contact_rest: float = 3e-3) -> Workload:
    """C4: two flat n x n layers 2 mm apart, top shifted by s/2 in x and y.

    Contacts: every top vertex (i, j) to bottom vertex (i, j); each step a
    seeded 5% of them retarget to a random bottom vertex among
    (i..i+1, j..j+1), clipped to the grid.  Rest length 3 mm, k = 1e3.
    """
    grid = grid_positions(n)
    bottom = grid.copy()
    top = grid.copy()
    top[:, 0] += 0.5 * SPACING
    top[:, 1] += 0.5 * SPACING
    top[:, 2] += gap
    x0 = np.concatenate([bottom, top])
    N = 2 * n * n
    nc = n * n

    def contact_fn(step, _x):
        g = step_rng(seed, step)
        top_id = np.arange(n * n, dtype=np.int64)
        ti, tj = top_id // n, top_id % n
        bi, bj = ti.copy(), tj.copy()
        m = int(churn * nc)
        sel = g.choice(nc, size=m, replace=False)
        bi[sel] = np.minimum(ti[sel] + g.integers(0, 2, size=m), n - 1)
        bj[sel] = np.minimum(tj[sel] + g.integers(0, 2, size=m), n - 1)
        return Contacts((top_id + n * n).astype(np.int32),
                        (bi * n + bj).astype(np.int32),
                        np.full(nc, K_CONTACT, np.float32),
                        np.full(nc, contact_rest, np.float32))

    return _base("two_layer_cloth_%d" % n, n, 2, x0, x0,
                 np.zeros_like(x0), 1e-2, steps, nc, contact_fn=contact_fn,
                 seed=seed,
                 description="2 x %dx%d layers, gap %g m, top shifted s/2, "
                 "%d contacts/step, %g%% churn" % (n, n, gap, nc, churn * 100))


def folded_stack(n: int = 455, layers: int = 4, seed: int = 1004,
                 steps: int = 20, gap: float = 1.5e-3, amp: float = 0.05,
                 contact_frac: float = 0.10, contact_rest: float = 2e-3,
                 h: float = 5e-3) -> Workload:
    """C5: four stacked n x n layers with random folds z += 0.05 sin(k_l x).

    k_l ~ U[3, 9] per layer, layer gap 1.5 mm, rest lengths from the flat
    grid.  Contacts: each step a seeded 10% of all vertices, drawn from layers
    0..layers-2, each joined to the vertex (i + U{0,1}, j + U{0,1}) (clipped)
    of the layer above.  Rest length 2 mm, k = 1e3, h = 5e-3.
    """
    rng = np.random.default_rng(seed)
    grid = grid_positions(n)
    kl = rng.uniform(3.0, 9.0, size=layers)
    rest_layers, x_layers = [], []
    for layer in range(layers):
        flat = grid.copy()
        flat[:, 2] = layer * gap
        rest_layers.append(flat)
        folded = flat.copy()
        folded[:, 2] += amp * np.sin(kl[layer] * grid[:, 0])
        x_layers.append(folded)
    rest_pos = np.concatenate(rest_layers)
    x0 = np.concatenate(x_layers)
    N = n * n * layers
    nc = int(contact_frac * N)
    pool = n * n * (layers - 1)

    def contact_fn(step, _x):
        g = step_rng(seed, step)
        a = g.choice(pool, size=nc, replace=False).astype(np.int64)
        layer = a // (n * n)
        loc = a % (n * n)
        ai, aj = loc // n, loc % n
        bi = np.minimum(ai + g.integers(0, 2, size=nc), n - 1)
        bj = np.minimum(aj + g.integers(0, 2, size=nc), n - 1)
        b = (layer + 1) * n * n + bi * n + bj
        return Contacts(a.astype(np.int32), b.astype(np.int32),
                        np.full(nc, K_CONTACT, np.float32),
                        np.full(nc, contact_rest, np.float32))

    w = _base("folded_stack_%dx%d" % (layers, n), n, layers, rest_pos, x0,
              np.zeros_like(x0), h, steps, nc, contact_fn=contact_fn,
              seed=seed,
              description="%d x %dx%d layers, gap %g m, folds amp %g k~U[3,9], "
              "%d contacts/step" % (layers, n, n, gap, amp, nc))
    return w


CONFIGS = {
    "C1": tiny_cloth,
    "C2": drooped_cloth,
    "C3": jittered_cloth,
    "C4": two_layer_cloth,
    "C5": folded_stack,
}


def make(name: str, **kw) -> Workload:
    """Build a named configuration (C1..C5); keyword args override sizes."""
    return CONFIGS[name](**kw)
