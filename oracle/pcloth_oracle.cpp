// Plain fp64 CPU oracle for the implicit-integration hot path of P-Cloth
// (arXiv 2008.00409, "P-Cloth: Interactive Complex Cloth Simulation on
// Multi-GPU Systems using Dynamic Matrix Assembly and Pipelined Implicit
// Integrators").
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
// this file; only the tests, the package's smoke check and the benchmark's
// CPU-baseline leg do.  It shares no code, header, table or helper with the
// CUDA library.
//
// What it computes, step by step, in the order the page gives it:
//
//   Sec. 2.5, Eq. (1)-(3): backward Euler, with the force linearised around
//     time t, gives the linear system
//         (M - h^2 J) dv = h f(x_t + h v_t),
//     J the force Jacobian evaluated at x_t.  With K_e = -df_i/dx_i >= 0 the
//     stiffness block of element e = (i, j), the matrix is
//         A = M + h^2 sum_e K_e   (K_e added to blocks (i,i), (j,j),
//                                  subtracted from (i,j) and (j,i)).
//   Element model (the configurations' spring law; the page only says
//     "piece-wise linear elastic"):
//         e = x_j - x_i,  l = |e|,  d = e / l,
//         K_e = k [ max(0, 1 - L0/l) (I - d d^T) + d d^T ]     at x_t,
//         F_e = k (l~ - L0) d~   on i  (and -F_e on j)        at x~ = x_t + h v_t.
//     Gravity adds m_i g to f_i.  Contacts are elements of the same law.
//   Sec. 3.2.2 (sparse matrix filling, steps 1-5): the block pattern is the
//     set of (row, col) pairs touched by any element plus the diagonal,
//     sorted per row with duplicates removed; every duplicate contribution is
//     summed into its one block.
//   Sec. 3.1 / Eq. (3) text: the system is solved by preconditioned conjugate
//     gradients; the page does not name the preconditioner, this oracle uses
//     the inverse of each 3x3 diagonal block (block Jacobi).
//   Sec. 4.2-4.3 (proximity contacts, restricted to vertex pairs): every pair
//     of vertices i < j closer than a radius r that is not a spring becomes a
//     contact (a spring of stiffness k_c and rest length r), listed in (i, j)
//     order.  This is a brute-force test of all pairs.  The distance decides
//     an integer outcome, so it is taken in the GPU's precision: float32
//     differences, squared distance ((dx dx + dy dy) + dz dz) rounded after
//     every operation, compared strictly with r r rounded to float32.
//
// Everything is double precision and single threaded.  The only library
// primitives used are std::sort / std::unique / std::lower_bound and sqrt.
// Compile without -ffast-math and with -ffp-contract=off so that the results
// do not depend on the host's fused multiply-add policy.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <utility>
#include <vector>

namespace {

// Status codes (kept numerically equal to the library's public codes so a
// test can compare them, but defined here independently).
enum : int {
  OR_OK = 0,
  OR_NOT_CONVERGED = 1,
  OR_INVALID_ARG = -1,
  OR_BAD_INDEX = -3,
  OR_NONFINITE = -4,
  OR_BREAKDOWN = -5,
};

struct Element {
  int32_t a, b;   // vertex indices, a != b
  double k, rest; // stiffness, rest length
};

// One assembled system: BSR with 3x3 row-major blocks, all fp64.
struct System {
  int32_t n = 0;
  std::vector<int64_t> rowptr;  // n + 1
  std::vector<int32_t> colind;  // nnzb
  std::vector<double> vals;     // nnzb * 9
  std::vector<double> rhs;      // 3n: b = h f(x~)
  std::vector<double> pinv;     // 9n: inverse of each diagonal block
  int status = OR_OK;
};

inline double dot3(const double* u, const double* v) {
  return u[0] * v[0] + u[1] * v[1] + u[2] * v[2];
}

// Stiffness block K (row-major 3x3) of one element at positions (xa, xb),
// and the force on vertex a at the advanced positions (ya, yb).
// Returns false when a length is zero (the direction is undefined).
bool element_terms(const double* xa, const double* xb, const double* ya,
                   const double* yb, double k, double rest, double K[9],
                   double F[3]) {
  double e[3] = {xb[0] - xa[0], xb[1] - xa[1], xb[2] - xa[2]};
  double l = std::sqrt(dot3(e, e));
  double d[3] = {e[0] / l, e[1] / l, e[2] / l};
  double tension = 1.0 - rest / l;
  if (tension < 0.0) tension = 0.0;
  for (int r = 0; r < 3; ++r)
    for (int c = 0; c < 3; ++c) {
      double ident = (r == c) ? 1.0 : 0.0;
      K[r * 3 + c] = k * (tension * (ident - d[r] * d[c]) + d[r] * d[c]);
    }
  double et[3] = {yb[0] - ya[0], yb[1] - ya[1], yb[2] - ya[2]};
  double lt = std::sqrt(dot3(et, et));
  for (int r = 0; r < 3; ++r) F[r] = k * (lt - rest) * (et[r] / lt);
  return l > 0.0 && lt > 0.0;
}

// Inverse of a 3x3 matrix by Gauss-Jordan elimination with partial pivoting.
bool invert3(const double* m, double* inv) {
  double a[3][6];
  for (int r = 0; r < 3; ++r) {
    for (int c = 0; c < 3; ++c) a[r][c] = m[r * 3 + c];
    for (int c = 0; c < 3; ++c) a[r][3 + c] = (r == c) ? 1.0 : 0.0;
  }
  for (int col = 0; col < 3; ++col) {
    int piv = col;
    for (int r = col + 1; r < 3; ++r)
      if (std::fabs(a[r][col]) > std::fabs(a[piv][col])) piv = r;
    if (a[piv][col] == 0.0) return false;
    if (piv != col)
      for (int c = 0; c < 6; ++c) std::swap(a[piv][c], a[col][c]);
    double s = a[col][col];
    for (int c = 0; c < 6; ++c) a[col][c] /= s;
    for (int r = 0; r < 3; ++r) {
      if (r == col) continue;
      double f = a[r][col];
      for (int c = 0; c < 6; ++c) a[r][c] -= f * a[col][c];
    }
  }
  for (int r = 0; r < 3; ++r)
    for (int c = 0; c < 3; ++c) inv[r * 3 + c] = a[r][3 + c];
  return true;
}

// Position of block (row, col) in the assembled pattern.
int64_t find_block(const System& s, int32_t row, int32_t col) {
  auto first = s.colind.begin() + s.rowptr[row];
  auto last = s.colind.begin() + s.rowptr[row + 1];
  auto it = std::lower_bound(first, last, col);
  return int64_t(it - s.colind.begin());
}

void gather_elements(std::vector<Element>& out, int32_t n, const int32_t* ei,
                     const int32_t* ej, const float* ek, const float* er) {
  for (int32_t e = 0; e < n; ++e)
    out.push_back(Element{ei[e], ej[e], double(ek[e]), double(er[e])});
}

System* assemble(int32_t n, const float* mass, const float* gravity,
                 int32_t ns, const int32_t* si, const int32_t* sj,
                 const float* sk, const float* sr, int32_t nc,
                 const int32_t* ci, const int32_t* cj, const float* ck,
                 const float* cr, const float* x, const float* v, double h) {
  System* s = new System();
  s->n = n;
  if (n <= 0 || ns < 0 || nc < 0) {
    s->status = OR_INVALID_ARG;
    return s;
  }
  // The element list: springs first, then contacts, each in input order.
  std::vector<Element> elems;
  elems.reserve(size_t(ns) + size_t(nc));
  gather_elements(elems, ns, si, sj, sk, sr);
  gather_elements(elems, nc, ci, cj, ck, cr);
  for (const Element& e : elems) {
    if (e.a < 0 || e.a >= n || e.b < 0 || e.b >= n || e.a == e.b) {
      s->status = OR_BAD_INDEX;
      return s;
    }
  }

  // Pattern (filling steps 1-3): every (row, col) touched, plus the
  // diagonal; sort; drop duplicates.
  std::vector<std::pair<int32_t, int32_t>> keys;
  keys.reserve(size_t(n) + 2 * elems.size());
  for (int32_t i = 0; i < n; ++i) keys.emplace_back(i, i);
  for (const Element& e : elems) {
    keys.emplace_back(e.a, e.b);
    keys.emplace_back(e.b, e.a);
  }
  std::sort(keys.begin(), keys.end());
  keys.erase(std::unique(keys.begin(), keys.end()), keys.end());
  s->rowptr.assign(size_t(n) + 1, 0);
  s->colind.resize(keys.size());
  for (size_t t = 0; t < keys.size(); ++t) {
    s->rowptr[keys[t].first + 1] += 1;
    s->colind[t] = keys[t].second;
  }
  for (int32_t i = 0; i < n; ++i) s->rowptr[i + 1] += s->rowptr[i];

  // Values (filling step 5) and the right-hand side.
  s->vals.assign(keys.size() * 9, 0.0);
  std::vector<double> f(size_t(n) * 3, 0.0);
  const double h2 = h * h;
  for (int32_t i = 0; i < n; ++i) {
    double* D = &s->vals[size_t(find_block(*s, i, i)) * 9];
    for (int r = 0; r < 3; ++r) D[r * 4] += double(mass[i]);
    for (int r = 0; r < 3; ++r) f[size_t(i) * 3 + r] += double(mass[i]) * double(gravity[r]);
  }
  bool finite = true;
  for (const Element& e : elems) {
    double xa[3], xb[3], ya[3], yb[3];
    for (int r = 0; r < 3; ++r) {
      xa[r] = x[size_t(e.a) * 3 + r];
      xb[r] = x[size_t(e.b) * 3 + r];
      ya[r] = xa[r] + h * double(v[size_t(e.a) * 3 + r]);
      yb[r] = xb[r] + h * double(v[size_t(e.b) * 3 + r]);
    }
    double K[9], F[3];
    if (!element_terms(xa, xb, ya, yb, e.k, e.rest, K, F)) finite = false;
    double* Aaa = &s->vals[size_t(find_block(*s, e.a, e.a)) * 9];
    double* Abb = &s->vals[size_t(find_block(*s, e.b, e.b)) * 9];
    double* Aab = &s->vals[size_t(find_block(*s, e.a, e.b)) * 9];
    double* Aba = &s->vals[size_t(find_block(*s, e.b, e.a)) * 9];
    for (int t = 0; t < 9; ++t) {
      Aaa[t] += h2 * K[t];
      Abb[t] += h2 * K[t];
      Aab[t] -= h2 * K[t];
      Aba[t] -= h2 * K[t];
    }
    for (int r = 0; r < 3; ++r) {
      f[size_t(e.a) * 3 + r] += F[r];
      f[size_t(e.b) * 3 + r] -= F[r];
    }
  }
  s->rhs.resize(size_t(n) * 3);
  for (size_t t = 0; t < s->rhs.size(); ++t) s->rhs[t] = h * f[t];

  // Block-Jacobi preconditioner: P_i = (A_ii)^-1.
  s->pinv.assign(size_t(n) * 9, 0.0);
  for (int32_t i = 0; i < n; ++i) {
    const double* D = &s->vals[size_t(find_block(*s, i, i)) * 9];
    if (!invert3(D, &s->pinv[size_t(i) * 9])) finite = false;
  }
  for (double t : s->vals)
    if (!std::isfinite(t)) finite = false;
  for (double t : s->rhs)
    if (!std::isfinite(t)) finite = false;
  if (!finite) s->status = OR_NONFINITE;
  return s;
}

// y = A x (fp64), the block definition of the product.
void spmv(const System& s, const double* xin, double* y) {
  for (int32_t i = 0; i < s.n; ++i) {
    double acc[3] = {0.0, 0.0, 0.0};
    for (int64_t p = s.rowptr[i]; p < s.rowptr[i + 1]; ++p) {
      const double* B = &s.vals[size_t(p) * 9];
      const double* xj = &xin[size_t(s.colind[p]) * 3];
      for (int r = 0; r < 3; ++r)
        acc[r] += B[r * 3 + 0] * xj[0] + B[r * 3 + 1] * xj[1] + B[r * 3 + 2] * xj[2];
    }
    for (int r = 0; r < 3; ++r) y[size_t(i) * 3 + r] = acc[r];
  }
}

double dot(const std::vector<double>& u, const std::vector<double>& v) {
  double acc = 0.0;
  for (size_t t = 0; t < u.size(); ++t) acc += u[t] * v[t];
  return acc;
}

void apply_pinv(const System& s, const std::vector<double>& r,
                std::vector<double>& z) {
  for (int32_t i = 0; i < s.n; ++i) {
    const double* P = &s.pinv[size_t(i) * 9];
    const double* ri = &r[size_t(i) * 3];
    for (int c = 0; c < 3; ++c)
      z[size_t(i) * 3 + c] = P[c * 3 + 0] * ri[0] + P[c * 3 + 1] * ri[1] + P[c * 3 + 2] * ri[2];
  }
}

// Textbook preconditioned CG on A dv = b, dv_0 = 0, stop when the recursive
// residual satisfies |r|_2 <= tol |b|_2 (checked after each update of r).
// PCG from the initial guess x0 (nullptr: dv = 0).  With a guess the
// residual starts as r = b - A x0 and the iteration is otherwise unchanged;
// the stop test stays |r| <= tol |b|, and a guess that already meets it is
// returned after 0 iterations.
int pcg(const System& s, double tol, int32_t maxit, double* dv_out,
        int32_t* iters, double* relres, const double* x0 = nullptr) {
  const size_t m = size_t(s.n) * 3;
  std::vector<double> dv(m, 0.0), r(s.rhs), z(m), p(m), q(m);
  *iters = 0;
  double bnorm = std::sqrt(dot(s.rhs, s.rhs));
  if (bnorm == 0.0) {
    std::fill(dv_out, dv_out + m, 0.0);
    *relres = 0.0;
    return OR_OK;
  }
  if (x0 != nullptr) {
    std::copy(x0, x0 + m, dv.begin());
    spmv(s, dv.data(), q.data());
    for (size_t t = 0; t < m; ++t) r[t] = s.rhs[t] - q[t];
  }
  double rnorm = std::sqrt(dot(r, r));
  if (x0 != nullptr) {
    *relres = rnorm / bnorm;
    if (rnorm <= tol * bnorm || maxit <= 0) {
      std::copy(dv.begin(), dv.end(), dv_out);
      return rnorm <= tol * bnorm ? OR_OK : OR_NOT_CONVERGED;
    }
  }
  apply_pinv(s, r, z);
  p = z;
  double rz = dot(r, z);
  for (int32_t it = 1; it <= maxit; ++it) {
    spmv(s, p.data(), q.data());
    double pq = dot(p, q);
    if (!(pq > 0.0)) {
      *iters = it;
      *relres = rnorm / bnorm;
      std::copy(dv.begin(), dv.end(), dv_out);
      return std::isfinite(pq) ? OR_BREAKDOWN : OR_NONFINITE;
    }
    double alpha = rz / pq;
    for (size_t t = 0; t < m; ++t) {
      dv[t] += alpha * p[t];
      r[t] -= alpha * q[t];
    }
    rnorm = std::sqrt(dot(r, r));
    *iters = it;
    *relres = rnorm / bnorm;
    if (rnorm <= tol * bnorm) {
      std::copy(dv.begin(), dv.end(), dv_out);
      return OR_OK;
    }
    apply_pinv(s, r, z);
    double rz_new = dot(r, z);
    if (!(rz_new > 0.0)) {
      std::copy(dv.begin(), dv.end(), dv_out);
      return std::isfinite(rz_new) ? OR_BREAKDOWN : OR_NONFINITE;
    }
    double beta = rz_new / rz;
    rz = rz_new;
    for (size_t t = 0; t < m; ++t) p[t] = z[t] + beta * p[t];
  }
  std::copy(dv.begin(), dv.end(), dv_out);
  return OR_NOT_CONVERGED;
}

}  // namespace

extern "C" {

// Stiffness block and force of one element (see element_terms above).
// xa, xb: positions at t; va, vb: velocities; the force is evaluated at
// x + h v.  Returns 1 when both lengths are nonzero, else 0.
int oracle_element(const double* xa, const double* xb, const double* va,
                   const double* vb, double k, double rest, double h,
                   double* K, double* F) {
  double ya[3], yb[3];
  for (int r = 0; r < 3; ++r) {
    ya[r] = xa[r] + h * va[r];
    yb[r] = xb[r] + h * vb[r];
  }
  return element_terms(xa, xb, ya, yb, k, rest, K, F) ? 1 : 0;
}

void* oracle_assemble(int32_t n, const float* mass, const float* gravity,
                      int32_t ns, const int32_t* si, const int32_t* sj,
                      const float* sk, const float* sr, int32_t nc,
                      const int32_t* ci, const int32_t* cj, const float* ck,
                      const float* cr, const float* x, const float* v,
                      double h) {
  try {
    return assemble(n, mass, gravity, ns, si, sj, sk, sr, nc, ci, cj, ck, cr,
                    x, v, h);
  } catch (const std::bad_alloc&) {
    return nullptr;
  }
}

int oracle_status(const void* sys) {
  return static_cast<const System*>(sys)->status;
}

int64_t oracle_nnzb(const void* sys) {
  const System* s = static_cast<const System*>(sys);
  return s->rowptr.empty() ? 0 : s->rowptr.back();
}

// Copies the assembled system out; any pointer may be null.
void oracle_export(const void* sys, int64_t* rowptr, int32_t* colind,
                   double* vals, double* rhs, double* pinv) {
  const System* s = static_cast<const System*>(sys);
  if (rowptr) std::copy(s->rowptr.begin(), s->rowptr.end(), rowptr);
  if (colind) std::copy(s->colind.begin(), s->colind.end(), colind);
  if (vals) std::copy(s->vals.begin(), s->vals.end(), vals);
  if (rhs) std::copy(s->rhs.begin(), s->rhs.end(), rhs);
  if (pinv) std::copy(s->pinv.begin(), s->pinv.end(), pinv);
}

void oracle_spmv(const void* sys, const double* xin, double* y) {
  spmv(*static_cast<const System*>(sys), xin, y);
}

int oracle_pcg(const void* sys, double tol, int32_t maxit, double* dv,
               int32_t* iters, double* relres) {
  return pcg(*static_cast<const System*>(sys), tol, maxit, dv, iters, relres);
}

// The same PCG started from the guess x0 (float64[n][3]).
int oracle_pcg_x0(const void* sys, double tol, int32_t maxit, const double* x0, double* dv,
                  int32_t* iters, double* relres) {
  return pcg(*static_cast<const System*>(sys), tol, maxit, dv, iters, relres, x0);
}

// Backward-Euler state update of Eq. (3): v <- v + dv, then x <- x + h v.
void oracle_update(int32_t n, const float* x, const float* v, const double* dv,
                   double h, double* x_out, double* v_out) {
  for (size_t t = 0; t < size_t(n) * 3; ++t) {
    v_out[t] = double(v[t]) + dv[t];
    x_out[t] = double(x[t]) + h * v_out[t];
  }
}

void oracle_free(void* sys) { delete static_cast<System*>(sys); }

// Vertex-vertex proximity contacts (see the header): writes up to `capacity`
// pairs (i, j), i < j, in (i, j) order and returns how many exist.  Spring
// pairs (si[s], sj[s]), in either order, are not contacts.
int64_t oracle_find_contacts(int32_t n, const float* x, float radius, int32_t ns,
                             const int32_t* si, const int32_t* sj, int32_t* out_i,
                             int32_t* out_j, int64_t capacity) {
  std::vector<std::pair<int32_t, int32_t>> springs;
  springs.reserve(size_t(ns));
  for (int32_t s = 0; s < ns; ++s)
    springs.emplace_back(std::min(si[s], sj[s]), std::max(si[s], sj[s]));
  std::sort(springs.begin(), springs.end());
  const float r2 = radius * radius;
  int64_t count = 0;
  for (int32_t i = 0; i < n; ++i) {
    for (int32_t j = i + 1; j < n; ++j) {
      const float dx = x[3 * size_t(j)] - x[3 * size_t(i)];
      const float dy = x[3 * size_t(j) + 1] - x[3 * size_t(i) + 1];
      const float dz = x[3 * size_t(j) + 2] - x[3 * size_t(i) + 2];
      const float xx = dx * dx;
      const float yy = dy * dy;
      const float zz = dz * dz;
      const float d2 = (xx + yy) + zz;
      if (!(d2 < r2)) continue;
      if (std::binary_search(springs.begin(), springs.end(), std::make_pair(i, j))) continue;
      if (count < capacity) {
        out_i[count] = i;
        out_j[count] = j;
      }
      ++count;
    }
  }
  return count;
}

}  // extern "C"
