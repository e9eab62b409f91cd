// Per-step assembly of A dv = b (P-Cloth, arXiv 2008.00409: Sec. 2.5
// Eq. (3) for the system, Sec. 3.2 for the assembly elements, Sec. 3.2.2 for
// the sparse matrix filling).
//
// The page fills an ELL index table with atomics, sorts and compacts each row
// with one thread per row, then fills values with atomics.  This design keeps
// BSR3 and replaces those steps with deterministic ones:
//
//   contact_keys     two directed keys (row << B | col) per contact
//   radix sort       stable, so equal keys keep their input order
//   contact_classify flag the first entry of every (row, col) pair that is
//                    not already a block of the static spring pattern
//   scan + compact   list of new blocks, sorted by (row, col)
//   tile_bounds      per tile of rows: first new block / first entry
//   assemble_rows    per tile: rebuild rowptr and colind in place (static
//                    blocks shifted by the new blocks of earlier rows, new
//                    blocks merged into their rows), evaluate every element
//                    of every off-diagonal block, reduce each row into its
//                    diagonal block, b = h f and the block-Jacobi inverse.
//
// No float atomics: every sum has a fixed order, so the assembled system is
// bitwise reproducible.  Each off-diagonal block is computed by its own row;
// the block (j, i) is computed from the negated edge vector and is therefore
// bitwise equal to the block (i, j).  Every block is a symmetric 3x3 (a sum
// of element stiffnesses k[a I + c d d^T], plus m I on the diagonal) and is
// stored packed, six floats (a00 a01 a02 a11 a12 a22) per block, which cuts
// the bytes every SpMV streams by a third.

#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

constexpr uint64_t kSentinel = ~0ull;
constexpr int kRowLanes = kAsmThreads / kAsmRows;   // threads per row in the row reductions
static_assert(kRowLanes == 8, "the row reduction merges eight lanes");

struct AsmArgs {
  int32_t n;
  int B;                 // bits per index in a key
  float dt, h2;
  float gx, gy, gz;
  const float* x;
  const float* v;
  const float* mass;
  const int32_t* rowptr_s;
  const int32_t* colind_s;
  const int32_t* sblk_ptr;
  const float2* sentry;
  int has_contacts;
  const uint64_t* skey;    // sorted contact keys
  const int32_t* sval;     // contact id of each sorted key
  const float* ck;
  const float* cr;
  const uint64_t* newkey;
  const int32_t* newfirst;
  const int32_t* tile_nb;
  const int32_t* tile_eb;
  const int32_t* counters;  // [0] new blocks, [1] valid entries
  int32_t* rowptr;
  int32_t* colind;
  float* vals;
  float* rhs;
  float* pinv6;      // [6][vs]
  int64_t vs;
  uint32_t* status;
};

__global__ void contact_keys(int32_t nc, int32_t n, int B, const int32_t* __restrict__ ci,
                             const int32_t* __restrict__ cj, const float* __restrict__ ck,
                             const float* __restrict__ cr, uint64_t* __restrict__ keys,
                             int32_t* __restrict__ vals, uint32_t* status) {
  const int32_t c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= nc) return;
  const int32_t i = ci[c], j = cj[c];
  const bool ok = i >= 0 && i < n && j >= 0 && j < n && i != j;
  if (!ok) atomicOr(status, ST_BAD_INDEX);
  if (!isfinite(ck[c]) || !isfinite(cr[c])) atomicOr(status, ST_NONFINITE);
  keys[2 * int64_t(c)] = ok ? (uint64_t(i) << B) | uint64_t(j) : kSentinel;
  keys[2 * int64_t(c) + 1] = ok ? (uint64_t(j) << B) | uint64_t(i) : kSentinel;
  vals[2 * int64_t(c)] = c;
  vals[2 * int64_t(c) + 1] = c;
}

__device__ __forceinline__ bool static_has(const int32_t* __restrict__ colind_s,
                                           int32_t lo, int32_t hi, int32_t col) {
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    const int32_t c = colind_s[mid];
    if (c == col) return true;
    if (c < col) lo = mid + 1; else hi = mid;
  }
  return false;
}

__global__ void contact_classify(int32_t m, int B, const uint64_t* __restrict__ skey,
                                 const int32_t* __restrict__ rowptr_s,
                                 const int32_t* __restrict__ colind_s,
                                 int32_t* __restrict__ flags, int32_t* __restrict__ counters) {
  const int32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= m) return;
  const uint64_t key = skey[t];
  int32_t f = 0;
  if (key != kSentinel) {
    const uint64_t mask = (uint64_t(1) << B) - 1;
    const int32_t row = int32_t(key >> B), col = int32_t(key & mask);
    const bool first = (t == 0) || skey[t - 1] != key;
    if (first && !static_has(colind_s, rowptr_s[row], rowptr_s[row + 1], col)) f = 1;
    // sentinels sort last: the last valid entry records the valid count
    if (t + 1 == m || skey[t + 1] == kSentinel) counters[1] = t + 1;
  }
  flags[t] = f;
}

__global__ void contact_compact(int32_t m, const uint64_t* __restrict__ skey,
                                const int32_t* __restrict__ prefix,
                                const int32_t* __restrict__ counters,
                                uint64_t* __restrict__ newkey, int32_t* __restrict__ newfirst) {
  const int32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= m) return;
  const int32_t next = (t + 1 < m) ? prefix[t + 1] : counters[0];
  if (next != prefix[t]) {
    newkey[prefix[t]] = skey[t];
    newfirst[prefix[t]] = t;
  }
}

__device__ __forceinline__ int32_t lower_bound_key(const uint64_t* __restrict__ a,
                                                   int32_t lo, int32_t hi, uint64_t key) {
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void tile_bounds(int32_t ntiles, int32_t n, int B, int has_contacts,
                            const uint64_t* __restrict__ newkey,
                            const uint64_t* __restrict__ skey,
                            const int32_t* __restrict__ counters,
                            int32_t* __restrict__ tile_nb, int32_t* __restrict__ tile_eb) {
  const int32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t > ntiles) return;
  if (!has_contacts) {
    tile_nb[t] = 0;
    tile_eb[t] = 0;
    return;
  }
  const int64_t r = min(int64_t(t) * kAsmRows, int64_t(n));
  const uint64_t key = uint64_t(r) << B;
  tile_nb[t] = lower_bound_key(newkey, 0, counters[0], key);
  tile_eb[t] = lower_bound_key(skey, 0, counters[1], key);
}

// An edge vector carried exactly as hi + lo: the difference of two fp32
// coordinates is rounded in fp32, and near the rest shape of a flat sheet
// that rounding alone (a tilt of the spring axis by ~1e-8) shifts the
// solution along the soft out-of-plane modes by ~1e-4.  TwoSum recovers the
// rounding error exactly; x_i - x_j gives exactly (-hi, -lo), so the blocks
// (i, j) and (j, i) stay bitwise equal.
struct Edge {
  float3 hi, lo;
};

__device__ __forceinline__ float two_diff_lo(float a, float b, float s) {  // s = fl(a - b)
  const float bp = s - a;
  return (a - (s - bp)) + (-b - bp);
}

__device__ __forceinline__ Edge edge_of(float3 xi, float3 xj) {
  Edge e;
  e.hi = make_float3(xj.x - xi.x, xj.y - xi.y, xj.z - xi.z);
  e.lo = make_float3(two_diff_lo(xj.x, xi.x, e.hi.x), two_diff_lo(xj.y, xi.y, e.hi.y),
                     two_diff_lo(xj.z, xi.z, e.hi.z));
  return e;
}

// |e|^2 - L0^2 from an exact edge e = hi + lo, in fp32 pairs: the four large
// terms hi.x^2, hi.y^2, hi.z^2 and -L0^2 are split exactly into product and
// residual by an FMA and the products summed by TwoSum, so the cancellation
// near the rest length loses nothing; the residuals, the cross terms
// 2 hi.lo and lo.lo (all about 2^-24 of the squares or smaller) are added in
// plain fp32.  The error is about 2^-48 |e|^2, like an fp64 evaluation, at
// fp32 speed (fp64 is a slow path on this GPU).  Every term is even in e, so
// the edges e and -e give the same bits.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& t) {
  s = a + b;
  const float bp = s - a;
  t = (a - (s - bp)) + (b - bp);
}

__device__ __forceinline__ float excess_sq(float3 hi, float3 lo, float L0) {
  const float px = hi.x * hi.x, py = hi.y * hi.y, pz = hi.z * hi.z, pl = -(L0 * L0);
  const float rx = fmaf(hi.x, hi.x, -px), ry = fmaf(hi.y, hi.y, -py);
  const float rz = fmaf(hi.z, hi.z, -pz), rl = fmaf(-L0, L0, -pl);
  float s, t1, t2, t3;
  two_sum(px, py, s, t1);
  two_sum(s, pz, s, t2);
  two_sum(s, pl, s, t3);
  const float cross = 2.0f * fmaf(hi.x, lo.x, fmaf(hi.y, lo.y, hi.z * lo.z)) +
                      fmaf(lo.x, lo.x, fmaf(lo.y, lo.y, lo.z * lo.z));
  const float small = ((t1 + t2) + t3) + (((rx + ry) + rz) + rl) + cross;
  return s + small;
}

// Scaled stiffness block K' = -h^2 K (6 unique entries of the symmetric
// block) and force F of one element seen from vertex i: K at x, force at
// x~ = x + h v.  e = x_j - x_i (exact, see Edge) is shared by all elements of
// a block and w = v_j - v_i.
//
// K = a I + c d d^T with a = k max(0, 1 - L0/l), c = k - a.  The length
// excess l - L0 is formed as (|e|^2 - L0^2) / (l + L0) with the squares in
// fp32 pairs: near the rest length the plain fp32 difference is pure rounding noise
// (~1e-7 L0) that would give a spring at rest a spurious transverse stiffness
// along exactly the soft out-of-plane directions of a flat sheet.  Written
// as K' = A I + S e e^T with A = -h^2 a and S = -h^2 c / l^2, each product
// e_r e_c is formed in double-float (exact hi*hi by an FMA plus the hi*lo
// cross terms) and scaled by S with about one rounding; any error in S is
// common to the whole e e^T term, so the block keeps its rank-one-plus-
// identity structure.
//
// The advanced edge is formed as e + h w, not as a difference of advanced
// positions, so it keeps the accuracy of the short edge instead of that of
// the (possibly metres-large) coordinates.
__device__ __forceinline__ float scaled_entry(float S, float hr, float lr, float hc, float lc) {
  const float p = hr * hc;
  const float pe = fmaf(hr, hc, -p);             // hr * hc == p + pe exactly
  const float tail = pe + fmaf(hr, lc, lr * hc);
  return fmaf(S, p, S * tail);
}

__device__ __forceinline__ void element_terms(const Edge& e, float3 w, float dt, float h2,
                                              float k, float L0, float (&K)[6], float (&F)[3]) {
  const float3 h = e.hi, o = e.lo;
  const float l2 = fmaf(h.x, h.x, fmaf(h.y, h.y, h.z * h.z)) +
                   2.0f * fmaf(h.x, o.x, fmaf(h.y, o.y, h.z * o.z));
  const float l = sqrtf(l2);
  const float stretch = excess_sq(h, o, L0) / (l + L0);    // l - L0
  const float tension = fmaxf(0.0f, stretch / l);                  // max(0, 1 - L0/l)
  const float a = k * tension;
  const float c = k - a;
  const float A = -h2 * a;
  const float S = (-h2 * c) / l2;
  K[0] += scaled_entry(S, h.x, o.x, h.x, o.x) + A;
  K[1] += scaled_entry(S, h.x, o.x, h.y, o.y);
  K[2] += scaled_entry(S, h.x, o.x, h.z, o.z);
  K[3] += scaled_entry(S, h.y, o.y, h.y, o.y) + A;
  K[4] += scaled_entry(S, h.y, o.y, h.z, o.z);
  K[5] += scaled_entry(S, h.z, o.z, h.z, o.z) + A;
  // force at the advanced positions
  const float fx = fmaf(dt, w.x, h.x) + o.x, fy = fmaf(dt, w.y, h.y) + o.y,
              fz = fmaf(dt, w.z, h.z) + o.z;
  const float lt = sqrtf(fx * fx + fy * fy + fz * fz);
  const float3 fz3 = make_float3(0.f, 0.f, 0.f);
  const float st = excess_sq(make_float3(fx, fy, fz), fz3, L0) / (lt + L0);   // l~ - L0
  const float s = k * st / lt;
  F[0] += s * fx;
  F[1] += s * fy;
  F[2] += s * fz;
}

__device__ __forceinline__ float3 ld3(const float* p, int64_t i) {
  return make_float3(p[3 * i], p[3 * i + 1], p[3 * i + 2]);
}

// Merge position p of two sorted disjoint lists S (static cols) and T (new
// contact cols): returns a = number of S entries before position p.
__device__ __forceinline__ int32_t merge_split(const int32_t* __restrict__ S, int32_t nS,
                                               const uint64_t* __restrict__ T, int32_t nT,
                                               uint64_t mask, int32_t p) {
  int32_t lo = max(0, p - nT), hi = min(p, nS);
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (S[mid - 1] < int32_t(T[p - mid] & mask)) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct RowInfo {
  int32_t sb, se;   // static slots
  int32_t nb, ne;   // new blocks
  int32_t eb, ee;   // sorted contact entries
  int32_t ob;       // first output block
};

// Computes block `o` (absolute output index) of tile-local row `ri`; writes
// the value (-h^2 sum K as a packed symmetric block, 6 floats) and the force
// sum into shared staging.
__device__ __forceinline__ void compute_block(const AsmArgs& a, int32_t i, const RowInfo& R,
                                              int32_t p, float* __restrict__ stv,
                                              float* __restrict__ stf, int32_t* __restrict__ stc,
                                              int32_t m_valid) {
  const uint64_t mask = (uint64_t(1) << a.B) - 1;
  const int32_t nS = R.se - R.sb, nT = R.ne - R.nb;
  int32_t col, sslot = -1, nk = -1;
  if (nT == 0) {
    sslot = R.sb + p;
    col = a.colind_s[sslot];
  } else {
    const int32_t s = merge_split(a.colind_s + R.sb, nS, a.newkey + R.nb, nT, mask, p);
    const int32_t t = p - s;
    if (s < nS && (t >= nT || a.colind_s[R.sb + s] < int32_t(a.newkey[R.nb + t] & mask))) {
      sslot = R.sb + s;
      col = a.colind_s[sslot];
    } else {
      nk = R.nb + t;
      col = int32_t(a.newkey[nk] & mask);
    }
  }
  float K[6] = {0, 0, 0, 0, 0, 0}, F[3] = {0, 0, 0};
  if (col != i) {
    const float3 xi = ld3(a.x, i), vi = ld3(a.v, i);
    const float3 xj = ld3(a.x, col), vj = ld3(a.v, col);
    const Edge ed = edge_of(xi, xj);
    const float3 wd = make_float3(vj.x - vi.x, vj.y - vi.y, vj.z - vi.z);
    if (sslot >= 0) {
      const int32_t e1 = a.sblk_ptr[sslot + 1];
      for (int32_t e = a.sblk_ptr[sslot]; e < e1; ++e) {
        const float2 kl = a.sentry[e];
        element_terms(ed, wd, a.dt, a.h2, kl.x, kl.y, K, F);
      }
    }
    // contacts on this (row, col) pair: a run of equal sorted keys
    int32_t t0 = -1;
    const uint64_t key = (uint64_t(i) << a.B) | uint64_t(col);
    if (nk >= 0) {
      t0 = a.newfirst[nk];
    } else if (R.ee > R.eb) {
      const int32_t t = lower_bound_key(a.skey, R.eb, R.ee, key);
      if (t < R.ee && a.skey[t] == key) t0 = t;
    }
    if (t0 >= 0) {
      for (int32_t t = t0; t < m_valid && a.skey[t] == key; ++t) {
        const int32_t c = a.sval[t];
        element_terms(ed, wd, a.dt, a.h2, a.ck[c], a.cr[c], K, F);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kSymBlock; ++t) stv[t] = K[t];
  stf[0] = F[0]; stf[1] = F[1]; stf[2] = F[2];
  *stc = col;
}

// Diagonal block, right-hand side and block-Jacobi inverse of row i from the
// row's compensated sum h^2 sum K = Ks + Kc (6 unique entries, Kc the
// TwoSum compensation) and its force sum.  The mass is added to the small
// compensation term first, so the diagonal is rounded once from the exact
// total: adding m after rounding the large sum would round the same m to the
// same ulp grid in every row of a binade -- a coherent shift of the mass by
// ~0.1%, which the soft modes of the system amplify.
__device__ __forceinline__ void finish_row(const AsmArgs& a, int32_t i, const float (&Ks)[6],
                                           const float (&Kc)[6], const float (&Fs)[3],
                                           float (&D)[kSymBlock]) {
  const float m = a.mass[i];
  // packed symmetric diagonal block (d00 d01 d02 d11 d12 d22)
  D[0] = Ks[0] + (Kc[0] + m); D[1] = Ks[1] + Kc[1]; D[2] = Ks[2] + Kc[2];
  D[3] = Ks[3] + (Kc[3] + m); D[4] = Ks[4] + Kc[4]; D[5] = Ks[5] + (Kc[5] + m);
  const float b0 = a.dt * (Fs[0] + m * a.gx);
  const float b1 = a.dt * (Fs[1] + m * a.gy);
  const float b2 = a.dt * (Fs[2] + m * a.gz);
  a.rhs[3 * int64_t(i)] = b0;
  a.rhs[3 * int64_t(i) + 1] = b1;
  a.rhs[3 * int64_t(i) + 2] = b2;
  // inverse of the symmetric block by its adjugate
  const float d00 = D[0], d01 = D[1], d02 = D[2], d11 = D[3], d12 = D[4], d22 = D[5];
  const float c00 = d11 * d22 - d12 * d12;
  const float c01 = d12 * d02 - d01 * d22;
  const float c02 = d01 * d12 - d11 * d02;
  const float c11 = d00 * d22 - d02 * d02;
  const float c12 = d02 * d01 - d00 * d12;
  const float c22 = d00 * d11 - d01 * d01;
  const float det = d00 * c00 + d01 * c01 + d02 * c02;
  const float id = 1.0f / det;
  // the inverse of a symmetric block is symmetric: six entries, one plane each
  a.pinv6[i] = c00 * id;
  a.pinv6[a.vs + i] = c01 * id;
  a.pinv6[2 * a.vs + i] = c02 * id;
  a.pinv6[3 * a.vs + i] = c11 * id;
  a.pinv6[4 * a.vs + i] = c12 * id;
  a.pinv6[5 * a.vs + i] = c22 * id;
  bool ok = finite3(b0, b1, b2) && isfinite(det) && det > 0.0f;
#pragma unroll
  for (int t = 0; t < kSymBlock; ++t) ok = ok && isfinite(D[t]);
  if (!ok) atomicOr(a.status, ST_NONFINITE);
}

// Four CTAs per SM (64 registers a thread): the kernel is bound by the
// latency of its gathers and of the per-row reductions, so occupancy pays
// more than the few spills it costs.
__global__ void __launch_bounds__(kAsmThreads, 4)
assemble_rows(AsmArgs a) {
  __shared__ RowInfo rows[kAsmRows + 1];
  __shared__ float stv[kAsmCap * kSymBlock];
  __shared__ float stf[kAsmCap * 3];
  __shared__ int32_t stc[kAsmCap];
  __shared__ double red[9][kAsmThreads / 32];
  __shared__ double acc[9];

  const int32_t r0 = blockIdx.x * kAsmRows;
  const int32_t nrows = min(kAsmRows, a.n - r0);
  const int32_t m_valid = a.has_contacts ? a.counters[1] : 0;
  const uint64_t mask = (uint64_t(1) << a.B) - 1;
  (void)mask;

  // ---- phase 1: row bounds, rebuilt row pointers ------------------------
  if (threadIdx.x <= nrows) {
    const int32_t ri = threadIdx.x, i = r0 + ri;
    RowInfo R;
    R.sb = a.rowptr_s[i];
    R.se = (ri < nrows) ? a.rowptr_s[i + 1] : R.sb;
    if (a.has_contacts) {
      const int32_t nb0 = a.tile_nb[blockIdx.x], nb1 = a.tile_nb[blockIdx.x + 1];
      const int32_t eb0 = a.tile_eb[blockIdx.x], eb1 = a.tile_eb[blockIdx.x + 1];
      const uint64_t key = uint64_t(i) << a.B;
      R.nb = (ri == 0) ? nb0 : (ri == nrows ? nb1 : lower_bound_key(a.newkey, nb0, nb1, key));
      R.eb = (ri == 0) ? eb0 : (ri == nrows ? eb1 : lower_bound_key(a.skey, eb0, eb1, key));
    } else {
      R.nb = 0;
      R.eb = 0;
    }
    R.ob = R.sb + R.nb;
    rows[ri] = R;
    if (ri < nrows || i == a.n) a.rowptr[i] = R.ob;
  }
  __syncthreads();
  if (threadIdx.x < nrows) {
    rows[threadIdx.x].ne = rows[threadIdx.x + 1].nb;
    rows[threadIdx.x].ee = rows[threadIdx.x + 1].eb;
  }
  __syncthreads();

  // ---- phase 2..4: groups of whole rows that fit in the staging ---------
  int32_t g = 0;
  while (g < nrows) {
    int32_t e = g + 1;
    while (e < nrows && rows[e + 1].ob - rows[g].ob <= kAsmCap) ++e;
    const int32_t gob = rows[g].ob;
    const int32_t nblk = rows[e].ob - gob;
    if (nblk <= kAsmCap) {
      // phase 2: every block of the group, one thread per block
      for (int32_t o = threadIdx.x; o < nblk; o += kAsmThreads) {
        // row of block o: last ri in [g, e) with rows[ri].ob <= gob + o
        int32_t lo = g, hi = e - 1;
        while (lo < hi) {
          const int32_t mid = (lo + hi + 1) >> 1;
          if (rows[mid].ob <= gob + o) lo = mid; else hi = mid - 1;
        }
        const RowInfo R = rows[lo];
        compute_block(a, r0 + lo, R, gob + o - R.ob, &stv[kSymBlock * o], &stf[3 * o], &stc[o],
                      m_valid);
      }
      __syncthreads();
      // phase 3: eight threads per row (kAsmRows x 8 = kAsmThreads) reduce
      // its blocks into the diagonal.  h^2 sum K is compensated (TwoSum):
      // the diagonal is ~h^2 k while the mass it must preserve is far
      // smaller.  Thread q of a row takes blocks q, q + 8, ... in column
      // order; the eight (sum, compensation) pairs are then merged by a
      // butterfly whose steps are commutative, so the order is fixed and
      // all eight threads hold the same bits.
      {
        const int32_t ri = g + int32_t(threadIdx.x) / kRowLanes;
        const int32_t q = int32_t(threadIdx.x) % kRowLanes;
        const bool live = ri < e;
        const int32_t i = r0 + ri;
        float Ks[6] = {0, 0, 0, 0, 0, 0}, Kc[6] = {0, 0, 0, 0, 0, 0}, Fs[3] = {0, 0, 0};
        int32_t dpos = -1;
        if (live) {
          const int32_t o0 = rows[ri].ob - gob, o1 = rows[ri + 1].ob - gob;
          for (int32_t o = o0 + q; o < o1; o += kRowLanes) {
            if (stc[o] == i) { dpos = o; continue; }
            const float* sv = &stv[kSymBlock * o];
#pragma unroll
            for (int t = 0; t < 6; ++t) {
              const float x = -sv[t];
              const float sum = Ks[t] + x;
              const float bp = sum - Ks[t];
              Kc[t] += (Ks[t] - (sum - bp)) + (x - bp);
              Ks[t] = sum;
            }
            Fs[0] += stf[3 * o]; Fs[1] += stf[3 * o + 1]; Fs[2] += stf[3 * o + 2];
          }
        }
#pragma unroll
        for (int off = kRowLanes / 2; off > 0; off >>= 1) {
#pragma unroll
          for (int t = 0; t < 6; ++t) {
            const float so = __shfl_xor_sync(0xffffffffu, Ks[t], off);
            const float co = __shfl_xor_sync(0xffffffffu, Kc[t], off);
            // TwoSum's error is the exact rounding error of the sum, so
            // both lanes of the pair get the same bits in either order
            const float sum = Ks[t] + so;
            const float bp = sum - Ks[t];
            const float err = (Ks[t] - (sum - bp)) + (so - bp);
            Kc[t] = (Kc[t] + co) + err;
            Ks[t] = sum;
          }
#pragma unroll
          for (int t = 0; t < 3; ++t) Fs[t] += __shfl_xor_sync(0xffffffffu, Fs[t], off);
          dpos = max(dpos, __shfl_xor_sync(0xffffffffu, dpos, off));
        }
        if (live && q == 0) {
          float D[kSymBlock];
          finish_row(a, i, Ks, Kc, Fs, D);
          if (dpos >= 0) {
#pragma unroll
            for (int t = 0; t < kSymBlock; ++t) stv[kSymBlock * dpos + t] = D[t];
          } else {
            atomicOr(a.status, ST_CAPACITY);  // diagonal missing: cannot happen
          }
        }
      }
      __syncthreads();
      // phase 4: coalesced write-out of values and column indices
      float* dst = a.vals + kSymBlock * int64_t(gob);
      for (int32_t f = threadIdx.x; f < kSymBlock * nblk; f += kAsmThreads) dst[f] = stv[f];
      for (int32_t o = threadIdx.x; o < nblk; o += kAsmThreads) a.colind[gob + o] = stc[o];
      __syncthreads();
    } else {
      // one row longer than the staging: stream it through in pieces
      const int32_t ri = g, i = r0 + ri;
      const RowInfo R = rows[ri];
      if (threadIdx.x < 9) acc[threadIdx.x] = 0.0;
      int32_t dpos_abs = -1;
      for (int32_t c0 = 0; c0 < nblk; c0 += kAsmCap) {
        const int32_t cn = min(kAsmCap, nblk - c0);
        __syncthreads();
        for (int32_t o = threadIdx.x; o < cn; o += kAsmThreads)
          compute_block(a, i, R, c0 + o, &stv[kSymBlock * o], &stf[3 * o], &stc[o], m_valid);
        __syncthreads();
        // fixed-order fp64 partial sums (one row: the cost is negligible):
        // thread t owns blocks t, t+T, ...
        double part[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
        for (int32_t o = threadIdx.x; o < cn; o += kAsmThreads) {
          if (stc[o] == i) { dpos_abs = gob + c0 + o; continue; }
          const float* s = &stv[kSymBlock * o];
          part[0] -= s[0]; part[1] -= s[1]; part[2] -= s[2];
          part[3] -= s[3]; part[4] -= s[4]; part[5] -= s[5];
          part[6] += stf[3 * o]; part[7] += stf[3 * o + 1]; part[8] += stf[3 * o + 2];
        }
#pragma unroll
        for (int q = 0; q < 9; ++q) {
          double vq = part[q];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) vq += __shfl_down_sync(0xffffffffu, vq, off);
          if ((threadIdx.x & 31) == 0) red[q][threadIdx.x >> 5] = vq;
        }
        __syncthreads();
        if (threadIdx.x < 9) {
          double s = 0.0;
          for (int w = 0; w < kAsmThreads / 32; ++w) s += red[threadIdx.x][w];
          acc[threadIdx.x] += s;
        }
        float* dst = a.vals + kSymBlock * (int64_t(gob) + c0);
        for (int32_t f = threadIdx.x; f < kSymBlock * cn; f += kAsmThreads) dst[f] = stv[f];
        for (int32_t o = threadIdx.x; o < cn; o += kAsmThreads) a.colind[gob + c0 + o] = stc[o];
      }
      __syncthreads();
      // the thread that saw the diagonal writes it (exactly one does)
      if (dpos_abs >= 0) {
        float Ks[6], Kc[6];
#pragma unroll
        for (int t = 0; t < 6; ++t) {   // exact split of the fp64 sum into hi + lo
          Ks[t] = float(acc[t]);
          Kc[t] = float(acc[t] - double(Ks[t]));
        }
        const float Fs[3] = {float(acc[6]), float(acc[7]), float(acc[8])};
        float D[kSymBlock];
        finish_row(a, i, Ks, Kc, Fs, D);
        float* dst = a.vals + kSymBlock * int64_t(dpos_abs);
#pragma unroll
        for (int t = 0; t < kSymBlock; ++t) dst[t] = D[t];
      }
      __syncthreads();
    }
    g = e;
  }
}

__global__ void pinv_expand(int32_t n, const float* __restrict__ p6, int64_t vs,
                            float* __restrict__ out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float p00 = p6[i], p01 = p6[vs + i], p02 = p6[2 * vs + i];
  const float p11 = p6[3 * vs + i], p12 = p6[4 * vs + i], p22 = p6[5 * vs + i];
  float* o = out + 9 * i;
  o[0] = p00; o[1] = p01; o[2] = p02;
  o[3] = p01; o[4] = p11; o[5] = p12;
  o[6] = p02; o[7] = p12; o[8] = p22;
}

// Packed symmetric blocks (a00 a01 a02 a11 a12 a22) to row-major 3x3.
__global__ void vals_expand(int64_t nnzb, const float* __restrict__ v6, float* __restrict__ out) {
  const int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= nnzb) return;
  const float* s = v6 + kSymBlock * b;
  const float a00 = s[0], a01 = s[1], a02 = s[2], a11 = s[3], a12 = s[4], a22 = s[5];
  float* o = out + 9 * b;
  o[0] = a00; o[1] = a01; o[2] = a02;
  o[3] = a01; o[4] = a11; o[5] = a12;
  o[6] = a02; o[7] = a12; o[8] = a22;
}

}  // namespace

int launch_vals_expand(Handle* h, float* out9, int64_t nnzb) {
  if (nnzb <= 0) return PCLOTH_OK;
  vals_expand<<<unsigned((nnzb + 255) / 256), 256, 0, h->stream>>>(nnzb, h->vals, out9);
  h->launches += 1;
  return check_launch(h, "vals expand");
}

int launch_pinv_expand(Handle* h, float* out9) {
  pinv_expand<<<(h->n + 255) / 256, 256, 0, h->stream>>>(h->n, h->pinv6, h->vstride, out9);
  h->launches += 1;
  return check_launch(h, "pinv expand");
}

int assemble_system(Handle* h, const float* x, const float* v,
                    const pcloth_springs* contacts, float dt) {
  const int32_t nc = contacts ? contacts->n : 0;
  const int B = h->key_bits;
  const int32_t ntiles = (h->n + kAsmRows - 1) / kAsmRows;
  cudaStream_t s = h->stream;
  h->bell_valid = false;   // the pattern changes below
  if (h->prof.on) cudaEventRecord(h->ev[0], s);
  int rc = PCLOTH_OK;
  AsmArgs a{};
  a.has_contacts = nc > 0;
  if (nc > 0) {
    const int32_t m = 2 * nc;
    contact_keys<<<(nc + 255) / 256, 256, 0, s>>>(nc, h->n, B, contacts->i, contacts->j,
                                                   contacts->k, contacts->rest, h->ckey[0],
                                                   h->cval[0], h->d_status);
    cudaMemsetAsync(h->counters, 0, 4 * sizeof(int32_t), s);
    h->launches += 1;
    int cur = radix_sort_pairs(h, h->ckey, h->cval, m, 2 * B);
    if (cur < 0) return cur;
    contact_classify<<<(m + 255) / 256, 256, 0, s>>>(m, B, h->ckey[cur], h->rowptr_s,
                                                     h->colind_s, h->flags, h->counters);
    h->launches += 1;
    rc = scan_exclusive(h, h->flags, m, h->counters);
    if (rc != PCLOTH_OK) return rc;
    contact_compact<<<(m + 255) / 256, 256, 0, s>>>(m, h->ckey[cur], h->flags, h->counters,
                                                    h->newkey, h->newfirst);
    h->launches += 1;
    a.skey = h->ckey[cur];
    a.sval = h->cval[cur];
    a.ck = contacts->k;
    a.cr = contacts->rest;
  }
  tile_bounds<<<(ntiles + 1 + 255) / 256, 256, 0, s>>>(ntiles, h->n, B, nc > 0, h->newkey,
                                                        a.skey, h->counters, h->tile_nb,
                                                        h->tile_eb);
  h->launches += 1;
  a.n = h->n;
  a.B = B;
  a.dt = dt;
  a.h2 = dt * dt;
  a.gx = h->gravity[0];
  a.gy = h->gravity[1];
  a.gz = h->gravity[2];
  a.x = x;
  a.v = v;
  a.mass = h->mass;
  a.rowptr_s = h->rowptr_s;
  a.colind_s = h->colind_s;
  a.sblk_ptr = h->sblk_ptr;
  a.sentry = h->sentry;
  a.newkey = h->newkey;
  a.newfirst = h->newfirst;
  a.tile_nb = h->tile_nb;
  a.tile_eb = h->tile_eb;
  a.counters = h->counters;
  a.rowptr = h->rowptr;
  a.colind = h->colind;
  a.vals = h->vals;
  a.rhs = h->rhs;
  a.pinv6 = h->pinv6;
  a.vs = h->vstride;
  a.status = h->d_status;
  assemble_rows<<<ntiles, kAsmThreads, 0, s>>>(a);
  h->launches += 1;
  if (h->prof.on) {
    cudaEventRecord(h->ev[1], s);
    cudaEventSynchronize(h->ev[1]);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, h->ev[0], h->ev[1]);
    h->prof.assemble_ms += ms;
    h->prof.assemble_calls += 1;
  }
  return check_launch(h, "assembly");
}

}  // namespace pcloth_impl
