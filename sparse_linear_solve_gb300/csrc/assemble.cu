// Per-step assembly of A dv = b (P-Cloth, arXiv 2008.00409: Sec. 2.5
// Eq. (3) for the system, Sec. 3.2 for the assembly elements, Sec. 3.2.2 for
// the sparse matrix filling).
//
// The page fills an index table with atomics, sorts and compacts each row
// with one thread per row, then fills values with atomics.  Here the spring
// pattern is built once (pcloth_create) and each step's contacts go through
// the same steps, made deterministic:
//
//   contact_count     entries per row (a contact (i, j) is an entry of row i
//                     with column j and one of row j with column i), atomics
//   scan              first entry of each row
//   contact_scatter   the entries into their rows (any order within a row)
//   row_classify      one thread per row sorts its entries by (column,
//                     contact id) -- so equal blocks sum in input order --
//                     and lists the columns that are not spring blocks: the
//                     row's new blocks
//   scan              new blocks before each row
//   assemble_rows     two lanes per row: the row's blocks in column order
//                     (spring and new blocks merged), every element of every
//                     off-diagonal block evaluated and written, the row's
//                     compensated sum into its diagonal block, b = h f and
//                     the block-Jacobi inverse.  No shared memory, no CTA
//                     barrier: rows are independent.
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

#ifndef PCLOTH_ASM_LANES
#define PCLOTH_ASM_LANES 2
#endif
constexpr int kRowLanes = PCLOTH_ASM_LANES;   // lanes of a warp that assemble one row
static_assert(kAsmThreads % 32 == 0 && 32 % kRowLanes == 0, "whole rows per warp");

struct AsmArgs {
  int32_t n;
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
  const int32_t* ebefore;   // [n+1] first contact entry of each row
  const int32_t* nbefore;   // [n+1] new blocks before each row
  const uint64_t* centry;   // entries, per row sorted by (column << 32 | contact id)
  const int32_t* newcol;    // a row's new columns, at the row's first entry index
  const float* ck;
  const float* cr;
  int32_t* rowptr;
  int32_t* colind;
  float* vals;        // packed symmetric blocks, six floats each
  float* rhs;
  float* pinv6;      // [6][vs]
  int64_t vs;
  uint32_t* status;
};

// The one validity test of a contact, shared by the counting and the
// scattering pass so that both skip the same contacts.
__device__ __forceinline__ bool contact_ok(int32_t i, int32_t j, int32_t n) {
  return i >= 0 && i < n && j >= 0 && j < n && i != j;
}

__global__ void contact_count(int32_t nc, int32_t n, const int32_t* __restrict__ ci,
                              const int32_t* __restrict__ cj, const float* __restrict__ ck,
                              const float* __restrict__ cr, int32_t* __restrict__ rowcnt,
                              uint32_t* status) {
  const int32_t c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= nc) return;
  const int32_t i = ci[c], j = cj[c];
  if (!isfinite(ck[c]) || !isfinite(cr[c])) atomicOr(status, ST_NONFINITE);
  if (!contact_ok(i, j, n)) {
    atomicOr(status, ST_BAD_INDEX);
    return;
  }
  atomicAdd(&rowcnt[i], 1);
  atomicAdd(&rowcnt[j], 1);
}

__global__ void contact_scatter(int32_t nc, int32_t n, const int32_t* __restrict__ ci,
                                const int32_t* __restrict__ cj,
                                const int32_t* __restrict__ ebefore, int32_t* __restrict__ fill,
                                uint64_t* __restrict__ centry) {
  const int32_t c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= nc) return;
  const int32_t i = ci[c], j = cj[c];
  if (!contact_ok(i, j, n)) return;
  const int32_t pi = ebefore[i] + atomicAdd(&fill[i], 1);
  const int32_t pj = ebefore[j] + atomicAdd(&fill[j], 1);
  centry[pi] = (uint64_t(uint32_t(j)) << 32) | uint32_t(c);
  centry[pj] = (uint64_t(uint32_t(i)) << 32) | uint32_t(c);
}

// Sorts a row's few entries in place: insertion sort, or heapsort for long
// rows (a vertex in contact with hundreds of others).
__device__ __forceinline__ void sort_entries(uint64_t* a, int32_t m) {
  if (m <= 32) {
    for (int32_t t = 1; t < m; ++t) {
      const uint64_t key = a[t];
      int32_t u = t - 1;
      while (u >= 0 && a[u] > key) {
        a[u + 1] = a[u];
        --u;
      }
      a[u + 1] = key;
    }
    return;
  }
  auto sift = [&](int32_t root, int32_t end) {   // max-heap on [0, end)
    while (true) {
      int32_t child = 2 * root + 1;
      if (child >= end) return;
      if (child + 1 < end && a[child + 1] > a[child]) ++child;
      if (a[root] >= a[child]) return;
      const uint64_t t = a[root];
      a[root] = a[child];
      a[child] = t;
      root = child;
    }
  };
  for (int32_t r = m / 2 - 1; r >= 0; --r) sift(r, m);
  for (int32_t end = m - 1; end > 0; --end) {
    const uint64_t t = a[0];
    a[0] = a[end];
    a[end] = t;
    sift(0, end);
  }
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

// One thread per row (thread n writes newcnt[n] = 0, the scan's total slot).
__global__ void row_classify(int32_t n, const int32_t* __restrict__ ebefore,
                             uint64_t* __restrict__ centry, const int32_t* __restrict__ rowptr_s,
                             const int32_t* __restrict__ colind_s, int32_t* __restrict__ newcol,
                             int32_t* __restrict__ newcnt) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i > n) return;
  if (i == n) {
    newcnt[n] = 0;
    return;
  }
  const int32_t e0 = ebefore[i], e1 = ebefore[i + 1];
  int32_t k = 0;
  if (e1 > e0) {
    sort_entries(centry + e0, e1 - e0);
    const int32_t s0 = rowptr_s[i], s1 = rowptr_s[i + 1];
    int32_t last = -1;
    for (int32_t t = e0; t < e1; ++t) {
      const int32_t col = int32_t(centry[t] >> 32);
      if (col == last) continue;
      last = col;
      if (!static_has(colind_s, s0, s1, col)) {
        newcol[e0 + k] = col;
        ++k;
      }
    }
  }
  newcnt[i] = k;
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
// the edges e and -e give the same bits.  The squares are rounded with
// __fmul_rn, which the compiler never fuses into a multiply-add: fused into
// the TwoSum that follows, a square would enter that sum unrounded and its
// error term would no longer be exact.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& t) {
  s = a + b;
  const float bp = s - a;
  t = (a - (s - bp)) + (b - bp);
}

__device__ __forceinline__ float excess_sq(float3 hi, float3 lo, float L0) {
  const float px = __fmul_rn(hi.x, hi.x), py = __fmul_rn(hi.y, hi.y);
  const float pz = __fmul_rn(hi.z, hi.z), pl = -__fmul_rn(L0, L0);
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

// The same for an edge held in one fp32 vector (no lo part).
__device__ __forceinline__ float excess_sq(float3 v, float L0) {
  const float px = __fmul_rn(v.x, v.x), py = __fmul_rn(v.y, v.y);
  const float pz = __fmul_rn(v.z, v.z), pl = -__fmul_rn(L0, L0);
  const float rx = fmaf(v.x, v.x, -px), ry = fmaf(v.y, v.y, -py);
  const float rz = fmaf(v.z, v.z, -pz), rl = fmaf(-L0, L0, -pl);
  float s, t1, t2, t3;
  two_sum(px, py, s, t1);
  two_sum(s, pz, s, t2);
  two_sum(s, pl, s, t3);
  return s + (((t1 + t2) + t3) + (((rx + ry) + rz) + rl));
}

// Scaled stiffness block K' = -h^2 K (6 unique entries of the symmetric
// block) and force F of one element seen from vertex i: K at x, force at
// x~ = x + h v.  e = x_j - x_i (exact, see Edge), its length and the
// advanced edge are shared by all elements of a block (BlockEdge, formed
// once per block); each element costs two divisions.  The square roots and
// divisions are the IEEE ones (correctly rounded): rsqrtf and __fdividef,
// good to a few units in the last place, made the assembly 4% faster and
// are left out so that every operation of the element terms is IEEE.
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

// What the elements of one block share: the edge at x_t (exact, with
// l2 = |e|^2, l = |e| and 1 / l2) and the advanced edge at x~ with its length.
struct BlockEdge {
  Edge e;
  float l2, l, inv_l2;
  float3 adv;
  float lt;
};

__device__ __forceinline__ BlockEdge block_edge(float3 xi, float3 xj, float3 vi, float3 vj,
                                                float dt) {
  BlockEdge b;
  b.e = edge_of(xi, xj);
  const float3 h = b.e.hi, o = b.e.lo;
  b.l2 = fmaf(h.x, h.x, fmaf(h.y, h.y, h.z * h.z)) +
         2.0f * fmaf(h.x, o.x, fmaf(h.y, o.y, h.z * o.z));
  b.l = sqrtf(b.l2);
  b.inv_l2 = 1.0f / b.l2;
  const float3 w = make_float3(vj.x - vi.x, vj.y - vi.y, vj.z - vi.z);
  b.adv = make_float3(fmaf(dt, w.x, h.x) + o.x, fmaf(dt, w.y, h.y) + o.y,
                      fmaf(dt, w.z, h.z) + o.z);
  b.lt = sqrtf(b.adv.x * b.adv.x + b.adv.y * b.adv.y + b.adv.z * b.adv.z);
  return b;
}

__device__ __forceinline__ void element_terms(const BlockEdge& b, float h2, float k, float L0,
                                              float (&K)[6], float (&F)[3]) {
  const float3 h = b.e.hi, o = b.e.lo;
  const float l = b.l;
  // max(0, 1 - L0/l) = max(0, (l - L0) / l), with l - L0 = (|e|^2 - L0^2) / (l + L0)
  const float tension = fmaxf(0.0f, excess_sq(h, o, L0) / ((l + L0) * l));
  const float a = k * tension;
  const float c = k - a;
  const float A = -h2 * a;
  const float S = (-h2 * c) * b.inv_l2;
  K[0] += scaled_entry(S, h.x, o.x, h.x, o.x) + A;
  K[1] += scaled_entry(S, h.x, o.x, h.y, o.y);
  K[2] += scaled_entry(S, h.x, o.x, h.z, o.z);
  K[3] += scaled_entry(S, h.y, o.y, h.y, o.y) + A;
  K[4] += scaled_entry(S, h.y, o.y, h.z, o.z);
  K[5] += scaled_entry(S, h.z, o.z, h.z, o.z) + A;
  // force at the advanced positions: k (l~ - L0) / l~ along the advanced edge
  const float s = k * excess_sq(b.adv, L0) / ((b.lt + L0) * b.lt);
  F[0] += s * b.adv.x;
  F[1] += s * b.adv.y;
  F[2] += s * b.adv.z;
}

__device__ __forceinline__ float3 ld3(const float* p, int64_t i) {
  return make_float3(p[3 * i], p[3 * i + 1], p[3 * i + 2]);
}

// Writes a packed block (six floats from float offset 6 q) with one 16-byte
// and one 8-byte store, without a branch: 24 q bytes is 16-byte aligned for
// even q, so the 16-byte word holds entries 0-3 there and 2-5 for odd q.
// Six 4-byte stores from the lanes of a warp, whose blocks lie in 16
// different rows, reach L2 as six partial-sector writes per block.
__device__ __forceinline__ void st_block(float* vals, int64_t q, const float (&K)[6]) {
  float* d = vals + kSymBlock * q;
  const bool odd = (q & 1) != 0;
  const float4 w4 =
      odd ? make_float4(K[2], K[3], K[4], K[5]) : make_float4(K[0], K[1], K[2], K[3]);
  const float2 w2 = odd ? make_float2(K[0], K[1]) : make_float2(K[4], K[5]);
  *reinterpret_cast<float4*>(d + (odd ? 2 : 0)) = w4;
  *reinterpret_cast<float2*>(d + (odd ? 0 : 4)) = w2;
}

// Merge position p of two sorted disjoint column lists S (spring blocks) and
// T (new blocks): returns the number of S entries before position p.
__device__ __forceinline__ int32_t merge_split(const int32_t* __restrict__ S, int32_t nS,
                                               const int32_t* __restrict__ T, int32_t nT,
                                               int32_t p) {
  int32_t lo = max(0, p - nT), hi = min(p, nS);
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (S[mid - 1] < T[p - mid]) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Diagonal block (written to the row's diagonal slot dpos), right-hand side
// and block-Jacobi inverse of row i from the row's compensated sum
// -sum_j A_ij = h^2 sum K = Ks + Kc over its off-diagonal blocks as stored
// (6 unique entries, Kc the TwoSum compensation) and its force sum.  The mass is added to the small
// compensation term first, so the diagonal is rounded once from the exact
// total: adding m after rounding the large sum would round the same m to the
// same ulp grid in every row of a binade -- a coherent shift of the mass by
// ~0.1%, which the soft modes of the system amplify.
__device__ __forceinline__ void finish_row(const AsmArgs& a, int32_t i, int64_t dpos,
                                           const float (&Ks)[6], const float (&Kc)[6],
                                           const float (&Fs)[3]) {
  float D[kSymBlock];
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
  st_block(a.vals, dpos, D);
  bool ok = finite3(b0, b1, b2) && isfinite(det) && det > 0.0f;
#pragma unroll
  for (int t = 0; t < kSymBlock; ++t) ok = ok && isfinite(D[t]);
  if (!ok) atomicOr(a.status, ST_NONFINITE);
}

// kRowLanes lanes per row.  The diagonal's position dpos in the row is
// found first (the spring columns below i plus the new columns below i);
// lane l then takes the row's off-diagonal blocks l, l + kRowLanes, ... in
// column order (block k sits at slot k + (k >= dpos)): it finds the block's
// column by walking the spring and new columns with two cursors, evaluates
// every element of the block -- the spring entries of a spring block, then
// the block's contacts in input order, found by a third cursor -- writes
// the block's column and packed value, and adds the negated value and the
// block's force into its compensated (TwoSum) partial sums.  A butterfly whose steps are
// commutative merges the lanes' partials (all lanes end with the same
// bits), and lane 0 writes the diagonal's column and forms the diagonal
// block, b and the block-Jacobi inverse.  Rows are independent: no shared
// memory and no CTA barrier.
//
// Two lanes per row at three CTAs per SM (80 registers) were the fastest of
// a sweep on the 1.65M-triangle cloth (whole assembly per step): 16 lanes
// 0.78 ms, 8 lanes 0.58 ms, 4 lanes 0.51 ms (four CTAs per SM), 2 lanes
// 0.47 ms, 1 lane 0.62 ms; four or more CTAs per SM spill and lose.  Fewer
// lanes cut the butterfly's and the row finish's share of the
// instructions; one lane per row leaves each row's loads in a serial chain.
// On that cloth the kernel then took 380 us (ncu); the block stores as one
// 16- and one 8-byte word and the diagonal taken out of the lanes' loop cut
// it most.  Contacts cost the most per element: without them the assembly
// takes 0.20 ms.  One element loop for springs and contacts, and cursors in
// place of a merge-path search per block and a search of the contact run,
// brought the whole assembly from 0.45 to 0.305 ms per step.
#ifndef PCLOTH_ASM_CTAS
#define PCLOTH_ASM_CTAS 3
#endif
__global__ void __launch_bounds__(kAsmThreads, PCLOTH_ASM_CTAS)
assemble_rows(AsmArgs a) {
  const int32_t lane = int32_t(threadIdx.x) % kRowLanes;
  const int64_t row = (int64_t(blockIdx.x) * kAsmThreads + threadIdx.x) / kRowLanes;
  const bool live = row < a.n;
  // lanes past the last row shadow it (same loads, no writes), so that every
  // lane of the warp takes part in the shuffles
  const int32_t i = live ? int32_t(row) : a.n - 1;
  const int32_t sb = a.rowptr_s[i], se = a.rowptr_s[i + 1];
  int32_t nb = 0, ne = 0, eb = 0, ee = 0;
  if (a.has_contacts) {
    nb = a.nbefore[i];
    ne = a.nbefore[i + 1];
    eb = a.ebefore[i];
    ee = a.ebefore[i + 1];
  }
  const int32_t ob = sb + nb;   // the row's first block in the full pattern
  const int32_t nS = se - sb, nT = ne - nb, len = nS + nT;
  if (live && lane == 0) {
    a.rowptr[i] = ob;
    if (i == a.n - 1) a.rowptr[a.n] = se + ne;
  }
  const float3 xi = ld3(a.x, i), vi = ld3(a.v, i);
  float Ks[6] = {0, 0, 0, 0, 0, 0}, Kc[6] = {0, 0, 0, 0, 0, 0}, Fs[3] = {0, 0, 0};
  int32_t dpos;   // the diagonal's position in the row
  {
    int32_t lo = sb, hi = se;
    while (lo < hi) {
      const int32_t mid = (lo + hi) >> 1;
      if (a.colind_s[mid] < i) lo = mid + 1; else hi = mid;
    }
    dpos = lo - sb;
    for (int32_t t = 0; t < nT; ++t) dpos += a.newcol[eb + t] < i;
  }
  // Cursors that walk the row with the lane: sc into the spring columns S
  // and tn into the new columns T (heads hs and ht, kEnd past the end), and
  // tc into the row's sorted contact entries (head hen).  The lane's first
  // block is found by a merge-path search, each later one by stepping the
  // cursors over the other lane's blocks.
  const int32_t* S = a.colind_s + sb;
  const int32_t* T = a.newcol + eb;
  constexpr int32_t kEnd = INT32_MAX;
  int32_t sc, tn, hs, ht;
  {
    const int32_t p0 = lane + (lane >= dpos);
    sc = merge_split(S, nS, T, nT, p0);
    tn = p0 - sc;
    hs = sc < nS ? S[sc] : kEnd;
    ht = tn < nT ? T[tn] : kEnd;
  }
  int32_t tc = eb;
  uint64_t hen = tc < ee ? a.centry[tc] : ~uint64_t(0);
  for (int32_t k = lane; k < len - 1; k += kRowLanes) {
    const int32_t p = k + (k >= dpos);
    const bool from_s = hs < ht;   // the two lists are disjoint
    const int32_t col = from_s ? hs : ht;
    const int32_t sslot = from_s ? sb + sc : -1;
    if (live) a.colind[ob + p] = col;
    float K[6] = {0, 0, 0, 0, 0, 0}, F[3] = {0, 0, 0};
    const float3 xj = ld3(a.x, col), vj = ld3(a.v, col);
    const BlockEdge be = block_edge(xi, xj, vi, vj, a.dt);
    // The block's elements in one loop, so that the lanes of a warp
    // evaluate springs and contacts in the same passes: the spring entries,
    // then the block's contacts, the run of the row's sorted entries with
    // this column (the contact cursor first passes the entries of the other
    // lane's columns).
    int32_t e = 0, e1 = 0;
    if (sslot >= 0) {
      e = a.sblk_ptr[sslot];
      e1 = a.sblk_ptr[sslot + 1];
    }
    const uint64_t col_key = uint64_t(uint32_t(col)) << 32;
    while (hen < col_key) {
      ++tc;
      hen = tc < ee ? a.centry[tc] : ~uint64_t(0);
    }
    while (true) {
      float kk, L0;
      if (e < e1) {
        const float2 kl = a.sentry[e++];
        kk = kl.x;
        L0 = kl.y;
      } else {
        if ((hen >> 32) != uint64_t(uint32_t(col))) break;
        const int32_t c = int32_t(uint32_t(hen));
        kk = a.ck[c];
        L0 = a.cr[c];
        ++tc;
        hen = tc < ee ? a.centry[tc] : ~uint64_t(0);
      }
      element_terms(be, a.h2, kk, L0, K, F);
    }
    if (live) {
      st_block(a.vals, int64_t(ob) + p, K);
    }
    // the diagonal takes -(the block as stored), so that the rows of A sum
    // to M up to the compensated sums' own error
#pragma unroll
    for (int t = 0; t < 6; ++t) add_comp(Ks[t], Kc[t], -K[t]);
    Fs[0] += F[0];
    Fs[1] += F[1];
    Fs[2] += F[2];
    // step the column cursors to the lane's next block (d slots on); with no
    // new column left the spring cursor jumps
    const int32_t kn = k + kRowLanes;
    int32_t d = kn + (kn >= dpos) - p;
    while (d > 0) {
      if (ht == kEnd) {
        sc += d;
        break;
      }
      if (hs < ht) {
        ++sc;
        hs = sc < nS ? S[sc] : kEnd;
      } else {
        ++tn;
        ht = tn < nT ? T[tn] : kEnd;
      }
      --d;
    }
    hs = sc < nS ? S[sc] : kEnd;
  }
  // merge the lanes' partials: TwoSum's error is the exact rounding error of
  // the sum, so both lanes of a pair get the same bits in either order
#pragma unroll
  for (int off = kRowLanes / 2; off > 0; off >>= 1) {
#pragma unroll
    for (int t = 0; t < 6; ++t) {
      const float so = __shfl_xor_sync(0xffffffffu, Ks[t], off);
      const float co = __shfl_xor_sync(0xffffffffu, Kc[t], off);
      const float sum = Ks[t] + so;
      const float bp = sum - Ks[t];
      const float err = (Ks[t] - (sum - bp)) + (so - bp);
      Kc[t] = (Kc[t] + co) + err;
      Ks[t] = sum;
    }
#pragma unroll
    for (int t = 0; t < 3; ++t) Fs[t] += __shfl_xor_sync(0xffffffffu, Fs[t], off);
  }
  if (live && lane == 0) {
    a.colind[ob + dpos] = i;
    finish_row(a, i, int64_t(ob) + dpos, Ks, Kc, Fs);
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
  const int32_t n = h->n;
  cudaStream_t s = h->stream;
  h->bell_valid = false;   // the pattern changes below
  if (h->prof.on) cudaEventRecord(h->ev[0], s);
  AsmArgs a{};
  a.has_contacts = nc > 0;
  if (nc > 0) {
    int32_t* rowcnt = h->rowcnt;          // [n+1]: counts, then first entry per row
    int32_t* fill = h->rowcnt + (n + 1);  // [n+1]: scatter cursors
    uint64_t* centry = h->centry;
    cudaError_t e = cudaMemsetAsync(h->rowcnt, 0, 2 * (size_t(n) + 1) * sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_fail(h, e, "contact counts reset");
    const int cgrid = (nc + 255) / 256, rgrid = (n + 1 + 255) / 256;
    contact_count<<<cgrid, 256, 0, s>>>(nc, n, contacts->i, contacts->j, contacts->k,
                                        contacts->rest, rowcnt, h->d_status);
    h->launches += 1;
    int rc = scan_exclusive(h, rowcnt, n + 1, h->counters + 1);
    if (rc != PCLOTH_OK) return rc;
    contact_scatter<<<cgrid, 256, 0, s>>>(nc, n, contacts->i, contacts->j, rowcnt, fill,
                                          centry);
    row_classify<<<rgrid, 256, 0, s>>>(n, rowcnt, centry, h->rowptr_s, h->colind_s, h->newcol,
                                       h->newcnt);
    h->launches += 2;
    rc = scan_exclusive(h, h->newcnt, n + 1, h->counters);
    if (rc != PCLOTH_OK) return rc;
    a.ebefore = rowcnt;
    a.nbefore = h->newcnt;
    a.centry = centry;
    a.newcol = h->newcol;
    a.ck = contacts->k;
    a.cr = contacts->rest;
  }
  a.n = n;
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
  a.rowptr = h->rowptr;
  a.colind = h->colind;
  a.vals = h->vals;
  a.rhs = h->rhs;
  a.pinv6 = h->pinv6;
  a.vs = h->vstride;
  a.status = h->d_status;
  const int64_t rows_per_cta = kAsmThreads / kRowLanes;
  assemble_rows<<<unsigned((n + rows_per_cta - 1) / rows_per_cta), kAsmThreads, 0, s>>>(a);
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
