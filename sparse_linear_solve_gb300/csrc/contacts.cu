// Vertex-vertex proximity contacts by spatial hashing (P-Cloth, arXiv
// 2008.00409, Sec. 4.2: a spatial-hash table built on the fly every step,
// then proximity tests; Sec. 4.3: proximities enter the implicit integrator
// as forces).  Restricted to pairs of vertices: every pair i < j closer than
// a radius r that is not a spring becomes a contact (a spring of stiffness
// k_c and rest length r), listed in (i, j) order.
//
//   hash_count    each vertex to its cell of edge 2r (1 + 2^-7); the cell to
//                 a bucket of a table of T >= 2n buckets by the hash of
//                 Teschner et al. (2003, "Optimized Spatial Hashing for
//                 Collision Detection of Deformable Objects"), counted with
//                 an atomic that also gives the vertex its place in the bucket
//   scan          the buckets' first slots
//   hash_fill     each vertex's position and index into its bucket's slot
//   hash_ranges   each bucket's slot range as one 8-byte word
//   pair_pass     per vertex i, twice: the 8 cells that can hold a partner
//                 -- per axis its own cell and the next one on the side of
//                 the half of the cell that holds the vertex, as a partner
//                 is less than half a cell away.  The enlargement 1 + 2^-7
//                 keeps that true despite the rounding of x / edge, for
//                 coordinates up to 2^14 cells from the origin (65 m at
//                 r = 2 mm).  A candidate j > i counts if it lies in the
//                 searched cell (buckets are shared by colliding cells),
//                 passes the exact float32 test ((dx dx + dy dy) + dz dz <
//                 r r, each operation rounded) and is no spring (a binary
//                 search in the static pattern).  The first pass counts, a scan gives
//                 every vertex its first output slot, and the second pass
//                 writes the partners and sorts them, so the list comes out
//                 in (i, j) order whatever the order inside the buckets.
//
// The distance test decides an integer outcome, so it is written with
// explicitly rounded operations (no fused multiply-add) to be reproducible
// by a plain float32 restatement.

#include <algorithm>

#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

constexpr int32_t kCellLimit = 1 << 20;   // cells clamped to [-2^20 + 2, 2^20 - 3]

__device__ __forceinline__ int32_t cell_of(float v, float inv_edge) {
  const float c = floorf(v * inv_edge);
  return int32_t(fminf(fmaxf(c, float(-kCellLimit + 2)), float(kCellLimit - 3)));
}

// Teschner et al.'s spatial hash: the cell's coordinates times three large
// primes, combined by exclusive or, modulo the table size (a power of two).
__device__ __forceinline__ uint32_t cell_hash(int32_t cx, int32_t cy, int32_t cz, uint32_t mask) {
  return ((uint32_t(cx) * 73856093u) ^ (uint32_t(cy) * 19349663u) ^ (uint32_t(cz) * 83492791u)) &
         mask;
}

__global__ void hash_count(int32_t n, const float* __restrict__ x, float inv_edge, uint32_t mask,
                           int32_t* __restrict__ count, int2* __restrict__ where,
                           uint32_t* status) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float px = x[3 * i], py = x[3 * i + 1], pz = x[3 * i + 2];
  if (!finite3(px, py, pz)) atomicOr(status, ST_NONFINITE);
  const uint32_t b =
      cell_hash(cell_of(px, inv_edge), cell_of(py, inv_edge), cell_of(pz, inv_edge), mask);
  where[i] = make_int2(int32_t(b), atomicAdd(&count[b], 1));
}

__global__ void hash_fill(int32_t n, const float* __restrict__ x, const int2* __restrict__ where,
                          const int32_t* __restrict__ first, float4* __restrict__ slot) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int2 w = where[i];
  slot[first[w.x] + w.y] = make_float4(x[3 * i], x[3 * i + 1], x[3 * i + 2], __int_as_float(int32_t(i)));
}

// Each bucket's slot range as one 8-byte word, so that a lookup is one load.
__global__ void hash_ranges(int32_t nb, const int32_t* __restrict__ first,
                            int2* __restrict__ range) {
  const int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b < nb) range[b] = make_int2(first[b], first[b + 1]);
}

__device__ __forceinline__ bool is_spring(const int32_t* __restrict__ rowptr_s,
                                          const int32_t* __restrict__ colind_s, int32_t i,
                                          int32_t j) {
  int32_t lo = rowptr_s[i], hi = rowptr_s[i + 1];
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    const int32_t c = colind_s[mid];
    if (c == j) return true;
    if (c < j) lo = mid + 1; else hi = mid;
  }
  return false;
}

// Sorts a vertex's few partners in place: insertion sort, or heapsort for
// many (a vertex inside a dense cluster).
__device__ void sort_partners(int32_t* a, int32_t m) {
  if (m <= 32) {
    for (int32_t t = 1; t < m; ++t) {
      const int32_t key = a[t];
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
      const int32_t t = a[root];
      a[root] = a[child];
      a[child] = t;
      root = child;
    }
  };
  for (int32_t r = m / 2 - 1; r >= 0; --r) sift(r, m);
  for (int32_t end = m - 1; end > 0; --end) {
    const int32_t t = a[0];
    a[0] = a[end];
    a[end] = t;
    sift(0, end);
  }
}

struct PairArgs {
  int32_t n;
  float r2, inv_edge;
  uint32_t mask;
  const float* x;
  const int2* range;       // [T] first and end slot of each bucket
  const float4* slot;      // [n] (x, y, z, index) in bucket order
  const int32_t* rowptr_s;
  const int32_t* colind_s;
  int32_t* count;          // count pass: partners of each vertex
  unsigned long long* total;  // count pass: all partners, in 64 bits
  const int32_t* out_first;  // write pass: each vertex's first output slot
  int32_t* oi;
  int32_t* oj;
  float* ok;
  float* orest;
  float k, rest;
};

template <bool kWrite>
__global__ void pair_pass(PairArgs a) {
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int32_t i = int32_t(t);
  int32_t c = 0;
  int32_t base = 0;
  if (t < a.n) {
    const float px = a.x[3 * t], py = a.x[3 * t + 1], pz = a.x[3 * t + 2];
    const int32_t cx = cell_of(px, a.inv_edge), cy = cell_of(py, a.inv_edge);
    const int32_t cz = cell_of(pz, a.inv_edge);
    // cells of edge 2r: the partners lie in this cell or the next one on
    // the side of the half of the cell that holds the vertex, per axis
    const float tx = px * a.inv_edge, ty = py * a.inv_edge, tz = pz * a.inv_edge;
    const int sx = (tx - floorf(tx) >= 0.5f) ? 1 : -1;
    const int sy = (ty - floorf(ty) >= 0.5f) ? 1 : -1;
    const int sz = (tz - floorf(tz) >= 0.5f) ? 1 : -1;
    if (kWrite) base = a.out_first[i];
    for (int ox = 0; ox <= 1; ++ox) {
      for (int oy = 0; oy <= 1; ++oy) {
        for (int oz = 0; oz <= 1; ++oz) {
          const int32_t nx = cx + ox * sx, ny = cy + oy * sy, nz = cz + oz * sz;
          const uint32_t b = cell_hash(nx, ny, nz, a.mask);
          const int2 rg = a.range[b];
          for (int32_t u = rg.x; u < rg.y; ++u) {
            const float4 s = a.slot[u];
            const int32_t j = __float_as_int(s.w);
            if (j <= i) continue;
            if (cell_of(s.x, a.inv_edge) != nx || cell_of(s.y, a.inv_edge) != ny ||
                cell_of(s.z, a.inv_edge) != nz)
              continue;   // another cell with the same hash
            const float dx = __fsub_rn(s.x, px);
            const float dy = __fsub_rn(s.y, py);
            const float dz = __fsub_rn(s.z, pz);
            const float d2 = __fadd_rn(__fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy)),
                                       __fmul_rn(dz, dz));
            if (!(d2 < a.r2)) continue;
            if (is_spring(a.rowptr_s, a.colind_s, i, j)) continue;
            if (kWrite) a.oj[base + c] = j;
            ++c;
          }
        }
      }
    }
  }
  if (kWrite) {
    if (t < a.n) {
      sort_partners(a.oj + base, c);
      for (int32_t q = 0; q < c; ++q) {
        a.oi[base + q] = i;
        a.ok[base + q] = a.k;
        a.orest[base + q] = a.rest;
      }
    }
    return;
  }
  if (t < a.n) {
    a.count[i] = c;
    if (i == a.n - 1) a.count[a.n] = 0;   // the scan's total slot
  }
  // The total in 64 bits (a warp's sum, then one atomic per warp): past 2^31
  // pairs (a collapsed cloud) the int32 scan of the counts wraps, and the
  // capacity test must still see the true number.  Every thread of the block
  // gets here, so the warp is whole.
  unsigned long long w = static_cast<unsigned long long>(c);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) w += __shfl_down_sync(0xffffffffu, w, o);
  if ((threadIdx.x & 31) == 0 && w != 0) atomicAdd(a.total, w);
}

}  // namespace

int find_contacts(Handle* h, const float* x, float radius, float stiffness,
                  pcloth_springs* out, int32_t capacity, int32_t* found) {
  cudaStream_t s = h->stream;
  const int32_t n = h->n;
  const float edge = 2.0f * radius * (1.0f + 1.0f / 128.0f);
  const float inv_edge = 1.0f / edge;
  const float r2 = radius * radius;   // float32, as the test compares
  const int32_t nb = int32_t(h->hash_mask) + 1;   // buckets
  const int grid = (n + 255) / 256;
  // the hash table: bucket counts, their scan, the vertices in bucket order
  cudaError_t e = cudaMemsetAsync(h->hash_first, 0, (size_t(nb) + 1) * sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "hash table reset");
  hash_count<<<grid, 256, 0, s>>>(n, x, inv_edge, h->hash_mask, h->hash_first, h->hash_where,
                                  h->d_status);
  h->launches += 1;
  int rc = check_launch(h, "hash count");
  if (rc != PCLOTH_OK) return rc;
  rc = scan_exclusive(h, h->hash_first, nb + 1, h->counters + 2);
  if (rc != PCLOTH_OK) return rc;
  hash_fill<<<grid, 256, 0, s>>>(n, x, h->hash_where, h->hash_first, h->hash_slot);
  hash_ranges<<<(nb + 255) / 256, 256, 0, s>>>(nb, h->hash_first, h->hash_range);
  h->launches += 2;
  rc = check_launch(h, "hash fill");
  if (rc != PCLOTH_OK) return rc;
  // partners per vertex, their scan, and the total on the host
  PairArgs a{};
  a.n = n;
  a.r2 = r2;
  a.inv_edge = inv_edge;
  a.mask = h->hash_mask;
  a.x = x;
  a.range = h->hash_range;
  a.slot = h->hash_slot;
  a.rowptr_s = h->rowptr_s;
  a.colind_s = h->colind_s;
  a.count = h->pair_first;
  a.total = reinterpret_cast<unsigned long long*>(h->counters + 4);
  e = cudaMemsetAsync(a.total, 0, sizeof(unsigned long long), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "pair total reset");
  pair_pass<false><<<grid, 256, 0, s>>>(a);
  h->launches += 1;
  rc = check_launch(h, "pair count");
  if (rc != PCLOTH_OK) return rc;
  rc = scan_exclusive(h, h->pair_first, n + 1, h->counters + 2);
  if (rc != PCLOTH_OK) return rc;
  unsigned long long total64 = 0;
  e = cudaMemcpyAsync(&total64, a.total, sizeof(total64), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e, "pair count");
  const int32_t total = int32_t(std::min<unsigned long long>(total64, INT32_MAX));
  if (found) *found = total;
  const int32_t cap = std::min<int32_t>(capacity, h->max_contacts);
  if (total64 > static_cast<unsigned long long>(cap)) {
    out->n = 0;
    return fail(h, PCLOTH_ERR_CAPACITY,
                "found " + std::to_string(total64) + " contacts, capacity " + std::to_string(cap));
  }
  if (total > 0) {
    a.out_first = h->pair_first;
    a.oi = const_cast<int32_t*>(out->i);
    a.oj = const_cast<int32_t*>(out->j);
    a.ok = const_cast<float*>(out->k);
    a.orest = const_cast<float*>(out->rest);
    a.k = stiffness;
    a.rest = radius;
    pair_pass<true><<<grid, 256, 0, s>>>(a);
    h->launches += 1;
    rc = check_launch(h, "pair write");
    if (rc != PCLOTH_OK) return rc;
  }
  out->n = total;
  return collect_status(h);
}

}  // namespace pcloth_impl
