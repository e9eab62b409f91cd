// Vertex-vertex proximity contacts by spatial hashing (P-Cloth, arXiv
// 2008.00409, Sec. 4.2: a spatial-hash table built on the fly every step,
// then proximity tests; Sec. 4.3: proximities enter the implicit integrator
// as forces).  Restricted to pairs of vertices: every pair i < j closer than
// a radius r that is not a spring becomes a contact (a spring of stiffness
// k_c and rest length r), listed in (i, j) order.
//
//   cell_keys     each vertex to its cell of edge r (1 + 2^-7): the slight
//                 enlargement keeps every pair closer than r in neighbouring
//                 cells despite the rounding of x / edge, for coordinates up
//                 to 2^15 cells from the origin (65 m at r = 2 mm)
//   radix sort    vertices by cell key (z fastest, so the three cells of a
//                 column along z are contiguous in key order)
//   find_pairs    per vertex: the 3 x 3 columns of neighbouring cells, one
//                 binary search each; every candidate j > i gets the exact
//                 test in float32 ((dx dx + dy dy) + dz dz < r r, each
//                 operation rounded) and spring pairs are dropped by a
//                 binary search in the static pattern; survivors are
//                 appended
//   radix sort    the appended (i, j) keys, so the list is deterministic
//   unpack        into the caller's i, j, k, rest arrays
//
// The distance test decides an integer outcome, so it is written with
// explicitly rounded operations (no fused multiply-add) to be reproducible
// by a plain float32 restatement.

#include <algorithm>

#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

constexpr int kCellBits = 21;                          // per axis
constexpr int32_t kCellBias = 1 << (kCellBits - 1);    // cells -2^20 .. 2^20 - 1
constexpr uint64_t kCellMask = (uint64_t(1) << kCellBits) - 1;

__device__ __forceinline__ uint64_t cell_key(int32_t cx, int32_t cy, int32_t cz) {
  return (uint64_t(uint32_t(cx + kCellBias) & kCellMask) << (2 * kCellBits)) |
         (uint64_t(uint32_t(cy + kCellBias) & kCellMask) << kCellBits) |
         uint64_t(uint32_t(cz + kCellBias) & kCellMask);
}

__device__ __forceinline__ int32_t cell_of(float v, float inv_edge) {
  const float c = floorf(v * inv_edge);
  return int32_t(fminf(fmaxf(c, float(-kCellBias + 2)), float(kCellBias - 3)));
}

__global__ void cell_keys(int32_t n, const float* __restrict__ x, float inv_edge,
                          uint64_t* __restrict__ keys, int32_t* __restrict__ ids,
                          uint32_t* status) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float px = x[3 * i], py = x[3 * i + 1], pz = x[3 * i + 2];
  if (!finite3(px, py, pz)) atomicOr(status, ST_NONFINITE);
  keys[i] = cell_key(cell_of(px, inv_edge), cell_of(py, inv_edge), cell_of(pz, inv_edge));
  ids[i] = int32_t(i);
}

__device__ __forceinline__ int32_t lower_bound_u64(const uint64_t* a, int32_t n, uint64_t v) {
  int32_t lo = 0, hi = n;
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (a[mid] < v) lo = mid + 1; else hi = mid;
  }
  return lo;
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

// One thread per sorted position t (vertex i = ids[t]).
__global__ void find_pairs(int32_t n, const float* __restrict__ x, float r2, float inv_edge,
                           const uint64_t* __restrict__ keys, const int32_t* __restrict__ ids,
                           const int32_t* __restrict__ rowptr_s,
                           const int32_t* __restrict__ colind_s, int key_bits,
                           unsigned long long* __restrict__ pairs, int32_t capacity,
                           int32_t* counter) {
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n) return;
  const int32_t i = ids[t];
  const float px = x[3 * int64_t(i)], py = x[3 * int64_t(i) + 1], pz = x[3 * int64_t(i) + 2];
  const int32_t cx = cell_of(px, inv_edge), cy = cell_of(py, inv_edge), cz = cell_of(pz, inv_edge);
  for (int ox = -1; ox <= 1; ++ox) {
    for (int oy = -1; oy <= 1; ++oy) {
      const int32_t b = lower_bound_u64(keys, n, cell_key(cx + ox, cy + oy, cz - 1));
      const uint64_t last = cell_key(cx + ox, cy + oy, cz + 1);
      for (int32_t u = b; u < n && keys[u] <= last; ++u) {
        const int32_t j = ids[u];
        if (j <= i) continue;
        const float dx = __fsub_rn(x[3 * int64_t(j)], px);
        const float dy = __fsub_rn(x[3 * int64_t(j) + 1], py);
        const float dz = __fsub_rn(x[3 * int64_t(j) + 2], pz);
        const float d2 = __fadd_rn(__fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy)),
                                   __fmul_rn(dz, dz));
        if (!(d2 < r2)) continue;
        if (is_spring(rowptr_s, colind_s, i, j)) continue;
        const int32_t slot = atomicAdd(counter, 1);
        if (slot < capacity)
          pairs[slot] = (static_cast<unsigned long long>(i) << key_bits) |
                        static_cast<unsigned long long>(j);
      }
    }
  }
}

__global__ void unpack_pairs(int32_t m, const uint64_t* __restrict__ pairs, int key_bits,
                             float k, float rest, int32_t* __restrict__ oi,
                             int32_t* __restrict__ oj, float* __restrict__ ok,
                             float* __restrict__ orest) {
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= m) return;
  const uint64_t p = pairs[t];
  oi[t] = int32_t(p >> key_bits);
  oj[t] = int32_t(p & ((uint64_t(1) << key_bits) - 1));
  ok[t] = k;
  orest[t] = rest;
}

}  // namespace

int find_contacts(Handle* h, const float* x, float radius, float stiffness,
                  pcloth_springs* out, int32_t capacity, int32_t* found) {
  cudaStream_t s = h->stream;
  const int32_t n = h->n;
  const float edge = radius * (1.0f + 1.0f / 128.0f);
  const float inv_edge = 1.0f / edge;
  const float r2 = radius * radius;   // float32, as the test compares
  // vertices by cell
  cell_keys<<<(n + 255) / 256, 256, 0, s>>>(n, x, inv_edge, h->vkey[0], h->vid[0], h->d_status);
  h->launches += 1;
  int rc = check_launch(h, "cell keys");
  if (rc != PCLOTH_OK) return rc;
  const int cur = radix_sort_pairs(h, h->vkey, h->vid, n, 3 * 21);
  if (cur < 0) return cur;
  // candidate pairs, appended
  cudaError_t e = cudaMemsetAsync(h->counters + 2, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "pair counter");
  const int32_t cap = std::min<int32_t>(capacity, h->max_contacts);
  find_pairs<<<(n + 255) / 256, 256, 0, s>>>(
      n, x, r2, inv_edge, h->vkey[cur], h->vid[cur], h->rowptr_s, h->colind_s, h->key_bits,
      reinterpret_cast<unsigned long long*>(h->ckey[0]), cap, h->counters + 2);
  h->launches += 1;
  rc = check_launch(h, "find pairs");
  if (rc != PCLOTH_OK) return rc;
  int32_t total = 0;
  e = cudaMemcpyAsync(&total, h->counters + 2, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e, "pair count");
  if (found) *found = total;
  if (total > cap) {
    out->n = 0;
    return fail(h, PCLOTH_ERR_CAPACITY,
                "found " + std::to_string(total) + " contacts, capacity " + std::to_string(cap));
  }
  // (i, j) order
  const int cur2 = radix_sort_pairs(h, h->ckey, h->cval, total, 2 * h->key_bits);
  if (cur2 < 0) return cur2;
  if (total > 0) {
    unpack_pairs<<<(total + 255) / 256, 256, 0, s>>>(
        total, h->ckey[cur2], h->key_bits, stiffness, radius, const_cast<int32_t*>(out->i),
        const_cast<int32_t*>(out->j), const_cast<float*>(out->k),
        const_cast<float*>(out->rest));
    h->launches += 1;
    rc = check_launch(h, "unpack pairs");
    if (rc != PCLOTH_OK) return rc;
  }
  out->n = total;
  return collect_status(h);
}

}  // namespace pcloth_impl
