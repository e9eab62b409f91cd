// Block-ELL (BELL) copy of the assembled matrix and its SpMV, for comparison
// with the streaming BSR3 product.  P-Cloth (arXiv 2008.00409), Sec. 3.2.2:
// the pages store the matrix as an index table and a value table padded to
// the longest compacted row, so that one thread per row reads coalesced
// columns of the tables.
//
// Layout here: W = the longest row (in blocks) of the current pattern; slot
// s of row i sits at s * n + i.  colind_ell int32[W * n] (-1 past the end of
// a row) and six value planes (the packed symmetric block a00 a01 a02 a11
// a12 a22), plane k at k * W * n.  One thread per row walks its slots in
// column order and adds the same products in the same order as the BSR3
// kernel, so the two give the same bits.

#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

__global__ void row_width_max(int32_t n, const int32_t* __restrict__ rowptr, int32_t* wmax) {
  int32_t w = 0;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    w = max(w, rowptr[i + 1] - rowptr[i]);
  for (int o = 16; o > 0; o >>= 1) w = max(w, __shfl_down_sync(0xffffffffu, w, o));
  if ((threadIdx.x & 31) == 0) atomicMax(wmax, w);
}

__global__ void bell_convert(int32_t n, int32_t W, const int32_t* __restrict__ rowptr,
                             const int32_t* __restrict__ colind,
                             const float* __restrict__ vals, int32_t* __restrict__ col_ell,
                             float* __restrict__ val_ell) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t plane = int64_t(W) * n;
  const int32_t b0 = rowptr[i], len = rowptr[i + 1] - b0;
  for (int32_t s = 0; s < W; ++s) {
    const int64_t e = int64_t(s) * n + i;
    if (s < len) {
      const int64_t b = b0 + s;
      col_ell[e] = colind[b];
#pragma unroll
      for (int k = 0; k < kSymBlock; ++k) val_ell[k * plane + e] = vals[kSymBlock * b + k];
    } else {
      col_ell[e] = -1;
#pragma unroll
      for (int k = 0; k < kSymBlock; ++k) val_ell[k * plane + e] = 0.f;
    }
  }
}

__global__ void __launch_bounds__(256)
bell_spmv(int32_t n, int32_t W, const int32_t* __restrict__ col_ell,
          const float* __restrict__ val_ell, const int32_t* __restrict__ rowptr,
          const float* __restrict__ in, float* __restrict__ out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t plane = int64_t(W) * n;
  // long rows are summed with compensation, as in the BSR3 kernel
  const bool comp = rowptr[i + 1] - rowptr[i] > kCompRow;
  float ax = 0.f, ay = 0.f, az = 0.f, cx = 0.f, cy = 0.f, cz = 0.f;
  for (int32_t s = 0; s < W; ++s) {
    const int64_t e = int64_t(s) * n + i;
    const int32_t c = col_ell[e];
    if (c < 0) break;   // slots past a row's end are all padding
    const float a00 = val_ell[e], a01 = val_ell[plane + e], a02 = val_ell[2 * plane + e];
    const float a11 = val_ell[3 * plane + e], a12 = val_ell[4 * plane + e];
    const float a22 = val_ell[5 * plane + e];
    const int64_t c3 = int64_t(c) * 3;
    const float x = in[c3], y = in[c3 + 1], z = in[c3 + 2];
    // the same products, in the same order, as the packed block of the BSR3 kernel
    const float px = fmaf(a00, x, fmaf(a01, y, a02 * z));
    const float py = fmaf(a01, x, fmaf(a11, y, a12 * z));
    const float pz = fmaf(a02, x, fmaf(a12, y, a22 * z));
    if (comp) {
      add_comp(ax, cx, px);
      add_comp(ay, cy, py);
      add_comp(az, cz, pz);
    } else {
      ax += px;
      ay += py;
      az += pz;
    }
  }
  out[3 * i] = ax + cx;
  out[3 * i + 1] = ay + cy;
  out[3 * i + 2] = az + cz;
}

}  // namespace

int bell_build(Handle* h) {
  cudaStream_t s = h->stream;
  const int32_t n = h->n;
  cudaError_t e = cudaMemsetAsync(h->bell_wmax, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "bell width reset");
  row_width_max<<<h->vec_grid, 256, 0, s>>>(n, h->rowptr, h->bell_wmax);
  h->launches += 1;
  int rc = check_launch(h, "bell width");
  if (rc != PCLOTH_OK) return rc;
  int32_t W = 0;
  e = cudaMemcpyAsync(&W, h->bell_wmax, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(h, e, "bell width");
  if (W <= 0) return fail(h, PCLOTH_ERR_STATE, "empty pattern");
  const int64_t slots = int64_t(W) * n;
  if (slots > h->bell_cap) {   // grows only; freed with the handle
    if (h->bell_col) cudaFree(h->bell_col);
    if (h->bell_val) cudaFree(h->bell_val);
    h->bell_col = nullptr;
    h->bell_val = nullptr;
    h->bell_cap = 0;
    e = cudaMalloc(reinterpret_cast<void**>(&h->bell_col), size_t(slots) * sizeof(int32_t));
    if (e == cudaSuccess)
      e = cudaMalloc(reinterpret_cast<void**>(&h->bell_val),
                     size_t(slots) * kSymBlock * sizeof(float));
    if (e != cudaSuccess) return cuda_fail(h, e, "bell tables");
    h->bell_cap = slots;
  }
  h->bell_w = W;
  bell_convert<<<(n + 255) / 256, 256, 0, s>>>(n, W, h->rowptr, h->colind, h->vals, h->bell_col,
                                               h->bell_val);
  h->launches += 1;
  rc = check_launch(h, "bell convert");
  if (rc != PCLOTH_OK) return rc;
  h->bell_valid = true;
  return PCLOTH_OK;
}

int launch_bell_spmv(Handle* h, const float* in, float* out) {
  bell_spmv<<<(h->n + 255) / 256, 256, 0, h->stream>>>(h->n, h->bell_w, h->bell_col, h->bell_val,
                                                       h->rowptr, in, out);
  h->launches += 1;
  return check_launch(h, "bell spmv");
}

}  // namespace pcloth_impl
