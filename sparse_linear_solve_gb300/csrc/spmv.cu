// Block (3x3) sparse matrix-vector product q = A p (P-Cloth, arXiv
// 2008.00409, Sec. 3.1: SpMV is the most expensive operator of the PCG
// solve; Eq. (4) with one GPU is the plain product).
//
// The pages use a block-ELL layout on Pascal/Volta so that one thread per
// row streams coalesced SoA planes.  On GB300 the matrix stays BSR3 and each
// CTA streams whole tiles of rows instead:
//
//   1. the tile's value and column-index ranges are contiguous, so the CTA
//      copies them into shared memory with aligned 16-byte loads (a single
//      HBM pass at full sector efficiency, whatever the row lengths);
//   2. one thread per block multiplies its 3x3 block (stride-9 shared reads,
//      bank-conflict free) by the gathered input vertex (L2/L1 resident);
//   3. one thread per (row, component) sums its row's block products in
//      column order and writes the output coalesced.
//
// Tiles longer than the staging are processed in chunks; a row's partial
// sum simply carries over, so every output has a fixed summation order and
// the product is bitwise reproducible.
//
// The PCG variant fuses two neighbouring steps of the iteration into the
// same pass: the search direction p_k = z_k + beta p_{k-1} is formed on the
// fly where p is gathered (and written once for the block's own rows), and
// the partial dot product p_k . q_k is reduced per CTA.

#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

constexpr int kValFloats = kSpmvCap * 9 + 8;
constexpr int kColInts = kSpmvCap + 8;
constexpr size_t kSpmvSmem =
    size_t(kValFloats) * 4 + size_t(kColInts) * 4 + size_t(kSpmvCap) * 3 * 4 +
    size_t(kSpmvRows + 1 + 7) * 4;

struct SpmvArgs {
  int32_t n;
  int32_t ntiles;
  const int32_t* rowptr;
  const int32_t* colind;
  const float* vals;
  const float* in;       // plain product input
  float* out;            // plain output, or q for PCG
  // PCG fields
  const float* z;
  const float* p_old;
  float* p_new;
  const double* rz_cur;  // partials of r_k . z_k (slot 0) and r_k . r_k (slot 1)
  const double* rz_prev; // partials of r_{k-1} . z_{k-1}
  const double* bb;      // partials of b . b (slot 0)
  int red_n;             // number of partial records of rz_* and bb
  double* pq_out;        // this kernel's partials of p . q
  PcgState* state;
  uint32_t* status;
  int first;
  int k;
  double tol2;
};

template <bool PCG>
__global__ void __launch_bounds__(kSpmvThreads)
spmv_tiles(SpmvArgs a) {
  extern __shared__ float4 smem4[];
  float* sv = reinterpret_cast<float*>(smem4);
  int32_t* sc = reinterpret_cast<int32_t*>(sv + kValFloats);
  float* part = reinterpret_cast<float*>(sc + kColInts);
  int32_t* srp = reinterpret_cast<int32_t*>(part + kSpmvCap * 3);
  __shared__ double rsh[33];
  __shared__ int done_sh;

  float beta = 0.f;
  if (PCG) {
    if (threadIdx.x == 0) done_sh = a.state->done;
    __syncthreads();
    if (done_sh) return;
    const double bb = reduce_partials<kSpmvThreads>(a.bb, a.red_n, kRedSlots, 0, rsh);
    if (a.first) {
      if (!(bb > 0.0) || !isfinite(bb)) {
        // b = 0: dv = 0 solves exactly; non-finite b: report it
        if (blockIdx.x == 0 && threadIdx.x == 0) {
          a.state->done = 1;
          a.state->iterations = 0;
          a.state->relres = 0.0;
          a.state->code = isfinite(bb) ? PCLOTH_OK : PCLOTH_ERR_NONFINITE;
          if (!isfinite(bb)) atomicOr(a.status, ST_NONFINITE);
        }
        return;
      }
    } else {
      const double rr = reduce_partials<kSpmvThreads>(a.rz_cur, a.red_n, kRedSlots, 1, rsh);
      const double rz = reduce_partials<kSpmvThreads>(a.rz_cur, a.red_n, kRedSlots, 0, rsh);
      const double rzp = reduce_partials<kSpmvThreads>(a.rz_prev, a.red_n, kRedSlots, 0, rsh);
      const bool conv = rr <= a.tol2 * bb;
      const bool bad = !isfinite(rr) || !isfinite(rz) || !(rz > 0.0) || !(rzp > 0.0);
      if (conv || bad) {
        if (blockIdx.x == 0 && threadIdx.x == 0) {
          a.state->done = 1;
          a.state->iterations = a.k;
          a.state->relres = sqrt(rr / bb);
          a.state->code = conv ? PCLOTH_OK
                               : (isfinite(rr) && isfinite(rz) ? PCLOTH_ERR_BREAKDOWN
                                                               : PCLOTH_ERR_NONFINITE);
          if (!conv) atomicOr(a.status, isfinite(rz) ? ST_BREAKDOWN : ST_NONFINITE);
        }
        return;
      }
      beta = float(rz / rzp);
    }
  }

  const int tid = threadIdx.x;
  const int lr = tid / 3, comp = tid - 3 * (tid / 3);
  float pq = 0.f;
  for (int32_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    const int32_t r0 = tile * kSpmvRows;
    const int32_t nrows = min(kSpmvRows, a.n - r0);
    if (tid <= nrows) srp[tid] = a.rowptr[r0 + tid];
    __syncthreads();
    const int32_t b0 = srp[0], b1 = srp[nrows];
    float acc = 0.f;
    for (int32_t c0 = b0; c0 < b1; c0 += kSpmvCap) {
      const int32_t c1 = min(b1, c0 + kSpmvCap);
      const int32_t cn = c1 - c0;
      // aligned 16-byte copies of the chunk's values and column indices
      const int64_t w0 = (int64_t(c0) * 9) & ~int64_t(3);
      const int64_t w1 = (int64_t(c1) * 9 + 3) & ~int64_t(3);
      const int voff = int(int64_t(c0) * 9 - w0);
      const float4* gv = reinterpret_cast<const float4*>(a.vals) + (w0 >> 2);
      const int nv4 = int((w1 - w0) >> 2);
      for (int q = tid; q < nv4; q += kSpmvThreads)
        reinterpret_cast<float4*>(sv)[q] = __ldcs(gv + q);
      const int32_t k0 = c0 & ~3, k1 = (c1 + 3) & ~3;
      const int coff = c0 - k0;
      const int4* gc = reinterpret_cast<const int4*>(a.colind) + (k0 >> 2);
      const int nk4 = (k1 - k0) >> 2;
      for (int q = tid; q < nk4; q += kSpmvThreads)
        reinterpret_cast<int4*>(sc)[q] = __ldcs(gc + q);
      __syncthreads();
      for (int j = tid; j < cn; j += kSpmvThreads) {
        const int32_t col = sc[coff + j];
        const float* B = sv + voff + 9 * j;
        const int64_t c3 = int64_t(col) * 3;
        float x0, x1, x2;
        if (PCG) {
          x0 = a.z[c3]; x1 = a.z[c3 + 1]; x2 = a.z[c3 + 2];
          if (!a.first) {
            x0 = fmaf(beta, a.p_old[c3], x0);
            x1 = fmaf(beta, a.p_old[c3 + 1], x1);
            x2 = fmaf(beta, a.p_old[c3 + 2], x2);
          }
        } else {
          x0 = a.in[c3]; x1 = a.in[c3 + 1]; x2 = a.in[c3 + 2];
        }
        part[3 * j + 0] = fmaf(B[0], x0, fmaf(B[1], x1, B[2] * x2));
        part[3 * j + 1] = fmaf(B[3], x0, fmaf(B[4], x1, B[5] * x2));
        part[3 * j + 2] = fmaf(B[6], x0, fmaf(B[7], x1, B[8] * x2));
      }
      __syncthreads();
      if (tid < 3 * nrows) {
        const int32_t rs = max(srp[lr], c0), re = min(srp[lr + 1], c1);
        for (int32_t b = rs; b < re; ++b) acc += part[3 * (b - c0) + comp];
      }
      __syncthreads();
    }
    if (tid < 3 * nrows) {
      const int64_t gi = int64_t(r0 + lr) * 3 + comp;
      a.out[gi] = acc;
      if (PCG) {
        const float pn = a.first ? a.z[gi] : fmaf(beta, a.p_old[gi], a.z[gi]);
        a.p_new[gi] = pn;
        pq = fmaf(pn, acc, pq);
      }
    }
    __syncthreads();
  }
  if (PCG) {
    const double t = block_sum<kSpmvThreads>(double(pq), rsh);
    if (tid == 0) a.pq_out[int64_t(blockIdx.x) * kRedSlots] = t;
  }
}

bool g_attr_done[64] = {};

int ensure_attr(Handle* h) {
  if (h->device >= 0 && h->device < 64 && g_attr_done[h->device]) return PCLOTH_OK;
  cudaError_t e = cudaFuncSetAttribute(spmv_tiles<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kSpmvSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(spmv_tiles<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSpmvSmem));
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(spmv)");
  if (h->device >= 0 && h->device < 64) g_attr_done[h->device] = true;
  return PCLOTH_OK;
}

}  // namespace

int launch_spmv(Handle* h, const float* in, float* out) {
  int rc = ensure_attr(h);
  if (rc != PCLOTH_OK) return rc;
  SpmvArgs a{};
  a.n = h->n;
  a.ntiles = (h->n + kSpmvRows - 1) / kSpmvRows;
  a.rowptr = h->rowptr;
  a.colind = h->colind;
  a.vals = h->vals;
  a.in = in;
  a.out = out;
  spmv_tiles<false><<<h->spmv_grid, kSpmvThreads, kSpmvSmem, h->stream>>>(a);
  h->launches += 1;
  return check_launch(h, "spmv");
}

// One PCG SpMV of iteration k (0-based): q = A p_k with p_k = z_k + beta p_{k-1}.
int launch_spmv_pcg(Handle* h, int k, double tol) {
  int rc = ensure_attr(h);
  if (rc != PCLOTH_OK) return rc;
  SpmvArgs a{};
  a.n = h->n;
  a.ntiles = (h->n + kSpmvRows - 1) / kSpmvRows;
  a.rowptr = h->rowptr;
  a.colind = h->colind;
  a.vals = h->vals;
  a.out = h->q;
  a.z = h->z;
  a.p_old = h->p[(k + 1) & 1];
  a.p_new = h->p[k & 1];
  a.rz_cur = h->red_upd[k & 1];
  a.rz_prev = h->red_upd[(k + 1) & 1];
  a.bb = h->red_init;
  a.red_n = h->vec_grid;
  a.pq_out = h->red_spmv;
  a.state = h->state;
  a.status = h->d_status;
  a.first = (k == 0);
  a.k = k;
  a.tol2 = tol * tol;
  spmv_tiles<true><<<h->spmv_grid, kSpmvThreads, kSpmvSmem, h->stream>>>(a);
  h->launches += 1;
  return check_launch(h, "spmv (pcg)");
}

}  // namespace pcloth_impl
