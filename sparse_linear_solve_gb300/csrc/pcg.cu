// Block-Jacobi preconditioned conjugate gradients on A dv = b (P-Cloth,
// arXiv 2008.00409, Sec. 2.5 Eq. (3) and Sec. 3.1: the linear system of each
// step is solved by PCG; the pages do not name the preconditioner, this uses
// the inverses of the 3x3 diagonal blocks), plus the backward-Euler state
// update v += dv, x += h v.
//
// One iteration is two kernels:
//   spmv_tiles<true>  p_k = z_k + beta p_{k-1} (formed where gathered),
//                     q = A p_k, partial p_k . q
//   pcg_update        alpha = (r.z)/(p.q); dv += alpha p; r -= alpha q;
//                     z = P r; partials r.z and r.r
// Every scalar (alpha, beta, the convergence test |r| <= tol |b|) is formed
// on the device by each CTA from the previous kernel's per-CTA partials in a
// fixed order, so no host round trip is needed inside the loop and the
// iteration is bitwise reproducible.  Dot products accumulate a few terms in
// fp32 per thread and everything after that in fp64.  The host enqueues
// `chunk` iterations at a time and reads the device state of the previous
// chunk while the current one runs; kernels enqueued after convergence
// return at once.

#include <algorithm>

#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

// Vertex-to-lane mapping of the vector kernels: a warp covers 10 vertices,
// lanes 3v..3v+2 hold the components of vertex v (lanes 30, 31 idle), so the
// three components of a vertex are always read before any is written.
constexpr int kVertsPerWarp = 10;

__device__ __forceinline__ bool lane_vertex(int64_t wglobal, int lane, int32_t n,
                                            int64_t& i, int& c) {
  i = wglobal * kVertsPerWarp + lane / 3;
  c = lane - 3 * (lane / 3);
  return lane < 3 * kVertsPerWarp && i < n;
}

__global__ void __launch_bounds__(kVecThreads)
pcg_init(int32_t n, const float* __restrict__ b, const float* __restrict__ pinv,
         float* __restrict__ r, float* __restrict__ z, float* __restrict__ dv,
         float* __restrict__ p_old, double* __restrict__ red_rz0,
         double* __restrict__ red_bb, PcgState* state) {
  __shared__ double sh[33];
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(n) + kVertsPerWarp - 1) / kVertsPerWarp;
  const int64_t wstride = int64_t(gridDim.x) * (kVecThreads / 32);
  float rz = 0.f, bb = 0.f;
  for (int64_t w = int64_t(blockIdx.x) * (kVecThreads / 32) + (threadIdx.x >> 5); w < nwarps;
       w += wstride) {
    int64_t i;
    int c;
    if (!lane_vertex(w, lane, n, i, c)) continue;
    const int64_t e = 3 * i + c;
    const float* P = pinv + 9 * i + 3 * c;
    const float b0 = b[3 * i], b1 = b[3 * i + 1], b2 = b[3 * i + 2];
    const float be = b[e];
    const float ze = fmaf(P[0], b0, fmaf(P[1], b1, P[2] * b2));
    r[e] = be;
    z[e] = ze;
    dv[e] = 0.f;
    p_old[e] = 0.f;
    rz = fmaf(be, ze, rz);
    bb = fmaf(be, be, bb);
  }
  const double trz = block_sum<kVecThreads>(double(rz), sh);
  const double tbb = block_sum<kVecThreads>(double(bb), sh);
  if (threadIdx.x == 0) {
    red_rz0[int64_t(blockIdx.x) * kRedSlots + 0] = trz;
    red_rz0[int64_t(blockIdx.x) * kRedSlots + 1] = tbb;
    red_bb[int64_t(blockIdx.x) * kRedSlots + 0] = tbb;
    if (blockIdx.x == 0) {
      state->done = 0;
      state->iterations = 0;
      state->code = PCLOTH_NOT_CONVERGED;
      state->relres = 1.0;
    }
  }
}

__global__ void __launch_bounds__(kVecThreads)
pcg_update(int32_t n, int k, const float* __restrict__ p, const float* __restrict__ q,
           const float* __restrict__ pinv, float* __restrict__ r, float* __restrict__ z,
           float* __restrict__ dv, const double* __restrict__ red_pq, int npq,
           const double* __restrict__ red_rz, const double* __restrict__ red_bb, int nrz,
           double* __restrict__ red_out, PcgState* state, uint32_t* status) {
  __shared__ double sh[33];
  __shared__ int done_sh;
  if (threadIdx.x == 0) done_sh = state->done;
  __syncthreads();
  if (done_sh) return;
  const double pq = reduce_partials<kVecThreads>(red_pq, npq, kRedSlots, 0, sh);
  const double rz = reduce_partials<kVecThreads>(red_rz, nrz, kRedSlots, 0, sh);
  if (!(pq > 0.0) || !isfinite(pq) || !isfinite(rz)) {
    const double rr = reduce_partials<kVecThreads>(red_rz, nrz, kRedSlots, 1, sh);
    const double bb = reduce_partials<kVecThreads>(red_bb, nrz, kRedSlots, 0, sh);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      const bool fin = isfinite(pq) && isfinite(rz);
      state->done = 1;
      state->iterations = k;
      state->relres = sqrt(rr / bb);
      state->code = fin ? PCLOTH_ERR_BREAKDOWN : PCLOTH_ERR_NONFINITE;
      atomicOr(status, fin ? ST_BREAKDOWN : ST_NONFINITE);
    }
    return;
  }
  const float alpha = float(rz / pq);
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t(n) + kVertsPerWarp - 1) / kVertsPerWarp;
  const int64_t wstride = int64_t(gridDim.x) * (kVecThreads / 32);
  float arz = 0.f, arr = 0.f;
  for (int64_t w = int64_t(blockIdx.x) * (kVecThreads / 32) + (threadIdx.x >> 5); w < nwarps;
       w += wstride) {
    int64_t i;
    int c;
    const bool on = lane_vertex(w, lane, n, i, c);
    float r0 = 0.f, r1 = 0.f, r2 = 0.f, re = 0.f, ze = 0.f;
    if (on) {
      const int64_t v3 = 3 * i, e = v3 + c;
      dv[e] = fmaf(alpha, p[e], dv[e]);
      r0 = fmaf(-alpha, q[v3], r[v3]);
      r1 = fmaf(-alpha, q[v3 + 1], r[v3 + 1]);
      r2 = fmaf(-alpha, q[v3 + 2], r[v3 + 2]);
      re = c == 0 ? r0 : (c == 1 ? r1 : r2);
      const float* P = pinv + 9 * i + 3 * c;
      ze = fmaf(P[0], r0, fmaf(P[1], r1, P[2] * r2));
    }
    __syncwarp();  // all three lanes of a vertex have read r before any writes it
    if (on) {
      const int64_t e = 3 * i + c;
      r[e] = re;
      z[e] = ze;
      arz = fmaf(re, ze, arz);
      arr = fmaf(re, re, arr);
    }
  }
  const double trz = block_sum<kVecThreads>(double(arz), sh);
  const double trr = block_sum<kVecThreads>(double(arr), sh);
  if (threadIdx.x == 0) {
    red_out[int64_t(blockIdx.x) * kRedSlots + 0] = trz;
    red_out[int64_t(blockIdx.x) * kRedSlots + 1] = trr;
  }
}

// Closes a solve that used all its iterations (or none).
__global__ void pcg_finish(int k, double tol2, const double* __restrict__ red_rz,
                           const double* __restrict__ red_bb, int nrz, PcgState* state) {
  __shared__ double sh[33];
  __shared__ int done_sh;
  if (threadIdx.x == 0) done_sh = state->done;
  __syncthreads();
  if (done_sh) return;
  const double rr = reduce_partials<kVecThreads>(red_rz, nrz, kRedSlots, 1, sh);
  const double bb = reduce_partials<kVecThreads>(red_bb, nrz, kRedSlots, 0, sh);
  if (threadIdx.x == 0) {
    state->done = 1;
    state->iterations = k;
    state->relres = bb > 0.0 ? sqrt(rr / bb) : 0.0;
    state->code = (rr <= tol2 * bb) ? PCLOTH_OK : PCLOTH_NOT_CONVERGED;
    if (!isfinite(rr) || !isfinite(bb)) state->code = PCLOTH_ERR_NONFINITE;
  }
}

__global__ void __launch_bounds__(kVecThreads)
state_update(int64_t m, float* __restrict__ x, float* __restrict__ v,
             const float* __restrict__ dv, float dt, uint32_t* status) {
  bool ok = true;
  for (int64_t e = int64_t(blockIdx.x) * kVecThreads + threadIdx.x; e < m;
       e += int64_t(gridDim.x) * kVecThreads) {
    const float vn = v[e] + dv[e];
    const float xn = fmaf(dt, vn, x[e]);
    v[e] = vn;
    x[e] = xn;
    ok = ok && isfinite(xn) && isfinite(vn);
  }
  if (!ok) atomicOr(status, ST_NONFINITE);
}

}  // namespace

int launch_state_update(Handle* h, float* x, float* v, const float* dv, float dt) {
  state_update<<<h->vec_grid, kVecThreads, 0, h->stream>>>(int64_t(h->n) * 3, x, v, dv, dt,
                                                           h->d_status);
  h->launches += 1;
  return check_launch(h, "state update");
}

int pcg_solve(Handle* h, double tol, int32_t maxit, float* dv, int32_t* iterations,
              double* rel_residual) {
  cudaStream_t s = h->stream;
  const double tol2 = tol * tol;
  const bool prof = h->prof.on;
  const int vg = h->vec_grid;
  if (prof) cudaEventRecord(h->ev[2], s);
  pcg_init<<<vg, kVecThreads, 0, s>>>(h->n, h->rhs, h->pinv, h->r, h->z, dv, h->p[1],
                                      h->red_upd[0], h->red_init, h->state);
  h->launches += 1;
  int rc = check_launch(h, "pcg init");
  if (rc != PCLOTH_OK) return rc;

  int32_t k = 0;
  int chunk_id = 0, pending = -1;
  bool done = false;
  const int per = 2 * h->chunk + 1;  // events per chunk slot
  auto consume = [&](int slot, int launched) {
    if (!prof) return;
    cudaEvent_t* ev = h->pev.data() + size_t(slot) * per;
    for (int j = 0; j < launched; ++j) {
      float a = 0.f, b = 0.f;
      if (cudaEventElapsedTime(&a, ev[2 * j], ev[2 * j + 1]) == cudaSuccess)
        h->prof.spmv_ms += a;
      if (cudaEventElapsedTime(&b, ev[2 * j + 1], ev[2 * j + 2]) == cudaSuccess)
        h->prof.update_ms += b;
    }
  };
  int launched_in[2] = {0, 0};
  while (k < maxit && !done) {
    const int slot = chunk_id & 1;
    const int m = std::min<int32_t>(h->chunk, maxit - k);
    cudaEvent_t* ev = h->pev.data() + size_t(slot) * per;
    for (int j = 0; j < m; ++j, ++k) {
      if (prof && j == 0) cudaEventRecord(ev[0], s);
      rc = launch_spmv_pcg(h, k, tol);
      if (rc != PCLOTH_OK) return rc;
      if (prof) cudaEventRecord(ev[2 * j + 1], s);
      pcg_update<<<vg, kVecThreads, 0, s>>>(h->n, k, h->p[k & 1], h->q, h->pinv, h->r, h->z, dv,
                                            h->red_spmv, h->spmv_grid, h->red_upd[k & 1],
                                            h->red_init, vg, h->red_upd[(k + 1) & 1], h->state,
                                            h->d_status);
      h->launches += 1;
      if (prof) cudaEventRecord(ev[2 * j + 2], s);
    }
    launched_in[slot] = m;
    rc = check_launch(h, "pcg update");
    if (rc != PCLOTH_OK) return rc;
    cudaMemcpyAsync(&h->state_host[slot], h->state, sizeof(PcgState), cudaMemcpyDeviceToHost, s);
    cudaEventRecord(h->chunk_ev[slot], s);
    if (pending >= 0) {
      cudaError_t e = cudaEventSynchronize(h->chunk_ev[pending]);
      if (e != cudaSuccess) return cuda_fail(h, e, "pcg poll");
      consume(pending, launched_in[pending]);
      if (h->state_host[pending].done) done = true;
    }
    pending = slot;
    ++chunk_id;
  }
  if (pending >= 0) {
    cudaError_t e = cudaEventSynchronize(h->chunk_ev[pending]);
    if (e != cudaSuccess) return cuda_fail(h, e, "pcg poll");
    consume(pending, launched_in[pending]);
  }
  pcg_finish<<<1, kVecThreads, 0, s>>>(k, tol2, h->red_upd[k & 1], h->red_init, vg, h->state);
  h->launches += 1;
  rc = check_launch(h, "pcg finish");
  if (rc != PCLOTH_OK) return rc;
  cudaMemcpyAsync(&h->state_host[0], h->state, sizeof(PcgState), cudaMemcpyDeviceToHost, s);
  if (prof) cudaEventRecord(h->ev[3], s);
  rc = collect_status(h);  // synchronises
  const PcgState st = h->state_host[0];
  if (iterations) *iterations = st.iterations;
  if (rel_residual) *rel_residual = st.relres;
  if (prof) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, h->ev[2], h->ev[3]);
    h->prof.solve_ms += ms;
    h->prof.solves += 1;
    h->prof.iterations += st.iterations;
    h->prof.spmv_launches += k;
    h->prof.update_launches += k;
  }
  if (rc != PCLOTH_OK && rc != PCLOTH_ERR_BREAKDOWN && rc != PCLOTH_ERR_NONFINITE) return rc;
  if (st.code != PCLOTH_OK && st.code != PCLOTH_NOT_CONVERGED) {
    fail(h, st.code, st.code == PCLOTH_ERR_BREAKDOWN ? "PCG breakdown (p.Ap <= 0 or r.z <= 0)"
                                                     : "non-finite value in PCG");
    return st.code;
  }
  if (rc != PCLOTH_OK) return rc;
  if (st.code == PCLOTH_NOT_CONVERGED) fail(h, st.code, "PCG reached maxit");
  return st.code;
}

}  // namespace pcloth_impl
