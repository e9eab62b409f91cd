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

// Vector kernels: one thread per vertex on the padded vectors (one float4
// (x, y, z, 0) per vertex), so every access of a warp is one contiguous,
// aligned 512-byte transaction; the symmetric block-Jacobi inverse is two
// float4 per vertex.  Dot products accumulate a vertex's three terms in fp32
// and everything after that in fp64.
__device__ __forceinline__ float3 apply_p(float4 u, float4 w, float3 r) {
  // P = [[u.x u.y u.z] [u.y u.w w.x] [u.z w.x w.y]]
  return make_float3(fmaf(u.x, r.x, fmaf(u.y, r.y, u.z * r.z)),
                     fmaf(u.y, r.x, fmaf(u.w, r.y, w.x * r.z)),
                     fmaf(u.z, r.x, fmaf(w.x, r.y, w.y * r.z)));
}

__device__ __forceinline__ float dot3(float3 a, float3 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, a.z * b.z));
}

__global__ void __launch_bounds__(kVecThreads)
pcg_init(int32_t n, const float* __restrict__ b, const float4* __restrict__ pinv8,
         float4* __restrict__ r, float4* __restrict__ z, float4* __restrict__ dv,
         float4* __restrict__ p_old, float2* __restrict__ red_rz0,
         float2* __restrict__ red_bb, PcgState* state) {
  __shared__ float2 sh[33 * 2];
  float rz = 0.f, bb = 0.f;
  for (int64_t i = int64_t(blockIdx.x) * kVecThreads + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * kVecThreads) {
    const float3 bv = make_float3(b[3 * i], b[3 * i + 1], b[3 * i + 2]);
    const float3 zv = apply_p(pinv8[2 * i], pinv8[2 * i + 1], bv);
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    r[i] = make_float4(bv.x, bv.y, bv.z, 0.f);
    z[i] = make_float4(zv.x, zv.y, zv.z, 0.f);
    dv[i] = zero;
    p_old[i] = zero;
    rz += dot3(bv, zv);
    bb += dot3(bv, bv);
  }
  Dfloat v[2] = {df_of(rz), df_of(bb)};
  block_sum_df<kVecThreads, 2>(v, sh);
  if (threadIdx.x == 0) {
    red_rz0[int64_t(blockIdx.x) * kRedSlots + 0] = df_pack(v[0]);
    red_rz0[int64_t(blockIdx.x) * kRedSlots + 1] = df_pack(v[1]);
    red_bb[int64_t(blockIdx.x) * kRedSlots + 0] = df_pack(v[1]);
    if (blockIdx.x == 0) {
      state->done = 0;
      state->iterations = 0;
      state->code = PCLOTH_NOT_CONVERGED;
      state->relres = 1.0;
    }
  }
}

// dv += alpha p; r -= alpha q; z = P r; partials of r.z and r.r.  The first
// vertex's loads are issued before alpha is known, so their latency
// overlaps the reduction of the previous kernels' partials.
__global__ void __launch_bounds__(kVecThreads, 4)
pcg_update(int32_t n, int k, const float4* __restrict__ p, const float4* __restrict__ q,
           const float4* __restrict__ pinv8, float4* __restrict__ r, float4* __restrict__ z,
           float4* __restrict__ dv, const float2* __restrict__ red_pq, int npq,
           const float2* __restrict__ red_rz, const float2* __restrict__ red_bb, int nrz,
           float2* __restrict__ red_out, PcgState* state, uint32_t* status) {
  __shared__ float2 sh[33 * 4];
  __shared__ int flag_sh;
  __shared__ float alpha_sh;
  if (threadIdx.x == 0) flag_sh = state->done;
  __syncthreads();
  if (flag_sh) return;
  const int64_t stride = int64_t(gridDim.x) * kVecThreads;
  int64_t i = int64_t(blockIdx.x) * kVecThreads + threadIdx.x;
  float4 pv, qv, rv, dvv, pu, pw;
  if (i < n) {
    pv = p[i]; qv = q[i]; rv = r[i]; dvv = dv[i]; pu = pinv8[2 * i]; pw = pinv8[2 * i + 1];
  }
  Dfloat v[4];   // p.q, r.z, r.r, b.b
  v[0] = records_share(red_pq, npq, 0, kVecThreads);
  v[1] = records_share(red_rz, nrz, 0, kVecThreads);
  v[2] = records_share(red_rz, nrz, 1, kVecThreads);
  v[3] = records_share(red_bb, nrz, 0, kVecThreads);
  block_sum_df<kVecThreads, 4>(v, sh);
  if (threadIdx.x == 0) {
    const double pq = df_value(v[0]), rz = df_value(v[1]);
    int stop = 0;
    if (!(pq > 0.0) || !isfinite(pq) || !isfinite(rz)) {
      stop = 1;
      if (blockIdx.x == 0) {
        const bool fin = isfinite(pq) && isfinite(rz);
        state->done = 1;
        state->iterations = k;
        state->relres = sqrt(df_value(v[2]) / df_value(v[3]));
        state->code = fin ? PCLOTH_ERR_BREAKDOWN : PCLOTH_ERR_NONFINITE;
        atomicOr(status, fin ? ST_BREAKDOWN : ST_NONFINITE);
      }
    }
    alpha_sh = float(rz / pq);
    flag_sh = stop;
  }
  __syncthreads();
  if (flag_sh) return;
  const float alpha = alpha_sh;
  float arz = 0.f, arr = 0.f;
  while (i < n) {
    const float3 rn = make_float3(fmaf(-alpha, qv.x, rv.x), fmaf(-alpha, qv.y, rv.y),
                                  fmaf(-alpha, qv.z, rv.z));
    const float3 zn = apply_p(pu, pw, rn);
    dv[i] = make_float4(fmaf(alpha, pv.x, dvv.x), fmaf(alpha, pv.y, dvv.y),
                        fmaf(alpha, pv.z, dvv.z), 0.f);
    r[i] = make_float4(rn.x, rn.y, rn.z, 0.f);
    z[i] = make_float4(zn.x, zn.y, zn.z, 0.f);
    arz += dot3(rn, zn);
    arr += dot3(rn, rn);
    i += stride;
    if (i < n) {
      pv = p[i]; qv = q[i]; rv = r[i]; dvv = dv[i]; pu = pinv8[2 * i]; pw = pinv8[2 * i + 1];
    }
  }
  Dfloat o[2] = {df_of(arz), df_of(arr)};
  block_sum_df<kVecThreads, 2>(o, sh);
  if (threadIdx.x == 0) {
    red_out[int64_t(blockIdx.x) * kRedSlots + 0] = df_pack(o[0]);
    red_out[int64_t(blockIdx.x) * kRedSlots + 1] = df_pack(o[1]);
  }
}

// dv (padded) -> caller's float[n][3].
__global__ void unpack_dv(int32_t n, const float4* __restrict__ dv4, float* __restrict__ out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float4 d = dv4[i];
  out[3 * i] = d.x;
  out[3 * i + 1] = d.y;
  out[3 * i + 2] = d.z;
}

// Closes a solve that used all its iterations (or none).
__global__ void __launch_bounds__(kVecThreads)
pcg_finish(int k, double tol2, const float2* __restrict__ red_rz,
           const float2* __restrict__ red_bb, int nrz, PcgState* state) {
  __shared__ float2 sh[33 * 2];
  __shared__ int done_sh;
  if (threadIdx.x == 0) done_sh = state->done;
  __syncthreads();
  if (done_sh) return;
  Dfloat v[2] = {records_share(red_rz, nrz, 1, kVecThreads), records_share(red_bb, nrz, 0, kVecThreads)};
  block_sum_df<kVecThreads, 2>(v, sh);
  if (threadIdx.x == 0) {
    const double rr = df_value(v[0]), bb = df_value(v[1]);
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

int pcg_solve(Handle* h, double tol, int32_t maxit, float* dv_out, int32_t* iterations,
              double* rel_residual) {
  cudaStream_t s = h->stream;
  float4* dv = h->dv4;  // padded; unpacked into dv_out at the end
  const double tol2 = tol * tol;
  const bool prof = h->prof.on;
  const int vg = h->vec_grid;
  if (prof) cudaEventRecord(h->ev[2], s);
  pcg_init<<<vg, kVecThreads, 0, s>>>(h->n, h->rhs, h->pinv8, h->r4, h->z4, dv, h->p4[1],
                                      h->red_upd[0], h->red_init, h->state);
  h->launches += 1;
  int rc = check_launch(h, "pcg init");
  if (rc != PCLOTH_OK) return rc;

  int32_t k = 0;
  int chunk_id = 0, pending = -1;
  h->prof_done_at = INT32_MAX;
  bool done = false;
  const int per = 2 * h->chunk + 1;  // events per chunk slot
  // Profiling mode 1 times the first iteration of every chunk (events around
  // its two launches); mode 2 times every iteration.  Iterations enqueued
  // after convergence return at once and are not counted.
  const bool every = h->prof.mode == 2;
  auto consume = [&](int slot, int launched) {
    if (!prof || launched <= 0) return;
    cudaEvent_t* ev = h->pev.data() + size_t(slot) * per;
    const int timed = every ? launched : 1;
    const int32_t first_k = h->prof_chunk_k[slot];
    for (int j = 0; j < timed; ++j) {
      if (first_k + j >= h->prof_done_at) break;   // launches from here on were no-ops
      float a = 0.f, b = 0.f;
      if (cudaEventElapsedTime(&a, ev[2 * j], ev[2 * j + 1]) == cudaSuccess &&
          cudaEventElapsedTime(&b, ev[2 * j + 1], ev[2 * j + 2]) == cudaSuccess) {
        h->prof.spmv_ms += a;
        h->prof.update_ms += b;
        h->prof.samples += 1;
      }
    }
  };
  int launched_in[2] = {0, 0};
  while (k < maxit && !done) {
    const int slot = chunk_id & 1;
    const int m = std::min<int32_t>(h->chunk, maxit - k);
    cudaEvent_t* ev = h->pev.data() + size_t(slot) * per;
    h->prof_chunk_k[slot] = k;
    for (int j = 0; j < m; ++j, ++k) {
      const bool rec = prof && (every || j == 0);
      if (rec && j == 0) cudaEventRecord(ev[0], s);
      rc = launch_spmv_pcg(h, k, tol);
      if (rc != PCLOTH_OK) return rc;
      if (rec) cudaEventRecord(ev[2 * j + 1], s);
      pcg_update<<<vg, kVecThreads, 0, s>>>(h->n, k, h->p4[k & 1], h->q4, h->pinv8, h->r4, h->z4, dv,
                                            h->red_spmv, h->spmv_grid, h->red_upd[k & 1],
                                            h->red_init, vg, h->red_upd[(k + 1) & 1], h->state,
                                            h->d_status);
      h->launches += 1;
      if (rec) cudaEventRecord(ev[2 * j + 2], s);
    }
    launched_in[slot] = m;
    rc = check_launch(h, "pcg update");
    if (rc != PCLOTH_OK) return rc;
    cudaMemcpyAsync(&h->state_host[slot], h->state, sizeof(PcgState), cudaMemcpyDeviceToHost, s);
    cudaEventRecord(h->chunk_ev[slot], s);
    if (pending >= 0) {
      cudaError_t e = cudaEventSynchronize(h->chunk_ev[pending]);
      if (e != cudaSuccess) return cuda_fail(h, e, "pcg poll");
      if (h->state_host[pending].done) {
        done = true;
        h->prof_done_at = h->state_host[pending].iterations;
      }
      consume(pending, launched_in[pending]);
    }
    pending = slot;
    ++chunk_id;
  }
  if (pending >= 0) {
    cudaError_t e = cudaEventSynchronize(h->chunk_ev[pending]);
    if (e != cudaSuccess) return cuda_fail(h, e, "pcg poll");
    if (h->state_host[pending].done && h->prof_done_at > h->state_host[pending].iterations)
      h->prof_done_at = h->state_host[pending].iterations;
    consume(pending, launched_in[pending]);
  }
  pcg_finish<<<1, kVecThreads, 0, s>>>(k, tol2, h->red_upd[k & 1], h->red_init, vg, h->state);
  h->launches += 1;
  rc = check_launch(h, "pcg finish");
  if (rc != PCLOTH_OK) return rc;
  unpack_dv<<<(h->n + 255) / 256, 256, 0, s>>>(h->n, dv, dv_out);
  h->launches += 1;
  rc = check_launch(h, "dv unpack");
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

// ===========================================================================
// Allocation-free solve.
//
// Some callers cannot allocate GPU memory at the time they need a solve: a
// host application (an animation tool, a game engine) that reserves the
// GPU's memory budget for itself and forbids allocation by plug-ins, or a
// real-time loop in which an allocation's latency, or an allocation that
// fails in the middle of a frame, is not acceptable.  pcloth_solve_bsr3_static
// serves them: it runs the same block-Jacobi PCG kernels as pcloth_solve on a
// BSR3 system the caller already holds, and keeps every work vector, every
// reduction record and the status words in one fixed array compiled into
// this library, so it never calls cudaMalloc, cudaFree or any allocating
// routine.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (about 2.2 MiB) until the process exits, and every call
// on that GPU shares it.  Calls that overlap on the GPU therefore race on it;
// a caller must order them (one stream, or events).  Each call re-initialises
// everything it reads before reading it, so nothing leaks from one call into
// the next.
// ===========================================================================
namespace {

constexpr int64_t kStaticVec = int64_t(PCLOTH_STATIC_MAX_VERTS) + 64;  // float4 per vector
constexpr int kStaticMaxRecords = 1024;                                 // per reduction buffer
constexpr size_t kStaticBytes =
    sizeof(float4) * size_t(2 * kStaticVec        // block-Jacobi inverses (2 per vertex)
                            + 5 * kStaticVec)     // dv, r, z, q and the spare p
    + sizeof(float4) * size_t(kStaticVec)         // second p (ping-pong)
    + sizeof(float2) * size_t(kRedSlots) * size_t(4 * kStaticMaxRecords) + 256;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

// Device address of g_static_scratch per device ordinal (set up on first use).
void* g_static_addr[64] = {};

// Inverse of the diagonal block of each row of a caller's BSR3 matrix, packed
// like the library's own: (P00 P01 P02 P11) (P12 P22 0 0).  A row without a
// diagonal block, or with a non-invertible one, is reported as non-finite.
__global__ void bsr3_diag_inverse(int32_t n, const int32_t* __restrict__ rowptr,
                                  const int32_t* __restrict__ colind,
                                  const float* __restrict__ vals, float4* __restrict__ pinv8,
                                  uint32_t* status) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int32_t lo = rowptr[i], hi = rowptr[i + 1];
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (colind[mid] < i) lo = mid + 1; else hi = mid;
  }
  float det = 0.f, c00 = 0.f, c01 = 0.f, c02 = 0.f, c11 = 0.f, c12 = 0.f, c22 = 0.f;
  if (lo < rowptr[i + 1] && colind[lo] == i) {
    const float* D = vals + 9 * int64_t(lo);
    c00 = D[4] * D[8] - D[5] * D[7];
    c01 = D[5] * D[6] - D[3] * D[8];
    c02 = D[3] * D[7] - D[4] * D[6];
    c11 = D[0] * D[8] - D[2] * D[6];
    c12 = D[2] * D[3] - D[0] * D[5];
    c22 = D[0] * D[4] - D[1] * D[3];
    det = D[0] * c00 + D[1] * c01 + D[2] * c02;
  }
  if (!(det > 0.f) || !isfinite(det)) {
    atomicOr(status, ST_NONFINITE);
    det = 1.f;
  }
  const float id = 1.0f / det;
  pinv8[2 * i] = make_float4(c00 * id, c01 * id, c02 * id, c11 * id);
  pinv8[2 * i + 1] = make_float4(c12 * id, c22 * id, 0.f, 0.f);
}

}  // namespace

int pcg_solve_static(int32_t n, const int32_t* rowptr, const int32_t* colind, const float* vals,
                     const float* b, double tol, int32_t maxit, float* dv_out,
                     int32_t* iterations, double* rel_residual, cudaStream_t stream) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
  if (device < 0 || device >= 64) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "device ordinal");
  if (!g_static_addr[device]) {
    // g_static_scratch names a host-side stand-in here; the kernels need the
    // array's device address on this device.
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetSymbolAddress(scratch)");
    g_static_addr[device] = ptr;
  }
  // A stack handle pointing into the fixed array and the caller's buffers:
  // its containers stay empty and nothing in it is allocated or freed.
  Handle h;
  h.device = device;
  h.stream = stream;
  h.n = n;
  h.chunk = 32;
  cudaDeviceGetAttribute(&h.sm_count, cudaDevAttrMultiProcessorCount, device);
  if (h.sm_count <= 0) h.sm_count = 1;
  h.spmv_grid = spmv_grid_for(n, h.sm_count);
  h.vec_grid = int(std::min<int64_t>((int64_t(n) + kVecThreads - 1) / kVecThreads,
                                     int64_t(h.sm_count) * 4));
  if (h.spmv_grid > kStaticMaxRecords || h.vec_grid > kStaticMaxRecords)
    return fail(nullptr, PCLOTH_ERR_CAPACITY, "too many CTAs for the fixed reduction records");
  unsigned char* base = static_cast<unsigned char*>(g_static_addr[device]);
  float4* v4 = reinterpret_cast<float4*>(base);
  h.pinv8 = v4;
  h.dv4 = v4 + 2 * kStaticVec;
  h.r4 = v4 + 3 * kStaticVec;
  h.z4 = v4 + 4 * kStaticVec;
  h.q4 = v4 + 5 * kStaticVec;
  h.p4[0] = v4 + 6 * kStaticVec;
  h.p4[1] = v4 + 7 * kStaticVec;
  float2* rec = reinterpret_cast<float2*>(v4 + 8 * kStaticVec);
  h.red_spmv = rec;
  h.red_upd[0] = rec + size_t(kRedSlots) * kStaticMaxRecords;
  h.red_upd[1] = rec + size_t(2 * kRedSlots) * kStaticMaxRecords;
  h.red_init = rec + size_t(3 * kRedSlots) * kStaticMaxRecords;
  unsigned char* tail = reinterpret_cast<unsigned char*>(rec + size_t(4 * kRedSlots) * kStaticMaxRecords);
  h.state = reinterpret_cast<PcgState*>(tail);
  h.d_status = reinterpret_cast<uint32_t*>(tail + 64);
  h.rowptr = const_cast<int32_t*>(rowptr);
  h.colind = const_cast<int32_t*>(colind);
  h.vals = const_cast<float*>(vals);
  h.blk = 9;   // the caller's blocks are general row-major 3x3
  h.rhs = const_cast<float*>(b);

  const int vg = h.vec_grid;
  e = cudaMemsetAsync(h.d_status, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "status reset");
  bsr3_diag_inverse<<<(n + 255) / 256, 256, 0, stream>>>(n, rowptr, colind, vals, h.pinv8,
                                                        h.d_status);
  pcg_init<<<vg, kVecThreads, 0, stream>>>(n, b, h.pinv8, h.r4, h.z4, h.dv4, h.p4[1],
                                           h.red_upd[0], h.red_init, h.state);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "static solve launch");
  PcgState st{};
  int32_t k = 0;
  while (k < maxit) {
    const int m = std::min<int32_t>(h.chunk, maxit - k);
    for (int j = 0; j < m; ++j, ++k) {
      if (launch_spmv_pcg(&h, k, tol) != PCLOTH_OK) return fail(nullptr, PCLOTH_ERR_CUDA, h.err);
      pcg_update<<<vg, kVecThreads, 0, stream>>>(n, k, h.p4[k & 1], h.q4, h.pinv8, h.r4, h.z4,
                                                 h.dv4, h.red_spmv, h.spmv_grid,
                                                 h.red_upd[k & 1], h.red_init, vg,
                                                 h.red_upd[(k + 1) & 1], h.state, h.d_status);
    }
    e = cudaMemcpyAsync(&st, h.state, sizeof(PcgState), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "static solve poll");
    if (st.done) break;
  }
  pcg_finish<<<1, kVecThreads, 0, stream>>>(k, tol * tol, h.red_upd[k & 1], h.red_init, vg, h.state);
  unpack_dv<<<(n + 255) / 256, 256, 0, stream>>>(n, h.dv4, dv_out);
  uint32_t status = 0;
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(&st, h.state, sizeof(PcgState), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&status, h.d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "static solve result");
  if (iterations) *iterations = st.iterations;
  if (rel_residual) *rel_residual = st.relres;
  if (status & ST_WAIT_TIMEOUT) return fail(nullptr, PCLOTH_ERR_CUDA, "device wait timed out");
  if (status & ST_NONFINITE)
    return fail(nullptr, PCLOTH_ERR_NONFINITE, "non-finite value or missing/singular diagonal block");
  if (st.code == PCLOTH_ERR_BREAKDOWN) return fail(nullptr, st.code, "PCG breakdown");
  if (st.code == PCLOTH_ERR_NONFINITE) return fail(nullptr, st.code, "non-finite value in PCG");
  return st.code;
}

}  // namespace pcloth_impl
