// Block-Jacobi preconditioned conjugate gradients on A dv = b (P-Cloth,
// arXiv 2008.00409, Sec. 2.5 Eq. (3) and Sec. 3.1: the linear system of each
// step is solved by PCG; the pages do not name the preconditioner, this uses
// the inverses of the 3x3 diagonal blocks), plus the backward-Euler state
// update v += dv, x += h v.
//
// The whole solve is one persistent kernel, launched cooperatively so that
// all of its CTAs are resident at once.  Each CTA owns the rows of its SpMV
// tiles (blockIdx.x, +gridDim.x, ...) in every phase, and the phases of an
// iteration are separated by grid-wide barriers:
//
//   S  q = A p (the streaming SpMV of spmv_pipe.cuh, gathering p only);
//      partial p.q over the CTA's rows                              barrier
//   U  alpha = r.z / p.q; r -= alpha q; z = P r; partials r.z, r.r  barrier
//   P  dv += alpha p; stop if |r| <= tol |b| (or breakdown, or maxit);
//      otherwise beta = r.z / r.z_old and p = z + beta p            barrier
//
// (dv is updated in P rather than U: both it and the new direction read the
// same p, so each row's p is read once per iteration.)
//
// Every scalar is formed by every CTA from the same per-CTA partials in the
// same order (double-float sums), so all CTAs take the same decisions and
// the solve is bitwise reproducible.  No host round trip happens inside the
// solve.  A barrier's arrival and wait are separate, and a CTA uses the time
// between them for work that needs nothing from the other CTAs: before U and
// P each thread loads its first rows of the phase, before S thread 0 issues
// the next SpMV's first stages.
//
// Every wait (mbarrier, grid barrier) is bounded in time: on a timeout the
// CTA records ST_WAIT_TIMEOUT and marks its next barrier arrival, so that
// every CTA leaves the loop at that barrier; each then waits (bounded) for
// its own copies in flight and returns, and the host reports an error.

#include <algorithm>

#include "spmv_pipe.cuh"


namespace pcloth_impl {
namespace {

// The SpMV's gathers of p carry an L2 evict-last policy, so that the matrix
// streamed past them (evict-first) does not push p out.
struct Vec {
  uint64_t pol;
  __device__ __forceinline__ float4 ld(const float4* p) const { return ld_policy(p, pol); }
};

__device__ __forceinline__ Vec vec_access() { return Vec{policy_evict_last()}; }

// Row i of a vector stored as three planes (x, y, z) of vs floats.
__device__ __forceinline__ float3 ld3(const float* __restrict__ v, int64_t vs, int64_t i) {
  return make_float3(v[i], v[vs + i], v[2 * vs + i]);
}

__device__ __forceinline__ void st3(float* __restrict__ v, int64_t vs, int64_t i, float3 x) {
  v[i] = x.x;
  v[vs + i] = x.y;
  v[2 * vs + i] = x.z;
}

// The symmetric block-Jacobi inverse of row i, stored as six planes.
struct Sym3 {
  float p00, p01, p02, p11, p12, p22;
};

__device__ __forceinline__ Sym3 ld_sym(const float* __restrict__ v, int64_t vs, int64_t i) {
  return Sym3{v[i], v[vs + i], v[2 * vs + i], v[3 * vs + i], v[4 * vs + i], v[5 * vs + i]};
}

__device__ __forceinline__ float3 apply_p(const Sym3& P, float3 r) {
  return make_float3(fmaf(P.p00, r.x, fmaf(P.p01, r.y, P.p02 * r.z)),
                     fmaf(P.p01, r.x, fmaf(P.p11, r.y, P.p12 * r.z)),
                     fmaf(P.p02, r.x, fmaf(P.p12, r.y, P.p22 * r.z)));
}

__device__ __forceinline__ float dot3(float3 a, float3 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, a.z * b.z));
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// A CTA in which a wait timed out adds kPoison to the barrier counter with
// its next arrival, so that every CTA sees the timeout in the value that
// completes its own wait: the arrivals are counted in the bits below.
constexpr unsigned long long kPoison = 1ull << 40;

// Polls the counter until its arrival count reaches `target`; false once
// `limit_ns` has passed.  *seen: the last value read.
__device__ __forceinline__ bool poll_bounded(const unsigned long long* counter,
                                             unsigned long long target, uint64_t limit_ns,
                                             unsigned long long* seen) {
  unsigned long long v = ld_acquire(counter);
  if ((v & (kPoison - 1)) < target) {
    const uint64_t t0 = now_ns();
    while (((v = ld_acquire(counter)) & (kPoison - 1)) < target)
      if (now_ns() - t0 > limit_ns) {
        *seen = v;
        return false;
      }
  }
  *seen = v;
  return true;
}

// Grid-wide barrier.  Every CTA adds 1 to the counter (zeroed before the
// launch) once per barrier, so the b-th barrier is complete when the
// arrivals reach b * gridDim.x.  Thread 0 arrives with a release add and
// waits with acquire loads, and the CTA barriers on both sides carry the
// ordering to its other threads: each CTA's writes before the barrier are
// visible to every CTA after it.  Returns false, the same in every thread of
// the CTA, if the wait ran past kWaitNs or any CTA of the grid arrived
// poisoned (fail_sh set: one of its waits timed out); the caller then
// leaves its loop.
//
// The barrier comes in two halves, so that a CTA can load its own rows for
// the next phase between its arrival and its wait (grid_arrive, then
// grid_wait; grid_barrier is both).  epoch is thread 0's.
__device__ __forceinline__ void grid_arrive(unsigned long long* bar, unsigned long long& epoch,
                                            const int* fail_sh) {
  __syncthreads();
  if (threadIdx.x == 0) {
    ++epoch;
    const unsigned long long inc = 1ull + (*fail_sh ? kPoison : 0ull);
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(bar), "l"(inc) : "memory");
  }
}

__device__ __forceinline__ bool grid_wait(const unsigned long long* bar,
                                          const unsigned long long& epoch, int* ok_sh) {
  if (threadIdx.x == 0) {
    unsigned long long v = 0;
    const bool ok = poll_bounded(bar, epoch * gridDim.x, kWaitNs, &v);
    *ok_sh = ok && v < kPoison;
  }
  __syncthreads();
  return *ok_sh != 0;
}

__device__ __forceinline__ bool grid_barrier(unsigned long long* bar, unsigned long long& epoch,
                                             const int* fail_sh, int* ok_sh) {
  grid_arrive(bar, epoch, fail_sh);
  return grid_wait(bar, epoch, ok_sh);
}

// Records a wait that gave up: in the status word for the host, and in the
// CTA's flag, which poisons its next barrier arrival.
__device__ __forceinline__ void timed_out(uint32_t* status, int* fail_sh) {
  atomicOr(status, ST_WAIT_TIMEOUT);
  *fail_sh = 1;
}

constexpr int kTileCache = 256;   // tiles per CTA whose block ranges stay in shared memory
// Rows per thread of the update and direction phases loaded between the CTA's
// barrier arrival and its wait (they are its own rows and need no scalar).
// Each row moves about 3.7 MB of the phase's traffic into the wait on the
// 1.65M-triangle cloth, about 0.5 us per iteration; five rows spill.
#ifndef PCLOTH_PCG_PRE
#define PCLOTH_PCG_PRE 4
#endif
constexpr int kPreRows = PCLOTH_PCG_PRE;
static_assert(kPreRows >= 1, "at least one row loads under the barrier");
// Stages of the next SpMV that thread 0 issues between its CTA's arrival at
// the direction phase's barrier and its wait: the matrix does not change, so
// the copies need nothing from the other CTAs.  Two beat one and three on
// the 1.65M-triangle cloth (67.9 against 69.5 and 68.6 us per iteration).
#ifndef PCLOTH_PCG_EARLY
#define PCLOTH_PCG_EARLY 2
#endif
constexpr int kEarlyStages = PCLOTH_PCG_EARLY;

struct LoopArgs {
  PipeMatrix m;
  const float* b;          // float[n][3]
  const float* pinv;       // [6][vs] planes P00 P01 P02 P11 P12 P22
  float* dv;               // [3][vs] planes x, y, z
  float* r;                // [3][vs]
  float* z;                // [3][vs]
  float4* p;               // one float4 per vertex: the SpMV gathers it
  float* q;                // [3][vs]
  int64_t vs;              // floats per plane
  float2* rec;             // [gridDim.x][kRecSlots]
  unsigned long long* bar; // grid-barrier counter, zero at launch
  PcgState* state;
  uint32_t* status;
  float* dv_out;           // caller's float[n][3]
  const float* x0;         // caller's float[n][3] initial guess (the kGuess kernel only)
  unsigned long long* phase_ns;  // [4] = S, U, P nanoseconds, timed SpMV phases (or null)
  double tol2;
  int32_t maxit;
};

// The CTA's rows: slot f is row (f % kPipeRows) of its tile number f / kPipeRows.
__device__ __forceinline__ int32_t own_row(int32_t f) {
  return (int32_t(blockIdx.x) + (f / kPipeRows) * int32_t(gridDim.x)) * kPipeRows +
         f % kPipeRows;
}

struct PGather {
  const float4* p;
  Vec vm;
  __device__ __forceinline__ float3 operator()(int32_t col) const {
    const float4 v = vm.ld(p + col);
    return make_float3(v.x, v.y, v.z);
  }
};

struct PEpi {
  const float4* p;
  float* q;
  int64_t vs;
  Vec vm;
  float pq;
  float4 pr;   // p of this thread's row, loaded when its tile starts
  __device__ __forceinline__ void begin(int32_t row) { pr = vm.ld(p + row); }
  __device__ __forceinline__ void operator()(int32_t row, float3 acc) {
    st3(q, vs, row, acc);
    pq = fmaf(pr.x, acc.x, fmaf(pr.y, acc.y, fmaf(pr.z, acc.z, pq)));
  }
};

// State that only thread 0 of a CTA uses (the producer lane, the grid
// barrier, the scalar decisions, the phase timers), kept in shared memory so
// that it takes no registers in the other threads.  Thread 0 copies the
// producer's cursor into registers for each stretch of stage issues.
struct Lead {
  Producer P;
  unsigned long long epoch, t_s, t_u, t_p, n_timed, t_prev;
  double rz_old, bbd, rr_last;
};

// Start of a solve from the caller's guess x0 (P-Cloth Sec. 3.1's PCG with a
// nonzero first iterate): dv = x0, r = b - A x0 (one SpMV pass of the same
// pipeline), z = P r, p = z.  A guess that already meets |r| <= tol |b|
// stops with 0 iterations (and b = 0 gives dv = 0, whatever the guess).
// Returns whether the iteration runs; every CTA takes the same decision from
// the same records.  *stop_sh and *zero_sh are the CTA's shared flags.
template <int BW>
__device__ __forceinline__ bool start_from_guess(const LoopArgs& a, const PipeMatrix& m,
                                                 const PipeShared& sh, Consumer& C, Lead& L,
                                                 int32_t n, int32_t nslots, float2* my_rec,
                                                 float2* red_sh, int* ok_sh, int* fail_sh,
                                                 int* stop_sh, int* zero_sh) {
  const int32_t tid = threadIdx.x;
  // p = x0 (the SpMV below gathers it), dv = x0
  for (int32_t f = tid; f < nslots; f += kPipeThreads) {
    const int32_t i = own_row(f);
    if (i >= n) continue;
    const float3 x = make_float3(a.x0[3 * int64_t(i)], a.x0[3 * int64_t(i) + 1],
                                 a.x0[3 * int64_t(i) + 2]);
    a.p[i] = make_float4(x.x, x.y, x.z, 0.f);
    st3(a.dv, a.vs, i, x);
  }
  if (!grid_barrier(a.bar, L.epoch, fail_sh, ok_sh)) return false;
  // q = A x0: one pass of the streaming product
  if (tid < 32) {
    if (tid == 0) {
      Producer P = L.P;
      if (!producer_pass<BW>(P, sh, m)) timed_out(a.status, fail_sh);
      L.P = P;
    }
  } else {
    const Vec vm = vec_access();
    PGather g{a.p, vm};
    PEpi e{a.p, a.q, a.vs, vm, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
    if (!consumer_pass<BW>(C, sh, g, e)) timed_out(a.status, fail_sh);
  }
  __syncthreads();   // this CTA's rows of q are written
  // r = b - A x0, z = P r; partials r.z, b.b, r.r
  {
    float rz = 0.f, bb = 0.f, rr = 0.f;
    for (int32_t f = tid; f < nslots; f += kPipeThreads) {
      const int32_t i = own_row(f);
      if (i >= n) continue;
      const float3 bv = make_float3(a.b[3 * int64_t(i)], a.b[3 * int64_t(i) + 1],
                                    a.b[3 * int64_t(i) + 2]);
      const float3 qv = ld3(a.q, a.vs, i);
      const float3 rv = make_float3(bv.x - qv.x, bv.y - qv.y, bv.z - qv.z);
      const float3 zv = apply_p(ld_sym(a.pinv, a.vs, i), rv);
      st3(a.r, a.vs, i, rv);
      st3(a.z, a.vs, i, zv);
      rz += dot3(rv, zv);
      bb += dot3(bv, bv);
      rr += dot3(rv, rv);
    }
    Dfloat v[2] = {df_of(rz), df_of(bb)};
    block_sum_df0<kPipeThreads, 2>(v, red_sh);
    if (tid == 0) {
      my_rec[REC_RZ] = df_pack(v[0]);
      my_rec[REC_BB] = df_pack(v[1]);
    }
    __syncthreads();
    Dfloat w[1] = {df_of(rr)};
    block_sum_df0<kPipeThreads, 1>(w, red_sh);
    if (tid == 0) my_rec[REC_RR] = df_pack(w[0]);
  }
  if (!grid_barrier(a.bar, L.epoch, fail_sh, ok_sh)) return false;
  {
    Dfloat rzrr[2], bb[1];
    records_share<2>(a.rec, gridDim.x, REC_RZ, kPipeThreads, rzrr);
    records_share<1>(a.rec, gridDim.x, REC_BB, kPipeThreads, bb);
    Dfloat v[2] = {rzrr[0], bb[0]};
    block_sum_df0<kPipeThreads, 2>(v, red_sh);
    if (tid == 0) {
      L.rz_old = df_value(v[0]);
      L.bbd = df_value(v[1]);
    }
    __syncthreads();
    Dfloat w[1] = {rzrr[1]};
    block_sum_df0<kPipeThreads, 1>(w, red_sh);
    if (tid == 0) {
      const double rzd = L.rz_old, bbd = L.bbd, rrd = df_value(w[0]);
      L.rr_last = rrd;
      int stop = 1;
      PcgState st{1, 0, PCLOTH_OK, 0, 0.0, sqrt(bbd)};
      if (!isfinite(bbd) || !isfinite(rrd) || !isfinite(rzd)) {
        st.code = PCLOTH_ERR_NONFINITE;
        if (blockIdx.x == 0) atomicOr(a.status, ST_NONFINITE);
      } else if (!(bbd > 0.0)) {
        *zero_sh = 1;                      // b = 0: dv = 0 is exact
      } else {
        st.relres = sqrt(rrd / bbd);
        if (rrd <= a.tol2 * bbd)
          st.code = PCLOTH_OK;             // the guess already meets the tolerance
        else if (a.maxit <= 0)
          st.code = PCLOTH_NOT_CONVERGED;
        else
          stop = 0;
      }
      if (stop && blockIdx.x == 0) *a.state = st;
      *stop_sh = stop;
    }
    __syncthreads();
  }
  if (*stop_sh) return false;
  // p = z; the loop's first product gathers it only after the next barrier
  for (int32_t f = tid; f < nslots; f += kPipeThreads) {
    const int32_t i = own_row(f);
    if (i >= n) continue;
    const float3 zv = ld3(a.z, a.vs, i);
    a.p[i] = make_float4(zv.x, zv.y, zv.z, 0.f);
  }
  if (!grid_barrier(a.bar, L.epoch, fail_sh, ok_sh)) return false;
  if (tid == 0) {   // the first stages of the first SpMV
    Producer P = L.P;
    for (int j = 0; j < kPipeStages && !P.ended; ++j)
      if (producer_step<BW>(P, sh, m) < 0) timed_out(a.status, fail_sh);
    L.P = P;
  }
  __syncthreads();
  return true;
}

// kGuess: the solve starts from the caller's guess x0 instead of 0 -- one
// extra SpMV pass and two extra grid barriers before the loop; the loop
// itself is the same code.
template <int BW, bool kGuess>
__global__ void __launch_bounds__(kPipeThreads, kPipeCtasPerSm)
pcg_loop(LoopArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const PipeShared sh = pipe_shared<BW>(smem);
  __shared__ float2 red_sh[33 * 2];
  __shared__ int ok_sh;
  __shared__ int fail_sh;   // a wait of this CTA timed out
  __shared__ int stop_sh;
  __shared__ float scal_sh;
  __shared__ int zero_sh;   // b = 0: dv = 0 is exact, whatever the guess
  __shared__ Lead L;
  // every SpMV pass walks the same tiles: their block ranges, once
  __shared__ int2 tb_sh[kTileCache];
  PipeMatrix m = a.m;
  m.tb = tb_sh;
  m.ntb = fill_tile_bounds(m, tb_sh, kTileCache);
  pipe_init(sh);
  __syncthreads();

  const int32_t n = a.m.n;
  const int32_t tid = threadIdx.x;
  const int32_t my_tiles = (a.m.ntiles - int32_t(blockIdx.x) + int32_t(gridDim.x) - 1) /
                           int32_t(gridDim.x);
  const int32_t nslots = my_tiles * kPipeRows;
  float2* my_rec = a.rec + size_t(blockIdx.x) * kRecSlots;
  const bool timer = a.phase_ns != nullptr && blockIdx.x == 0 && tid == 0;
  Consumer C;
  if (tid == 0) {
    fail_sh = 0;
    zero_sh = 0;
    producer_begin(L.P, m);
    L.epoch = L.t_s = L.t_u = L.t_p = L.n_timed = L.t_prev = 0;
  }
  consumer_begin(C);

  bool run;
  if constexpr (kGuess) {
    run = start_from_guess<BW>(a, m, sh, C, L, n, nslots, my_rec, red_sh, &ok_sh, &fail_sh,
                               &stop_sh, &zero_sh);
  } else {
    // ---- init: r = b, z = P b, dv = 0, p = z; partials r.z and b.b ---------
    {
      float rz = 0.f, bb = 0.f;
      for (int32_t f = tid; f < nslots; f += kPipeThreads) {
        const int32_t i = own_row(f);
        if (i >= n) continue;
        const float3 bv = make_float3(a.b[3 * int64_t(i)], a.b[3 * int64_t(i) + 1],
                                      a.b[3 * int64_t(i) + 2]);
        const float3 zv = apply_p(ld_sym(a.pinv, a.vs, i), bv);
        st3(a.r, a.vs, i, bv);
        st3(a.z, a.vs, i, zv);
        a.p[i] = make_float4(zv.x, zv.y, zv.z, 0.f);
        st3(a.dv, a.vs, i, make_float3(0.f, 0.f, 0.f));
        rz += dot3(bv, zv);
        bb += dot3(bv, bv);
      }
      Dfloat v[2] = {df_of(rz), df_of(bb)};
      block_sum_df0<kPipeThreads, 2>(v, red_sh);
      if (tid == 0) {
        my_rec[REC_RZ] = df_pack(v[0]);
        my_rec[REC_BB] = df_pack(v[1]);
      }
    }
    run = grid_barrier(a.bar, L.epoch, &fail_sh, &ok_sh);

    if (run) {
      Dfloat v[2], rz[1], bb[1];
      records_share<1>(a.rec, gridDim.x, REC_RZ, kPipeThreads, rz);
      records_share<1>(a.rec, gridDim.x, REC_BB, kPipeThreads, bb);
      v[0] = rz[0];
      v[1] = bb[0];
      block_sum_df0<kPipeThreads, 2>(v, red_sh);
      if (tid == 0) {
        const double bbd = df_value(v[1]);
        L.rz_old = df_value(v[0]);
        L.bbd = bbd;
        L.rr_last = bbd;
        int stop = 1;
        PcgState st{1, 0, PCLOTH_OK, 0, 0.0, sqrt(bbd)};
        if (!isfinite(bbd)) {
          st.code = PCLOTH_ERR_NONFINITE;
          if (blockIdx.x == 0) atomicOr(a.status, ST_NONFINITE);
        } else if (!(bbd > 0.0)) {
          st.code = PCLOTH_OK;             // b = 0: dv = 0 is exact
        } else if (a.maxit <= 0) {
          st.relres = 1.0;
          st.code = (1.0 <= a.tol2) ? PCLOTH_OK : PCLOTH_NOT_CONVERGED;
        } else {
          stop = 0;
        }
        if (stop && blockIdx.x == 0) *a.state = st;
        stop_sh = stop;
        // the first stages of the first SpMV
        if (!stop) {
          Producer P = L.P;
          for (int j = 0; j < kPipeStages && !P.ended; ++j)
            if (producer_step<BW>(P, sh, m) < 0) timed_out(a.status, &fail_sh);
          L.P = P;
        }
      }
      __syncthreads();
      run = stop_sh == 0;
    }
  }

  if (timer) L.t_prev = now_ns();
  for (int32_t k = 0; run; ++k) {
    // ---- S: q = A p, partial p.q ------------------------------------------
    float pq = 0.f;
    if (tid < 32) {
      if (tid == 0) {
        Producer P = L.P;
        if (!producer_pass<BW>(P, sh, m)) timed_out(a.status, &fail_sh);
        L.P = P;
      }
    } else {
      const Vec vm = vec_access();
      PGather g{a.p, vm};
      PEpi e{a.p, a.q, a.vs, vm, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
      if (!consumer_pass<BW>(C, sh, g, e)) timed_out(a.status, &fail_sh);
      pq = e.pq;
    }
    {
      Dfloat t[1] = {df_of(pq)};
      block_sum_df0<kPipeThreads, 1>(t, red_sh);
      if (tid == 0) my_rec[REC_PQ] = df_pack(t[0]);
    }
    grid_arrive(a.bar, L.epoch, &fail_sh);
    // The update's first kPreRows rows of this thread: their inputs are this
    // CTA's own rows and do not depend on alpha, so they load while the other
    // CTAs arrive.  (Rows grow with the slot; past the end, i = n.)
    int32_t i_pre[kPreRows];
    float3 q_pre[kPreRows], r_pre[kPreRows];
    Sym3 s_pre[kPreRows];
#pragma unroll
    for (int u = 0; u < kPreRows; ++u) {
      const int32_t f = tid + u * kPipeThreads;
      i_pre[u] = f < nslots ? min(own_row(f), n) : n;
      q_pre[u] = r_pre[u] = make_float3(0.f, 0.f, 0.f);
      s_pre[u] = Sym3{0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (i_pre[u] < n) {
        q_pre[u] = ld3(a.q, a.vs, i_pre[u]);
        r_pre[u] = ld3(a.r, a.vs, i_pre[u]);
        s_pre[u] = ld_sym(a.pinv, a.vs, i_pre[u]);
      }
    }
    if (!grid_wait(a.bar, L.epoch, &ok_sh)) break;
    if (timer) {
      const unsigned long long t = now_ns();
      L.t_s += t - L.t_prev;
      L.t_prev = t;
      ++L.n_timed;
    }

    // ---- U: alpha; r, z; partials r.z, r.r ----------------------------------
    {
      Dfloat v[1];
      records_share<1>(a.rec, gridDim.x, REC_PQ, kPipeThreads, v);
      block_sum_df0<kPipeThreads, 1>(v, red_sh);
      if (tid == 0) {
        const double pqd = df_value(v[0]), rz_old = L.rz_old, bbd = L.bbd;
        int stop = 0;
        if (!(pqd > 0.0) || !isfinite(pqd) || !isfinite(rz_old)) {
          stop = 1;
          const bool fin = isfinite(pqd) && isfinite(rz_old);
          if (blockIdx.x == 0) {
            *a.state = PcgState{1, k, fin ? PCLOTH_ERR_BREAKDOWN : PCLOTH_ERR_NONFINITE, 0,
                                sqrt(L.rr_last / bbd), sqrt(bbd)};
            atomicOr(a.status, fin ? ST_BREAKDOWN : ST_NONFINITE);
          }
        }
        // alpha in fp32 from the fp64-rounded sums: the vectors are updated
        // in fp32 anyway, and an fp64 division is a slow path on this GPU
        scal_sh = float(rz_old) / float(pqd);
        stop_sh = stop;
      }
      __syncthreads();
    }
    if (stop_sh) break;
    const float alpha = scal_sh;
    // z of the preloaded rows stays in registers for the direction phase (the
    // same thread updates the same rows there): 24 bytes a row saved, 0.7 us
    // per iteration on the 1.65M-triangle cloth
    float3 z_pre[kPreRows];
    {
      float arz = 0.f, arr = 0.f;
      {
        const float* __restrict__ qv_ = a.q;
        const float* __restrict__ pinv = a.pinv;
        float* __restrict__ rv_ = a.r;
        float* __restrict__ zv_ = a.z;
        const int64_t vs = a.vs;
#pragma unroll
        for (int u = 0; u < kPreRows; ++u) {
          if (i_pre[u] < n) {
            const float3 rn = make_float3(fmaf(-alpha, q_pre[u].x, r_pre[u].x),
                                          fmaf(-alpha, q_pre[u].y, r_pre[u].y),
                                          fmaf(-alpha, q_pre[u].z, r_pre[u].z));
            const float3 zn = apply_p(s_pre[u], rn);
            st3(rv_, vs, i_pre[u], rn);
            z_pre[u] = zn;
            arz += dot3(rn, zn);
            arr += dot3(rn, rn);
          }
        }
#pragma unroll 2
        for (int32_t f = tid + kPreRows * kPipeThreads; f < nslots; f += kPipeThreads) {
          const int32_t i = own_row(f);
          if (i >= n) break;   // rows grow with f: the rest are past the end too
          const float3 qv = ld3(qv_, vs, i), rv = ld3(rv_, vs, i);
          const Sym3 P = ld_sym(pinv, vs, i);
          const float3 rn = make_float3(fmaf(-alpha, qv.x, rv.x), fmaf(-alpha, qv.y, rv.y),
                                        fmaf(-alpha, qv.z, rv.z));
          const float3 zn = apply_p(P, rn);
          st3(rv_, vs, i, rn);
          st3(zv_, vs, i, zn);
          arz += dot3(rn, zn);
          arr += dot3(rn, rn);
        }
      }
      Dfloat o[2] = {df_of(arz), df_of(arr)};
      block_sum_df0<kPipeThreads, 2>(o, red_sh);
      if (tid == 0) {
        my_rec[REC_RZ] = df_pack(o[0]);
        my_rec[REC_RR] = df_pack(o[1]);
      }
    }
    grid_arrive(a.bar, L.epoch, &fail_sh);
    // the direction phase's first kPreRows rows (the update's: their z is
    // still in registers), loaded while the other CTAs arrive
    float4 p_pre[kPreRows];
    float3 d_pre[kPreRows];
#pragma unroll
    for (int u = 0; u < kPreRows; ++u) {
      p_pre[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      d_pre[u] = make_float3(0.f, 0.f, 0.f);
      if (i_pre[u] < n) {
        p_pre[u] = a.p[i_pre[u]];
        d_pre[u] = ld3(a.dv, a.vs, i_pre[u]);
      }
    }
    if (!grid_wait(a.bar, L.epoch, &ok_sh)) break;
    if (timer) {
      const unsigned long long t = now_ns();
      L.t_u += t - L.t_prev;
      L.t_prev = t;
    }

    // ---- P: convergence, beta; dv += alpha p, p = z + beta p ------------------
    {
      static_assert(REC_RR == REC_RZ + 1 && REC_RZ % 2 == 0, "r.z, r.r: one 16-byte load");
      Dfloat v[2];
      records_share<2>(a.rec, gridDim.x, REC_RZ, kPipeThreads, v);
      block_sum_df0<kPipeThreads, 2>(v, red_sh);
      if (tid == 0) {
        const double rz = df_value(v[0]), rr = df_value(v[1]);
        const double rz_old = L.rz_old, bbd = L.bbd;
        const bool conv = rr <= a.tol2 * bbd;
        const bool bad = !isfinite(rr) || !isfinite(rz) || !(rz > 0.0) || !(rz_old > 0.0);
        int stop = 1;
        int code = PCLOTH_OK;
        if (conv) {
          code = PCLOTH_OK;
        } else if (bad) {
          code = (isfinite(rr) && isfinite(rz)) ? PCLOTH_ERR_BREAKDOWN : PCLOTH_ERR_NONFINITE;
          if (blockIdx.x == 0)
            atomicOr(a.status, code == PCLOTH_ERR_BREAKDOWN ? ST_BREAKDOWN : ST_NONFINITE);
        } else if (k + 1 >= a.maxit) {
          code = PCLOTH_NOT_CONVERGED;
        } else {
          stop = 0;
        }
        if (stop && blockIdx.x == 0)
          *a.state = PcgState{1, k + 1, code, 0, sqrt(rr / bbd), sqrt(bbd)};
        scal_sh = float(rz) / float(rz_old);   // beta, likewise in fp32
        stop_sh = stop;
        L.rr_last = rr;
        L.rz_old = rz;
      }
      __syncthreads();
    }
    // dv += alpha p_k (every exit from here on keeps it), then, to go on,
    // p_{k+1} = z_{k+1} + beta p_k
    const bool stop = stop_sh != 0;
    {
      const float beta = scal_sh;
      float4* __restrict__ pv_ = a.p;
      float* __restrict__ dv_ = a.dv;
      const float* __restrict__ zv_ = a.z;
      const int64_t vs = a.vs;
#pragma unroll
      for (int u = 0; u < kPreRows; ++u) {
        if (i_pre[u] < n) {
          const float4 pv = p_pre[u];
          st3(dv_, vs, i_pre[u],
              make_float3(fmaf(alpha, pv.x, d_pre[u].x), fmaf(alpha, pv.y, d_pre[u].y),
                          fmaf(alpha, pv.z, d_pre[u].z)));
          if (!stop)
            pv_[i_pre[u]] = make_float4(fmaf(beta, pv.x, z_pre[u].x),
                                        fmaf(beta, pv.y, z_pre[u].y),
                                        fmaf(beta, pv.z, z_pre[u].z), 0.f);
        }
      }
#pragma unroll 2
      for (int32_t f = tid + kPreRows * kPipeThreads; f < nslots; f += kPipeThreads) {
        const int32_t i = own_row(f);
        if (i >= n) break;
        const float4 pv = pv_[i];
        const float3 dvv = ld3(dv_, vs, i);
        const float3 zv = stop ? make_float3(pv.x, pv.y, pv.z) : ld3(zv_, vs, i);
        st3(dv_, vs, i, make_float3(fmaf(alpha, pv.x, dvv.x), fmaf(alpha, pv.y, dvv.y),
                                    fmaf(alpha, pv.z, dvv.z)));
        if (!stop)
          pv_[i] = make_float4(fmaf(beta, pv.x, zv.x), fmaf(beta, pv.y, zv.y),
                               fmaf(beta, pv.z, zv.z), 0.f);
      }
    }
    if (stop) break;
    grid_arrive(a.bar, L.epoch, &fail_sh);
    if (tid == 0) {
      Producer P = L.P;
      for (int j = 0; j < kEarlyStages && !P.ended; ++j)
        if (producer_step<BW>(P, sh, m) < 0) timed_out(a.status, &fail_sh);
      L.P = P;
    }
    if (!grid_wait(a.bar, L.epoch, &ok_sh)) break;
    if (timer) {
      const unsigned long long t = now_ns();
      L.t_p += t - L.t_prev;
      L.t_prev = t;
    }
  }

  // ---- copies still in flight (only after a timeout), timers, dv out -------
  if (tid == 0) {
    producer_drain(L.P, sh);
    if (timer) {
      a.phase_ns[0] = L.t_s;
      a.phase_ns[1] = L.t_u;
      a.phase_ns[2] = L.t_p;
      a.phase_ns[3] = L.n_timed;
    }
  }
  const bool zero = zero_sh != 0;
  for (int32_t f = tid; f < nslots; f += kPipeThreads) {
    const int32_t i = own_row(f);
    if (i >= n) continue;
    const float3 d = zero ? make_float3(0.f, 0.f, 0.f) : ld3(a.dv, a.vs, i);
    a.dv_out[3 * int64_t(i)] = d.x;
    a.dv_out[3 * int64_t(i) + 1] = d.y;
    a.dv_out[3 * int64_t(i) + 2] = d.z;
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

bool g_loop_attr[3][64] = {};

template <int BW, bool G>
int loop_attrs(int device) {
  const int w = BW == kSymBlock ? (G ? 1 : 0) : 2;
  if (device >= 0 && device < 64 && g_loop_attr[w][device]) return 0;
  constexpr size_t smem = Pipe<BW>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(pcg_loop<BW, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  cudaFuncAttributes fa{};
  if (PCLOTH_PIPE_CARVE && e == cudaSuccess) e = cudaFuncGetAttributes(&fa, pcg_loop<BW, G>);
  if (PCLOTH_PIPE_CARVE && e == cudaSuccess)
    e = cudaFuncSetAttribute(pcg_loop<BW, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             pipe_carveout_percent(smem, fa.sharedSizeBytes));
  if (e != cudaSuccess) return int(e);
  if (device >= 0 && device < 64) g_loop_attr[w][device] = true;
  return 0;
}

// Grid of the persistent kernel: the streaming grid, capped at the CTAs
// that can be resident at once.
template <int BW, bool G>
int loop_grid_for(int32_t n, int device, int sm_count, int* grid) {
  const int e = loop_attrs<BW, G>(device);
  if (e != 0) return e;
  int per_sm = 0;
  const cudaError_t o = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, pcg_loop<BW, G>, kPipeThreads, Pipe<BW>::kSmem);
  if (o != cudaSuccess) return int(o);
  if (per_sm <= 0) return int(cudaErrorCooperativeLaunchTooLarge);
  *grid = std::min(spmv_grid_for(n, sm_count), per_sm * sm_count);
  return 0;
}

// Enqueues the persistent solve (cooperative launch) on `stream`.  Should the
// device refuse to hold the whole grid at once (the occupancy estimate and
// the launch disagree), the grid is halved until it fits -- any grid is
// correct, each CTA then walks more tiles -- and *grid keeps the size that
// launched.
template <int BW, bool G>
cudaError_t launch_loop(const LoopArgs& a, int* grid, cudaStream_t stream) {
  LoopArgs args = a;
  void* params[] = {&args};
  while (true) {
    const cudaError_t e = cudaLaunchCooperativeKernel(
        reinterpret_cast<const void*>(pcg_loop<BW, G>), dim3(*grid), dim3(kPipeThreads), params,
        Pipe<BW>::kSmem, stream);
    if (e != cudaErrorCooperativeLaunchTooLarge || *grid <= 1) return e;
    cudaGetLastError();   // a launch-configuration error: not sticky
    *grid = (*grid + 1) / 2;
  }
}

// Self-tests of the bounded waits: each kernel waits, with a short limit, on
// something nothing will ever complete -- an mbarrier phase that gets no
// arrival, or a barrier counter that gets one arrival of the two it waits
// for -- and must return with ST_WAIT_TIMEOUT set instead of hanging.
__global__ void selftest_mbarrier(uint64_t limit_ns, uint32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !wait_bounded(&bar, 0u, limit_ns)) atomicOr(status, ST_WAIT_TIMEOUT);
}

// Two CTAs of one cooperative launch meet at the PCG kernel's grid barrier;
// CTA 1 arrives poisoned, as after a timeout.  Both must leave the barrier
// with the timeout verdict (each adds 1 to `seen`) instead of going on.
__global__ void selftest_poison(unsigned long long* bar, unsigned int* seen, uint32_t* status) {
  __shared__ int fail_sh, ok_sh;
  unsigned long long epoch = 0;
  if (threadIdx.x == 0) fail_sh = blockIdx.x == 1 ? 1 : 0;
  if (!grid_barrier(bar, epoch, &fail_sh, &ok_sh) && threadIdx.x == 0) {
    atomicOr(status, ST_WAIT_TIMEOUT);
    atomicAdd(seen, 1u);
  }
}

__global__ void selftest_counter(unsigned long long* counter, uint64_t limit_ns,
                                 uint32_t* status) {
  if (threadIdx.x == 0) {
    atomicAdd(counter, 1ull);
    unsigned long long v = 0;
    if (!poll_bounded(counter, 2ull, limit_ns, &v)) atomicOr(status, ST_WAIT_TIMEOUT);
  }
}

}  // namespace

int selftest_bounded_wait(int which, double limit_s, uint32_t* status_out) {
  unsigned char* buf = nullptr;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&buf), 64);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "self-test buffer");
  uint32_t* status = reinterpret_cast<uint32_t*>(buf);
  unsigned int* seen = reinterpret_cast<unsigned int*>(buf + 4);
  unsigned long long* counter = reinterpret_cast<unsigned long long*>(buf + 16);
  e = cudaMemset(buf, 0, 64);
  const uint64_t limit_ns = uint64_t(limit_s * 1e9);
  if (e == cudaSuccess) {
    if (which == 0) {
      selftest_mbarrier<<<1, 32>>>(limit_ns, status);
      e = cudaGetLastError();
    } else if (which == 1) {
      selftest_counter<<<1, 32>>>(counter, limit_ns, status);
      e = cudaGetLastError();
    } else {
      void* args[] = {&counter, &seen, &status};
      e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(selftest_poison), dim3(2),
                                      dim3(32), args, 0, nullptr);
    }
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  uint32_t st = 0, sn = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&st, status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&sn, seen, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  cudaFree(buf);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "self-test wait");
  if (status_out) *status_out = st | (sn << 8);
  if (st & ST_WAIT_TIMEOUT) return fail(nullptr, PCLOTH_ERR_CUDA, "device wait timed out");
  return PCLOTH_OK;
}

int pcg_loop_grid(int blk, int32_t n, int device, int sm_count, int* grid, bool guess) {
  if (blk != kSymBlock) return loop_grid_for<9, false>(n, device, sm_count, grid);
  return guess ? loop_grid_for<kSymBlock, true>(n, device, sm_count, grid)
               : loop_grid_for<kSymBlock, false>(n, device, sm_count, grid);
}

int launch_state_update(Handle* h, float* x, float* v, const float* dv, float dt) {
  state_update<<<h->vec_grid, kVecThreads, 0, h->stream>>>(int64_t(h->n) * 3, x, v, dv, dt,
                                                           h->d_status);
  h->launches += 1;
  return check_launch(h, "state update");
}

int pcg_solve(Handle* h, double tol, int32_t maxit, float* dv_out, int32_t* iterations,
              double* rel_residual, const float* x0, bool async) {
  cudaStream_t s = h->stream;
  const bool prof = h->prof.on && !async;
  LoopArgs a{};
  a.m = PipeMatrix{h->n, (h->n + kPipeRows - 1) / kPipeRows, h->rowptr, h->colind, h->vals,
                   nullptr, 0};
  a.b = h->rhs;
  a.pinv = h->pinv6;
  a.dv = h->dv3;
  a.r = h->r3;
  a.z = h->z3;
  a.p = h->p4;
  a.q = h->q3;
  a.vs = h->vstride;
  a.rec = h->rec;
  a.bar = h->bar;
  a.state = h->state;
  a.status = h->d_status;
  a.dv_out = dv_out;
  a.x0 = x0;
  a.phase_ns = prof ? h->phase_ns : nullptr;
  a.tol2 = tol * tol;
  a.maxit = maxit;
  cudaError_t e = cudaMemsetAsync(h->bar, 0, sizeof(unsigned long long), s);
  if (e != cudaSuccess) return cuda_fail(h, e, "pcg barrier reset");
  if (prof) cudaEventRecord(h->ev[2], s);
  if (x0) {
    if (h->loop_grid_guess <= 0) {
      const int ge = pcg_loop_grid(kSymBlock, h->n, h->device, h->sm_count, &h->loop_grid_guess,
                                   true);
      if (ge != 0) return cuda_fail(h, cudaError_t(ge), "PCG kernel occupancy (guess)");
    }
    e = launch_loop<kSymBlock, true>(a, &h->loop_grid_guess, s);
  } else {
    e = launch_loop<kSymBlock, false>(a, &h->loop_grid, s);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "pcg launch");
  h->launches += 1;
  // the asynchronous form reads nothing back: pcloth_step_result does, later
  if (async) return PCLOTH_OK;
  if (prof) cudaEventRecord(h->ev[3], s);
  e = cudaMemcpyAsync(h->state_host, h->state, sizeof(PcgState), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && prof)
    e = cudaMemcpyAsync(h->phase_host, h->phase_ns, 4 * sizeof(unsigned long long),
                        cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "pcg state copy");
  int rc = collect_status(h);  // synchronises
  const PcgState st = *h->state_host;
  if (prof) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, h->ev[2], h->ev[3]);
    h->prof.solve_ms += ms;
    h->prof.solves += 1;
    h->prof.iterations += st.iterations;
    h->prof.spmv_ms += double(h->phase_host[0]) * 1e-6;
    h->prof.update_ms += double(h->phase_host[1] + h->phase_host[2]) * 1e-6;
    h->prof.samples += int64_t(h->phase_host[3]);
    h->prof.spmv_launches += st.iterations;
    h->prof.update_launches += st.iterations;
  }
  return solve_code(h, rc, st, iterations, rel_residual);
}

// The outcome of the last solve from its device state, after the status word
// was collected (rc).
int solve_code(Handle* h, int rc, const PcgState& st, int32_t* iterations,
               double* rel_residual) {
  if (iterations) *iterations = st.iterations;
  if (rel_residual) *rel_residual = st.relres;
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

int pcg_result(Handle* h, int32_t* iterations, double* rel_residual) {
  cudaError_t e = cudaMemcpyAsync(h->state_host, h->state, sizeof(PcgState),
                                  cudaMemcpyDeviceToHost, h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "pcg state copy");
  const int rc = collect_status(h);  // synchronises
  return solve_code(h, rc, *h->state_host, iterations, rel_residual);
}

// ===========================================================================
// Allocation-free solve (pcloth_solve_bsr3_static).  It runs the same
// persistent PCG on a symmetric positive-definite BSR3 system the caller
// already holds, and keeps every work vector, every partial sum, the barrier
// counter and the status words in one fixed array compiled into this
// library, so it never calls cudaMalloc, cudaFree or any allocating routine.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kStaticBytes = 1,513,216 bytes, about 1.44 MiB) until
// the process exits, and every call on that GPU shares it.  Calls that
// overlap on the GPU therefore race on it; a caller must order them (one
// stream, or events).  Each call re-initialises everything it reads before
// reading it, so nothing leaks from one call into the next.
//
// The caller's arrays are checked before the solve is launched: alignment on
// the host, and the pattern on the device by a kernel that reads rowptr and
// colind only as values (it reads colind[k] only for k inside a row range
// it has already checked), so a malformed pattern is reported as
// PCLOTH_ERR_BAD_INDEX instead of steering the solve's copies and gathers
// out of bounds.
// ===========================================================================
namespace {

constexpr int64_t kStaticVec = int64_t(PCLOTH_STATIC_MAX_VERTS) + 64;   // float4 slots of p
constexpr int64_t kStaticPlane =                                          // floats per plane
    (int64_t(PCLOTH_STATIC_MAX_VERTS) + 31) / 32 * 32 + 64;
constexpr int kStaticPlanes = 6 + 4 * 3;   // P; dv, r, z, q
constexpr int kStaticMaxRecords = 2048;    // CTAs of the solve
static_assert((sizeof(float4) * kStaticVec + sizeof(float) * kStaticPlanes * kStaticPlane) % 16 ==
                  0, "the partial-sum records start 16-byte aligned");
constexpr size_t kStaticBytes = sizeof(float4) * size_t(kStaticVec) +
                                sizeof(float) * size_t(kStaticPlanes) * size_t(kStaticPlane) +
                                sizeof(float2) * size_t(kRecSlots) * size_t(kStaticMaxRecords) +
                                256;
static_assert(kStaticBytes == 1513216, "the size the header states");

static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

// Device address of g_static_scratch per device ordinal (set up on first use).
void* g_static_addr[64] = {};

// Pattern check of a caller's BSR3 matrix, one thread per row: rowptr[0] = 0,
// 0 <= rowptr[i] <= rowptr[i+1] <= rowptr[n], and inside the row every
// column in [0, n), strictly increasing, with the diagonal present.  A row
// whose bounds fail is not read further.  Any violation sets ST_BAD_INDEX.
__global__ void bsr3_validate(int32_t n, const int32_t* __restrict__ rowptr,
                              const int32_t* __restrict__ colind, uint32_t* status) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int32_t lo = rowptr[i], hi = rowptr[i + 1], total = rowptr[n];
  bool ok = lo >= 0 && lo <= hi && hi <= total && (i != 0 || lo == 0);
  if (ok) {
    int32_t prev = -1;
    bool diag = false;
    for (int32_t k = lo; k < hi && ok; ++k) {
      const int32_t c = colind[k];
      ok = c > prev && c < n;
      diag = diag || c == int32_t(i);
      prev = c;
    }
    ok = ok && diag;
  }
  if (!ok) atomicOr(status, ST_BAD_INDEX);
}

// Inverse of the diagonal block of each row of a caller's BSR3 matrix, stored
// like the library's own: six planes P00 P01 P02 P11 P12 P22 of vs floats.
// The block must be symmetric (A is symmetric positive definite): the
// inverse is formed from the six cofactors of the upper triangle.  The block
// is first scaled by its largest entry, so that the determinant of a tiny
// (or huge) but well-conditioned block neither underflows nor overflows in
// fp32; a block that is not positive definite by its determinant is
// reported as non-finite.  The pattern has passed bsr3_validate, so the
// diagonal is present.
__global__ void bsr3_diag_inverse(int32_t n, const int32_t* __restrict__ rowptr,
                                  const int32_t* __restrict__ colind,
                                  const float* __restrict__ vals, float* __restrict__ pinv6,
                                  int64_t vs, uint32_t* status) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  int32_t lo = rowptr[i], hi = rowptr[i + 1];
  while (lo < hi) {
    const int32_t mid = (lo + hi) >> 1;
    if (colind[mid] < i) lo = mid + 1; else hi = mid;
  }
  const float* D = vals + 9 * int64_t(lo);
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < 9; ++t) s = fmaxf(s, fabsf(D[t]));
  const float inv_s = s > 0.f ? 1.0f / s : 0.f;
  const float d00 = D[0] * inv_s, d01 = D[1] * inv_s, d02 = D[2] * inv_s;
  const float d11 = D[4] * inv_s, d12 = D[5] * inv_s, d22 = D[8] * inv_s;
  const float c00 = d11 * d22 - d12 * d12;
  const float c01 = d12 * d02 - d01 * d22;
  const float c02 = d01 * d12 - d11 * d02;
  const float c11 = d00 * d22 - d02 * d02;
  const float c12 = d02 * d01 - d00 * d12;
  const float c22 = d00 * d11 - d01 * d01;
  float det = d00 * c00 + d01 * c01 + d02 * c02;
  if (!(det > 0.f) || !isfinite(det) || !(s > 0.f) || !isfinite(s)) {
    atomicOr(status, ST_NONFINITE);
    det = 1.f;
  }
  // (D / s)^-1 = s D^-1, so D^-1 = adj(D / s) / (det(D / s) s)
  const float id = inv_s / det;
  pinv6[i] = c00 * id;
  pinv6[vs + i] = c01 * id;
  pinv6[2 * vs + i] = c02 * id;
  pinv6[3 * vs + i] = c11 * id;
  pinv6[4 * vs + i] = c12 * id;
  pinv6[5 * vs + i] = c22 * id;
}

}  // namespace

int pcg_solve_static(int32_t n, const int32_t* rowptr, const int32_t* colind, const float* vals,
                     const float* b, double tol, int32_t maxit, float* dv_out,
                     int32_t* iterations, double* rel_residual, cudaStream_t stream) {
  // The solve streams rowptr, colind and vals with 16-byte bulk copies.
  for (const void* p : {static_cast<const void*>(rowptr), static_cast<const void*>(colind),
                        static_cast<const void*>(vals)})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
      return fail(nullptr, PCLOTH_ERR_INVALID_ARG,
                  "rowptr, colind and vals must be 16-byte aligned device pointers");
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
  int sm_count = 0;
  cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, device);
  if (sm_count <= 0) sm_count = 1;
  int grid = 0;
  const int ge = pcg_loop_grid(9, n, device, sm_count, &grid, false);
  if (ge != 0) return cuda_fail(nullptr, cudaError_t(ge), "pcg grid");
  if (grid > kStaticMaxRecords)
    return fail(nullptr, PCLOTH_ERR_CAPACITY, "too many CTAs for the fixed partial sums");
  unsigned char* base = static_cast<unsigned char*>(g_static_addr[device]);
  float4* p4 = reinterpret_cast<float4*>(base);
  float* planes = reinterpret_cast<float*>(p4 + kStaticVec);
  float2* rec = reinterpret_cast<float2*>(planes + size_t(kStaticPlanes) * kStaticPlane);
  unsigned char* tail = reinterpret_cast<unsigned char*>(rec + size_t(kRecSlots) * kStaticMaxRecords);
  LoopArgs a{};
  a.m = PipeMatrix{n, (n + kPipeRows - 1) / kPipeRows, rowptr, colind, vals, nullptr, 0};
  a.b = b;
  float* pinv6 = planes;
  a.pinv = pinv6;
  a.dv = planes + 6 * kStaticPlane;
  a.r = planes + 9 * kStaticPlane;
  a.z = planes + 12 * kStaticPlane;
  a.q = planes + 15 * kStaticPlane;
  a.p = p4;
  a.vs = kStaticPlane;
  a.rec = rec;
  a.state = reinterpret_cast<PcgState*>(tail);
  uint32_t* status = reinterpret_cast<uint32_t*>(tail + 64);
  a.bar = reinterpret_cast<unsigned long long*>(tail + 128);
  a.status = status;
  a.dv_out = dv_out;
  a.phase_ns = nullptr;
  a.tol2 = tol * tol;
  a.maxit = maxit;

  e = cudaMemsetAsync(tail, 0, 256, stream);   // state, status and barrier counter
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "static solve reset");
  // the pattern first: nothing below runs on a malformed one
  bsr3_validate<<<(n + 255) / 256, 256, 0, stream>>>(n, rowptr, colind, status);
  e = cudaGetLastError();
  uint32_t st_bits = 0;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&st_bits, status, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "static solve pattern check");
  if (st_bits & ST_BAD_INDEX)
    return fail(nullptr, PCLOTH_ERR_BAD_INDEX,
                "malformed BSR3 pattern: rowptr not starting at 0 or decreasing, a column "
                "outside [0, n), columns of a row not strictly increasing, or no diagonal block");
  bsr3_diag_inverse<<<(n + 255) / 256, 256, 0, stream>>>(n, rowptr, colind, vals, pinv6,
                                                        kStaticPlane, status);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = launch_loop<9, false>(a, &grid, stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "static solve launch");
  PcgState st{};
  e = cudaMemcpyAsync(&st, a.state, sizeof(PcgState), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&st_bits, status, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "static solve result");
  if (iterations) *iterations = st.iterations;
  if (rel_residual) *rel_residual = st.relres;
  if (st_bits & ST_WAIT_TIMEOUT) return fail(nullptr, PCLOTH_ERR_CUDA, "device wait timed out");
  if (st_bits & ST_NONFINITE)
    return fail(nullptr, PCLOTH_ERR_NONFINITE,
                "non-finite value, or a diagonal block that is not positive definite");
  if (st.code == PCLOTH_ERR_BREAKDOWN) return fail(nullptr, st.code, "PCG breakdown");
  if (st.code == PCLOTH_ERR_NONFINITE) return fail(nullptr, st.code, "non-finite value in PCG");
  return st.code;
}

}  // namespace pcloth_impl
