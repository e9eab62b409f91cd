// Internal declarations shared by the CUDA sources of libpcloth.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

#include <string>
#include <vector>

#include "pcloth.h"

namespace pcloth_impl {

// ---------------------------------------------------------------- status --
// Device-side error bits (ORed into Handle::d_status by kernels).
enum : uint32_t {
  ST_BAD_INDEX = 1u << 0,
  ST_NONFINITE = 1u << 1,
  ST_BREAKDOWN = 1u << 2,
  ST_CAPACITY = 1u << 3,
  ST_WAIT_TIMEOUT = 1u << 4,   // a bounded device wait gave up
};

// Device state of one PCG solve (written by kernels, read by the host).
struct PcgState {
  int32_t done;        // 1 once converged, broken down or non-finite
  int32_t iterations;  // iterations completed when done was set
  int32_t code;        // PCLOTH_OK / _NOT_CONVERGED / _ERR_*
  int32_t pad;
  double relres;       // |r| / |b| at stop
  double bnorm;        // |b|
};

// ------------------------------------------------------------ sizes --------
constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;

constexpr int kSymBlock = 6;   // floats per packed symmetric 3x3 block
constexpr int kAsmThreads = 256;  // threads per CTA of the row assembly

// Rows of A longer than this many blocks are summed with compensation
// (TwoSum) in every product A x: the plain fp32 sum of n products errs by up
// to about n eps times the sum of their magnitudes, and a vertex in contact
// with hundreds of others sums hundreds of terms that cancel to a small
// fraction of their size.  Cloth rows (13 to 20 blocks) keep the plain sum,
// which costs nothing; compensating every row cost 3% per PCG iteration and
// 18% on the plain product.  The choice depends on the row's length only,
// so the streaming and the block-ELL products agree bit for bit.
constexpr int kCompRow = 32;

constexpr int kVecThreads = 256;
// Bytes by which the PCG's row vectors are staggered past their 2 MB
// boundaries (array k at k times this), see pcloth_create.  Measured per
// PCG iteration on the 1.65M-triangle cloth: separate allocations 67.7 us;
// one arena with staggers of 0, 4, 16, 32, 64, 96, 128, 256 KB, 1 and 1.5 MB
// gave 66.7, 66.7, 66.35, 66.6, 66.4, 66.7, 66.8, 67.5, 68.2 and 68.4 us (the
// vector phases move with it: 15.5 us at 64 KB, 17.1 us at 1.5 MB).
#ifndef PCLOTH_VEC_STAGGER
#define PCLOTH_VEC_STAGGER 65536
#endif
constexpr size_t kVecStagger = PCLOTH_VEC_STAGGER;
// Per-CTA partial sums of the PCG dot products, one double-float (float2)
// per slot: p.q, r.z, r.r, b.b.
constexpr int kRecSlots = 4;
// r.z and r.r share a 16-byte half of the record: one load reads both
enum { REC_PQ = 0, REC_BB = 1, REC_RZ = 2, REC_RR = 3 };

// --------------------------------------------------------------- handle ----
struct Profile {
  bool on = false;
  int mode = 1;          // accepted for compatibility: 1 and 2 behave alike
  double assemble_ms = 0, spmv_ms = 0, update_ms = 0, solve_ms = 0;
  int64_t spmv_launches = 0, update_launches = 0, assemble_calls = 0;
  int64_t solves = 0, iterations = 0;
  int64_t samples = 0;   // PCG iterations whose phases were timed
};

struct Handle {
  int device = 0;
  cudaStream_t stream = nullptr;
  int32_t n = 0;             // vertices
  int32_t ns = 0;            // springs
  int32_t max_contacts = 0;
  int64_t nnzb_static = 0;
  int64_t nnzb_cap = 0;
  float gravity[3] = {0, 0, 0};
  bool assembled = false;
  float last_dt = 0.f;
  int sm_count = 0;
  int spmv_grid = 0, vec_grid = 0;
  int loop_grid = 0;         // CTAs of the persistent PCG kernel (co-resident)
  int loop_grid_guess = 0;   // the same for its warm-start form (set on first use)
  int64_t launches = 0;      // kernels launched by this handle
  std::string err;

  // static data
  float* mass = nullptr;         // n
  int32_t* rowptr_s = nullptr;   // n+1
  int32_t* colind_s = nullptr;   // nnzb_static
  int32_t* sblk_ptr = nullptr;   // nnzb_static+1 (range of spring entries)
  float2* sentry = nullptr;      // 2*ns (k, L0), grouped by static block

  // assembled system
  int32_t* rowptr = nullptr;     // n+1
  int32_t* colind = nullptr;     // nnzb_cap (+pad)
  // Block values.  Every block of A is a symmetric 3x3 (a sum of symmetric
  // element stiffnesses, plus m I on the diagonal), so the library stores
  // six floats per block, (a00 a01 a02 a11 a12 a22): 24 bytes instead of 36.
  // A caller's general BSR3 (allocation-free solve) has blk = 9, row-major.
  float* vals = nullptr;         // nnzb_cap*blk (+pad)
  int32_t blk = kSymBlock;       // floats per block in vals
  float* rhs = nullptr;          // 3n
  float* pinv6 = nullptr;        // [6][vstride] planes P00 P01 P02 P11 P12 P22

  // per-step contact workspace (capacity 2*max_contacts entries).  The
  // assembly buckets a step's contact entries by row: centry holds them,
  // per row sorted by (column << 32 | contact id).
  uint64_t* centry = nullptr;
  int32_t* scan_tmp = nullptr;     // per-tile sums
  int32_t* rowcnt = nullptr;       // [2(n+1)]: entries per row, scanned to the first
                                   // entry of each row; then the scatter cursors
  int32_t* newcnt = nullptr;       // [n+1]: new blocks per row, scanned to those before it
  int32_t* newcol = nullptr;       // a row's new columns, at its first entry's index
  int32_t* counters = nullptr;     // [0] = #new blocks, [1] = #valid entries, [2] scan totals
                                   // of contact finding, [4..5] its pair count as uint64

  // host-input staging for pcloth_step_host
  float* hx = nullptr;
  float* hv = nullptr;
  int32_t* hci = nullptr;
  int32_t* hcj = nullptr;
  float* hck = nullptr;
  float* hcr = nullptr;

  // PCG workspace.  p, which the SpMV gathers, holds one float4 (x, y, z, 0)
  // per vertex, so that a gather is one aligned 16-byte load.  The vectors
  // that are only read and written row by row are three planes (x, y, z) of
  // vstride floats each, so that a warp's loads and stores cover whole
  // sectors and move no padding.
  void* vec_arena = nullptr;       // one allocation holding p, q, r, z, dv and P
  float* dv = nullptr;             // float[n][3] scratch (pcloth_step without dv)
  int64_t vstride = 0;             // floats per plane: n rounded up to 32
  float* dv3 = nullptr;            // [3][vstride]
  float* r3 = nullptr;
  float* z3 = nullptr;
  float* q3 = nullptr;
  float4* p4 = nullptr;
  float2* rec = nullptr;           // loop_grid * kRecSlots partial sums
  unsigned long long* bar = nullptr;       // grid-barrier arrival counter
  unsigned long long* phase_ns = nullptr;  // [4] phase times of the last solve
  unsigned long long* phase_host = nullptr;  // pinned copy
  PcgState* state = nullptr;       // device
  PcgState* state_host = nullptr;  // pinned
  uint32_t* d_status = nullptr;    // device error bits
  uint32_t* h_status = nullptr;    // pinned copy

  // contact finding: a spatial-hash table of hash_mask + 1 buckets
  uint32_t hash_mask = 0;
  int32_t* hash_first = nullptr;   // [buckets + 1]: counts, scanned to each bucket's first slot
  int2* hash_where = nullptr;      // [n]: each vertex's bucket and place in it
  float4* hash_slot = nullptr;     // [n]: (x, y, z, index) in bucket order
  int2* hash_range = nullptr;      // [buckets]: each bucket's first and end slot
  int32_t* pair_first = nullptr;   // [n + 1]: partners per vertex, scanned to first output

  // block-ELL copy of the assembled matrix (the pages' layout), built on
  // request for the head-to-head SpMV; invalid after the next assembly
  int32_t* bell_wmax = nullptr;    // device: longest row
  int32_t* bell_col = nullptr;     // [W * n]
  float* bell_val = nullptr;       // [6][W * n]
  int64_t bell_cap = 0;            // slots allocated
  int32_t bell_w = 0;
  bool bell_valid = false;

  // profiling
  Profile prof;
  cudaEvent_t ev[8] = {};
};

// ------------------------------------------------------------- helpers ----
int fail(Handle* h, int code, const std::string& msg);
int cuda_fail(Handle* h, cudaError_t e, const char* what);
int check_launch(Handle* h, const char* what);
int collect_status(Handle* h);  // sync + read d_status; returns error code

// scan.cu
// Exclusive scan of int32 counts in place; writes the total to *total_dev.
int scan_exclusive(Handle* h, int32_t* data, int32_t n, int32_t* total_dev);

// assemble.cu
int assemble_system(Handle* h, const float* x, const float* v,
                    const pcloth_springs* contacts, float dt);

// spmv.cu
int spmv_grid_for(int32_t n, int sm_count);
int pipe_carveout_percent(size_t dyn_smem, size_t static_smem);
int launch_spmv(Handle* h, const float* in, float* out);

// contacts.cu: vertex-vertex proximity contacts by spatial hashing
int find_contacts(Handle* h, const float* x, float radius, float stiffness,
                  pcloth_springs* out, int32_t capacity, int32_t* found);

// bell.cu: block-ELL copy of the assembled matrix and its product
int bell_build(Handle* h);
int launch_bell_spmv(Handle* h, const float* in, float* out);

// assemble.cu: expand the packed symmetric inverses to float[n][3][3]
int launch_pinv_expand(Handle* h, float* out9);
// assemble.cu: expand the packed symmetric blocks to float[nnzb][3][3]
int launch_vals_expand(Handle* h, float* out9, int64_t nnzb);

// pcg.cu
// CTAs of the persistent PCG kernel for blocks of blk floats: the streaming
// grid, capped at what can be co-resident (a cooperative launch needs all).
int pcg_loop_grid(int blk, int32_t n, int device, int sm_count, int* grid, bool guess = false);
int selftest_bounded_wait(int which, double limit_s, uint32_t* status_out);
// x0: the initial iterate (device float[n][3], may alias dv), or null for
// dv = 0.  async: enqueue only -- no host synchronisation or read; the
// result stays in h->state and the status word (pcloth_step_result).
int pcg_solve(Handle* h, double tol, int32_t maxit, float* dv,
              int32_t* iterations, double* rel_residual, const float* x0 = nullptr,
              bool async = false);
int launch_state_update(Handle* h, float* x, float* v, const float* dv, float dt);
// The outcome of the last (asynchronous) solve: synchronises, reads its
// device state and the status word.
int pcg_result(Handle* h, int32_t* iterations, double* rel_residual);
int solve_code(Handle* h, int rc, const PcgState& st, int32_t* iterations,
               double* rel_residual);
int pcg_solve_static(int32_t n, const int32_t* rowptr, const int32_t* colind, const float* vals,
                     const float* b, double tol, int32_t maxit, float* dv_out,
                     int32_t* iterations, double* rel_residual, cudaStream_t stream);

// ---------------------------------------------------------- device code ---
#ifdef __CUDACC__
__device__ __forceinline__ bool finite3(float a, float b, float c) {
  return isfinite(a) && isfinite(b) && isfinite(c);
}

// Double-float numbers (value = hi + lo, |lo| <= ulp(hi) / 2) for the PCG
// reductions.  FP64 arithmetic is slow on this part, so every sum is carried
// in pairs of fp32 with TwoSum, which keeps ~44 bits; each reduction adds in
// a fixed order, so all CTAs that reduce the same partials get the same bits.
struct Dfloat {
  float hi, lo;
};

__device__ __forceinline__ Dfloat df_add(Dfloat a, Dfloat b) {
  const float s = a.hi + b.hi;
  const float bp = s - a.hi;
  float e = (a.hi - (s - bp)) + (b.hi - bp);   // exact rounding error of a.hi + b.hi
  e += a.lo + b.lo;
  const float hi = s + e;
  return Dfloat{hi, e - (hi - s)};
}

__device__ __forceinline__ Dfloat df_of(float x) { return Dfloat{x, 0.f}; }

// Compensated running sum (TwoSum, Knuth): s + c carries the sum of the
// terms added so far with the rounding error of every addition kept in c,
// so a row of many terms that cancel (a vertex in contact with thousands of
// others) loses nothing to the additions; read the total as s + c.
__device__ __forceinline__ void add_comp(float& s, float& c, float x) {
  const float t = s + x;
  const float bp = t - s;
  c += (s - (t - bp)) + (x - bp);
  s = t;
}
__device__ __forceinline__ Dfloat df_of(float2 x) { return Dfloat{x.x, x.y}; }
__device__ __forceinline__ float2 df_pack(Dfloat x) { return make_float2(x.hi, x.lo); }
__device__ __forceinline__ double df_value(Dfloat x) { return double(x.hi) + double(x.lo); }

// Block-wide sums of N double-floats per thread, for thread 0 only: a
// shuffle tree per warp, then lane q of warp 0 adds the warp totals of value
// q in order and hands it to lane 0.  The result is valid in thread 0; the
// caller synchronises the block again before sh is reused.
template <int THREADS, int N>
__device__ __forceinline__ void block_sum_df0(Dfloat (&v)[N], float2* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q < N; ++q) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const Dfloat u{__shfl_down_sync(0xffffffffu, v[q].hi, o),
                     __shfl_down_sync(0xffffffffu, v[q].lo, o)};
      v[q] = df_add(v[q], u);
    }
    if (lane == 0) sh[q * 32 + warp] = df_pack(v[q]);
  }
  __syncthreads();
  if (warp == 0) {
    Dfloat t{0.f, 0.f};
    if (lane < N) {
      t = df_of(sh[lane * 32]);
      for (int w = 1; w < THREADS / 32; ++w) t = df_add(t, df_of(sh[lane * 32 + w]));
    }
#pragma unroll
    for (int q = 0; q < N; ++q)
      v[q] = Dfloat{__shfl_sync(0xffffffffu, t.hi, q), __shfl_sync(0xffffffffu, t.lo, q)};
  }
}

// Adds slots slot0 .. slot0 + N - 1 of `count` partial records (kRecSlots
// float2 each) that the CTAs of the grid wrote: this thread's share, records
// threadIdx.x, + threads, ..., in index order.  The loads bypass L1 (other
// SMs wrote the records) and are issued two records at a time before they
// are added, so that their latencies overlap; with N = 2 (slot0 even) a
// record's two slots are one 16-byte load.
template <int N>
__device__ __forceinline__ void records_share(const float2* rec, int count, int slot0,
                                              int threads, Dfloat (&a)[N]) {
  static_assert(N == 1 || N == 2, "one or two slots");
#pragma unroll
  for (int q = 0; q < N; ++q) a[q] = Dfloat{0.f, 0.f};
  auto load = [&](int t, float2(&x)[N]) {
    if constexpr (N == 2) {
      const float4 w = __ldcg(reinterpret_cast<const float4*>(rec + t * kRecSlots + slot0));
      x[0] = make_float2(w.x, w.y);
      x[1] = make_float2(w.z, w.w);
    } else {
      x[0] = __ldcg(&rec[t * kRecSlots + slot0]);
    }
  };
  int t = threadIdx.x;
  for (; t + threads < count; t += 2 * threads) {
    float2 x0[N], x1[N];
    load(t, x0);
    load(t + threads, x1);
#pragma unroll
    for (int q = 0; q < N; ++q) a[q] = df_add(df_add(a[q], df_of(x0[q])), df_of(x1[q]));
  }
  if (t < count) {
    float2 x0[N];
    load(t, x0);
#pragma unroll
    for (int q = 0; q < N; ++q) a[q] = df_add(a[q], df_of(x0[q]));
  }
}
#endif

}  // namespace pcloth_impl
