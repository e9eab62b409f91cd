// Block (3x3) sparse matrix-vector product q = A p (P-Cloth, arXiv
// 2008.00409, Sec. 3.1: SpMV is the most expensive operator of the PCG
// solve; Eq. (4) with one GPU is the plain product).
//
// The pages use a block-ELL layout on Pascal/Volta so that one thread per
// row streams coalesced SoA planes.  On GB300 the matrix stays BSR3 and is
// streamed tile by tile through shared memory:
//
//   * a persistent CTA owns tiles blockIdx.x, +gridDim.x, ... of kPipeRows
//     rows; one producer lane copies each tile's row pointers, block values
//     and column indices (three contiguous ranges, whatever the row lengths)
//     into a ring of shared-memory stages with bulk asynchronous copies,
//     completion counted on mbarriers, with an L2 evict-first hint so that
//     the gathered input vector stays L2-resident;
//   * the consumer warps work in two phases per stage: one thread per block
//     multiplies its 3x3 block (stride-9 shared reads, conflict free) by the
//     gathered input vertex -- a thread issues all of its gathers before
//     using any -- and stores the three products; then one thread per row
//     adds its row's products in column order and writes the output row.
//
// Tiles longer than a stage are split into chunks and the row sums carry
// over, so every output has a fixed summation order and the product is
// bitwise reproducible.  Every wait on an mbarrier is bounded in time and
// reports ST_WAIT_TIMEOUT instead of hanging.
//
// The PCG variant reads the solver's padded vectors (one float4 per vertex,
// so a gather is one aligned 16-byte load) and fuses two neighbouring steps
// of the iteration into the same pass: the search direction
// p_k = z_k + beta p_{k-1} is formed on the fly where it is gathered (and
// written once per own row), and the partial dot product p_k . q_k is
// reduced per CTA.  beta and the convergence test come from the previous
// kernel's per-CTA partials, reduced in a fixed order by every CTA.

#include <algorithm>

#include "async_copy.cuh"
#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

#ifndef PCLOTH_PIPE_ROWS
#define PCLOTH_PIPE_ROWS 48
#endif
#ifndef PCLOTH_PIPE_CAP
#define PCLOTH_PIPE_CAP 640
#endif
#ifndef PCLOTH_PIPE_STAGES
#define PCLOTH_PIPE_STAGES 2
#endif
#ifndef PCLOTH_PIPE_CTAS
#define PCLOTH_PIPE_CTAS 3
#endif
#ifndef PCLOTH_PIPE_CARVE
#define PCLOTH_PIPE_CARVE 1
#endif
constexpr int kPipeRows = PCLOTH_PIPE_ROWS;   // rows per tile (multiple of 4)
constexpr int kPipeCap = PCLOTH_PIPE_CAP;     // blocks per stage
constexpr int kPipeStages = PCLOTH_PIPE_STAGES;
constexpr int kPipeCtasPerSm = PCLOTH_PIPE_CTAS;
constexpr int kPipeConsumerWarps = 8;
constexpr int kPipeConsumers = 32 * kPipeConsumerWarps;
constexpr int kPipeThreads = 32 + kPipeConsumers;
constexpr int kPipePerThread = (kPipeCap + kPipeConsumers - 1) / kPipeConsumers;
constexpr int kPipeRpInts = kPipeRows + 4;
constexpr int kPipeColBytes = kPipeCap * 4 + 32;
constexpr int kPipeHeadBytes = 256;           // barriers and descriptors
constexpr int kPipePartBytes = kPipeCap * 16; // one float4 of products per block

// Shared-memory geometry of one stage for blocks of BW floats: row pointers,
// block values, column indices (each copy window has 16-byte slack at both
// ends), then the double-buffered products after the stages.
template <int BW>
struct Pipe {
  static constexpr int kValBytes = kPipeCap * 4 * BW + 32;
  static constexpr int kStageBytes =
      ((kPipeRpInts * 4 + kValBytes + kPipeColBytes) + 127) / 128 * 128;
  static constexpr size_t kSmem = size_t(kPipeHeadBytes) + size_t(kPipeStages) * kStageBytes +
                                  2 * size_t(kPipePartBytes);
};
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s: far beyond any legal wait
static_assert(kPipeRows % 4 == 0, "row-pointer copies must start 16-byte aligned");
static_assert(kPipeRows <= kPipeConsumers, "one consumer per row");

struct SpmvArgs {
  int32_t n;
  int32_t ntiles;
  const int32_t* rowptr;
  const int32_t* colind;
  const float* vals;
  const float* in;       // plain product: input  float[n][3]
  float* out;            // plain product: output float[n][3]
  // PCG fields (padded vectors, one float4 per vertex)
  const float4* z;
  const float4* p_old;
  float4* p_new;
  float4* q;
  const float2* rz_cur;  // records of r_k . z_k (slot 0) and r_k . r_k (slot 1)
  const float2* rz_prev; // records of r_{k-1} . z_{k-1}
  const float2* bb;      // records of b . b (slot 0)
  int red_n;             // number of records of rz_* and bb
  float2* pq_out;        // this kernel's records of p . q
  PcgState* state;
  uint32_t* status;
  int first;
  int k;
  double tol2;
};

struct StageDesc {
  int32_t tile, r0, nrows, c0, c1, voff, coff, flags;  // flags: 1 first, 2 last chunk
};

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait with a wall-clock bound; false when the bound is hit.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (now_ns() - t0 > kWaitNs) return false;
  }
}

// PCG prologue: returns false when the solve is already finished (converged,
// broken down or b = 0); otherwise sets beta for this iteration.  The four
// sums come from one fused, fixed-order double-float reduction of the
// previous kernels' records; thread 0 alone forms the scalars in fp64.
__device__ __forceinline__ bool pcg_prologue(const SpmvArgs& a, float2* rsh, int* flag_sh,
                                             float* beta_sh, float& beta) {
  if (threadIdx.x == 0) *flag_sh = a.state->done;
  __syncthreads();
  if (*flag_sh) return false;
  Dfloat v[4];   // b.b, r.r, r.z, previous r.z
  v[0] = records_share(a.bb, a.red_n, 0, kPipeThreads);
  if (a.first) {
    v[1] = v[2] = v[3] = Dfloat{0.f, 0.f};
  } else {
    v[1] = records_share(a.rz_cur, a.red_n, 1, kPipeThreads);
    v[2] = records_share(a.rz_cur, a.red_n, 0, kPipeThreads);
    v[3] = records_share(a.rz_prev, a.red_n, 0, kPipeThreads);
  }
  block_sum_df<kPipeThreads, 4>(v, rsh);
  if (threadIdx.x == 0) {
    const double bb = df_value(v[0]), rr = df_value(v[1]), rz = df_value(v[2]),
                 rzp = df_value(v[3]);
    int stop = 0;
    if (a.first) {
      if (!(bb > 0.0) || !isfinite(bb)) {   // b = 0: dv = 0 is exact
        stop = 1;
        if (blockIdx.x == 0) {
          a.state->done = 1;
          a.state->iterations = 0;
          a.state->relres = 0.0;
          a.state->code = isfinite(bb) ? PCLOTH_OK : PCLOTH_ERR_NONFINITE;
          if (!isfinite(bb)) atomicOr(a.status, ST_NONFINITE);
        }
      }
      *beta_sh = 0.f;
    } else {
      const bool conv = rr <= a.tol2 * bb;
      const bool bad = !isfinite(rr) || !isfinite(rz) || !(rz > 0.0) || !(rzp > 0.0);
      if (conv || bad) {
        stop = 1;
        if (blockIdx.x == 0) {
          a.state->done = 1;
          a.state->iterations = a.k;
          a.state->relres = sqrt(rr / bb);
          a.state->code = conv ? PCLOTH_OK
                               : (isfinite(rr) && isfinite(rz) ? PCLOTH_ERR_BREAKDOWN
                                                               : PCLOTH_ERR_NONFINITE);
          if (!conv) atomicOr(a.status, isfinite(rz) ? ST_BREAKDOWN : ST_NONFINITE);
        }
      }
      *beta_sh = float(rz / rzp);
    }
    *flag_sh = stop;
  }
  __syncthreads();
  beta = *beta_sh;
  return *flag_sh == 0;
}

template <bool PCG>
__device__ __forceinline__ float3 gather_x(const SpmvArgs& a, int32_t col, float beta) {
  if (PCG) {
    const float4 zc = a.z[col];
    if (a.first) return make_float3(zc.x, zc.y, zc.z);
    const float4 pc = a.p_old[col];
    return make_float3(fmaf(beta, pc.x, zc.x), fmaf(beta, pc.y, zc.y), fmaf(beta, pc.z, zc.z));
  }
  const int64_t c3 = int64_t(col) * 3;
  return make_float3(a.in[c3], a.in[c3 + 1], a.in[c3 + 2]);
}

// Product of one block with x.  BW = 6: packed symmetric block
// (a00 a01 a02 a11 a12 a22), read as three 8-byte words (a thread's stride of
// 24 bytes keeps the 16 threads of each half-warp on distinct banks); BW = 9:
// general row-major block.  Both give the same bits for a symmetric block.
template <int BW>
__device__ __forceinline__ float4 block_times(const float* __restrict__ B, float3 x) {
  if (BW == kSymBlock) {
    const float2* B2 = reinterpret_cast<const float2*>(B);
    const float2 u = B2[0], v = B2[1], w = B2[2];   // (a00 a01) (a02 a11) (a12 a22)
    return make_float4(fmaf(u.x, x.x, fmaf(u.y, x.y, v.x * x.z)),
                       fmaf(u.y, x.x, fmaf(v.y, x.y, w.x * x.z)),
                       fmaf(v.x, x.x, fmaf(w.x, x.y, w.y * x.z)), 0.f);
  }
  return make_float4(fmaf(B[0], x.x, fmaf(B[1], x.y, B[2] * x.z)),
                     fmaf(B[3], x.x, fmaf(B[4], x.y, B[5] * x.z)),
                     fmaf(B[6], x.x, fmaf(B[7], x.y, B[8] * x.z)), 0.f);
}

template <bool PCG, int BW>
__global__ void __launch_bounds__(kPipeThreads)
spmv_pipe(SpmvArgs a) {
  static_assert(BW == kSymBlock || BW == 9, "block width");
  constexpr int kPipeStageBytes = Pipe<BW>::kStageBytes;
  constexpr int kPipeValBytes = Pipe<BW>::kValBytes;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kPipeStages;
  StageDesc* desc = reinterpret_cast<StageDesc*>(smem + 64);
  unsigned char* stages = smem + kPipeHeadBytes;
  float4* parts = reinterpret_cast<float4*>(stages + size_t(kPipeStages) * kPipeStageBytes);
  __shared__ float2 rsh[33 * 4];
  __shared__ int flag_sh;
  __shared__ float beta_sh;

  float beta = 0.f;
  if (PCG && !pcg_prologue(a, rsh, &flag_sh, &beta_sh, beta)) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPipeStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kPipeConsumers);
    }
    mbar_init_fence();
  }
  __syncthreads();

  float pq = 0.f;
  if (threadIdx.x < 32) {
    // ------------------------------------------------------------ producer
    if (threadIdx.x == 0) {
      const uint64_t pol = policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int32_t tile = blockIdx.x; tile < a.ntiles && ok; tile += gridDim.x) {
        const int32_t r0 = tile * kPipeRows;
        const int32_t nrows = min(kPipeRows, a.n - r0);
        const int32_t b0 = a.rowptr[r0], b1 = a.rowptr[r0 + nrows];
        for (int32_t c0 = b0; ok;) {
          const int32_t c1 = min(b1, c0 + kPipeCap);
          if (!wait_bounded(&empty[s], ph ^ 1u)) { ok = false; break; }
          unsigned char* st = stages + size_t(s) * kPipeStageBytes;
          const int64_t va0 = (int64_t(c0) * (4 * BW)) & ~int64_t(15);
          const int64_t va1 = (int64_t(c1) * (4 * BW) + 15) & ~int64_t(15);
          const int64_t ca0 = (int64_t(c0) * 4) & ~int64_t(15);
          const int64_t ca1 = (int64_t(c1) * 4 + 15) & ~int64_t(15);
          const uint32_t rp_bytes = uint32_t(((nrows + 1 + 3) & ~3) * 4);
          const uint32_t v_bytes = uint32_t(va1 - va0), c_bytes = uint32_t(ca1 - ca0);
          StageDesc d;
          d.tile = tile; d.r0 = r0; d.nrows = nrows; d.c0 = c0; d.c1 = c1;
          d.voff = int32_t((int64_t(c0) * (4 * BW) - va0) >> 2);
          d.coff = int32_t((int64_t(c0) * 4 - ca0) >> 2);
          d.flags = (c0 == b0 ? 1 : 0) | (c1 == b1 ? 2 : 0);
          desc[s] = d;
          mbar_arrive_expect_tx(&full[s], rp_bytes + v_bytes + c_bytes);
          bulk_g2s(st, a.rowptr + r0, rp_bytes, &full[s], pol);
          bulk_g2s(st + kPipeRpInts * 4, reinterpret_cast<const unsigned char*>(a.vals) + va0,
                   v_bytes, &full[s], pol);
          bulk_g2s(st + kPipeRpInts * 4 + kPipeValBytes,
                   reinterpret_cast<const unsigned char*>(a.colind) + ca0, c_bytes, &full[s], pol);
          if (++s == kPipeStages) { s = 0; ph ^= 1u; }
          if (c1 >= b1) break;
          c0 = c1;
        }
      }
      // end marker (a plain arrival: no bytes)
      if (ok && wait_bounded(&empty[s], ph ^ 1u)) {
        desc[s].tile = -1;
        mbar_arrive(&full[s]);
      } else {
        ok = false;
      }
      if (!ok) atomicOr(a.status, ST_WAIT_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int ct = threadIdx.x - 32;
    int s = 0, buf = 0;
    uint32_t ph = 0;
    float3 acc = make_float3(0.f, 0.f, 0.f);
    float4 zown = make_float4(0.f, 0.f, 0.f, 0.f), pown = zown;
    while (true) {
      if (!wait_bounded(&full[s], ph)) {
        atomicOr(a.status, ST_WAIT_TIMEOUT);
        break;
      }
      const StageDesc d = desc[s];
      if (d.tile < 0) break;
      const unsigned char* st = stages + size_t(s) * kPipeStageBytes;
      const int32_t* rp = reinterpret_cast<const int32_t*>(st);
      const float* sv = reinterpret_cast<const float*>(st + kPipeRpInts * 4) + d.voff;
      const int32_t* sc =
          reinterpret_cast<const int32_t*>(st + kPipeRpInts * 4 + kPipeValBytes) + d.coff;
      float4* part = parts + buf * kPipeCap;
      const int32_t cn = d.c1 - d.c0;
      const bool row_owner = ct < d.nrows;
      const int32_t grow = d.r0 + ct;
      if (PCG && row_owner && (d.flags & 1)) {
        zown = a.z[grow];
        if (!a.first) pown = a.p_old[grow];
      }
      // phase B: block products, all of a thread's gathers in flight at once
      {
        int32_t col[kPipePerThread];
        float3 xv[kPipePerThread];
#pragma unroll
        for (int u = 0; u < kPipePerThread; ++u) {
          const int j = ct + u * kPipeConsumers;
          col[u] = j < cn ? sc[j] : -1;
        }
#pragma unroll
        for (int u = 0; u < kPipePerThread; ++u)
          if (col[u] >= 0) xv[u] = gather_x<PCG>(a, col[u], beta);
#pragma unroll
        for (int u = 0; u < kPipePerThread; ++u) {
          const int j = ct + u * kPipeConsumers;
          if (col[u] >= 0) part[j] = block_times<BW>(sv + BW * j, xv[u]);
        }
      }
      named_barrier_sync(1, kPipeConsumers);
      // phase C: row sums in column order, one thread per row
      if (row_owner) {
        const int32_t rs = max(rp[ct], d.c0) - d.c0, re = min(rp[ct + 1], d.c1) - d.c0;
        for (int32_t j = rs; j < re; ++j) {
          const float4 t = part[j];
          acc.x += t.x;
          acc.y += t.y;
          acc.z += t.z;
        }
      }
      mbar_arrive(&empty[s]);   // this thread no longer reads the stage
      if (row_owner && (d.flags & 2)) {
        if (PCG) {
          a.q[grow] = make_float4(acc.x, acc.y, acc.z, 0.f);
          const float4 pn = a.first ? zown
                                    : make_float4(fmaf(beta, pown.x, zown.x),
                                                  fmaf(beta, pown.y, zown.y),
                                                  fmaf(beta, pown.z, zown.z), 0.f);
          a.p_new[grow] = pn;
          pq = fmaf(pn.x, acc.x, fmaf(pn.y, acc.y, fmaf(pn.z, acc.z, pq)));
        } else {
          const int64_t g3 = int64_t(grow) * 3;
          a.out[g3] = acc.x;
          a.out[g3 + 1] = acc.y;
          a.out[g3 + 2] = acc.z;
        }
        acc = make_float3(0.f, 0.f, 0.f);
      }
      buf ^= 1;
      if (++s == kPipeStages) { s = 0; ph ^= 1u; }
    }
  }
  __syncthreads();
  if (PCG) {
    Dfloat t[1] = {df_of(pq)};
    block_sum_df<kPipeThreads, 1>(t, rsh);
    if (threadIdx.x == 0) a.pq_out[int64_t(blockIdx.x) * kRedSlots] = df_pack(t[0]);
  }
}

bool g_attr_done[64] = {};

// Shared-memory carveout: just enough for kPipeCtasPerSm CTAs, so that the
// rest of the unified L1/shared storage stays L1 cache for the gathers.
int carveout_percent(size_t smem) {
  const size_t need = size_t(kPipeCtasPerSm) * (smem + 2048);
  const size_t max_smem = 228 * 1024;
  int pct = int((need * 100 + max_smem - 1) / max_smem);
  return pct > 100 ? 100 : pct;
}

template <typename F>
cudaError_t set_attrs(F* f, size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(smem));
  if (PCLOTH_PIPE_CARVE && e == cudaSuccess)
    e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                             carveout_percent(smem));
  return e;
}

int ensure_attr(Handle* h) {
  if (h->device >= 0 && h->device < 64 && g_attr_done[h->device]) return PCLOTH_OK;
  cudaError_t e = set_attrs(spmv_pipe<false, kSymBlock>, Pipe<kSymBlock>::kSmem);
  if (e == cudaSuccess) e = set_attrs(spmv_pipe<true, kSymBlock>, Pipe<kSymBlock>::kSmem);
  if (e == cudaSuccess) e = set_attrs(spmv_pipe<true, 9>, Pipe<9>::kSmem);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(spmv)");
  if (h->device >= 0 && h->device < 64) g_attr_done[h->device] = true;
  return PCLOTH_OK;
}

SpmvArgs base_args(Handle* h) {
  SpmvArgs a{};
  a.n = h->n;
  a.ntiles = (h->n + kPipeRows - 1) / kPipeRows;
  a.rowptr = h->rowptr;
  a.colind = h->colind;
  a.vals = h->vals;
  a.status = h->d_status;
  return a;
}

}  // namespace

int spmv_grid_for(int32_t n, int sm_count) {
  return int(std::min<int64_t>((int64_t(n) + kPipeRows - 1) / kPipeRows,
                               int64_t(sm_count) * kPipeCtasPerSm));
}

int launch_spmv(Handle* h, const float* in, float* out) {
  int rc = ensure_attr(h);
  if (rc != PCLOTH_OK) return rc;
  SpmvArgs a = base_args(h);
  a.in = in;
  a.out = out;
  if (h->blk != kSymBlock) return fail(h, PCLOTH_ERR_INVALID_ARG, "spmv: packed blocks only");
  spmv_pipe<false, kSymBlock>
      <<<h->spmv_grid, kPipeThreads, Pipe<kSymBlock>::kSmem, h->stream>>>(a);
  h->launches += 1;
  return check_launch(h, "spmv");
}

// One PCG SpMV of iteration k (0-based): q = A p_k with p_k = z_k + beta p_{k-1}.
int launch_spmv_pcg(Handle* h, int k, double tol) {
  int rc = ensure_attr(h);
  if (rc != PCLOTH_OK) return rc;
  SpmvArgs a = base_args(h);
  a.z = h->z4;
  a.p_old = h->p4[(k + 1) & 1];
  a.p_new = h->p4[k & 1];
  a.q = h->q4;
  a.rz_cur = h->red_upd[k & 1];
  a.rz_prev = h->red_upd[(k + 1) & 1];
  a.bb = h->red_init;
  a.red_n = h->vec_grid;
  a.pq_out = h->red_spmv;
  a.state = h->state;
  a.first = (k == 0);
  a.k = k;
  a.tol2 = tol * tol;
  if (h->blk == kSymBlock)
    spmv_pipe<true, kSymBlock>
        <<<h->spmv_grid, kPipeThreads, Pipe<kSymBlock>::kSmem, h->stream>>>(a);
  else
    spmv_pipe<true, 9><<<h->spmv_grid, kPipeThreads, Pipe<9>::kSmem, h->stream>>>(a);
  h->launches += 1;
  return check_launch(h, "spmv (pcg)");
}

}  // namespace pcloth_impl
