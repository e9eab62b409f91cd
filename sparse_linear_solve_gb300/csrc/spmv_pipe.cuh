// Streaming pipeline of the block (3x3) sparse matrix-vector product: the
// machinery shared by the plain product q = A x (spmv.cu) and the SpMV phase
// of the persistent PCG kernel (pcg.cu).  P-Cloth (arXiv 2008.00409,
// Sec. 3.1): SpMV is the most expensive operator of the PCG solve; Eq. (4)
// with one GPU is the plain product.
//
// The pages use a block-ELL layout on Pascal/Volta so that one thread per
// row streams coalesced SoA planes.  On GB300 the matrix stays BSR3 and is
// streamed tile by tile through shared memory:
//
//   * a CTA owns row tiles blockIdx.x, +gridDim.x, ... of kPipeRows rows; one
//     producer lane copies each tile's row pointers, block values and column
//     indices (three contiguous ranges, whatever the row lengths) into a ring
//     of shared-memory stages with bulk asynchronous copies, completion
//     counted on mbarriers, with an L2 evict-first hint so that the gathered
//     vector stays L2-resident;
//   * the consumer warps have two roles.  Five product warps take one thread
//     per block: it multiplies its block (packed symmetric or general, see
//     block_times) by the gathered input vertex -- a thread issues all of
//     its gathers before using any -- and stores the three products.  Two
//     row warps take one thread per row of the tile: it adds its row's
//     products in column order (rows longer than kCompRow blocks as a
//     compensated TwoSum sum, see below) and hands the row to an epilogue.  The products are double-buffered and pass
//     between the roles on mbarriers, so the row sums of one stage overlap
//     the gathers of the next and are off the product warps' path.
//
// Tiles longer than a stage are split into chunks and the row sums carry
// over, so every output has a fixed summation order and the product is
// bitwise reproducible.  The producer walks the CTA's tiles and then issues
// an end marker; the walk can be repeated any number of times (the
// persistent solver runs one pass per iteration), with the ring's slots and
// phases carried across passes.  Every wait on an mbarrier is bounded in
// time and reports ST_WAIT_TIMEOUT instead of hanging.
#pragma once

#include "async_copy.cuh"
#include "pcloth_internal.cuh"

namespace pcloth_impl {

// Pipeline geometry.  A tile of 64 cloth rows holds about 13.2 x 64 = 845
// blocks (13 per interior row plus contacts), so a stage of 896 blocks takes
// most tiles whole (a tile split across two stages costs a nearly empty
// second stage); three stages keep two tiles' copies in flight while one is
// consumed.  With packed blocks a CTA needs 103 KB of shared memory, so two
// CTAs run per SM.  Measured on the 1.65M-triangle cloth, this beat 48-row
// tiles of 640 blocks at 3 CTAs per SM by 15% per PCG iteration.  Seven
// consumer warps (five product, two row) beat six, eight, nine and ten per
// PCG iteration: a CTA of 256 threads keeps 128 registers a thread.
#ifndef PCLOTH_PIPE_ROWS
#define PCLOTH_PIPE_ROWS 64
#endif
#ifndef PCLOTH_PIPE_CAP
#define PCLOTH_PIPE_CAP 896
#endif
#ifndef PCLOTH_PIPE_STAGES
#define PCLOTH_PIPE_STAGES 3
#endif
#ifndef PCLOTH_PIPE_CTAS
#define PCLOTH_PIPE_CTAS 2
#endif
#ifndef PCLOTH_PIPE_CARVE
#define PCLOTH_PIPE_CARVE 1
#endif
constexpr int kPipeRows = PCLOTH_PIPE_ROWS;   // rows per tile (multiple of 4)
constexpr int kPipeCap = PCLOTH_PIPE_CAP;     // blocks per stage
constexpr int kPipeStages = PCLOTH_PIPE_STAGES;
constexpr int kPipeCtasPerSm = PCLOTH_PIPE_CTAS;
#ifndef PCLOTH_PIPE_CWARPS
#define PCLOTH_PIPE_CWARPS 7
#endif
constexpr int kPipeConsumerWarps = PCLOTH_PIPE_CWARPS;
constexpr int kPipeConsumers = 32 * kPipeConsumerWarps;
constexpr int kPipeThreads = 32 + kPipeConsumers;
constexpr int kPipePerThread = (kPipeCap + kPipeConsumers - 1) / kPipeConsumers;
constexpr int kPipeRpInts = kPipeRows + 4;
constexpr int kPipeColBytes = kPipeCap * 4 + 32;
constexpr int kPipeHeadBytes = 256;           // barriers and descriptors
constexpr int kPipePartBytes = kPipeCap * 16; // one float4 of products per block
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s: far beyond any legal wait
static_assert(kPipeRows % 4 == 0, "row-pointer copies must start 16-byte aligned");
static_assert(kPipeRows <= kPipeConsumers, "one consumer per row");
static_assert(2 * kPipeStages * 8 <= 64 && 64 + kPipeStages * 32 + 32 <= kPipeHeadBytes,
              "ring barriers at offset 0, stage descriptors at offset 64, then the four "
              "product-buffer barriers");
// The consumers split in two roles: kPipeProd threads form the block
// products of a stage, kPipeRows threads (two warps) add the rows of the
// stage before, and the double-buffered products pass between them on
// mbarriers (ready: products written; free: products read).
constexpr int kPipeProd = kPipeConsumers - kPipeRows;
constexpr int kPipeProdPerThread = (kPipeCap + kPipeProd - 1) / kPipeProd;
static_assert(kPipeProd % 32 == 0 && kPipeProd > 0, "whole warps per role");

// Shared-memory geometry for blocks of BW floats: per stage the row
// pointers, block values and column indices (each copy window has 16 bytes
// of slack at both ends), then the double-buffered products.
template <int BW>
struct Pipe {
  static constexpr int kValBytes = kPipeCap * 4 * BW + 32;
  static constexpr int kStageBytes =
      ((kPipeRpInts * 4 + kValBytes + kPipeColBytes) + 127) / 128 * 128;
  static constexpr size_t kSmem = size_t(kPipeHeadBytes) + size_t(kPipeStages) * kStageBytes +
                                  2 * size_t(kPipePartBytes);
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
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (now_ns() - t0 > limit_ns) return false;
  }
}

// Product of one block with x.  BW = 6: packed symmetric block
// (a00 a01 a02 a11 a12 a22), read as three 8-byte words (a thread stride of
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

// The matrix a pass streams.  tb, if set, is a shared-memory copy of the
// block ranges of this CTA's first ntb tiles (entry j: tile blockIdx.x +
// j * gridDim.x), for kernels that walk the same tiles many times.
struct PipeMatrix {
  int32_t n, ntiles;
  const int32_t* rowptr;
  const int32_t* colind;
  const float* vals;
  const int2* tb;
  int32_t ntb;
};

struct PipeShared {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* ready;   // [2] products of a buffer written (kPipeProd arrivals)
  uint64_t* freed;   // [2] products of a buffer read (kPipeRows arrivals)
  StageDesc* desc;
  unsigned char* stages;
  float4* parts;
};

template <int BW>
__device__ __forceinline__ PipeShared pipe_shared(unsigned char* smem) {
  PipeShared s;
  s.full = reinterpret_cast<uint64_t*>(smem);
  s.empty = s.full + kPipeStages;
  s.desc = reinterpret_cast<StageDesc*>(smem + 64);
  s.ready = reinterpret_cast<uint64_t*>(smem + 64 + kPipeStages * 32);
  s.freed = s.ready + 2;
  s.stages = smem + kPipeHeadBytes;
  s.parts = reinterpret_cast<float4*>(s.stages + size_t(kPipeStages) * Pipe<BW>::kStageBytes);
  return s;
}

// Thread 0 initialises the ring; the caller synchronises the CTA afterwards.
__device__ __forceinline__ void pipe_init(const PipeShared& sh) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPipeStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kPipeConsumers);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.ready[b], kPipeProd);
      mbar_init(&sh.freed[b], kPipeRows);
    }
    mbar_init_fence();
  }
}

// ---------------------------------------------------------------- producer
// One lane (thread 0).  The cursor names the next stage: a tile and the
// first block of the chunk (-1: the tile's first chunk).  `ended` is set once
// the end marker of the current pass is issued (stages may be issued ahead
// of the pass that consumes them).  Bit s of `used` / `last_ph` records
// whether a stage was ever issued into slot s and the parity of the last
// one, so that a kernel leaving early can wait for its own copies in flight.
struct Producer {
  int s;
  uint32_t ph;
  int32_t tile, c0;
  int32_t b1;            // end block of the current tile
  int32_t nb0, nb1;      // block range of the next tile to start (loaded ahead)
  bool ended;
  uint32_t used, last_ph;
  uint64_t pol;
};

// Block range [rowptr[r0], rowptr[r0 + rows]) of a tile: from the shared
// copy when there is one, else loaded here and consumed a stage or more
// later, so that the load's latency is off the producer's path.
__device__ __forceinline__ void tile_bounds_of(const PipeMatrix& m, int32_t tile, int32_t& b0,
                                               int32_t& b1) {
  if (tile < m.ntiles) {
    const int32_t j = (tile - int32_t(blockIdx.x)) / int32_t(gridDim.x);
    if (m.tb != nullptr && j < m.ntb) {
      const int2 t = m.tb[j];
      b0 = t.x;
      b1 = t.y;
    } else {
      const int32_t r0 = tile * kPipeRows;
      b0 = m.rowptr[r0];
      b1 = m.rowptr[min(r0 + kPipeRows, m.n)];
    }
  } else {
    b0 = b1 = 0;
  }
}

// Fills a shared copy of the block ranges of this CTA's first `cap` tiles
// (all threads of the CTA; the caller synchronises afterwards).  Returns the
// number of entries.
__device__ __forceinline__ int32_t fill_tile_bounds(const PipeMatrix& m, int2* tb, int32_t cap) {
  const int32_t mine = (m.ntiles - int32_t(blockIdx.x) + int32_t(gridDim.x) - 1) /
                       int32_t(gridDim.x);
  const int32_t cnt = mine < cap ? mine : cap;
  for (int32_t j = threadIdx.x; j < cnt; j += blockDim.x) {
    const int32_t r0 = (int32_t(blockIdx.x) + j * int32_t(gridDim.x)) * kPipeRows;
    tb[j] = make_int2(m.rowptr[r0], m.rowptr[min(r0 + kPipeRows, m.n)]);
  }
  return cnt;
}
static_assert(kPipeStages <= 32, "slot bit masks");

__device__ __forceinline__ void producer_begin(Producer& P, const PipeMatrix& m) {
  P.s = 0;
  P.ph = 0;
  P.tile = blockIdx.x;
  P.c0 = -1;
  P.b1 = 0;
  tile_bounds_of(m, P.tile, P.nb0, P.nb1);
  P.ended = false;
  P.used = 0;
  P.last_ph = 0;
  P.pol = policy_evict_first();
}

// Waits (bounded) until the copies of every stage the producer issued have
// landed; a kernel calls this before it exits early.
__device__ __forceinline__ void producer_drain(const Producer& P, const PipeShared& sh) {
#pragma unroll
  for (int s = 0; s < kPipeStages; ++s)
    if ((P.used >> s) & 1u) wait_bounded(&sh.full[s], (P.last_ph >> s) & 1u);
}

// Issues the next stage of the walk, or the end marker after the CTA's last
// tile (which rewinds the cursor for the next pass).  Returns 1 for a data
// stage, 0 for the end marker, -1 if the slot never became free.
template <int BW>
__device__ __forceinline__ int producer_step(Producer& P, const PipeShared& sh,
                                             const PipeMatrix& m) {
  if (!wait_bounded(&sh.empty[P.s], P.ph ^ 1u)) return -1;
  int ret = 1;
  P.used |= 1u << P.s;
  P.last_ph = (P.last_ph & ~(1u << P.s)) | (P.ph << P.s);
  if (P.tile >= m.ntiles) {
    sh.desc[P.s].tile = -1;   // end marker: a plain arrival, no bytes
    mbar_arrive(&sh.full[P.s]);
    P.tile = blockIdx.x;      // the next pass starts over
    P.c0 = -1;
    tile_bounds_of(m, P.tile, P.nb0, P.nb1);
    P.ended = true;
    ret = 0;
  } else {
    const int32_t r0 = P.tile * kPipeRows;
    const int32_t nrows = min(kPipeRows, m.n - r0);
    const bool first = P.c0 < 0;
    if (first) {              // start of a tile: its bounds were loaded ahead
      P.b1 = P.nb1;
      P.c0 = P.nb0;
      tile_bounds_of(m, P.tile + int32_t(gridDim.x), P.nb0, P.nb1);
    }
    const int32_t b1 = P.b1;
    const int32_t c0 = P.c0;
    const int32_t c1 = min(b1, c0 + kPipeCap);
    unsigned char* st = sh.stages + size_t(P.s) * Pipe<BW>::kStageBytes;
    const int64_t va0 = (int64_t(c0) * (4 * BW)) & ~int64_t(15);
    const int64_t va1 = (int64_t(c1) * (4 * BW) + 15) & ~int64_t(15);
    const int64_t ca0 = (int64_t(c0) * 4) & ~int64_t(15);
    const int64_t ca1 = (int64_t(c1) * 4 + 15) & ~int64_t(15);
    const uint32_t rp_bytes = uint32_t(((nrows + 1 + 3) & ~3) * 4);
    const uint32_t v_bytes = uint32_t(va1 - va0), c_bytes = uint32_t(ca1 - ca0);
    StageDesc d;
    d.tile = P.tile; d.r0 = r0; d.nrows = nrows; d.c0 = c0; d.c1 = c1;
    d.voff = int32_t((int64_t(c0) * (4 * BW) - va0) >> 2);
    d.coff = int32_t((int64_t(c0) * 4 - ca0) >> 2);
    d.flags = (first ? 1 : 0) | (c1 == b1 ? 2 : 0);
    sh.desc[P.s] = d;
    mbar_arrive_expect_tx(&sh.full[P.s], rp_bytes + v_bytes + c_bytes);
    bulk_g2s(st, m.rowptr + r0, rp_bytes, &sh.full[P.s], P.pol);
    bulk_g2s(st + kPipeRpInts * 4, reinterpret_cast<const unsigned char*>(m.vals) + va0, v_bytes,
             &sh.full[P.s], P.pol);
    bulk_g2s(st + kPipeRpInts * 4 + Pipe<BW>::kValBytes,
             reinterpret_cast<const unsigned char*>(m.colind) + ca0, c_bytes, &sh.full[P.s],
             P.pol);
    if (c1 >= b1) {
      P.tile += gridDim.x;
      P.c0 = -1;
    } else {
      P.c0 = c1;
    }
  }
  if (++P.s == kPipeStages) {
    P.s = 0;
    P.ph ^= 1u;
  }
  return ret;
}

// Producer side of one whole pass: the stages not yet issued ahead of time,
// up to and including the end marker.
template <int BW>
__device__ __forceinline__ bool producer_pass(Producer& P, const PipeShared& sh,
                                              const PipeMatrix& m) {
  while (!P.ended)
    if (producer_step<BW>(P, sh, m) < 0) return false;
  P.ended = false;
  return true;
}

// --------------------------------------------------------------- consumers
struct Consumer {
  int s;
  uint32_t ph;
  int buf;   // data stages consumed so far: buffer buf & 1, its (buf >> 1)-th use
};

__device__ __forceinline__ void consumer_begin(Consumer& C) {
  C.s = 0;
  C.ph = 0;
  C.buf = 0;
}

// Consumer side of one pass (threads 32 .. kPipeThreads-1): processes stages
// up to and including the end marker.  gather(col) returns the input vertex
// col as a float3; epi.begin(row) is called when a tile starts and epi(row,
// acc) receives each finished row's sum (both in the row threads).  Returns
// false if a stage, or the other role, never arrived.
template <int BW, class Gather, class Epi>
__device__ __forceinline__ bool consumer_pass(Consumer& C, const PipeShared& sh, Gather& gather,
                                              Epi& epi) {
  const int ct = threadIdx.x - 32;
  const bool prod = ct < kPipeProd;
  const int rt = ct - kPipeProd;    // row thread index (row threads only)
  float3 acc = make_float3(0.f, 0.f, 0.f), cmp = make_float3(0.f, 0.f, 0.f);
  while (true) {
    if (!wait_bounded(&sh.full[C.s], C.ph)) return false;
    const StageDesc d = sh.desc[C.s];
    if (d.tile < 0) {
      mbar_arrive(&sh.empty[C.s]);
      if (++C.s == kPipeStages) { C.s = 0; C.ph ^= 1u; }
      return true;
    }
    const unsigned char* st = sh.stages + size_t(C.s) * Pipe<BW>::kStageBytes;
    const int b = C.buf & 1;
    const uint32_t use = uint32_t(C.buf >> 1) & 1u;
    float4* part = sh.parts + b * kPipeCap;
    if (prod) {
      const float* sv = reinterpret_cast<const float*>(st + kPipeRpInts * 4) + d.voff;
      const int32_t* sc =
          reinterpret_cast<const int32_t*>(st + kPipeRpInts * 4 + Pipe<BW>::kValBytes) + d.coff;
      const int32_t cn = d.c1 - d.c0;
      int32_t col[kPipeProdPerThread];
      float3 xv[kPipeProdPerThread];
#pragma unroll
      for (int u = 0; u < kPipeProdPerThread; ++u) {
        const int j = ct + u * kPipeProd;
        col[u] = j < cn ? sc[j] : -1;
      }
#pragma unroll
      for (int u = 0; u < kPipeProdPerThread; ++u)
        if (col[u] >= 0) xv[u] = gather(col[u]);
      // the buffer is free once the row threads have added its last use
      if (!wait_bounded(&sh.freed[b], use ^ 1u)) return false;
#pragma unroll
      for (int u = 0; u < kPipeProdPerThread; ++u) {
        const int j = ct + u * kPipeProd;
        if (col[u] >= 0) part[j] = block_times<BW>(sv + BW * j, xv[u]);
      }
      mbar_arrive(&sh.empty[C.s]);   // this thread no longer reads the stage
      mbar_arrive(&sh.ready[b]);
    } else {
      const int32_t* rp = reinterpret_cast<const int32_t*>(st);
      const bool row_owner = rt < d.nrows;
      int32_t rs = 0, re = 0;
      bool comp = false;
      if (row_owner) {
        rs = max(rp[rt], d.c0) - d.c0;
        re = min(rp[rt + 1], d.c1) - d.c0;
        comp = rp[rt + 1] - rp[rt] > kCompRow;
        if (d.flags & 1) epi.begin(d.r0 + rt);
      }
      const int r0 = d.r0, last = d.flags & 2;
      mbar_arrive(&sh.empty[C.s]);   // desc and row pointers read
      if (!wait_bounded(&sh.ready[b], use)) return false;
      if (row_owner && comp) {
        for (int32_t j = rs; j < re; ++j) {
          const float4 t = part[j];
          add_comp(acc.x, cmp.x, t.x);
          add_comp(acc.y, cmp.y, t.y);
          add_comp(acc.z, cmp.z, t.z);
        }
      } else if (row_owner) {
        for (int32_t j = rs; j < re; ++j) {
          const float4 t = part[j];
          acc.x += t.x;
          acc.y += t.y;
          acc.z += t.z;
        }
      }
      mbar_arrive(&sh.freed[b]);
      if (row_owner && last) {
        epi(r0 + rt, make_float3(acc.x + cmp.x, acc.y + cmp.y, acc.z + cmp.z));
        acc = cmp = make_float3(0.f, 0.f, 0.f);
      }
    }
    ++C.buf;
    if (++C.s == kPipeStages) { C.s = 0; C.ph ^= 1u; }
  }
}

// Grid size of the streaming kernels: kPipeCtasPerSm CTAs per SM, never more
// CTAs than row tiles.
int spmv_grid_for(int32_t n, int sm_count);

}  // namespace pcloth_impl
