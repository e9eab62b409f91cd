// Exclusive scans of int32 counts, in place: the assembly's per-row contact
// entries and new blocks (assemble.cu) and the contact finder's bucket and
// pair counts (contacts.cu).  Two launches: per-tile sums, then each tile's
// scan plus its offset, which the tile adds up itself from the sums before
// it (up to kInlineTiles tiles; a longer scan scans the sums in a launch of
// its own, between the two).

#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

// Exclusive scan of data[0, n) by a single block of 1024 threads, carrying a
// running total across chunks of 4096 values.  Writes the grand total to
// *total when total != nullptr.
__global__ void __launch_bounds__(1024)
scan_one_block(int32_t* __restrict__ data, int32_t n, int32_t* __restrict__ total) {
  __shared__ int32_t wsum[32];
  __shared__ int32_t carry_sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t carry = 0;
  for (int64_t base = 0; base < n; base += 4096) {
    int32_t v[4];
    const int64_t i0 = base + int64_t(threadIdx.x) * 4;
    int32_t s = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = (i0 + k < n) ? data[i0 + k] : 0;
      s += v[k];
    }
    // inclusive warp scan of the per-thread sums
    int32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int32_t w = wsum[lane];
      int32_t wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int32_t t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      wsum[lane] = wi - w;  // exclusive prefix of warp totals
      if (lane == 31) carry_sh = wi;
    }
    __syncthreads();
    int32_t run = carry + wsum[warp] + (incl - s);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (i0 + k < n) data[i0 + k] = run;
      run += v[k];
    }
    carry += carry_sh;
    __syncthreads();
  }
  if (threadIdx.x == 0 && total) *total = carry;
}

// Exclusive block scan of kScanItems values per thread; returns the block
// total to every thread.
__device__ __forceinline__ int32_t block_scan_items(int32_t (&v)[kScanItems],
                                                    int32_t* wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t s = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    const int32_t t = v[k];
    v[k] = s;
    s += t;
  }
  int32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int32_t w = (lane < kScanThreads / 32) ? wsum[lane] : 0;
    int32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kScanThreads / 32) wsum[lane] = wi - w;
    if (lane == 31) wsum[32] = wi;
  }
  __syncthreads();
  const int32_t off = wsum[warp] + (incl - s);
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) v[k] += off;
  const int32_t tot = wsum[32];
  __syncthreads();
  return tot;
}

__global__ void __launch_bounds__(kScanThreads)
scan_tile_sums(const int32_t* __restrict__ data, int32_t n, int32_t* __restrict__ sums) {
  __shared__ int32_t wsum[33];
  int32_t v[kScanItems];
  const int64_t base = int64_t(blockIdx.x) * kScanTile + int64_t(threadIdx.x) * kScanItems;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) v[k] = (base + k < n) ? data[base + k] : 0;
  const int32_t tot = block_scan_items(v, wsum);
  if (threadIdx.x == 0) sums[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kScanThreads)
scan_tiles_apply(int32_t* __restrict__ data, int32_t n, const int32_t* __restrict__ offs) {
  __shared__ int32_t wsum[33];
  int32_t v[kScanItems];
  const int64_t base = int64_t(blockIdx.x) * kScanTile + int64_t(threadIdx.x) * kScanItems;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) v[k] = (base + k < n) ? data[base + k] : 0;
  block_scan_items(v, wsum);
  const int32_t o = offs[blockIdx.x];
#pragma unroll
  for (int k = 0; k < kScanItems; ++k)
    if (base + k < n) data[base + k] = v[k] + o;
}

// The tile's exclusive scan plus its offset, the sum of the totals of the
// tiles before it, which the block adds up itself (at most kInlineTiles of
// them, read from L2): the single-block scan of the tile totals and its
// launch are saved.  The last block writes the grand total.
constexpr int kInlineTiles = 2048;

__global__ void __launch_bounds__(kScanThreads)
scan_tiles_apply_inline(int32_t* __restrict__ data, int32_t n,
                        const int32_t* __restrict__ sums, int32_t* __restrict__ total) {
  __shared__ int32_t wsum[33];
  __shared__ int32_t red[kScanThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t part = 0;
  for (int b = threadIdx.x; b < int(blockIdx.x); b += kScanThreads) part += sums[b];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_down_sync(0xffffffffu, part, o);
  if (lane == 0) red[warp] = part;
  int32_t v[kScanItems];
  const int64_t base = int64_t(blockIdx.x) * kScanTile + int64_t(threadIdx.x) * kScanItems;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) v[k] = (base + k < n) ? data[base + k] : 0;
  const int32_t tot = block_scan_items(v, wsum);   // synchronises the block: red[] is complete
  int32_t off = 0;
#pragma unroll
  for (int w = 0; w < kScanThreads / 32; ++w) off += red[w];
#pragma unroll
  for (int k = 0; k < kScanItems; ++k)
    if (base + k < n) data[base + k] = v[k] + off;
  if (total && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) *total = off + tot;
}

}  // namespace

int scan_exclusive(Handle* h, int32_t* data, int32_t n, int32_t* total_dev) {
  if (n <= 0) {
    cudaError_t e = cudaMemsetAsync(total_dev, 0, sizeof(int32_t), h->stream);
    return e == cudaSuccess ? PCLOTH_OK : cuda_fail(h, e, "scan memset");
  }
  const int ntiles = (n + kScanTile - 1) / kScanTile;
  if (ntiles == 1) {
    scan_one_block<<<1, 1024, 0, h->stream>>>(data, n, total_dev);
    h->launches += 1;
    return check_launch(h, "scan");
  }
  scan_tile_sums<<<ntiles, kScanThreads, 0, h->stream>>>(data, n, h->scan_tmp);
  if (ntiles <= kInlineTiles) {
    scan_tiles_apply_inline<<<ntiles, kScanThreads, 0, h->stream>>>(data, n, h->scan_tmp,
                                                                   total_dev);
    h->launches += 2;
    return check_launch(h, "scan");
  }
  scan_one_block<<<1, 1024, 0, h->stream>>>(h->scan_tmp, ntiles, total_dev);
  scan_tiles_apply<<<ntiles, kScanThreads, 0, h->stream>>>(data, n, h->scan_tmp);
  h->launches += 3;
  return check_launch(h, "scan");
}

}  // namespace pcloth_impl
