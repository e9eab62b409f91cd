// Stable LSD radix sort of (uint64 key, int32 value) pairs and an exclusive
// int32 scan.
//
// The sort orders the vertices by spatial-hash cell and the found contact
// pairs by (i, j) for contact finding (contacts.cu; P-Cloth Sec. 4.2): equal
// keys keep their input order, so the results are deterministic.  Each pass
// over one 8-bit digit is three kernels: per-tile digit histograms, one
// exclusive scan of the digit-major histogram table, and a stable scatter
// that ranks keys inside each warp with match_any.  The scan also serves
// the assembly's per-row counts (assemble.cu): per-tile sums, then each
// tile's scan plus its offset, which the tile adds up from the sums before
// it (up to 1024 tiles; larger scans scan the sums in a launch of their own).

#include "pcloth_internal.cuh"

namespace pcloth_impl {
namespace {

constexpr int kWarps = kSortThreads / 32;

__global__ void __launch_bounds__(kSortThreads)
rs_upsweep(const uint64_t* __restrict__ keys, int32_t n, int shift,
           int32_t* __restrict__ counts, int ntiles) {
  __shared__ int32_t hist[kSortRadix];
  for (int d = threadIdx.x; d < kSortRadix; d += kSortThreads) hist[d] = 0;
  __syncthreads();
  const int64_t base = int64_t(blockIdx.x) * kSortTile;
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const int64_t idx = base + it * kSortThreads + threadIdx.x;
    if (idx < n) atomicAdd(&hist[int((keys[idx] >> shift) & (kSortRadix - 1))], 1);
  }
  __syncthreads();
  for (int d = threadIdx.x; d < kSortRadix; d += kSortThreads)
    counts[int64_t(d) * ntiles + blockIdx.x] = hist[d];
}

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

__global__ void __launch_bounds__(kSortThreads)
rs_downsweep(const uint64_t* __restrict__ kin, const int32_t* __restrict__ vin,
             uint64_t* __restrict__ kout, int32_t* __restrict__ vout, int32_t n,
             int shift, const int32_t* __restrict__ offsets, int ntiles) {
  __shared__ int32_t whist[kWarps][kSortRadix];
  __shared__ int32_t toff[kSortRadix];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int d = threadIdx.x; d < kSortRadix; d += kSortThreads) {
    toff[d] = offsets[int64_t(d) * ntiles + blockIdx.x];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) whist[w][d] = 0;
  }
  __syncthreads();
  const int64_t wbase = int64_t(blockIdx.x) * kSortTile + warp * (32 * kSortItems);
  uint64_t key[kSortItems];
  int32_t val[kSortItems];
  int dig[kSortItems];
  int rank[kSortItems];
  const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const int64_t idx = wbase + it * 32 + lane;
    const bool valid = idx < n;
    key[it] = valid ? kin[idx] : 0ull;
    val[it] = valid ? vin[idx] : 0;
    dig[it] = valid ? int((key[it] >> shift) & (kSortRadix - 1)) : kSortRadix;
    const unsigned peers = __match_any_sync(0xffffffffu, dig[it]);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (valid) base = whist[warp][dig[it]];
    __syncwarp();
    if (valid && lane == leader) whist[warp][dig[it]] = base + __popc(peers);
    __syncwarp();
    rank[it] = base + __popc(peers & lt_mask);
  }
  __syncthreads();
  // exclusive scan across warps, per digit
  for (int d = threadIdx.x; d < kSortRadix; d += kSortThreads) {
    int32_t run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int32_t t = whist[w][d];
      whist[w][d] = run;
      run += t;
    }
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    if (dig[it] < kSortRadix) {
      const int64_t pos = int64_t(toff[dig[it]]) + whist[warp][dig[it]] + rank[it];
      kout[pos] = key[it];
      vout[pos] = val[it];
    }
  }
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
constexpr int kInlineTiles = 1024;

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

int radix_sort_pairs(Handle* h, uint64_t* keys[2], int32_t* vals[2], int32_t n,
                     int bits) {
  int cur = 0;
  if (n <= 1) return cur;
  const int ntiles = (n + kSortTile - 1) / kSortTile;
  for (int shift = 0; shift < bits; shift += kSortBits) {
    rs_upsweep<<<ntiles, kSortThreads, 0, h->stream>>>(keys[cur], n, shift,
                                                       h->sort_counts, ntiles);
    scan_one_block<<<1, 1024, 0, h->stream>>>(h->sort_counts, kSortRadix * ntiles, nullptr);
    rs_downsweep<<<ntiles, kSortThreads, 0, h->stream>>>(
        keys[cur], vals[cur], keys[cur ^ 1], vals[cur ^ 1], n, shift,
        h->sort_counts, ntiles);
    h->launches += 3;
    cur ^= 1;
  }
  int rc = check_launch(h, "radix sort");
  return rc == PCLOTH_OK ? cur : rc;
}

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
