// Block (3x3) sparse matrix-vector product out = A in (P-Cloth, arXiv
// 2008.00409, Sec. 3.1; Eq. (4) with one GPU is the plain product), for
// pcloth_spmv.  One persistent CTA per (SM x kPipeCtasPerSm) streams its row
// tiles through the pipeline of spmv_pipe.cuh once; the input and output
// are the caller's float[n][3] vectors.  The PCG solve runs the same
// pipeline inside its persistent kernel (pcg.cu).

#include <algorithm>

#include "spmv_pipe.cuh"

namespace pcloth_impl {
namespace {

struct PlainGather {
  const float* in;
  __device__ __forceinline__ float3 operator()(int32_t col) const {
    const int64_t c3 = int64_t(col) * 3;
    return make_float3(in[c3], in[c3 + 1], in[c3 + 2]);
  }
};

struct PlainEpi {
  float* out;
  __device__ __forceinline__ void begin(int32_t) const {}
  __device__ __forceinline__ void operator()(int32_t row, float3 acc) const {
    const int64_t g3 = int64_t(row) * 3;
    out[g3] = acc.x;
    out[g3 + 1] = acc.y;
    out[g3 + 2] = acc.z;
  }
};

constexpr int kTileCacheSpmv = 256;   // tiles per CTA whose block ranges go to shared memory

template <int BW>
__global__ void __launch_bounds__(kPipeThreads)
spmv_plain(PipeMatrix m, const float* __restrict__ in, float* __restrict__ out,
           uint32_t* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int2 tb_sh[kTileCacheSpmv];
  const PipeShared sh = pipe_shared<BW>(smem);
  m.tb = tb_sh;
  m.ntb = fill_tile_bounds(m, tb_sh, kTileCacheSpmv);
  pipe_init(sh);
  __syncthreads();
  if (threadIdx.x < 32) {
    if (threadIdx.x == 0) {
      Producer P;
      producer_begin(P, m);
      if (!producer_pass<BW>(P, sh, m)) atomicOr(status, ST_WAIT_TIMEOUT);
    }
  } else {
    Consumer C;
    consumer_begin(C);
    PlainGather g{in};
    PlainEpi e{out};
    if (!consumer_pass<BW>(C, sh, g, e)) atomicOr(status, ST_WAIT_TIMEOUT);
  }
}

bool g_attr_done[64] = {};

}  // namespace

// Shared-memory carveout: just enough for kPipeCtasPerSm CTAs, so that the
// rest of the unified L1/shared storage stays L1 cache for the gathers.  A
// CTA takes its dynamic and static shared memory plus the 1 KB the runtime
// reserves per CTA; the carveout is the smallest shared-memory capacity the
// SM offers that holds that many CTAs (a hint that rounded down would leave
// room for fewer CTAs than a cooperative launch of the full grid needs).
int pipe_carveout_percent(size_t dyn_smem, size_t static_smem) {
  const size_t need = size_t(kPipeCtasPerSm) * (dyn_smem + static_smem + 1024);
  static const int kCapsKb[] = {0, 8, 16, 32, 64, 100, 132, 164, 196, 228};
  for (int c : kCapsKb)
    if (size_t(c) * 1024 >= need) return (c * 100 + 227) / 228;
  return 100;
}

int spmv_grid_for(int32_t n, int sm_count) {
  return int(std::min<int64_t>((int64_t(n) + kPipeRows - 1) / kPipeRows,
                               int64_t(sm_count) * kPipeCtasPerSm));
}

int launch_spmv(Handle* h, const float* in, float* out) {
  if (h->blk != kSymBlock) return fail(h, PCLOTH_ERR_INVALID_ARG, "spmv: packed blocks only");
  constexpr size_t smem = Pipe<kSymBlock>::kSmem;
  if (!(h->device >= 0 && h->device < 64 && g_attr_done[h->device])) {
    cudaError_t e = cudaFuncSetAttribute(spmv_plain<kSymBlock>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    cudaFuncAttributes fa{};
    if (PCLOTH_PIPE_CARVE && e == cudaSuccess) e = cudaFuncGetAttributes(&fa, spmv_plain<kSymBlock>);
    if (PCLOTH_PIPE_CARVE && e == cudaSuccess)
      e = cudaFuncSetAttribute(spmv_plain<kSymBlock>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               pipe_carveout_percent(smem, fa.sharedSizeBytes));
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(spmv)");
    if (h->device >= 0 && h->device < 64) g_attr_done[h->device] = true;
  }
  PipeMatrix m{h->n, (h->n + kPipeRows - 1) / kPipeRows, h->rowptr, h->colind, h->vals,
               nullptr, 0};
  spmv_plain<kSymBlock><<<h->spmv_grid, kPipeThreads, smem, h->stream>>>(m, in, out,
                                                                        h->d_status);
  h->launches += 1;
  return check_launch(h, "spmv");
}

}  // namespace pcloth_impl
