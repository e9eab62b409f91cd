// C ABI of libpcloth: handle lifetime, static pattern, error reporting.
//
// The static block pattern is built here once, on the host, from the springs
// (P-Cloth, arXiv 2008.00409, Sec. 3.2.2, sparse matrix filling steps 1-3:
// count the entries of every row, fill the column indices, sort each row and
// drop duplicates).  Everything per step runs in the kernels of
// assemble.cu, spmv.cu and pcg.cu.

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "pcloth_internal.cuh"

using namespace pcloth_impl;

namespace {
thread_local std::string g_create_err;

template <typename T>
cudaError_t dalloc(T** p, size_t count) {
  *p = nullptr;
  if (count == 0) count = 1;
  return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
}

void free_handle(Handle* h) {
  if (!h) return;
  cudaSetDevice(h->device);
  cudaStreamSynchronize(h->stream);
  void* bufs[] = {h->mass, h->rowptr_s, h->colind_s, h->sblk_ptr, h->sentry,
                  h->rowptr, h->colind, h->vals, h->rhs, h->vec_arena,
                  h->centry, h->hash_first, h->hash_where, h->hash_slot, h->hash_range, h->pair_first,
                  h->scan_tmp, h->rowcnt, h->newcnt, h->newcol,
                  h->counters,
                  h->hx, h->hv, h->hci, h->hcj, h->hck, h->hcr,
                  h->dv, h->rec, h->bar,
                  h->phase_ns, h->state, h->d_status, h->bell_wmax, h->bell_col, h->bell_val,
                  };
  for (void* b : bufs)
    if (b) cudaFree(b);
  if (h->state_host) cudaFreeHost(h->state_host);
  if (h->h_status) cudaFreeHost(h->h_status);
  if (h->phase_host) cudaFreeHost(h->phase_host);
  for (auto& e : h->ev)
    if (e) cudaEventDestroy(e);
  delete h;
}

}  // namespace

namespace pcloth_impl {

int fail(Handle* h, int code, const std::string& msg) {
  if (h)
    h->err = msg;
  else
    g_create_err = msg;
  return code;
}

int cuda_fail(Handle* h, cudaError_t e, const char* what) {
  std::string m = std::string(what) + ": " + cudaGetErrorString(e);
  return fail(h, PCLOTH_ERR_CUDA, m);
}

int check_launch(Handle* h, const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(h, e, what);
  return PCLOTH_OK;
}

int collect_status(Handle* h) {
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  e = cudaMemcpy(h->h_status, h->d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "status copy");
  uint32_t st = *h->h_status;
  if (st == 0) return PCLOTH_OK;
  e = cudaMemset(h->d_status, 0, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(h, e, "status reset");
  if (st & ST_BAD_INDEX)
    return fail(h, PCLOTH_ERR_BAD_INDEX, "element index out of range or i == j");
  if (st & ST_CAPACITY) return fail(h, PCLOTH_ERR_CAPACITY, "capacity exceeded");
  if (st & ST_NONFINITE)
    return fail(h, PCLOTH_ERR_NONFINITE, "non-finite value or zero-length element");
  if (st & ST_BREAKDOWN) return fail(h, PCLOTH_ERR_BREAKDOWN, "PCG breakdown");
  if (st & ST_WAIT_TIMEOUT) return fail(h, PCLOTH_ERR_CUDA, "device wait timed out");
  return fail(h, PCLOTH_ERR_CUDA, "unknown device status");
}

}  // namespace pcloth_impl

extern "C" {

int pcloth_create(const pcloth_mesh* mesh, const pcloth_springs* sp,
                  const pcloth_opts* opts, pcloth_t* out) {
  if (!out) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  g_create_err.clear();
  if (!mesh || !sp || !opts)
    return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL mesh, springs or opts");
  if (mesh->n_verts <= 0 || !mesh->mass)
    return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "n_verts <= 0 or mass NULL");
  if (sp->n < 0 || opts->max_contacts < 0)
    return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "negative spring or contact count");
  if (sp->n > 0 && (!sp->i || !sp->j || !sp->k || !sp->rest))
    return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL spring array");
  const int64_t n = mesh->n_verts, ns = sp->n, mc = opts->max_contacts;
  const int64_t cap = n + 2 * ns + 2 * mc;
  if (cap > (int64_t(1) << 31) - 4096 || 2 * mc > (int64_t(1) << 30))
    return fail(nullptr, PCLOTH_ERR_CAPACITY, "sizes exceed the int32 index range");

  cudaError_t e = cudaSetDevice(opts->device);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaSetDevice");

  Handle* h = new Handle();
  h->device = opts->device;
  h->stream = static_cast<cudaStream_t>(opts->stream);
  h->n = int32_t(n);
  h->ns = int32_t(ns);
  h->max_contacts = int32_t(mc);
  for (int c = 0; c < 3; ++c) h->gravity[c] = mesh->gravity[c];
  h->nnzb_cap = cap;
  cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device);
  if (h->sm_count <= 0) h->sm_count = 1;

  // ---- springs to the host, validated --------------------------------
  std::vector<int32_t> si(ns), sj(ns);
  std::vector<float> sk(ns), sr(ns);
  if (ns > 0) {
    e = cudaMemcpy(si.data(), sp->i, ns * 4, cudaMemcpyDefault);
    if (e == cudaSuccess) e = cudaMemcpy(sj.data(), sp->j, ns * 4, cudaMemcpyDefault);
    if (e == cudaSuccess) e = cudaMemcpy(sk.data(), sp->k, ns * 4, cudaMemcpyDefault);
    if (e == cudaSuccess) e = cudaMemcpy(sr.data(), sp->rest, ns * 4, cudaMemcpyDefault);
    if (e != cudaSuccess) {
      free_handle(h);
      return cuda_fail(nullptr, e, "copying springs");
    }
  }
  for (int64_t s = 0; s < ns; ++s) {
    if (si[s] < 0 || si[s] >= n || sj[s] < 0 || sj[s] >= n || si[s] == sj[s]) {
      free_handle(h);
      return fail(nullptr, PCLOTH_ERR_BAD_INDEX,
                  "spring " + std::to_string(s) + " has a bad vertex index");
    }
  }

  // ---- static pattern: per-row counting sort, then sort inside rows -----
  // entry = (col, spring id) in row; the diagonal is entry (row, -1).
  std::vector<int64_t> cnt(n + 1, 0);
  for (int64_t i = 0; i < n; ++i) cnt[i + 1] += 1;
  for (int64_t s = 0; s < ns; ++s) {
    cnt[si[s] + 1] += 1;
    cnt[sj[s] + 1] += 1;
  }
  for (int64_t i = 0; i < n; ++i) cnt[i + 1] += cnt[i];
  const int64_t nent = cnt[n];
  std::vector<std::pair<int32_t, int32_t>> ent(nent);
  {
    std::vector<int64_t> fill(cnt.begin(), cnt.end() - 1);
    for (int64_t i = 0; i < n; ++i) ent[fill[i]++] = {int32_t(i), -1};
    for (int64_t s = 0; s < ns; ++s) {
      ent[fill[si[s]]++] = {sj[s], int32_t(s)};
      ent[fill[sj[s]]++] = {si[s], int32_t(s)};
    }
  }
  std::vector<int32_t> rowptr_s(n + 1, 0), colind_s, sblk_ptr;
  std::vector<float2> sentry;
  colind_s.reserve(nent);
  sblk_ptr.reserve(nent + 1);
  sentry.reserve(2 * ns);
  for (int64_t i = 0; i < n; ++i) {
    std::sort(ent.begin() + cnt[i], ent.begin() + cnt[i + 1]);
    int32_t last = -1;
    for (int64_t t = cnt[i]; t < cnt[i + 1]; ++t) {
      if (ent[t].first != last) {
        colind_s.push_back(ent[t].first);
        sblk_ptr.push_back(int32_t(sentry.size()));
        last = ent[t].first;
      }
      if (ent[t].second >= 0)
        sentry.push_back(make_float2(sk[ent[t].second], sr[ent[t].second]));
    }
    rowptr_s[i + 1] = int32_t(colind_s.size());
  }
  sblk_ptr.push_back(int32_t(sentry.size()));
  h->nnzb_static = int64_t(colind_s.size());
  ent.clear();
  ent.shrink_to_fit();

  // ---- device buffers ---------------------------------------------------
  const int64_t ent2 = std::max<int64_t>(2 * mc, 1);
  // contact finding hashes cells into a power-of-two table of at least 2n
  // buckets
  int64_t buckets = 1024;
  while (buckets < 2 * n && buckets < (int64_t(1) << 30)) buckets *= 2;
  h->hash_mask = uint32_t(buckets - 1);
  // scans run over the n + 1 per-row counts of the assembly, the n + 1
  // per-vertex pair counts and the buckets + 1 hash counts
  const int64_t scan_tiles =
      (std::max<int64_t>(ent2, buckets + 1) + kScanTile - 1) / kScanTile;
  h->spmv_grid = spmv_grid_for(int32_t(n), h->sm_count);
  {
    const int ge = pcg_loop_grid(kSymBlock, int32_t(n), h->device, h->sm_count, &h->loop_grid);
    if (ge != 0) {
      free_handle(h);
      return cuda_fail(nullptr, cudaError_t(ge), "PCG kernel occupancy");
    }
  }
  h->vec_grid = int(std::min<int64_t>((n + kVecThreads - 1) / kVecThreads,
                                      int64_t(h->sm_count) * 4));
  const int64_t vpad = 64;  // floats of slack after each vector / value array
  bool ok = true;
  auto A = [&](cudaError_t r) { ok = ok && (r == cudaSuccess); };
  A(dalloc(&h->mass, n));
  A(dalloc(&h->rowptr_s, n + 1 + vpad));
  A(dalloc(&h->colind_s, h->nnzb_static + vpad));
  A(dalloc(&h->sblk_ptr, h->nnzb_static + 1 + vpad));
  A(dalloc(&h->sentry, std::max<int64_t>(2 * ns, 1)));
  A(dalloc(&h->rowptr, n + 1 + vpad));
  A(dalloc(&h->colind, cap + vpad));
  A(dalloc(&h->vals, cap * kSymBlock + vpad));
  A(dalloc(&h->rhs, 3 * n + vpad));
  h->vstride = (n + 31) / 32 * 32;
  const int64_t vs = h->vstride;
  {
    // The vectors of the PCG's row phases in one allocation, each array on
    // its own 2 MB boundary plus a stagger of kVecStagger bytes times its
    // index, so that the streams a phase reads at the same row index do not
    // all sit at the same offset within their pages.
    const size_t sizes[6] = {size_t(n + vpad) * sizeof(float4),           // p
                             size_t(3 * vs + vpad) * sizeof(float),       // q
                             size_t(3 * vs + vpad) * sizeof(float),       // r
                             size_t(3 * vs + vpad) * sizeof(float),       // z
                             size_t(3 * vs + vpad) * sizeof(float),       // dv
                             size_t(6 * vs + vpad) * sizeof(float)};      // P
    constexpr size_t kPage = size_t(2) << 20;
    size_t off[6], cursor = 0;
    for (int k = 0; k < 6; ++k) {
      off[k] = (cursor + kPage - 1) / kPage * kPage + size_t(k) * kVecStagger;
      cursor = off[k] + sizes[k];
    }
    unsigned char* base = nullptr;
    A(cudaMalloc(reinterpret_cast<void**>(&base), cursor));
    h->vec_arena = base;
    if (base) {
      h->p4 = reinterpret_cast<float4*>(base + off[0]);
      h->q3 = reinterpret_cast<float*>(base + off[1]);
      h->r3 = reinterpret_cast<float*>(base + off[2]);
      h->z3 = reinterpret_cast<float*>(base + off[3]);
      h->dv3 = reinterpret_cast<float*>(base + off[4]);
      h->pinv6 = reinterpret_cast<float*>(base + off[5]);
    }
  }
  A(dalloc(&h->centry, ent2));
  A(dalloc(&h->hash_first, buckets + 1));
  A(dalloc(&h->hash_where, n));
  A(dalloc(&h->hash_slot, n));
  A(dalloc(&h->hash_range, buckets));
  A(dalloc(&h->pair_first, n + 1));
  A(dalloc(&h->scan_tmp, scan_tiles + 1));
  A(dalloc(&h->rowcnt, 2 * (n + 1)));
  A(dalloc(&h->newcnt, n + 1));
  A(dalloc(&h->newcol, ent2));
  A(dalloc(&h->counters, 8));
  A(dalloc(&h->hx, 3 * n));
  A(dalloc(&h->hv, 3 * n));
  A(dalloc(&h->hci, std::max<int64_t>(mc, 1)));
  A(dalloc(&h->hcj, std::max<int64_t>(mc, 1)));
  A(dalloc(&h->hck, std::max<int64_t>(mc, 1)));
  A(dalloc(&h->hcr, std::max<int64_t>(mc, 1)));
  A(dalloc(&h->dv, 3 * n + vpad));
  A(dalloc(&h->rec, int64_t(h->loop_grid) * kRecSlots));
  A(dalloc(&h->bar, 1));
  A(dalloc(&h->phase_ns, 4));
  A(dalloc(&h->bell_wmax, 1));
  A(dalloc(&h->state, 1));
  A(dalloc(&h->d_status, 1));
  A(cudaMallocHost(reinterpret_cast<void**>(&h->state_host), sizeof(PcgState)));
  A(cudaMallocHost(reinterpret_cast<void**>(&h->phase_host), 4 * sizeof(unsigned long long)));
  A(cudaMallocHost(reinterpret_cast<void**>(&h->h_status), sizeof(uint32_t)));
  for (auto& ev : h->ev) A(cudaEventCreate(&ev));
  if (!ok) {
    cudaGetLastError();
    free_handle(h);
    return fail(nullptr, PCLOTH_ERR_CUDA, "device allocation failed");
  }
  e = cudaMemcpy(h->mass, mesh->mass, n * 4, cudaMemcpyDefault);
  if (e == cudaSuccess) e = cudaMemcpy(h->rowptr_s, rowptr_s.data(), (n + 1) * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && h->nnzb_static)
    e = cudaMemcpy(h->colind_s, colind_s.data(), h->nnzb_static * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(h->sblk_ptr, sblk_ptr.data(), sblk_ptr.size() * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !sentry.empty())
    e = cudaMemcpy(h->sentry, sentry.data(), sentry.size() * sizeof(float2), cudaMemcpyHostToDevice);
  // zero the padding and workspaces so that no read ever sees garbage
  if (e == cudaSuccess) e = cudaMemset(h->vals, 0, (cap * kSymBlock + vpad) * 4);
  if (e == cudaSuccess) e = cudaMemset(h->colind, 0, (cap + vpad) * 4);
  if (e == cudaSuccess) e = cudaMemset(h->rowptr, 0, (n + 1 + vpad) * 4);
  for (float* v : {h->dv, h->rhs})
    if (e == cudaSuccess) e = cudaMemset(v, 0, (3 * n + vpad) * 4);
  for (float* v : {h->dv3, h->r3, h->z3, h->q3})
    if (e == cudaSuccess) e = cudaMemset(v, 0, (3 * vs + vpad) * sizeof(float));
  if (e == cudaSuccess) e = cudaMemset(h->p4, 0, (n + vpad) * sizeof(float4));
  if (e == cudaSuccess) e = cudaMemset(h->pinv6, 0, (6 * vs + vpad) * sizeof(float));
  if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, 4);
  if (e == cudaSuccess) e = cudaMemset(h->state, 0, sizeof(PcgState));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_handle(h);
    return cuda_fail(nullptr, e, "uploading the static pattern");
  }
  *out = reinterpret_cast<pcloth_t>(h);
  return PCLOTH_OK;
}

int pcloth_assemble(pcloth_t ht, const float* x, const float* v,
                    const pcloth_springs* contacts, float dt) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (!x || !v) return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL x or v");
  if (!(dt > 0.f) || !std::isfinite(dt)) return fail(h, PCLOTH_ERR_INVALID_ARG, "dt must be > 0");
  if (contacts && contacts->n < 0) return fail(h, PCLOTH_ERR_INVALID_ARG, "negative contact count");
  if (contacts && contacts->n > h->max_contacts)
    return fail(h, PCLOTH_ERR_CAPACITY, "contacts exceed max_contacts");
  if (contacts && contacts->n > 0 &&
      (!contacts->i || !contacts->j || !contacts->k || !contacts->rest))
    return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL contact array");
  cudaSetDevice(h->device);
  int rc = assemble_system(h, x, v, contacts, dt);
  if (rc == PCLOTH_OK) {
    h->assembled = true;
    h->last_dt = dt;
  }
  return rc;
}

int pcloth_spmv(pcloth_t ht, const float* in, float* out) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (!in || !out) return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL vector");
  if (!h->assembled) return fail(h, PCLOTH_ERR_STATE, "spmv before assemble");
  cudaSetDevice(h->device);
  return launch_spmv(h, in, out);
}

int pcloth_find_contacts(pcloth_t ht, const float* x, float radius, float stiffness,
                         pcloth_springs* out, int32_t capacity, int32_t* found) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (!x || !out) return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL x or out");
  if (!(radius > 0.f) || !std::isfinite(radius) || !(stiffness >= 0.f) ||
      !std::isfinite(stiffness))
    return fail(h, PCLOTH_ERR_INVALID_ARG, "radius must be > 0 and stiffness >= 0");
  if (capacity < 0) return fail(h, PCLOTH_ERR_INVALID_ARG, "negative capacity");
  if (capacity > 0 && (!out->i || !out->j || !out->k || !out->rest))
    return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL output array");
  cudaSetDevice(h->device);
  return find_contacts(h, x, radius, stiffness, out, capacity, found);
}

int pcloth_bell_build(pcloth_t ht, int32_t* width) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (!h->assembled) return fail(h, PCLOTH_ERR_STATE, "block-ELL copy before assemble");
  cudaSetDevice(h->device);
  const int rc = bell_build(h);
  if (rc == PCLOTH_OK && width) *width = h->bell_w;
  return rc;
}

int pcloth_spmv_bell(pcloth_t ht, const float* in, float* out) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (!in || !out) return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL vector");
  if (!h->bell_valid)
    return fail(h, PCLOTH_ERR_STATE, "no block-ELL copy of the current matrix (pcloth_bell_build)");
  cudaSetDevice(h->device);
  return launch_bell_spmv(h, in, out);
}

int pcloth_solve(pcloth_t ht, double tol, int32_t maxit, float* dv,
                 int32_t* iterations, double* rel_residual) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (!dv || maxit < 0 || !(tol >= 0.0))
    return fail(h, PCLOTH_ERR_INVALID_ARG, "bad dv, tol or maxit");
  if (!h->assembled) return fail(h, PCLOTH_ERR_STATE, "solve before assemble");
  cudaSetDevice(h->device);
  return pcg_solve(h, tol, maxit, dv, iterations, rel_residual);
}

int pcloth_solve_guess(pcloth_t ht, double tol, int32_t maxit, float* dv,
                       int32_t* iterations, double* rel_residual) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (!dv || maxit < 0 || !(tol >= 0.0))
    return fail(h, PCLOTH_ERR_INVALID_ARG, "bad dv, tol or maxit");
  if (!h->assembled) return fail(h, PCLOTH_ERR_STATE, "solve before assemble");
  cudaSetDevice(h->device);
  return pcg_solve(h, tol, maxit, dv, iterations, rel_residual, dv, false);
}

int pcloth_step_async(pcloth_t ht, float* x, float* v, const pcloth_springs* contacts,
                      float dt, double tol, int32_t maxit, float* dv) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (h->prof.on)
    return fail(h, PCLOTH_ERR_STATE,
                "profiling synchronises: turn it off for the asynchronous step");
  if (maxit < 0 || !(tol >= 0.0)) return fail(h, PCLOTH_ERR_INVALID_ARG, "bad tol or maxit");
  int rc = pcloth_assemble(ht, x, v, contacts, dt);
  if (rc != PCLOTH_OK) return rc;
  float* d = dv ? dv : h->dv;
  rc = pcg_solve(h, tol, maxit, d, nullptr, nullptr, nullptr, true);
  if (rc != PCLOTH_OK) return rc;
  return launch_state_update(h, x, v, d, dt);
}

int pcloth_step_result(pcloth_t ht, int32_t* iterations, double* rel_residual) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  cudaSetDevice(h->device);
  return pcg_result(h, iterations, rel_residual);
}

int pcloth_step(pcloth_t ht, float* x, float* v, const pcloth_springs* contacts,
                float dt, double tol, int32_t maxit, float* dv,
                int32_t* iterations, double* rel_residual) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  int rc = pcloth_assemble(ht, x, v, contacts, dt);
  if (rc != PCLOTH_OK) return rc;
  float* d = dv ? dv : h->dv;
  rc = pcloth_solve(ht, tol, maxit, d, iterations, rel_residual);
  if (rc != PCLOTH_OK && rc != PCLOTH_NOT_CONVERGED) return rc;
  int rc2 = launch_state_update(h, x, v, d, dt);
  if (rc2 != PCLOTH_OK) return rc2;
  int rc3 = collect_status(h);
  if (rc3 != PCLOTH_OK) return rc3;
  return rc;
}

int pcloth_step_host(pcloth_t ht, float* x, float* v,
                     const pcloth_springs* contacts, float dt, double tol,
                     int32_t maxit, int32_t* iterations, double* rel_residual) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (!x || !v) return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL x or v");
  if (contacts && (contacts->n < 0 || contacts->n > h->max_contacts))
    return fail(h, contacts->n < 0 ? PCLOTH_ERR_INVALID_ARG : PCLOTH_ERR_CAPACITY,
                "bad contact count");
  cudaSetDevice(h->device);
  const size_t vb = size_t(h->n) * 3 * sizeof(float);
  cudaError_t e = cudaMemcpyAsync(h->hx, x, vb, cudaMemcpyHostToDevice, h->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h->hv, v, vb, cudaMemcpyHostToDevice, h->stream);
  pcloth_springs dc{0, h->hci, h->hcj, h->hck, h->hcr};
  if (contacts && contacts->n > 0) {
    if (!contacts->i || !contacts->j || !contacts->k || !contacts->rest)
      return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL contact array");
    const size_t cb = size_t(contacts->n) * 4;
    dc.n = contacts->n;
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->hci, contacts->i, cb, cudaMemcpyHostToDevice, h->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->hcj, contacts->j, cb, cudaMemcpyHostToDevice, h->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->hck, contacts->k, cb, cudaMemcpyHostToDevice, h->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->hcr, contacts->rest, cb, cudaMemcpyHostToDevice, h->stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "host-to-device copy");
  int rc = pcloth_step(ht, h->hx, h->hv, &dc, dt, tol, maxit, nullptr, iterations,
                       rel_residual);
  if (rc != PCLOTH_OK && rc != PCLOTH_NOT_CONVERGED) return rc;
  e = cudaMemcpyAsync(x, h->hx, vb, cudaMemcpyDeviceToHost, h->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v, h->hv, vb, cudaMemcpyDeviceToHost, h->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "device-to-host copy");
  return rc;
}

int pcloth_nnzb(pcloth_t ht, int64_t* nnzb) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h || !nnzb) return fail(h, PCLOTH_ERR_INVALID_ARG, "NULL argument");
  if (!h->assembled) return fail(h, PCLOTH_ERR_STATE, "nnzb before assemble");
  cudaSetDevice(h->device);
  int rc = collect_status(h);
  if (rc != PCLOTH_OK) return rc;
  int32_t last = 0;
  cudaError_t e = cudaMemcpy(&last, h->rowptr + h->n, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "reading rowptr[n]");
  *nnzb = last;
  return PCLOTH_OK;
}

int pcloth_export(pcloth_t ht, int32_t* rowptr, int32_t* colind, float* vals,
                  float* b, float* pinv) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  int64_t nnzb = 0;
  int rc = pcloth_nnzb(ht, &nnzb);
  if (rc != PCLOTH_OK) return rc;
  cudaError_t e = cudaSuccess;
  const size_t n = size_t(h->n);
  if (rowptr) e = cudaMemcpyAsync(rowptr, h->rowptr, (n + 1) * 4, cudaMemcpyDefault, h->stream);
  if (colind && e == cudaSuccess)
    e = cudaMemcpyAsync(colind, h->colind, size_t(nnzb) * 4, cudaMemcpyDefault, h->stream);
  if (b && e == cudaSuccess)
    e = cudaMemcpyAsync(b, h->rhs, n * 12, cudaMemcpyDefault, h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "export copy");
  if (vals) {
    rc = launch_vals_expand(h, vals, nnzb);   // packed symmetric -> row-major 3x3
    if (rc != PCLOTH_OK) return rc;
  }
  if (pinv) {
    rc = launch_pinv_expand(h, pinv);
    if (rc != PCLOTH_OK) return rc;
  }
  e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "export copy");
  return PCLOTH_OK;
}

int pcloth_set_stream(pcloth_t ht, void* stream) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  h->stream = static_cast<cudaStream_t>(stream);
  return PCLOTH_OK;
}

int pcloth_sync(pcloth_t ht) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  cudaSetDevice(h->device);
  return collect_status(h);
}

const char* pcloth_last_error(pcloth_t ht) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  return h ? h->err.c_str() : g_create_err.c_str();
}

void pcloth_destroy(pcloth_t ht) { free_handle(reinterpret_cast<Handle*>(ht)); }

int pcloth_selftest_bounded_wait(int which, double limit_seconds, uint32_t* status) {
  g_create_err.clear();
  if (which < 0 || which > 2) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "which must be 0, 1 or 2");
  if (!(limit_seconds > 0.0) || !(limit_seconds <= 10.0))
    return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "limit_seconds must be in (0, 10]");
  return selftest_bounded_wait(which, limit_seconds, status);
}

int pcloth_solve_bsr3_static(int32_t n, const int32_t* rowptr, const int32_t* colind,
                             const float* vals, const float* b, double tol, int32_t maxit,
                             float* dv, int32_t* iterations, double* rel_residual,
                             void* stream) {
  g_create_err.clear();
  if (n > PCLOTH_STATIC_MAX_VERTS)
    return fail(nullptr, PCLOTH_ERR_CAPACITY,
                "n = " + std::to_string(n) + " exceeds PCLOTH_STATIC_MAX_VERTS = " +
                    std::to_string(PCLOTH_STATIC_MAX_VERTS));
  if (n <= 0 || !rowptr || !colind || !vals || !b || !dv || maxit < 0 || !(tol >= 0.0))
    return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "bad argument to pcloth_solve_bsr3_static");
  return pcg_solve_static(n, rowptr, colind, vals, b, tol, maxit, dv, iterations, rel_residual,
                          static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------- profiling ---
// Per-kernel-class device time accumulated from CUDA events recorded on the
// handle's stream around every launch while profiling is on.
int pcloth_profile_enable(pcloth_t ht, int on) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  h->prof.on = on != 0;
  h->prof.mode = on == 2 ? 2 : 1;
  return PCLOTH_OK;
}

int pcloth_profile_read(pcloth_t ht, double* ms_out, int64_t* counts_out, int reset) {
  Handle* h = reinterpret_cast<Handle*>(ht);
  if (!h) return fail(nullptr, PCLOTH_ERR_INVALID_ARG, "NULL handle");
  if (ms_out) {
    ms_out[0] = h->prof.assemble_ms;
    ms_out[1] = h->prof.spmv_ms;
    ms_out[2] = h->prof.update_ms;
    ms_out[3] = h->prof.solve_ms;
  }
  if (counts_out) {
    counts_out[0] = h->prof.assemble_calls;
    counts_out[1] = h->prof.spmv_launches;
    counts_out[2] = h->prof.update_launches;
    counts_out[3] = h->prof.solves;
    counts_out[4] = h->prof.iterations;
    counts_out[5] = h->launches;
    counts_out[6] = h->prof.samples;
  }
  if (reset) {
    const bool on = h->prof.on;
    const int mode = h->prof.mode;
    h->prof = Profile();
    h->prof.on = on;
    h->prof.mode = mode;
    h->launches = 0;
  }
  return PCLOTH_OK;
}

}  // extern "C"
