/*
 * pcloth.h - C ABI of the GB300 implicit-integration hot path of P-Cloth.
 *
 * P-Cloth (arXiv 2008.00409, "P-Cloth: Interactive Complex Cloth Simulation on
 * Multi-GPU Systems using Dynamic Matrix Assembly and Pipelined Implicit
 * Integrators") integrates a cloth of p vertices with backward Euler
 * (Sec. 2.5, Eq. (1)-(3)).  Each time step it
 *
 *   1. assembles the 3x3-block sparse system
 *        A dv = b,   A = M + h^2 sum_e K_e,   b = h f(x_t + h v_t)
 *      from every spring and contact element e = (i, j, k, L0) (Sec. 3.2,
 *      "assembly elements"; Sec. 3.2.2, sparse matrix filling), with
 *        K_e = k [ max(0, 1 - L0/l) (I - d d^T) + d d^T ]  at x_t,
 *        F_e = k (l~ - L0) d~                             at x~ = x_t + h v_t,
 *      K_e added to blocks (i,i), (j,j) and subtracted from (i,j), (j,i);
 *      f_i = sum of element forces on i plus m_i g;
 *   2. solves it by preconditioned conjugate gradients (Sec. 3.1 and the text
 *      after Eq. (3)); the preconditioner here is block Jacobi (the inverse
 *      of each 3x3 diagonal block), whose inner loop is the block sparse
 *      matrix-vector product (Sec. 3.1, "the most computationally expensive
 *      operator");
 *   3. updates the state v += dv, x += h v.
 *
 * Storage (all on the device, owned by the library unless noted):
 *   matrix     BSR3: rowptr int32[n+1], colind int32[nnzb] (sorted per row,
 *              unique, diagonal always present), block values with rows
 *              consecutive.  Every block of A is symmetric (a sum of the
 *              symmetric K_e, plus m_i I on the diagonal), so the library
 *              holds each packed as six floats (a00 a01 a02 a11 a12 a22),
 *              float32[nnzb][6]; pcloth_export expands them to row-major
 *              float32[nnzb][3][3];
 *   vectors    float32[n][3] (x, y, z interleaved per vertex).
 * The pattern of the springs is built once by pcloth_create; every
 * pcloth_assemble merges that step's contact pairs into it in place, inside
 * buffers sized at create for n + 2 * n_springs + 2 * max_contacts blocks, so
 * no call after create allocates device memory.
 *
 * Streams: every call enqueues its work on the stream given at create (or by
 * pcloth_set_stream) and returns without waiting, except where a call's
 * comment says it synchronises.  Calls on one handle are not thread safe.
 *
 * Errors: every int-returning call returns PCLOTH_OK (0), PCLOTH_NOT_CONVERGED
 * (1, results still valid) or a negative code.  Errors found by a kernel
 * (bad index, capacity, non-finite value) are recorded in a device status
 * word and reported by the next synchronising call (pcloth_solve,
 * pcloth_step, pcloth_export, pcloth_nnzb, pcloth_sync); the status is then
 * cleared.  pcloth_last_error returns a message for the last failure.
 */
#ifndef PCLOTH_H_
#define PCLOTH_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  PCLOTH_OK = 0,
  PCLOTH_NOT_CONVERGED = 1,    /* maxit reached; dv, iterations, residual valid */
  PCLOTH_ERR_INVALID_ARG = -1, /* null/negative/out-of-order argument         */
  PCLOTH_ERR_CAPACITY = -2,    /* more contacts than max_contacts, or sizes
                                  beyond the int32 index range               */
  PCLOTH_ERR_BAD_INDEX = -3,   /* element index outside [0, n) or i == j      */
  PCLOTH_ERR_NONFINITE = -4,   /* NaN/Inf in x, v, the system or a residual,
                                  or a zero-length element                   */
  PCLOTH_ERR_BREAKDOWN = -5,   /* PCG: p.Ap <= 0 or r.z < 0 (not SPD)         */
  PCLOTH_ERR_CUDA = -6,        /* a CUDA runtime call failed                  */
  PCLOTH_ERR_STATE = -7        /* call out of order (solve before assemble)   */
};

typedef struct pcloth* pcloth_t; /* opaque handle, owned by the library */

/* The cloth: n_verts vertices with masses (device pointer, float32[n_verts],
 * kg) and a uniform gravity acceleration (m/s^2, e.g. {0, 0, -9.8}).
 * Sec. 2.5: M is the (block-diagonal) mass matrix of Eq. (1). */
typedef struct {
  int32_t n_verts;
  const float* mass;
  float gravity[3];
} pcloth_mesh;

/* A list of n elements (springs or contacts), device pointers:
 * i, j int32[n] vertex indices (i != j, both in [0, n_verts)), k float32[n]
 * stiffness (N/m), rest float32[n] rest length (m).  Sec. 3.2: the
 * "assembly elements" that form f and J of Eq. (3); contacts are penalty
 * springs of the same law.  Duplicated pairs are summed into one block. */
typedef struct {
  int32_t n;
  const int32_t* i;
  const int32_t* j;
  const float* k;
  const float* rest;
} pcloth_springs;

/* Options: max_contacts sizes the per-step contact buffers; device is the
 * CUDA device ordinal; stream is a cudaStream_t (0 = the legacy default
 * stream). */
typedef struct {
  int32_t max_contacts;
  int device;
  void* stream;
} pcloth_opts;

/* Create a handle for a cloth and its (static) springs.  Copies the springs
 * to the host once, validates them (PCLOTH_ERR_BAD_INDEX on a bad index),
 * builds the static block pattern (Sec. 3.2.2 steps 1-3: diagonal plus both
 * directions of every spring, sorted, duplicates merged) and allocates every
 * device buffer at its capacity.  Synchronises.  On failure *out is NULL. */
int pcloth_create(const pcloth_mesh* mesh, const pcloth_springs* springs,
                  const pcloth_opts* opts, pcloth_t* out);

/* Assemble the step's system at state (x, v) (device float32[n][3]) with
 * time step h and this step's contacts (may be NULL or n = 0): evaluates
 * every element (K_e at x, F_e at x + h v), merges the contact pairs into the
 * pattern (key sort, rows rebuilt in place), fills the block values
 * A = M + h^2 sum K_e, the right-hand side b = h f and the block-Jacobi
 * inverses.  Sec. 2.5 Eq. (3); Sec. 3.2.2 steps 1-5.  Asynchronous;
 * PCLOTH_ERR_CAPACITY if contacts->n > max_contacts (checked on the host). */
int pcloth_assemble(pcloth_t h, const float* x, const float* v,
                    const pcloth_springs* contacts, float dt);

/* out = A in for the last assembled A (device float32[n][3] each; in and
 * out must not overlap).  Sec. 3.1 (SpMV).  Asynchronous. */
int pcloth_spmv(pcloth_t h, const float* in, float* out);

/* Vertex-vertex proximity contacts by spatial hashing (P-Cloth Sec. 4.2: a
 * spatial-hash table built every step, then proximity tests; Sec. 4.3:
 * proximities enter the implicit integrator as forces), restricted to pairs
 * of vertices.  Every pair i < j of vertices at x (device float32[n][3])
 * closer than `radius` that is not a spring becomes a contact: a spring
 * (i, j, stiffness, rest = radius), the same element law as the springs.
 * The distance test is taken in float32 with every operation rounded:
 * ((dx dx + dy dy) + dz dz) < radius * radius, d = x_j - x_i.  The pairs are
 * written in (i, j) order into the caller's device arrays out->i, out->j
 * (int32), out->k, out->rest (float32) of length `capacity`; out->n is set
 * to their number, which is ready to pass to pcloth_assemble / pcloth_step.
 * *found (may be NULL) receives the number of pairs found (at most
 * 2^31 - 1; the count itself is taken in 64 bits).  If more than
 * min(capacity, max_contacts) exist, nothing is written, out->n = 0 and
 * PCLOTH_ERR_CAPACITY is returned.  Cells have edge 2 radius (1 + 2^-7) and
 * each vertex searches the 8 cells that can hold a partner, which finds
 * every pair for coordinates within 2^14 cells of the origin.
 * Synchronises. */
int pcloth_find_contacts(pcloth_t h, const float* x, float radius, float stiffness,
                         pcloth_springs* out, int32_t capacity, int32_t* found);

/* Block-ELL comparison path (P-Cloth Sec. 3.2.2: the pages' index and value
 * tables, padded to the longest compacted row, read by one thread per row).
 * pcloth_bell_build copies the last assembled matrix into that layout:
 * W = the longest row in blocks, slot s of row i at s * n + i, column
 * indices int32[W * n] (-1 past a row's end) and six planes of the packed
 * symmetric block values float32[6][W * n].  It writes W to *width (may be
 * NULL) and synchronises.  It is the one call after create that may
 * allocate device memory (the tables grow to the largest W * n seen, and are
 * freed by pcloth_destroy).  The copy is invalid after the next assembly.
 * pcloth_spmv_bell computes out = A in (device float32[n][3] each) from the
 * copy, adding the same products in the same order as pcloth_spmv, so the
 * two give the same bits; PCLOTH_ERR_STATE if there is no valid copy.
 * Asynchronous. */
int pcloth_bell_build(pcloth_t h, int32_t* width);
int pcloth_spmv_bell(pcloth_t h, const float* in, float* out);

/* Solve A dv = b by block-Jacobi PCG from dv = 0 until
 * |r|_2 <= tol |b|_2 (recursive residual) or maxit iterations; dv is device
 * float32[n][3]; *iterations and *rel_residual (= |r|/|b|) are written on
 * the host.  Sec. 3.1 / Eq. (3).  The whole solve is one cooperative kernel
 * launch (all of its CTAs resident; grid-wide barriers between the SpMV and
 * vector phases of each iteration), so the host does not take part in the
 * iteration.  Synchronises at the end. */
int pcloth_solve(pcloth_t h, double tol, int32_t maxit, float* dv,
                 int32_t* iterations, double* rel_residual);

/* pcloth_solve from an initial iterate: dv (device float32[n][3]) holds the
 * guess on entry and the solution on return.  The iteration starts from
 * r = b - A dv, z = P r, p = z (the textbook PCG with a nonzero first
 * iterate; Sec. 3.1 / Eq. (3)); the stop test is the same, |r|_2 <= tol |b|_2
 * on the recursive residual, and a guess that already meets it returns after
 * 0 iterations with *rel_residual = |b - A dv| / |b|.  b = 0 gives dv = 0.
 * Costs one extra SpMV pass.  Synchronises at the end. */
int pcloth_solve_guess(pcloth_t h, double tol, int32_t maxit, float* dv,
                       int32_t* iterations, double* rel_residual);

/* pcloth_step with no host synchronisation and no host-side read, so that a
 * caller can capture it in a CUDA graph (with the handle's stream set to the
 * capturing stream) and replay it: it enqueues the assembly, the solve and
 * the state update on the handle's stream and returns.  The solve's
 * iterations, residual and status stay on the device until
 * pcloth_step_result reads them.  Pointers (x, v, dv and the contacts'
 * arrays) are baked into a captured graph: to replay it for another step,
 * write that step's contacts into the same arrays (contacts->n is captured
 * too).  dv may be NULL (library scratch).  Profiling must be off
 * (PCLOTH_ERR_STATE otherwise: it synchronises).  Errors found on the host
 * (arguments, contact count) are returned at once. */
int pcloth_step_async(pcloth_t h, float* x, float* v, const pcloth_springs* contacts,
                      float dt, double tol, int32_t maxit, float* dv);

/* The outcome of the last solve enqueued by pcloth_step_async: waits for the
 * handle's stream, writes *iterations and *rel_residual (either may be NULL)
 * and returns the solve's code (PCLOTH_OK, PCLOTH_NOT_CONVERGED or an error,
 * as pcloth_step would have).  Synchronises. */
int pcloth_step_result(pcloth_t h, int32_t* iterations, double* rel_residual);

/* One whole implicit step: assemble at (x, v), solve, then update the state
 * in place: v += dv, x += dt v (Eq. (3) with backward Euler).  x, v device
 * float32[n][3]; dv may be NULL (library scratch is used).  Synchronises. */
int pcloth_step(pcloth_t h, float* x, float* v, const pcloth_springs* contacts,
                float dt, double tol, int32_t maxit, float* dv,
                int32_t* iterations, double* rel_residual);

/* pcloth_step with HOST buffers: x, v are host float32[n][3] (pinned memory
 * recommended), contacts' pointers are host arrays.  Copies the inputs to
 * library-owned device buffers, runs the step and copies x, v back.
 * Synchronises. */
int pcloth_step_host(pcloth_t h, float* x, float* v,
                     const pcloth_springs* contacts, float dt, double tol,
                     int32_t maxit, int32_t* iterations, double* rel_residual);

/* Number of blocks of the last assembled matrix (synchronises). */
int pcloth_nnzb(pcloth_t h, int64_t* nnzb);

/* Copy the last assembled system into caller-owned device buffers (any may
 * be NULL): rowptr int32[n+1], colind int32[nnzb], vals float32[nnzb*9]
 * (row-major 3x3 blocks, expanded from the packed symmetric storage), b
 * float32[n*3], pinv float32[n*9] (the block-Jacobi inverses, row-major).
 * vals and pinv must be device memory (a kernel writes them).
 * Synchronises. */
int pcloth_export(pcloth_t h, int32_t* rowptr, int32_t* colind, float* vals,
                  float* b, float* pinv);

/* Replace the stream used by later calls. */
int pcloth_set_stream(pcloth_t h, void* stream);

/* Wait for the handle's stream and report any device-side error. */
int pcloth_sync(pcloth_t h);

/* Message for the last error on this handle ("" if none); NULL handle gives
 * the message of the last failed pcloth_create. */
const char* pcloth_last_error(pcloth_t h);

/* Profiling: while enabled (on != 0; 1 and 2 behave alike), the library
 * records CUDA events on its stream around every assembly and around every
 * launch of the PCG kernel, and the PCG kernel times its phases with the
 * GPU's global timer (the SpMV phase up to the barrier after it; the two
 * vector phases up to theirs).  pcloth_profile_read fills ms_out[4] =
 * {assembly, PCG SpMV phases, PCG vector phases, PCG kernel launches} in
 * milliseconds and counts_out[7] = {assemblies, SpMV phases, vector-phase
 * pairs, solves, PCG iterations, kernels launched by this handle, timed SpMV
 * phases}; divide a phase time by the timed count for a per-iteration
 * average.  reset != 0 zeroes the accumulators and keeps the mode. */
int pcloth_profile_enable(pcloth_t h, int on);
int pcloth_profile_read(pcloth_t h, double* ms_out, int64_t* counts_out,
                        int reset);

/* Allocation-free solve.  The paper has no counterpart: this entry point is
 * for callers that cannot allocate GPU memory when they need a solve -- a
 * host application that reserves the GPU's memory for itself and forbids
 * plug-ins to allocate, or a real-time loop in which an allocation's latency
 * or failure mid-frame is unacceptable.  It solves A dv = b for a BSR3
 * matrix the caller already holds, with the same block-Jacobi PCG as
 * pcloth_solve, on the current device and the given stream (a cudaStream_t,
 * 0 = legacy default), and returns *iterations and *rel_residual on the
 * host.
 *
 * Arguments (device pointers, owned by the caller):
 *   rowptr  int32[n+1], rowptr[0] = 0, non-decreasing;
 *   colind  int32[rowptr[n]], each row's columns in [0, n), strictly
 *           increasing, with the diagonal block present;
 *   vals    float32[rowptr[n]][3][3], row-major blocks;
 *   b       float32[n][3];  dv  float32[n][3] (output).
 * A must be symmetric positive definite (so every diagonal block is
 * symmetric); the preconditioner inverts each diagonal block from the six
 * entries of its upper triangle.  rowptr, colind and vals must be 16-byte
 * aligned (PCLOTH_ERR_INVALID_ARG otherwise, checked before any launch), and
 * each must be followed by at least 16 bytes of readable device memory
 * (for example the rest of a larger allocation): the solve streams them in
 * whole 16-byte words, so its last copy of each can read up to 12 bytes past
 * the end.  The pattern is checked on the device before the solve starts --
 * reading rowptr and colind only as values -- and a malformed one returns
 * PCLOTH_ERR_BAD_INDEX without launching the solve.
 *
 * It allocates nothing: all of its scratch is one fixed array compiled into
 * this library, 1,513,216 bytes (about 1.44 MiB), which every GPU that loads
 * the library holds until the process exits.  n may be at most
 * PCLOTH_STATIC_MAX_VERTS; larger n returns PCLOTH_ERR_CAPACITY without
 * touching the GPU.  Every call on a device shares that array, which keeps
 * the last call's contents (each call sets up what it reads), so calls that
 * overlap on the GPU race: order them (one stream, or events).
 *
 * The first call on each device looks up the array's device address and,
 * with CUDA's lazy module loading, may be what loads this library's device
 * code and with it the array itself: make one warm-up call at
 * initialisation, before any window in which nothing may allocate and
 * before any stream capture.  Synchronises (once after the pattern check,
 * once at the end).  Errors are described by pcloth_last_error(NULL). */
#define PCLOTH_STATIC_MAX_VERTS 16384
int pcloth_solve_bsr3_static(int32_t n, const int32_t* rowptr, const int32_t* colind,
                             const float* vals, const float* b, double tol, int32_t maxit,
                             float* dv, int32_t* iterations, double* rel_residual,
                             void* stream);

/* Self-test of the device-side bounded waits that keep every kernel of this
 * library from hanging.  which = 0 runs the SpMV pipeline's mbarrier wait on
 * a barrier phase that gets no arrival; which = 1 runs the PCG grid
 * barrier's counter poll on a counter that gets one arrival of the two it
 * waits for; both wait limit_seconds (0 < limit_seconds <= 10; the
 * library's own waits use 2 s), give up and record the timeout.  which = 2
 * runs the PCG grid barrier itself in one cooperative launch of two CTAs,
 * one of which arrives marked as having timed out (its arrival carries the
 * mark, as after a real timeout): both CTAs must leave the barrier with the
 * timeout verdict at once.  The device status word is copied to *status (if
 * not NULL): bit 4 = a wait gave up; for which = 2, bits 8-15 = how many of
 * the two CTAs left the barrier with the verdict.  Runs on the current
 * device's legacy stream.  Returns PCLOTH_ERR_CUDA with the message "device
 * wait timed out" -- what a real timeout reports -- when the timeout was
 * recorded as designed, PCLOTH_OK if it was not, PCLOTH_ERR_INVALID_ARG for
 * a bad argument.  Allocates 64 bytes of device memory for the call and
 * synchronises the device; the GPU context stays usable afterwards.  Errors
 * are described by pcloth_last_error(NULL). */
int pcloth_selftest_bounded_wait(int which, double limit_seconds, uint32_t* status);

/* Free every buffer of the handle (synchronises its stream first). */
void pcloth_destroy(pcloth_t h);

#ifdef __cplusplus
}
#endif

#endif /* PCLOTH_H_ */
