/*
 * muon_ns.h — C ABI of a GB300 (sm_103a) library for batched quintic
 * Newton–Schulz (NS) orthogonalisation, the inner loop of the Muon optimizer
 * step.
 *
 * What is computed (per matrix G of a stack, rows x cols, bf16 in and out):
 *
 *   X <- G / (||G||_F + eps)
 *   if rows > cols: X <- X^T                       (internal m x n, m <= n)
 *   repeat `steps` times:  A = X X^T;  B = b A + c A A;  X = a X + B X
 *   if transposed: X <- X^T
 *
 * The three products are those of prime-rl PR #3873, Summary item 1
 * ("Symmetric-GEMM Newton–Schulz": X·X^T, b·A + c·A·A, a·X + B·X, inside
 * Dion's dense zeropower_via_newtonschulz5).  The leading axis of a stack is a
 * batch of independent matrices (prime-rl PR #3873, Summary item 2;
 * param-decomp PR #978 "stacked-NS Muon", What).  `steps` is the `ns_steps`
 * setting of param-decomp PR #978 (default 5).  The default coefficients
 * (a, b, c) = (3.4445, -4.7750, 2.0315), eps = 1e-7 and the transpose rule
 * (transpose iff rows > cols) are the standard Muon quintic, which the pages
 * name but do not print.
 *
 * Numerics: bf16 storage of X, A and B between steps; every product
 * accumulates in fp32 on the tensor cores and every epilogue (b·A + c·(A A),
 * a·X + B X) runs in fp32 and rounds once to bf16, as the fp32 alpha/beta
 * epilogue of prime-rl PR #3873 (Results, note under the microbenchmark).
 * A and B are symmetric and one triangle of each is computed (prime-rl PR
 * #3873, Summary item 1; Megatron-LM PR #6381 "Add --muon-use-syrk option",
 * Summary).  The per-step entry points mirror it, so the stored matrix is
 * bit-symmetric; the whole-call entry points store it half (MUON_NS_HALF
 * below): whole inside the diagonal 256 x 256 blocks, the lower triangle
 * elsewhere, and the next product reads the rest of the upper triangle
 * transposed from the lower one.  The diagonal of B is kept in fp32
 * (B = D + O, O bf16 with a zero diagonal) and the update applies (a + D)
 * in its fp32 epilogue: the same arithmetic, with the part of B that
 * dominates near convergence kept out of bf16 rounding.
 *
 * Conventions for every entry point below:
 *   - Matrices are contiguous row-major stacks [batch][rows][cols] of raw
 *     bf16 bit patterns (muon_bf16) in DEVICE memory owned by the caller
 *     (muon_ns_host() alone takes its stacks in host memory).
 *   - rows and cols must be multiples of 8 and every device pointer must be
 *     16-byte aligned (16-byte rows for TMA; prime-rl PR #3873, Summary
 *     item 1, has the same divisible-by-8 rule).  This is an
 *     error (MUON_NS_ERR_ALIGNMENT), never a silent fallback (Megatron-LM PR
 *     #6381, "Version compatibility": a hard failure instead of a fallback).
 *   - batch == 0, rows == 0 or cols == 0 is an empty problem: MUON_NS_OK,
 *     nothing is launched and pointers may be NULL.
 *   - Work is enqueued on `stream` (NULL = legacy default stream) and the call
 *     returns without synchronising.  Arguments are validated on the host
 *     before anything is launched; a non-OK status means nothing was enqueued
 *     (except MUON_NS_ERR_CUDA, which reports a failed launch).
 *   - Only GPUs of compute capability 10.3 (sm_103) are supported; others get
 *     MUON_NS_ERR_UNSUPPORTED_DEVICE.  The kernels are built for sm_103a
 *     alone (tcgen05, TMA), so no other device could run them.
 *   - One GPU per process.  Products with contractions up to 1024 run on
 *     pairs of CTAs that load a shared operand panel with TMA multicast within
 *     their cluster; every tensor map covers only buffers on the calling GPU,
 *     and nothing in the library exchanges data between GPUs.  Processes that
 *     drive more than one GPU are not a supported use.
 *   - Limits: batch, rows, cols <= 1<<20 and each matrix below 2^31 elements.
 *     Magnitudes: ||G_k||_F below about 1.8e19 (the norm and the first Gram
 *     accumulate in fp32); above it the norm overflows and the output is 0.
 *   - Errors found on the device (a bounded wait inside a kernel that ran out)
 *     set a device error word; the call that launched the kernels cannot
 *     see it, muon_ns_read_error() / muon_ns_cached_error() can.
 */
#ifndef MUON_NS_H
#define MUON_NS_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t muon_bf16; /* raw bfloat16 bit pattern */

/* Status codes returned by every entry point. */
enum {
  MUON_NS_OK = 0,
  MUON_NS_ERR_INVALID_ARG = 1,        /* NULL pointer, negative size, steps < 0, bad eps, too large */
  MUON_NS_ERR_ALIGNMENT = 2,          /* rows/cols not multiples of 8, or a pointer not 16-byte aligned */
  MUON_NS_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
  MUON_NS_ERR_WORKSPACE = 4,          /* workspace NULL/too small, or cache too small during graph capture */
  MUON_NS_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
  MUON_NS_ERR_TIMEOUT = 6             /* a kernel's bounded wait ran out (reported through the error word) */
};

/* Bits of the device error word. */
#define MUON_NS_DEVERR_WAIT_TIMEOUT 1

/* Library version string, e.g. "0.1.0". */
const char* muon_ns_version(void);

/* Human-readable name of a status code (static storage). */
const char* muon_ns_status_string(int status);

/* Returns MUON_NS_OK if `device` (or the current device when device < 0) is
 * supported, else MUON_NS_ERR_UNSUPPORTED_DEVICE (or MUON_NS_ERR_CUDA). */
int muon_ns_device_supported(int device);

/* ---------------------------------------------------------------------------
 * Whole NS call.
 * ------------------------------------------------------------------------- */

/* Workspace regions, for muon_ns_workspace_region(). */
enum {
  MUON_NS_WS_TOTAL = 0,   /* whole workspace (offset 0) */
  MUON_NS_WS_ERROR = 1,   /* int32 device error word */
  MUON_NS_WS_NORMS = 2,   /* fp32 [batch]: ||G_k||_F of the last call */
  MUON_NS_WS_X = 3,       /* bf16 [batch][rows][cols]: ping-pong iterate */
  MUON_NS_WS_GRAM = 4,    /* bf16 [batch][m][m]: A of the last step, m = min(rows, cols); the
                             whole-call entry points store its lower triangle and its diagonal
                             256 x 256 blocks only (the products read the rest transposed) */
  MUON_NS_WS_POLY = 5,    /* bf16 [batch][m][m]: off-diagonal part of B of the last step, stored
                             like A */
  MUON_NS_WS_DIAG = 6     /* fp32 [batch][m]: diagonal of B of the last step */
};

/* Size of the workspace muon_ns_ws() needs for this problem, in bytes.
 * Returns MUON_NS_OK or MUON_NS_ERR_INVALID_ARG / MUON_NS_ERR_ALIGNMENT. */
int muon_ns_workspace_size(int batch, int rows, int cols, size_t* bytes);

/* Offset and size in bytes of one region of the workspace (layout above).
 * Tests read A (MUON_NS_WS_GRAM) after a call with steps = 1 to check its
 * stored part against the definition. */
int muon_ns_workspace_region(int batch, int rows, int cols, int region, size_t* offset, size_t* bytes);

/* out = NS(G) for a stack of `batch` matrices of rows x cols.
 *   G, out     device, bf16 [batch][rows][cols]; out == G is allowed (in-place);
 *              otherwise the two must not overlap.
 *   steps      >= 0; steps == 0 returns G / (||G||_F + eps).
 *   coeffs     host pointer to (a, b, c); NULL selects (3.4445, -4.7750, 2.0315).
 *   eps        >= 0 and finite.  With eps == 0 an all-zero matrix gives NaN (0/0),
 *              as the definition does; with eps > 0 it gives zeros.
 *   workspace  device, >= muon_ns_workspace_size() bytes, 256-byte aligned,
 *              caller-owned.  Nothing is allocated and nothing synchronises,
 *              so the call can be captured in a CUDA graph.
 * Kernel launches per call: 1 + 3 * steps (the norm, then per step the Gram,
 * polynomial and update kernels); 2 when steps == 0 (norm and scale).  The
 * first step reads G itself and applies s = 1 / (||G||_F + eps) in its
 * epilogues (A0 = s^2 G G^T, X1 = s (a + D) G + s O G), so no scaled copy of G
 * is made and X0 is never rounded to bf16.  In place with an odd step count
 * the result is copied once from the workspace into out at the end.
 * For stacks of two or more matrices each product kernel waits for the
 * previous product of the same matrix (per-matrix completion counters in the
 * workspace, bounded waits that report MUON_NS_ERR_TIMEOUT through the error
 * word) rather than for the whole previous kernel, so consecutive kernels
 * overlap; the call's last kernel still completes after all the others, so
 * work queued after the call on `stream` sees every result. */
int muon_ns_ws(const muon_bf16* G, muon_bf16* out, int batch, int rows, int cols, int steps,
               const float* coeffs, float eps, void* workspace, size_t workspace_bytes,
               cudaStream_t stream);

/* As muon_ns_ws() with a workspace cached by the library per device (grown
 * with cudaMalloc when too small, never freed before exit).  Growing is
 * refused with MUON_NS_ERR_WORKSPACE while `stream` is being captured.
 * Every muon_ns() call on a device shares that workspace, so calls that may
 * run at the same time on the GPU (different streams) must use muon_ns_ws()
 * with a workspace each: a shared workspace would mix their iterates and
 * their per-matrix completion counters. */
int muon_ns(const muon_bf16* G, muon_bf16* out, int batch, int rows, int cols, int steps,
            const float* coeffs, float eps, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * fp32 NS (the `ns_dtype: float32` setting of param-decomp PR #978, What).
 * G and out are fp32 [batch][rows][cols]; X, A and B are stored in fp32
 * rounded to tf32 (10-bit mantissa, round to nearest even) and multiplied on
 * the tf32 tensor cores with fp32 accumulation; the epilogues, B's diagonal
 * and the final output are full fp32.  About 7x closer to the exact result
 * than the bf16 path, at about twice its time and memory.  Every tensor-core
 * operand is read K-major here: the iterate is kept in both orientations (the
 * update also writes its transpose), and the first step makes one transposed
 * copy of G.  Same argument
 * rules as the bf16 calls (rows and cols multiples of 8, 16-byte aligned
 * pointers, out == G allowed).
 * ------------------------------------------------------------------------- */

/* Workspace bytes / regions for muon_ns_ws_f32 (regions as for the bf16 call,
 * with fp32 X, GRAM and POLY regions). */
int muon_ns_f32_workspace_size(int batch, int rows, int cols, size_t* bytes);
int muon_ns_f32_workspace_region(int batch, int rows, int cols, int region, size_t* offset,
                                 size_t* bytes);

/* out = NS(G) in fp32 mode; otherwise as muon_ns_ws().  Launches per call:
 * 1 + 3 * steps (2 if steps == 0). */
int muon_ns_ws_f32(const float* G, float* out, int batch, int rows, int cols, int steps,
                   const float* coeffs, float eps, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Several stacks in one call (e.g. every Muon parameter group of an optimizer
 * step): same-shape matrices are stacked, as param-decomp PR #978 (What)
 * stacks same-shape leaves; stacks of different shapes run through the same
 * launches, so small stacks do not leave SMs idle.
 * ------------------------------------------------------------------------- */

/* One stack of a grouped call: `batch` matrices of rows x cols, device bf16,
 * contiguous [batch][rows][cols]; out == G allowed, otherwise no overlap
 * (with any other stack either). */
typedef struct {
  const muon_bf16* G;
  muon_bf16* out;
  int batch;
  int rows;
  int cols;
} muon_ns_stack;

/* Workspace bytes for muon_ns_grouped(): the per-stack workspaces of
 * muon_ns_workspace_size() laid end to end (non-empty stacks, in order). */
int muon_ns_grouped_workspace_size(const muon_ns_stack* stacks, int num_stacks, size_t* bytes);

/* NS of every stack (host array of num_stacks <= 64 descriptors) with one set
 * of steps / coefficients / eps.  Each step runs as one Gram, one polynomial
 * and one update launch for up to 8 stacks of the same orientation (wide:
 * rows <= cols; tall: rows > cols) at a time, plus one norm launch per stack.
 * Results are bit-identical to calling muon_ns_ws() on each stack alone.
 * The device error word is the first 4 bytes of the workspace
 * (muon_ns_read_error).  Validation, aliasing and errors as for muon_ns_ws;
 * empty stacks are skipped. */
int muon_ns_grouped(const muon_ns_stack* stacks, int num_stacks, int steps, const float* coeffs,
                    float eps, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Stacks held in host memory (e.g. optimizer states kept on the CPU).  The
 * stack is processed in chunks of `chunk` matrices: each chunk is uploaded,
 * orthogonalised and downloaded, and the copies of one chunk overlap the
 * compute of its neighbours (two chunks in flight; uploads, each followed by
 * its chunk's norm pass, and downloads run on two streams the library creates
 * once per device, the products on `stream`).  The matrices of a stack are independent (the leading axis is
 * the batch, prime-rl PR #3873, Summary item 2), so the result equals
 * muon_ns_ws() on the whole stack bit for bit.  Host buffers should be
 * page-locked (cudaHostAlloc, or a pinned torch tensor) for the copies to
 * overlap; pageable memory gives the same result without overlap.
 * ------------------------------------------------------------------------- */

/* Device workspace bytes for muon_ns_host(): the call's error word (256
 * bytes, then padding to 1 KB) and two slots of (input chunk, output chunk,
 * muon_ns_ws() workspace of one chunk of `chunk` matrices).  `chunk` is the
 * largest chunk: when the stack is larger, the first and the last chunk take
 * ceil(chunk / 2) matrices (shorter upload before the first compute and
 * download after the last) and the ones between `chunk`, the one before the
 * last the remainder (muon_ns_host_plan gives the sizes).  chunk <= 0 selects
 * the default: the whole stack if it holds less than 32 MiB, else
 * ceil(96 MiB / (2 * rows * cols)) matrices but at most ceil(batch / 2).
 * chunk > batch is clamped to batch.  Returns MUON_NS_OK or
 * MUON_NS_ERR_INVALID_ARG / MUON_NS_ERR_ALIGNMENT as muon_ns_workspace_size(). */
int muon_ns_host_workspace_size(int batch, int rows, int cols, int chunk, size_t* bytes);

/* Largest chunk, in matrices, that muon_ns_host() uses for this stack and
 * `chunk` argument (the default rule above for chunk <= 0); 0 for an empty
 * stack or invalid sizes. */
int muon_ns_host_chunk(int batch, int rows, int cols, int chunk);

/* The chunk sizes, in order, that muon_ns_host() uses for this stack and
 * `chunk` argument: writes min(count, max_chunks) sizes to `sizes` (may be
 * NULL) and returns the count (0 for an empty stack, -1 on invalid sizes).
 * Host-only. */
int muon_ns_host_plan(int batch, int rows, int cols, int chunk, int* sizes, int max_chunks);

/* out_host = NS(G_host).
 *   G_host, out_host  host, bf16 [batch][rows][cols]; they may be the same
 *                     buffer, otherwise they must not overlap;
 *   chunk             largest chunk, as above (<= 0: the default);
 *   workspace         device, >= muon_ns_host_workspace_size() bytes,
 *                     256-byte aligned, caller-owned.
 * Everything is enqueued and the call returns: `stream` completes after the
 * last download, so synchronise it before reading out_host.  The device
 * error word is the workspace's first int (muon_ns_read_error()).  Kernel
 * launches: 1 + 3 * steps per chunk; one cudaMemcpyAsync per chunk and
 * direction.  Errors as muon_ns_ws(); MUON_NS_ERR_CUDA if a copy, stream or
 * event operation fails. */
int muon_ns_host(const muon_bf16* G_host, muon_bf16* out_host, int batch, int rows, int cols,
                 int steps, const float* coeffs, float eps, int chunk, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/* Synchronises `stream`, copies the device error word of `workspace` into
 * *device_error (0 = none) and, if `clear` is nonzero, resets it.  Returns
 * MUON_NS_ERR_TIMEOUT if the word is nonzero, else MUON_NS_OK or an error. */
int muon_ns_read_error(const void* workspace, int* device_error, int clear, cudaStream_t stream);

/* Asynchronous check of a call's device error word: enqueues on `stream` one
 * copy of the first int of `workspace` (a muon_ns_ws(), muon_ns_grouped() or
 * muon_ns_host() workspace) into *host_word and returns without
 * synchronising or allocating, so the check can follow a call inside a
 * captured CUDA graph and is replayed with it.
 *   host_word  page-locked (cudaHostAlloc, cudaHostRegister, a pinned torch
 *              tensor) or managed memory, owned by the caller; pageable memory
 *              is rejected with MUON_NS_ERR_INVALID_ARG, since its copy would
 *              synchronise.
 * Read *host_word once the stream has passed the copy (synchronise the stream
 * or an event recorded after this call): 0 = no kernel reported an error;
 * MUON_NS_DEVERR_WAIT_TIMEOUT set = a bounded wait ran out, i.e. the call's
 * status is MUON_NS_ERR_TIMEOUT.  The next whole call on the workspace clears
 * the word.  Returns MUON_NS_OK, MUON_NS_ERR_INVALID_ARG (NULL or pageable
 * pointer), MUON_NS_ERR_ALIGNMENT (workspace not 256-byte aligned) or
 * MUON_NS_ERR_CUDA (the copy could not be enqueued).  This is the
 * asynchronous counterpart of muon_ns_read_error(), which synchronises. */
int muon_ns_check(const void* workspace, int* host_word, cudaStream_t stream);

/* Same for the workspace cached by muon_ns() on `device` (synchronises the
 * device).  *device_error = 0 if no cached workspace exists yet. */
int muon_ns_cached_error(int device, int* device_error);

/* Budget of every bounded wait inside the kernels (barrier phases, per-matrix
 * counters), in SM clock cycles (clock64); 0 restores the default of 4e9
 * cycles, about 2 s at 2 GHz.  A wait that runs out sets the error word
 * (read as MUON_NS_ERR_TIMEOUT) and its kernel returns; a budget shorter than
 * the waits of a healthy call gives spurious timeouts, never a hang.  Applies
 * to calls made afterwards, from any thread.  MUON_NS_ERR_INVALID_ARG if
 * cycles < 0. */
int muon_ns_set_wait_budget(long long cycles);

/* Host-side fault injection for tests of the bounded waits.  With `enable`
 * nonzero, later whole calls of stacks with two or more matrices give the
 * first step's polynomial kernel a completion target one unit above what the
 * Gram kernel signals: its waits run out, every later kernel of the call gives
 * up when it sees the error word, and the call reports MUON_NS_ERR_TIMEOUT
 * through it.  Nothing faults; the device stays usable.  Off by default;
 * returns MUON_NS_OK. */
int muon_ns_inject_stall(int enable);

/* ---------------------------------------------------------------------------
 * The steps of the path, one kernel each (the same kernels muon_ns_ws runs).
 * `device_error` is an optional device int32 that receives
 * MUON_NS_DEVERR_WAIT_TIMEOUT if a bounded wait runs out (may be NULL).
 * ------------------------------------------------------------------------- */

/* X = bf16(G * (1 / (||G_k||_F + eps))) per matrix, in the input orientation,
 * and norms[k] = ||G_k||_F (fp32, sum of squares accumulated in fp32 in a
 * fixed order, so the result is the same for a matrix alone or in any stack)
 * in the workspace's MUON_NS_WS_NORMS region.  `workspace` as for muon_ns_ws
 * (only its header and norm regions are used).  X == G is allowed; X == NULL
 * computes the norms only (one launch instead of two). */
int muon_ns_normalize(const muon_bf16* G, muon_bf16* X, int batch, int rows, int cols, float eps,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Gram matrix of the internal orientation, bf16 [batch][m][m], m = min(rows, cols):
 *   rows <= cols:  A = X X^T        rows > cols:  A = X^T X
 * Only lower-triangle tiles are computed; each value is written to (i, j) and
 * (j, i), so A is bit-symmetric.  fp32 accumulation, one rounding to bf16.
 *   norms  NULL, or device fp32 [batch]: then X is taken as unscaled and the
 *          Gram of X_k / (norms[k] + eps) is computed (the first NS step). */
int muon_ns_gram(const muon_bf16* X, muon_bf16* A, int batch, int rows, int cols,
                 const float* norms, float eps, int* device_error, cudaStream_t stream);

/* B = b A + c (A A) for a bit-symmetric A, bf16 [batch][m][m].  A A is formed
 * as A A^T (equal for a bit-symmetric A) over lower-triangle tiles; the
 * epilogue reads A and computes in fp32; B is bit-symmetric.  B != A.
 *   diag  NULL: B is stored whole in bf16.
 *         Non-NULL (device fp32 [batch][m], 16-byte aligned): B's diagonal is
 *         written here in fp32 and zeros are stored on B's bf16 diagonal, i.e.
 *         B = diag(D) + O with O bf16 and zero-diagonal.  muon_ns_ws does this:
 *         near convergence B is close to a multiple of the identity and its
 *         diagonal is the part bf16 would round worst. */
int muon_ns_poly(const muon_bf16* A, muon_bf16* B, float* diag, int batch, int m, float b,
                 float c, int* device_error, cudaStream_t stream);

/* The update of the iterate, in the input orientation, with m = min(rows, cols):
 *   rows <= cols:  Xn = a X + B X     (B is rows x rows)
 *   rows >  cols:  Xn = a X + X B     (B is cols x cols; this is (a X^T + B X^T)^T
 *                                      for the bit-symmetric B)
 * fp32 epilogue reading X.  Xn must not overlap X or B.
 *   diag  NULL, or the fp32 diagonal written by muon_ns_poly (then B's stored
 *         diagonal must be zero): the epilogue applies (a + diag_i) to X in
 *         fp32, row i for rows <= cols, column i for rows > cols.
 *   norms NULL, or device fp32 [batch]: then X is taken as unscaled and the
 *         update of X_k / (norms[k] + eps) is computed (the first NS step). */
int muon_ns_update(const muon_bf16* X, const muon_bf16* B, const float* diag, muon_bf16* Xn,
                   int batch, int rows, int cols, float a, const float* norms, float eps,
                   int* device_error, cudaStream_t stream);

/* Half storage of the symmetric matrices, as the whole-call entry points keep
 * them: A (or B) [batch][m][m] holds every diagonal 256 x 256 block whole
 * (rows and columns 256 k .. 256 k + 255) and, outside them, only the lower
 * triangle (i > j); the entries above the diagonal outside those blocks are
 * neither written nor read.  A per-step chain in this form moves fewer bytes
 * and runs the very kernels a whole call runs, with the same results bit for
 * bit.  Each _ex function takes `flags` = 0 (as the function without _ex) or
 * MUON_NS_HALF:
 *   muon_ns_gram_ex    writes A half;
 *   muon_ns_poly_ex    reads A half, writes B half;
 *   muon_ns_update_ex  reads B half.
 * Other flag bits return MUON_NS_ERR_INVALID_ARG.  The other arguments are as
 * for muon_ns_gram(), muon_ns_poly() and muon_ns_update(). */
#define MUON_NS_HALF 1
int muon_ns_gram_ex(const muon_bf16* X, muon_bf16* A, int batch, int rows, int cols, const float* norms,
                    float eps, int flags, int* device_error, cudaStream_t stream);
int muon_ns_poly_ex(const muon_bf16* A, muon_bf16* B, float* diag, int batch, int m, float b, float c,
                    int flags, int* device_error, cudaStream_t stream);
int muon_ns_update_ex(const muon_bf16* X, const muon_bf16* B, const float* diag, muon_bf16* Xn, int batch,
                      int rows, int cols, float a, const float* norms, float eps, int flags, int* device_error,
                      cudaStream_t stream);

/* X = bf16(G * (1 / (||G_k||_F + eps))) exactly as muon_ns_normalize(), for
 * callers that cannot allocate device memory (plugins handed only their
 * buffers, hosts whose allocator forbids cudaMalloc, loops that cannot take
 * cudaMalloc's synchronisation).  It allocates nothing and takes no
 * workspace: its scratch is a 1 MiB static device array of the library, held
 * by every GPU that loads it until the process exits.  The pages have no
 * counterpart; this is a deployment variant of the first NS step.
 *   - Size limit: 4 * batch * (ceil(rows * cols / 16384) + 2) bytes, each of
 *     the three parts rounded up to 256, must fit in 1 MiB; larger problems
 *     return MUON_NS_ERR_WORKSPACE and launch nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture on the device.
 *   - Every call shares the one array; it keeps the last call's contents and
 *     the call zeroes what must start at zero.  Calls that overlap on the GPU
 *     (different streams, no ordering) race on it and give wrong results.
 *   - X must not be NULL (MUON_NS_ERR_INVALID_ARG): the norms stay in the
 *     library's private array, where the caller cannot read them, so a
 *     norms-only call would have no result.
 *   - Other arguments, errors and aliasing (X == G allowed) as for
 *     muon_ns_normalize(). */
int muon_ns_normalize_static(const muon_bf16* G, muon_bf16* X, int batch, int rows, int cols,
                             float eps, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * The Muon optimizer step around NS.  prime-rl PR #3873 (Summary) speeds up
 * "the Muon optimizer step" whose inner loop is the NS above; param-decomp PR
 * #978 (What, `ns_dtype`) runs that NS in bf16 while "masters/momentum stay
 * fp32".  The pages print no formula for the step; the one taken here, per
 * matrix W (fp32 master), G (fp32 gradient), M (fp32 momentum buffer), is
 *
 *   M' = mu M + G
 *   U  = G + mu M'   (nesterov != 0)      or   U = M'   (nesterov == 0)
 *   O  = NS(bf16(U))                      (the bf16 NS of muon_ns_ws)
 *   W' = (1 - lr wd) W - lr scale O
 *
 * in fp32 (fused multiply-adds), with U rounded once to bf16 (nearest, ties
 * to even).  `scale` is the caller's shape factor on the update; the Python
 * binding defaults it to sqrt(max(1, rows / cols)).  W, M and G are device
 * fp32 [batch][rows][cols], contiguous, 16-byte aligned and pairwise
 * disjoint; the shape rules are those of muon_ns_ws.
 * ------------------------------------------------------------------------- */

typedef struct {
  float lr;            /* learning rate */
  float momentum;      /* mu */
  float weight_decay;  /* decoupled: W <- (1 - lr weight_decay) W - ... */
  float scale;         /* factor on the orthogonalised update */
  int nesterov;        /* nonzero: U = G + mu M'; zero: U = M' */
} muon_step_hparams;

/* Workspace bytes of muon_step_ws(): the muon_ns_ws() workspace of the stack
 * (same regions, muon_ns_workspace_region) followed by the bf16 U. */
int muon_step_workspace_size(int batch, int rows, int cols, size_t* bytes);

/* One Muon step of a stack, in place on W and M, G read only.  Kernel
 * launches: 1 + 3 * steps (3 if steps == 0).  The first kernel does the
 * momentum update, writes U and computes ||U||_F (the same fp32 value the NS
 * norm kernel would compute on U), so the NS needs no norm pass; the last
 * update product writes W' directly instead of storing O, so neither O nor
 * a separate update pass exists.  Results equal muon_momentum() ->
 * muon_ns_ws() on U -> muon_apply() bit for bit.  Hyperparameters must be
 * finite (MUON_NS_ERR_INVALID_ARG); the other arguments, errors and the
 * device error word (first int of the workspace) are as for muon_ns_ws().
 * Nothing is allocated and nothing synchronises. */
int muon_step_ws(float* W, float* M, const float* G, int batch, int rows, int cols,
                 const muon_step_hparams* hp, int steps, const float* coeffs, float eps, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/* The step's first kernel alone: M = mu M + G in place, U = bf16 NS input
 * (device bf16 [batch][rows][cols]), and ||U||_F into the MUON_NS_WS_NORMS
 * region of `workspace` (a muon_ns_ws() workspace of the stack).  M and G
 * must not overlap. */
int muon_momentum(float* M, const float* G, muon_bf16* U, int batch, int rows, int cols, float momentum,
                  int nesterov, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The step's update alone: W = (1 - lr wd) W - lr scale O for a device bf16 O
 * of W's shape (the NS output); hp->momentum and hp->nesterov are unused. */
int muon_apply(float* W, const muon_bf16* O, int batch, int rows, int cols, const muon_step_hparams* hp,
               cudaStream_t stream);

/* One stack of a grouped Muon step: `batch` matrices of rows x cols, device
 * fp32 W and M (updated in place) and G, contiguous, 16-byte aligned, with
 * this stack's hyperparameters. */
typedef struct {
  float* W;
  float* M;
  const float* G;
  int batch;
  int rows;
  int cols;
  muon_step_hparams hp;
} muon_step_stack;

/* Workspace bytes of muon_step_grouped(): the muon_step_ws() workspaces of
 * the non-empty stacks, end to end, in order.  Checks the stacks as the call
 * does (no device needed). */
int muon_step_grouped_workspace_size(const muon_step_stack* stacks, int num_stacks, size_t* bytes);

/* One Muon step over several stacks (an optimizer step's parameter groups of
 * different shapes and hyperparameters; host array of num_stacks <= 64
 * descriptors), with one NS setting (steps, coeffs, eps).  Each stack gets its
 * momentum kernel; the NS products of all stacks then share launches as in
 * muon_ns_grouped(), the last update of each writing its own W.  Results equal
 * muon_step_ws() on each stack alone, bit for bit.  No W or M may overlap any
 * stack's W, M or G (MUON_NS_ERR_INVALID_ARG); empty stacks are skipped.  The
 * device error word is the first non-empty stack's, at the start of the
 * workspace.  Errors otherwise as muon_step_ws(). */
int muon_step_grouped(const muon_step_stack* stacks, int num_stacks, int steps, const float* coeffs, float eps,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Kernel launches of one muon_step_ws() call: 1 + 3 * steps (3 if steps == 0). */
int muon_step_launches(int steps);

/* ---------------------------------------------------------------------------
 * Host-only helpers (no GPU needed).
 * ------------------------------------------------------------------------- */

/* Kernel launches made by one muon_ns_ws() call: 1 + 3 * steps (2 if steps == 0). */
int muon_ns_launches_per_call(int steps);

/* Persistent tile scheduler of the tensor-core kernels.  kind 0 = lower
 * triangle of an m x m output (M == N), kind 1 = full M x N output.  Tiles are
 * 128 x 256.  kinds 2 and 3 are the same spaces walked by clusters of two
 * CTAs: a unit is a pair of row tiles (2p, 2p + 1) of one column tile, and
 * row_tile returns p.  muon_ns_tile_count() returns the number of units of a
 * launch (-1 on bad arguments); muon_ns_tile_coords() maps a linear unit
 * index to (matrix, row tile or pair row, column tile) exactly as the kernels
 * do. */
long long muon_ns_tile_count(int kind, int batch, int M, int N);
int muon_ns_tile_coords(int kind, int batch, int M, int N, long long tile, int* matrix,
                        int* row_tile, int* col_tile);

#ifdef __cplusplus
}
#endif

#endif /* MUON_NS_H */
