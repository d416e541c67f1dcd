/*
 * dion3.h -- C ABI of the GB300 (sm_103a) Dion3 / Gram Newton-Schulz library (libdion3.so).
 *
 * The library implements the data-parallel hot path of the Dion3 optimizer:
 *   - a symmetric GEMM (lower triangle computed, upper triangle written as its exact mirror),
 *   - batched Gram Newton-Schulz orthogonalization with restarts,
 *   - one Dion3 step (momentum update, exact top-k row selection, orthogonalization of the
 *     selected rows, W row update, error-feedback decay of the selected rows).
 *
 * Citations name a page and a section of it:
 *   [D3]  "Dion3: Full-Stack Orthogonal Updates", structured summary (paper.rainbus.top):
 *         prerequisites, "core method" (Theorem 2), "method details" (Algorithms 3 and 4),
 *         table "structured data" (FLOP formulas), "limitations".
 *   [D3m] "Dion3: Full-Stack Orthogonal Updates", summary (m.montaan.com).
 *   [MB]  "Muon: Orthogonalized Momentum and Why It Trains LLMs 2x Cheaper",
 *         section "Doing an SVD without an SVD".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Matrices are row-major.  A batch of matrices is [batch][rows][cols] with a leading
 *   dimension `ld` (elements between consecutive rows, >= cols) and a batch stride
 *   `stride` (elements between consecutive matrices, >= rows*ld when batch > 1).
 * - All matrix pointers are DEVICE pointers owned by the caller.  `abc`, `restart_after`
 *   are HOST arrays.  `stream` is a cudaStream_t (NULL = legacy default stream).
 * - The library allocates no memory, keeps no state between calls and never synchronizes
 *   the stream.  Scratch memory is the caller's `workspace` (query its size first).
 * - Host-detectable errors are returned synchronously and nothing is enqueued.  A launch
 *   failure returns DION3_ECUDA.
 * - Conditions found on the device are OR-ed into `*status_dev` (a device int, may be
 *   NULL) as DION3_DEV_* bits; the caller reads it whenever it wants.  No kernel traps.
 * - Every wait inside a kernel is bounded; a wait that gives up sets DION3_DEV_TIMEOUT
 *   and the kernel returns (its outputs are then undefined).
 */
#ifndef DION3_H
#define DION3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DION3_ABI_VERSION 1

/* Return codes. */
typedef enum {
  DION3_OK = 0,
  DION3_EINVAL = 1,        /* a null pointer, negative or inconsistent size, bad schedule */
  DION3_EUNSUPPORTED = 2,  /* valid but outside what the library supports (dtype mix, limits) */
  DION3_EWORKSPACE = 3,    /* workspace missing or smaller than the query says */
  DION3_ECUDA = 4,         /* a CUDA call (launch, tensor-map encode, attribute) failed */
  DION3_EALIGN = 5         /* a pointer, leading dimension or stride breaks the 16-byte rule */
} dion3_status;

/* Element types. */
typedef enum { DION3_BF16 = 0, DION3_FP16 = 1, DION3_FP32 = 2 } dion3_dtype;

/* norm_p value of the step entry points for a caller-chosen row set S (see dion3_step). */
#define DION3_SELECT_GIVEN 0

/* Bits OR-ed into *status_dev by kernels. */
#define DION3_DEV_NONFINITE 0x1 /* a non-finite momentum key, norm or input value was seen, or
                                   the last product of the orthogonalisation wrote a non-finite
                                   value (into Out, or into W by the row update): the iteration
                                   diverged ("half precision and numerical stability") */
#define DION3_DEV_TIMEOUT   0x2 /* a bounded wait gave up; outputs of that call are undefined */
#define DION3_DEV_SELECT    0x4 /* row selection could not certify k rows (internal error), or a
                                   caller-chosen S was not k distinct ascending rows in [0, n) */
#define DION3_DEV_RANGE     0x8 /* checked builds only (libdion3_checked.so, see dion3_range_checks):
                                   a kernel found an index outside its buffer -- a selected or
                                   carried row outside [-1, n), or a tile outside its matrix -- and
                                   skipped the access.  -1 is the blank a failed selection leaves
                                   and is not flagged. */

/*
 * dion3_sym_gemm -- D = alpha * A * B^T + beta * C + gamma * I, for results known to be
 * symmetric.  [D3] prerequisite "symmetric GEMM kernels" (compute the lower triangle and the
 * diagonal, write the transpose into the upper triangle) and [D3] "technical novelty" (the
 * fused symmetric alpha*A*B + beta*C the Gram form needs).  [D3m] reports the ~2x over cuBLAS.
 *
 *   A : [batch][n][k], element type in_dtype, leading dim lda, batch stride strideA.
 *   B : same shape and type as A, or NULL for B = A (the Gram product A*A^T).  When B != A
 *       the caller asserts that A*B^T is symmetric (for Gram Newton-Schulz: products of
 *       polynomials in the same R, which commute).  Only tiles with row-block >= column-block
 *       are computed.
 *   C : [batch][n][n] of out_dtype, read only where beta != 0 and only in its lower triangle
 *       (diagonal included).  May alias D (same ld and stride).
 *   D : [batch][n][n] of out_dtype.  Every element is written; D[j][i] is the bit-exact copy
 *       of D[i][j] for i > j.
 *   in_dtype  : DION3_BF16 / DION3_FP16 (5th-gen tensor cores, fp32 accumulation) or
 *               DION3_FP32 (fp32 FFMA, no TF32).
 *   out_dtype : in_dtype or DION3_FP32 for 16-bit inputs; DION3_FP32 for fp32 inputs.
 *   Alignment: all pointers 16-byte aligned; ld*elemsize and stride*elemsize multiples of 16.
 *   k == 0 is allowed (D = beta*C + gamma*I; A and B are then not read and may be NULL).
 *   n == 0 or batch == 0 is a no-op.
 *   Errors: EINVAL (nulls, sizes, ld < cols), EALIGN, EUNSUPPORTED (dtype mix), ECUDA.
 */
int dion3_sym_gemm(int batch, int n, int k,
                   const void* A, int64_t lda, int64_t strideA,
                   const void* B, int64_t ldb, int64_t strideB,
                   const void* C, int64_t ldc, int64_t strideC,
                   void* D, int64_t ldd, int64_t strideD,
                   float alpha, float beta, float gamma,
                   int in_dtype, int out_dtype,
                   int* status_dev, void* stream);

/*
 * dion3_gram_ns_workspace_bytes -- bytes of device workspace dion3_gram_ns needs for these
 * sizes, dtypes and number of restarts (n_restart).  Returns 0 for invalid sizes.
 */
size_t dion3_gram_ns_workspace_bytes(int batch, int n, int m, int x_dtype, int compute_dtype,
                                     int n_restart);

/*
 * dion3_gram_ns -- Out = GramNS(X) for a batch of n x m matrices, 1 <= n <= m.
 * [D3] "core method" Theorem 2 and "method details" Algorithm 3; [MB] for the prescale:
 *   Xs = X / (||X||_F + eps)  (norm in fp32 on the stored values);
 *   R = Xs Xs^T;  Q = I;
 *   for t = 1..T:  Z = a_t I + b_t R + c_t R^2;   Q = Q Z;
 *                  if t is in restart_after:  Xs = Q Xs;  R = Xs Xs^T;  Q = I;
 *                  else if t < T:             R = Z R Z;
 *   Out = Q Xs.
 * Products with Q = I are skipped (Q = Z), as is the R update a restart or the end makes
 * dead.  16-bit compute keeps R, Z, Q and the restarted Xs in that type with fp32
 * accumulation; fp32 compute uses fp32 FFMA throughout.  [D3] Algorithm 3 runs the
 * iteration in float16 (DION3_FP16): the half-precision rounding of R is what the restarts
 * repair.  DION3_BF16 iterates work the same way with an 8-bit mantissa, which costs about an
 * order of magnitude in accuracy.
 *
 *   X   : [batch][n][m] of x_dtype (ldx, strideX), not modified.  X is read in place when
 *         x_dtype == compute_dtype and its pointer, ldx and strideX are 16-byte multiples;
 *         otherwise it is copied into the workspace.  The workspace query reserves room for
 *         that copy unless x_dtype == compute_dtype and m * elemsize is a multiple of 16; a
 *         call that needs the copy without having queried for it returns DION3_EWORKSPACE.
 *   Out : [batch][n][m] of out_dtype (ldo, strideO); 16-byte aligned rows.  Must not
 *         overlap X or the workspace.
 *   T, abc : T >= 1 iterations, abc = host float[3*T] = (a_1,b_1,c_1, a_2,b_2,c_2, ...).
 *   restart_after : host int[n_restart], strictly increasing, each in [1, T-1]; may be NULL
 *         when n_restart == 0.
 *   eps : added to the Frobenius norm (the pages use 1e-7).
 *   compute_dtype : DION3_BF16, DION3_FP16 or DION3_FP32.
 *   workspace : device buffer of at least dion3_gram_ns_workspace_bytes(...) bytes,
 *         256-byte aligned.
 *   Errors: EINVAL (n > m, T < 1, schedule), EWORKSPACE, EALIGN (Out, workspace),
 *           EUNSUPPORTED (fp32 compute with a 16-bit output), ECUDA.
 *   Device: DION3_DEV_NONFINITE if a norm or an element of Out is not finite.
 */
int dion3_gram_ns(int batch, int n, int m,
                  const void* X, int64_t ldx, int64_t strideX, int x_dtype,
                  void* Out, int64_t ldo, int64_t strideO, int out_dtype,
                  int T, const float* abc, const int* restart_after, int n_restart,
                  float eps, int compute_dtype,
                  void* workspace, size_t workspace_bytes,
                  int* status_dev, void* stream);

/*
 * dion3_ns_standard_workspace_bytes -- bytes of device workspace dion3_ns_standard needs.
 * Returns 0 for invalid sizes.
 */
size_t dion3_ns_standard_workspace_bytes(int batch, int n, int m, int compute_dtype);

/*
 * dion3_ns_standard -- Out = NS(X), the standard quintic Newton-Schulz iteration, for a batch
 * of n x m matrices, 1 <= n <= m.  [D3] prerequisite "Newton-Schulz iteration" and [MB]
 * "Doing an SVD without an SVD" define the iteration; [D3] "limitations" names it as the
 * fallback for square matrices (alpha = 1), where Gram Newton-Schulz saves nothing and its
 * restarts cost 3(alpha-1)n^3 = 0 anyway:
 *   Xs = X / (||X||_F + eps);
 *   for t = 1..T:  A = Xs Xs^T;  B = b_t A + c_t A^2;  Xs = a_t Xs + B Xs;
 *   Out = Xs.
 * A and B are symmetric products (lower triangle computed, mirrored); Xs = B Xs + a_t Xs is
 * one general product with the a_t Xs term added in its epilogue, so an iteration costs
 * (3 alpha + 1) n^3 useful FLOPs.  The iterates Xs, A, B are stored in compute_dtype (fp32
 * accumulation).
 *   X, Out, T, abc, eps, compute_dtype, workspace, status_dev, stream: as dion3_gram_ns (X is
 *   always copied, prescaled, into the workspace).
 *   Errors: EINVAL (n > m, T < 1), EWORKSPACE, EALIGN (Out, workspace), EUNSUPPORTED (fp32
 *           compute with a 16-bit output), ECUDA.
 *   Device: DION3_DEV_NONFINITE if a norm or an element of Out is not finite.
 */
int dion3_ns_standard(int batch, int n, int m,
                      const void* X, int64_t ldx, int64_t strideX, int x_dtype,
                      void* Out, int64_t ldo, int64_t strideO, int out_dtype,
                      int T, const float* abc, float eps, int compute_dtype,
                      void* workspace, size_t workspace_bytes,
                      int* status_dev, void* stream);

/*
 * dion3_k -- k = ceil(n * f_num / f_den) in exact integers ([D3] "existing work": k = ceil(f n)).
 * Returns -1 unless n >= 0 and 0 < f_num <= f_den.
 */
int dion3_k(int n, int f_num, int f_den);

/*
 * dion3_step_workspace_bytes -- bytes of workspace dion3_step needs.  0 for invalid sizes.
 */
size_t dion3_step_workspace_bytes(int batch, int n, int m, int f_num, int f_den, int norm_p,
                                  int compute_dtype, int n_restart);

/*
 * dion3_step -- one Dion3 step on a megabatch of same-shape matrices, n <= m.
 * [D3] "method details" Algorithm 4, prerequisite "error feedback", prerequisite
 * "spectral-norm steepest descent" (eta' = eta / sqrt(f)):
 *   M <- M + G                                  (fp32 state, one rounding)
 *   key_i = sum_j |M_ij|   (norm_p = 1, the pages' l1 rule)
 *         = sum_j M_ij^2   (norm_p = 2, same order as the row L2 norm)
 *   S = the k = ceil(f n) rows with the largest exact keys, ties to the lower row index,
 *       written ascending to sel_out.  Keys are compared as exact real numbers: fp32 keys
 *       with a proven error bound decide every row they can, and the rows they cannot are
 *       re-ranked with exact integer sums on the device.
 *   norm_p = DION3_SELECT_GIVEN: S is chosen by the caller and read from sel_out (k strictly
 *       ascending rows in [0, n) per matrix; e.g. a random subset, which [D3] "limitations"
 *       reports to work about as well, and which [D3] "future directions" notes can be drawn
 *       without knowing M).  No keys are computed.  A matrix whose S breaks the rule gets
 *       DION3_DEV_SELECT, its sel_out entries are set to -1 and none of its rows change
 *       except by M <- M + G (and the decay of W).
 *   O = GramNS(M[S,:])                          (as dion3_gram_ns, compute_dtype)
 *   W <- (1 - eta' wd) W  (all rows; skipped when wd == 0)
 *   W[S,:] <- W[S,:] - eta' O,  eta' = eta * sqrt(f_den / f_num)
 *   M[S,:] <- mu * M[S,:]                       (fp32, one rounding; mu taken as given)
 *
 *   W, M : fp32 [batch][n][m], contiguous (ld = m, stride = n*m), updated in place.
 *   G    : [batch][n][m] contiguous, g_dtype DION3_BF16, DION3_FP16 or DION3_FP32.
 *   sel_out : int32 [batch][k] device output, ascending row indices.
 *   Limits: n <= 16384 and m <= 65536 (exact selection); 0 < f_num <= f_den.
 *   W, M, G, sel_out 16-byte aligned.  Errors as dion3_gram_ns.
 *   Device: DION3_DEV_NONFINITE (a non-finite momentum or norm, or a non-finite updated W
 *           row element), DION3_DEV_SELECT.
 */
int dion3_step(int batch, int n, int m,
               float* W, float* M, const void* G, int g_dtype,
               int f_num, int f_den, float mu, float eta, float wd, int norm_p,
               int T, const float* abc, const int* restart_after, int n_restart, float eps,
               int compute_dtype, int32_t* sel_out,
               void* workspace, size_t workspace_bytes,
               int* status_dev, void* stream);

/*
 * dion3_step_timed -- dion3_step, and in addition records the caller's events (cudaEvent_t
 * handles, created by the caller) on `stream` at the step's phase boundaries:
 *   events[0] before the momentum pass, [1] after it, [2] after the row selection,
 *   [3] after the gather of M[S,:], [4] after the Gram Newton-Schulz products (the end).
 * Only the first n_events entries are used; NULL entries are skipped.  Use it to split a
 * step's device time by phase.  (No counterpart on the pages: a measurement hook.)
 */
int dion3_step_timed(int batch, int n, int m,
                     float* W, float* M, const void* G, int g_dtype,
                     int f_num, int f_den, float mu, float eta, float wd, int norm_p,
                     int T, const float* abc, const int* restart_after, int n_restart, float eps,
                     int compute_dtype, int32_t* sel_out,
                     void* workspace, size_t workspace_bytes,
                     int* status_dev, void* stream, void* const* events, int n_events);

/*
 * dion3_step_cols_workspace_bytes -- bytes of workspace dion3_step_cols needs.  0 for invalid sizes.
 */
size_t dion3_step_cols_workspace_bytes(int batch, int m, int n, int f_num, int f_den, int norm_p,
                                       int compute_dtype, int n_restart);

/*
 * dion3_step_cols -- one Dion3 step on matrices stored un-oriented, [batch][m][n] with the short
 * side n as columns (n <= m), selecting columns: [D3m] update-rule paragraph (f is the fraction
 * of rows or columns selected) with everything else as dion3_step.  In exact arithmetic it is
 * dion3_step on the transposed matrices, transposed back:
 *   M <- M + G;  key_j = sum_i |M_ij| (norm_p = 1) or sum_i M_ij^2 (norm_p = 2);
 *   S = the k = ceil(f n) columns with the largest exact keys (ties to the lower index);
 *   O = GramNS(M[:, S]^T) (k x m);  W <- (1 - eta' wd) W;  W[:, S] <- W[:, S] - eta' O^T;
 *   M[:, S] <- mu M[:, S].
 *   W, M : fp32 [batch][m][n] contiguous (ld = n, stride = m*n), updated in place.
 *   G    : [batch][m][n] contiguous, g_dtype as dion3_step.
 *   sel_out : int32 [batch][k], ascending column indices (read when norm_p = DION3_SELECT_GIVEN).
 *   The columns are gathered and scattered through shared-memory transposes; O passes through
 *   the workspace in the compute dtype (one rounding that dion3_step's fused update avoids).
 *   Limits: n <= 16384, m <= 65536, batch <= 65535.  Errors and device flags as dion3_step.
 */
int dion3_step_cols(int batch, int m, int n,
                    float* W, float* M, const void* G, int g_dtype,
                    int f_num, int f_den, float mu, float eta, float wd, int norm_p,
                    int T, const float* abc, const int* restart_after, int n_restart, float eps,
                    int compute_dtype, int32_t* sel_out,
                    void* workspace, size_t workspace_bytes,
                    int* status_dev, void* stream);

/*
 * dion3_step_dev -- dion3_step with the hyperparameters read on the device, for CUDA-graph
 * capture: a graph captured around one call replays every later step with whatever values
 * hyper_dev holds when it runs (a learning-rate schedule without re-capture).  [D3] "method
 * details" Algorithm 4 (mu, eta, weight decay) and the step-time figures it reports for
 * graph-captured optimizer steps.
 *   hyper_dev : device float[3] = {mu, eta, wd}, 4-byte aligned, read by the kernels when they
 *               run.  eta' = double(eta) * sqrt(f_den / f_num) and 1 - eta' wd are formed in
 *               double and rounded once to fp32, exactly as dion3_step forms them on the host,
 *               so both entry points give bit-identical results for the same values.
 *   decay     : nonzero runs the W <- (1 - eta' wd) W pass (read-modify-write of all of W);
 *               zero skips it whatever wd holds.  It is fixed at capture time.
 *   Everything else as dion3_step.  The values are not checked for finiteness on the host.
 *   Errors: as dion3_step; EINVAL if hyper_dev is NULL, EALIGN if it is not 4-byte aligned.
 */
int dion3_step_dev(int batch, int n, int m,
                   float* W, float* M, const void* G, int g_dtype,
                   int f_num, int f_den, const float* hyper_dev, int decay, int norm_p,
                   int T, const float* abc, const int* restart_after, int n_restart, float eps,
                   int compute_dtype, int32_t* sel_out,
                   void* workspace, size_t workspace_bytes,
                   int* status_dev, void* stream);

/*
 * dion3_step_carry -- dion3_step_timed whose error-feedback decay of M[S,:] moves into the next
 * call's momentum pass.  [D3] "method details" Algorithm 4 and prerequisite "error feedback":
 * the decay M[S,:] <- mu M[S,:] ends one step and the next step's first operation is
 * M <- M + G, so it can be applied as M_i <- (mu M_i) + G_i by the pass that reads and writes
 * every row of M anyway, saving the gather pass its write of M[S,:] (4 of its 10 bytes per
 * selected element).  Each product is rounded to fp32 before the sum, so the results are
 * bit-identical to dion3_step's.  (Not a step of the pages: a reordering of theirs.)
 *   carry_rows : NULL, or int32 [batch][k] device rows (same k as this call) whose decay by
 *                carry_mu an earlier call left pending -- that call's sel_out.  They are
 *                applied before M <- M + G.  Entries outside [0, n) (the -1 of a failed
 *                selection) are skipped; a row listed more than once is scaled once.  4-byte
 *                aligned.  It may be the same buffer as sel_out (it is read before the new S
 *                is written), except with norm_p = DION3_SELECT_GIVEN, where sel_out holds
 *                the new S on entry: that aliasing is EINVAL.
 *   carry_mu   : the factor of the pending decay (that call's mu); must be finite.
 *   defer      : nonzero leaves this call's own decay of M[S,:] by mu pending: on return
 *                M[S,:] holds M + G, and the caller passes (sel_out, mu) as the next call's
 *                (carry_rows, carry_mu) or applies it with dion3_decay_rows.  Zero applies it
 *                as dion3_step does.
 *   Workspace: dion3_step_workspace_bytes.  Everything else as dion3_step_timed (events may
 *   be NULL with n_events = 0).  One extra launch (the per-row flags) when carry_rows is set.
 *   Errors: as dion3_step; EINVAL for a non-finite carry_mu or the aliasing above, EALIGN
 *   for a misaligned carry_rows.
 */
int dion3_step_carry(int batch, int n, int m,
                     float* W, float* M, const void* G, int g_dtype,
                     int f_num, int f_den, float mu, float eta, float wd, int norm_p,
                     int T, const float* abc, const int* restart_after, int n_restart, float eps,
                     int compute_dtype, int32_t* sel_out,
                     const int32_t* carry_rows, float carry_mu, int defer,
                     void* workspace, size_t workspace_bytes,
                     int* status_dev, void* stream, void* const* events, int n_events);

/*
 * dion3_step_dev_carry -- dion3_step_dev with the carried decay of dion3_step_carry, for a
 * graph captured once and replayed every step: the carried factor lives on the device.
 *   carry_rows   : as dion3_step_carry (typically sel_out itself).
 *   carry_mu_dev : device float, 4-byte aligned; required when carry_rows is set or defer is
 *                  nonzero.  The momentum pass reads the pending factor from it (when carry_rows
 *                  is set); with defer, the gather pass then stores this call's mu
 *                  (hyper_dev[0]) there, so the next replay applies it.  Before the first
 *                  replay set it to 1.0f (and sel_out to -1 or any rows in range): a factor of
 *                  1 leaves every row exactly as it is.  The value is not checked for
 *                  finiteness.
 *   defer        : as dion3_step_carry.  Everything else as dion3_step_dev.
 *   Errors: as dion3_step_dev; EINVAL when carry_mu_dev is needed and NULL, EALIGN when it is
 *   misaligned; the carry_rows rules of dion3_step_carry.
 */
int dion3_step_dev_carry(int batch, int n, int m,
                         float* W, float* M, const void* G, int g_dtype,
                         int f_num, int f_den, const float* hyper_dev, int decay, int norm_p,
                         int T, const float* abc, const int* restart_after, int n_restart, float eps,
                         int compute_dtype, int32_t* sel_out,
                         const int32_t* carry_rows, float* carry_mu_dev, int defer,
                         void* workspace, size_t workspace_bytes,
                         int* status_dev, void* stream);

/*
 * dion3_decay_rows -- applies a decay that dion3_step_carry left pending:
 *   M[b][rows[b][j]][:] <- mu * M[b][rows[b][j]][:]  (fp32, one rounding)
 * for j < k and rows in [0, n); other entries are skipped.  List each row once (as sel_out
 * does): a repeated row is scaled once per listing.
 *   M    : fp32 [batch][n][m] contiguous, 4-byte aligned.  rows : int32 [batch][k], 4-byte aligned.
 *   Errors: EINVAL (negative sizes, k > n, non-finite mu, NULL pointers with work to do),
 *   EALIGN, ECUDA.  Nothing to do (batch, k or m zero) returns DION3_OK.
 */
int dion3_decay_rows(int batch, int n, int m, float* M, const int32_t* rows, int k, float mu, void* stream);

/*
 * dion3_gram_ns_noalloc -- dion3_gram_ns for callers that cannot allocate device memory
 * (no counterpart in the paper).  Same arguments and results as dion3_gram_ns, minus the
 * workspace: the scratch comes from an array of DION3_NOALLOC_SCRATCH_BYTES compiled into the
 * library, resident on every GPU that loads the library until the process exits.
 *   - Arguments are checked exactly as dion3_gram_ns checks them, in the same order, so a bad
 *     call returns the same code from either entry point.
 *   - Sizes whose workspace (dion3_gram_ns_workspace_bytes, plus the copy of a misaligned X)
 *     exceeds DION3_NOALLOC_SCRATCH_BYTES are then rejected with DION3_EWORKSPACE, nothing
 *     enqueued.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and keeps it; make that first call before any stream capture.  The address
 *     belongs to the device's primary context: after cudaDeviceReset on that device it is
 *     stale, so do not call this entry point there again in the same process.
 *   - It allocates nothing and frees nothing.
 *   - Every call uses the same array and leaves its contents behind; nothing in it needs to
 *     start at zero.  Calls whose work overlaps on the GPU (other streams, other host
 *     threads) race on the array: serialise them.
 */
#define DION3_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int dion3_gram_ns_noalloc(int batch, int n, int m,
                          const void* X, int64_t ldx, int64_t strideX, int x_dtype,
                          void* Out, int64_t ldo, int64_t strideO, int out_dtype,
                          int T, const float* abc, const int* restart_after, int n_restart,
                          float eps, int compute_dtype,
                          int* status_dev, void* stream);

/* Human-readable name of a return code. */
const char* dion3_status_str(int code);

/* DION3_ABI_VERSION of the loaded library. */
int dion3_abi_version(void);

/*
 * dion3_range_checks -- 1 if this library was built with in-kernel range checks
 * (libdion3_checked.so: every entry point above, same arguments and results, plus
 * DION3_DEV_RANGE in *status_dev when an index leaves its buffer), 0 for the default build.
 * The checked build stands in for a memory checker, which the GPUs this library is tested on
 * do not offer; it never traps.  No counterpart on the pages.
 */
int dion3_range_checks(void);

/*
 * dion3_selftest_watchdog -- diagnostic for the bounded-wait machinery (no counterpart on the
 * pages).  Launches one small kernel that waits on a barrier nothing will ever complete,
 * giving up after `spin_limit_cycles` clock cycles; it then sets DION3_DEV_TIMEOUT in
 * *status_dev and returns normally.  status_dev must be non-NULL.
 */
int dion3_selftest_watchdog(long long spin_limit_cycles, int* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DION3_H */
