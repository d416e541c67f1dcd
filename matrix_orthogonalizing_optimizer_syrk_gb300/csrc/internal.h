// Internal host interface shared by the translation units of libdion3.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "dion3.h"

namespace dion3 {

enum DType { BF16 = DION3_BF16, FP16 = DION3_FP16, FP32 = DION3_FP32 };

inline int dtype_size(int t) { return t == FP32 ? 4 : 2; }
inline bool dtype_valid(int t) { return t == BF16 || t == FP16 || t == FP32; }
inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// One batched matrix operand: [batch][rows][cols] with leading dim and batch stride (elements).
struct Mat {
  const void* ptr = nullptr;
  int64_t ld = 0;
  int64_t stride = 0;
  int dtype = BF16;
};

enum Epi { EPI_SYM = 0, EPI_GEN = 1, EPI_WUPD = 2 };

// One batched GEMM as the drivers see it.
//   SYM : D[b] (M x M) = alpha_b * A[b] B[b]^T + beta * C[b] + gamma * I, lower tiles only,
//         upper triangle mirrored.  A, B are K-major ([b][M][K]).
//   GEN : D[b] (M x N) = alpha_b * A[b] B[b] + beta * C[b]; A is [b][M][K], B is [b][K][N]
//         (N contiguous); C (read when beta != 0) has D's dtype.
//   WUPD: like GEN, but instead of storing D the epilogue adds alpha_b * acc into
//         W[b][sel[b][r]][c] (fp32 read-modify-write).
// alpha_b = alpha * (alpha_batch ? alpha_batch[b] : 1).
struct GemmCall {
  int batch = 0, M = 0, N = 0, K = 0;
  int epi = EPI_SYM;
  Mat A, B;
  Mat C;
  float beta = 0.f;
  Mat D;
  float alpha = 1.f;
  const float* alpha_batch = nullptr;
  float gamma = 0.f;
  float* W = nullptr;
  int64_t ldw = 0, sW = 0;
  const int* sel = nullptr;
  int64_t ssel = 0;
  int w_rows = 0;  // rows of each W matrix (bounds for sel entries)
  int* status = nullptr;
  long long spin_limit = 0;  // clock cycles for bounded waits; 0 = default
  // When set, alpha is replaced on the device by float(-(double(*eta_dev) * eta_scale)): the W
  // row update's -eta' read from device memory at run time.
  const float* eta_dev = nullptr;
  double eta_scale = 0.0;
  // Last product of an orthogonalisation: a non-finite stored element (or updated W element)
  // sets DION3_DEV_NONFINITE in *status.
  bool check_finite = false;
};

// 16-bit inputs on the tcgen05 tensor cores (gemm_tc.cu).
int gemm_tc(const GemmCall& g, cudaStream_t s);
// fp32 inputs on FFMA (gemm_simt.cu).
int gemm_simt(const GemmCall& g, cudaStream_t s);
inline int gemm(const GemmCall& g, cudaStream_t s) {
  return g.A.dtype == FP32 ? gemm_simt(g, s) : gemm_tc(g, s);
}

// Number of SMs of the current device (cached per device).
int sm_count();

// 3-D TMA map over a 16-bit [batch][rows][cols] matrix (ld and stride from m), box
// box_cols x box_rows, 128-byte swizzle (gemm_tc.cu).
bool tensor_map_16(CUtensorMap* map, const Mat& m, int rows, int cols, int batch, int box_cols, int box_rows);

// One restart segment of Gram Newton-Schulz on n x n Gram matrices, n <= 128, 16-bit (gram_small.cu):
// from R (batch x n x n) run `iters` iterations with the (a, b, c) triples abc[0 .. 3 iters) and
// write Q.  The R update after the segment's last iteration is skipped.
#define DION3_SEG_MAX_ITERS 32
int gram_segment(int batch, int n, const Mat& R, const Mat& Q, int iters, const float* abc, int* status,
                 cudaStream_t s);

// ---- elementwise / reduction launchers (elementwise.cu) ----
// Per-row sum of squares of X (any dtype, any ld) into rowsq[b*n + i] (fp32).
int rows_sumsq(int batch, int n, int m, Mat X, float* rowsq, int* status, cudaStream_t s);
// scale[b] = 1 / (sqrt(sum_i rowsq[b*rows + i]) + eps); alpha2[b] = scale[b]^2 (alpha2 may be null).
int finalize_scale(int batch, int rows, const float* rowsq, float eps, float* scale, float* alpha2,
                   int* status, cudaStream_t s);
// Xc[b] = scale[b] * X[b] in dtype cdt (ld ldc, stride sc); scale == nullptr converts only.
int scaled_cast(int batch, int n, int m, Mat X, const float* scale, void* Xc, int64_t ldc, int64_t sc, int cdt,
                cudaStream_t s);

// ---- Dion3 step launchers (step.cu) ----
struct StepArgs {
  int batch, n, m, k;
  float* W;
  float* M;
  const void* G;
  int g_dtype;
  int norm_p;
  float mu;
  float w_decay;  // 1 - eta' * wd
  bool decay;     // run the W <- w_decay W pass
  // When set, mu, eta, wd are read from hyper[0..2] on the device (mu and w_decay then come
  // from there; eta' = double(eta) * eta_scale).
  const float* hyper;
  double eta_scale;
  int32_t* sel;
  float* key_lo;
  float* key_hi;
  uint64_t* exact;  // [batch][n][limbs]
  void* XS;         // [batch][k][ldx] compute dtype, = scale_b * M[S,:]
  int64_t ldx;
  int cdt;
  float* rowsq;  // [batch][n]: per-row sum of squares of M after + G
  float* scale;  // [batch]: 1 / (||M[S,:]||_F + eps)
  float eps;
  int* status;
  // Column selection: W, M, G stored [batch][m][n] and the n keys belong to columns (each a
  // vector of m entries).  Pass A then writes per-chunk column partial sums (part_s, part_q:
  // [batch][nchunk][n]) that a finalize kernel turns into keys and column sums of squares.
  bool cols = false;
  float* part_s = nullptr;
  float* part_q = nullptr;
  int nchunk = 0;
  // Carried decay.  carry_rows ([batch][k], or null): rows whose decay by carry_mu an earlier
  // step left pending; pass A first turns them into per-row flags (carry_flag, [batch][n]) and
  // scales those rows by carry_mu before adding G.  defer: pass C leaves this step's decay of
  // M[S,:] pending instead of storing mu M[S,:].
  const int32_t* carry_rows = nullptr;
  uint8_t* carry_flag = nullptr;
  float carry_mu = 1.f;
  bool defer = false;
  // Device form (graph capture): the pending factor is read from carry_mu_dev, and with defer
  // pass C stores this step's mu there once it has been read.
  float* carry_mu_dev = nullptr;
};
int step_momentum_keys(const StepArgs& a, cudaStream_t s);
int step_select(const StepArgs& a, cudaStream_t s);
int step_gather(const StepArgs& a, cudaStream_t s);
// Column selection only (step_cols.cu): pass A with column keys (and its finalize), and pass C.
int step_colkeys(const StepArgs& a, cudaStream_t s);
int step_gather_cols(const StepArgs& a, cudaStream_t s);
// Column selection only: W[b][i][S_j] += alpha * O[b][j][i] for the k x m matrices O (compute
// dtype, leading dimension ldo); alpha is float(-double(*eta_dev) * eta_scale) when eta_dev is set.
int step_scatter_cols(const StepArgs& a, const void* O, int64_t ldo, float alpha, const float* eta_dev,
                      double eta_scale, cudaStream_t s);
constexpr int STEP_COL_CHUNK = 256;  // rows per partial sum of a column key
int step_exact_limbs(int norm_p);
// M[b][rows[b][j]][:] <- mu M[b][rows[b][j]][:] for the listed rows in [0, n).
int step_decay_rows(int batch, int n, int m, int k, float* M, const int32_t* rows, float mu, cudaStream_t s);

// Argument checks of dion3_gram_ns, in its order (api.cu).  Returns the code dion3_gram_ns would
// return before looking at its workspace; on DION3_OK, *need is the workspace size the call needs
// (0: nothing to do, e.g. an empty batch).
int gram_ns_validate(int batch, int n, int m, const void* X, int64_t ldx, int64_t strideX, int x_dtype,
                     const void* Out, int64_t ldo, int64_t strideO, int out_dtype, int T, const float* abc,
                     const int* restart_after, int n_restart, float eps, int compute_dtype, size_t* need);

// Watchdog self-test kernel (gemm_tc.cu).
int selftest_watchdog(long long spin_limit, int* status, cudaStream_t s);

}  // namespace dion3
