// C ABI of libdion3.so: argument validation, workspace layout and the launch sequences of
// Gram Newton-Schulz ("Dion3: Full-Stack Orthogonal Updates", core method Theorem 2 and
// method details Algorithm 3) and of one Dion3 step (Algorithm 4).  Everything here runs on
// the host and only enqueues kernels on the caller's stream.
#include <cmath>
#include <cstring>

#include "internal.h"

using namespace dion3;

namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ld_ok(int64_t ld, int dt) { return (ld * dtype_size(dt)) % 16 == 0; }

constexpr size_t WS_ALIGN = 256;

struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    off = static_cast<size_t>(round_up(static_cast<int64_t>(off), WS_ALIGN));
    const size_t at = off;
    off += bytes;
    return at;
  }
};

// Buffers of the Gram Newton-Schulz core for `batch` matrices of n x m.
struct CoreLayout {
  size_t R = 0, Z = 0, Q = 0, Tm = 0, X1 = 0, X2 = 0;
  int64_t ldn = 0, ldm = 0;
};

void core_layout(Carve& cv, CoreLayout& L, int batch, int n, int m, int cdt, int n_restart) {
  const int es = dtype_size(cdt);
  L.ldn = round_up(n, 8);
  L.ldm = round_up(m, 8);
  const size_t nn = static_cast<size_t>(batch) * n * L.ldn * es;
  const size_t nm = static_cast<size_t>(batch) * n * L.ldm * es;
  L.R = cv.take(nn);
  L.Z = cv.take(nn);
  L.Q = cv.take(nn);
  L.Tm = cv.take(nn);
  L.X1 = n_restart >= 1 ? cv.take(nm) : 0;
  L.X2 = n_restart >= 2 ? cv.take(nm) : 0;
}

struct GramLayout {
  size_t rowsq, scale, alpha2, xcopy;
  CoreLayout core;
  size_t total;
};

GramLayout gram_layout(int batch, int n, int m, bool need_copy, int cdt, int n_restart) {
  GramLayout L{};
  Carve cv;
  L.rowsq = cv.take(sizeof(float) * static_cast<size_t>(batch) * n);
  L.scale = cv.take(sizeof(float) * batch);
  L.alpha2 = cv.take(sizeof(float) * batch);
  L.xcopy = need_copy ? cv.take(static_cast<size_t>(batch) * n * round_up(m, 8) * dtype_size(cdt)) : 0;
  core_layout(cv, L.core, batch, n, m, cdt, n_restart);
  L.total = round_up(static_cast<int64_t>(cv.off), WS_ALIGN);
  return L;
}

// Standard Newton-Schulz: the prescaled X in two ping-pong buffers, A = X X^T and
// B = b A + c A^2.
struct NsLayout {
  size_t rowsq, scale, X[2], A, B;
  int64_t ldn, ldm;
  size_t total;
};

NsLayout ns_layout(int batch, int n, int m, int cdt) {
  NsLayout L{};
  Carve cv;
  const int es = dtype_size(cdt);
  L.ldn = round_up(n, 8);
  L.ldm = round_up(m, 8);
  L.rowsq = cv.take(sizeof(float) * static_cast<size_t>(batch) * n);
  L.scale = cv.take(sizeof(float) * batch);
  for (int i = 0; i < 2; ++i) L.X[i] = cv.take(static_cast<size_t>(batch) * n * L.ldm * es);
  L.A = cv.take(static_cast<size_t>(batch) * n * L.ldn * es);
  L.B = cv.take(static_cast<size_t>(batch) * n * L.ldn * es);
  L.total = round_up(static_cast<int64_t>(cv.off), WS_ALIGN);
  return L;
}

struct StepLayout {
  size_t key_lo, key_hi, exact, rowsq, scale, xs, carry;
  size_t part_s, part_q, obuf;  // column selection: chunk sums of the column keys, and O
  int nchunk;
  CoreLayout core;
  size_t total;
};

// n keys (rows, or columns with `cols`), each a vector of m entries.
StepLayout step_layout(int batch, int n, int m, int k, int norm_p, int cdt, int n_restart, bool cols = false) {
  StepLayout L{};
  Carve cv;
  L.key_lo = cv.take(sizeof(float) * static_cast<size_t>(batch) * n);
  L.key_hi = cv.take(sizeof(float) * static_cast<size_t>(batch) * n);
  L.exact = cv.take(sizeof(uint64_t) * static_cast<size_t>(batch) * n * step_exact_limbs(norm_p));
  L.rowsq = cv.take(sizeof(float) * static_cast<size_t>(batch) * n);
  L.scale = cv.take(sizeof(float) * batch);
  L.xs = cv.take(static_cast<size_t>(batch) * k * round_up(m, 8) * dtype_size(cdt));
  L.carry = cols ? 0 : cv.take(static_cast<size_t>(batch) * n);  // per-row flags of a carried decay
  if (cols) {
    L.nchunk = (m + STEP_COL_CHUNK - 1) / STEP_COL_CHUNK;
    L.part_s = cv.take(sizeof(float) * static_cast<size_t>(batch) * L.nchunk * n);
    L.part_q = cv.take(sizeof(float) * static_cast<size_t>(batch) * L.nchunk * n);
    L.obuf = cv.take(static_cast<size_t>(batch) * k * round_up(m, 8) * dtype_size(cdt));
  }
  core_layout(cv, L.core, batch, k, m, cdt, n_restart);
  L.total = round_up(static_cast<int64_t>(cv.off), WS_ALIGN);
  return L;
}

int check_schedule(int T, const float* abc, const int* restart_after, int n_restart) {
  if (T < 1 || abc == nullptr) return DION3_EINVAL;
  if (n_restart < 0) return DION3_EINVAL;
  if (n_restart > 0 && restart_after == nullptr) return DION3_EINVAL;
  for (int i = 0; i < n_restart; ++i) {
    if (restart_after[i] < 1 || restart_after[i] > T - 1) return DION3_EINVAL;
    if (i > 0 && restart_after[i] <= restart_after[i - 1]) return DION3_EINVAL;
  }
  for (int i = 0; i < 3 * T; ++i)
    if (!std::isfinite(abc[i])) return DION3_EINVAL;
  return DION3_OK;
}

// The Gram Newton-Schulz iteration on a batch of n x m matrices whose prescale is folded
// into alpha: R_0 = alpha2_b * X0 X0^T and the first Q X product uses alpha = xscale_b.
struct Core {
  int batch = 0, n = 0, m = 0, cdt = BF16;
  Mat X0;
  const float* xscale = nullptr;
  const float* alpha2 = nullptr;
  char* ws = nullptr;
  CoreLayout L;
  int T = 0;
  const float* abc = nullptr;
  const int* restarts = nullptr;
  int n_restart = 0;
  bool wupd = false;
  Mat Out;
  float* W = nullptr;
  int64_t ldw = 0, sW = 0;
  const int* sel = nullptr;
  int w_rows = 0;
  float w_alpha = 0.f;
  const float* eta_dev = nullptr;  // when set, the W update's alpha is -double(*eta_dev) * eta_scale
  double eta_scale = 0.0;
  int* status = nullptr;
};

int run_core(const Core& c, cudaStream_t s) {
  auto nn = [&](size_t off) {
    Mat mm;
    mm.ptr = c.ws + off;
    mm.ld = c.L.ldn;
    mm.stride = static_cast<int64_t>(c.n) * c.L.ldn;
    mm.dtype = c.cdt;
    return mm;
  };
  auto sym = [&](const Mat& A, const Mat& B, const Mat& D, int K, float alpha, const float* ab, const Mat& C,
                 float beta, float gamma) {
    GemmCall g;
    g.batch = c.batch;
    g.M = c.n;
    g.N = c.n;
    g.K = K;
    g.epi = EPI_SYM;
    g.A = A;
    g.B = B;
    g.C = C;
    g.beta = beta;
    g.D = D;
    g.alpha = alpha;
    g.alpha_batch = ab;
    g.gamma = gamma;
    g.status = c.status;
    return gemm(g, s);
  };
  // `last`: the product that writes the result (Out, or W through the row update).
  auto gen = [&](const Mat& Q, const Mat& X, float alpha, const float* ab, int epi, const Mat& D, bool last) {
    GemmCall g;
    g.batch = c.batch;
    g.M = c.n;
    g.N = c.m;
    g.K = c.n;
    g.epi = epi;
    g.A = Q;
    g.B = X;
    g.D = D;
    g.alpha = alpha;
    g.alpha_batch = ab;
    g.W = c.W;
    g.ldw = c.ldw;
    g.sW = c.sW;
    g.sel = c.sel;
    g.ssel = c.n;
    g.w_rows = c.w_rows;
    if (epi == EPI_WUPD) {
      g.eta_dev = c.eta_dev;
      g.eta_scale = c.eta_scale;
    }
    g.status = c.status;
    g.check_finite = last;
    return gemm(g, s);
  };

  size_t Rb = c.L.R, Zb = c.L.Z, Qb = c.L.Q, Tb = c.L.Tm;
  const Mat none;
  int rc = sym(c.X0, c.X0, nn(Rb), c.m, 1.f, c.alpha2, none, 0.f, 0.f);
  if (rc) return rc;

  // Small Gram matrices: every restart segment (its iterations from a (re)start up to the next
  // restart or the end) is one fused launch that keeps R, Z and Q on chip.
  bool fused = c.n <= 128 && c.cdt != FP32;
  for (int i = 0, t0 = 1; fused && i <= c.n_restart; ++i) {
    const int t1 = i < c.n_restart ? c.restarts[i] : c.T;
    if (t1 - t0 + 1 > DION3_SEG_MAX_ITERS) fused = false;
    t0 = t1 + 1;
  }
  if (fused) {
    Mat Xcur = c.X0;
    const float* xs = c.xscale;
    int next_x = 0;
    for (int i = 0, t0 = 1; i <= c.n_restart; ++i) {
      const int t1 = i < c.n_restart ? c.restarts[i] : c.T;
      rc = gram_segment(c.batch, c.n, nn(Rb), nn(Qb), t1 - t0 + 1, c.abc + 3 * (t0 - 1), c.status, s);
      if (rc) return rc;
      if (i < c.n_restart) {  // X <- Q X, R <- X X^T
        Mat Xn;
        Xn.ptr = c.ws + (next_x == 0 ? c.L.X1 : c.L.X2);
        Xn.ld = c.L.ldm;
        Xn.stride = static_cast<int64_t>(c.n) * c.L.ldm;
        Xn.dtype = c.cdt;
        next_x ^= 1;
        rc = gen(nn(Qb), Xcur, 1.f, xs, EPI_GEN, Xn, false);
        if (rc) return rc;
        Xcur = Xn;
        xs = nullptr;
        rc = sym(Xcur, Xcur, nn(Rb), c.m, 1.f, nullptr, none, 0.f, 0.f);
        if (rc) return rc;
      }
      t0 = t1 + 1;
    }
    if (c.wupd) return gen(nn(Qb), Xcur, c.w_alpha, xs, EPI_WUPD, none, true);
    return gen(nn(Qb), Xcur, 1.f, xs, EPI_GEN, c.Out, true);
  }

  bool q_identity = true;
  Mat Xcur = c.X0;
  const float* xs = c.xscale;
  int next_x = 0;
  int ri = 0;
  for (int t = 1; t <= c.T; ++t) {
    const float a = c.abc[3 * (t - 1)], b = c.abc[3 * (t - 1) + 1], cc = c.abc[3 * (t - 1) + 2];
    // Z = c R R + b R + a I
    rc = sym(nn(Rb), nn(Rb), nn(Zb), c.n, cc, nullptr, nn(Rb), b, a);
    if (rc) return rc;
    size_t Zcur = Zb;
    if (q_identity) {
      // Q = I Z = Z: Q takes over Z's buffer (still read below as Z); the old Q buffer
      // becomes the next iteration's Z buffer.
      std::swap(Qb, Zb);
      Zcur = Qb;
      q_identity = false;
    } else {
      rc = sym(nn(Qb), nn(Zb), nn(Tb), c.n, 1.f, nullptr, none, 0.f, 0.f);
      if (rc) return rc;
      std::swap(Qb, Tb);
    }
    const bool restart = ri < c.n_restart && c.restarts[ri] == t;
    if (restart) {
      ++ri;
      Mat Xn;
      Xn.ptr = c.ws + (next_x == 0 ? c.L.X1 : c.L.X2);
      Xn.ld = c.L.ldm;
      Xn.stride = static_cast<int64_t>(c.n) * c.L.ldm;
      Xn.dtype = c.cdt;
      next_x ^= 1;
      rc = gen(nn(Qb), Xcur, 1.f, xs, EPI_GEN, Xn, false);
      if (rc) return rc;
      Xcur = Xn;
      xs = nullptr;
      rc = sym(Xcur, Xcur, nn(Rb), c.m, 1.f, nullptr, none, 0.f, 0.f);
      if (rc) return rc;
      q_identity = true;
    } else if (t < c.T) {
      rc = sym(nn(Rb), nn(Zcur), nn(Tb), c.n, 1.f, nullptr, none, 0.f, 0.f);  // R Z
      if (rc) return rc;
      rc = sym(nn(Tb), nn(Zcur), nn(Rb), c.n, 1.f, nullptr, none, 0.f, 0.f);  // (R Z) Z
      if (rc) return rc;
    }
  }
  if (c.wupd) return gen(nn(Qb), Xcur, c.w_alpha, xs, EPI_WUPD, none, true);
  return gen(nn(Qb), Xcur, 1.f, xs, EPI_GEN, c.Out, true);
}

}  // namespace

extern "C" {

int dion3_abi_version(void) { return DION3_ABI_VERSION; }

#ifndef DION3_RANGE_CHECKS
#define DION3_RANGE_CHECKS 0
#endif
int dion3_range_checks(void) { return DION3_RANGE_CHECKS; }

const char* dion3_status_str(int code) {
  switch (code) {
    case DION3_OK:
      return "DION3_OK";
    case DION3_EINVAL:
      return "DION3_EINVAL: invalid argument";
    case DION3_EUNSUPPORTED:
      return "DION3_EUNSUPPORTED: unsupported dtype combination or size";
    case DION3_EWORKSPACE:
      return "DION3_EWORKSPACE: workspace missing or too small";
    case DION3_ECUDA:
      return "DION3_ECUDA: a CUDA call failed";
    case DION3_EALIGN:
      return "DION3_EALIGN: pointer, leading dimension or stride not 16-byte aligned";
    default:
      return "unknown dion3 status";
  }
}

int dion3_k(int n, int f_num, int f_den) {
  if (n < 0 || f_num <= 0 || f_den <= 0 || f_num > f_den) return -1;
  const int64_t v = (static_cast<int64_t>(n) * f_num + f_den - 1) / f_den;
  return static_cast<int>(v);
}

int dion3_sym_gemm(int batch, int n, int k, const void* A, int64_t lda, int64_t strideA, const void* B, int64_t ldb,
                   int64_t strideB, const void* C, int64_t ldc, int64_t strideC, void* D, int64_t ldd,
                   int64_t strideD, float alpha, float beta, float gamma, int in_dtype, int out_dtype,
                   int* status_dev, void* stream) {
  if (batch < 0 || n < 0 || k < 0) return DION3_EINVAL;
  if (!dtype_valid(in_dtype) || !dtype_valid(out_dtype)) return DION3_EINVAL;
  if (in_dtype == FP32 ? out_dtype != FP32 : (out_dtype != in_dtype && out_dtype != FP32)) return DION3_EUNSUPPORTED;
  if (batch == 0 || n == 0) return DION3_OK;
  if (D == nullptr || (beta != 0.f && C == nullptr)) return DION3_EINVAL;
  if (k == 0) {  // A and B are never read: D = beta C + gamma I
    A = B = D;
    lda = ldb = ldd;
    strideA = strideB = strideD;
  }
  if (A == nullptr) return DION3_EINVAL;
  if (lda < k || ldd < n) return DION3_EINVAL;
  if (B == nullptr) {
    B = A;
    ldb = lda;
    strideB = strideA;
  }
  if (ldb < k) return DION3_EINVAL;
  if (beta != 0.f && ldc < n) return DION3_EINVAL;
  if (batch > 1) {
    if (strideA < n * lda || strideB < n * ldb || strideD < n * ldd) return DION3_EINVAL;
    if (beta != 0.f && strideC < n * ldc) return DION3_EINVAL;
  }
  if (C != nullptr && C == D && beta != 0.f && (ldc != ldd || (batch > 1 && strideC != strideD))) return DION3_EINVAL;
  const bool reads_ab = k > 0;
  if (!al16(D) || (beta != 0.f && !al16(C))) return DION3_EALIGN;
  if (reads_ab && (!al16(A) || !al16(B) || !ld_ok(lda, in_dtype) || !ld_ok(ldb, in_dtype))) return DION3_EALIGN;
  if (!ld_ok(ldd, out_dtype) || (beta != 0.f && !ld_ok(ldc, out_dtype))) return DION3_EALIGN;
  if (batch > 1) {
    if (reads_ab && (!ld_ok(strideA, in_dtype) || !ld_ok(strideB, in_dtype))) return DION3_EALIGN;
    if (!ld_ok(strideD, out_dtype) || (beta != 0.f && !ld_ok(strideC, out_dtype))) return DION3_EALIGN;
  }
  GemmCall g;
  g.batch = batch;
  g.M = n;
  g.N = n;
  g.K = k;
  g.epi = EPI_SYM;
  g.A = Mat{A, lda, strideA, in_dtype};
  g.B = Mat{B, ldb, strideB, in_dtype};
  if (beta != 0.f) g.C = Mat{C, ldc, strideC, out_dtype};
  g.beta = beta;
  g.D = Mat{D, ldd, strideD, out_dtype};
  g.alpha = alpha;
  g.gamma = gamma;
  g.status = status_dev;
  return gemm(g, static_cast<cudaStream_t>(stream));
}

// The workspace holds a copy of X unless X can be read in place: same dtype as the compute
// dtype and rows of a whole number of 16-byte units.
static bool query_needs_copy(int m, int x_dtype, int compute_dtype) {
  return x_dtype != compute_dtype || (static_cast<int64_t>(m) * dtype_size(x_dtype)) % 16 != 0;
}

size_t dion3_gram_ns_workspace_bytes(int batch, int n, int m, int x_dtype, int compute_dtype, int n_restart) {
  if (batch < 0 || n < 0 || m < n || n_restart < 0) return 0;
  if (!dtype_valid(x_dtype) || !dtype_valid(compute_dtype)) return 0;
  return gram_layout(batch, n, m, query_needs_copy(m, x_dtype, compute_dtype), compute_dtype, n_restart).total;
}

}  // extern "C"

namespace dion3 {

int gram_ns_validate(int batch, int n, int m, const void* X, int64_t ldx, int64_t strideX, int x_dtype,
                     const void* Out, int64_t ldo, int64_t strideO, int out_dtype, int T, const float* abc,
                     const int* restart_after, int n_restart, float eps, int compute_dtype, size_t* need) {
  *need = 0;
  if (batch < 0 || n < 0 || m < 0) return DION3_EINVAL;
  if (!dtype_valid(x_dtype) || !dtype_valid(out_dtype) || !dtype_valid(compute_dtype)) return DION3_EINVAL;
  if (int rc = check_schedule(T, abc, restart_after, n_restart)) return rc;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return DION3_EINVAL;
  if (batch == 0 || n == 0) return DION3_OK;
  if (n > m) return DION3_EINVAL;
  if (compute_dtype == FP32 && out_dtype != FP32) return DION3_EUNSUPPORTED;
  if (X == nullptr || Out == nullptr) return DION3_EINVAL;
  if (ldx < m || ldo < m) return DION3_EINVAL;
  if (batch > 1 && (strideX < n * ldx || strideO < n * ldo)) return DION3_EINVAL;
  if (!al16(Out) || !ld_ok(ldo, out_dtype) || (batch > 1 && !ld_ok(strideO, out_dtype))) return DION3_EALIGN;
  const bool x_aligned = al16(X) && ld_ok(ldx, x_dtype) && (batch <= 1 || ld_ok(strideX, x_dtype));
  const bool need_copy = x_dtype != compute_dtype || !x_aligned;
  *need = gram_layout(batch, n, m, need_copy, compute_dtype, n_restart).total;
  return DION3_OK;
}

}  // namespace dion3

extern "C" {

int dion3_gram_ns(int batch, int n, int m, const void* X, int64_t ldx, int64_t strideX, int x_dtype, void* Out,
                  int64_t ldo, int64_t strideO, int out_dtype, int T, const float* abc, const int* restart_after,
                  int n_restart, float eps, int compute_dtype, void* workspace, size_t workspace_bytes,
                  int* status_dev, void* stream) {
  size_t need = 0;
  if (int rc = gram_ns_validate(batch, n, m, X, ldx, strideX, x_dtype, Out, ldo, strideO, out_dtype, T, abc,
                                restart_after, n_restart, eps, compute_dtype, &need))
    return rc;
  if (need == 0) return DION3_OK;  // empty batch or n == 0: nothing to do
  const bool x_aligned = al16(X) && ld_ok(ldx, x_dtype) && (batch <= 1 || ld_ok(strideX, x_dtype));
  const bool need_copy = x_dtype != compute_dtype || !x_aligned;
  const GramLayout L = gram_layout(batch, n, m, need_copy, compute_dtype, n_restart);
  if (workspace == nullptr || workspace_bytes < L.total) return DION3_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (WS_ALIGN - 1)) != 0) return DION3_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  float* rowsq = reinterpret_cast<float*>(ws + L.rowsq);
  float* scale = reinterpret_cast<float*>(ws + L.scale);
  float* alpha2 = reinterpret_cast<float*>(ws + L.alpha2);
  const int64_t ldm = round_up(m, 8);
  Mat Xin{X, ldx, strideX, x_dtype};
  int rc = rows_sumsq(batch, n, m, Xin, rowsq, status_dev, s);
  if (rc) return rc;
  rc = finalize_scale(batch, n, rowsq, eps, scale, need_copy ? nullptr : alpha2, status_dev, s);
  if (rc) return rc;
  if (need_copy) {  // the copy carries the prescale; nothing is folded into the GEMMs
    rc = scaled_cast(batch, n, m, Xin, scale, ws + L.xcopy, ldm, static_cast<int64_t>(n) * ldm, compute_dtype, s);
    if (rc) return rc;
  }
  Core c;
  c.batch = batch;
  c.n = n;
  c.m = m;
  c.cdt = compute_dtype;
  c.X0 = need_copy ? Mat{ws + L.xcopy, ldm, static_cast<int64_t>(n) * ldm, compute_dtype} : Xin;
  c.xscale = need_copy ? nullptr : scale;
  c.alpha2 = need_copy ? nullptr : alpha2;
  c.ws = ws;
  c.L = L.core;
  c.T = T;
  c.abc = abc;
  c.restarts = restart_after;
  c.n_restart = n_restart;
  c.Out = Mat{Out, ldo, strideO, out_dtype};
  c.status = status_dev;
  return run_core(c, s);
}

size_t dion3_ns_standard_workspace_bytes(int batch, int n, int m, int compute_dtype) {
  if (batch < 0 || n < 0 || m < n) return 0;
  if (!dtype_valid(compute_dtype)) return 0;
  return ns_layout(batch, n, m, compute_dtype).total;
}

int dion3_ns_standard(int batch, int n, int m, const void* X, int64_t ldx, int64_t strideX, int x_dtype, void* Out,
                      int64_t ldo, int64_t strideO, int out_dtype, int T, const float* abc, float eps,
                      int compute_dtype, void* workspace, size_t workspace_bytes, int* status_dev, void* stream) {
  if (batch < 0 || n < 0 || m < 0) return DION3_EINVAL;
  if (!dtype_valid(x_dtype) || !dtype_valid(out_dtype) || !dtype_valid(compute_dtype)) return DION3_EINVAL;
  if (int rc = check_schedule(T, abc, nullptr, 0)) return rc;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return DION3_EINVAL;
  if (batch == 0 || n == 0) return DION3_OK;
  if (n > m) return DION3_EINVAL;
  if (compute_dtype == FP32 && out_dtype != FP32) return DION3_EUNSUPPORTED;
  if (X == nullptr || Out == nullptr) return DION3_EINVAL;
  if (ldx < m || ldo < m) return DION3_EINVAL;
  if (batch > 1 && (strideX < n * ldx || strideO < n * ldo)) return DION3_EINVAL;
  if (!al16(Out) || !ld_ok(ldo, out_dtype) || (batch > 1 && !ld_ok(strideO, out_dtype))) return DION3_EALIGN;
  const NsLayout L = ns_layout(batch, n, m, compute_dtype);
  if (workspace == nullptr || workspace_bytes < L.total) return DION3_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (WS_ALIGN - 1)) != 0) return DION3_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  float* rowsq = reinterpret_cast<float*>(ws + L.rowsq);
  float* scale = reinterpret_cast<float*>(ws + L.scale);
  const int64_t snm = static_cast<int64_t>(n) * L.ldm, snn = static_cast<int64_t>(n) * L.ldn;
  const Mat Xb[2] = {Mat{ws + L.X[0], L.ldm, snm, compute_dtype}, Mat{ws + L.X[1], L.ldm, snm, compute_dtype}};
  const Mat Am{ws + L.A, L.ldn, snn, compute_dtype}, Bm{ws + L.B, L.ldn, snn, compute_dtype};
  const Mat Om{Out, ldo, strideO, out_dtype};
  // The last product writes Out directly when Out has the compute dtype (the a X term is read
  // in that dtype); otherwise it lands in a buffer that is converted at the end.
  const bool direct = out_dtype == compute_dtype;

  const Mat Xin{X, ldx, strideX, x_dtype};
  int rc = rows_sumsq(batch, n, m, Xin, rowsq, status_dev, s);
  if (rc) return rc;
  rc = finalize_scale(batch, n, rowsq, eps, scale, nullptr, status_dev, s);
  if (rc) return rc;
  rc = scaled_cast(batch, n, m, Xin, scale, const_cast<void*>(Xb[0].ptr), L.ldm, snm, compute_dtype, s);
  if (rc) return rc;
  int cur = 0;
  for (int t = 1; t <= T; ++t) {
    const float a = abc[3 * (t - 1)], b = abc[3 * (t - 1) + 1], c = abc[3 * (t - 1) + 2];
    GemmCall g;  // A = X X^T
    g.batch = batch;
    g.M = g.N = n;
    g.K = m;
    g.epi = EPI_SYM;
    g.A = g.B = Xb[cur];
    g.D = Am;
    g.status = status_dev;
    if ((rc = gemm(g, s))) return rc;
    GemmCall h;  // B = c A A + b A
    h.batch = batch;
    h.M = h.N = h.K = n;
    h.epi = EPI_SYM;
    h.A = h.B = Am;
    h.C = Am;
    h.beta = b;
    h.alpha = c;
    h.D = Bm;
    h.status = status_dev;
    if ((rc = gemm(h, s))) return rc;
    GemmCall u;  // X' = B X + a X
    u.batch = batch;
    u.M = n;
    u.N = m;
    u.K = n;
    u.epi = EPI_GEN;
    u.A = Bm;
    u.B = Xb[cur];
    u.C = Xb[cur];
    u.beta = a;
    u.D = (t == T && direct) ? Om : Xb[cur ^ 1];
    u.status = status_dev;
    u.check_finite = t == T;
    if ((rc = gemm(u, s))) return rc;
    cur ^= 1;
  }
  if (!direct) return scaled_cast(batch, n, m, Xb[cur], nullptr, Out, ldo, strideO, out_dtype, s);
  return DION3_OK;
}

size_t dion3_step_workspace_bytes(int batch, int n, int m, int f_num, int f_den, int norm_p, int compute_dtype,
                                  int n_restart) {
  if (batch < 0 || n < 0 || m < n || n_restart < 0) return 0;
  if (norm_p != DION3_SELECT_GIVEN && norm_p != 1 && norm_p != 2) return 0;
  if (!dtype_valid(compute_dtype)) return 0;
  const int k = dion3_k(n, f_num, f_den);
  if (k < 0) return 0;
  return step_layout(batch, n, m, k, norm_p, compute_dtype, n_restart).total;
}

int dion3_step_timed(int batch, int n, int m, float* W, float* M, const void* G, int g_dtype, int f_num, int f_den,
                     float mu, float eta, float wd, int norm_p, int T, const float* abc, const int* restart_after,
                     int n_restart, float eps, int compute_dtype, int32_t* sel_out, void* workspace,
                     size_t workspace_bytes, int* status_dev, void* stream, void* const* events, int n_events);

int dion3_step(int batch, int n, int m, float* W, float* M, const void* G, int g_dtype, int f_num, int f_den,
               float mu, float eta, float wd, int norm_p, int T, const float* abc, const int* restart_after,
               int n_restart, float eps, int compute_dtype, int32_t* sel_out, void* workspace,
               size_t workspace_bytes, int* status_dev, void* stream) {
  return dion3_step_timed(batch, n, m, W, M, G, g_dtype, f_num, f_den, mu, eta, wd, norm_p, T, abc, restart_after,
                          n_restart, eps, compute_dtype, sel_out, workspace, workspace_bytes, status_dev, stream,
                          nullptr, 0);
}

}  // extern "C"

namespace {

// One Dion3 step.  With hyper_dev == nullptr, mu, eta, wd are the host values; otherwise they
// are read on the device from hyper_dev[0..2] and `decay` says whether the W decay pass runs.
int step_impl(int batch, int n, int m, float* W, float* M, const void* G, int g_dtype, int f_num, int f_den,
              float mu, float eta, float wd, const float* hyper_dev, bool decay, int norm_p, int T, const float* abc,
              const int* restart_after, int n_restart, float eps, int compute_dtype, int32_t* sel_out,
              void* workspace, size_t workspace_bytes, int* status_dev, void* stream, void* const* events,
              int n_events, bool cols = false, const int32_t* carry_rows = nullptr, float carry_mu = 1.f,
              bool defer = false, float* carry_mu_dev = nullptr) {
  if (n_events < 0 || (n_events > 0 && events == nullptr)) return DION3_EINVAL;
  if (cols && (carry_rows != nullptr || defer)) return DION3_EUNSUPPORTED;
  if (carry_mu_dev != nullptr && (reinterpret_cast<uintptr_t>(carry_mu_dev) & 3u) != 0) return DION3_EALIGN;
  if (carry_rows != nullptr) {
    if (carry_mu_dev == nullptr && !std::isfinite(carry_mu)) return DION3_EINVAL;
    // A caller-chosen S is read from sel_out: a carried list there would be the new S.
    if (norm_p == DION3_SELECT_GIVEN && carry_rows == sel_out) return DION3_EINVAL;
    if ((reinterpret_cast<uintptr_t>(carry_rows) & 3u) != 0) return DION3_EALIGN;
  }
  if (batch < 0 || n < 0 || m < 0) return DION3_EINVAL;
  if (!dtype_valid(g_dtype) || !dtype_valid(compute_dtype)) return DION3_EINVAL;
  if (norm_p != DION3_SELECT_GIVEN && norm_p != 1 && norm_p != 2) return DION3_EINVAL;
  const int k = dion3_k(n, f_num, f_den);
  if (k < 0) return DION3_EINVAL;
  if (int rc = check_schedule(T, abc, restart_after, n_restart)) return rc;
  if (!std::isfinite(mu) || !std::isfinite(eta) || !std::isfinite(wd) || !(eps >= 0.f) || !std::isfinite(eps))
    return DION3_EINVAL;
  if (batch == 0 || n == 0) return DION3_OK;
  if (n > m) return DION3_EINVAL;
  if (n > 16384 || m > 65536) return DION3_EUNSUPPORTED;
  if (W == nullptr || M == nullptr || G == nullptr || sel_out == nullptr) return DION3_EINVAL;
  if (!al16(W) || !al16(M) || !al16(G) || !al16(sel_out)) return DION3_EALIGN;
  if (hyper_dev != nullptr && (reinterpret_cast<uintptr_t>(hyper_dev) & 3u) != 0) return DION3_EALIGN;
  if (cols && batch > 65535) return DION3_EUNSUPPORTED;
  const StepLayout L = step_layout(batch, n, m, k, norm_p, compute_dtype, n_restart, cols);
  if (workspace == nullptr || workspace_bytes < L.total) return DION3_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (WS_ALIGN - 1)) != 0) return DION3_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  // eta' = eta / sqrt(f); double arithmetic, rounded once to fp32 where it is used.  The device
  // path (hyper_dev) repeats exactly these operations on the value it reads.
  const double eta_scale = std::sqrt(static_cast<double>(f_den) / static_cast<double>(f_num));
  const double eta_p = static_cast<double>(eta) * eta_scale;
  const int64_t ldm = round_up(m, 8);

  StepArgs sa{};
  sa.batch = batch;
  sa.n = n;
  sa.m = m;
  sa.k = k;
  sa.W = W;
  sa.M = M;
  sa.G = G;
  sa.g_dtype = g_dtype;
  sa.norm_p = norm_p;
  sa.mu = mu;
  const double wd_term = eta_p * static_cast<double>(wd);
  sa.w_decay = static_cast<float>(1.0 - wd_term);
  sa.decay = hyper_dev != nullptr ? decay : (wd != 0.f && sa.w_decay != 1.0f);
  sa.hyper = hyper_dev;
  sa.eta_scale = eta_scale;
  sa.sel = sel_out;
  sa.key_lo = reinterpret_cast<float*>(ws + L.key_lo);
  sa.key_hi = reinterpret_cast<float*>(ws + L.key_hi);
  sa.exact = reinterpret_cast<uint64_t*>(ws + L.exact);
  sa.XS = ws + L.xs;
  sa.ldx = ldm;
  sa.cdt = compute_dtype;
  sa.rowsq = reinterpret_cast<float*>(ws + L.rowsq);
  sa.scale = reinterpret_cast<float*>(ws + L.scale);
  sa.eps = eps;
  sa.status = status_dev;
  sa.cols = cols;
  if (cols) {
    sa.part_s = reinterpret_cast<float*>(ws + L.part_s);
    sa.part_q = reinterpret_cast<float*>(ws + L.part_q);
    sa.nchunk = L.nchunk;
  } else {
    sa.carry_rows = carry_rows;
    sa.carry_flag = reinterpret_cast<uint8_t*>(ws + L.carry);
    sa.carry_mu = carry_mu;
    sa.defer = defer;
    sa.carry_mu_dev = carry_mu_dev;
  }

  // Phase boundaries for the caller's timing events (0: start ... 4: end).
  auto mark = [&](int i) {
    if (i < n_events && events[i] != nullptr) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
  };
  mark(0);
  int rc = cols ? step_colkeys(sa, s) : step_momentum_keys(sa, s);
  if (rc) return rc;
  mark(1);
  rc = step_select(sa, s);
  if (rc) return rc;
  mark(2);
  if (k == 0) {
    mark(3);
    mark(4);
    return DION3_OK;
  }
  rc = cols ? step_gather_cols(sa, s) : step_gather(sa, s);
  if (rc) return rc;
  mark(3);
  Core c;
  c.batch = batch;
  c.n = k;
  c.m = m;
  c.cdt = compute_dtype;
  c.X0 = Mat{sa.XS, ldm, static_cast<int64_t>(k) * ldm, compute_dtype};  // already prescaled
  c.ws = ws;
  c.L = L.core;
  c.T = T;
  c.abc = abc;
  c.restarts = restart_after;
  c.n_restart = n_restart;
  c.wupd = !cols;  // columns: O goes to the workspace and a transposing pass updates W
  if (cols) c.Out = Mat{ws + L.obuf, ldm, static_cast<int64_t>(k) * ldm, compute_dtype};
  c.W = W;
  c.ldw = m;
  c.sW = static_cast<int64_t>(n) * m;
  c.sel = sel_out;
  c.w_rows = n;
  c.w_alpha = static_cast<float>(-eta_p);
  if (hyper_dev != nullptr) {
    c.eta_dev = hyper_dev + 1;
    c.eta_scale = eta_scale;
  }
  c.status = status_dev;
  rc = run_core(c, s);
  if (rc) return rc;
  if (cols) {
    rc = step_scatter_cols(sa, ws + L.obuf, ldm, c.w_alpha, c.eta_dev, c.eta_scale, s);
    if (rc) return rc;
  }
  mark(4);
  return DION3_OK;
}

}  // namespace

extern "C" {

int dion3_step_timed(int batch, int n, int m, float* W, float* M, const void* G, int g_dtype, int f_num, int f_den,
                     float mu, float eta, float wd, int norm_p, int T, const float* abc, const int* restart_after,
                     int n_restart, float eps, int compute_dtype, int32_t* sel_out, void* workspace,
                     size_t workspace_bytes, int* status_dev, void* stream, void* const* events, int n_events) {
  return step_impl(batch, n, m, W, M, G, g_dtype, f_num, f_den, mu, eta, wd, nullptr, false, norm_p, T, abc,
                   restart_after, n_restart, eps, compute_dtype, sel_out, workspace, workspace_bytes, status_dev,
                   stream, events, n_events);
}

size_t dion3_step_cols_workspace_bytes(int batch, int m, int n, int f_num, int f_den, int norm_p, int compute_dtype,
                                       int n_restart) {
  if (batch < 0 || n < 0 || m < n || n_restart < 0) return 0;
  if (norm_p != DION3_SELECT_GIVEN && norm_p != 1 && norm_p != 2) return 0;
  if (!dtype_valid(compute_dtype)) return 0;
  const int k = dion3_k(n, f_num, f_den);
  if (k < 0) return 0;
  return step_layout(batch, n, m, k, norm_p, compute_dtype, n_restart, true).total;
}

int dion3_step_cols(int batch, int m, int n, float* W, float* M, const void* G, int g_dtype, int f_num, int f_den,
                    float mu, float eta, float wd, int norm_p, int T, const float* abc, const int* restart_after,
                    int n_restart, float eps, int compute_dtype, int32_t* sel_out, void* workspace,
                    size_t workspace_bytes, int* status_dev, void* stream) {
  return step_impl(batch, n, m, W, M, G, g_dtype, f_num, f_den, mu, eta, wd, nullptr, false, norm_p, T, abc,
                   restart_after, n_restart, eps, compute_dtype, sel_out, workspace, workspace_bytes, status_dev,
                   stream, nullptr, 0, true);
}

int dion3_step_dev(int batch, int n, int m, float* W, float* M, const void* G, int g_dtype, int f_num, int f_den,
                   const float* hyper_dev, int decay, int norm_p, int T, const float* abc, const int* restart_after,
                   int n_restart, float eps, int compute_dtype, int32_t* sel_out, void* workspace,
                   size_t workspace_bytes, int* status_dev, void* stream) {
  if (hyper_dev == nullptr) return DION3_EINVAL;
  return step_impl(batch, n, m, W, M, G, g_dtype, f_num, f_den, 0.f, 0.f, 0.f, hyper_dev, decay != 0, norm_p, T,
                   abc, restart_after, n_restart, eps, compute_dtype, sel_out, workspace, workspace_bytes, status_dev,
                   stream, nullptr, 0);
}

int dion3_step_carry(int batch, int n, int m, float* W, float* M, const void* G, int g_dtype, int f_num, int f_den,
                     float mu, float eta, float wd, int norm_p, int T, const float* abc, const int* restart_after,
                     int n_restart, float eps, int compute_dtype, int32_t* sel_out, const int32_t* carry_rows,
                     float carry_mu, int defer, void* workspace, size_t workspace_bytes, int* status_dev,
                     void* stream, void* const* events, int n_events) {
  return step_impl(batch, n, m, W, M, G, g_dtype, f_num, f_den, mu, eta, wd, nullptr, false, norm_p, T, abc,
                   restart_after, n_restart, eps, compute_dtype, sel_out, workspace, workspace_bytes, status_dev,
                   stream, events, n_events, false, carry_rows, carry_mu, defer != 0);
}

int dion3_step_dev_carry(int batch, int n, int m, float* W, float* M, const void* G, int g_dtype, int f_num,
                         int f_den, const float* hyper_dev, int decay, int norm_p, int T, const float* abc,
                         const int* restart_after, int n_restart, float eps, int compute_dtype, int32_t* sel_out,
                         const int32_t* carry_rows, float* carry_mu_dev, int defer, void* workspace,
                         size_t workspace_bytes, int* status_dev, void* stream) {
  if (hyper_dev == nullptr) return DION3_EINVAL;
  if ((carry_rows != nullptr || defer != 0) && carry_mu_dev == nullptr) return DION3_EINVAL;
  return step_impl(batch, n, m, W, M, G, g_dtype, f_num, f_den, 0.f, 0.f, 0.f, hyper_dev, decay != 0, norm_p, T,
                   abc, restart_after, n_restart, eps, compute_dtype, sel_out, workspace, workspace_bytes, status_dev,
                   stream, nullptr, 0, false, carry_rows, 1.f, defer != 0, carry_mu_dev);
}

int dion3_decay_rows(int batch, int n, int m, float* M, const int32_t* rows, int k, float mu, void* stream) {
  if (batch < 0 || n < 0 || m < 0 || k < 0 || k > n) return DION3_EINVAL;
  if (!std::isfinite(mu)) return DION3_EINVAL;
  if (batch == 0 || k == 0 || m == 0) return DION3_OK;
  if (M == nullptr || rows == nullptr) return DION3_EINVAL;
  if ((reinterpret_cast<uintptr_t>(M) & 3u) != 0 || (reinterpret_cast<uintptr_t>(rows) & 3u) != 0)
    return DION3_EALIGN;
  return step_decay_rows(batch, n, m, k, M, rows, mu, static_cast<cudaStream_t>(stream));
}

int dion3_selftest_watchdog(long long spin_limit_cycles, int* status_dev, void* stream) {
  if (status_dev == nullptr || spin_limit_cycles <= 0) return DION3_EINVAL;
  return selftest_watchdog(spin_limit_cycles, status_dev, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
