// Column selection for matrices stored un-oriented: W, M, G are [batch][m][n] with the short
// side n as columns, and the step selects k = ceil(f n) columns ("Dion3" summary, update-rule
// paragraph: a fraction of rows or columns).  The mathematics is the row step of the transpose;
// these passes move the data in the stored layout:
//
//   pass A  M <- M + G, optional W decay, and per column Kahan sums of |M_ij| (or M_ij^2) and
//           sums of squares over chunks of STEP_COL_CHUNK rows; a finalize kernel adds the chunks
//           in a fixed order (fp64) into the same certified key intervals the row pass produces.
//   pass C  X_S[j][i] = scale * M[i][S_j] in the compute dtype, M[i][S_j] <- mu M[i][S_j]: a
//           32 x 32 shared-memory transpose per block of rows.
//   update  W[i][S_j] += alpha * O[j][i] from O = GramNS(X_S), transposed the same way.
// Selection itself is the row selection kernel with strided vectors (step.cu).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dev_common.cuh"
#include "internal.h"

namespace dion3 {
namespace {

using dev::kahan_add;

using dev::from_f;
using dev::to_f;

struct ColA {
  int m, n, nchunk;
  float* M;
  const void* G;
  float* W;
  float w_decay;
  bool decay;
  const float* hyper;
  double eta_scale;
  bool keys;
  float* part_s;
  float* part_q;
};

// Pass A: one thread per (column, chunk of rows); consecutive threads take consecutive columns,
// so every row access of a warp is 128 contiguous bytes.  Four rows are loaded before use.
template <typename TG, int NORM_P>
__global__ void __launch_bounds__(256) colkeys_kernel(const ColA a) {
  const int c = blockIdx.y * 256 + threadIdx.x;
  const int ch = blockIdx.x;
  const long long b = blockIdx.z;
  if (c >= a.n) return;
  const float w_decay =
      a.hyper ? __double2float_rn(__dsub_rn(1.0, __dmul_rn(__dmul_rn(static_cast<double>(a.hyper[1]), a.eta_scale),
                                                            static_cast<double>(a.hyper[2]))))
              : a.w_decay;
  const long long base = b * a.m * a.n + c;
  const int i0 = ch * STEP_COL_CHUNK;
  const int i1 = min(a.m, i0 + STEP_COL_CHUNK);
  const TG* G = static_cast<const TG*>(a.G);
  float s = 0.f, comp = 0.f, q2 = 0.f;
  bool bad = false;
  for (int i = i0; i < i1; i += 4) {
    float x[4], g[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long off = base + static_cast<long long>(i + u) * a.n;
      x[u] = i + u < i1 ? a.M[off] : 0.f;
      g[u] = i + u < i1 ? to_f<TG>(G[off]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (i + u >= i1) break;
      const long long off = base + static_cast<long long>(i + u) * a.n;
      const float v = __fadd_rn(x[u], g[u]);
      a.M[off] = v;
      if (a.decay) a.W[off] = __fmul_rn(a.W[off], w_decay);
      q2 = fmaf(v, v, q2);
      if (a.keys) {
        bad |= !isfinite(v);
        kahan_add(s, comp, NORM_P == 1 ? fabsf(v) : __fmul_rn(v, v));
      }
    }
  }
  const long long po = (b * a.nchunk + ch) * a.n + c;
  a.part_q[po] = q2;
  if (a.keys) a.part_s[po] = bad ? __int_as_float(0x7fc00000) : s;  // NaN marks a non-finite momentum
}

struct ColF {
  long long total;  // batch * n
  int m, n, nchunk;
  bool keys;
  const float* part_s;
  const float* part_q;
  float* key_lo;
  float* key_hi;
  float* colsq;
  int* status;
};

// Chunk sums of each column, added in chunk order in fp64.  Every chunk's Kahan sum of at most
// STEP_COL_CHUNK nonnegative terms is within (2u + O(N u^2)) of its exact value (3u for
// squares), and the fp64 combination adds less than nchunk * 2^-53; the 2^-21 (8u) margin of
// the row pass covers it, and the absolute term covers gradual underflow.
__global__ void __launch_bounds__(256) colkeys_finalize_kernel(const ColF a) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= a.total) return;
  const long long b = idx / a.n, c = idx - b * a.n;
  double tot = 0.0, q = 0.0;
  bool nan = false, inf = false;
  for (int ch = 0; ch < a.nchunk; ++ch) {
    const long long po = (b * a.nchunk + ch) * a.n + c;
    q += static_cast<double>(a.part_q[po]);
    if (a.keys) {
      const float ps = a.part_s[po];
      nan |= isnan(ps);
      inf |= isinf(ps);
      tot += static_cast<double>(ps);
    }
  }
  a.colsq[idx] = static_cast<float>(q);
  if (!a.keys) return;
  float lo, hi;
  if (nan) {
    if (a.status) atomicOr(a.status, DION3_DEV_NONFINITE);
    lo = hi = __int_as_float(0x7f800000);  // ranks as the largest, like the row pass
  } else if (inf) {
    lo = 0.f;  // fp32 overflow of a chunk sum: the exact path decides
    hi = __int_as_float(0x7f800000);
  } else {
    const double bound = tot * 0x1p-21 + static_cast<double>(a.m) * 0x1p-146;
    lo = __double2float_rd(fmax(tot - bound, 0.0));
    hi = __double2float_ru(tot + bound);
  }
  a.key_lo[idx] = lo;
  a.key_hi[idx] = hi;
}

struct ColC {
  int m, n, k;
  float* M;
  const int32_t* sel;
  void* XS;
  long long ldx;
  float mu;
  const float* mu_dev;
  const float* scale;
  int* status;
};

// Pass C: a block of 32 rows; 8 warps.  Lanes over 32 selected columns read M[i][S_j] (and
// decay it), the tile is transposed in shared memory, lanes over 32 rows write X_S[j][i].
template <typename TC>
__global__ void __launch_bounds__(256) gather_cols_kernel(const ColC a) {
  __shared__ float tile[32][33];
  const long long b = blockIdx.y;
  const int i0 = blockIdx.x * 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const float f = a.scale[b];
  const float mu = a.mu_dev ? *a.mu_dev : a.mu;
  const int32_t* sel = a.sel + b * a.k;
  float* Mb = a.M + b * a.m * a.n;
  TC* Xb = static_cast<TC*>(a.XS) + b * a.k * a.ldx;
  for (int jc = 0; jc < a.k; jc += 32) {
    const int j = jc + lane;
    const int col = j < a.k ? sel[j] : -1;
    dev::range_check(col >= -1 && col < a.n, a.status);
    const bool ok = col >= 0 && col < a.n;  // -1 only after a failed selection
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int il = 4 * w + rr, i = i0 + il;
      float x = 0.f;
      if (ok && i < a.m) {
        float* p = Mb + static_cast<long long>(i) * a.n + col;
        x = *p;
        *p = __fmul_rn(mu, x);
      }
      tile[il][lane] = x;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int jl = 4 * w + rr, jj = jc + jl;
      if (jj < a.k && i0 + lane < a.m) Xb[jj * a.ldx + i0 + lane] = from_f<TC>(tile[lane][jl] * f);
    }
    __syncthreads();
  }
}

struct ColU {
  int m, n, k;
  float* W;
  const int32_t* sel;
  const void* O;
  long long ldo;
  float alpha;
  const float* eta_dev;
  double eta_scale;
  int* status;
};

// W update: lanes over 32 rows read O[j][i] (coalesced), the tile is transposed, lanes over 32
// selected columns add alpha * O[j][i] into W[i][S_j].
template <typename TC>
__global__ void __launch_bounds__(256) scatter_cols_kernel(const ColU a) {
  __shared__ float tile[32][33];
  const long long b = blockIdx.y;
  const int i0 = blockIdx.x * 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const float alpha =
      a.eta_dev ? __double2float_rn(-__dmul_rn(static_cast<double>(*a.eta_dev), a.eta_scale)) : a.alpha;
  const int32_t* sel = a.sel + b * a.k;
  float* Wb = a.W + b * a.m * a.n;
  const TC* Ob = static_cast<const TC*>(a.O) + b * a.k * a.ldo;
  for (int jc = 0; jc < a.k; jc += 32) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int jl = 4 * w + rr, jj = jc + jl;
      tile[jl][lane] = (jj < a.k && i0 + lane < a.m) ? to_f<TC>(Ob[jj * a.ldo + i0 + lane]) : 0.f;
    }
    __syncthreads();
    const int j = jc + lane;
    const int col = j < a.k ? sel[j] : -1;
    dev::range_check(col >= -1 && col < a.n, a.status);
    const bool ok = col >= 0 && col < a.n;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int il = 4 * w + rr, i = i0 + il;
      if (ok && i < a.m) {
        float* p = Wb + static_cast<long long>(i) * a.n + col;
        *p = fmaf(tile[lane][il], alpha, *p);
      }
    }
    __syncthreads();
  }
}

template <typename TG>
int launch_colkeys(const ColA& a, int batch, int norm_p, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(a.nchunk), static_cast<unsigned>((a.n + 255) / 256),
                  static_cast<unsigned>(batch));
  if (norm_p == 2)
    colkeys_kernel<TG, 2><<<grid, 256, 0, s>>>(a);
  else
    colkeys_kernel<TG, 1><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

}  // namespace

int step_colkeys(const StepArgs& s, cudaStream_t st) {
  if (s.batch <= 0 || s.n <= 0) return DION3_OK;
  if (s.batch > 65535) return DION3_EUNSUPPORTED;
  ColA a{};
  a.m = s.m;
  a.n = s.n;
  a.nchunk = s.nchunk;
  a.M = s.M;
  a.G = s.G;
  a.W = s.W;
  a.w_decay = s.w_decay;
  a.decay = s.decay;
  a.hyper = s.hyper;
  a.eta_scale = s.eta_scale;
  a.keys = s.norm_p != DION3_SELECT_GIVEN && s.k < s.n;
  a.part_s = s.part_s;
  a.part_q = s.part_q;
  int rc;
  switch (s.g_dtype) {
    case FP32:
      rc = launch_colkeys<float>(a, s.batch, s.norm_p, st);
      break;
    case FP16:
      rc = launch_colkeys<__half>(a, s.batch, s.norm_p, st);
      break;
    default:
      rc = launch_colkeys<__nv_bfloat16>(a, s.batch, s.norm_p, st);
      break;
  }
  if (rc) return rc;
  ColF f{};
  f.total = static_cast<long long>(s.batch) * s.n;
  f.m = s.m;
  f.n = s.n;
  f.nchunk = s.nchunk;
  f.keys = a.keys;
  f.part_s = s.part_s;
  f.part_q = s.part_q;
  f.key_lo = s.key_lo;
  f.key_hi = s.key_hi;
  f.colsq = s.rowsq;
  f.status = s.status;
  colkeys_finalize_kernel<<<static_cast<unsigned>((f.total + 255) / 256), 256, 0, st>>>(f);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

int step_gather_cols(const StepArgs& s, cudaStream_t st) {
  if (s.batch <= 0 || s.k <= 0) return DION3_OK;
  if (s.batch > 65535) return DION3_EUNSUPPORTED;
  ColC c{};
  c.m = s.m;
  c.n = s.n;
  c.k = s.k;
  c.M = s.M;
  c.sel = s.sel;
  c.XS = s.XS;
  c.ldx = s.ldx;
  c.mu = s.mu;
  c.mu_dev = s.hyper;
  c.scale = s.scale;
  c.status = s.status;
  const dim3 grid(static_cast<unsigned>((s.m + 31) / 32), static_cast<unsigned>(s.batch));
  switch (s.cdt) {
    case FP32:
      gather_cols_kernel<float><<<grid, 256, 0, st>>>(c);
      break;
    case FP16:
      gather_cols_kernel<__half><<<grid, 256, 0, st>>>(c);
      break;
    default:
      gather_cols_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(c);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

int step_scatter_cols(const StepArgs& s, const void* O, int64_t ldo, float alpha, const float* eta_dev,
                      double eta_scale, cudaStream_t st) {
  if (s.batch <= 0 || s.k <= 0) return DION3_OK;
  if (s.batch > 65535) return DION3_EUNSUPPORTED;
  ColU u{};
  u.m = s.m;
  u.n = s.n;
  u.k = s.k;
  u.W = s.W;
  u.sel = s.sel;
  u.O = O;
  u.ldo = ldo;
  u.alpha = alpha;
  u.eta_dev = eta_dev;
  u.eta_scale = eta_scale;
  u.status = s.status;
  const dim3 grid(static_cast<unsigned>((s.m + 31) / 32), static_cast<unsigned>(s.batch));
  switch (s.cdt) {
    case FP32:
      scatter_cols_kernel<float><<<grid, 256, 0, st>>>(u);
      break;
    case FP16:
      scatter_cols_kernel<__half><<<grid, 256, 0, st>>>(u);
      break;
    default:
      scatter_cols_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(u);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

}  // namespace dion3
