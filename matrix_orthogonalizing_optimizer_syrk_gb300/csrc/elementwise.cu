// Frobenius prescale support ("Muon: Orthogonalized Momentum ...", section "Doing an SVD
// without an SVD": X / (||X||_F + eps), norm in fp32).
//
// When X is read in place, the scale is folded into the alpha of the first X X^T product
// (alpha = scale^2) and of the first Q X product (alpha = scale).  When X has to be
// converted to the compute dtype, the conversion applies the scale, so that a 16-bit copy
// never sees values outside its range.  Reductions run in a fixed order (deterministic).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dev_common.cuh"
#include "internal.h"

namespace dion3 {
namespace {

using dev::from_f;
using dev::to_f;

// Per-row sum of squares (fp32 FMA chain per lane, fixed warp tree): one warp per row,
// grid-stride over all batch*n rows.
template <typename Tin>
__global__ void __launch_bounds__(256) rows_sumsq_kernel(int batch, int n, int m, const Tin* X, long long ldx,
                                                         long long sx, float* rowsq, int* status) {
  const long long rows = static_cast<long long>(batch) * n;
  const int lane = threadIdx.x & 31;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long row = w0; row < rows; row += nw) {
    const long long b = row / n, i = row - b * n;
    const Tin* src = X + b * sx + i * ldx;
    float acc = 0.f;
    for (int j = lane; j < m; j += 32) {
      const float x = to_f<Tin>(src[j]);
      acc = fmaf(x, x, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      rowsq[row] = acc;
      if (!isfinite(acc) && status) atomicOr(status, DION3_DEV_NONFINITE);
    }
  }
}

// Xc = X * scale[b] (scale == nullptr: a plain conversion), converted to Xc's dtype (one warp
// per row).
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) scaled_cast_kernel(int batch, int n, int m, const Tin* X, long long ldx,
                                                          long long sx, const float* scale, Tout* Xc,
                                                          long long ldc, long long sc) {
  const long long rows = static_cast<long long>(batch) * n;
  const int lane = threadIdx.x & 31;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long row = w0; row < rows; row += nw) {
    const long long b = row / n, i = row - b * n;
    const Tin* src = X + b * sx + i * ldx;
    Tout* dst = Xc + b * sc + i * ldc;
    const float f = scale ? scale[b] : 1.f;
    for (int j = lane; j < m; j += 32) dst[j] = from_f<Tout>(to_f<Tin>(src[j]) * f);
  }
}

__global__ void finalize_scale_kernel(int batch, int rows, const float* rowsq, float eps, float* scale,
                                      float* alpha2, int* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  double s = 0.0;
  const float* r = rowsq + static_cast<long long>(b) * rows;
  for (int i = 0; i < rows; ++i) s += static_cast<double>(r[i]);
  const double sc = 1.0 / (sqrt(s) + static_cast<double>(eps));
  if (!isfinite(s) && status) atomicOr(status, DION3_DEV_NONFINITE);
  scale[b] = static_cast<float>(sc);
  if (alpha2) alpha2[b] = static_cast<float>(sc * sc);
}

unsigned grid_for_rows(long long rows) {
  long long blocks = (rows + 7) / 8;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

template <typename Tin>
int launch_sumsq(int batch, int n, int m, const Mat& X, float* rowsq, int* status, cudaStream_t s) {
  rows_sumsq_kernel<Tin><<<grid_for_rows(static_cast<long long>(batch) * n), 256, 0, s>>>(
      batch, n, m, static_cast<const Tin*>(X.ptr), X.ld, X.stride, rowsq, status);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

template <typename Tin, typename Tout>
int launch_cast(int batch, int n, int m, const Mat& X, const float* scale, void* Xc, int64_t ldc, int64_t sc,
                cudaStream_t s) {
  scaled_cast_kernel<Tin, Tout><<<grid_for_rows(static_cast<long long>(batch) * n), 256, 0, s>>>(
      batch, n, m, static_cast<const Tin*>(X.ptr), X.ld, X.stride, scale, static_cast<Tout*>(Xc), ldc, sc);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

template <typename Tin>
int cast_out(int batch, int n, int m, const Mat& X, const float* scale, void* Xc, int64_t ldc, int64_t sc, int cdt,
             cudaStream_t s) {
  switch (cdt) {
    case FP32:
      return launch_cast<Tin, float>(batch, n, m, X, scale, Xc, ldc, sc, s);
    case FP16:
      return launch_cast<Tin, __half>(batch, n, m, X, scale, Xc, ldc, sc, s);
    default:
      return launch_cast<Tin, __nv_bfloat16>(batch, n, m, X, scale, Xc, ldc, sc, s);
  }
}

}  // namespace

int rows_sumsq(int batch, int n, int m, Mat X, float* rowsq, int* status, cudaStream_t s) {
  if (batch <= 0 || n <= 0) return DION3_OK;
  switch (X.dtype) {
    case FP32:
      return launch_sumsq<float>(batch, n, m, X, rowsq, status, s);
    case FP16:
      return launch_sumsq<__half>(batch, n, m, X, rowsq, status, s);
    default:
      return launch_sumsq<__nv_bfloat16>(batch, n, m, X, rowsq, status, s);
  }
}

int scaled_cast(int batch, int n, int m, Mat X, const float* scale, void* Xc, int64_t ldc, int64_t sc, int cdt,
                cudaStream_t s) {
  if (batch <= 0 || n <= 0) return DION3_OK;
  switch (X.dtype) {
    case FP32:
      return cast_out<float>(batch, n, m, X, scale, Xc, ldc, sc, cdt, s);
    case FP16:
      return cast_out<__half>(batch, n, m, X, scale, Xc, ldc, sc, cdt, s);
    default:
      return cast_out<__nv_bfloat16>(batch, n, m, X, scale, Xc, ldc, sc, cdt, s);
  }
}

int finalize_scale(int batch, int rows, const float* rowsq, float eps, float* scale, float* alpha2, int* status,
                   cudaStream_t s) {
  if (batch <= 0) return DION3_OK;
  finalize_scale_kernel<<<(batch + 127) / 128, 128, 0, s>>>(batch, rows, rowsq, eps, scale, alpha2, status);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

}  // namespace dion3
