// fp32 GEMMs on FFMA for the fp32 compute mode (true fp32, no TF32).
//
// Same three epilogues as the tensor-core path (symmetric lower-triangle + mirror,
// general, fused W row update), 64 x 64 output tiles, 256 threads, 4 x 4 outputs per
// thread, K staged through shared memory 16 at a time.  This path exists for the
// 1e-4 parity mode on small matrices; the 16-bit path is the fast one.
#include "internal.h"

namespace dion3 {
namespace {

constexpr int TS = 64;
constexpr int TK = 16;

struct SParams {
  int M, N, K;
  int tiles_m, tiles_n, tiles_per_batch;
  const float* A;
  long long lda, sA;
  const float* B;
  long long ldb, sB;
  float* D;
  long long ldd, sD;
  const float* C;
  long long ldc, sC;
  float beta, alpha, gamma;
  const float* alpha_batch;
  float* W;
  long long ldw, sW;
  const int* sel;
  long long ssel;
  int w_rows;
};

template <bool B_MN, int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const SParams p) {
  const int b = blockIdx.y;
  int mi, nj;
  int t = blockIdx.x;
  if (EPI == EPI_SYM) {
    int row = 0;
    while (t >= row + 1) {
      t -= row + 1;
      ++row;
    }
    mi = row;
    nj = t;
  } else {
    mi = t % p.tiles_m;
    nj = t / p.tiles_m;
  }
  __shared__ float As[TK][TS + 4];
  __shared__ float Bs[TK][TS + 4];
  const float* A = p.A + static_cast<long long>(b) * p.sA;
  const float* B = p.B + static_cast<long long>(b) * p.sB;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < p.K; k0 += TK) {
    for (int e = threadIdx.x; e < TS * TK; e += 256) {
      const int rr = e / TK, kk = e % TK;
      const int gr = mi * TS + rr, gk = k0 + kk;
      As[kk][rr] = (gr < p.M && gk < p.K) ? A[static_cast<long long>(gr) * p.lda + gk] : 0.f;
    }
    if (!B_MN) {
      for (int e = threadIdx.x; e < TS * TK; e += 256) {
        const int cc = e / TK, kk = e % TK;
        const int gc = nj * TS + cc, gk = k0 + kk;
        Bs[kk][cc] = (gc < p.N && gk < p.K) ? B[static_cast<long long>(gc) * p.ldb + gk] : 0.f;
      }
    } else {
      for (int e = threadIdx.x; e < TS * TK; e += 256) {
        const int kk = e / TS, cc = e % TS;
        const int gc = nj * TS + cc, gk = k0 + kk;
        Bs[kk][cc] = (gc < p.N && gk < p.K) ? B[static_cast<long long>(gk) * p.ldb + gc] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], bb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bb[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
  const float ab = p.alpha * (p.alpha_batch ? p.alpha_batch[b] : 1.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = mi * TS + ty * 4 + i;
    if (r >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = nj * TS + tx * 4 + j;
      if (c >= p.N) continue;
      float v = acc[i][j] * ab;
      if (EPI == EPI_SYM) {
        if (c > r) continue;
        float* D = p.D + static_cast<long long>(b) * p.sD;
        if (p.beta != 0.f) v = fmaf(p.beta, p.C[static_cast<long long>(b) * p.sC + static_cast<long long>(r) * p.ldc + c], v);
        if (r == c) v += p.gamma;
        D[static_cast<long long>(r) * p.ldd + c] = v;
        if (c < r) D[static_cast<long long>(c) * p.ldd + r] = v;
      } else if (EPI == EPI_GEN) {
        p.D[static_cast<long long>(b) * p.sD + static_cast<long long>(r) * p.ldd + c] = v;
      } else {
        const int row = p.sel[static_cast<long long>(b) * p.ssel + r];
        if (row < 0 || row >= p.w_rows) continue;
        p.W[static_cast<long long>(b) * p.sW + static_cast<long long>(row) * p.ldw + c] += v;
      }
    }
  }
}

template <bool B_MN, int EPI>
int launch(const GemmCall& g, cudaStream_t s) {
  SParams p{};
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.tiles_m = (g.M + TS - 1) / TS;
  p.tiles_n = (g.N + TS - 1) / TS;
  p.tiles_per_batch = EPI == EPI_SYM ? p.tiles_m * (p.tiles_m + 1) / 2 : p.tiles_m * p.tiles_n;
  p.A = static_cast<const float*>(g.A.ptr);
  p.lda = g.A.ld;
  p.sA = g.A.stride;
  p.B = static_cast<const float*>(g.B.ptr);
  p.ldb = g.B.ld;
  p.sB = g.B.stride;
  p.D = static_cast<float*>(const_cast<void*>(g.D.ptr));
  p.ldd = g.D.ld;
  p.sD = g.D.stride;
  p.C = static_cast<const float*>(g.C.ptr);
  p.ldc = g.C.ld;
  p.sC = g.C.stride;
  p.beta = g.beta;
  p.alpha = g.alpha;
  p.gamma = g.gamma;
  p.alpha_batch = g.alpha_batch;
  p.W = g.W;
  p.ldw = g.ldw;
  p.sW = g.sW;
  p.sel = g.sel;
  p.ssel = g.ssel;
  p.w_rows = g.w_rows;
  if (g.batch > 65535) return DION3_EUNSUPPORTED;
  dim3 grid(p.tiles_per_batch, g.batch);
  simt_gemm_kernel<B_MN, EPI><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

}  // namespace

int gemm_simt(const GemmCall& g, cudaStream_t s) {
  if (g.batch <= 0 || g.M <= 0 || g.N <= 0) return DION3_OK;
  if (g.D.dtype != FP32 && g.epi != EPI_WUPD) return DION3_EUNSUPPORTED;
  switch (g.epi) {
    case EPI_SYM:
      return launch<false, EPI_SYM>(g, s);
    case EPI_GEN:
      return launch<true, EPI_GEN>(g, s);
    case EPI_WUPD:
      return launch<true, EPI_WUPD>(g, s);
    default:
      return DION3_EINVAL;
  }
}

}  // namespace dion3
