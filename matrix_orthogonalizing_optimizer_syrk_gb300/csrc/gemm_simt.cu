// fp32 GEMMs on FFMA for the fp32 compute mode (true fp32, no TF32).
//
// Same three epilogues as the tensor-core path (symmetric lower-triangle + mirror, general,
// fused W row update).  256 threads per CTA compute a TS x TS output tile (TS = 64, or 32 when
// 64-wide tiles would leave most SMs idle); K advances 32 at a time through double-buffered
// shared memory, the next K block being loaded into registers while the current one is used,
// so global-load latency is hidden behind the FMAs.  This path serves the 1e-4 parity mode;
// the 16-bit path is the fast one.
#include "dev_common.cuh"
#include "internal.h"

namespace dion3 {
namespace {

constexpr int TK = 32;
constexpr int NT = 256;

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
  const float* eta_dev;
  double eta_scale;
  int* status;
  int check_finite;  // last product: flag non-finite stored values (DION3_DEV_NONFINITE)
};

template <int TS, bool B_MN, int EPI>
__global__ void __launch_bounds__(NT) simt_gemm_kernel(const SParams p) {
  constexpr int R = TS / 16;           // outputs per thread along each dimension
  constexpr int LD = TS * TK / NT;     // elements of each operand a thread loads per K block
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
  __shared__ float As[2][TK][TS + 4];
  __shared__ float Bs[2][TK][TS + 4];
  const float* A = p.A + static_cast<long long>(b) * p.sA;
  const float* B = p.B + static_cast<long long>(b) * p.sB;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[R][R] = {};
  float ra[LD], rb[LD];

  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < LD; ++q) {
      const int e = threadIdx.x + q * NT;
      const int rr = e / TK, kk = e % TK;  // A: K fastest (contiguous in memory)
      const int gr = mi * TS + rr, gk = k0 + kk;
      ra[q] = (gr < p.M && gk < p.K) ? A[static_cast<long long>(gr) * p.lda + gk] : 0.f;
      if (!B_MN) {
        const int gc = nj * TS + rr;
        rb[q] = (gc < p.N && gk < p.K) ? B[static_cast<long long>(gc) * p.ldb + gk] : 0.f;
      } else {
        const int kk2 = e / TS, cc = e % TS;  // B stored K x N: N fastest
        const int gc = nj * TS + cc, gk2 = k0 + kk2;
        rb[q] = (gc < p.N && gk2 < p.K) ? B[static_cast<long long>(gk2) * p.ldb + gc] : 0.f;
      }
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int q = 0; q < LD; ++q) {
      const int e = threadIdx.x + q * NT;
      As[buf][e % TK][e / TK] = ra[q];
      if (!B_MN)
        Bs[buf][e % TK][e / TK] = rb[q];
      else
        Bs[buf][e / TS][e % TS] = rb[q];
    }
  };

  const int nkb = (p.K + TK - 1) / TK;
  if (nkb > 0) {
    load(0);
    stash(0);
  }
  __syncthreads();
  for (int kb = 0; kb < nkb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < nkb) load((kb + 1) * TK);
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[R], bb[R];
#pragma unroll
      for (int i = 0; i < R; ++i) a[i] = As[buf][kk][ty * R + i];
#pragma unroll
      for (int j = 0; j < R; ++j) bb[j] = Bs[buf][kk][tx * R + j];
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < R; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    if (kb + 1 < nkb) stash(buf ^ 1);
    __syncthreads();
  }
  const float alpha = p.eta_dev ? __double2float_rn(-__dmul_rn(static_cast<double>(*p.eta_dev), p.eta_scale)) : p.alpha;
  const float ab = alpha * (p.alpha_batch ? p.alpha_batch[b] : 1.f);
  bool bad = false;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int r = mi * TS + ty * R + i;
    if (r >= p.M) continue;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int c = nj * TS + tx * R + j;
      if (c >= p.N) continue;
      float v = acc[i][j] * ab;
      if (EPI == EPI_SYM) {
        if (c > r) continue;
        float* D = p.D + static_cast<long long>(b) * p.sD;
        if (p.beta != 0.f)
          v = fmaf(p.beta, p.C[static_cast<long long>(b) * p.sC + static_cast<long long>(r) * p.ldc + c], v);
        if (r == c) v += p.gamma;
        D[static_cast<long long>(r) * p.ldd + c] = v;
        if (c < r) D[static_cast<long long>(c) * p.ldd + r] = v;
      } else if (EPI == EPI_GEN) {
        if (p.beta != 0.f)
          v = fmaf(p.beta, p.C[static_cast<long long>(b) * p.sC + static_cast<long long>(r) * p.ldc + c], v);
        p.D[static_cast<long long>(b) * p.sD + static_cast<long long>(r) * p.ldd + c] = v;
        bad |= !isfinite(v);
      } else {
        const int row = p.sel[static_cast<long long>(b) * p.ssel + r];
        dev::range_check(row >= -1 && row < p.w_rows, p.status);
        if (row < 0 || row >= p.w_rows) continue;
        float* w = p.W + static_cast<long long>(b) * p.sW + static_cast<long long>(row) * p.ldw + c;
        const float nw = *w + v;
        *w = nw;
        bad |= !isfinite(nw);
      }
    }
  }
  if (p.check_finite && __syncthreads_or(bad) && threadIdx.x == 0 && p.status != nullptr)
    atomicOr(p.status, DION3_DEV_NONFINITE);
}

template <int TS, bool B_MN, int EPI>
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
  p.eta_dev = g.eta_dev;
  p.eta_scale = g.eta_scale;
  p.status = g.status;
  p.check_finite = g.check_finite ? 1 : 0;
  if (g.batch > 65535) return DION3_EUNSUPPORTED;
  dim3 grid(p.tiles_per_batch, g.batch);
  simt_gemm_kernel<TS, B_MN, EPI><<<grid, NT, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

// 64-wide tiles unless they would give fewer CTAs than two per SM.
template <bool B_MN, int EPI>
int launch_sized(const GemmCall& g, cudaStream_t s) {
  const long long t64m = (g.M + 63) / 64, t64n = (g.N + 63) / 64;
  const long long tiles64 = (EPI == EPI_SYM ? t64m * (t64m + 1) / 2 : t64m * t64n) * g.batch;
  if (tiles64 < 2LL * sm_count()) return launch<32, B_MN, EPI>(g, s);
  return launch<64, B_MN, EPI>(g, s);
}

}  // namespace

int gemm_simt(const GemmCall& g, cudaStream_t s) {
  if (g.batch <= 0 || g.M <= 0 || g.N <= 0) return DION3_OK;
  if (g.D.dtype != FP32 && g.epi != EPI_WUPD) return DION3_EUNSUPPORTED;
  switch (g.epi) {
    case EPI_SYM:
      return launch_sized<false, EPI_SYM>(g, s);
    case EPI_GEN:
      return launch_sized<true, EPI_GEN>(g, s);
    case EPI_WUPD:
      return launch_sized<true, EPI_WUPD>(g, s);
    default:
      return DION3_EINVAL;
  }
}

}  // namespace dion3
