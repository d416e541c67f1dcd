// The memory-bound passes of one Dion3 step ("Dion3: Full-Stack Orthogonal Updates",
// method details, Algorithm 4, and prerequisite "error feedback"):
//
//   pass A  M <- M + G (fp32, one rounding) for every row, optional W <- (1 - eta' wd) W,
//           and per-row selection keys: fp32 Kahan sums of |M_ij| (or M_ij^2) with a proven
//           error bound, stored as an interval [lo, hi] that contains the exact key.
//   pass B  per matrix: the k rows of largest exact key, ties to the lower index, written
//           ascending.  The intervals decide every row they can; rows whose interval
//           straddles the boundary are re-ranked with exact integer sums computed on the
//           device from the stored fp32 row (every fp32 value is an integer multiple of
//           2^-149, every square one of 2^-298).
//           Pass A also stores each row's sum of squares; pass B adds them up over S for the
//           Frobenius prescale, scale_b = 1 / (||M[S,:]||_F + eps).
//           With a caller-chosen S (norm_p = DION3_SELECT_GIVEN: the pages' random selection)
//           pass A computes no keys and pass B only checks S (k distinct ascending rows).
//   pass C  X_S = scale_b * M[S,:] packed in the compute dtype, and M[S,:] <- mu * M[S,:]
//           (fp32, one rounding).
// The W row update W[S,:] -= eta' O is fused into the last GEMM's epilogue (gemm_tc.cu).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>

#include "dev_common.cuh"
#include "internal.h"

namespace dion3 {
namespace {

constexpr int SEL_THREADS = 1024;
constexpr int MAX_N = 16384;

using dev::kahan_add;

using dev::to_f;

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&g)[8]) {
  if constexpr (sizeof(T) == 2) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = to_f<T>(h[i]);
  } else {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
    g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
  }
}

struct AArgs {
  long long rows;
  int m;
  float* M;
  const void* G;
  float* W;
  float w_decay;
  bool decay;
  const float* hyper;  // device {mu, eta, wd}: w_decay = 1 - double(eta) eta_scale double(wd)
  double eta_scale;
  bool keys;
  float* key_lo;
  float* key_hi;
  float* rowsq;
  int* status;
  const uint8_t* carry;  // [rows]: nonzero where an earlier step's decay of the row is pending
  float carry_mu;
  const float* carry_mu_dev;  // when set (and carry is), the pending factor is read from here
};

// ------------------------------------------------------------------------------ pass A
template <typename TG, int NORM_P, bool VEC>
__global__ void __launch_bounds__(256) momentum_keys_kernel(const AArgs a) {
  const int lane = threadIdx.x & 31;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int m = a.m;
  const float w_decay =
      a.hyper ? __double2float_rn(__dsub_rn(1.0, __dmul_rn(__dmul_rn(static_cast<double>(a.hyper[1]), a.eta_scale),
                                                            static_cast<double>(a.hyper[2]))))
              : a.w_decay;
  const float cm = (a.carry != nullptr && a.carry_mu_dev != nullptr) ? *a.carry_mu_dev : a.carry_mu;
  for (long long row = w0; row < a.rows; row += nw) {
    float* Mr = a.M + row * m;
    const TG* Gr = static_cast<const TG*>(a.G) + row * m;
    float* Wr = a.W + row * m;
    float s[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
    float q2[4] = {0.f, 0.f, 0.f, 0.f};  // sums of squares for the Frobenius prescale
    bool bad = false;
    // A pending decay is applied first, rounded to fp32 on its own, so the row ends exactly as
    // if the earlier step had stored mu M and this pass then added G.
    const bool cr = a.carry != nullptr && a.carry[row] != 0;
    if constexpr (VEC) {
      for (int j = lane * 8; j < m; j += 256) {
        float g[8];
        load8<TG>(Gr + j, g);
        float4* m4 = reinterpret_cast<float4*>(Mr + j);
        float4 ma = m4[0], mb = m4[1];
        float x[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        if (cr) {
#pragma unroll
          for (int q = 0; q < 8; ++q) x[q] = __fmul_rn(cm, x[q]);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = __fadd_rn(x[q], g[q]);
        m4[0] = make_float4(x[0], x[1], x[2], x[3]);
        m4[1] = make_float4(x[4], x[5], x[6], x[7]);
        if (a.decay) {
          float4* w4 = reinterpret_cast<float4*>(Wr + j);
          float4 wa = w4[0], wb = w4[1];
          wa.x = __fmul_rn(wa.x, w_decay); wa.y = __fmul_rn(wa.y, w_decay);
          wa.z = __fmul_rn(wa.z, w_decay); wa.w = __fmul_rn(wa.w, w_decay);
          wb.x = __fmul_rn(wb.x, w_decay); wb.y = __fmul_rn(wb.y, w_decay);
          wb.z = __fmul_rn(wb.z, w_decay); wb.w = __fmul_rn(wb.w, w_decay);
          w4[0] = wa;
          w4[1] = wb;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) q2[q & 3] = fmaf(x[q], x[q], q2[q & 3]);
        if (a.keys) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            bad |= !isfinite(x[q]);
            const float t = NORM_P == 1 ? fabsf(x[q]) : __fmul_rn(x[q], x[q]);
            kahan_add(s[q & 3], c[q & 3], t);
          }
        }
      }
    } else {
      for (int j = lane; j < m; j += 32) {
        const float mv = cr ? __fmul_rn(cm, Mr[j]) : Mr[j];
        const float x = __fadd_rn(mv, to_f<TG>(Gr[j]));
        Mr[j] = x;
        q2[0] = fmaf(x, x, q2[0]);
        if (a.decay) Wr[j] = __fmul_rn(Wr[j], w_decay);
        if (a.keys) {
          bad |= !isfinite(x);
          const float t = NORM_P == 1 ? fabsf(x) : __fmul_rn(x, x);
          kahan_add(s[0], c[0], t);
        }
      }
    }
    double sq = static_cast<double>(q2[0]) + static_cast<double>(q2[1]) + static_cast<double>(q2[2]) +
                static_cast<double>(q2[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) a.rowsq[row] = static_cast<float>(sq);
    if (!a.keys) continue;
    double tot = static_cast<double>(s[0]) + static_cast<double>(s[1]) + static_cast<double>(s[2]) +
                 static_cast<double>(s[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      float lo, hi;
      if (any_bad) {
        // Non-finite momentum: flagged; the row ranks as the largest.
        if (a.status) atomicOr(a.status, DION3_DEV_NONFINITE);
        lo = hi = __int_as_float(0x7f800000);
      } else if (!isfinite(tot)) {
        // fp32 overflow of the running sum: leave the decision to the exact path.
        lo = 0.f;
        hi = __int_as_float(0x7f800000);
      } else {
        // Kahan sums of nonnegative terms are within (2u + O(N u^2)) of the exact sum; a squared
        // term adds u more; the fp64 combination of 128 partial sums adds < 2^-45.  2^-21 = 8u
        // covers all of it with room to spare; the absolute term covers gradual underflow.
        const double bound = tot * 0x1p-21 + static_cast<double>(m) * 0x1p-146;
        lo = __double2float_rd(fmax(tot - bound, 0.0));
        hi = __double2float_ru(tot + bound);
      }
      a.key_lo[row] = lo;
      a.key_hi[row] = hi;
    }
  }
}

// ------------------------------------------------------------------------------ pass B helpers
// Exclusive prefix sum over the block (blockDim.x a multiple of 32); *total gets the sum.
__device__ int block_exclusive_scan(int v, int* total, int* warp_sums) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const int prefix = (wid > 0 ? warp_sums[wid - 1] : 0) + x - v;
  *total = warp_sums[nwarps - 1];
  __syncthreads();
  return prefix;
}

// k-th largest (1-based) of n nonnegative-float bit patterns (monotone as unsigned ints).
__device__ uint32_t radix_kth_largest(const uint32_t* v, int n, int k, uint32_t* hist, int* sh) {
  uint32_t prefix = 0, mask = 0;
  int kk = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint32_t x = v[i];
      if ((x & mask) == prefix) atomicAdd(&hist[(x >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int cum = 0, d = 255;
      for (; d > 0; --d) {
        if (cum + static_cast<int>(hist[d]) >= kk) break;
        cum += static_cast<int>(hist[d]);
      }
      sh[0] = d;
      sh[1] = kk - cum;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sh[0]) << shift;
    mask |= 255u << shift;
    kk = sh[1];
    __syncthreads();
  }
  return prefix;
}

// Adds v << off (v < 2^40, off < 64) into the 128-bit value (hi, lo).
__device__ __forceinline__ void add_shifted128(uint64_t& lo, uint64_t& hi, uint64_t v, int off) {
  const uint64_t l = v << off;
  lo += l;
  hi += (off ? v >> (64 - off) : 0ull) + (lo < l ? 1ull : 0ull);
}

// The exact key of one row from its exponent buckets, written as NL little-endian 64-bit limbs
// to `out` (value * 2^149 for norm_p = 1: sum over w of bkt[w] 2^w; value * 2^298 for norm_p = 2:
// sum of bkt[w] 2^(2w) and bkt[256 + w] 2^(2w + 24)).  Warp 0 only: lane q < NL adds the
// buckets whose shift falls in [64q, 64q + 64) into 128 bits (at most 64 terms below 2^103), then
// lane 0 chains the carries.  `part` holds 2 NL words of shared memory.
template <int NORM_P, int NL>
__device__ void buckets_to_limbs(const unsigned long long* bkt, uint64_t* part, uint64_t* out) {
  const int q = threadIdx.x;
  if (q < NL) {
    uint64_t lo = 0ull, hi = 0ull;
    const int s0 = 64 * q;
    if constexpr (NORM_P == 1) {
      for (int w = s0; w < s0 + 64 && w < 256; ++w) add_shifted128(lo, hi, bkt[w], w - s0);
    } else {
      for (int w = s0 / 2; w < s0 / 2 + 32 && w < 256; ++w) add_shifted128(lo, hi, bkt[w], 2 * w - s0);
      for (int w = max(0, s0 / 2 - 12); w < s0 / 2 + 20 && w < 256; ++w)
        add_shifted128(lo, hi, bkt[256 + w], 2 * w + 24 - s0);
    }
    part[2 * q] = lo;
    part[2 * q + 1] = hi;
  }
  __syncwarp();
  if (q == 0) {
    uint64_t carry = 0ull;  // the previous window's high word plus the carry out of its limb
    for (int l = 0; l < NL; ++l) {
      const uint64_t lo = part[2 * l];
      const uint64_t v = lo + carry;
      out[l] = v;
      carry = part[2 * l + 1] + (v < lo ? 1ull : 0ull);
    }
  }
}

// Digit p (most significant first, 8 bits each) of the unique sort key (exact key, 0xFFFF - row)
// of ambiguous entry j: the NL limbs of the key, then two digits of the inverted row index, so
// that equal keys rank the lower row first.
template <int NL>
__device__ __forceinline__ uint32_t rank_digit(const uint64_t* ex, int j, int row, int p) {
  if (p < NL * 8) {
    const uint64_t limb = ex[static_cast<long long>(j) * NL + (NL - 1 - p / 8)];
    return static_cast<uint32_t>(limb >> (56 - 8 * (p % 8))) & 255u;
  }
  const uint32_t inv = 0xFFFFu - static_cast<uint32_t>(row);
  return p == NL * 8 ? (inv >> 8) & 255u : inv & 255u;
}

template <int NL>
__device__ __forceinline__ int limbs_cmp(const uint64_t* a, const uint64_t* b) {
  for (int q = NL - 1; q >= 0; --q) {
    if (a[q] != b[q]) return a[q] > b[q] ? 1 : -1;
  }
  return 0;
}

struct BArgs {
  int n, m, k;
  const float* M;
  long long kstride, estride;  // key i's vector: M + b*n*m + i*kstride, entries estride apart
  const float* key_lo;
  const float* key_hi;
  uint64_t* exact;
  int32_t* sel;
  const float* rowsq;
  float* scale;
  float eps;
  int* status;
};

// scale[b] = 1 / (sqrt(sum of rowsq over the selected rows) + eps), summed in a fixed order by
// warp 0 (lane l takes entries l, l+32, ...; then a fixed shuffle tree).
__device__ void selected_scale(const BArgs& a, int b, const int32_t* sel) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const float* rq = a.rowsq + static_cast<long long>(b) * a.n;
  double acc = 0.0;
  for (int j = lane; j < a.k; j += 32) {
    const int i = sel[j];
    dev::range_check(i >= -1 && i < a.n, a.status);
    if (i >= 0 && i < a.n) acc += static_cast<double>(rq[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    if (!isfinite(acc) && a.status) atomicOr(a.status, DION3_DEV_NONFINITE);
    a.scale[b] = static_cast<float>(1.0 / (sqrt(acc) + static_cast<double>(a.eps)));
  }
}

// ------------------------------------------------------------------------------ pass B
// THREADS = 256 (n <= 2048: many small matrices, e.g. MoE experts) is bounded to 32 registers so
// that eight CTAs share an SM; THREADS = 1024 runs one large matrix per CTA.
template <int NORM_P, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS == 256 ? 8 : 1) select_kernel(const BArgs a) {
  constexpr int NL = NORM_P == 1 ? 5 : 9;
  constexpr int NB = NORM_P == 1 ? 256 : 512;
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ uint32_t hist[256];
  __shared__ unsigned long long bkt[NB];
  __shared__ int warp_sums[32];
  __shared__ int sh[4];
  __shared__ int s_bad;
  __shared__ uint64_t s_part[2 * NL];

  const int b = blockIdx.x, n = a.n, k = a.k, tid = threadIdx.x, bd = blockDim.x;
  int32_t* sel = a.sel + static_cast<long long>(b) * k;
  if (k >= n) {
    for (int i = tid; i < n; i += bd) sel[i] = i;
    __syncthreads();
    selected_scale(a, b, sel);
    return;
  }
  if (k <= 0) return;
  uint32_t* lo = reinterpret_cast<uint32_t*>(sm);
  uint32_t* hi = lo + n;
  uint16_t* amb = reinterpret_cast<uint16_t*>(hi + n);
  uint8_t* flag = reinterpret_cast<uint8_t*>(amb + ((n + 1) & ~1));
  const float* klo = a.key_lo + static_cast<long long>(b) * n;
  const float* khi = a.key_hi + static_cast<long long>(b) * n;
  for (int i = tid; i < n; i += bd) {
    lo[i] = __float_as_uint(klo[i]);
    hi[i] = __float_as_uint(khi[i]);
  }
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // At least k rows have exact key >= L; at most k rows have hi > H.
  const uint32_t L = radix_kth_largest(lo, n, k, hist, sh);
  const uint32_t H = radix_kth_largest(hi, n, k + 1, hist, sh);
  for (int i = tid; i < n; i += bd) flag[i] = lo[i] > H ? 1 : (hi[i] < L ? 0 : 2);
  __syncthreads();

  const int chunk = (n + bd - 1) / bd;
  const int i0 = min(n, tid * chunk), i1 = min(n, i0 + chunk);
  int c_in = 0, c_amb = 0;
  for (int i = i0; i < i1; ++i) {
    c_in += flag[i] == 1;
    c_amb += flag[i] == 2;
  }
  int tot_in, tot_amb;
  block_exclusive_scan(c_in, &tot_in, warp_sums);
  int pos = block_exclusive_scan(c_amb, &tot_amb, warp_sums);
  for (int i = i0; i < i1; ++i)
    if (flag[i] == 2) amb[pos++] = static_cast<uint16_t>(i);
  __syncthreads();

  int r = k - tot_in;
  if (r < 0 || r > tot_amb) {
    if (tid == 0 && a.status) atomicOr(a.status, DION3_DEV_SELECT);
    r = r < 0 ? 0 : tot_amb;
  }
  if (r > 0 && r < tot_amb) {
    uint64_t* ex = a.exact + static_cast<long long>(b) * n * NL;
    for (int j = 0; j < tot_amb; ++j) {
      const int row = amb[j];
      for (int q = tid; q < NB; q += bd) bkt[q] = 0ull;
      __syncthreads();
      const uint32_t* src =
          reinterpret_cast<const uint32_t*>(a.M + static_cast<long long>(b) * n * a.m + row * a.kstride);
      // Four loads in flight per thread; lanes past the row's end contribute zero.
      for (int base = 0; base < a.m; base += 4 * bd) {
        uint32_t bits4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = base + u * bd + tid;
          bits4[u] = e < a.m ? src[e * a.estride] : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t bits = bits4[u];
          const uint32_t e8 = (bits >> 23) & 255u;
          uint32_t mant = (bits & 0x7FFFFFu) | (e8 ? 0x800000u : 0u);
          if (e8 == 255u) {
            s_bad = 1;
            mant = 0;
          }
          const uint32_t w = e8 ? e8 - 1u : 0u;
          const unsigned grp = __match_any_sync(0xffffffffu, w);
          const bool leader = (threadIdx.x & 31) == (__ffs(grp) - 1);
          if constexpr (NORM_P == 1) {
            const unsigned sum = __reduce_add_sync(grp, mant);
            if (leader && sum) atomicAdd(&bkt[w], static_cast<unsigned long long>(sum));
          } else {
            const uint64_t sq = static_cast<uint64_t>(mant) * mant;
            const unsigned l24 = static_cast<unsigned>(sq & 0xFFFFFFull);
            const unsigned h24 = static_cast<unsigned>(sq >> 24);
            const unsigned sl = __reduce_add_sync(grp, l24);
            const unsigned shh = __reduce_add_sync(grp, h24);
            if (leader) {
              if (sl) atomicAdd(&bkt[w], static_cast<unsigned long long>(sl));
              if (shh) atomicAdd(&bkt[256 + w], static_cast<unsigned long long>(shh));
            }
          }
        }
      }
      __syncthreads();
      uint64_t* exj = ex + static_cast<long long>(j) * NL;
      if (s_bad) {
        if (tid < NL) exj[tid] = ~0ull;
        if (tid == 0 && a.status) atomicOr(a.status, DION3_DEV_NONFINITE);
      } else if (tid < 32) {
        buckets_to_limbs<NORM_P, NL>(bkt, s_part, exj);
      }
      __syncthreads();
      if (tid == 0) s_bad = 0;  // every thread has read it; the next row's barrier follows
    }
    if (tot_amb <= bd) {
      // Few ambiguous rows: each thread ranks one against all others.
      for (int j = tid; j < tot_amb; j += bd) {
        const uint64_t* kj = ex + static_cast<long long>(j) * NL;
        const int ij = amb[j];
        int rank = 0;
        for (int q = 0; q < tot_amb; ++q) {
          if (q == j) continue;
          const int cmp = limbs_cmp<NL>(ex + static_cast<long long>(q) * NL, kj);
          if (cmp > 0 || (cmp == 0 && amb[q] < ij)) ++rank;
        }
        flag[ij] = rank < r ? 1 : 0;
      }
    } else {
      // Many (ties, e.g. rows that are permutations of one another): MSB-first radix select of
      // the r largest unique sort keys (exact key, 0xFFFF - row).  Candidates keep flag 2; each
      // digit marks those above the r-th candidate's digit in (1) and those below out (0).
      // Invariant: at least rr candidates remain, and rr of them are still to be taken.
      int rr = r;
      for (int p = 0; p < NL * 8 + 2; ++p) {
        for (int q = tid; q < 256; q += bd) hist[q] = 0;
        __syncthreads();
        for (int j = tid; j < tot_amb; j += bd) {
          const int row = amb[j];
          if (flag[row] == 2) atomicAdd(&hist[rank_digit<NL>(ex, j, row, p)], 1u);
        }
        __syncthreads();
        if (tid == 0) {
          int cum = 0, d = 255;
          for (; d > 0; --d) {
            if (cum + static_cast<int>(hist[d]) >= rr) break;
            cum += static_cast<int>(hist[d]);
          }
          sh[0] = d;
          sh[1] = rr - cum;
          sh[2] = static_cast<int>(hist[d]);
        }
        __syncthreads();
        const uint32_t d = static_cast<uint32_t>(sh[0]);
        for (int j = tid; j < tot_amb; j += bd) {
          const int row = amb[j];
          if (flag[row] != 2) continue;
          const uint32_t dj = rank_digit<NL>(ex, j, row, p);
          if (dj != d) flag[row] = dj > d ? 1 : 0;
        }
        rr = sh[1];
        const bool done = sh[2] == rr;  // every remaining candidate is taken
        __syncthreads();
        if (done) break;
      }
      // The keys are unique, so the loop ends with exactly rr candidates left, all taken.
      for (int j = tid; j < tot_amb; j += bd)
        if (flag[amb[j]] == 2) flag[amb[j]] = 1;
    }
  } else {
    for (int j = tid; j < tot_amb; j += bd) flag[amb[j]] = (r == tot_amb) ? 1 : 0;
  }
  __syncthreads();

  int c_sel = 0;
  for (int i = i0; i < i1; ++i) c_sel += flag[i] == 1;
  int tot_sel;
  int p = block_exclusive_scan(c_sel, &tot_sel, warp_sums);
  for (int i = i0; i < i1; ++i)
    if (flag[i] == 1 && p < k) sel[p++] = i;
  // Never leave an entry unwritten: consumers skip rows outside [0, n).
  for (int q = tot_sel + tid; q < k; q += bd) sel[q] = -1;
  if (tid == 0 && tot_sel != k && a.status) atomicOr(a.status, DION3_DEV_SELECT);
  __syncthreads();
  selected_scale(a, b, sel);
}

// Pass B for a caller-chosen S: sel[b] must hold k strictly ascending rows in [0, n).  A set
// that breaks this is flagged (DION3_DEV_SELECT) and replaced by -1 entries, so that no row
// of W or M is touched for that matrix.
__global__ void __launch_bounds__(256) given_kernel(const BArgs a) {
  const int b = blockIdx.x;
  int32_t* sel = a.sel + static_cast<long long>(b) * a.k;
  int bad = 0;
  for (int j = threadIdx.x; j < a.k; j += blockDim.x) {
    const int i = sel[j];
    bad |= i < 0 || i >= a.n || (j > 0 && sel[j - 1] >= i);
  }
  if (__syncthreads_or(bad)) {
    for (int j = threadIdx.x; j < a.k; j += blockDim.x) sel[j] = -1;
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, DION3_DEV_SELECT);
  }
  __syncthreads();
  selected_scale(a, b, sel);
}

// ------------------------------------------------------------------------------ pass C
struct CArgs {
  int n, m, k;
  long long rows;  // batch * k
  float* M;
  const int32_t* sel;
  void* XS;
  long long ldx;
  float mu;
  const float* mu_dev;  // when set, mu is read from here
  const float* scale;
  float* mu_out;  // when set, the mu of this step is stored here (a decay left pending)
  int* status;
};

template <typename T>
__device__ __forceinline__ T cvt_out(float v);
template <>
__device__ __forceinline__ float cvt_out<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <>
__device__ __forceinline__ __half cvt_out<__half>(float v) { return __float2half_rn(v); }

// WRITE_M = false leaves M[S,:] as it is: its decay is carried to a later pass.
template <typename TC, bool VEC, bool WRITE_M>
__global__ void __launch_bounds__(256) gather_kernel(const CArgs a) {
  const int lane = threadIdx.x & 31;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const float mu = a.mu_dev ? *a.mu_dev : a.mu;
  if (a.mu_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.mu_out = mu;
  for (long long row = w0; row < a.rows; row += nw) {
    const long long b = row / a.k;
    const int i = a.sel[row];
    TC* dst = static_cast<TC*>(a.XS) + row * a.ldx;
    dev::range_check(i >= -1 && i < a.n, a.status);  // -1: the blank left by a failed selection
    if (i < 0 || i >= a.n) {  // only after a failed selection (DION3_DEV_SELECT is set)
      for (int c = lane; c < a.m; c += 32) dst[c] = cvt_out<TC>(0.f);
      continue;
    }
    float* src = a.M + (b * a.n + i) * a.m;
    const float f = a.scale[b];
    if constexpr (VEC) {
      // Four 16-byte loads per lane are issued before any store, so each warp keeps 2 KB of the
      // row in flight.
      auto put = [&](int c, const float4& x) {
        if constexpr (sizeof(TC) == 2) {
          TC o[4] = {cvt_out<TC>(x.x * f), cvt_out<TC>(x.y * f), cvt_out<TC>(x.z * f), cvt_out<TC>(x.w * f)};
          *reinterpret_cast<uint2*>(dst + c) = *reinterpret_cast<const uint2*>(o);
        } else {
          *reinterpret_cast<float4*>(dst + c) = make_float4(x.x * f, x.y * f, x.z * f, x.w * f);
        }
        if constexpr (WRITE_M)
          *reinterpret_cast<float4*>(src + c) =
              make_float4(__fmul_rn(mu, x.x), __fmul_rn(mu, x.y), __fmul_rn(mu, x.z), __fmul_rn(mu, x.w));
      };
      int c = lane * 4;
      for (; c + 384 < a.m; c += 512) {
        float4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = *reinterpret_cast<const float4*>(src + c + 128 * u);
#pragma unroll
        for (int u = 0; u < 4; ++u) put(c + 128 * u, x[u]);
      }
      for (; c < a.m; c += 128) put(c, *reinterpret_cast<const float4*>(src + c));
    } else {
      for (int c = lane; c < a.m; c += 32) {
        const float x = src[c];
        dst[c] = cvt_out<TC>(x * f);
        if constexpr (WRITE_M) src[c] = __fmul_rn(mu, x);
      }
    }
  }
}

template <typename TG, int NORM_P>
int launch_a(const AArgs& a, bool vec, cudaStream_t s) {
  long long blocks = (a.rows + 7) / 8;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (vec)
    momentum_keys_kernel<TG, NORM_P, true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  else
    momentum_keys_kernel<TG, NORM_P, false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

template <typename TG>
int launch_a_p(const AArgs& a, int norm_p, bool vec, cudaStream_t s) {
  return norm_p == 2 ? launch_a<TG, 2>(a, vec, s) : launch_a<TG, 1>(a, vec, s);  // no keys: a.keys is off
}

template <typename TC>
int launch_c(const CArgs& c, bool vec, bool write_m, cudaStream_t s) {
  long long blocks = (c.rows + 7) / 8;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) return DION3_OK;
  const unsigned g = static_cast<unsigned>(blocks);
  if (vec && write_m)
    gather_kernel<TC, true, true><<<g, 256, 0, s>>>(c);
  else if (vec)
    gather_kernel<TC, true, false><<<g, 256, 0, s>>>(c);
  else if (write_m)
    gather_kernel<TC, false, true><<<g, 256, 0, s>>>(c);
  else
    gather_kernel<TC, false, false><<<g, 256, 0, s>>>(c);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

// Carried decay, flag pass: flag[b][i] = 1 for the listed rows of matrix b, 0 elsewhere.  One CTA
// per matrix; entries outside [0, n) (the -1 of a failed selection) list nothing.
__global__ void __launch_bounds__(256) carry_flags_kernel(int n, int k, const int32_t* rows, uint8_t* flag,
                                                          int* status) {
  const int b = blockIdx.x;
  uint8_t* f = flag + static_cast<long long>(b) * n;
  for (int i = threadIdx.x; i < n; i += blockDim.x) f[i] = 0;
  __syncthreads();
  const int32_t* r = rows + static_cast<long long>(b) * k;
  for (int j = threadIdx.x; j < k; j += blockDim.x) {
    const int i = r[j];
    dev::range_check(i >= -1 && i < n, status);
    if (i >= 0 && i < n) f[i] = 1;
  }
}

// Explicit decay: M[b][rows[b][j]][:] <- mu M[...] (one fp32 rounding), one warp per listed row;
// entries outside [0, n) are skipped.
template <bool VEC>
__global__ void __launch_bounds__(256) decay_rows_kernel(int n, int m, int k, long long nrows, float* M,
                                                         const int32_t* rows, float mu) {
  const int lane = threadIdx.x & 31;
  const long long w0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long r = w0; r < nrows; r += nw) {
    const long long b = r / k;
    const int i = rows[r];
    if (i < 0 || i >= n) continue;
    float* p = M + (b * n + i) * m;
    if constexpr (VEC) {
      for (int c = lane * 4; c < m; c += 128) {
        float4 x = *reinterpret_cast<const float4*>(p + c);
        x = make_float4(__fmul_rn(mu, x.x), __fmul_rn(mu, x.y), __fmul_rn(mu, x.z), __fmul_rn(mu, x.w));
        *reinterpret_cast<float4*>(p + c) = x;
      }
    } else {
      for (int c = lane; c < m; c += 32) p[c] = __fmul_rn(mu, p[c]);
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int step_exact_limbs(int norm_p) { return norm_p == 1 ? 5 : (norm_p == 2 ? 9 : 0); }

int step_momentum_keys(const StepArgs& s, cudaStream_t st) {
  AArgs a{};
  a.rows = static_cast<long long>(s.batch) * s.n;
  a.m = s.m;
  a.M = s.M;
  a.G = s.G;
  a.W = s.W;
  a.w_decay = s.w_decay;
  a.decay = s.decay;
  a.hyper = s.hyper;
  a.eta_scale = s.eta_scale;
  a.keys = s.norm_p != DION3_SELECT_GIVEN && s.k < s.n;
  a.key_lo = s.key_lo;
  a.key_hi = s.key_hi;
  a.rowsq = s.rowsq;
  a.status = s.status;
  a.carry = s.carry_rows != nullptr ? s.carry_flag : nullptr;
  a.carry_mu = s.carry_mu;
  a.carry_mu_dev = s.carry_mu_dev;
  if (a.rows == 0) return DION3_OK;
  if (a.carry != nullptr) {
    carry_flags_kernel<<<s.batch, 256, 0, st>>>(s.n, s.k, s.carry_rows, s.carry_flag, s.status);
    if (cudaGetLastError() != cudaSuccess) return DION3_ECUDA;
  }
  const bool vec = (s.m % 8 == 0) && aligned16(s.M) && aligned16(s.G) && aligned16(s.W);
  switch (s.g_dtype) {
    case FP32:
      return launch_a_p<float>(a, s.norm_p, vec, st);
    case FP16:
      return launch_a_p<__half>(a, s.norm_p, vec, st);
    default:
      return launch_a_p<__nv_bfloat16>(a, s.norm_p, vec, st);
  }
}

int step_select(const StepArgs& s, cudaStream_t st) {
  if (s.batch <= 0 || s.n <= 0) return DION3_OK;
  if (s.n > MAX_N) return DION3_EUNSUPPORTED;
  BArgs a{};
  a.n = s.n;
  a.m = s.m;
  a.k = s.k;
  a.M = s.M;
  a.key_lo = s.key_lo;
  a.key_hi = s.key_hi;
  a.exact = s.exact;
  a.sel = s.sel;
  a.rowsq = s.rowsq;
  a.scale = s.scale;
  a.eps = s.eps;
  a.status = s.status;
  a.kstride = s.cols ? 1 : s.m;
  a.estride = s.cols ? s.n : 1;
  if (s.norm_p == DION3_SELECT_GIVEN) {
    if (s.k <= 0) return DION3_OK;
    given_kernel<<<s.batch, 256, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
  }
  const int smem = 11 * s.n + 16;
  // One CTA per matrix; small matrices (many of them, e.g. MoE experts) get 256 threads so that
  // several CTAs share an SM.
  auto launch = [&](auto kern, int threads) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
    kern<<<s.batch, threads, smem, st>>>(a);
    return true;
  };
  bool ok;
  if (s.n <= 2048)
    ok = s.norm_p == 1 ? launch(select_kernel<1, 256>, 256) : launch(select_kernel<2, 256>, 256);
  else
    ok = s.norm_p == 1 ? launch(select_kernel<1, SEL_THREADS>, SEL_THREADS)
                       : launch(select_kernel<2, SEL_THREADS>, SEL_THREADS);
  if (!ok) return DION3_ECUDA;
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

int step_gather(const StepArgs& s, cudaStream_t st) {
  CArgs c{};
  c.n = s.n;
  c.m = s.m;
  c.k = s.k;
  c.rows = static_cast<long long>(s.batch) * s.k;
  c.M = s.M;
  c.sel = s.sel;
  c.XS = s.XS;
  c.ldx = s.ldx;
  c.mu = s.mu;
  c.mu_dev = s.hyper;
  c.scale = s.scale;
  c.mu_out = s.defer ? s.carry_mu_dev : nullptr;
  c.status = s.status;
  const bool vec = (s.m % 4 == 0) && aligned16(s.M) && (s.ldx % 8 == 0);
  switch (s.cdt) {
    case FP32:
      return launch_c<float>(c, vec, !s.defer, st);
    case FP16:
      return launch_c<__half>(c, vec, !s.defer, st);
    default:
      return launch_c<__nv_bfloat16>(c, vec, !s.defer, st);
  }
}

int step_decay_rows(int batch, int n, int m, int k, float* M, const int32_t* rows, float mu, cudaStream_t st) {
  const long long nrows = static_cast<long long>(batch) * k;
  if (nrows == 0 || m == 0) return DION3_OK;
  long long blocks = (nrows + 7) / 8;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  const bool vec = (m % 4 == 0) && aligned16(M);
  if (vec)
    decay_rows_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, st>>>(n, m, k, nrows, M, rows, mu);
  else
    decay_rows_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, st>>>(n, m, k, nrows, M, rows, mu);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

}  // namespace dion3
