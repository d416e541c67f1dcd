// 16-bit GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA) for sm_103a.
//
// One persistent kernel template serves the three products Gram Newton-Schulz needs
// ("Dion3: Full-Stack Orthogonal Updates", method details, Algorithm 3; prerequisite
// "symmetric GEMM kernels"):
//   EPI_SYM  D = alpha*A*B^T + beta*C + gamma*I for symmetric results (X X^T, R^2 with the
//            polynomial epilogue, Q Z, R Z, (R Z) Z).  Only tiles that reach the lower
//            triangle are computed; the epilogue stores each lower element and its mirror,
//            so D[j][i] is bit-identical to D[i][j].
//   EPI_GEN  D = alpha*A*B + beta*C with B stored K x N (N contiguous, "MN-major"): Q X, and
//            the standard Newton-Schulz update X' = B X + a X.
//   EPI_WUPD like EPI_GEN, but the epilogue adds alpha*acc into W[b][sel[b][r]][:] -- the
//            Dion3 row update W[S,:] -= eta' O fused into the last product (Algorithm 4).
//
// CTA = 320 threads: warp 0 issues TMA loads, warp 1 owns TMEM and issues tcgen05.mma
// (one thread), warps 2-9 drain the accumulators.  Tiles are BM=128 rows x BN (128 or 256)
// columns, K in steps of 64 16-bit elements (one 128-byte swizzled row).  Two TMEM
// accumulators let the epilogue of one tile overlap the main loop of the next.  Every
// wait is bounded (clock64); a wait that gives up raises DION3_DEV_TIMEOUT and the CTA
// drains its in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "dev_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dion3 {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
// Warp 0 issues TMA loads, warp 1 the MMAs, eight warps drain the accumulators: two per TMEM
// lane quarter, which split each tile's 32-column chunks between them (a chunk's TMEM load,
// conversion, staging and store is a dependent chain; two warps keep two chains in flight).
template <int EPI>
constexpr int epi_warps() { return 8; }
template <int EPI>
constexpr int num_threads() { return 64 + 32 * epi_warps<EPI>(); }
constexpr long long DEFAULT_SPIN = 4000000000LL;  // clock cycles (about 2 s)

// CL = 1: one CTA computes a 128 x BN tile.  CL = 2: a CTA pair computes a 256 x BN tile with
// tcgen05.mma.cta_group::2 -- each CTA holds its 128 rows of A and half (BN / 2) of B, so
// every SM stages and reads only half of the B tile.
template <int BN, int CL, int EPI>
struct Cfg {
  static constexpr int EPIW = epi_warps<EPI>();
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (BN / CL) * BK * 2;
  // Epilogue staging per warp: two buffers of {32x32 block, its transpose} in 16 bits (stored
  // products), or one 32 x 36 fp32 block and 32 row pointers (W row update).
  static constexpr int STG_WARP = EPI == EPI_WUPD ? 5120 : 2 * 2 * 2048;
  static constexpr int STAGE_BUDGET = 232448 - EPIW * STG_WARP - 2048;  // 227 KB minus staging and barriers
  static constexpr int STAGES = (STAGE_BUDGET / (A_BYTES + B_BYTES)) < 8 ? (STAGE_BUDGET / (A_BYTES + B_BYTES)) : 8;
  static constexpr int STG_OFF = STAGES * (A_BYTES + B_BYTES);
  static constexpr int BAR_OFF = STG_OFF + EPIW * STG_WARP;
  static constexpr int NBARS = 2 * STAGES + 5;  // full, empty, tmem_full[2], tmem_empty[2], drain
  static constexpr int SMEM = BAR_OFF + NBARS * 8 + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr uint32_t TX_BYTES = CL * (A_BYTES + B_BYTES);  // what the MMA-issuing CTA waits for
};

struct KParams {
  int batch, M, N, K;
  int tiles_m, tiles_n, tiles_per_batch;
  long long total_tiles;
  int num_kb;
  uint32_t idesc;
  void* D;
  long long ldd, sD;
  int d_type;
  const void* C;
  long long ldc, sC;
  float beta;
  float alpha;
  const float* alpha_batch;
  float gamma;
  float* W;
  long long ldw, sW;
  const int* sel;
  long long ssel;
  int w_rows;
  int* status;
  long long spin_limit;
  const float* eta_dev;
  double eta_scale;
  int check_finite;  // last product: flag non-finite stored values (DION3_DEV_NONFINITE)
};

// ----------------------------------------------------------------------------- tile order
// Work unit t -> (batch b, row block mi, column block nj).  With CL = 2 the unit is a pair of
// row blocks (2q, 2q+1) sharing column block nj; CTA `rank` of the cluster takes row block
// 2q + rank.
template <int EPI, int BN, int CL>
__device__ __forceinline__ void decode_tile(const KParams& p, long long t, uint32_t rank, int& b, int& mi, int& nj) {
  b = static_cast<int>(t / p.tiles_per_batch);
  int r = static_cast<int>(t - static_cast<long long>(b) * p.tiles_per_batch);
  if constexpr (EPI == EPI_SYM) {
    if constexpr (CL == 1) {
      // Row block i holds column blocks 0 .. i*BM/BN (the blocks that reach the lower triangle).
      constexpr int RATIO = BN / BM;
      int row = 0;
      for (;;) {
        const int c = row / RATIO + 1;
        if (r < c) break;
        r -= c;
        ++row;
      }
      mi = row;
      nj = r;
    } else {
      // BN = 2 BM: row blocks 2q and 2q+1 both hold column blocks 0 .. q.
      int q = 0;
      for (;;) {
        if (r < q + 1) break;
        r -= q + 1;
        ++q;
      }
      mi = 2 * q + static_cast<int>(rank);
      nj = r;
    }
  } else {
    if constexpr (CL == 1) {
      mi = r % p.tiles_m;
      nj = r / p.tiles_m;
    } else {
      const int P = (p.tiles_m + 1) / 2;
      mi = 2 * (r % P) + static_cast<int>(rank);
      nj = r / P;
    }
  }
}

// ----------------------------------------------------------------------------- epilogue
using dev::from_f;
using dev::to_f;

// 32 consecutive values of one row, written with 16-byte stores (caller checked alignment).
template <typename T>
__device__ __forceinline__ void store_row32(T* dst, const T (&o)[32]) {
  const uint4* src = reinterpret_cast<const uint4*>(o);
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < static_cast<int>(32 * sizeof(T) / 16); ++i) d[i] = src[i];
}
template <typename T>
__device__ __forceinline__ void load_row32(const T* src, float (&v)[32]) {
  T tmp[32];
  uint4* t = reinterpret_cast<uint4*>(tmp);
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < static_cast<int>(32 * sizeof(T) / 16); ++i) t[i] = s[i];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = to_f<T>(tmp[i]);
}

__device__ __forceinline__ bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

template <typename T>
__device__ __forceinline__ void epi_sym(const KParams& p, int b, int r, int c0, float (&acc)[32]) {
  T* D = static_cast<T*>(p.D) + static_cast<long long>(b) * p.sD;
  const T* C = static_cast<const T*>(p.C) + static_cast<long long>(b) * p.sC;
  T* drow = D + static_cast<long long>(r) * p.ldd;
  const bool interior = (c0 + 31 < p.N) && (c0 + 31 < r);
  if (p.beta != 0.f) {
    const T* crow = C + static_cast<long long>(r) * p.ldc;
    if (interior && aligned16(crow + c0)) {
      float cv[32];
      load_row32<T>(crow + c0, cv);
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = fmaf(p.beta, cv[i], acc[i]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c = c0 + i;
        if (c < p.N && c <= r) acc[i] = fmaf(p.beta, to_f<T>(crow[c]), acc[i]);
      }
    }
  }
  if (p.gamma != 0.f) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c0 + i == r) acc[i] += p.gamma;
  }
  T o[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] = from_f<T>(acc[i]);
  if (interior && aligned16(drow + c0)) {
    store_row32<T>(drow + c0, o);
#pragma unroll
    for (int i = 0; i < 32; ++i) D[static_cast<long long>(c0 + i) * p.ldd + r] = o[i];
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int c = c0 + i;
      if (c < p.N && c <= r) {
        drow[c] = o[i];
        if (c < r) D[static_cast<long long>(c) * p.ldd + r] = o[i];
      }
    }
  }
}

template <typename T>
__device__ __forceinline__ void epi_gen(const KParams& p, int b, int r, int c0, float (&acc)[32]) {
  T* drow = static_cast<T*>(p.D) + static_cast<long long>(b) * p.sD + static_cast<long long>(r) * p.ldd;
  if (p.beta != 0.f) {
    const T* crow = static_cast<const T*>(p.C) + static_cast<long long>(b) * p.sC + static_cast<long long>(r) * p.ldc;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c0 + i < p.N) acc[i] = fmaf(p.beta, to_f<T>(crow[c0 + i]), acc[i]);
  }
  T o[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] = from_f<T>(acc[i]);
  if (c0 + 31 < p.N && aligned16(drow + c0)) {
    store_row32<T>(drow + c0, o);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c0 + i < p.N) drow[c0 + i] = o[i];
  }
}

__device__ __forceinline__ void epi_wupd(const KParams& p, int b, int r, int c0, const float (&acc)[32]) {
  const int row = __ldg(p.sel + static_cast<long long>(b) * p.ssel + r);
  dev::range_check(row >= -1 && row < p.w_rows, p.status);
  if (row < 0 || row >= p.w_rows) return;  // only after a failed selection
  float* wrow = p.W + static_cast<long long>(b) * p.sW + static_cast<long long>(row) * p.ldw;
  if (c0 + 31 < p.N && aligned16(wrow + c0)) {
    float4* w4 = reinterpret_cast<float4*>(wrow + c0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 w = w4[i];
      w.x += acc[4 * i + 0];
      w.y += acc[4 * i + 1];
      w.z += acc[4 * i + 2];
      w.w += acc[4 * i + 3];
      w4[i] = w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c0 + i < p.N) wrow[c0 + i] += acc[i];
  }
}

template <int EPI>
__device__ __forceinline__ void epi_dispatch(const KParams& p, int b, int r, int c0, float (&acc)[32]) {
  if constexpr (EPI == EPI_WUPD) {
    epi_wupd(p, b, r, c0, acc);
  } else {
    switch (p.d_type) {
      case FP32:
        if constexpr (EPI == EPI_SYM) epi_sym<float>(p, b, r, c0, acc); else epi_gen<float>(p, b, r, c0, acc);
        break;
      case FP16:
        if constexpr (EPI == EPI_SYM) epi_sym<__half>(p, b, r, c0, acc); else epi_gen<__half>(p, b, r, c0, acc);
        break;
      default:
        if constexpr (EPI == EPI_SYM) epi_sym<__nv_bfloat16>(p, b, r, c0, acc);
        else epi_gen<__nv_bfloat16>(p, b, r, c0, acc);
        break;
    }
  }
}

using dev::pack2;
using dev::unpack2;

// Non-finite test of 16-bit pairs by carries: (w & E) + A sets bit 15 (31) of a half-word exactly
// when its exponent bits are all ones (an infinity or a NaN), and never carries into the other
// half.  OR-ing the sums of many pairs and testing 0x80008000 once checks them all.
template <typename T>
struct NonFinite16 {
  static constexpr uint32_t E = std::is_same<T, __half>::value ? 0x7C007C00u : 0x7F807F80u;
  static constexpr uint32_t A = std::is_same<T, __half>::value ? 0x04000400u : 0x00800080u;
  static __device__ __forceinline__ uint32_t acc(uint32_t w, uint32_t keep) { return ((w & keep) & E) + (A & keep); }
};

// One lane of each warp that saw a non-finite value sets DION3_DEV_NONFINITE (warp-uniform call).
__device__ __forceinline__ void flag_nonfinite(const KParams& p, bool bad, int lane) {
  if (__any_sync(0xffffffffu, bad) && lane == 0 && p.status != nullptr) atomicOr(p.status, DION3_DEV_NONFINITE);
}

// 32 consecutive C values of row r starting at c0, packed in pairs (zeros where out of range).
template <typename T>
__device__ __forceinline__ void load_c32(const KParams& p, const T* crow, int c0, uint32_t (&w)[16]) {
  if (crow == nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = 0u;
    return;
  }
  if (c0 + 31 < p.N && aligned16(crow + c0)) {
    const uint4* s4 = reinterpret_cast<const uint4*>(crow + c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = s4[q];
      w[4 * q + 0] = u.x;
      w[4 * q + 1] = u.y;
      w[4 * q + 2] = u.z;
      w[4 * q + 3] = u.w;
    }
  } else {
    const uint16_t* c16 = reinterpret_cast<const uint16_t*>(crow);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t lo = (c0 + 2 * i < p.N) ? c16[c0 + 2 * i] : 0u;
      const uint32_t hi = (c0 + 2 * i + 1 < p.N) ? c16[c0 + 2 * i + 1] : 0u;
      w[i] = lo | (hi << 16);
    }
  }
}

// Byte offset of element (row, col) in a 32 x 32 block of 16-bit values laid out the way a
// TMA box of {32, 32} with 64-byte swizzle expects it: 64-byte rows, 16-byte units permuted
// by (row / 2) mod 4.
__device__ __forceinline__ uint32_t stg_off(int row, int col) {
  return static_cast<uint32_t>(row * 64 + ((((col >> 3) ^ (row >> 1)) & 3) << 4) + ((col & 7) << 1));
}

// Row `lane` of a staged 32 x 32 block (layout of stg_off) into D[b][row0 + lane][col0 ..], clipped
// to the matrix; used where a TMA store would write past the end of a row.  Kept out of line:
// it runs only for blocks on a ragged right edge.
__device__ __noinline__ void store_block_plain(const KParams& p, int b, const uint8_t* blk, int row0, int col0,
                                               int lane) {
  const int row = row0 + lane;
  if (row >= p.M) return;
  uint16_t* drow = static_cast<uint16_t*>(p.D) + static_cast<long long>(b) * p.sD + static_cast<long long>(row) * p.ldd;
  for (int c = col0; c < p.N && c < col0 + 32; ++c)
    drow[c] = *reinterpret_cast<const uint16_t*>(blk + stg_off(lane, c - col0));
}

// Epilogue of one tile for a 16-bit D (EPI_SYM or EPI_GEN).  Each warp owns 32 rows and every
// other 32-column chunk (its partner warp on the same TMEM lanes takes the rest); a chunk is
// converted, written into a swizzled staging block (and, for blocks below
// the diagonal, into a transposed block: lane pairs exchange halves so every shared store is a
// full word), and stored with TMA bulk stores.  A diagonal block is made exactly symmetric in
// shared memory (its upper half copied from the transposed lower half) and stored once.
// Chunks whose columns lie entirely above the warp's rows are skipped; TMA clips rows and
// columns outside the matrix, and a warp whose rows all lie outside stores nothing.
template <typename T, int BN, int EPI>
__device__ __forceinline__ void epi_tile_tma(const KParams& p, const CUtensorMap* tmD, uint8_t* stg, int& buf,
                                             uint32_t t_acc, int b, int mi, int nj, int ew, int half, int lane,
                                             float ab) {
  const int r0w = mi * BM + ew * 32;
  const int r = r0w + lane;
  const bool use_c = p.beta != 0.f;  // D = alpha acc + beta C (C has D's type and layout)
  const T* crow = nullptr;
  if (use_c && r < p.M)
    crow = static_cast<const T*>(p.C) + static_cast<long long>(b) * p.sC + static_cast<long long>(r) * p.ldc;
  int nch = 0;
  for (int ch = 0; r0w < p.M && ch < BN / 32; ++ch) {
    const int c0 = nj * BN + ch * 32;
    if (c0 >= p.N || (EPI == EPI_SYM && c0 > r0w)) break;
    ++nch;
  }
  uint32_t cnx[16];
  bool bad = false;
  if (use_c && half < nch) load_c32<T>(p, crow, nj * BN + half * 32, cnx);
#pragma unroll 1
  for (int ch = half; ch < nch; ch += 2) {
    const int c0 = nj * BN + ch * 32;
    uint32_t cw[16];
    if (use_c) {
#pragma unroll
      for (int i = 0; i < 16; ++i) cw[i] = cnx[i];
      if (ch + 2 < nch) load_c32<T>(p, crow, c0 + 64, cnx);  // prefetch this warp's next chunk of C
    }
    uint32_t v[32];
    __syncwarp();
    if (p.num_kb > 0) {
      ptx::tmem_ld_32x32b_x32(t_acc + ch * 32, v);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;
    }
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float lo = __uint_as_float(v[2 * i]) * ab;
      float hi = __uint_as_float(v[2 * i + 1]) * ab;
      if (use_c) {
        const float2 c2 = unpack2<T>(cw[i]);
        lo = fmaf(p.beta, c2.x, lo);
        hi = fmaf(p.beta, c2.y, hi);
      }
      if (EPI == EPI_SYM && p.gamma != 0.f) {
        if (c0 + 2 * i == r) lo += p.gamma;
        if (c0 + 2 * i + 1 == r) hi += p.gamma;
      }
      w[i] = pack2<T>(lo, hi);
    }
    if (p.check_finite && r < p.M) {
      uint32_t carry = 0u;
      if (c0 + 32 <= p.N) {
#pragma unroll
        for (int i = 0; i < 16; ++i) carry |= NonFinite16<T>::acc(w[i], 0xFFFFFFFFu);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t keep = c0 + 2 * i < p.N ? (c0 + 2 * i + 1 < p.N ? 0xFFFFFFFFu : 0x0000FFFFu) : 0u;
          carry |= NonFinite16<T>::acc(w[i], keep);
        }
      }
      bad |= (carry & 0x80008000u) != 0u;
    }
    const bool diag = (EPI == EPI_SYM) && (c0 == r0w);
    const bool below = (EPI == EPI_SYM) && (c0 < r0w);
    // the buffer used two chunks ago must have been read by its TMA store
    if (lane == 0) ptx::bulk_wait_read_le1();
    __syncwarp();
    uint8_t* S = stg + buf * 4096;
    uint8_t* Tt = S + 2048;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(S + lane * 64 + ((((q) ^ (lane >> 1)) & 3) << 4)) =
          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    if (diag || below) {
      const bool odd = lane & 1;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t s0 = odd ? (w[2 * j] & 0xFFFFu) : (w[2 * j] >> 16);
        const uint32_t s1 = odd ? (w[2 * j + 1] & 0xFFFFu) : (w[2 * j + 1] >> 16);
        const uint32_t rcv = __shfl_xor_sync(0xffffffffu, s0 | (s1 << 16), 1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int k = 2 * j + h;
          const uint32_t rk = h ? (rcv >> 16) : (rcv & 0xFFFFu);
          const uint32_t word = odd ? (rk | (w[k] & 0xFFFF0000u)) : ((w[k] & 0xFFFFu) | (rk << 16));
          const int c = 2 * k + (odd ? 1 : 0);
          *reinterpret_cast<uint32_t*>(Tt + c * 64 + ((((lane >> 3) ^ (c >> 1)) & 3) << 4) + (((lane >> 1) & 3) << 2)) =
              word;
        }
      }
      if (diag) {
        __syncwarp();
        for (int c = lane + 1; c < 32; ++c)
          *reinterpret_cast<uint16_t*>(S + stg_off(lane, c)) = *reinterpret_cast<const uint16_t*>(Tt + stg_off(lane, c));
      }
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    // A TMA store writes whole 16-byte units of a row, so a block whose columns run past a row
    // end that is not 16-byte aligned is written with plain stores instead (lane = block row).
    const bool ragged = (p.N & 7) != 0;
    const bool blk_plain = ragged && c0 + 32 > p.N;
    const bool tr_plain = ragged && below && r0w + 32 > p.N;
    if (lane == 0) {
      if (!blk_plain) ptx::tma_store_3d(tmD, ptx::smem_u32(S), c0, r0w, b);
      if (below && !tr_plain) ptx::tma_store_3d(tmD, ptx::smem_u32(Tt), r0w, c0, b);
      ptx::bulk_commit_group();
    }
    if (blk_plain) store_block_plain(p, b, S, r0w, c0, lane);
    if (tr_plain) store_block_plain(p, b, Tt, c0, r0w, lane);
    buf ^= 1;
  }
  if (p.check_finite) flag_nonfinite(p, bad, lane);
}

// Epilogue of the fused row update W[sel[r], :] += alpha * acc.  tcgen05.ld hands each lane one
// accumulator row; addressed that way, every warp access to W would touch 32 scattered rows.
// So each 32 x 32 chunk goes through shared memory and is read back transposed: in the global
// loads and stores, lanes 8j .. 8j+7 cover 128 contiguous bytes of one W row and a warp
// instruction covers four rows.  NHALF warps share a lane quarter and take every NHALF-th
// chunk; each runs its W loads AHEAD chunks in front of the adds and stores.  Staging per warp:
// the 32 x 36 fp32 chunk and 32 row pointers (4864 bytes).
template <bool CHECKED>
__device__ __forceinline__ void load_w_chunk(float* const (&wr)[8], int c, int N, float4 (&x)[8]) {
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const float* w = wr[it];
    if (!CHECKED) {
      x[it] = *reinterpret_cast<const float4*>(w + c);
    } else {
      x[it].x = (w && c < N) ? w[c] : 0.f;
      x[it].y = (w && c + 1 < N) ? w[c + 1] : 0.f;
      x[it].z = (w && c + 2 < N) ? w[c + 2] : 0.f;
      x[it].w = (w && c + 3 < N) ? w[c + 3] : 0.f;
    }
  }
}

template <int BN, int NHALF>
__device__ __forceinline__ void epi_tile_wupd(const KParams& p, uint8_t* stg, uint32_t t_acc, int b, int mi, int nj,
                                              int ew, int half, int lane, float ab) {
  constexpr int NCHW = BN / 32 / NHALF;  // chunks of this warp
  constexpr int AHEAD = NHALF == 1 ? 3 : 2;
  constexpr int LDT = 36;  // staged row stride in floats (16-byte aligned, conflict-free phases)
  const int r0w = mi * BM + ew * 32;
  if (r0w >= p.M) return;
  float* tile = reinterpret_cast<float*>(stg);
  float** rowp = reinterpret_cast<float**>(stg + 32 * LDT * 4);
  {
    const int r = r0w + lane;
    float* wrow = nullptr;
    if (r < p.M) {
      const int row = __ldg(p.sel + static_cast<long long>(b) * p.ssel + r);
      dev::range_check(row >= -1 && row < p.w_rows, p.status);
      if (row >= 0 && row < p.w_rows)  // only a failed selection leaves rows outside [0, w_rows)
        wrow = p.W + static_cast<long long>(b) * p.sW + static_cast<long long>(row) * p.ldw;
    }
    __syncwarp();
    rowp[lane] = wrow;
    __syncwarp();
  }
  const int sub = lane >> 3;      // row within each group of four
  const int cq = (lane & 7) * 4;  // first of this lane's four columns in a chunk
  float* wr[8];
  bool rows_ok = true;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    wr[it] = rowp[it * 4 + sub];
    rows_ok &= wr[it] != nullptr;
  }
  // Fast path: 16-byte aligned W rows, all 32 rows present; then only the chunk's columns matter.
  const bool fast = __all_sync(0xffffffffu, rows_ok) && ((p.ldw & 3) == 0) && ((p.sW & 3) == 0) && aligned16(p.W);
  float4 ring[AHEAD][8];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < AHEAD && j < NCHW; ++j) {
    const int c0 = nj * BN + (half + j * NHALF) * 32;
    if (c0 < p.N) {
      if (fast && c0 + 32 <= p.N) load_w_chunk<false>(wr, c0 + cq, p.N, ring[j]);
      else load_w_chunk<true>(wr, c0 + cq, p.N, ring[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < NCHW; ++j) {
    const int ch = half + j * NHALF;
    const int c0 = nj * BN + ch * 32;
    if (c0 < p.N) {
      float4 x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = ring[j % AHEAD][i];
      if (j + AHEAD < NCHW) {
        const int cn = c0 + AHEAD * NHALF * 32;
        if (cn < p.N) {
          if (fast && cn + 32 <= p.N) load_w_chunk<false>(wr, cn + cq, p.N, ring[j % AHEAD]);
          else load_w_chunk<true>(wr, cn + cq, p.N, ring[j % AHEAD]);
        }
      }
      uint32_t v[32];
      __syncwarp();
      if (p.num_kb > 0) {
        ptx::tmem_ld_32x32b_x32(t_acc + ch * 32, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(tile + lane * LDT + 4 * q) = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      __syncwarp();
      const int c = c0 + cq;
      const bool full_chunk = fast && c0 + 32 <= p.N;
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const float4 a = *reinterpret_cast<const float4*>(tile + (it * 4 + sub) * LDT + cq);
        float4 y = x[it];
        y.x = fmaf(a.x, ab, y.x);
        y.y = fmaf(a.y, ab, y.y);
        y.z = fmaf(a.z, ab, y.z);
        y.w = fmaf(a.w, ab, y.w);
        float* w = wr[it];
        if (full_chunk) {
          // one sum per four values; only a non-finite sum (a non-finite value, or a sum of
          // huge ones) is looked at value by value
          if (!isfinite((y.x + y.y) + (y.z + y.w)))
            bad |= !(isfinite(y.x) && isfinite(y.y) && isfinite(y.z) && isfinite(y.w));
          *reinterpret_cast<float4*>(w + c) = y;
        } else if (w != nullptr) {
          bad |= (c < p.N && !isfinite(y.x)) || (c + 1 < p.N && !isfinite(y.y)) || (c + 2 < p.N && !isfinite(y.z)) ||
                 (c + 3 < p.N && !isfinite(y.w));
          if (c < p.N) w[c] = y.x;
          if (c + 1 < p.N) w[c + 1] = y.y;
          if (c + 2 < p.N) w[c + 2] = y.z;
          if (c + 3 < p.N) w[c + 3] = y.w;
        }
      }
    }
  }
  flag_nonfinite(p, bad, lane);
}

using dev::drain_wait;

// ----------------------------------------------------------------------------- kernel
template <int BN, bool B_MN, int EPI, int CL>
__global__ void __launch_bounds__(num_threads<EPI>(), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const KParams p) {
  using Cf = Cfg<BN, CL, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + Cf::STAGES * Cf::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cf::BAR_OFF);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + Cf::NBARS);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * Cf::STAGES;
  const uint32_t tfull0 = empty0 + 8 * Cf::STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain_bar = tempty0 + 16;

  const uint32_t rank = CL == 2 ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;  // the CTA that issues the MMAs (CL = 2: the even CTA)
  const long long unit0 = blockIdx.x / CL, unit_step = gridDim.x / CL;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cf::STAGES; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull0 + 8 * a, 1);
      ptx::mbar_init(tempty0 + 8 * a, Cf::EPIW * CL);  // every epilogue warp of the pair releases it
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    if (EPI != EPI_WUPD && p.d_type != FP32) ptx::tma_prefetch_desc(&tmD);
  }
  if (warp == 1) {
    if constexpr (CL == 2) {
      ptx::tmem_alloc_pair(ptx::smem_u32(tmem_holder), Cf::TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_holder), Cf::TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (CL == 2) ptx::cluster_sync();  // both CTAs' barriers exist before either signals the other
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  volatile int* abort = abort_flag;
  const long long lim = p.spin_limit;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0, fill_parity = 0;
      bool ok = true;
      for (long long t = unit0; ok && t < p.total_tiles; t += unit_step) {
        int b, mi, nj;
        decode_tile<EPI, BN, CL>(p, t, rank, b, mi, nj);
        // the tile scheduler's invariants: a matrix of the batch, a row block of the (pair-rounded)
        // row grid, a column block of the column grid (and at or below the diagonal for SYM)
        dev::range_check(b >= 0 && b < p.batch && mi >= 0 && mi < (p.tiles_m + CL - 1) / CL * CL && nj >= 0 &&
                             nj < p.tiles_n && (EPI != EPI_SYM || nj * BN <= mi * BM + BM - 1),
                         p.status);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!ptx::mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort, lim)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t adst = ptx::smem_u32(sA + stage * Cf::A_BYTES);
          const uint32_t bdst = ptx::smem_u32(sB + stage * Cf::B_BYTES);
          if constexpr (CL == 1) {
            ptx::mbar_arrive_expect_tx(fb, Cf::TX_BYTES);
            ptx::tma_load_3d(adst, &tmA, fb, kb * BK, mi * BM, b);
            if constexpr (!B_MN) {
              ptx::tma_load_3d(bdst, &tmB, fb, kb * BK, nj * BN, b);
            } else {
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                ptx::tma_load_3d(bdst + c * (BK * 128), &tmB, fb, nj * BN + c * 64, kb * BK, b);
            }
          } else {
            // Each CTA stages its own 128 rows of A and its half of B; all the bytes of the pair
            // complete the even CTA's barrier, which the MMA issuer waits on.
            const uint32_t fb_lead = ptx::mapa_shared(fb, 0);
            if (leader) ptx::mbar_arrive_expect_tx(fb, Cf::TX_BYTES);
            ptx::tma_load_3d_pair(adst, &tmA, fb_lead, kb * BK, mi * BM, b);
            if constexpr (!B_MN) {
              ptx::tma_load_3d_pair(bdst, &tmB, fb_lead, kb * BK, nj * BN + static_cast<int>(rank) * (BN / 2), b);
            } else {
#pragma unroll
              for (int c = 0; c < BN / 128; ++c)
                ptx::tma_load_3d_pair(bdst + c * (BK * 128), &tmB, fb_lead,
                                      nj * BN + (static_cast<int>(rank) * (BN / 128) + c) * 64, kb * BK, b);
            }
          }
          filled |= 1u << stage;
          fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == Cf::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // Let every issued copy land before the CTA's shared memory is released (in a pair,
        // all copies complete the even CTA's barriers, and the final cluster barrier keeps
        // the odd CTA alive until the even one has drained).
        for (int s = 0; s < Cf::STAGES; ++s)
          if (filled & (1u << s)) drain_wait(full0 + 8 * s, (fill_parity >> s) & 1u, lim);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (long long t = unit0; ok && t < p.total_tiles; t += unit_step) {
        if (!ptx::mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1u, abort, lim)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!ptx::mbar_wait(full0 + 8 * stage, phase, abort, lim)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_base = ptx::smem_u32(sA + stage * Cf::A_BYTES);
          const uint32_t b_base = ptx::smem_u32(sB + stage * Cf::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = ptx::smem_desc_sw128(a_base + kk * 32, 16, 1024);
            uint64_t bd;
            if constexpr (!B_MN) bd = ptx::smem_desc_sw128(b_base + kk * 32, 16, 1024);
            else bd = ptx::smem_desc_sw128(b_base + kk * 16 * 128, BK * 128, 1024);
            if constexpr (CL == 2)
              ptx::tc_mma_f16_pair(d_tmem, ad, bd, p.idesc, (kb | kk) != 0 ? 1u : 0u);
            else
              ptx::tc_mma_f16(d_tmem, ad, bd, p.idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          if constexpr (CL == 2)
            ptx::tc_commit_pair_mc(empty0 + 8 * stage, 0x3);  // frees the stage in both CTAs
          else
            ptx::tc_commit(empty0 + 8 * stage);
          if (++stage == Cf::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (CL == 2)
          ptx::tc_commit_pair_mc(tfull0 + 8 * acc, 0x3);  // both CTAs' epilogues may start
        else
          ptx::tc_commit(tfull0 + 8 * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA this thread issued has completed once the drain barrier fires.
      if constexpr (CL == 2)
        ptx::tc_commit_pair(drain_bar);
      else
        ptx::tc_commit(drain_bar);
      drain_wait(drain_bar, 0, lim);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int ew = warp & 3;  // TMEM lanes 32*ew .. 32*ew+31
    const int half = (warp - 2) >> 2;  // the two warps of a lane quarter split the chunks
    uint8_t* stg = smem + Cf::STG_OFF + (warp - 2) * Cf::STG_WARP;
    int buf = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (long long t = unit0; t < p.total_tiles; t += unit_step) {
      int b, mi, nj;
      decode_tile<EPI, BN, CL>(p, t, rank, b, mi, nj);
      if (!ptx::mbar_wait(tfull0 + 8 * acc, acc_phase, abort, lim)) break;
      ptx::tc_fence_after();
      const float alpha =
          p.eta_dev ? __double2float_rn(-__dmul_rn(static_cast<double>(__ldg(p.eta_dev)), p.eta_scale)) : p.alpha;
      const float ab = alpha * (p.alpha_batch ? __ldg(p.alpha_batch + b) : 1.f);
      const int r = mi * BM + ew * 32 + lane;
      const int rmax_warp = mi * BM + ew * 32 + 31;
      const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(acc * BN);
      bool done = false;
      if constexpr (EPI == EPI_WUPD) {
        epi_tile_wupd<BN, Cf::EPIW / 4>(p, stg, t_acc, b, mi, nj, ew, half, lane, ab);
        done = true;
      } else {
        if (p.d_type != FP32) {
          if (p.d_type == FP16)
            epi_tile_tma<__half, BN, EPI>(p, &tmD, stg, buf, t_acc, b, mi, nj, ew, half, lane, ab);
          else
            epi_tile_tma<__nv_bfloat16, BN, EPI>(p, &tmD, stg, buf, t_acc, b, mi, nj, ew, half, lane, ab);
          done = true;
        }
      }
      if (!done) {
        bool bad = false;
#pragma unroll 1
        for (int ch = half; ch < BN / 32; ch += 2) {
          const int c0 = nj * BN + ch * 32;
          if (c0 >= p.N) break;
          if (EPI == EPI_SYM && c0 > rmax_warp) break;
          uint32_t v[32];
          __syncwarp();
          if (p.num_kb > 0) {
            ptx::tmem_ld_32x32b_x32(t_acc + ch * 32, v);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
          if (r < p.M) {
            float a[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = __uint_as_float(v[i]) * ab;
            epi_dispatch<EPI>(p, b, r, c0, a);
            if (p.check_finite) {
#pragma unroll
              for (int i = 0; i < 32; ++i) bad |= c0 + i < p.N && !isfinite(a[i]);
            }
          }
        }
        if (p.check_finite) flag_nonfinite(p, bad, lane);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CL == 2)
          ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty0 + 8 * acc, 0));
        else
          ptx::mbar_arrive(tempty0 + 8 * acc);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // Every TMA store of this warp has finished before the CTA (and its staging) goes away.
    if (lane == 0) ptx::bulk_wait_all();
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (CL == 2) ptx::cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (CL == 2)
      ptx::tmem_dealloc_pair(tmem_base, Cf::TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem_base, Cf::TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort && p.status) atomicOr(p.status, DION3_DEV_TIMEOUT);
}

__global__ void watchdog_kernel(long long limit, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the wait must give up on its own.
    if (!ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag, limit)) atomicOr(status, DION3_DEV_TIMEOUT);
  }
}

// ----------------------------------------------------------------------------- host side
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeFn>(nullptr);
    return reinterpret_cast<EncodeFn>(ptr);
  }();
  return fn;
}

// Encoded maps are a pure function of their arguments; a product chain encodes the same few
// again and again, so the last ones are kept (direct-mapped on a hash of the arguments).
struct MapKey {
  const void* ptr;
  int64_t ld, stride;
  int dtype, rows, cols, batch, box_cols, box_rows, swz;
};

bool same_key(const MapKey& a, const MapKey& b) {
  return a.ptr == b.ptr && a.ld == b.ld && a.stride == b.stride && a.dtype == b.dtype && a.rows == b.rows &&
         a.cols == b.cols && a.batch == b.batch && a.box_cols == b.box_cols && a.box_rows == b.box_rows &&
         a.swz == b.swz;
}

constexpr int MAP_CACHE = 256;
struct MapCache {
  std::mutex mu;
  bool used[MAP_CACHE] = {};
  MapKey key[MAP_CACHE];
  CUtensorMap map[MAP_CACHE];
};
MapCache& map_cache() {
  static MapCache c;
  return c;
}

size_t key_slot(const MapKey& k) {
  uint64_t h = 1469598103934665603ull;
  auto mix = [&](uint64_t v) { h = (h ^ v) * 1099511628211ull; };
  mix(reinterpret_cast<uintptr_t>(k.ptr));
  mix(static_cast<uint64_t>(k.ld));
  mix(static_cast<uint64_t>(k.stride));
  mix((static_cast<uint64_t>(k.rows) << 32) ^ static_cast<uint32_t>(k.cols));
  mix((static_cast<uint64_t>(k.batch) << 32) ^ static_cast<uint32_t>(k.box_cols * 4096 + k.box_rows));
  mix(static_cast<uint64_t>(k.dtype * 16 + k.swz));
  return static_cast<size_t>(h % MAP_CACHE);
}

bool encode_map(CUtensorMap* map, const Mat& m, int rows, int cols, int batch, int box_cols, int box_rows,
                CUtensorMapSwizzle swz);

// 3-D map over a 16-bit [batch][rows][cols] operand, box = box_cols x box_rows, 128-byte swizzle
// (operand loads) or 64-byte swizzle (32 x 32 epilogue stores).
bool make_map(CUtensorMap* map, const Mat& m, int rows, int cols, int batch, int box_cols, int box_rows,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  const MapKey k{m.ptr, m.ld, m.stride, m.dtype, rows, cols, batch, box_cols, box_rows, static_cast<int>(swz)};
  const size_t slot = key_slot(k);
  MapCache& c = map_cache();
  {
    std::lock_guard<std::mutex> lock(c.mu);
    if (c.used[slot] && same_key(c.key[slot], k)) {
      *map = c.map[slot];
      return true;
    }
  }
  if (!encode_map(map, m, rows, cols, batch, box_cols, box_rows, swz)) return false;
  std::lock_guard<std::mutex> lock(c.mu);
  c.used[slot] = true;
  c.key[slot] = k;
  c.map[slot] = *map;
  return true;
}

bool encode_map(CUtensorMap* map, const Mat& m, int rows, int cols, int batch, int box_cols, int box_rows,
                CUtensorMapSwizzle swz) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  const cuuint64_t es = 2;
  cuuint64_t ld_b = static_cast<cuuint64_t>(m.ld) * es;
  if (ld_b < 16) ld_b = 16;  // K == 0: the map is never read, but must be well formed
  cuuint64_t st_b = static_cast<cuuint64_t>(m.stride) * es;
  if (batch <= 1 || st_b == 0) st_b = ld_b * static_cast<cuuint64_t>(rows > 0 ? rows : 1);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {ld_b, st_b};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = m.dtype == FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, dt, 3, const_cast<void*>(m.ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Number of 2-CTA clusters of this kernel that fit on the device at once (cached per device).
template <int BN, bool B_MN, int EPI>
int max_clusters() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  auto kern = tc_gemm_kernel<BN, B_MN, EPI, 2>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(num_threads<EPI>(), 1, 1);
  cfg.dynamicSmemBytes = Cfg<BN, 2, EPI>::SMEM;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sm_count() / 2;
  }
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

template <int BN, bool B_MN, int EPI, int CL>
int launch(const GemmCall& g, cudaStream_t s) {
  using Cf = Cfg<BN, CL, EPI>;
  KParams p{};
  p.batch = g.batch;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.tiles_m = (g.M + BM - 1) / BM;
  p.tiles_n = (g.N + BN - 1) / BN;
  const int pairs = (p.tiles_m + 1) / 2;
  if (EPI == EPI_SYM) {
    int cnt = 0;
    if (CL == 1)
      for (int i = 0; i < p.tiles_m; ++i) cnt += i * BM / BN + 1;
    else
      cnt = pairs * (pairs + 1) / 2;
    p.tiles_per_batch = cnt;
  } else {
    p.tiles_per_batch = (CL == 1 ? p.tiles_m : pairs) * p.tiles_n;
  }
  p.total_tiles = static_cast<long long>(p.tiles_per_batch) * g.batch;
  p.num_kb = (g.K + BK - 1) / BK;
  p.idesc = ptx::make_idesc_f16(g.A.dtype == FP16 ? 0 : 1, B_MN, BM * CL, BN);
  p.D = const_cast<void*>(g.D.ptr);
  p.ldd = g.D.ld;
  p.sD = g.D.stride;
  p.d_type = g.D.dtype;
  p.C = g.C.ptr;
  p.ldc = g.C.ld;
  p.sC = g.C.stride;
  p.beta = g.beta;
  p.alpha = g.alpha;
  p.alpha_batch = g.alpha_batch;
  p.gamma = g.gamma;
  p.W = g.W;
  p.ldw = g.ldw;
  p.sW = g.sW;
  p.sel = g.sel;
  p.ssel = g.ssel;
  p.w_rows = g.w_rows;
  p.status = g.status;
  p.spin_limit = g.spin_limit > 0 ? g.spin_limit : DEFAULT_SPIN;
  p.eta_dev = g.eta_dev;
  p.eta_scale = g.eta_scale;
  p.check_finite = g.check_finite ? 1 : 0;
  if (p.total_tiles == 0) return DION3_OK;

  CUtensorMap ta, tb;
  // A is [batch][M][K].  With K == 0 nothing is loaded, but the maps must still be well
  // formed: they then describe a 16-byte-wide window at D, which is never read.
  Mat Ae = g.A, Be = g.B;
  if (g.K == 0) {
    Ae.ptr = Be.ptr = g.D.ptr;
    Ae.ld = Be.ld = 8;
    Ae.stride = Be.stride = 8LL * (g.M > g.N ? g.M : g.N);
    Ae.dtype = Be.dtype = BF16;
  }
  const int kdim = g.K > 0 ? g.K : 1;
  if (!make_map(&ta, Ae, g.M, kdim, g.batch, BK, BM)) return DION3_ECUDA;
  if (!B_MN) {
    if (!make_map(&tb, Be, g.N, kdim, g.batch, BK, BN / CL)) return DION3_ECUDA;
  } else {
    if (!make_map(&tb, Be, kdim, g.N, g.batch, 64, BK)) return DION3_ECUDA;
  }
  CUtensorMap td = ta;  // D as a TMA store target (16-bit D of EPI_SYM / EPI_GEN)
  if (EPI != EPI_WUPD && g.D.dtype != FP32) {
    if (!make_map(&td, g.D, g.M, g.N, g.batch, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) return DION3_ECUDA;
  }
  auto kern = tc_gemm_kernel<BN, B_MN, EPI, CL>;
  // The shared-memory opt-in is set once per device for each instantiation.
  static std::atomic<bool> smem_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DION3_ECUDA;
  if (dev < 0 || dev >= 64 || !smem_set[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM) != cudaSuccess)
      return DION3_ECUDA;
    if (dev >= 0 && dev < 64) smem_set[dev].store(true, std::memory_order_release);
  }
  if constexpr (CL == 1) {
    long long grid = sm_count();
    if (grid > p.total_tiles) grid = p.total_tiles;
    kern<<<static_cast<unsigned>(grid), num_threads<EPI>(), Cf::SMEM, s>>>(ta, tb, td, p);
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(num_threads<EPI>(), 1, 1);
    cfg.dynamicSmemBytes = Cf::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2 * max_clusters<BN, B_MN, EPI>(), 1, 1);
    long long clusters = cfg.gridDim.x / 2;
    if (clusters > p.total_tiles) clusters = p.total_tiles;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, td, p) != cudaSuccess) return DION3_ECUDA;
  }
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

}  // namespace

bool tensor_map_16(CUtensorMap* map, const Mat& m, int rows, int cols, int batch, int box_cols, int box_rows) {
  return make_map(map, m, rows, cols, batch, box_cols, box_rows);
}

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

int gemm_tc(const GemmCall& g, cudaStream_t s) {
  if (g.batch <= 0 || g.M <= 0 || g.N <= 0) return DION3_OK;
  if (g.beta != 0.f && (g.C.ptr == nullptr || g.C.dtype != g.D.dtype)) return DION3_EUNSUPPORTED;
  // Two CTAs (a cta_group::2 pair) compute each 256 x 256 tile when there are at least two row
  // blocks, each staging half of the B tile; otherwise one CTA per 128-row tile.
  switch (g.epi) {
    case EPI_SYM: {
      // CTA pairs on 256 x 256 tiles, unless that leaves SMs idle: then 128 x 128 tiles, which
      // give about twice as many CTAs (small single products such as n <= 2048).
      const long long pairs = (g.M + 255) / 256;
      const long long pair_ctas = 2 * pairs * (pairs + 1) / 2 * g.batch;
      if (g.M <= 128 || pair_ctas < sm_count()) return launch<128, false, EPI_SYM, 1>(g, s);
      return launch<256, false, EPI_SYM, 2>(g, s);
    }
    case EPI_GEN:
      if (g.N <= 128) return launch<128, true, EPI_GEN, 1>(g, s);
      return g.M <= 128 ? launch<256, true, EPI_GEN, 1>(g, s) : launch<256, true, EPI_GEN, 2>(g, s);
    case EPI_WUPD:
      if (g.N <= 128) return launch<128, true, EPI_WUPD, 1>(g, s);
      return g.M <= 128 ? launch<256, true, EPI_WUPD, 1>(g, s) : launch<256, true, EPI_WUPD, 2>(g, s);
    default:
      return DION3_EINVAL;
  }
}

int selftest_watchdog(long long spin_limit, int* status, cudaStream_t s) {
  watchdog_kernel<<<1, 32, 0, s>>>(spin_limit, status);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

}  // namespace dion3
