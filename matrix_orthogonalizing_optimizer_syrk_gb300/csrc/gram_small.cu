// One restart segment of Gram Newton-Schulz for small Gram matrices (n <= 128), fused into a
// single persistent kernel ("Dion3: Full-Stack Orthogonal Updates", core method Theorem 2 and
// method details Algorithm 3).
//
// For each matrix of the batch one CTA loads R (n x n, 16-bit) and runs the iterations of the
// segment entirely on chip:
//   Z = a_t I + b_t R + c_t R^2;  Q = Z (first iteration) or Q Z;  R = (R Z) Z (not after the
//   segment's last iteration)
// and stores Q.  R, Z, Q and R Z live in shared memory as n16 x n16 16-bit matrices (n16 = n
// rounded up to 16) in the 128-byte-swizzled layout of 64-column panels of n16 rows -- the
// layout TMA writes for a {64, n16} box -- which the tensor cores read directly as the K-major
// A operand (rows = M) and as the MN-major B operand (rows = K), so no product needs a
// transpose or assumes symmetry.  The products run on tcgen05.mma (M = 128, N = n16) into two
// TMEM accumulators; an A operand's rows past n16 run into the next panel, which only fills
// accumulator rows that are never read.  128 threads (one per TMEM lane = matrix row) convert
// the accumulators back into shared memory.  At n = 96 a CTA needs about 100 KB of shared
// memory and 256 TMEM columns, so two CTAs share an SM and overlap their dependent chains.
//
// This replaces, for k x k Gram matrices of a few dozen to 128 rows (fine-grained MoE experts
// at f = 1/8), the separate product launches whose 128 x 128 tiles are latency-bound.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dev_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dion3 {
namespace {

constexpr int SEG_THREADS = 128;
constexpr int SEG_TMEM_COLS = 256;       // two accumulators of up to 128 columns
constexpr int SEG_SMEM_TWO_PER_SM = 115712;  // per-CTA shared memory that still fits two CTAs per SM
constexpr long long SEG_SPIN = 4000000000LL;

struct SegParams {
  int batch, n, n16;
  int panel;        // bytes of one 64-column panel: n16 rows x 128 bytes
  int npanels;      // ceil(n16 / 64)
  int mat;          // bytes of one matrix buffer: npanels panels
  int nbuf;         // 4 (R, Z, Q, T = R Z) or 5 (plus the next matrix's R)
  int iters;        // iterations in this segment (>= 1)
  float a[DION3_SEG_MAX_ITERS], b[DION3_SEG_MAX_ITERS], c[DION3_SEG_MAX_ITERS];
  uint32_t idesc;
  int* status;
  long long spin_limit;
};

// Byte offset of element (row, col) in a 16-bit matrix stored as 128-byte-swizzled panels of 64
// columns (`panel` bytes each, a multiple of 2048): 16-byte units of each 128-byte row permuted
// by row % 8.
__device__ __forceinline__ uint32_t sw_off(int row, int col, int panel) {
  return static_cast<uint32_t>((col >> 6) * panel + row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) +
                               ((col & 7) << 1));
}

using dev::pack2;
using dev::unpack2;

// acc = A * B over K = n16 (K-major A, MN-major B, both in the panel layout).  One thread.
__device__ __forceinline__ void mma_nn(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, int n16, int panel,
                                       uint32_t idesc) {
  for (int kk = 0; kk < n16 / 16; ++kk) {
    const uint64_t ad = ptx::smem_desc_sw128(a_base + (kk >> 2) * panel + (kk & 3) * 32, 16, 1024);
    const uint64_t bd = ptx::smem_desc_sw128(b_base + kk * 16 * 128, panel, 1024);
    ptx::tc_mma_f16(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
  }
}

// Row `row` (this thread's TMEM lane) of an accumulator, turned into 16-bit values in the panel
// layout of `dst`:  v = cs * acc + bs * src[row][col] + (col == row ? as : 0), zero outside
// the n x n matrix.  `src` is read only when bs != 0.  Rows from n16 on are not stored (the
// buffers hold n16 rows); the TMEM load itself is warp-wide, so every lane takes part.
template <typename T>
__device__ __forceinline__ void drain_row(uint32_t t_acc, int row, int n, int n16, int panel, float cs, float bs,
                                          float as, const uint8_t* src, uint8_t* dst) {
  for (int q = 0; q < n16; q += 32) {
    uint32_t v[32];
    ptx::tmem_ld_32x32b_x32(t_acc + q, v);
    if (row >= n16) continue;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c0 = q + 8 * u;
      uint4 rv = make_uint4(0u, 0u, 0u, 0u);
      if (bs != 0.f) rv = *reinterpret_cast<const uint4*>(src + sw_off(row, c0, panel));
      const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int ca = c0 + 2 * h;
        const float2 r2 = unpack2<T>(rw[h]);
        float lo = cs * __uint_as_float(v[8 * u + 2 * h]);
        float hi = cs * __uint_as_float(v[8 * u + 2 * h + 1]);
        if (bs != 0.f) {
          lo = fmaf(bs, r2.x, lo);
          hi = fmaf(bs, r2.y, hi);
        }
        if (ca == row) lo += as;
        if (ca + 1 == row) hi += as;
        if (row >= n || ca >= n) lo = 0.f;
        if (row >= n || ca + 1 >= n) hi = 0.f;
        w[h] = pack2<T>(lo, hi);
      }
      *reinterpret_cast<uint4*>(dst + sw_off(row, c0, panel)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Shared-memory layout: nbuf matrix buffers; then the bytes an A operand read of the last panel
// runs past it (the MMA reads 128 rows, a panel holds n16); then three mbarriers, the TMEM
// address and the abort flag.
__host__ __device__ __forceinline__ int seg_bars_offset(const SegParams& p) {
  return p.nbuf * p.mat + (128 * 128 - p.panel);
}
__host__ __device__ __forceinline__ int seg_smem_bytes(const SegParams& p) {
  return seg_bars_offset(p) + 64 + 1024;  // + barriers, + alignment of the dynamic base to 1024
}

// Make this thread's shared-memory writes visible to the tensor cores and TMA, then sync.
__device__ __forceinline__ void publish() {
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
}

using dev::drain_wait;

template <typename T>
__global__ void __launch_bounds__(SEG_THREADS, 1)
    gram_seg_kernel(const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmQ,
                    const SegParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // Buffers, then room for the rows an A operand reads past the last panel, then the barriers.
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + seg_bars_offset(p));
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  const uint32_t bar_load = ptx::smem_u32(bars), bar_mma = bar_load + 8, bar_drain = bar_load + 16;
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    ptx::mbar_init(bar_load, 1);
    ptx::mbar_init(bar_mma, 1);
    ptx::mbar_init(bar_drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tmR);
    ptx::tma_prefetch_desc(&tmQ);
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_holder), SEG_TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's TMEM lanes
  volatile int* abort = abort_flag;
  const long long lim = p.spin_limit;
  uint32_t ph_load = 0, ph_mma = 0;
  bool ok = true, load_pending = false;

  // One thread waits on the mbarrier (bounded); the CTA barrier hands its verdict to every
  // thread, so all of them take the same path, and orders their TMEM reads after the MMAs.
  auto cta_wait = [&](uint32_t bar, uint32_t& ph) {
    int failed = 0;
    if (tid == 0) failed = ptx::mbar_wait(bar, ph, abort, lim) ? 0 : 1;
    if (__syncthreads_or(failed)) return false;
    ph ^= 1u;
    ptx::tc_fence_after();
    return true;
  };

  // With a fifth buffer, R of the next matrix is loaded into the spare S while this one is
  // computed, and the buffers rotate (the old R becomes the next spare); otherwise each
  // matrix's R is loaded when the previous matrix is done.
  const bool prefetch = p.nbuf == 5;
  const int panel = p.panel;
  uint8_t* R = smem;
  uint8_t* Z = smem + p.mat;
  uint8_t* Q = smem + 2 * p.mat;
  uint8_t* Tm = smem + 3 * p.mat;
  uint8_t* S = smem + 4 * p.mat;
  auto issue_load = [&](uint8_t* dst, int mat) {
    ptx::mbar_arrive_expect_tx(bar_load, static_cast<uint32_t>(p.mat));
    for (int pi = 0; pi < p.npanels; ++pi)
      ptx::tma_load_3d(ptx::smem_u32(dst + pi * panel), &tmR, bar_load, 64 * pi, 0, mat);
    load_pending = true;
  };
  if (tid == 0 && static_cast<int>(blockIdx.x) < p.batch) issue_load(R, blockIdx.x);
  for (int mat = blockIdx.x; ok && mat < p.batch; mat += gridDim.x) {
    if (!cta_wait(bar_load, ph_load)) {
      ok = false;
      break;
    }
    load_pending = false;
    const int next = mat + static_cast<int>(gridDim.x);
    if (tid == 0 && prefetch && next < p.batch) issue_load(S, next);
    bool q_identity = true;
    for (int j = 0; j < p.iters; ++j) {
      const bool last = j + 1 == p.iters;
      // R^2, then Z = a I + b R + c R^2
      if (tid == 0) {
        mma_nn(tmem + 0, ptx::smem_u32(R), ptx::smem_u32(R), p.n16, panel, p.idesc);
        ptx::tc_commit(bar_mma);
        // The previous matrix's Q store must have read its buffer before anything is written.
        if (j == 0) ptx::bulk_wait_read_0();
      }
      if (!cta_wait(bar_mma, ph_mma)) {
        ok = false;
        break;
      }
      drain_row<T>(t_lane + 0, tid, p.n, p.n16, panel, p.c[j], p.b[j], p.a[j], R, Z);
      publish();
      // Q Z (or Q = Z after a start) and R Z (unless this is the segment's last iteration)
      const bool do_qz = !q_identity, do_rz = !last;
      if (q_identity) {  // Q takes over Z's buffer; the old Q buffer receives the next Z
        uint8_t* t = Q;
        Q = Z;
        Z = t;
        q_identity = false;
      }
      uint8_t* Zc = do_qz ? Z : Q;  // where this iteration's Z lives
      if (do_qz || do_rz) {
        if (tid == 0) {
          if (do_qz) mma_nn(tmem + 0, ptx::smem_u32(Q), ptx::smem_u32(Zc), p.n16, panel, p.idesc);
          if (do_rz) mma_nn(tmem + 128, ptx::smem_u32(R), ptx::smem_u32(Zc), p.n16, panel, p.idesc);
          ptx::tc_commit(bar_mma);
        }
        if (!cta_wait(bar_mma, ph_mma)) {
          ok = false;
          break;
        }
        if (do_qz) drain_row<T>(t_lane + 0, tid, p.n, p.n16, panel, 1.f, 0.f, 0.f, nullptr, Q);
        if (do_rz) drain_row<T>(t_lane + 128, tid, p.n, p.n16, panel, 1.f, 0.f, 0.f, nullptr, Tm);
        publish();
      }
      if (do_rz) {  // R = (R Z) Z
        if (tid == 0) {
          mma_nn(tmem + 0, ptx::smem_u32(Tm), ptx::smem_u32(Zc), p.n16, panel, p.idesc);
          ptx::tc_commit(bar_mma);
        }
        if (!cta_wait(bar_mma, ph_mma)) {
          ok = false;
          break;
        }
        drain_row<T>(t_lane + 0, tid, p.n, p.n16, panel, 1.f, 0.f, 0.f, nullptr, R);
        publish();
      }
    }
    if (!ok) break;
    if (tid == 0) {
      for (int pi = 0; pi < p.npanels; ++pi) ptx::tma_store_3d(&tmQ, ptx::smem_u32(Q + pi * panel), 64 * pi, 0, mat);
      ptx::bulk_commit_group();
    }
    if (prefetch) {
      uint8_t* t = R;
      R = S;
      S = t;
    } else if (tid == 0 && next < p.batch) {
      issue_load(R, next);  // R is never the buffer the Q store reads
    }
  }
  if (tid == 0) {
    // Let every issued copy and MMA finish before the shared memory and TMEM are released.
    if (load_pending) drain_wait(bar_load, ph_load, lim);
    ptx::tc_commit(bar_drain);
    drain_wait(bar_drain, 0, lim);
    ptx::bulk_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, SEG_TMEM_COLS);
  }
  if (tid == 0 && *abort && p.status) atomicOr(p.status, DION3_DEV_TIMEOUT);
}

}  // namespace

int gram_segment(int batch, int n, const Mat& R, const Mat& Q, int iters, const float* abc, int* status,
                 cudaStream_t s) {
  if (batch <= 0 || n <= 0) return DION3_OK;
  if (n > 128 || iters < 1 || iters > DION3_SEG_MAX_ITERS) return DION3_EUNSUPPORTED;
  if (R.dtype == FP32 || R.dtype != Q.dtype) return DION3_EUNSUPPORTED;
  SegParams p{};
  p.batch = batch;
  p.n = n;
  p.n16 = (n + 15) / 16 * 16;
  p.iters = iters;
  for (int j = 0; j < iters; ++j) {
    p.a[j] = abc[3 * j];
    p.b[j] = abc[3 * j + 1];
    p.c[j] = abc[3 * j + 2];
  }
  p.idesc = ptx::make_idesc_f16(R.dtype == FP16 ? 0 : 1, true, 128, p.n16);
  p.status = status;
  p.spin_limit = SEG_SPIN;
  p.panel = p.n16 * 128;
  p.npanels = (p.n16 + 63) / 64;
  p.mat = p.npanels * p.panel;
  // Two CTAs per SM when four buffers leave room for them (TMEM allows two: 256 columns each);
  // the fifth, prefetch buffer only where it does not cost that.
  p.nbuf = 4;
  int per_sm = seg_smem_bytes(p) <= SEG_SMEM_TWO_PER_SM ? 2 : 1;
  p.nbuf = 5;
  if (per_sm == 2 && seg_smem_bytes(p) > SEG_SMEM_TWO_PER_SM) p.nbuf = 4;
  const int smem = seg_smem_bytes(p);
  CUtensorMap tr, tq;
  if (!tensor_map_16(&tr, R, n, n, batch, 64, p.n16) || !tensor_map_16(&tq, Q, n, n, batch, 64, p.n16))
    return DION3_ECUDA;
  const bool half = R.dtype == FP16;
  auto kern = half ? gram_seg_kernel<__half> : gram_seg_kernel<__nv_bfloat16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return DION3_ECUDA;
  long long grid = static_cast<long long>(sm_count()) * per_sm;
  if (grid > batch) grid = batch;
  kern<<<static_cast<unsigned>(grid), SEG_THREADS, smem, s>>>(tr, tq, p);
  return cudaGetLastError() == cudaSuccess ? DION3_OK : DION3_ECUDA;
}

}  // namespace dion3
