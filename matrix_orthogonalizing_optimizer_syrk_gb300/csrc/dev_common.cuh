// Small device helpers shared by the kernels of libdion3.so: element conversions, packing of
// 16-bit pairs, compensated summation and the bounded drain wait used after an abort.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "dion3.h"
#include "ptx.cuh"

// Checked builds (libdion3_checked.so) compile with DION3_RANGE_CHECKS=1: the index checks below
// then set DION3_DEV_RANGE in the caller's status word.  In the default build they compile to
// nothing; the accesses they guard are skipped by the kernels' own bounds in both builds.
#ifndef DION3_RANGE_CHECKS
#define DION3_RANGE_CHECKS 0
#endif

namespace dion3 {
namespace dev {

// An index that should lie in its buffer: `ok` false sets DION3_DEV_RANGE (checked builds only).
__device__ __forceinline__ void range_check(bool ok, int* status) {
#if DION3_RANGE_CHECKS
  if (!ok && status != nullptr) atomicOr(status, DION3_DEV_RANGE);
#else
  (void)ok;
  (void)status;
#endif
}

// Conversions between a stored element type (fp32, bf16, fp16) and fp32, round to nearest.
template <typename T>
struct Num;
template <>
struct Num<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <>
struct Num<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
};
template <>
struct Num<__half> {
  static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
  static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
};

template <typename T>
__device__ __forceinline__ float to_f(T v) { return Num<T>::to_f(v); }
template <typename T>
__device__ __forceinline__ T from_f(float v) { return Num<T>::from_f(v); }
// Two fp32 values rounded to a 16-bit pair (lo in the low half-word).
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) { return Num<T>::pack2(lo, hi); }
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w) { return Num<T>::unpack2(w); }

// One step of Kahan's compensated summation in fp32, with every operation rounded once
// (no contraction): s + c carries the running sum.
__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = __fsub_rn(x, c);
  const float t = __fadd_rn(s, y);
  c = __fsub_rn(__fsub_rn(t, s), y);
  s = t;
}

// Bounded wait on an mbarrier phase that ignores the abort flag: used while draining in-flight
// copies and MMAs after a wait gave up.  Returns after `limit` clock cycles at the latest.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) break;
  }
}

}  // namespace dev
}  // namespace dion3
