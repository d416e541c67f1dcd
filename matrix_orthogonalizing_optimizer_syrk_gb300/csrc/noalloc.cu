// Gram Newton-Schulz for callers that cannot allocate device memory.
//
// Some callers of this library may not allocate device memory: embedded runtimes whose
// device memory is carved up once at start-up, plug-ins that are handed raw device buffers
// by a host application that owns every allocation, and code running inside an allocator or
// memory-pool callback, where a new allocation would re-enter the allocator.  They cannot
// provide the scratch workspace dion3_gram_ns asks for.  dion3_gram_ns_noalloc serves them
// from a fixed scratch array compiled into this library: the array occupies
// DION3_NOALLOC_SCRATCH_BYTES of device memory on every GPU that loads the library's code, from
// then until the process exits.
//
// The array's device address is looked up once per device (cudaGetSymbolAddress, with that
// device current) by the first call made on that device, then reused; that first call should
// come before any stream capture.  The saved address belongs to the device's primary context:
// after cudaDeviceReset (which destroys that context and the library's module in it) it is no
// longer valid, so a process that resets a device must not call this entry point on it again.
// Host code never hands the array's name itself to a kernel: on the host that name is a
// stand-in, not a device address.
//
// All calls share the one array, and it keeps whatever the last call left in it.  No part of
// it needs to start at zero (every byte the computation reads was written earlier in the same
// call), but two calls whose work overlaps on the GPU -- on different streams, or from
// different host threads -- race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DION3_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on first use).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DION3_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return DION3_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DION3_ECUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return DION3_OK;
}

}  // namespace

extern "C" int dion3_gram_ns_noalloc(int batch, int n, int m, const void* X, int64_t ldx, int64_t strideX,
                                     int x_dtype, void* Out, int64_t ldo, int64_t strideO, int out_dtype, int T,
                                     const float* abc, const int* restart_after, int n_restart, float eps,
                                     int compute_dtype, int* status_dev, void* stream) {
  // The same checks, in the same order, as dion3_gram_ns: a bad call gets the same code from
  // both entry points.  Then problems that need more scratch than the array holds (including
  // the copy a misaligned X needs) are rejected before the GPU is touched.
  size_t need = 0;
  if (int rc = dion3::gram_ns_validate(batch, n, m, X, ldx, strideX, x_dtype, Out, ldo, strideO, out_dtype, T, abc,
                                       restart_after, n_restart, eps, compute_dtype, &need))
    return rc;
  if (need == 0) return DION3_OK;
  if (need > static_cast<size_t>(DION3_NOALLOC_SCRATCH_BYTES)) return DION3_EWORKSPACE;
  void* scratch = nullptr;
  if (int rc = scratch_address(&scratch)) return rc;
  return dion3_gram_ns(batch, n, m, X, ldx, strideX, x_dtype, Out, ldo, strideO, out_dtype, T, abc, restart_after,
                       n_restart, eps, compute_dtype, scratch, static_cast<size_t>(DION3_NOALLOC_SCRATCH_BYTES),
                       status_dev, stream);
}
