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
// come before any stream capture.  Host code never hands the array's name itself to a kernel:
// on the host that name is a stand-in, not a device address.
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
  if (batch < 0 || n < 0 || m < 0 || n > m || !dion3::dtype_valid(x_dtype) || !dion3::dtype_valid(compute_dtype))
    return DION3_EINVAL;
  // Reject problems that need more scratch than the array holds, before touching the GPU.
  if (dion3_gram_ns_workspace_bytes(batch, n, m, x_dtype, compute_dtype, n_restart < 0 ? 0 : n_restart) >
      static_cast<size_t>(DION3_NOALLOC_SCRATCH_BYTES))
    return DION3_EWORKSPACE;
  if (batch == 0 || n == 0) return DION3_OK;
  void* scratch = nullptr;
  if (int rc = scratch_address(&scratch)) return rc;
  return dion3_gram_ns(batch, n, m, X, ldx, strideX, x_dtype, Out, ldo, strideO, out_dtype, T, abc, restart_after,
                       n_restart, eps, compute_dtype, scratch, static_cast<size_t>(DION3_NOALLOC_SCRATCH_BYTES),
                       status_dev, stream);
}
