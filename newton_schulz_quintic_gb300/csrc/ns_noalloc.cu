// ns_noalloc.cu -- Newton-Schulz for callers that must not allocate device
// memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the moment they
// orthogonalize: a training process whose framework allocator has already
// reserved nearly all of HBM, so a foreign allocation fails or fragments the
// pool; an optimizer step on a latency budget that cannot absorb the
// allocator's implicit synchronisation; a runtime that forbids device
// allocation after start-up. ns_orthogonalize_batched_noalloc serves them: the
// scratch the method needs (working copies W and W^T, A, B, norms, tile lists
// and TMA descriptors) lives in one fixed array below, which the library
// reserves when the module loads and keeps on every device that loads it
// until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/ns.h"
#include "ns_internal.h"

namespace {

// Largest scratch a batch may use through this entry point.
constexpr size_t kNoAllocScratchBytes = size_t(256) << 20;  // 256 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device. In host code the array's
// name is only a host-side stand-in, never a device address, so the address
// is fetched with cudaGetSymbolAddress once per device, with that device
// current, the first time this entry point runs there.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

int scratch_address(void **out) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ? NS_ENODEV : NS_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return NS_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return NS_ECUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return NS_OK;
}

}  // namespace

extern "C" int ns_orthogonalize_batched_noalloc(void *const *X, const int64_t *shapes, int count, int steps,
                                                const float *coeffs, int dtype, void *stream) {
  // the arguments and the device first, with the codes every entry point
  // returns for them; only a valid batch is measured against the array
  int rc = ns::check_call(X, shapes, count, steps, dtype);
  if (rc != NS_OK || count == 0) return rc;
  const size_t need = ns_workspace_bytes(shapes, count, dtype);
  if (need == 0) return NS_EINVAL;
  if (need > kNoAllocScratchBytes) return NS_ETOOBIG;
  void *ws = nullptr;
  rc = scratch_address(&ws);
  if (rc != NS_OK) return rc;
  // the caller-workspace path: it launches into `ws` and allocates nothing
  return ns_orthogonalize_batched_ex(X, shapes, count, steps, coeffs, 1e-7f, dtype, ws, kNoAllocScratchBytes,
                                     stream);
}
