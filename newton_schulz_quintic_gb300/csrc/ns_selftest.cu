// ns_selftest.cu -- exercises the bounded-wait failure path on the device.
//
// One CTA initialises an mbarrier that expects one arrival which never comes
// and waits on it with the same bounded wait the GEMM kernels use, but with a
// short limit. The wait gives up, records NS_ETIMEOUT in the device status
// word and the kernel returns normally, so the context stays usable. Nothing
// faults, traps or hangs.
#include <cuda_runtime.h>

#include "ns_device.cuh"

namespace ns {

__global__ void __launch_bounds__(32) ns_wait_probe_kernel(int *status, uint64_t limit_ns, int *gave_up) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    const Waiter w{&abort_flag, status, limit_ns};
    const bool done = mbar_wait(&bar, 0, w);
    *gave_up = done ? 0 : 1;
  }
}

int launch_wait_probe(int *status, uint64_t limit_ns, int *gave_up, cudaStream_t s) {
  ns_wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns, gave_up);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace ns
