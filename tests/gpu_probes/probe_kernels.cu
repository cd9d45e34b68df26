// probe_kernels.cu -- test-only kernels for tests/test_gpu_error_paths.py,
// compiled by that test into a library of their own (never into libgdn.so).
//
//  * gdn_probe_timeout: one thread waits, with the library's bounded
//    mbarrier wait and a poll limit of a few polls, on a barrier that nothing
//    signals (no thread arrives, no copy or product is attached), so the wait
//    runs out at once and reports a timeout into the given error word. The
//    kernel then returns; nothing is left in flight.
//  * gdn_probe_delayed_copy: a kernel that lets the next kernel of the stream
//    be scheduled at its start (griddepcontrol.launch_dependents), spins on
//    the global timer for a bounded time and only then writes dst = src; it
//    stands for a producer of a state_in pointer array that triggers early.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace {

__global__ void wait_on_silent_barrier(int *err, int site, unsigned polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    gdn::mbar_init(&bar, 1);
    gdn::fence_mbar_init();
    gdn::mbar_wait_n(&bar, 0, err, site, polls);
  }
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void write_after_delay(const unsigned long long *src, unsigned long long *dst, int n,
                                  unsigned long long delay_ns) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const unsigned long long t0 = global_ns();
  while (global_ns() - t0 < delay_ns) {
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

}  // namespace

extern "C" int gdn_probe_timeout(int *err, int site, unsigned polls, cudaStream_t stream) {
  wait_on_silent_barrier<<<1, 32, 0, stream>>>(err, site, polls);
  return (int)cudaGetLastError();
}

extern "C" int gdn_probe_delayed_copy(const unsigned long long *src, unsigned long long *dst,
                                      int n, unsigned long long delay_ns, cudaStream_t stream) {
  write_after_delay<<<1, 128, 0, stream>>>(src, dst, n, delay_ns);
  return (int)cudaGetLastError();
}
