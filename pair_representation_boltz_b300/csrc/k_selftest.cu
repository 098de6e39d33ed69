// k_selftest.cu -- watchdog self-test: one thread waits, with the bounded wait
// of every libtm kernel, on an mbarrier that nothing arrives at. The wait runs
// out, the status word records the timeout, and the kernel returns.
#include "tm_kernels.h"

namespace tmk {
namespace {

__global__ void k_watchdog_selftest(Watch w) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    wait_bounded(&bar, 0, w, &abort_flag, 99);
  }
}

}  // namespace

cudaError_t launch_watchdog_selftest(const Watch& w, cudaStream_t s) {
  k_watchdog_selftest<<<1, 32, 0, s>>>(w);
  return cudaGetLastError();
}

}  // namespace tmk
