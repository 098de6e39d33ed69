// k_selftest.cu -- watchdog self-test: one thread waits, with the bounded wait
// of every libtm kernel, on an mbarrier that nothing arrives at. The wait runs
// out, the status word records the timeout, and the kernel returns.
// Also a probe of the special-function pipe's exponential rate (the unit the
// triangle attention's softmax leans on): independent ex2.approx chains.
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

// Every thread runs 8 independent chains of iters exponentials (each result scaled back below 1 by
// an FMA-pipe multiply, off the special-function pipe); the sink keeps the chains live.
__device__ float probe_sink;
__global__ void __launch_bounds__(512) k_probe_ex2(int iters) {
  float x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = (float)(threadIdx.x + k) * 1e-3f;
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float y;
      asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x[k]));
      x[k] = y * 0.5f;
    }
  }
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) sum += x[k];
  if (sum == 12345.f) probe_sink = sum;   // never true for these chains; keeps them from being removed
}

}  // namespace

cudaError_t launch_probe_ex2(int blocks, int iters, cudaStream_t s) {
  k_probe_ex2<<<blocks, 512, 0, s>>>(iters);
  return cudaGetLastError();
}

cudaError_t launch_watchdog_selftest(const Watch& w, cudaStream_t s) {
  k_watchdog_selftest<<<1, 32, 0, s>>>(w);
  return cudaGetLastError();
}

}  // namespace tmk
