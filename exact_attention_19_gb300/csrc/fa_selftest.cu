// fa_selftest.cu -- exercises the bounded waits every kernel of the library
// relies on, without any fault: a wait on an mbarrier phase that nothing
// completes must give up and report, and the CUDA context must stay usable.
//
// One CTA of two warps.  mode 0: thread 0 waits (mbar_wait, the kernels' own
// bounded wait) on a barrier nothing arrives at; it returns false once the
// time limit (kWaitLimitNs) has passed.  mode 1: thread 0 waits the same way
// while warp 1 raises the CTA's abort flag after about 1 ms; the wait must
// give up on the flag, long before the time limit.  The outcome is written to
// a status word of this file (bit 0: the wait gave up; bits 8.. : 1 time
// limit, 2 abort flag) and the wait's duration in nanoseconds.
#include <cuda_runtime.h>

#include <cstdint>

#include "fa.h"
#include "fa_ptx.cuh"

namespace {

__device__ unsigned int g_selftest_word;
__device__ unsigned long long g_selftest_ns;

__global__ void __launch_bounds__(64, 1) fa_wait_selftest_kernel(int mode) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_storage;
  const uint32_t bar = fa::smem_addr(&bar_storage);
  volatile int* abort_flag = &abort_storage;
  if (threadIdx.x == 0) {
    fa::mbar_init(bar, 1);  // one arrival completes phase 0; none ever comes
    *abort_flag = 0;
    fa::mbar_init_fence();
  }
  __syncthreads();
  if (mode == 1 && threadIdx.x == 32) {
    const unsigned long long t0 = fa::global_ns();
    while (fa::global_ns() - t0 < 1000000ull) {
    }
    *abort_flag = 1;
  }
  if (threadIdx.x == 0) {
    const unsigned long long t0 = fa::global_ns();
    const bool completed = fa::mbar_wait(bar, 0, abort_flag);
    g_selftest_ns = fa::global_ns() - t0;
    if (!completed) atomicOr(&g_selftest_word, 1u | ((*abort_flag ? 2u : 1u) << 8));
  }
  __syncthreads();
}

}  // namespace

extern "C" int fa_selftest_wait(int mode, unsigned int* word, unsigned long long* wait_ns, cudaStream_t stream) {
  if (word == nullptr || wait_ns == nullptr) return FA_ERR_NULL;
  if (mode != 0 && mode != 1) return FA_ERR_SHAPE;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (major != 10 || minor != 3) return FA_ERR_DEVICE;
  const unsigned int zero_word = 0;
  const unsigned long long zero_ns = 0;
  if (cudaMemcpyToSymbolAsync(g_selftest_word, &zero_word, sizeof(zero_word), 0, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_selftest_ns, &zero_ns, sizeof(zero_ns), 0, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess)
    return FA_ERR_LAUNCH;
  fa_wait_selftest_kernel<<<1, 64, 0, stream>>>(mode);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  if (cudaMemcpyFromSymbolAsync(word, g_selftest_word, sizeof(*word), 0, cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaMemcpyFromSymbolAsync(wait_ns, g_selftest_ns, sizeof(*wait_ns), 0, cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}
