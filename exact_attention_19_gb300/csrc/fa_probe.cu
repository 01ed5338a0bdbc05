// fa_probe.cu -- throughput probes of 2^x.
//
// The softmax of the attention forward issues one ex2.approx per score; the
// page "pinghaoyang FlashAttention 1-4 guide" (FA4 section) names this unit
// (MUFU) as the one that stops keeping pace with the tensor cores on
// Blackwell, and describes moving part of the exponentials onto the FMA
// pipes as a polynomial.  fa_probe_exp2 measures either way's rate on the
// device at hand: the MUFU rate is the third roofline of the forward kernel,
// the polynomial rate says what such an offload could add.
//
// One CTA per SM (the dynamic shared-memory request keeps a second CTA off
// the SM), 16 warps per CTA, each thread running 16 independent chains of
// x <- 2^x - 1.5 (x stays in [-1, -0.5]).
//   method 0: ex2.approx.ftz.f32 (MUFU); the subtraction runs on the FMA pipe.
//   method 1: 2^x = 2^n * p(f) with n = round(x) (the 1.5 * 2^23 shift), f =
//             x - n in [-1/2, 1/2], p the cubic Taylor polynomial of e^(f ln 2)
//             in Horner form, and 2^n added to p's exponent field; every step
//             runs on the FMA and integer pipes.  Only the rate matters here:
//             the cubic's relative error (about 1e-3 at f = 1/2) is not tuned.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "fa.h"
#include "fa_ptx.cuh"

namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeChains = 16;
constexpr int kProbeIters = 4096;
constexpr int kProbeMaxSms = 1024;
constexpr int kProbeSmem = 128 * 1024;  // more than half an SM's shared memory

__device__ long long g_probe_cycles[kProbeMaxSms];
__device__ float g_probe_sink[kProbeMaxSms];

__device__ __forceinline__ float poly_exp2(float x) {
  const float shift = 12582912.0f;  // 1.5 * 2^23: adding it rounds x to an integer in the low mantissa bits
  const float t = x + shift;
  const float f = x - (t - shift);
  // e^(f ln 2) = 1 + f ln2 + (f ln2)^2 / 2 + (f ln2)^3 / 6 + ...
  float p = fmaf(f, 0.05550410866f, 0.2402265070f);
  p = fmaf(p, f, 0.6931471806f);
  p = fmaf(p, f, 1.0f);
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

template <int METHOD>
__global__ void __launch_bounds__(kProbeThreads, 1) fa_exp2_probe_kernel() {
  extern __shared__ uint8_t probe_smem[];
  float x[kProbeChains];
#pragma unroll
  for (int u = 0; u < kProbeChains; ++u) x[u] = -0.5f - 0.03125f * static_cast<float>((threadIdx.x + u) & 15);
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < kProbeIters; ++i) {
#pragma unroll
    for (int u = 0; u < kProbeChains; ++u) x[u] = (METHOD == 0 ? fa::ex2(x[u]) : poly_exp2(x[u])) - 1.5f;
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int u = 0; u < kProbeChains; ++u) s += x[u];
  if (s > 1.0e30f) {  // never true: keeps the chains live without a store per thread
    probe_smem[threadIdx.x] = 1;
    g_probe_sink[blockIdx.x] = s + probe_smem[threadIdx.x ^ 1];
  }
  if (threadIdx.x == 0) g_probe_cycles[blockIdx.x] = t1 - t0;
}

template <int METHOD>
int run_probe(int grid, cudaStream_t stream) {
  if (cudaFuncSetAttribute(fa_exp2_probe_kernel<METHOD>, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) !=
      cudaSuccess)
    return FA_ERR_LAUNCH;
  // the first launch warms the clocks and the instruction cache; the second is read
  for (int rep = 0; rep < 2; ++rep) {
    fa_exp2_probe_kernel<METHOD><<<grid, kProbeThreads, kProbeSmem, stream>>>();
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

}  // namespace

extern "C" int fa_probe_exp2(int method, double* per_clk_sm, cudaStream_t stream) {
  if (per_clk_sm == nullptr) return FA_ERR_NULL;
  if (method != 0 && method != 1) return FA_ERR_SHAPE;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (major != 10 || minor != 3) return FA_ERR_DEVICE;
  const int grid = std::min(sms, kProbeMaxSms);
  if (grid <= 0) return FA_ERR_LAUNCH;
  const int launched = method == 0 ? run_probe<0>(grid, stream) : run_probe<1>(grid, stream);
  if (launched != FA_OK) return launched;
  std::vector<long long> cycles(static_cast<size_t>(grid));
  if (cudaMemcpyFromSymbolAsync(cycles.data(), g_probe_cycles, sizeof(long long) * grid, 0,
                                cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FA_ERR_LAUNCH;
  std::sort(cycles.begin(), cycles.end());
  const long long median = cycles[cycles.size() / 2];
  if (median <= 0) return FA_ERR_LAUNCH;
  *per_clk_sm = static_cast<double>(kProbeIters) * kProbeChains * kProbeThreads / static_cast<double>(median);
  return FA_OK;
}
