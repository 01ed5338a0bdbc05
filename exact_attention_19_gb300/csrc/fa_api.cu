// fa_api.cu -- C-ABI front end of libfa_gb300.so: argument checks, TMA
// tensor maps, kernel selection and launch.  See include/fa.h for the
// contract of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_fwd_kernel.cuh"

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Per-device one-time state: compute capability check and the kernels'
// shared-memory opt-in.  0 = not yet, 1 = ready, -1 = unsupported device.
std::atomic<int> g_dev_state[kMaxDevices];
std::mutex g_dev_mutex;

template <int D, bool CAUSAL>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(fa::fa_fwd_kernel<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::Cfg<D>::kSmemBytes));
}

int prepare_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
  int st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st == 1) return FA_OK;
  if (st == -1) return FA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st != 0) return st == 1 ? FA_OK : FA_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (major != 10 || minor != 3) {
    g_dev_state[dev].store(-1, std::memory_order_release);
    return FA_ERR_DEVICE;
  }
  if (set_smem_attr<64, false>() != cudaSuccess || set_smem_attr<64, true>() != cudaSuccess ||
      set_smem_attr<128, false>() != cudaSuccess || set_smem_attr<128, true>() != cudaSuccess)
    return FA_ERR_LAUNCH;
  g_dev_state[dev].store(1, std::memory_order_release);
  return FA_OK;
}

bool is_device_pointer(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state of this query
    return false;
  }
  if (a.type == cudaMemoryTypeManaged) return true;
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

// 3-D tensor map over a [BH, N, D] bf16 tensor: dims (D, N, BH), box
// (64, 128, 1), 128-byte swizzle.  Rows past N inside a head read as zero.
bool make_map(CUtensorMap* map, const void* ptr, int D, long long N, long long BH) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2u, static_cast<cuuint64_t>(N) * D * 2u};
  cuuint32_t box[3] = {64u, 128u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool CAUSAL>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const fa::FwdParams& p,
           long long grid, cudaStream_t stream) {
  fa::fa_fwd_kernel<D, CAUSAL><<<static_cast<unsigned>(grid), fa::Cfg<D>::kThreads, fa::Cfg<D>::kSmemBytes,
                                 stream>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int fa_version(void) { return kVersion; }

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case FA_ERR_SHAPE: return "invalid shape (B, H, Nk must be > 0, Nq >= 0, sizes within limits)";
    case FA_ERR_HEADDIM: return "head dimension must be 64 or 128";
    case FA_ERR_CAUSAL_SHAPE: return "causal attention needs Nq == Nk";
    case FA_ERR_LAUNCH: return "CUDA launch or set-up call failed";
    case FA_ERR_DEVICE: return "current device is not a compute capability 10.3 (GB300) GPU";
    case FA_ERR_TIMEOUT: return "a kernel wait timed out";
    case FA_ERR_SCALE: return "scale must be finite and > 0";
    case FA_ERR_POINTER: return "a tensor pointer is not device memory of the current device";
    default: return "unknown status";
  }
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
           int d, float scale, int causal, cudaStream_t stream) {
  // ---- host-side validation (nothing is launched on failure) --------------
  // With Nq == 0 nothing is read or written, so the (empty) tensors may be NULL.
  if ((Nq != 0 && (!q || !o || !lse)) || !k || !v) return FA_ERR_NULL;
  const uintptr_t mis = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                         reinterpret_cast<uintptr_t>(lse)) & 15u;
  if (mis) return FA_ERR_ALIGN;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (B <= 0 || H <= 0 || Nk <= 0 || Nq < 0) return FA_ERR_SHAPE;
  if (causal != 0 && causal != 1) return FA_ERR_SHAPE;
  if (causal && Nq != Nk) return FA_ERR_CAUSAL_SHAPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  const long long BH = static_cast<long long>(B) * H;
  const long long n_pairs = (static_cast<long long>(Nq) + 255) / 256;
  const long long grid = BH * n_pairs;
  // tensor-map limits: a stride below 2^40 bytes, grid below 2^31 CTAs
  if (static_cast<long long>(Nq > Nk ? Nq : Nk) * d * 2 >= (1ll << 40)) return FA_ERR_SHAPE;
  if (BH >= (1ll << 31) || grid >= (1ll << 31)) return FA_ERR_SHAPE;
  if (Nq == 0) return FA_OK;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_LAUNCH;
  const int prep = prepare_device(dev);
  if (prep != FA_OK) return prep;
  if (!is_device_pointer(q, dev) || !is_device_pointer(k, dev) || !is_device_pointer(v, dev) ||
      !is_device_pointer(o, dev) || !is_device_pointer(lse, dev))
    return FA_ERR_POINTER;

  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, d, Nq, BH) || !make_map(&mk, k, d, Nk, BH) || !make_map(&mv, v, d, Nk, BH))
    return FA_ERR_LAUNCH;

  fa::FwdParams p;
  p.o = o;
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_pairs = static_cast<int>(n_pairs);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);

  if (d == 64) return causal ? launch<64, true>(mq, mk, mv, p, grid, stream)
                             : launch<64, false>(mq, mk, mv, p, grid, stream);
  return causal ? launch<128, true>(mq, mk, mv, p, grid, stream) : launch<128, false>(mq, mk, mv, p, grid, stream);
}

int fa_fwd_status(cudaStream_t stream, unsigned int* detail, int clear) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_LAUNCH;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, fa::g_fa_status, sizeof(word)) != cudaSuccess) return FA_ERR_LAUNCH;
  if (detail) *detail = word;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return word ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"
