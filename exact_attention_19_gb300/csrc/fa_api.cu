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
#include "fa_fwd_persist.cuh"
#include "fa_bwd_kernel.cuh"

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
int g_dev_sms[kMaxDevices];  // multiprocessor count, valid once the state is 1
long long g_dev_l2[kMaxDevices];  // L2 bytes, valid once the state is 1

int g_dev_sms_or(int dev, int fallback) {
  return (dev >= 0 && dev < kMaxDevices && g_dev_sms[dev] > 0) ? g_dev_sms[dev] : fallback;
}
std::mutex g_dev_mutex;

// A kernel that moves registers between warpgroups with setmaxnreg assumes
// the register count it is launched with; with any other count an increase
// could wait forever, so the library refuses such a build.
template <typename K>
bool launch_regs_are(K kernel, int regs) {
  cudaFuncAttributes a;
  return cudaFuncGetAttributes(&a, kernel) == cudaSuccess && a.numRegs == regs;
}

template <int D, int MASK, bool SPLIT, int TILES = 2>
cudaError_t set_smem_attr() {
  if (TILES == 2 && !launch_regs_are(fa::fa_fwd_kernel<D, MASK, SPLIT, TILES>, fa::Cfg<D, TILES>::kRegLaunch))
    return cudaErrorInvalidDeviceFunction;
  return cudaFuncSetAttribute(fa::fa_fwd_kernel<D, MASK, SPLIT, TILES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::Cfg<D, TILES>::kSmemBytes));
}

template <int D, int MASK>
bool set_persist_attr() {
  return launch_regs_are(fa::fa_fwd_persist_kernel<D, MASK>, fa::PCfg<D>::kRegLaunch) &&
         cudaFuncSetAttribute(fa::fa_fwd_persist_kernel<D, MASK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::PCfg<D>::kSmemBytes)) == cudaSuccess;
}

template <int D, int MASK>
bool set_bwd_smem_attr() {
  using C = fa::BwdCfg<D>;
  return cudaFuncSetAttribute(fa::fa_bwd_dq_kernel<D, MASK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(C::kSmemQ)) == cudaSuccess &&
         cudaFuncSetAttribute(fa::fa_bwd_dkdv_kernel<D, MASK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(C::kSmemKV)) == cudaSuccess;
}

template <int D>
bool set_bwd_smem_attrs() {
  return set_bwd_smem_attr<D, fa::kBwdMaskNone>() && set_bwd_smem_attr<D, fa::kBwdMaskCausal>() &&
         set_bwd_smem_attr<D, fa::kBwdMaskWindow>();
}

template <int D>
bool set_smem_attrs() {
  bool ok = set_smem_attr<D, fa::kMaskNone, false>() == cudaSuccess &&
            set_smem_attr<D, fa::kMaskCausal, false>() == cudaSuccess &&
            set_smem_attr<D, fa::kMaskWindow, false>() == cudaSuccess &&
            set_smem_attr<D, fa::kMaskNone, true>() == cudaSuccess &&
            set_smem_attr<D, fa::kMaskCausal, true>() == cudaSuccess;
  ok = ok && set_persist_attr<D, fa::kMaskNone>() && set_persist_attr<D, fa::kMaskCausal>() &&
       set_persist_attr<D, fa::kMaskWindow>();
  if constexpr (D == 64)
    ok = ok && set_smem_attr<64, fa::kMaskCausal, false, 1>() == cudaSuccess &&
         set_smem_attr<64, fa::kMaskNone, true, 1>() == cudaSuccess &&
         set_smem_attr<64, fa::kMaskCausal, true, 1>() == cudaSuccess;
  return ok;
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
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return FA_ERR_LAUNCH;
  g_dev_sms[dev] = sms;
  int l2 = 0;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 <= 0) return FA_ERR_LAUNCH;
  g_dev_l2[dev] = l2;
  if (!set_smem_attrs<64>() || !set_smem_attrs<128>() || !set_bwd_smem_attrs<64>() || !set_bwd_smem_attrs<128>())
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

template <int D, int MASK, bool SPLIT, int TILES = 2>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
           const fa::FwdParams& p,
           long long grid, cudaStream_t stream) {
  using C = fa::Cfg<D, TILES>;
  fa::fa_fwd_kernel<D, MASK, SPLIT, TILES><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, stream>>>(
      mq, mk, mv, mo, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Single query tile per CTA (two CTAs per SM) for causal attention at d = 64
// over at most this many keys: there the fixed per-CTA cost weighs most
// (8 x 12 x 1024: +5.5%, 2 x 4 x 2048: +8%; 4 x 32 x 8192: -10%, so longer
// key ranges keep two tiles per CTA).
constexpr int kSingleTileMaxKeys = 2048;
// d = 64 without a mask: the persistent kernel up to this many keys (4 x 32 x
// 8192: 1.6% slower than one CTA per unit; 8 x 12 x 1024: 9% faster).
constexpr int kPersistD64MaxKeys = 2048;
// Causal d = 64 beyond kSingleTileMaxKeys keys: the persistent kernel under
// cluster launch control once there are this many query-tile pairs per SM
// (fewer, and single tiles balance better: causal 4 x 16 x 3072, 5 pairs per
// SM, 6% faster on single tiles; 4 x 16 x 4096, 6.7 per SM, 2.5% slower).
constexpr int kClcMinUnitsPerSm = 6;
// Causal d = 128: the same dynamic schedule from this many pairs per SM
// (4 x 32 x 8192, 27 per SM: +1%; 1 x 16 x 32000, 13 per SM with units of up
// to 250 K/V tiles: 4.6% slower, so one CTA per unit there).
constexpr int kClcMinUnitsPerSm128 = 20;
// A window bounded on both sides with Nq <= Nk (every row sees a key, units
// of about equal length): the persistent kernel's static schedule from this
// many query-tile pairs per SM (4 x 32 x 8192 d = 64 band of 1024 keys: +6%;
// 2 x 16 x 4096, 1.7 pairs per SM: 3% slower).  A band open on one side gives
// units of unequal length, which the static schedule balances badly.
constexpr int kPersistWindowMinUnitsPerSm = 4;

// no mask or the causal mask (split or not)
template <int D, bool SPLIT>
int launch_d(bool causal, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
             const CUtensorMap& mo, const fa::FwdParams& p, long long grid, cudaStream_t stream) {
  return causal ? launch<D, fa::kMaskCausal, SPLIT>(mq, mk, mv, mo, p, grid, stream)
                : launch<D, fa::kMaskNone, SPLIT>(mq, mk, mv, mo, p, grid, stream);
}

template <int D, int MASK>
int launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
               const CUtensorMap& mdq, const CUtensorMap& mdk, const CUtensorMap& mdv, const fa::BwdParams& p,
               long long bh, cudaStream_t stream) {
  using C = fa::BwdCfg<D>;
  fa::fa_bwd_dq_kernel<D, MASK><<<static_cast<unsigned>(bh * p.n_qt), C::kThreads, C::kSmemQ, stream>>>(
      mq, mk, mv, mdo, mdq, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  fa::fa_bwd_dkdv_kernel<D, MASK><<<static_cast<unsigned>(bh * p.n_kt), C::kThreads, C::kSmemKV, stream>>>(
      mq, mk, mv, mdo, mdk, mdv, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Host-only checks shared by fa_fwd, fa_fwd_window and both split-KV entry
// points, in the order fa.h documents; nothing here touches the device.
// *noop is set when Nq == 0 (nothing is read or written).
int check_args(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
               int d, float scale, int causal, bool* noop) {
  *noop = false;
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
  // tensor-map limits: a stride below 2^40 bytes, grid below 2^31 CTAs
  if (static_cast<long long>(Nq > Nk ? Nq : Nk) * d * 2 >= (1ll << 40)) return FA_ERR_SHAPE;
  if (BH >= (1ll << 31) || BH * n_pairs >= (1ll << 31)) return FA_ERR_SHAPE;
  if (Nq == 0) *noop = true;
  return FA_OK;
}

// The device side of a forward call whose arguments passed check_args (with
// Nq > 0): the current device, its one-time set-up, the pointer checks, the
// TMA tensor maps and the parameters common to every forward kernel.
int prepare_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                   int d, float scale, int causal, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv,
                   CUtensorMap* mo, fa::FwdParams* p, int* dev_out) {
  const long long BH = static_cast<long long>(B) * H;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_LAUNCH;
  const int prep = prepare_device(dev);
  if (prep != FA_OK) return prep;
  if (!is_device_pointer(q, dev) || !is_device_pointer(k, dev) || !is_device_pointer(v, dev) ||
      !is_device_pointer(o, dev) || !is_device_pointer(lse, dev))
    return FA_ERR_POINTER;
  if (!make_map(mq, q, d, Nq, BH) || !make_map(mk, k, d, Nk, BH) || !make_map(mv, v, d, Nk, BH) ||
      !make_map(mo, o, d, Nq, BH))
    return FA_ERR_LAUNCH;
  p->o = o;
  p->lse = lse;
  p->Nq = Nq;
  p->Nk = Nk;
  p->n_pairs = static_cast<int>((static_cast<long long>(Nq) + 255) / 256);
  p->scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  // causal = the window (-1, 0) on the main diagonal (Nq == Nk here)
  p->win_left = -1;
  p->win_right = causal ? 0 : -1;
  p->diag_off = 0;
  p->n_splits = 1;
  p->split_tiles = 0;
  p->o_part = nullptr;
  p->lse_part = nullptr;
  p->rows = BH * Nq;
  // heads per causal scheduling group: their K and V fill at most a quarter
  // of the L2 (with half, a cold causal 4 x 32 x 8192 launch re-read 350 MB of
  // K/V from DRAM; with a quarter it reads Q, K, V once)
  const long long kv_head_bytes = 4ll * Nk * d;
  const long long group = (g_dev_l2[dev] / 4) / (kv_head_bytes > 0 ? kv_head_bytes : 1);
  p->lpt_group = static_cast<int>(group < 1 ? 1 : (group > BH ? BH : group));
  *dev_out = dev;
  return FA_OK;
}

// check_args then prepare_launch; *noop is set (and nothing else done) when Nq == 0.
int prepare_call(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                 int d, float scale, int causal, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv,
                 CUtensorMap* mo, fa::FwdParams* p, int* dev_out, bool* noop) {
  const int st = check_args(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, noop);
  if (st != FA_OK || *noop) return st;
  return prepare_launch(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, mq, mk, mv, mo, p, dev_out);
}

// K/V tiles per split and the number of non-empty splits for a request.
void split_shape(int Nk, int n_splits, int* split_tiles, int* eff_splits) {
  const int n_kv = (Nk + 127) / 128;
  const int req = n_splits < 1 ? 1 : (n_splits > n_kv ? n_kv : n_splits);
  *split_tiles = (n_kv + req - 1) / req;
  *eff_splits = (n_kv + *split_tiles - 1) / *split_tiles;
}

// The persistent kernel: one CTA per multiprocessor, at most one per work
// unit (a head's pair of 128-row query tiles).
template <int D>
int launch_persist(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const fa::FwdParams& p,
                   long long n_units, int sms, cudaStream_t stream) {
  using C = fa::PCfg<D>;
  if (n_units >= (1ll << 31)) return FA_ERR_SHAPE;
  const long long grid = n_units < sms ? n_units : sms;
  fa::fa_fwd_persist_kernel<D, fa::kMaskNone><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, stream>>>(
      mq, mk, mv, p, static_cast<int>(n_units));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// The causal persistent kernel: one CTA per unit in the causal launch order;
// running CTAs take over the ones not yet started (cluster launch control).
template <int D>
int launch_persist_causal(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                          const fa::FwdParams& p, long long n_units, cudaStream_t stream) {
  using C = fa::PCfg<D>;
  if (n_units >= (1ll << 31)) return FA_ERR_SHAPE;
  fa::fa_fwd_persist_kernel<D, fa::kMaskCausal>
      <<<static_cast<unsigned>(n_units), C::kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, p, static_cast<int>(n_units));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Single-pass forward (no mask or causal) on prepared maps and parameters.
// Without a mask, at d = 128 or at d = 64 with at most kPersistD64MaxKeys
// keys: the persistent kernel (units of equal length, balanced by its static
// schedule; at d = 64 it pays only on short units).  Causal at d = 64: single
// query tiles, two CTAs per SM, up to kSingleTileMaxKeys keys or below
// kClcMinUnitsPerSm pairs per SM; beyond, the persistent kernel under cluster
// launch control (4 x 32 x 8192: +5%).
// Causal at d = 128: the dynamic persistent schedule from kClcMinUnitsPerSm128
// pairs per SM; below, one CTA per unit, so the hardware's dispatch balances
// long units of unequal length in their longest-first launch order.
int launch_single_pass(int B, int H, int Nq, int Nk, int d, int causal, const CUtensorMap& mq,
                       const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo, fa::FwdParams p,
                       int dev, cudaStream_t stream) {
  const long long n_units = static_cast<long long>(B) * H * p.n_pairs;  // query-tile pairs
  if (!causal && (d == 128 || Nk <= kPersistD64MaxKeys)) {
    return d == 64 ? launch_persist<64>(mq, mk, mv, p, n_units, g_dev_sms_or(dev, 148), stream)
                   : launch_persist<128>(mq, mk, mv, p, n_units, g_dev_sms_or(dev, 148), stream);
  }
  if (d == 64 && causal &&
      (Nk <= kSingleTileMaxKeys || n_units < kClcMinUnitsPerSm * static_cast<long long>(g_dev_sms_or(dev, 148)))) {
    p.n_pairs = (Nq + 127) / 128;  // one query tile per CTA
    const long long grid = static_cast<long long>(B) * H * p.n_pairs;
    if (grid >= (1ll << 31)) return FA_ERR_SHAPE;
    return launch<64, fa::kMaskCausal, false, 1>(mq, mk, mv, mo, p, grid, stream);
  }
  if (d == 64 && causal) return launch_persist_causal<64>(mq, mk, mv, p, n_units, stream);
  if (causal && n_units >= kClcMinUnitsPerSm128 * static_cast<long long>(g_dev_sms_or(dev, 148)))
    return launch_persist_causal<128>(mq, mk, mv, p, n_units, stream);
  const long long grid = static_cast<long long>(B) * H * p.n_pairs;
  return d == 64 ? launch_d<64, false>(causal, mq, mk, mv, mo, p, grid, stream)
                 : launch_d<128, false>(causal, mq, mk, mv, mo, p, grid, stream);
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
    case FA_ERR_WORKSPACE: return "split-KV workspace is missing or smaller than fa_splitkv_workspace_bytes()";
    default: return "unknown status";
  }
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
           int d, float scale, int causal, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo;
  fa::FwdParams p;
  int dev = -1;
  bool noop = false;
  const int st = prepare_call(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, &mq, &mk, &mv, &mo, &p, &dev, &noop);
  if (st != FA_OK || noop) return st;
  return launch_single_pass(B, H, Nq, Nk, d, causal, mq, mk, mv, mo, p, dev, stream);
}

int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                  int Nk, int d, float scale, int window_left, int window_right, cudaStream_t stream) {
  if (window_left < -1 || window_right < -1) return FA_ERR_SHAPE;
  CUtensorMap mq, mk, mv, mo;
  fa::FwdParams p;
  int dev = -1;
  bool noop = false;
  const int st = prepare_call(q, k, v, o, lse, B, H, Nq, Nk, d, scale, 0, &mq, &mk, &mv, &mo, &p, &dev, &noop);
  if (st != FA_OK || noop) return st;
  p.win_left = window_left;
  p.win_right = window_right;
  p.diag_off = Nk - Nq;  // bottom-right: the window's diagonal ends at (Nq - 1, Nk - 1)
  const long long grid = static_cast<long long>(B) * H * p.n_pairs;  // one CTA per query-tile pair
  const int sms = g_dev_sms_or(dev, 148);
  if (window_left >= 0 && window_right >= 0 && Nq <= Nk && grid < (1ll << 31) &&
      grid >= kPersistWindowMinUnitsPerSm * static_cast<long long>(sms)) {
    const unsigned pgrid = static_cast<unsigned>(grid < sms ? grid : sms);
    if (d == 64)
      fa::fa_fwd_persist_kernel<64, fa::kMaskWindow><<<pgrid, fa::PCfg<64>::kThreads, fa::PCfg<64>::kSmemBytes, stream>>>(
          mq, mk, mv, p, static_cast<int>(grid));
    else
      fa::fa_fwd_persist_kernel<128, fa::kMaskWindow><<<pgrid, fa::PCfg<128>::kThreads, fa::PCfg<128>::kSmemBytes, stream>>>(
          mq, mk, mv, p, static_cast<int>(grid));
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
  }
  if (window_left < 0 && window_right < 0)  // no bound on either side: no mask
    return d == 64 ? launch<64, fa::kMaskNone, false>(mq, mk, mv, mo, p, grid, stream)
                   : launch<128, fa::kMaskNone, false>(mq, mk, mv, mo, p, grid, stream);
  return d == 64 ? launch<64, fa::kMaskWindow, false>(mq, mk, mv, mo, p, grid, stream)
                 : launch<128, fa::kMaskWindow, false>(mq, mk, mv, mo, p, grid, stream);
}

size_t fa_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int n_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
  int tiles = 0, eff = 0;
  split_shape(Nk, n_splits, &tiles, &eff);
  const size_t rows = static_cast<size_t>(B) * H * Nq;
  return static_cast<size_t>(eff) * rows * (static_cast<size_t>(d) + 1) * sizeof(float);
}

int fa_splitkv_heuristic(int B, int H, int Nq, int Nk, int d, int causal) {
  (void)d;
  (void)causal;
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return 1;
  int dev = -1, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess && prepare_device(dev) == FA_OK) sms = g_dev_sms_or(dev, sms);
  const long long ctas = static_cast<long long>(B) * H * ((static_cast<long long>(Nq) + 255) / 256);
  if (ctas >= sms) return 1;
  const int n_kv = (Nk + 127) / 128;
  long long want = sms / ctas;  // fill the SMs once
  if (want > 16) want = 16;
  if (want > n_kv / 2) want = n_kv / 2;  // a slice of one tile costs more than it saves
  int tiles = 0, eff = 0;
  split_shape(Nk, static_cast<int>(want < 1 ? 1 : want), &tiles, &eff);
  return eff;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free split-KV: the slice buffers of fa_fwd_splitkv_noalloc.  For
// callers that may not allocate device memory themselves (a host framework
// that owns the whole device pool, or a latency path where a cudaMalloc and
// its implicit synchronisation are not allowed), they live in one fixed array
// in the library's own device memory.  Each GPU that loads the library holds
// this array until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {
std::atomic<void*> g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device
std::mutex g_noalloc_mutex;

// The host-side name of a __device__ array is only a stand-in; the address a
// kernel may use is asked of the runtime once per device, with that device
// current, and cached (later calls take the lock-free path).
void* noalloc_scratch(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  void* ptr = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (ptr) return ptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  ptr = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_noalloc_ptr[dev].store(ptr, std::memory_order_release);
  }
  return ptr;
}

// Both split-KV entry points.  Checks run in one order for both: the host
// checks of fa_fwd (and the Nq == 0 no-op), then, for the allocation-free
// call, the size limit of the fixed array, then the device and pointer checks,
// and only then the workspace: the caller's, or the fixed array's address.
int splitkv_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                 int d, float scale, int causal, int n_splits, void* workspace, size_t workspace_bytes,
                 bool noalloc, cudaStream_t stream) {
  if (n_splits < 1 || n_splits > 64) return FA_ERR_SHAPE;
  bool noop = false;
  int st = check_args(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, &noop);
  if (st != FA_OK || noop) return st;
  int tiles = 0, eff = 0;
  split_shape(Nk, n_splits, &tiles, &eff);
  // one slice runs the plain kernel and needs no workspace
  const size_t need = eff > 1 ? fa_splitkv_workspace_bytes(B, H, Nq, Nk, d, n_splits) : 0;
  if (noalloc && need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  CUtensorMap mq, mk, mv, mo;
  fa::FwdParams p;
  int dev = -1;
  st = prepare_launch(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, &mq, &mk, &mv, &mo, &p, &dev);
  if (st != FA_OK) return st;
  if (eff == 1) return launch_single_pass(B, H, Nq, Nk, d, causal, mq, mk, mv, mo, p, dev, stream);
  if (noalloc) {
    // Every partial the merge reads is written earlier in the same call (an
    // empty slice writes weight 2^-inf), so nothing in the array is cleared.
    workspace = noalloc_scratch(dev);
    if (!workspace) return FA_ERR_LAUNCH;
  } else {
    if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_ALIGN;
    if (!is_device_pointer(workspace, dev)) return FA_ERR_POINTER;
  }
  p.n_splits = eff;
  p.split_tiles = tiles;
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = p.o_part + static_cast<size_t>(eff) * p.rows * d;
  // d = 64: one query tile per CTA (two CTAs per SM) when the grid of
  // query-tile pairs would leave more than half of the SMs idle or spill into
  // a second wave; single tiles double the CTAs and halve each one's work
  const long long pair_grid = static_cast<long long>(B) * H * p.n_pairs * eff;
  const int sms = g_dev_sms_or(dev, 148);
  const bool single = d == 64 && (2 * pair_grid < sms || pair_grid > sms);
  if (single) p.n_pairs = (Nq + 127) / 128;
  const long long grid = static_cast<long long>(B) * H * p.n_pairs * eff;
  if (grid >= (1ll << 31)) return FA_ERR_SHAPE;
  int rc;
  if (single)
    rc = causal ? launch<64, fa::kMaskCausal, true, 1>(mq, mk, mv, mo, p, grid, stream)
                : launch<64, fa::kMaskNone, true, 1>(mq, mk, mv, mo, p, grid, stream);
  else
    rc = d == 64 ? launch_d<64, true>(causal, mq, mk, mv, mo, p, grid, stream)
                 : launch_d<128, true>(causal, mq, mk, mv, mo, p, grid, stream);
  if (rc != FA_OK) return rc;
  // The merge is a programmatic dependent launch: its CTAs may be scheduled
  // while the sliced kernel's last CTAs run, and wait in the kernel for its
  // completion, so its launch latency overlaps the forward's tail.
  const long long cgrid = (p.rows + 7) / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cgrid));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float* o_part = p.o_part;
  const float* lse_part = p.lse_part;
  const long long rows = p.rows;
  const cudaError_t e = d == 64
                            ? cudaLaunchKernelEx(&cfg, fa::fa_splitkv_combine_kernel<64>, o_part, lse_part, o, lse, rows, eff)
                            : cudaLaunchKernelEx(&cfg, fa::fa_splitkv_combine_kernel<128>, o_part, lse_part, o, lse, rows, eff);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? FA_OK : FA_ERR_LAUNCH;
}
}  // namespace

extern "C" {

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                   int d, float scale, int causal, int n_splits, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream) {
  return splitkv_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, n_splits, workspace, workspace_bytes, false,
                      stream);
}

int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                           int Nk, int d, float scale, int causal, int n_splits, cudaStream_t stream) {
  return splitkv_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, n_splits, nullptr, 0, true, stream);
}

// ---------------------------------------------------------------------------
// Backward pass
// ---------------------------------------------------------------------------
size_t fa_bwd_workspace_bytes(int B, int H, int Nq) {
  if (B <= 0 || H <= 0 || Nq <= 0) return 0;
  const size_t nq_pad = (static_cast<size_t>(Nq) + 127) / 128 * 128;
  return 2 * static_cast<size_t>(B) * H * nq_pad * sizeof(float);
}

}  // extern "C"

namespace {

// The backward under one of the three masks, with the checks shared by
// fa_bwd and fa_bwd_window in the order fa.h documents (`causal` is fa_bwd's
// argument, 0 for a window).
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal, int mask,
             int window_left, int window_right, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv, workspace};
  for (const void* x : ptrs)
    if (!x) return FA_ERR_NULL;
  for (const void* x : ptrs)
    if (reinterpret_cast<uintptr_t>(x) & 15u) return FA_ERR_ALIGN;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return FA_ERR_SHAPE;
  if (causal != 0 && causal != 1) return FA_ERR_SHAPE;
  if (causal && Nq != Nk) return FA_ERR_CAUSAL_SHAPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  const long long BH = static_cast<long long>(B) * H;
  const long long n_qt = (static_cast<long long>(Nq) + 127) / 128, n_kt = (static_cast<long long>(Nk) + 127) / 128;
  if (static_cast<long long>(Nq > Nk ? Nq : Nk) * d * 2 >= (1ll << 40)) return FA_ERR_SHAPE;
  if (BH >= (1ll << 31) || BH * n_qt >= (1ll << 31) || BH * n_kt >= (1ll << 31)) return FA_ERR_SHAPE;
  if (workspace_bytes < fa_bwd_workspace_bytes(B, H, Nq)) return FA_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_LAUNCH;
  const int prep = prepare_device(dev);
  if (prep != FA_OK) return prep;
  for (const void* x : ptrs)
    if (!is_device_pointer(x, dev)) return FA_ERR_POINTER;
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  if (!make_map(&mq, q, d, Nq, BH) || !make_map(&mk, k, d, Nk, BH) || !make_map(&mv, v, d, Nk, BH) ||
      !make_map(&mdo, dout, d, Nq, BH) || !make_map(&mdq, dq, d, Nq, BH) || !make_map(&mdk, dk, d, Nk, BH) ||
      !make_map(&mdv, dv, d, Nk, BH))
    return FA_ERR_LAUNCH;
  fa::BwdParams p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qt = static_cast<int>(n_qt);
  p.n_kt = static_cast<int>(n_kt);
  p.Nq_pad = static_cast<int>(n_qt * 128);
  p.lse2 = static_cast<float*>(workspace);
  p.dsum = p.lse2 + static_cast<size_t>(BH) * p.Nq_pad;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.win_left = window_left;
  p.win_right = window_right;
  p.diag_off = Nk - Nq;  // bottom-right, as in the forward
  if (mask == fa::kBwdMaskWindow)
    return d == 64 ? launch_bwd<64, fa::kBwdMaskWindow>(mq, mk, mv, mdo, mdq, mdk, mdv, p, BH, stream)
                   : launch_bwd<128, fa::kBwdMaskWindow>(mq, mk, mv, mdo, mdq, mdk, mdv, p, BH, stream);
  if (mask == fa::kBwdMaskCausal)
    return d == 64 ? launch_bwd<64, fa::kBwdMaskCausal>(mq, mk, mv, mdo, mdq, mdk, mdv, p, BH, stream)
                   : launch_bwd<128, fa::kBwdMaskCausal>(mq, mk, mv, mdo, mdq, mdk, mdv, p, BH, stream);
  return d == 64 ? launch_bwd<64, fa::kBwdMaskNone>(mq, mk, mv, mdo, mdq, mdk, mdv, p, BH, stream)
                 : launch_bwd<128, fa::kBwdMaskNone>(mq, mk, mv, mdo, mdq, mdk, mdv, p, BH, stream);
}

}  // namespace

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
           void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal, void* workspace,
           size_t workspace_bytes, cudaStream_t stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, causal,
                  causal == 1 ? fa::kBwdMaskCausal : fa::kBwdMaskNone, -1, -1, workspace, workspace_bytes, stream);
}

int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                  void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int window_left,
                  int window_right, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (window_left < -1 || window_right < -1) return FA_ERR_SHAPE;
  const int mask = (window_left < 0 && window_right < 0) ? fa::kBwdMaskNone : fa::kBwdMaskWindow;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, 0, mask, window_left, window_right,
                  workspace, workspace_bytes, stream);
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
