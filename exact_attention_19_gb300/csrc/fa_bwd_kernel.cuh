// fa_bwd_kernel.cuh -- the attention backward pass for sm_103a, by
// recomputation from the forward's LSE (page "llm-infra-atlas /
// FlashAttention 01", section 5: P = exp(S * scale - LSE), dV = P^T dO,
// dP = dO V^T, dS = P (dP - rowsum(dO O)), dQ = dS K * scale, dK = dS^T Q * scale).
//
// Two kernels, no atomics (the result is deterministic):
//   fa_bwd_dq_kernel    one CTA per 128-row query tile: streams K_j, V_j and
//                       accumulates dQ in TMEM; also writes, for the second
//                       kernel, L = LSE * log2(e) and D = rowsum(dO * O) per
//                       query, padded to whole query tiles (+inf and 0 past Nq).
//   fa_bwd_dkdv_kernel  one CTA per 128-key tile, keys on TMEM lanes: streams
//                       Q_i, dO_i (with their L and D) and accumulates dK, dV.
// Both use the tcgen05 forms of the forward kernel: SS MMAs with K-major
// operands for the two score-shaped products, TS MMAs (A = bf16 probabilities
// or score gradients from TMEM, B = an MN-major tile from shared memory) for
// the three accumulations.  Roles: warps 0-7 compute, warp 8 TMA producer,
// warp 9 TMEM allocation and MMA issue.  Compute warp 4h + q holds TMEM lanes
// 32q..32q+31 (one row per thread) and column half h of every 128-column
// tile: the elementwise work (P from the stored L, dS from the stored D) needs
// no reduction along a row, so the two halves never communicate, and two
// warps per SM sub-partition keep twice the exponentials in flight.  Each half
// writes its bf16 results into its own columns (64h..64h+31), so no half
// overwrites values the other has yet to read; the MMAs take their A operand
// from columns 64 (kk / 4) + 8 (kk % 4).  The gradients leave through TMA
// tensor stores, staged in bf16 in the resident tiles' buffers (Q for dQ, K and
// V for dK and dV) once the last MMA has read them.  Every wait is bounded as
// in the forward kernel.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "fa_ptx.cuh"

namespace fa {

struct BwdParams {
  const void* o;      // bf16 [BH, Nq, D] forward output
  const void* dout;   // bf16 [BH, Nq, D]
  const float* lse;   // fp32 [BH, Nq] forward LSE (natural log)
  void* dq;           // bf16 [BH, Nq, D]
  void* dk;           // bf16 [BH, Nk, D]
  void* dv;           // bf16 [BH, Nk, D]
  float* lse2;        // workspace fp32 [BH, Nq_pad]: LSE * log2(e), +inf past Nq
  float* dsum;        // workspace fp32 [BH, Nq_pad]: rowsum(dO * O), 0 past Nq
  int Nq, Nk, Nq_pad;
  int n_qt, n_kt;     // query / key tiles per head
  float scale;        // softmax scale
  float scale_log2;   // scale * log2(e)
  // window mask only: key j is kept for query row i iff
  //   i + diag_off - win_left <= j <= i + diag_off + win_right  (a negative bound: that side open)
  int win_left, win_right, diag_off;
};

// kBwdMaskCausal: key j kept for row i iff j <= i (Nq == Nk); kBwdMaskWindow:
// the general window of BwdParams (the forward's reading of the "sliding" mask
// named in page "llm-infra-atlas / FlashAttention 01", section 3).  Each kernel then visits only the tiles its
// rows (keys) can see; a tile that sees none writes zero gradients.
enum : int { kBwdMaskNone = 0, kBwdMaskCausal = 1, kBwdMaskWindow = 2 };

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kThreads = 320;
  static constexpr int kBoxes = D / 64;
  static constexpr uint32_t kBoxBytes = 128u * 128u;
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;  // 128 rows x D bf16
  static constexpr int kRingQ = (D == 128) ? 5 : 8;           // dQ kernel: K/V ring slots
  static constexpr int kRingKV = (D == 128) ? 4 : 8;          // dK/dV kernel: Q/dO ring slots
  static constexpr uint32_t kSideBytes = 1024;                // L and D of one query tile
  // dQ kernel smem: Q, dO, ring
  static constexpr uint32_t kQRingOff = 2 * kTileBytes;
  static constexpr uint32_t kQBarOff = kQRingOff + kRingQ * kTileBytes;
  // dK/dV kernel smem: K, V, ring, side buffers
  static constexpr uint32_t kKVRingOff = 2 * kTileBytes;
  static constexpr uint32_t kKVSideOff = kKVRingOff + kRingKV * kTileBytes;
  static constexpr uint32_t kKVBarOff = kKVSideOff + kRingKV * kSideBytes;
  static constexpr uint32_t kBarBytes = 512;
  static constexpr uint32_t kQPartOff = kQBarOff + kBarBytes;  // dQ kernel: half-row sums of D (2 x 128 fp32)
  static constexpr uint32_t kSmemQ = kQPartOff + 1024 + 1024;
  static constexpr uint32_t kSmemKV = kKVBarOff + kBarBytes + 1024;
  static constexpr uint32_t kIdescScore = idesc_bf16(128, 128, false);  // 128 x 128 over d
  static constexpr uint32_t kIdescAcc = idesc_bf16(128, D, true);       // 128 x D over 128 rows
  static_assert(kSmemQ <= 232448 && kSmemKV <= 232448, "shared memory budget");
};

// ---------------------------------------------------------------------------
// dQ kernel
// ---------------------------------------------------------------------------
// barriers: 0 q_full, 1 s_full, 2 dp_full, 3 s_free, 4 ds_full, 5 dq_full,
// 6 drain, 7..10 the D half-sum exchange (one per TMEM lane quarter), then
// ring full[kRingQ], empty[kRingQ], then the epilogue's staging barrier
template <int D, int MASK>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int R = C::kRingQ;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw_addr);
  const uint32_t bar0 = base + C::kQBarOff;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto full = [&](int s) -> uint32_t { return bar(11 + s); };
  auto empty = [&](int s) -> uint32_t { return bar(11 + R + s); };
  auto slot_addr = [&](int s) -> uint32_t { return base + C::kQRingOff + s * C::kTileBytes; };
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + C::kQBarOff + 448);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sbase + C::kQBarOff + 452);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(0), 1);
    mbar_init(bar(1), 1);
    mbar_init(bar(2), 1);
    mbar_init(bar(3), 256);
    mbar_init(bar(4), 256);
    mbar_init(bar(5), 1);
    mbar_init(bar(6), 1);
    for (int q = 0; q < 4; ++q) mbar_init(bar(7 + q), 64);
    for (int s = 0; s < R; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(bar(11 + 2 * R), 256);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM: S [0,128), two dP buffers [128,256) and [256,384) (K/V tile j uses
  // buffer j % 2; dS_j overwrites part of it), dQ [384, 384 + D)
  constexpr uint32_t kTmS = 0, kTmDP = 128, kTmDQ = 384;
  static_assert(kTmDQ + D <= 512, "TMEM columns");

  const int bh = blockIdx.x / p.n_qt;
  int qt = blockIdx.x % p.n_qt;
  if (MASK == kBwdMaskCausal) qt = p.n_qt - 1 - qt;  // heaviest tile of each head first
  const int row0 = qt * 128;
  const int n_kv_all = (p.Nk + 127) / 128;
  // visible K/V tiles [jlo, jlo + nkv) of this query tile; only a window
  // can leave a tile with none (any_kv is a compile-time true otherwise)
  int jlo = 0, nkv = n_kv_all;
  if (MASK == kBwdMaskCausal) nkv = min(n_kv_all, qt + 1);
  if (MASK == kBwdMaskWindow) {
    const long long r_first = row0, r_last = min(row0 + 128, p.Nq) - 1;
    long long key_lo = 0, key_hi = p.Nk - 1;
    if (p.win_left >= 0) key_lo = max(0ll, r_first + p.diag_off - p.win_left);
    if (p.win_right >= 0) key_hi = min(key_hi, r_last + p.diag_off + p.win_right);
    if (key_lo > key_hi) {
      nkv = 0;  // no row of this tile sees a key: dQ = 0
    } else {
      jlo = static_cast<int>(key_lo / 128);
      nkv = static_cast<int>(key_hi / 128) + 1 - jlo;
    }
  }
  const bool any_kv = MASK != kBwdMaskWindow || nkv > 0;

  if (warp == 8) {
    // ======================= TMA producer =================================
    if (lane == 0 && any_kv) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmDO);
      tma_prefetch_map(&tmDQ);
      mbar_arrive_expect_tx(bar(0), 2 * C::kTileBytes);
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_3d(base + b * C::kBoxBytes, &tmQ, bar(0), b * 64, row0, bh);
        tma_load_3d(base + C::kTileBytes + b * C::kBoxBytes, &tmDO, bar(0), b * 64, row0, bh);
      }
      int item = 0;
      bool ok = true;
      // V_0, K_0, V_1, K_1, ...: V_j is done early (after dP_j), K_j late (after
      // dQ_j), so each V reuses the slot of a K released two tiles before
      for (; item < 2 * nkv; ++item) {
        const int s = item % R;
        if (!(ok = mbar_wait(empty(s), ((item / R) & 1) ^ 1u, abort_flag))) break;
        mbar_arrive_expect_tx(full(s), C::kTileBytes);
        for (int b = 0; b < C::kBoxes; ++b)
          tma_load_3d(slot_addr(s) + b * C::kBoxBytes, (item & 1) ? &tmK : &tmV, full(s), b * 64,
                      (jlo + (item >> 1)) * 128, bh);
      }
      if (!ok) report_wait_failure(abort_flag, 2u);
      if (*abort_flag) {
        for (int it = max(0, item - R); it < item; ++it) mbar_wait(full(it % R), (it / R) & 1, nullptr);
        mbar_wait(bar(0), 0, nullptr);
      }
    }
  } else if (warp == 9) {
    // ======================= MMA issuer ====================================
    // The whole warp runs the issue loop on warp-uniform values (every barrier
    // outcome made uniform with a vote); one lane chosen by elect.sync issues
    // each tcgen05.mma and commit, with no branch around the instruction
    // (same-box A/B against lane 0 alone: +6.5% to +11.5%).
    auto uniform = [](bool v) -> bool { return __all_sync(0xffffffffu, v); };
    {
      const uint64_t dQd = sdesc_sw128(base, 16, 1024);                   // Q, K-major
      const uint64_t dDOd = sdesc_sw128(base + C::kTileBytes, 16, 1024);  // dO, K-major
      const uint64_t dRingK = sdesc_sw128(base + C::kQRingOff, 16, 1024);
      const uint64_t dRingMN = sdesc_sw128(base + C::kQRingOff, C::kBoxBytes, 1024);
      auto slot_off = [&](int s) -> uint64_t { return (s * C::kTileBytes) >> 4; };
      // S = Q K_j^T or dP = dO V_j^T: 128 x 128 over d, both K-major
      auto score = [&](uint64_t da, int s, uint32_t dst) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tmem + dst, da + off, dRingK + slot_off(s) + off, C::kIdescScore, kk > 0 ? 1u : 0u);
        }
      };
      // dQ += dS_j K_j: A = dS_j from TMEM (packed bf16 in dP buffer j % 2, keys
      // 16kk.. at column 64 (kk / 4) + 8 (kk % 4)), B = K_j MN-major
      auto acc_dq = [&](int s, uint32_t dp_buf, bool acc_prev) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_elect(tmem + kTmDQ, tmem + dp_buf + (kk >> 2) * 64 + (kk & 3) * 8,
                 dRingMN + slot_off(s) + ((kk * 2048) >> 4), C::kIdescAcc, (acc_prev || kk > 0) ? 1u : 0u);
      };
      auto wait_item = [&](int it) -> bool { return uniform(mbar_wait(full(it % R), (it / R) & 1, abort_flag)); };
      // ring items: V_j = 2j, K_j = 2j + 1 (tile jlo + j)
      bool ok = !any_kv || (uniform(mbar_wait(bar(0), 0, abort_flag)) && wait_item(0) && wait_item(1));
      if (ok && any_kv) {
        tc_fence_after();
        score(dQd, 1, kTmS);
        mma_commit_elect(bar(1));
        score(dDOd, 0, kTmDP);
        mma_commit_elect(bar(2));
        mma_commit_elect(empty(0));  // V_0 is done
      }
      // Per K/V tile j: [S_j read, K_{j+1}, V_{j+1}] S_{j+1}, dP_{j+1}; [dS_j] dQ += dS_j K_j.
      // The next tile's two score products run while the warps turn P_j and
      // dP_j into dS_j: S_{j+1} may overwrite S once it has been read (P stays
      // in registers), and dP_{j+1} goes to the other dP buffer, whose last
      // reader (dQ += dS_{j-1} K_{j-1}) was issued before it.
      auto general = [&](int j) -> bool {
        const bool has_next = j + 1 < nkv;
        const int sk = (2 * j + 1) % R;
        if (has_next) {
          const int iv = 2 * j + 2, ik = 2 * j + 3;
          const bool a = mbar_try_wait(bar(3), j & 1);
          const bool b = mbar_try_wait(full(ik % R), (ik / R) & 1);
          const bool c = mbar_try_wait(full(iv % R), (iv / R) & 1);
          if (!uniform(a && b && c)) {
            if (!uniform(mbar_wait(bar(3), j & 1, abort_flag)) || !wait_item(ik) || !wait_item(iv)) return false;
          }
          tc_fence_after();
          score(dQd, ik % R, kTmS);
          mma_commit_elect(bar(1));
          score(dDOd, iv % R, kTmDP + ((j + 1) & 1) * 128);
          mma_commit_elect(bar(2));
          mma_commit_elect(empty(iv % R));  // V_{j+1} is done
        }
        if (!uniform(mbar_wait(bar(4), j & 1, abort_flag))) return false;
        tc_fence_after();
        acc_dq(sk, kTmDP + (j & 1) * 128, j > 0);
        mma_commit_elect(empty(sk));  // K_j is done
        if (j == nkv - 1) mma_commit_elect(bar(5));
        return true;
      };
      // Tiles 1 .. nkv-2: the same products with no branch around the MMAs (a
      // branch next to a barrier test of this thread costs the pipe about 20
      // cycles per MMA; the test itself waits for the MMAs already queued).
      auto steady = [&](int j) -> bool {
        const int sk = (2 * j + 1) % R;
        const int iv = 2 * j + 2, ik = 2 * j + 3;
        const uint32_t p3 = j & 1, pk = (ik / R) & 1, pv = (iv / R) & 1;
        const bool a = mbar_try_wait(bar(3), p3);
        const bool b = mbar_try_wait(full(ik % R), pk);
        const bool c = mbar_try_wait(full(iv % R), pv);
        if (!uniform(a && b && c)) {
          if (!uniform(mbar_wait(bar(3), p3, abort_flag)) || !uniform(mbar_wait(full(ik % R), pk, abort_flag)) ||
              !uniform(mbar_wait(full(iv % R), pv, abort_flag)))
            return false;
        }
        tc_fence_after();
        score(dQd, ik % R, kTmS);
        mma_commit_elect(bar(1));
        score(dDOd, iv % R, kTmDP + ((j + 1) & 1) * 128);
        mma_commit_elect(bar(2));
        mma_commit_elect(empty(iv % R));  // V_{j+1} is done
        if (!uniform(mbar_try_wait(bar(4), p3))) {
          if (!uniform(mbar_wait(bar(4), p3, abort_flag))) return false;
        }
        tc_fence_after();
        acc_dq(sk, kTmDP + (j & 1) * 128, true);
        mma_commit_elect(empty(sk));  // K_j is done
        return true;
      };
      int j = 0;
      if (ok && nkv > 0) ok = general(j++);
      for (; ok && j < nkv - 1; ++j) ok = steady(j);
      for (; ok && j < nkv; ++j) ok = general(j);
      if (!ok) report_wait_failure(abort_flag, 4u);
      mma_commit_elect(bar(6));
      uniform(mbar_wait(bar(6), 0, nullptr));
    }
  } else {
    // ============== compute warps (0-7: one row per thread, one column half) =====
    const int h = warp >> 2;  // keys 64h..64h+63 of each K/V tile, dQ columns h*D/2..
    const int wq = warp & 3;  // TMEM lane quarter
    const int row_local = wq * 32 + lane;
    const int row = row0 + row_local;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float c = p.scale_log2;
    const float POS_INF = __int_as_float(0x7f800000);
    const bool valid = row < p.Nq;
    const size_t grow = static_cast<size_t>(bh) * p.Nq + row;
    // keys [row_key_lo, row_key_end) are visible to this row (window bounds
    // clamped into [-1, Nk], so every later difference fits an int)
    int row_key_lo = 0, row_key_end = p.Nk;
    if (MASK == kBwdMaskCausal) row_key_end = min(p.Nk, row + 1);
    if (MASK == kBwdMaskWindow) {
      if (p.win_left >= 0)
        row_key_lo = static_cast<int>(min(static_cast<long long>(p.Nk),
                                          max(-1ll, static_cast<long long>(row) + p.diag_off - p.win_left)));
      if (p.win_right >= 0)
        row_key_end = static_cast<int>(
            min(static_cast<long long>(p.Nk), max(-1ll, static_cast<long long>(row) + p.diag_off + p.win_right) + 1));
    }
    // D = rowsum(dO * O) in fp32, L = LSE * log2(e); padding rows: P = 0.
    // Each half sums its own D/2 columns with every load issued up front (one
    // memory round trip), then the two half sums meet in shared memory and
    // both halves add them in the same order (same value in both).
    float dsum = 0.f, lse2 = POS_INF;
    if (valid) {
      const uint4* orow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + grow * D + h * (D / 2));
      const uint4* drow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + grow * D + h * (D / 2));
      uint4 oa[D / 16], da[D / 16];
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        oa[i] = orow[i];
        da[i] = drow[i];
      }
      lse2 = p.lse[grow] * 1.4426950408889634074f;
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        const uint32_t aw[4] = {oa[i].x, oa[i].y, oa[i].z, oa[i].w}, bw[4] = {da[i].x, da[i].y, da[i].z, da[i].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          dsum = fmaf(__uint_as_float(aw[t] << 16), __uint_as_float(bw[t] << 16), dsum);
          dsum = fmaf(__uint_as_float(aw[t] & 0xFFFF0000u), __uint_as_float(bw[t] & 0xFFFF0000u), dsum);
        }
      }
    }
    {
      float* const part = reinterpret_cast<float*>(sbase + C::kQPartOff);  // [half][row]
      part[h * 128 + row_local] = dsum;
      mbar_arrive(bar(7 + wq));
      bool got = __all_sync(0xffffffffu, mbar_wait(bar(7 + wq), 0, abort_flag));
      if (got) {
        dsum = part[row_local] + part[128 + row_local];
      } else {
        report_wait_failure(abort_flag, 1u);
      }
    }
    if (h == 0) {
      const size_t prow = static_cast<size_t>(bh) * p.Nq_pad + row;
      p.lse2[prow] = lse2;
      p.dsum[prow] = valid ? dsum : 0.f;
    }
    const float neg_lse2 = -lse2;
    const uint32_t tSh = lane_base + kTmS + h * 64;    // this half's S columns
    // this half's columns of dP buffer 0 (tile j uses buffer j % 2; dS lands in the first 32)
    const uint32_t tDPh = lane_base + kTmDP + h * 64;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      // ---- P = 2^(S*c - L) in registers, then S's columns are free
      bool got = mbar_wait(bar(1), j & 1, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s0[32], s1[32];
      tmem_ld32(tSh + 0, s0);
      tmem_ld32(tSh + 32, s1);
      tmem_ld_wait(s0);
      reg_pin(s1);
      tc_fence_before();
      mbar_arrive(bar(3));
      float* const f[2] = {reinterpret_cast<float*>(s0), reinterpret_cast<float*>(s1)};
      // visible columns of this half [lo, lim): ragged key tail, the causal
      // diagonal or the window's two edges
      const int col0 = (jlo + j) * 128 + h * 64;
      const int lim = row_key_end - col0;
      const int lo = (MASK == kBwdMaskWindow) ? row_key_lo - col0 : 0;
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float x0, x1;
          fma2(x0, x1, f[q2][i], f[q2][i + 1], c, neg_lse2);
          const int e = q2 * 32 + i;
          if (MASK == kBwdMaskWindow) {
            f[q2][i] = (e < lim && e >= lo) ? ex2(x0) : 0.f;
            f[q2][i + 1] = (e + 1 < lim && e + 1 >= lo) ? ex2(x1) : 0.f;
          } else {
            f[q2][i] = (e < lim) ? ex2(x0) : 0.f;
            f[q2][i + 1] = (e + 1 < lim) ? ex2(x1) : 0.f;
          }
        }
      // ---- dS = P (dP - D), bf16, into the first 32 columns of this half's dP
      got = mbar_wait(bar(2), j & 1, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t dp[32];
        const uint32_t tdp = tDPh + (j & 1) * 128;
        tmem_ld32(tdp + q2 * 32, dp);
        tmem_ld_wait(dp);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = f[q2][2 * i] * (__uint_as_float(dp[2 * i]) - dsum);
          const float b = f[q2][2 * i + 1] * (__uint_as_float(dp[2 * i + 1]) - dsum);
          pk[i] = pack_bf16(a, b);
        }
        // columns [16*q2, 16*q2 + 16) of this half were read by the first chunk
        tmem_st16(tdp + q2 * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(4));
    }
    if (!ok) report_wait_failure(abort_flag, 1u);
    if (ok && nkv > 0) {
      bool got = mbar_wait(bar(5), 0, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        report_wait_failure(abort_flag, 8u);
      } else {
        tc_fence_after();
        // dQ in bf16 is staged in the Q buffer (free once dq_full has flipped)
        // in the 128-byte swizzled box layout of the dQ tensor map, then one
        // thread stores the tile with TMA (rows past Nq are dropped)
        const uint32_t stage = base + static_cast<uint32_t>(row_local) * 128u;
        const uint32_t swz = static_cast<uint32_t>(row_local & 7);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          uint32_t o[32];
          tmem_ld32(lane_base + kTmDQ + h * (D / 2) + cc * 32, o);
          tmem_ld_wait(o);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(o[2 * i]) * p.scale, __uint_as_float(o[2 * i + 1]) * p.scale);
          const int col = h * (D / 2) + cc * 32;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t chunk = static_cast<uint32_t>(((col & 63) >> 3) + i);
            st_shared_v4(stage + static_cast<uint32_t>(col >> 6) * C::kBoxBytes + ((chunk ^ swz) << 4), w[4 * i],
                         w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(11 + 2 * R));
        if (threadIdx.x == 0) {
          if (mbar_wait(bar(11 + 2 * R), 0, abort_flag)) {
#pragma unroll
            for (int b = 0; b < C::kBoxes; ++b) tma_store_3d(&tmDQ, base + b * C::kBoxBytes, b * 64, row0, bh);
            bulk_commit_group();
            bulk_wait_group_read0();
          } else {
            report_wait_failure(abort_flag, 8u);
          }
        }
      }
    } else if (MASK == kBwdMaskWindow && ok && nkv == 0 && valid) {
      // no row of this tile sees a key (possible under a window): dQ = 0
      uint4* const out = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + grow * D + h * (D / 2));
#pragma unroll
      for (int i = 0; i < D / 16; ++i) out[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// dK / dV kernel
// ---------------------------------------------------------------------------
// barriers: 0 kv_full, 1 s_full (S^T), 2 p_done (P^T written), 3 acc_full,
// 4 drain, 5 dp_full (dP^T), 6 ds_done (dS^T written), then ring
// full[kRingKV], empty[kRingKV], then the epilogue's staging barrier
template <int D, int MASK>
__global__ void __launch_bounds__(320, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                       const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int R = C::kRingKV;
  // Ring slot and phase of item `it` (even: Q_i with its L and D, odd: dO_i; i = it / 2).
  // Query tile i uses the slot pair i % (R/2), and Q and dO swap places each time a
  // pair comes round again, so Q_{i+1} lands in the slot that dO_{i-1} left: dV_{i-1}
  // frees it half an iteration before dK_{i-1} frees Q_{i-1}'s, and Q_{i+1} (needed
  // first, by S^T_{i+1}) gets that much more time to arrive.
  auto item_slot = [](int it) -> int {
    const int i = it >> 1;
    return 2 * (i % (R / 2)) + ((it & 1) ^ ((i / (R / 2)) & 1));
  };
  auto item_phase = [](int it) -> uint32_t { return static_cast<uint32_t>((it >> 1) / (R / 2)) & 1u; };
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw_addr);
  const uint32_t bar0 = base + C::kKVBarOff;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto full = [&](int s) -> uint32_t { return bar(7 + s); };
  auto empty = [&](int s) -> uint32_t { return bar(7 + R + s); };
  auto slot_addr = [&](int s) -> uint32_t { return base + C::kKVRingOff + s * C::kTileBytes; };
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + C::kKVBarOff + 448);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sbase + C::kKVBarOff + 452);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(0), 1);
    mbar_init(bar(1), 1);
    mbar_init(bar(2), 256);
    mbar_init(bar(3), 1);
    mbar_init(bar(4), 1);
    mbar_init(bar(5), 1);
    mbar_init(bar(6), 256);
    for (int s = 0; s < R; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(bar(7 + 2 * R), 256);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM: S^T [0,128) (P^T overwrites its first 64 columns), dP^T [128,256)
  // (dS^T likewise), dV [256, 256 + D), dK [256 + D, 256 + 2D)
  constexpr uint32_t kTmS = 0, kTmDP = 128, kTmDV = 256, kTmDK = 256 + D;

  const int bh = blockIdx.x / p.n_kt;
  const int kt = blockIdx.x % p.n_kt;  // causal: small kt sees the most query tiles
  const int key0 = kt * 128;
  // query tiles [i0, i0 + nq) see this key tile
  int i0 = (MASK == kBwdMaskCausal) ? kt : 0;
  int nq = p.n_qt - i0;
  if (MASK == kBwdMaskWindow) {
    // query i keeps key j iff j - diag_off - win_right <= i <= j - diag_off + win_left
    const long long k_first = key0, k_last = min(key0 + 128, p.Nk) - 1;
    long long q_lo = 0, q_hi = p.Nq - 1;
    if (p.win_right >= 0) q_lo = max(0ll, k_first - p.diag_off - p.win_right);
    if (p.win_left >= 0) q_hi = min(q_hi, k_last - p.diag_off + p.win_left);
    if (q_lo > q_hi) {
      nq = 0;  // no query sees a key of this tile: dK = dV = 0
    } else {
      i0 = static_cast<int>(q_lo / 128);
      nq = static_cast<int>(q_hi / 128) + 1 - i0;
    }
  }
  const bool any_q = MASK != kBwdMaskWindow || nq > 0;  // compile-time true without a window

  if (warp == 8) {
    // ======================= TMA producer =================================
    if (lane == 0 && any_q) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmDO);
      tma_prefetch_map(&tmDK);
      tma_prefetch_map(&tmDV);
      mbar_arrive_expect_tx(bar(0), 2 * C::kTileBytes);
      for (int b = 0; b < C::kBoxes; ++b) {
        tma_load_3d(base + b * C::kBoxBytes, &tmK, bar(0), b * 64, key0, bh);
        tma_load_3d(base + C::kTileBytes + b * C::kBoxBytes, &tmV, bar(0), b * 64, key0, bh);
      }
      int item = 0;
      bool ok = true;
      for (; item < 2 * nq; ++item) {  // Q_i (with its L, D), dO_i, ...
        const int s = item_slot(item);
        const int i = i0 + (item >> 1);
        if (!(ok = mbar_wait(empty(s), item_phase(item) ^ 1u, abort_flag))) break;
        if (item & 1) {
          mbar_arrive_expect_tx(full(s), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(slot_addr(s) + b * C::kBoxBytes, &tmDO, full(s), b * 64, i * 128, bh);
        } else {
          mbar_arrive_expect_tx(full(s), C::kTileBytes + C::kSideBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(slot_addr(s) + b * C::kBoxBytes, &tmQ, full(s), b * 64, i * 128, bh);
          const size_t off = static_cast<size_t>(bh) * p.Nq_pad + static_cast<size_t>(i) * 128;
          const uint32_t side = base + C::kKVSideOff + s * C::kSideBytes;
          bulk_load(side, p.lse2 + off, 512, full(s));
          bulk_load(side + 512, p.dsum + off, 512, full(s));
        }
      }
      if (!ok) report_wait_failure(abort_flag, 2u);
      if (*abort_flag) {
        for (int it = max(0, item - R); it < item; ++it) mbar_wait(full(item_slot(it)), item_phase(it), nullptr);
        mbar_wait(bar(0), 0, nullptr);
      }
    }
  } else if (warp == 9) {
    // ======================= MMA issuer ====================================
    // The whole warp runs the issue loop on warp-uniform values (every barrier
    // outcome made uniform with a vote); one lane chosen by elect.sync issues
    // each tcgen05.mma and commit, with no branch around the instruction
    // (same-box A/B against lane 0 alone: +6.5% to +11.5%).
    auto uniform = [](bool v) -> bool { return __all_sync(0xffffffffu, v); };
    {
      const uint64_t dKd = sdesc_sw128(base, 16, 1024);                  // K, K-major
      const uint64_t dVd = sdesc_sw128(base + C::kTileBytes, 16, 1024);  // V, K-major
      const uint64_t dRingK = sdesc_sw128(base + C::kKVRingOff, 16, 1024);
      const uint64_t dRingMN = sdesc_sw128(base + C::kKVRingOff, C::kBoxBytes, 1024);
      auto slot_off = [&](int s) -> uint64_t { return (s * C::kTileBytes) >> 4; };
      // S^T = K Q_i^T or dP^T = V dO_i^T: 128 keys x 128 queries over d
      auto score = [&](uint64_t da, int s, uint32_t dst) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tmem + dst, da + off, dRingK + slot_off(s) + off, C::kIdescScore, kk > 0 ? 1u : 0u);
        }
      };
      // acc += A^T-tile (TMEM, 128 keys x 128 queries; queries 16kk.. at column
      // a_cols + 64 (kk / 4) + 8 (kk % 4)) times B_i (queries x D, MN-major)
      auto accum = [&](uint32_t dst, uint32_t a_cols, int s, bool acc_prev) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_elect(tmem + dst, tmem + a_cols + (kk >> 2) * 64 + (kk & 3) * 8, dRingMN + slot_off(s) + ((kk * 2048) >> 4),
                 C::kIdescAcc, (acc_prev || kk > 0) ? 1u : 0u);
      };
      auto wait_item = [&](int it) -> bool { return uniform(mbar_wait(full(item_slot(it)), item_phase(it), abort_flag)); };
      bool ok = !any_q || (uniform(mbar_wait(bar(0), 0, abort_flag)) && wait_item(0) && wait_item(1));
      if (ok && any_q) {
        tc_fence_after();
        score(dKd, item_slot(0), kTmS);
        mma_commit_elect(bar(1));
        score(dVd, item_slot(1), kTmDP);
        mma_commit_elect(bar(5));
      }
      // Per query tile i: [P^T_i written, Q_{i+1}] dV += P^T_i dO_i, S^T_{i+1};
      // [dS^T_i written, dO_{i+1}] dK += dS^T_i Q_i, dP^T_{i+1}.  The next tile's
      // S^T runs while the warps turn dP^T_i into dS^T_i, and its dP^T while they
      // exponentiate S^T_{i+1}: S^T_{i+1} overwrites P^T_i only after the dV
      // product that reads it (issued first), dP^T_{i+1} overwrites dS^T_i only
      // after the dK product.
      auto general = [&](int ii) -> bool {
        const int iq = 2 * ii, ido = 2 * ii + 1;
        const bool has_next = ii + 1 < nq;
        {
          const bool a = mbar_try_wait(bar(2), ii & 1);
          const bool b = !has_next || mbar_try_wait(full(item_slot(iq + 2)), item_phase(iq + 2));
          if (!uniform(a && b)) {
            if (!uniform(mbar_wait(bar(2), ii & 1, abort_flag))) return false;
            if (has_next && !wait_item(iq + 2)) return false;
          }
        }
        tc_fence_after();
        accum(kTmDV, kTmS, item_slot(ido), ii > 0);  // dV += P^T dO_i
        mma_commit_elect(empty(item_slot(ido)));           // dO_i is done
        if (has_next) {
          score(dKd, item_slot(iq + 2), kTmS);  // S^T_{i+1}
          mma_commit_elect(bar(1));
        }
        {
          const bool a = mbar_try_wait(bar(6), ii & 1);
          const bool b = !has_next || mbar_try_wait(full(item_slot(ido + 2)), item_phase(ido + 2));
          if (!uniform(a && b)) {
            if (!uniform(mbar_wait(bar(6), ii & 1, abort_flag))) return false;
            if (has_next && !wait_item(ido + 2)) return false;
          }
        }
        tc_fence_after();
        accum(kTmDK, kTmDP, item_slot(iq), ii > 0);  // dK += dS^T Q_i
        mma_commit_elect(empty(item_slot(iq)));            // Q_i (and its L, D) is done
        if (has_next) {
          score(dVd, item_slot(ido + 2), kTmDP);  // dP^T_{i+1}
          mma_commit_elect(bar(5));
        }
        return true;
      };
      // Query tiles 1 .. nq-2: the same products with no branch around the
      // MMAs (a branch next to a barrier test of this thread costs the pipe
      // about 20 cycles per MMA).
      auto steady = [&](int ii) -> bool {
        const int iq = 2 * ii, ido = 2 * ii + 1;
        const uint32_t pb = ii & 1, pq = item_phase(iq + 2), pd = item_phase(ido + 2);
        const int sq = item_slot(iq + 2), sd = item_slot(ido + 2), sqi = item_slot(iq), sdi = item_slot(ido);
        {
          const bool a = mbar_try_wait(bar(2), pb);
          const bool b = mbar_try_wait(full(sq), pq);
          if (!uniform(a && b)) {
            if (!uniform(mbar_wait(bar(2), pb, abort_flag)) || !uniform(mbar_wait(full(sq), pq, abort_flag))) return false;
          }
        }
        tc_fence_after();
        accum(kTmDV, kTmS, sdi, true);  // dV += P^T dO_i
        mma_commit_elect(empty(sdi));         // dO_i is done
        score(dKd, sq, kTmS);           // S^T_{i+1}
        mma_commit_elect(bar(1));
        {
          const bool a = mbar_try_wait(bar(6), pb);
          const bool b = mbar_try_wait(full(sd), pd);
          if (!uniform(a && b)) {
            if (!uniform(mbar_wait(bar(6), pb, abort_flag)) || !uniform(mbar_wait(full(sd), pd, abort_flag))) return false;
          }
        }
        tc_fence_after();
        accum(kTmDK, kTmDP, sqi, true);  // dK += dS^T Q_i
        mma_commit_elect(empty(sqi));          // Q_i (and its L, D) is done
        score(dVd, sd, kTmDP);           // dP^T_{i+1}
        mma_commit_elect(bar(5));
        return true;
      };
      int ii = 0;
      if (ok && nq > 0) ok = general(ii++);
      for (; ok && ii < nq - 1; ++ii) ok = steady(ii);
      for (; ok && ii < nq; ++ii) ok = general(ii);
      if (ok) mma_commit_elect(bar(3));
      if (!ok) report_wait_failure(abort_flag, 4u);
      mma_commit_elect(bar(4));
      uniform(mbar_wait(bar(4), 0, nullptr));
    }
  } else {
    // ============== compute warps (0-7: one key per thread, one column half) =====
    const int h = warp >> 2;  // queries 64h..64h+63 of each query tile, dK/dV columns h*D/2..
    const int wq = warp & 3;  // TMEM lane quarter
    const int key_local = wq * 32 + lane;
    const int key = key0 + key_local;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tSh = lane_base + kTmS + h * 64;    // this half's S^T columns (P^T lands in the first 32)
    const uint32_t tDPh = lane_base + kTmDP + h * 64;  // this half's dP^T columns (dS^T likewise)
    const float c = p.scale_log2;
    // window: queries [key_q_lo, key_q_end) keep this key (bounds clamped into
    // [-1, Nq], so every later difference fits an int)
    int key_q_lo = 0, key_q_end = p.Nq;
    if (MASK == kBwdMaskWindow) {
      if (p.win_right >= 0)
        key_q_lo = static_cast<int>(min(static_cast<long long>(p.Nq),
                                        max(-1ll, static_cast<long long>(key) - p.diag_off - p.win_right)));
      if (p.win_left >= 0)
        key_q_end = static_cast<int>(
            min(static_cast<long long>(p.Nq), max(-1ll, static_cast<long long>(key) - p.diag_off + p.win_left) + 1));
    }
    bool ok = true;
    for (int ii = 0; ii < nq; ++ii) {
      const int i = i0 + ii;
      const int s = item_slot(2 * ii);  // slot of Q_i, which carries the side buffer
      const float* const Ls = reinterpret_cast<const float*>(sbase + C::kKVSideOff + s * C::kSideBytes) + h * 64;
      const float* const Ds = Ls + 128;
      // the Q_i item's TMA barrier covers the side buffer (L, D) read below;
      // S^T_i comes from its MMA commit (dP^T_i, from its own, is waited for later)
      bool got = mbar_wait(full(s), item_phase(2 * ii), abort_flag) && mbar_wait(bar(1), ii & 1, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s0[32], s1[32];
      tmem_ld32(tSh + 0, s0);
      tmem_ld32(tSh + 32, s1);
      tmem_ld_wait(s0);
      reg_pin(s1);
      float* const f[2] = {reinterpret_cast<float*>(s0), reinterpret_cast<float*>(s1)};
      // causal: query q sees this key iff q >= key; only the diagonal tile masks;
      // window: this half's columns [qlo, qend) are kept
      const int qlim = (MASK == kBwdMaskCausal && i == kt) ? key_local - h * 64 : 0;  // columns < qlim are masked
      const int qcol0 = i * 128 + h * 64;
      const int qlo = (MASK == kBwdMaskWindow) ? key_q_lo - qcol0 : 0;
      const int qend = (MASK == kBwdMaskWindow) ? key_q_end - qcol0 : 64;
      // P^T = 2^(S^T c - L[q]); padding queries have L = +inf, so P^T = 0 there
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t pk[16];
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 l4 = *reinterpret_cast<const float4*>(Ls + q2 * 32 + i4 * 4);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int col = q2 * 32 + i4 * 4 + t;
            const float x = fmaf(f[q2][i4 * 4 + t], c, -lv[t]);
            if (MASK == kBwdMaskWindow)
              f[q2][i4 * 4 + t] = (col >= qlo && col < qend) ? ex2(x) : 0.f;
            else
              f[q2][i4 * 4 + t] = (col >= qlim) ? ex2(x) : 0.f;
          }
        }
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2) pk[i2] = pack_bf16(f[q2][2 * i2], f[q2][2 * i2 + 1]);
        tmem_st16(tSh + q2 * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(2));  // P^T_i is in TMEM: dV may start
      got = __all_sync(0xffffffffu, mbar_wait(bar(5), ii & 1, abort_flag));
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dS^T = P^T (dP^T - D[q]) into the first 32 columns of this half's dP^T
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t dp[32];
        tmem_ld32(tDPh + q2 * 32, dp);
        tmem_ld_wait(dp);
        uint32_t pk[16];
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 d4 = *reinterpret_cast<const float4*>(Ds + q2 * 32 + i4 * 4);
          const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
          for (int t = 0; t < 4; t += 2) {
            const int e = i4 * 4 + t;
            const float a = f[q2][e] * (__uint_as_float(dp[e]) - dv[t]);
            const float b = f[q2][e + 1] * (__uint_as_float(dp[e + 1]) - dv[t + 1]);
            pk[e / 2] = pack_bf16(a, b);
          }
        }
        tmem_st16(tDPh + q2 * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(6));  // dS^T_i is in TMEM: dK may start
    }
    if (!ok) report_wait_failure(abort_flag, 1u);
    if (ok && nq > 0) {
      bool got = mbar_wait(bar(3), 0, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        report_wait_failure(abort_flag, 8u);
      } else {
        tc_fence_after();
        // dK and dV in bf16 are staged in the K and V buffers (free once
        // acc_full has flipped) in the 128-byte swizzled box layout of their
        // tensor maps, then one thread stores both tiles with TMA (keys past
        // Nk are dropped)
        const uint32_t stage_k = base + static_cast<uint32_t>(key_local) * 128u;
        const uint32_t stage_v = stage_k + C::kTileBytes;
        const uint32_t swz = static_cast<uint32_t>(key_local & 7);
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc) {
          const int col = h * (D / 2) + cc * 32;
          const uint32_t off = static_cast<uint32_t>(col >> 6) * C::kBoxBytes;
          const uint32_t chunk0 = static_cast<uint32_t>((col & 63) >> 3);
          uint32_t o[32];
          tmem_ld32(lane_base + kTmDV + h * (D / 2) + cc * 32, o);
          tmem_ld_wait(o);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = pack_bf16(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_shared_v4(stage_v + off + (((chunk0 + i) ^ swz) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2],
                         w[4 * i + 3]);
          tmem_ld32(lane_base + kTmDK + h * (D / 2) + cc * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16(__uint_as_float(o[2 * i]) * p.scale, __uint_as_float(o[2 * i + 1]) * p.scale);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_shared_v4(stage_k + off + (((chunk0 + i) ^ swz) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2],
                         w[4 * i + 3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(7 + 2 * R));
        if (threadIdx.x == 0) {
          if (mbar_wait(bar(7 + 2 * R), 0, abort_flag)) {
#pragma unroll
            for (int b = 0; b < C::kBoxes; ++b) {
              tma_store_3d(&tmDK, base + b * C::kBoxBytes, b * 64, key0, bh);
              tma_store_3d(&tmDV, base + C::kTileBytes + b * C::kBoxBytes, b * 64, key0, bh);
            }
            bulk_commit_group();
            bulk_wait_group_read0();
          } else {
            report_wait_failure(abort_flag, 8u);
          }
        }
      }
    } else if (MASK == kBwdMaskWindow && ok && nq == 0 && key < p.Nk) {
      // no query sees a key of this tile (possible under a window): dK = dV = 0
      const size_t grow = static_cast<size_t>(bh) * p.Nk + key;
      uint4* const outv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dv) + grow * D + h * (D / 2));
      uint4* const outk = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dk) + grow * D + h * (D / 2));
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        outv[i] = make_uint4(0u, 0u, 0u, 0u);
        outk[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
