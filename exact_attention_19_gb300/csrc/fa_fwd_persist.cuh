// fa_fwd_persist.cuh -- persistent fused exact-attention forward for sm_103a
// (no K/V split).  Without a mask: d = 128, and d = 64 for short key ranges,
// under a static schedule.  Causal with many query-tile pairs per SM (and at
// d = 64 long key ranges): under a dynamic schedule (cluster launch control).
//
// The arithmetic is that of fa_fwd_kernel (FA2 loop order, page "llm-infra-
// atlas / FlashAttention 01", sections 2-4; conditional rescaling with
// tau = 8 in base 2, page "pinghaoyang FlashAttention 1-4 guide", FA4
// section; O divided by the row sum with the row's largest P counted as
// rounded to bf16).  What differs is the schedule:
//
//  * One CTA per SM loops over work units (b*H + h, pair of 128-row query
//    tiles); CTA c takes units c, 2G-1-c, 2G+c, ... (G CTAs).  The K/V ring,
//    the S and P barriers and the MMA stream run on across unit boundaries:
//    in the last K/V step of a unit the MMA issuer computes the next unit's
//    first S products where it would otherwise compute the next tile's, so
//    the tensor pipe sees no start or end of a unit, and no CTA is launched,
//    set up or torn down per unit.
//  * 12 warps, launched with 168 registers each; setmaxnreg then gives
//    warps 0-7 184 and warps 8-11 128, or 192 and 120 at d = 64 (as in
//    fa_fwd_kernel):
//      warps 0-3   softmax, conditional rescale and epilogue of query tile 0
//      warps 4-7   the same for query tile 1
//      warp  8     TMA producer of the K/V ring
//      warp  9     MMA issuer: the whole warp runs the issue loop on
//                  warp-uniform values, one elected lane issues
//                  (as in fa_fwd_kernel)
//      warp 10     TMA producer of the Q tiles (and an L2 prefetch of the
//                  next unit's Q)
//      warp 11     idle
//    The epilogue of a unit's tile (O / l to bf16, stored by each row's
//    thread; LSE) runs in that tile's softmax warps before they take the next
//    unit's first S, so the next unit's first P V (which overwrites O) cannot
//    start before O has been read.
//  * d = 128: one Q buffer per tile; the next unit's Q is loaded as soon as
//    the last S product of the unit has read the old one (it was prefetched
//    into L2 a unit earlier).  d = 64: two Q buffers per tile, so the next
//    unit's Q is loaded while the unit runs.
//  * Causal units are of unequal length (1 to N / 128 K/V tiles): the grid
//    keeps one CTA per unit in fa_fwd_kernel's longest-first order, and a
//    running CTA asks the hardware for the next CTA not yet started
//    (clusterlaunchcontrol.try_cancel) and runs its unit instead, so the
//    hardware's greedy balance of that order is kept.  The K/V producer asks
//    for unit k + 1 as it starts unit k; the answers pass to the other roles
//    through a ring of kUnitRing 16-byte slots in shared memory.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "fa_fwd_kernel.cuh"

namespace fa {

template <int D>
struct PCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kThreads = 384;  // three warpgroups
  static constexpr int kWarpKV = 8, kWarpMma = 9, kWarpQ = 10;
  static constexpr int kBM = 128, kBN = 128;
  static constexpr int kQBufs = (D == 64) ? 2 : 1;  // Q buffers per query tile
  static constexpr int kRing = (D == 64) ? 8 : 5;    // K/V ring slots
  static constexpr int kUnitRing = 4;                // dynamic schedule: unit responses in flight
  static constexpr int kBoxes = D / 64;
  static constexpr uint32_t kBoxBytes = 128u * 128u;
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
  static constexpr uint32_t kQOff = 0;  // Q[qb][t] at (2 * qb + t) * kTileBytes
  static constexpr uint32_t kRingOff = 2 * kQBufs * kTileBytes;
  static constexpr uint32_t kBarOff = kRingOff + kRing * kTileBytes;
  static constexpr uint32_t kBarBytes = 512;
  static constexpr uint32_t kSmemBytes = kBarOff + kBarBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmO = 256;  // O[t] at kTmO + t * D
  static constexpr uint32_t kIdescS = idesc_bf16(128, 128, false);
  static constexpr uint32_t kIdescO = idesc_bf16(128, D, true);
  // registers per thread: at launch (checked by the host), softmax warpgroups, warpgroup 2
  static constexpr int kRegLaunch = 168, kRegSoftmax = (D == 64) ? 192 : 184, kRegMisc = (D == 64) ? 120 : 128;
  static_assert(2 * 128 * kRegSoftmax + 128 * kRegMisc <= kThreads * kRegLaunch, "register split");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// barrier slots (8 bytes each)
enum : int {
  kPBarQFull = 0,    // [qb][t]: 4
  kPBarQFree = 4,    // [qb][t]: 4
  kPBarS = 8,        // [t]
  kPBarP = 10,       // [t]
  kPBarOFinal = 12,  // [t]
  kPBarDrain = 14,
  kPBarRing = 15,      // full[kRing] then empty[kRing] (kRing <= 8)
  kPBarUnit = 31,      // dynamic schedule: response s has landed [kUnitRing]
  kPBarUnitFree = 35,  // dynamic schedule: every consumer has read response s [kUnitRing]
  kPBarEnd = 39
};
constexpr uint32_t kUnitRespOff = 320;  // kUnitRing 16-byte responses, after the barriers
static_assert(8 * kPBarEnd <= kUnitRespOff && kUnitRespOff + 16 * 4 <= 448, "barrier block");
// consumers of a unit response: the Q producer, the MMA warp, the 8 softmax warps
constexpr int kUnitConsumers = 10;

// L2 prefetch of one TMA box (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// One work unit as every role sees it.
struct PUnit {
  int bh;
  int j0;          // first K/V tile streamed (0 without a window)
  int row0[2];
  int jlo[2];      // K/V tiles [j0 + jlo[t], j0 + jhi[t]) visible to query tile t;
  int jhi[2];      // jlo = jhi = 0 when the tile is absent; jlo is 0 or 1
  int n_max;       // K/V tiles streamed: max(jhi)
};

// MASK kMaskNone: a static schedule over min(units, SMs) CTAs.  kMaskCausal:
// one CTA per unit in fa_fwd_kernel's causal launch order; a running CTA
// takes over CTAs that have not started yet with cluster launch control, so
// the hardware's greedy dispatch of that order is kept.
template <int D, int MASK>
__global__ void __launch_bounds__(PCfg<D>::kThreads, 1)
    fa_fwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const FwdParams p, const int n_units) {
  static_assert(MASK == kMaskNone || MASK == kMaskCausal || MASK == kMaskWindow, "mask");
  constexpr bool kDynamic = MASK == kMaskCausal;
  using C = PCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw_addr);

  const uint32_t bar0 = base + C::kBarOff;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto full = [&](int slot) -> uint32_t { return bar(kPBarRing + slot); };
  auto empty = [&](int slot) -> uint32_t { return bar(kPBarRing + C::kRing + slot); };
  auto slot_addr = [&](int slot) -> uint32_t { return base + C::kRingOff + slot * C::kTileBytes; };
  auto q_addr = [&](int qb, int t) -> uint32_t { return base + C::kQOff + (2 * qb + t) * C::kTileBytes; };
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + C::kBarOff + kTmemSlotOff);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sbase + C::kBarOff + kAbortOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(kPBarQFull + i), 1);
      mbar_init(bar(kPBarQFree + i), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kPBarS + t), 1);
      mbar_init(bar(kPBarP + t), 128);
      mbar_init(bar(kPBarOFinal + t), 1);
    }
    mbar_init(bar(kPBarDrain), 1);
    for (int s = 0; s < C::kRing; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < C::kUnitRing; ++s) {
      mbar_init(bar(kPBarUnit + s), 1);
      mbar_init(bar(kPBarUnitFree + s), kUnitConsumers);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == C::kWarpMma) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- the CTA's work units ---------------------------------------------
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  const int n_kv = (p.Nk + C::kBN - 1) / C::kBN;
  // the unit with index uid in launch order
  auto decode = [&](int uid, PUnit& u) {
    int bh = uid / p.n_pairs, pair = uid % p.n_pairs;
    if (MASK == kMaskCausal) {
      // heads in groups whose K/V fit a quarter of the L2, heaviest pairs of
      // a group first (fa_fwd_kernel's causal launch order)
      const int n_bh = n_units / p.n_pairs;
      const int per_group = p.lpt_group * p.n_pairs;
      const int grp = uid / per_group;
      const int g0 = grp * p.lpt_group;
      const int g_heads = min(p.lpt_group, n_bh - g0);
      const int within = uid - grp * per_group;
      bh = g0 + within % g_heads;
      pair = p.n_pairs - 1 - within / g_heads;
    }
    u.bh = bh;
    u.n_max = 0;
    int lo[2], hi[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int qt = 2 * pair + t;
      u.row0[t] = qt * C::kBM;
      lo[t] = 0;
      hi[t] = 0;
      if (u.row0[t] < p.Nq) {
        hi[t] = (MASK == kMaskCausal) ? min(n_kv, qt + 1) : n_kv;
        if (MASK == kMaskWindow) {
          // a bounded band with Nq <= Nk: every row sees a key, and the two
          // tiles' ranges are contiguous, tile 1's starting at most one later
          const long long r_first = u.row0[t], r_last = min(u.row0[t] + C::kBM, p.Nq) - 1;
          const long long key_lo = max(0ll, r_first + p.diag_off - p.win_left);
          long long key_hi = p.Nk - 1;
          if (p.win_right >= 0) key_hi = min(key_hi, r_last + p.diag_off + p.win_right);
          lo[t] = static_cast<int>(key_lo / C::kBN);
          hi[t] = static_cast<int>(key_hi / C::kBN) + 1;
        }
      }
    }
    u.j0 = lo[0];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      u.jlo[t] = hi[t] > lo[t] ? lo[t] - u.j0 : 0;
      u.jhi[t] = hi[t] > lo[t] ? hi[t] - u.j0 : 0;
      u.n_max = max(u.n_max, u.jhi[t]);
    }
  };
  // a unit's range start and first K/V tile: zero unless there is a window
  auto lo_ = [](const PUnit& u, int t) -> int { return MASK == kMaskWindow ? u.jlo[t] : 0; };
  auto j0_ = [](const PUnit& u) -> int { return MASK == kMaskWindow ? u.j0 : 0; };
  // Dynamic schedule: unit k >= 1 of this CTA is the answer to the k-th
  // cancellation request, in response slot (k - 1) % kUnitRing.
  auto resp_addr = [&](int s) -> uint32_t { return bar0 + kUnitRespOff + 16u * static_cast<uint32_t>(s); };
  // The k-th unit of this CTA: 1 with u filled in, 0 past the end, -1 when a
  // wait gave up.  `release`: 0 for the requesting thread, 1 for a single
  // consuming thread, 2 for a whole consuming warp (lane 0 releases the slot).
  auto get_unit = [&](int k, PUnit& u, int release) -> int {
    if constexpr (!kDynamic) {
      const long long id = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - cta) : cta);
      if (id >= n_units) return 0;
      decode(static_cast<int>(id), u);
      return 1;
    } else {
      if (k == 0) {
        decode(cta, u);
        return 1;
      }
      const int s = (k - 1) % C::kUnitRing;
      bool got = mbar_wait(bar(kPBarUnit + s), ((k - 1) / C::kUnitRing) & 1, abort_flag);
      if (release == 2) got = __all_sync(0xffffffffu, got);
      if (!got) return -1;
      int x = 0;
      const bool more = clc_query(resp_addr(s), x);
      if (release == 2) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kPBarUnitFree + s));
      } else if (release == 1) {
        mbar_arrive(bar(kPBarUnitFree + s));
      }
      if (!more) return 0;
      decode(x, u);
      return 1;
    }
  };
  // Dynamic schedule, requesting thread only: ask for the CTA's unit k.
  auto request_unit = [&](int k) -> bool {
    const int s = (k - 1) % C::kUnitRing, use = (k - 1) / C::kUnitRing;
    if (use > 0 && !mbar_wait(bar(kPBarUnitFree + s), (use - 1) & 1, abort_flag)) return false;
    mbar_arrive_expect_tx(bar(kPBarUnit + s), 16);
    clc_try_cancel(resp_addr(s), bar(kPBarUnit + s));
    return true;
  };

  if (warp >= 8) {
    regs_dec<C::kRegMisc>();
    if (warp == C::kWarpKV && lane == 0) {
      // ======================= K/V producer ===============================
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      int issued = 0;
      bool ok = true;
      int pending = 0;  // dynamic: unit whose request is answered but not yet read (0: none)
      PUnit u;
      int r = get_unit(0, u, 0);
      for (int k = 0; ok && r == 1; ++k) {
        // dynamic: ask now for the next unit; its answer is needed once this
        // unit's loads have been issued
        if (kDynamic) {
          if (!request_unit(k + 1)) {
            report_wait_failure(abort_flag, 2u);
            ok = false;
            break;
          }
          pending = k + 1;
        }
        for (int i = 0; i < 2 * u.n_max; ++i) {
          const int item = issued;
          const int s = item % C::kRing;
          if (!mbar_wait(empty(s), ((item / C::kRing) & 1) ^ 1u, abort_flag)) {
            report_wait_failure(abort_flag, 2u);
            ok = false;
            break;
          }
          const CUtensorMap* map = (i & 1) ? &tmV : &tmK;
          mbar_arrive_expect_tx(full(s), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(slot_addr(s) + b * C::kBoxBytes, map, full(s), b * 64, (j0_(u) + (i >> 1)) * C::kBN, u.bh);
          issued = item + 1;
        }
        if (!ok) break;
        r = get_unit(k + 1, u, 0);
        if (r < 0) {
          report_wait_failure(abort_flag, 2u);
          ok = false;
        } else {
          pending = 0;
        }
      }
      if (*abort_flag) {
        // let every copy already issued land before the CTA can exit
        for (int item = max(0, issued - C::kRing); item < issued; ++item)
          mbar_wait(full(item % C::kRing), (item / C::kRing) & 1, nullptr);
        // and the answer to an outstanding cancellation request
        if (kDynamic && pending > 0)
          mbar_wait(bar(kPBarUnit + (pending - 1) % C::kUnitRing), ((pending - 1) / C::kUnitRing) & 1, nullptr);
      }
    } else if (warp == C::kWarpQ && lane == 0) {
      // ======================= Q producer =================================
      tma_prefetch_map(&tmQ);
      int occ[2] = {0, 0};
      bool ok = true;
      PUnit u, un;
      int r = get_unit(0, u, 1);
      for (int k = 0; ok && r == 1; ++k) {
        for (int t = 0; t < 2 && ok; ++t) {
          if (u.jhi[t] == 0) continue;
          const int qb = occ[t] % C::kQBufs, use = occ[t] / C::kQBufs;
          if (use > 0 && !mbar_wait(bar(kPBarQFree + 2 * qb + t), (use - 1) & 1, abort_flag)) {
            report_wait_failure(abort_flag, 2u);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kPBarQFull + 2 * qb + t), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            tma_load_3d(q_addr(qb, t) + b * C::kBoxBytes, &tmQ, bar(kPBarQFull + 2 * qb + t), b * 64, u.row0[t],
                        u.bh);
          ++occ[t];
        }
        if (!ok) break;
        // the next unit's Q into L2 while this one runs
        r = get_unit(k + 1, un, 1);
        if (r < 0) {
          report_wait_failure(abort_flag, 2u);
          ok = false;
        } else if (r == 1) {
          for (int t = 0; t < 2; ++t)
            if (un.jhi[t] > 0)
              for (int b = 0; b < C::kBoxes; ++b) tma_prefetch_l2_3d(&tmQ, b * 64, un.row0[t], un.bh);
          u = un;
        }
      }
      if (*abort_flag) {
        // every Q copy issued lands before exit: the last fill of each buffer
        for (int t = 0; t < 2; ++t)
          for (int i = max(0, occ[t] - C::kQBufs); i < occ[t]; ++i)
            mbar_wait(bar(kPBarQFull + 2 * (i % C::kQBufs) + t), (i / C::kQBufs) & 1, nullptr);
      }
    } else if (warp == C::kWarpMma) {
      // ======================= MMA issuer ==================================
      // Every lane runs this loop; waits are made warp-uniform with
      // __all_sync, and each tcgen05.mma / commit is issued by the lane that
      // elect.sync picks inside the same asm statement.
      auto uniform = [](bool v) -> bool { return __all_sync(0xffffffffu, v); };
      // Per K/V step j of a unit, as in fa_fwd_kernel:
      //   [V_j, K_{j+1}, P_0(j)] PV_0(j), S_0(j+1); [P_1(j)] PV_1(j), S_1(j+1)
      // The interior steps of a unit run the same bodies as fa_fwd_kernel
      // (the general one, and the branch-free copy where both tiles are
      // inside their ranges); the last step computes the next unit's first
      // S products (after checking its Q tiles) in place of S(j+1).  O needs no
      // check: a tile's next first P V waits for its P, which that tile's
      // softmax warps hand over only after their epilogue has read O.
      const uint64_t dK0 = sdesc_sw128(base + C::kRingOff, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(base + C::kRingOff, C::kBoxBytes, 1024);
      const uint64_t dQ0 = sdesc_sw128(base + C::kQOff, 16, 1024);
      const uint32_t tS[2] = {tmem, tmem + 128u};
      uint64_t dq[2] = {dQ0, dQ0}, dq_n[2] = {dQ0, dQ0};  // Q descriptors of the unit's and the next unit's tiles
      const uint32_t to[2] = {tmem + C::kTmO, tmem + C::kTmO + D};
      int qb[2] = {0, 0}, qb_n[2] = {0, 0};
      auto gemm1 = [&](int t, uint64_t dqt, int slot) {
        const uint64_t dk = dK0 + ((slot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tS[t], dqt + off, dk + off, C::kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      auto gemm2 = [&](int t, int slot, bool acc_prev) {
        const uint64_t dv = dV0 + ((slot * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::kBN / 16; ++kk)
          mma_ts_elect(to[t], tS[t] + kk * 8, dv + ((kk * 2048) >> 4), C::kIdescO, (acc_prev || kk > 0) ? 1u : 0u);
      };
      auto qdesc = [&](int b, int t) -> uint64_t { return dQ0 + (((2 * b + t) * C::kTileBytes) >> 4); };
      int np[2] = {0, 0};  // P phases consumed per tile
      bool ok = true;
      PUnit cur = {}, nxt = {};
      bool has_nxt = false;
      int base_item = 0;
      int occ[2] = {0, 0}, occ_n[2] = {0, 0};
      // interior step (1 <= jj <= n_max - 2): the general body
      auto inner = [&](int jj) -> bool {
        const int iv = base_item + 2 * jj + 1, ik = iv + 1;
        const int sv = iv % C::kRing, sk = ik % C::kRing;
        const bool pv0 = jj < cur.jhi[0], pv1 = jj < cur.jhi[1];
        {
          const bool a = mbar_try_wait(full(sv), (iv / C::kRing) & 1);
          const bool b = mbar_try_wait(full(sk), (ik / C::kRing) & 1);
          const bool c = !pv0 || mbar_try_wait(bar(kPBarP + 0), np[0] & 1);
          if (!uniform(a && b && c)) {
            if (!uniform(mbar_wait(full(sv), (iv / C::kRing) & 1, abort_flag))) return false;
            if (!uniform(mbar_wait(full(sk), (ik / C::kRing) & 1, abort_flag))) return false;
            if (pv0 && !uniform(mbar_wait(bar(kPBarP + 0), np[0] & 1, abort_flag))) return false;
          }
        }
        tc_fence_after();
        if (pv0) {
          ++np[0];
          gemm2(0, sv, jj > lo_(cur, 0));
          if (jj == cur.jhi[0] - 1) mma_commit_elect(bar(kPBarOFinal + 0));
        }
        if (jj + 1 < cur.jhi[0]) {
          gemm1(0, dq[0], sk);
          mma_commit_elect(bar(kPBarS + 0));
          if (jj + 2 == cur.jhi[0]) mma_commit_elect(bar(kPBarQFree + 2 * qb[0] + 0));
        }
        if (pv1) {
          if (!uniform(mbar_wait(bar(kPBarP + 1), np[1] & 1, abort_flag))) return false;
          ++np[1];
          tc_fence_after();
          gemm2(1, sv, jj > lo_(cur, 1));
          if (jj == cur.jhi[1] - 1) mma_commit_elect(bar(kPBarOFinal + 1));
        }
        mma_commit_elect(empty(sv));
        if (jj + 1 < cur.jhi[1]) {
          gemm1(1, dq[1], sk);
          mma_commit_elect(bar(kPBarS + 1));
          if (jj + 2 == cur.jhi[1]) mma_commit_elect(bar(kPBarQFree + 2 * qb[1] + 1));
        }
        mma_commit_elect(empty(sk));
        return true;
      };
      // interior step with both tiles inside their ranges and no tile's last
      // S or P V in it: every product issued, no branch around the MMAs
      auto steady = [&](int jj) -> bool {
        const int iv = base_item + 2 * jj + 1, ik = iv + 1;
        const int sv = iv % C::kRing, sk = ik % C::kRing;
        const uint32_t phv = (iv / C::kRing) & 1, phk = (ik / C::kRing) & 1;
        const uint32_t ph0 = np[0] & 1, ph1 = np[1] & 1;
        const bool a = mbar_try_wait(full(sv), phv);
        const bool b = mbar_try_wait(full(sk), phk);
        const bool c = mbar_try_wait(bar(kPBarP + 0), ph0);
        if (!uniform(a && b && c)) {
          if (!uniform(mbar_wait(full(sv), phv, abort_flag)) || !uniform(mbar_wait(full(sk), phk, abort_flag)) ||
              !uniform(mbar_wait(bar(kPBarP + 0), ph0, abort_flag)))
            return false;
        }
        tc_fence_after();
        gemm2(0, sv, true);
        gemm1(0, dq[0], sk);
        mma_commit_elect(bar(kPBarS + 0));
        if (!uniform(mbar_try_wait(bar(kPBarP + 1), ph1))) {
          if (!uniform(mbar_wait(bar(kPBarP + 1), ph1, abort_flag))) return false;
        }
        tc_fence_after();
        gemm2(1, sv, true);
        mma_commit_elect(empty(sv));
        gemm1(1, dq[1], sk);
        mma_commit_elect(bar(kPBarS + 1));
        mma_commit_elect(empty(sk));
        ++np[0];
        ++np[1];
        return true;
      };
      // first and last step of a unit
      auto boundary = [&](int jj) -> bool {
        const bool last = jj + 1 == cur.n_max;
        const int iv = base_item + 2 * jj + 1, ik = iv + 1;
        const int sv = iv % C::kRing, sk = ik % C::kRing;
        const bool has_k = !last || has_nxt;
        const bool pv0 = jj >= lo_(cur, 0) && jj < cur.jhi[0], pv1 = jj >= lo_(cur, 1) && jj < cur.jhi[1];
        // the next unit's first S products: only for tiles whose range starts
        // at its first K/V tile (a tile starting one later gets its first S
        // in that unit's first step)
        const bool sn0 = last ? (has_nxt && nxt.jhi[0] > 0 && lo_(nxt, 0) == 0) : (jj + 1 < cur.jhi[0]);
        const bool sn1 = last ? (has_nxt && nxt.jhi[1] > 0 && lo_(nxt, 1) == 0) : (jj + 1 < cur.jhi[1]);
        if (!uniform(mbar_wait(full(sv), (iv / C::kRing) & 1, abort_flag))) return false;
        if (has_k && !uniform(mbar_wait(full(sk), (ik / C::kRing) & 1, abort_flag))) return false;
        if (pv0 && !uniform(mbar_wait(bar(kPBarP + 0), np[0] & 1, abort_flag))) return false;
        if (last) {
          if (sn0 && !uniform(mbar_wait(bar(kPBarQFull + 2 * qb_n[0] + 0), (occ_n[0] / C::kQBufs) & 1, abort_flag))) return false;
          if (sn1 && !uniform(mbar_wait(bar(kPBarQFull + 2 * qb_n[1] + 1), (occ_n[1] / C::kQBufs) & 1, abort_flag))) return false;
        } else if (jj == 0) {
          // a tile whose range starts one K/V tile late: its first S is issued here
          if (sn0 && lo_(cur, 0) == 1 &&
              !uniform(mbar_wait(bar(kPBarQFull + 2 * qb[0] + 0), (occ[0] / C::kQBufs) & 1, abort_flag))) return false;
          if (sn1 && lo_(cur, 1) == 1 &&
              !uniform(mbar_wait(bar(kPBarQFull + 2 * qb[1] + 1), (occ[1] / C::kQBufs) & 1, abort_flag))) return false;
        }
        tc_fence_after();
        if (pv0) {
          ++np[0];
          gemm2(0, sv, jj > lo_(cur, 0));
          if (jj == cur.jhi[0] - 1) mma_commit_elect(bar(kPBarOFinal + 0));
        }
        if (sn0) {
          gemm1(0, last ? dq_n[0] : dq[0], sk);
          mma_commit_elect(bar(kPBarS + 0));
          if (last ? (nxt.jhi[0] == 1) : (jj + 2 == cur.jhi[0]))
            mma_commit_elect(bar(kPBarQFree + 2 * (last ? qb_n[0] : qb[0]) + 0));
        }
        if (pv1) {
          if (!uniform(mbar_wait(bar(kPBarP + 1), np[1] & 1, abort_flag))) return false;
          ++np[1];
          tc_fence_after();
          gemm2(1, sv, jj > lo_(cur, 1));
          if (jj == cur.jhi[1] - 1) mma_commit_elect(bar(kPBarOFinal + 1));
        }
        mma_commit_elect(empty(sv));
        if (sn1) {
          gemm1(1, last ? dq_n[1] : dq[1], sk);
          mma_commit_elect(bar(kPBarS + 1));
          if (last ? (nxt.jhi[1] == 1) : (jj + 2 == cur.jhi[1]))
            mma_commit_elect(bar(kPBarQFree + 2 * (last ? qb_n[1] : qb[1]) + 1));
        }
        if (has_k) mma_commit_elect(empty(sk));
        return true;
      };
      if (get_unit(0, cur, 2) == 1) {
        // prologue: the first unit's first S products
        for (int t = 0; t < 2 && ok; ++t)
          if (cur.jhi[t] > 0) ok = uniform(mbar_wait(bar(kPBarQFull + t), 0, abort_flag));
        if (ok) ok = uniform(mbar_wait(full(0), 0, abort_flag));
        if (ok) {
          tc_fence_after();
          for (int t = 0; t < 2; ++t)
            if (cur.jhi[t] > 0 && lo_(cur, t) == 0) {
              gemm1(t, qdesc(0, t), 0);
              mma_commit_elect(bar(kPBarS + t));
              if (cur.jhi[t] == 1) mma_commit_elect(bar(kPBarQFree + t));
            }
          mma_commit_elect(empty(0));
        }
        for (int k = 0; ok; ++k) {
          const int rn = get_unit(k + 1, nxt, 2);
          if (rn < 0) {
            ok = false;
            break;
          }
          has_nxt = rn == 1;
          for (int t = 0; t < 2; ++t) {
            occ_n[t] = occ[t] + (cur.jhi[t] > 0 ? 1 : 0);
            qb[t] = occ[t] % C::kQBufs;
            qb_n[t] = occ_n[t] % C::kQBufs;
            dq[t] = qdesc(qb[t], t);
            dq_n[t] = qdesc(qb_n[t], t);
          }
          // steady range [1, s_hi): both tiles present, no last S or P V of either
          // (and past both tiles' first P V)
          const int s_lo = max(lo_(cur, 0), lo_(cur, 1)) + 1;
          int s_hi = 1;
          if (cur.jhi[1] > 0) s_hi = max(1, min(cur.jhi[0], cur.jhi[1]) - 2);
          const int n = cur.n_max;
          ok = boundary(0);
          int jj = 1;
          for (; ok && jj < s_lo && jj < n - 1; ++jj) ok = inner(jj);
          for (; ok && jj < s_hi && jj < n - 1; ++jj) ok = steady(jj);
          for (; ok && jj < n - 1; ++jj) ok = inner(jj);
          if (ok && n > 1) ok = boundary(n - 1);
          if (!ok || !has_nxt) break;
          base_item += 2 * cur.n_max;
          cur = nxt;
          occ[0] = occ_n[0];
          occ[1] = occ_n[1];
        }
      }
      if (!ok) report_wait_failure(abort_flag, 4u);
      // drain: every MMA issued so far has completed once this barrier flips
      mma_commit_elect(bar(kPBarDrain));
      uniform(mbar_wait(bar(kPBarDrain), 0, nullptr));
    }
  } else {
    regs_inc<C::kRegSoftmax>();
    // ============== softmax, correction and epilogue (warps 0-7) =============
    const int t = warp >> 2;
    const int q = warp & 3;
    const int row_local = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t tS = lane_base + (t ? 128u : 0u);
    const uint32_t tO = lane_base + C::kTmO + static_cast<uint32_t>(t * D);
    const float c = p.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const bool o_aligned32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
    int ns = 0;   // S phases consumed
    int occ = 0;  // units in which this tile was present so far (O-final phases)
    bool ok = true;
    PUnit u;
    for (int k = 0; ok; ++k) {
      const int r = get_unit(k, u, 2);
      if (r < 0) {
        ok = false;
        break;
      }
      if (r == 0) break;
      const int nt = u.jhi[t] - lo_(u, t);
      if (nt == 0) continue;
      const int row = u.row0[t] + row_local;
      const int key0 = (j0_(u) + lo_(u, t)) * C::kBN;  // first key of the tile's first K/V tile
      // keys past Nk (the ragged last tile), causal past the row, and outside
      // a window's band are masked
      int row_key_lo = 0, row_key_end = (MASK == kMaskCausal) ? min(p.Nk, row + 1) : p.Nk;
      if (MASK == kMaskWindow) {
        row_key_lo = static_cast<int>(max(-1ll, static_cast<long long>(row) + p.diag_off - p.win_left));
        if (p.win_right >= 0)
          row_key_end = static_cast<int>(
              min(static_cast<long long>(p.Nk), max(-1ll, static_cast<long long>(row) + p.diag_off + p.win_right) + 1));
      }
      float m_bar = NEG_INF;  // reference maximum, base-2 scaled units
      float l = 0.f;
      float r_max = NEG_INF;  // the row's largest score (raw units); see fa_fwd_kernel
      for (int j = 0; j < nt; ++j) {
        bool got = mbar_wait(bar(kPBarS + t), ns & 1, abort_flag);
        ++ns;
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s0[32], s1[32], s2[32], s3[32];
        tmem_ld32(tS + 0, s0);
        tmem_ld32(tS + 32, s1);
        tmem_ld_wait(s0);
        reg_pin(s1);
        tmem_ld32(tS + 64, s2);
        tmem_ld32(tS + 96, s3);
        float* const f0 = reinterpret_cast<float*>(s0);
        float* const f1 = reinterpret_cast<float*>(s1);
        float* const f2 = reinterpret_cast<float*>(s2);
        float* const f3 = reinterpret_cast<float*>(s3);
        const int k0 = key0 + j * C::kBN;
        const int lim_lo = MASK == kMaskWindow ? min(C::kBN, max(0, row_key_lo - k0)) : 0;
        const int lim_hi = min(C::kBN, max(0, row_key_end - k0));
        const bool masked = lim_lo > 0 || lim_hi < C::kBN;
        if (masked) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < lim_lo || i >= lim_hi) f0[i] = NEG_INF;
            if (32 + i < lim_lo || 32 + i >= lim_hi) f1[i] = NEG_INF;
          }
        }
        float mx0 = fmax3(f0[0], f0[1], f1[0]), mx1 = fmax3(f0[2], f0[3], f1[1]);
#pragma unroll
        for (int i = 2; i < 16; ++i) {
          if (i & 1) mx1 = fmax3(mx1, f0[2 * i], f0[2 * i + 1]);
          else mx0 = fmax3(mx0, f0[2 * i], f0[2 * i + 1]);
        }
#pragma unroll
        for (int i = 2; i < 32; i += 2) mx0 = fmax3(mx0, f1[i], f1[i + 1]);
        tmem_ld_wait(s2);
        reg_pin(s3);
        if (masked) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (64 + i < lim_lo || 64 + i >= lim_hi) f2[i] = NEG_INF;
            if (96 + i < lim_lo || 96 + i >= lim_hi) f3[i] = NEG_INF;
          }
        }
        float mx2 = fmax3(f2[0], f2[1], f3[0]), mx3 = fmax3(f2[2], f2[3], f3[1]);
#pragma unroll
        for (int i = 2; i < 16; ++i) {
          if (i & 1) mx3 = fmax3(mx3, f2[2 * i], f2[2 * i + 1]);
          else mx2 = fmax3(mx2, f2[2 * i], f2[2 * i + 1]);
        }
#pragma unroll
        for (int i = 2; i < 32; i += 2) mx2 = fmax3(mx2, f3[i], f3[i + 1]);
        const float s_max = fmaxf(fmax3(mx0, mx1, mx2), mx3);
        r_max = fmaxf(r_max, s_max);
        const float m_new = s_max * c;
        const bool need = m_new > m_bar + 8.0f;
        const bool any_need = __any_sync(0xffffffffu, need);
        float alpha = 1.0f;
        if (need) {
          alpha = ex2(m_bar - m_new);  // 0 on the first visible tile (m_bar = -inf)
          m_bar = m_new;
          l *= alpha;
        }
        const float neg_ref = (m_bar == NEG_INF) ? 0.f : -m_bar;
        float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
        auto emit = [&](const float* f, uint32_t col) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            fma2(x0, x1, f[2 * i], f[2 * i + 1], c, neg_ref);
            const float e0 = ex2(x0), e1 = ex2(x1);
            if (i & 1) add2(ls2, ls3, e0, e1);
            else add2(ls0, ls1, e0, e1);
            pk[i] = pack_bf16(e0, e1);
          }
          tmem_st16(tS + col, pk);
        };
        emit(f0, 0);
        emit(f1, 16);
        emit(f2, 32);
        emit(f3, 48);
        l += (ls0 + ls1) + (ls2 + ls3);
        // correction: O *= alpha for the rows whose reference moved (the
        // previous P V of this tile has completed: S of this tile was issued
        // after it and its commit covers it)
        if (any_need && j > 0) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + cc * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kPBarP + t));
      }
      if (!ok) break;
      // ---- epilogue of this unit's tile: O / l to bf16, LSE --------------
      bool got = mbar_wait(bar(kPBarOFinal + t), occ & 1, abort_flag);
      ++occ;
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the row's largest P counted as rounded for P V (see fa_fwd_kernel)
      float l_o = l;
      if (l > 0.f) {
        const float e_max = ex2(fmaf(r_max, c, -m_bar));
        l_o += __uint_as_float(pack_bf16(e_max, 0.f) << 16) - e_max;
      }
      const float inv_l = (l > 0.f) ? (1.0f / l_o) : 0.f;
      const bool store = row < p.Nq;
      uint16_t* const orow = static_cast<uint16_t*>(p.o) + (static_cast<size_t>(u.bh) * p.Nq + row) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_ld_wait(o);
        if (store) {
          // a row is D * 2 = 256 bytes from a 256-byte multiple: with a 32-byte
          // aligned O every store fills whole sectors
          if (o_aligned32) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                w[i] = pack_bf16(__uint_as_float(o[16 * h + 2 * i]) * inv_l, __uint_as_float(o[16 * h + 2 * i + 1]) * inv_l);
              st_global_v8(orow + cc * 32 + h * 16, w);
            }
          } else {
            uint4* const o4 = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              o4[cc * 4 + i] = make_uint4(pack_bf16(__uint_as_float(o[8 * i + 0]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l),
                                          pack_bf16(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l),
                                          pack_bf16(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l),
                                          pack_bf16(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l));
          }
        }
      }
      if (store)
        p.lse[static_cast<size_t>(u.bh) * p.Nq + row] =
            (l > 0.f) ? (m_bar + __log2f(l)) * 0.69314718055994530942f : NEG_INF;
      // O has been read before this tile hands over its next P: the next
      // unit's first P V (which overwrites O) cannot start earlier
      tc_fence_before();
    }
    if (!ok) report_wait_failure(abort_flag, 1u);
  }

  // ---- teardown -----------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == C::kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
