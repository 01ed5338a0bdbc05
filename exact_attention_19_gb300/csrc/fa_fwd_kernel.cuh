// fa_fwd_kernel.cuh -- the fused exact-attention forward kernel for sm_103a.
//
// Algorithm (FA2 loop order: page "llm-infra-atlas / FlashAttention 01",
// section 3): one CTA owns query tiles and streams every visible K/V tile
// past them.  Per K/V tile j and query tile Q_i:
//   S = Q_i K_j^T                 GEMM-I, tensor cores, fp32 in TMEM
//   mask (causal diagonal tile, ragged key tail) -> -inf
//   m_new = max(m, rowmax S)      online softmax, section 2 of the same page
//   P = 2^(S*c - m_bar)           c = scale * log2(e) (section 4, exp2 form)
//   l = alpha*l + rowsum P; O = alpha*O + P V_j   (GEMM-II into TMEM)
// and at the end O / l and LSE = ln 2 * (m_bar + log2 l) (section 3, 5).
// The l that divides O counts the row's largest P as rounded to bf16 for the
// P V product (LSE keeps the exact l), so that a row dominated by one key
// divides that key's rounded weight by itself.
// The reference m_bar moves only when the candidate maximum exceeds it by
// more than tau = 8 in base-2 units ("conditional softmax rescaling", page
// "pinghaoyang FlashAttention 1-4 guide", FA4 section); the final division
// by the true normaliser keeps the result exact.  S and P never leave the SM.
//
// GB300 mapping (one CTA per SM, 384 threads):
//   warps 0-3  softmax + correction + epilogue for query tile 0 (TMEM lanes 0-127)
//   warps 4-7  the same for query tile 1
//   warp  8    TMA producer: Q tiles once, then K_0, V_0, K_1, V_1, ... through
//              one ring of kRing tile-sized slots (mbarrier full/empty per slot)
//   warp  9    MMA issuer: the whole warp runs the loop, one elected lane
//              issues every tcgen05.mma and commit to mbarriers
//   warps 10-11 idle: they complete warpgroup 2 (warps 8-11), which hands
//              registers to the softmax warpgroups with setmaxnreg (168 at
//              launch; then 184 for warps 0-7 and 128 for warps 8-11, or
//              192 and 120 at d = 64, whose MMA issuer needs fewer), so that
//              the 128-float S row and the loop state fit without spilling
// TMEM (512 columns x 128 lanes x 32 bit):
//   S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D, 256+2D);
//   P_i (bf16, packed in pairs) overwrites the first 64 columns of S_i and is
//   the A operand of GEMM-II straight from TMEM.
// Shared memory: Q0, Q1, then the K/V ring; each tile is 128 rows x D bf16
// stored as D/64 boxes of 128 rows x 128 bytes with the 128-byte swizzle that
// TMA writes and the MMA descriptors read (K-major for Q and K, MN-major for V).
// Epilogue: once a query tile's last MMA has completed its Q buffer is free;
// its warps write O / l there as bf16 in the same swizzled box layout and one
// thread stores the tile with TMA (rows past Nq are clipped by the tensor map).
// The single-tile instantiation (TILES = 1, d = 64, short causal key ranges)
// keeps warps 0-3 for its one query tile, warp 4 as producer and warp 5 as MMA
// issuer, 256 TMEM columns (S [0,128), O [128,192)) and a 5-slot ring, so two
// CTAs share an SM.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "fa_ptx.cuh"

namespace fa {

// Device status word: bit 0 set when any wait gave up; bits 8.. hold the
// roles that gave up (1 softmax, 2 producer, 4 MMA, 8 epilogue).
__device__ unsigned int g_fa_status;

struct FwdParams {
  void* o;            // bf16 [BH, Nq, D]
  float* lse;         // fp32 [BH, Nq]
  int Nq, Nk;
  int n_pairs;        // CTAs per (b, h): ceil(Nq / (128 * TILES)), query-tile pairs or single tiles
  float scale_log2;   // scale * log2(e)
  // window mask only: key j is visible to query row i iff
  //   i + diag_off - win_left <= j <= i + diag_off + win_right  (a negative bound: unbounded)
  int win_left, win_right, diag_off;
  // split-KV only: CTAs per pair, K/V tiles per split, and the partial results
  int n_splits, split_tiles;
  // causal only: heads per scheduling group (their K/V fit in a quarter of the L2)
  int lpt_group;
  float* o_part;      // fp32 [n_splits, BH * Nq, D], each slice normalised by its own l
  float* lse_part;    // fp32 [n_splits, BH * Nq], m_bar + log2(l) in base-2 scaled units
  long long rows;     // BH * Nq
};

// TILES = 2: two query tiles per CTA (softmax ping-pong), one CTA per SM.
// TILES = 1 (d = 64): one query tile per CTA in half the TMEM and shared
// memory, so that two CTAs share an SM and each one's MMA checks, start and
// end overlap the other's work; taken for short causal key ranges, where the
// fixed per-CTA cost weighs most.
template <int D, int TILES = 2>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(TILES == 2 || (TILES == 1 && D == 64), "query tiles per CTA");
  static constexpr int kTiles = TILES;
  static constexpr int kWarpProd = 4 * kTiles, kWarpMma = 4 * kTiles + 1;
  // two query tiles: 12 warps (softmax 0-7, producer 8, MMA 9, idle 10-11),
  // so that warps 8-11 form a whole warpgroup whose registers setmaxnreg
  // moves to the softmax warpgroups; one tile: 6 warps, no register move
  static constexpr int kThreads = (kTiles == 2) ? 384 : 32 * (4 * kTiles + 2);
  static constexpr int kRegLaunch = 168;   // what ptxas gives 384 threads at one CTA per SM (checked by the host)
  static constexpr int kRegSoftmax = (D == 64) ? 192 : 184;  // warpgroups 0 and 1
  static constexpr int kRegMisc = (D == 64) ? 120 : 128;     // warpgroup 2
  static_assert(kTiles == 1 || 2 * 128 * kRegSoftmax + 128 * kRegMisc <= kThreads * kRegLaunch, "register split");
  static_assert(kRegMisc <= kRegLaunch && kRegSoftmax >= kRegLaunch, "setmaxnreg direction");
  static constexpr int kMinBlocks = (kTiles == 1) ? 2 : 1;  // CTAs per SM
  static constexpr int kBM = 128;  // query rows per tile (MMA M)
  static constexpr int kBN = 128;  // keys per tile
  static constexpr int kRing = (D == 128 || kTiles == 1) ? 5 : 8;  // K/V ring slots (K and V alternate)
  static constexpr int kBoxes = D / 64;  // 128-byte swizzle boxes per row
  static constexpr uint32_t kBoxBytes = 128u * 128u;
  static constexpr uint32_t kTileBytes = kBoxes * kBoxBytes;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kRingOff = kTiles * kTileBytes;
  static constexpr uint32_t kBarOff = kRingOff + kRing * kTileBytes;
  static constexpr uint32_t kBarBytes = 512;
  static constexpr uint32_t kSmemBytes = kBarOff + kBarBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = (kTiles == 1) ? 256 : 512;
  static constexpr uint32_t kTmS0 = 0, kTmS1 = 128, kTmO0 = (kTiles == 1) ? 128 : 256, kTmO1 = 256 + D;
  static constexpr uint32_t kIdescS = idesc_bf16(128, 128, false);  // S = Q K^T
  static constexpr uint32_t kIdescO = idesc_bf16(128, D, true);     // O += P V
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kMinBlocks == 1 || kMinBlocks * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
};

// barrier slots (8 bytes each) inside the barrier block; the ring's full
// barriers start at kBarRing, its empty barriers right after them
enum : int { kBarQ = 0, kBarS = 2, kBarP = 4, kBarO = 6, kBarDrain = 8, kBarEpi = 9, kBarRing = 11 };
constexpr uint32_t kTmemSlotOff = 448, kAbortOff = 452;

__device__ __forceinline__ void report_wait_failure(volatile int* abort, unsigned role) {
  *abort = 1;
  atomicOr(&g_fa_status, 1u | (role << 8));
}

// MASK: kMaskNone, kMaskCausal (key j visible to row i iff j <= i, Nq == Nk)
// or kMaskWindow (the general window of FwdParams); each query tile visits
// only the K/V tiles its rows can see and masks the partly visible ones.  The
// causal case is the window (-1, 0) with diag_off 0, specialised at compile
// time so that its bounds fold to constants.
// SPLIT: the CTA covers K/V tiles [split * split_tiles, (split+1) * split_tiles)
// of its pair and writes a partial result; fa_splitkv_combine_kernel merges them.
enum : int { kMaskNone = 0, kMaskCausal = 1, kMaskWindow = 2 };

template <int D, int MASK, bool SPLIT, int TILES = 2>
__global__ void __launch_bounds__(Cfg<D, TILES>::kThreads, Cfg<D, TILES>::kMinBlocks)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
  using C = Cfg<D, TILES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw_addr);

  const uint32_t bar0 = base + C::kBarOff;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  auto full = [&](int slot) -> uint32_t { return bar(kBarRing + slot); };
  auto empty = [&](int slot) -> uint32_t { return bar(kBarRing + C::kRing + slot); };
  auto slot_addr = [&](int slot) -> uint32_t { return base + C::kRingOff + slot * C::kTileBytes; };
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + C::kBarOff + kTmemSlotOff);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sbase + C::kBarOff + kAbortOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // split-KV: the merge kernel is launched as a programmatic dependent of this
  // grid; let it be scheduled once every CTA of this grid has started (it
  // waits for this grid's completion and memory before reading the partials)
  if (SPLIT) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQ + 0), 1);
    mbar_init(bar(kBarQ + 1), 1);
    mbar_init(bar(kBarS + 0), 1);
    mbar_init(bar(kBarS + 1), 1);
    mbar_init(bar(kBarP + 0), 128);
    mbar_init(bar(kBarP + 1), 128);
    mbar_init(bar(kBarO + 0), 1);
    mbar_init(bar(kBarO + 1), 1);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarEpi + 0), 128);
    mbar_init(bar(kBarEpi + 1), 128);
    for (int s = 0; s < C::kRing; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
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

  // ---- work item: (b*H + h, pair of query tiles[, K/V split]) -------------
  int cta = blockIdx.x;
  int split = 0;
  if (SPLIT) {
    split = cta % p.n_splits;
    cta /= p.n_splits;
  }
  int bh = cta / p.n_pairs;
  int pair = cta % p.n_pairs;
  if (MASK == kMaskCausal) {
    // Causal CTAs differ in work (pair i sees 2i + 2 K/V tiles, a single
    // tile i sees i + 1).  Heads are
    // taken in groups whose K/V fit in a quarter of the L2; inside a group the
    // heaviest pairs of all its heads run first, so a group's last wave holds
    // its lightest pairs (longest-processing-time-first order), while the
    // CTAs in flight at any time share the K/V tiles of a few heads.
    const int n_bh = static_cast<int>(gridDim.x / (SPLIT ? p.n_splits : 1)) / p.n_pairs;
    const int per_group = p.lpt_group * p.n_pairs;
    const int g0 = (cta / per_group) * p.lpt_group;
    const int g_heads = min(p.lpt_group, n_bh - g0);
    const int within = cta - (cta / per_group) * per_group;
    bh = g0 + within % g_heads;
    pair = p.n_pairs - 1 - within / g_heads;
  }
  const int n_kv_all = (p.Nk + C::kBN - 1) / C::kBN;
  const int kv_lo = SPLIT ? split * p.split_tiles : 0;  // this CTA's slice of K/V tiles
  const int kv_hi = SPLIT ? min(n_kv_all, kv_lo + p.split_tiles) : n_kv_all;
  // visible K/V tiles [jlo, jhi) of each query tile, within the slice
  int row0[2], jlo[2], jhi[2], nkv[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = C::kTiles * pair + t;
    row0[t] = qt * C::kBM;
    int lo = 0, hi = 0;
    if (t < C::kTiles && row0[t] < p.Nq) {
      hi = n_kv_all;
      if (MASK == kMaskCausal) {
        hi = min(n_kv_all, qt + 1);
      } else if (MASK == kMaskWindow) {
        const long long r_first = row0[t], r_last = min(row0[t] + C::kBM, p.Nq) - 1;
        long long key_lo = 0, key_hi = p.Nk - 1;
        if (p.win_left >= 0) key_lo = max(0ll, r_first + p.diag_off - p.win_left);
        if (p.win_right >= 0) key_hi = min(key_hi, r_last + p.diag_off + p.win_right);
        if (key_lo > key_hi) {
          hi = 0;  // no row of this tile sees a key
        } else {
          lo = static_cast<int>(key_lo / C::kBN);
          hi = static_cast<int>(key_hi / C::kBN) + 1;
        }
      }
      lo = max(lo, kv_lo);
      hi = min(hi, kv_hi);
      if (hi < lo) hi = lo;
    }
    jlo[t] = lo;
    jhi[t] = hi;
    nkv[t] = hi - lo;
  }
  // the CTA streams the union of the two ranges: K/V tiles [J0, J0 + n_max)
  int J0 = 0, n_max = 0;
  if (nkv[0] > 0 || nkv[1] > 0) {
    J0 = nkv[0] == 0 ? jlo[1] : (nkv[1] == 0 ? jlo[0] : min(jlo[0], jlo[1]));
    const int J1 = nkv[0] == 0 ? jhi[1] : (nkv[1] == 0 ? jhi[0] : max(jhi[0], jhi[1]));
    n_max = J1 - J0;
  }
  const int n_items = 2 * n_max;  // ring items: K_j = item 2j, V_j = item 2j+1

  if (warp >= 4 * TILES) {
    // warpgroup 2 (producer, MMA issuer and, with two tiles, two idle warps)
    // gives registers to the softmax warpgroups
    if constexpr (TILES == 2) regs_dec<C::kRegMisc>();
    if (warp == C::kWarpProd) {
      // ======================= TMA producer =================================
      // d = 64: the whole warp runs the loop (each barrier outcome made uniform
      // with a vote) and one lane chosen by elect.sync issues every expect-tx
      // and copy, as in the MMA issuer below.  A d = 64 K/V tile carries half
      // the MMA work of a d = 128 one, so the producer's issue latency weighs
      // twice as much there.  d = 128: lane 0 alone.
      auto uniform = [](bool v) -> bool {
        if constexpr (D == 64) return __all_sync(0xffffffffu, v);
        else return v;
      };
      auto expect_tx = [](uint32_t b, uint32_t bytes) {
        if constexpr (D == 64) mbar_arrive_expect_tx_elect(b, bytes);
        else mbar_arrive_expect_tx(b, bytes);
      };
      auto load = [](uint32_t dst, const CUtensorMap* map, uint32_t b, int x, int y, int z) {
        if constexpr (D == 64) tma_load_3d_elect(dst, map, b, x, y, z);
        else tma_load_3d(dst, map, b, x, y, z);
      };
      if (D == 64 || lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmO);
        for (int t = 0; t < 2; ++t) {
          if (nkv[t] == 0) continue;
          const uint32_t dst = base + C::kQOff + t * C::kTileBytes;
          expect_tx(bar(kBarQ + t), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            load(dst + b * C::kBoxBytes, &tmQ, bar(kBarQ + t), b * 64, row0[t], bh);
        }
        int issued = 0;
        for (int item = 0; item < n_items; ++item) {
          const int s = item % C::kRing;
          const uint32_t ph = (item / C::kRing) & 1;
          if (!uniform(mbar_wait(empty(s), ph ^ 1u, abort_flag))) {
            report_wait_failure(abort_flag, 2u);
            break;
          }
          const CUtensorMap* map = (item & 1) ? &tmV : &tmK;
          expect_tx(full(s), C::kTileBytes);
          for (int b = 0; b < C::kBoxes; ++b)
            load(slot_addr(s) + b * C::kBoxBytes, map, full(s), b * 64, (J0 + (item >> 1)) * C::kBN, bh);
          issued = item + 1;
        }
        if (*abort_flag) {
          // Let every copy already issued land before the CTA can exit: the
          // last item issued into each slot is among the final kRing items.
          for (int item = max(0, issued - C::kRing); item < issued; ++item)
            uniform(mbar_wait(full(item % C::kRing), (item / C::kRing) & 1, nullptr));
          for (int t = 0; t < 2; ++t)
            if (nkv[t] > 0) uniform(mbar_wait(bar(kBarQ + t), 0, nullptr));
        }
      }
    } else if (warp == C::kWarpMma) {
      // ======================= MMA issuer ====================================
      // The whole warp runs the issue loop on warp-uniform values (every
      // barrier outcome made uniform with a vote); one lane chosen by
      // elect.sync issues each tcgen05.mma and commit, with no branch around the
      // instruction.  Same-box A/B against lane 0 alone: +4% to +7.5% at d = 64,
      // and at d = 128 +1% together with the branch-free steady body below.
      auto mma_ss_x = [](uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
        mma_ss_elect(d_tmem, a_desc, b_desc, idesc, acc);
      };
      auto mma_ts_x = [](uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
        mma_ts_elect(d_tmem, a_tmem, b_desc, idesc, acc);
      };
      auto commit_x = [](uint32_t b) { mma_commit_elect(b); };
      auto uniform = [](bool v) -> bool { return __all_sync(0xffffffffu, v); };
      {
        // descriptors: start address lives in bits 0-13 (address >> 4), so a
        // byte offset is added to a base descriptor as (offset >> 4)
        const uint64_t dQ0 = sdesc_sw128(base + C::kQOff, 16, 1024);
        const uint64_t dQ1 = sdesc_sw128(base + C::kQOff + C::kTileBytes, 16, 1024);
        const uint64_t dK0 = sdesc_sw128(base + C::kRingOff, 16, 1024);
        const uint64_t dV0 = sdesc_sw128(base + C::kRingOff, C::kBoxBytes, 1024);
        const uint32_t tS[2] = {tmem + C::kTmS0, tmem + C::kTmS1};
        const uint32_t tO[2] = {tmem + C::kTmO0, tmem + C::kTmO1};
        auto gemm1 = [&](int t, int slot) {
          const uint64_t dq = t ? dQ1 : dQ0;
          const uint64_t dk = dK0 + ((slot * C::kTileBytes) >> 4);
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ss_x(tS[t], dq + off, dk + off, C::kIdescS, kk > 0 ? 1u : 0u);
          }
        };
        auto gemm2 = [&](int t, int slot, bool acc_prev) {
          const uint64_t dv = dV0 + ((slot * C::kTileBytes) >> 4);
  #pragma unroll
          for (int kk = 0; kk < C::kBN / 16; ++kk)
            mma_ts_x(tO[t], tS[t] + kk * 8, dv + ((kk * 2048) >> 4), C::kIdescO, (acc_prev || kk > 0) ? 1u : 0u);
        };
        auto wait_item = [&](int item) -> bool {
          return uniform(mbar_wait(full(item % C::kRing), (item / C::kRing) & 1, abort_flag));
        };
        auto uwait = [&](uint32_t b, uint32_t ph) -> bool { return uniform(mbar_wait(b, ph, abort_flag)); };
        // is K/V tile j (absolute index within the head) visible to query tile t?
        auto in_range = [&](int t, int j) -> bool { return j >= jlo[t] && j < jhi[t]; };
        bool ok = true;
        for (int t = 0; t < 2 && ok; ++t)
          if (nkv[t] > 0) ok = uwait(bar(kBarQ + t), 0);
        if (ok && n_max > 0) ok = wait_item(0);
        if (ok && n_max > 0) {
          tc_fence_after();
          for (int t = 0; t < 2; ++t)
            if (nkv[t] > 0 && jlo[t] == J0) {
              gemm1(t, 0);
              commit_x(bar(kBarS + t));
            }
          commit_x(empty(0));
        }
        // Issue order per K/V tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), with
        // every barrier check of the first half gathered in one place (each
        // check behind queued MMAs costs a pipe bubble, consecutive ones cost one).
        // A tile whose range starts after J0 gets its first S when j + 1 enters it.
        auto general = [&](int jj) -> bool {
          const int j = J0 + jj;
          const int iv = 2 * jj + 1, ik = 2 * jj + 2;  // ring items of V_j and K_{j+1}
          const int sv = iv % C::kRing, sk = ik % C::kRing;
          const bool has_next = (jj + 1) < n_max;
          const bool pv0 = in_range(0, j), pv1 = in_range(1, j);
          {
            // the three checks are issued back to back so their latencies overlap
            const bool a = mbar_try_wait(full(sv), (iv / C::kRing) & 1);
            const bool b = !has_next || mbar_try_wait(full(sk), (ik / C::kRing) & 1);
            const bool c = !pv0 || mbar_try_wait(bar(kBarP + 0), (j - jlo[0]) & 1);
            if (!uniform(a && b && c)) {
              if (!wait_item(iv)) return false;
              if (has_next && !wait_item(ik)) return false;
              if (pv0 && !uwait(bar(kBarP + 0), (j - jlo[0]) & 1)) return false;
            }
          }
          tc_fence_after();
          if (pv0) {
            gemm2(0, sv, j > jlo[0]);
            if (j == jhi[0] - 1) commit_x(bar(kBarO + 0));
          }
          if (has_next && in_range(0, j + 1)) {
            gemm1(0, sk);
            commit_x(bar(kBarS + 0));
          }
          if (pv1) {
            if (!uwait(bar(kBarP + 1), (j - jlo[1]) & 1)) return false;
            tc_fence_after();
            gemm2(1, sv, j > jlo[1]);
            if (j == jhi[1] - 1) commit_x(bar(kBarO + 1));
          }
          commit_x(empty(sv));
          if (has_next && in_range(1, j + 1)) {
            gemm1(1, sk);
            commit_x(bar(kBarS + 1));
          }
          if (has_next) commit_x(empty(sk));
          return true;
        };
        // The steady state: K/V tiles j with j - 1, j and j + 1 in both query
        // tiles' ranges, so every product of the tile is issued and none is the
        // last of its tile.  The same issue order without a branch around the
        // MMAs: a barrier test by this thread completes only after its queued
        // MMAs, and a branch next to it costs the pipe about 20 cycles per MMA.
        auto steady = [&](int jj) -> bool {
          const int j = J0 + jj;
          const int iv = 2 * jj + 1, ik = 2 * jj + 2;
          const int sv = iv % C::kRing, sk = ik % C::kRing;
          const uint32_t phv = (iv / C::kRing) & 1, phk = (ik / C::kRing) & 1;
          const uint32_t ph0 = (j - jlo[0]) & 1, ph1 = (j - jlo[1]) & 1;
          const bool a = mbar_try_wait(full(sv), phv);
          const bool b = mbar_try_wait(full(sk), phk);
          const bool c = mbar_try_wait(bar(kBarP + 0), ph0);
          if (!uniform(a && b && c)) {
            if (!uwait(full(sv), phv) || !uwait(full(sk), phk) || !uwait(bar(kBarP + 0), ph0)) return false;
          }
          tc_fence_after();
          gemm2(0, sv, true);
          gemm1(0, sk);
          commit_x(bar(kBarS + 0));
          if (!uniform(mbar_try_wait(bar(kBarP + 1), ph1))) {
            if (!uwait(bar(kBarP + 1), ph1)) return false;
          }
          tc_fence_after();
          gemm2(1, sv, true);
          commit_x(empty(sv));
          gemm1(1, sk);
          commit_x(bar(kBarS + 1));
          commit_x(empty(sk));
          return true;
        };
        // steady range [s_lo, s_hi) of jj; the tiles before and after it take
        // the general body.  With the elected issue it gains at both head sizes
        // (with lane 0 alone it had measured 3% slower at d = 128).
        int s_lo = n_max, s_hi = n_max;
        if (nkv[0] > 0 && nkv[1] > 0) {
          const int lo = max(jlo[0], jlo[1]) + 1 - J0, hi = min(jhi[0], jhi[1]) - 1 - J0;
          if (lo < hi) {
            s_lo = lo;
            s_hi = hi;
          }
        }
        int jj = 0;
        for (; ok && jj < s_lo; ++jj) ok = general(jj);
        for (; ok && jj < s_hi; ++jj) ok = steady(jj);
        for (; ok && jj < n_max; ++jj) ok = general(jj);
        if (!ok) report_wait_failure(abort_flag, 4u);
        // Drain: every MMA issued so far has completed once this barrier flips.
        commit_x(bar(kBarDrain));
        mbar_wait(bar(kBarDrain), 0, nullptr);
      }
    }
  } else {
    if constexpr (TILES == 2) regs_inc<C::kRegSoftmax>();
    // ============== softmax / correction / epilogue (warps 0-7) ===========
    const int t = warp >> 2;        // query tile of this warpgroup
    const int wq = warp & 3;        // TMEM lane quarter
    const int row_local = wq * 32 + lane;
    // this tile's values by select, not by a runtime index (which would put
    // the arrays in local memory and reload them inside the loop)
    const int row0_t = t ? row0[1] : row0[0];
    const int key0_t = (t ? jlo[1] : jlo[0]) * C::kBN;  // first key of the tile's first K/V tile
    const int nkv_t = t ? nkv[1] : nkv[0];
    const int row = row0_t + row_local;
    // keys [row_key_lo, row_key_end) are visible to this row; all sizes fit
    // an int (N < 2^31), the window bounds are clamped into [-1, Nk]
    int row_key_lo = 0, row_key_end = p.Nk;
    if (MASK == kMaskCausal) row_key_end = min(p.Nk, row + 1);
    if (MASK == kMaskWindow) {
      if (p.win_left >= 0)
        row_key_lo = static_cast<int>(max(-1ll, static_cast<long long>(row) + p.diag_off - p.win_left));
      if (p.win_right >= 0)
        row_key_end = static_cast<int>(
            min(static_cast<long long>(p.Nk), max(-1ll, static_cast<long long>(row) + p.diag_off + p.win_right) + 1));
    }
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tS = lane_base + (t == 0 ? C::kTmS0 : C::kTmS1);
    const uint32_t tO = lane_base + (t == 0 ? C::kTmO0 : C::kTmO1);
    const float c = p.scale_log2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    float m_bar = NEG_INF;  // reference maximum, base-2 scaled units
    float l = 0.f;
    // The row's largest score so far (raw units).  The reference only moves
    // when a tile raises the row's maximum, so the reference in force when the
    // largest score was exponentiated is the final m_bar: the epilogue can
    // recompute that P bit for bit.
    float r_max = NEG_INF;
    bool ok = true;
    const int nt = nkv_t;
    for (int j = 0; j < nt; ++j) {
      bool got = mbar_wait(bar(kBarS + t), j & 1, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) { ok = false; break; }
      tc_fence_after();
      // S row in two halves: the second half's TMEM load overlaps the first
      // half's row max.
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

      // masking: columns outside [lim_lo, lim_hi) of this K/V tile are not
      // visible to this row (window / causal bounds, ragged key tail)
      const int k0 = key0_t + j * C::kBN;  // first key of this K/V tile
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
      // P = 2^(S*c - m_ref), rounded to bf16 pairs into the first 64 columns
      // of this tile's S region (16 columns = 32 probabilities per store).
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
      // after it and its commit covers it).
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
      mbar_arrive(bar(kBarP + t));
    }
    if (!ok) report_wait_failure(abort_flag, 1u);
    if (ok && nt > 0) {
      bool got = mbar_wait(bar(kBarO + t), 0, abort_flag);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        report_wait_failure(abort_flag, 8u);
      } else {
        tc_fence_after();
        // O's normaliser counts the row's largest P as rounded to bf16 for P V
        float l_o = l;
        if (l > 0.f) {
          const float e_max = ex2(fmaf(r_max, c, -m_bar));
          l_o += __uint_as_float(pack_bf16(e_max, 0.f) << 16) - e_max;
        }
        const float inv_l = (l > 0.f) ? (1.0f / l_o) : 0.f;
        const bool store = row < p.Nq;
        const size_t grow = static_cast<size_t>(bh) * p.Nq + row;  // row within [BH * Nq]
        if (!SPLIT) {
          // O / l in bf16 is staged in this tile's Q buffer (no MMA reads it
          // once the tile's O barrier has flipped), laid out as the 128-byte
          // swizzled boxes the O tensor map describes: 16-byte chunk c of row
          // r of a box sits at r * 128 + ((c ^ (r & 7)) * 16), so a warp's 32
          // rows cover every bank once per 8 rows.  One thread then writes the
          // tile with TMA stores, which drop the rows past Nq.
          const uint32_t stage = base + C::kQOff + static_cast<uint32_t>(t) * C::kTileBytes +
                                 static_cast<uint32_t>(row_local) * 128u;
          const uint32_t swz = static_cast<uint32_t>(row_local & 7);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
            tmem_ld_wait(o);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t chunk = static_cast<uint32_t>((cc & 1) * 4 + i);  // 16-byte chunk within the box
              st_shared_v4(stage + static_cast<uint32_t>(cc >> 1) * C::kBoxBytes + ((chunk ^ swz) << 4), w[4 * i],
                           w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(kBarEpi + t));
          if (store) {
            const float lse = (l > 0.f) ? (m_bar + __log2f(l)) * 0.69314718055994530942f : NEG_INF;
            p.lse[grow] = lse;
          }
          if (row_local == 0) {
            if (mbar_wait(bar(kBarEpi + t), 0, abort_flag)) {
              const uint32_t src = base + C::kQOff + static_cast<uint32_t>(t) * C::kTileBytes;
#pragma unroll
              for (int b = 0; b < C::kBoxes; ++b) tma_store_3d(&tmO, src + b * C::kBoxBytes, b * 64, row0_t, bh);
              bulk_commit_group();
              bulk_wait_group_read0();
            } else {
              report_wait_failure(abort_flag, 8u);
            }
          }
        } else {
          // partial: O / l in fp32 and the base-2 log-sum-exp of this slice
          const size_t prow = static_cast<size_t>(split) * p.rows + grow;
          float4* const orow = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
            tmem_ld_wait(o);
            if (store) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                orow[cc * 8 + i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                               __uint_as_float(o[4 * i + 2]) * inv_l,
                                               __uint_as_float(o[4 * i + 3]) * inv_l);
            }
          }
          if (store) p.lse_part[prow] = (l > 0.f) ? (m_bar + __log2f(l)) : NEG_INF;
        }
      }
    } else if (!SPLIT && ok && nt == 0 && row < p.Nq) {
      // no row of this tile sees a key (possible under a window): O = 0, LSE = -inf
      uint4* const orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                                   (static_cast<size_t>(bh) * p.Nq + row) * D);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) orow[i] = make_uint4(0u, 0u, 0u, 0u);
      p.lse[static_cast<size_t>(bh) * p.Nq + row] = NEG_INF;
    } else if (SPLIT && ok && nt == 0 && row < p.Nq) {
      // no visible key in this slice: an empty partial (weight 2^-inf = 0)
      const size_t prow = static_cast<size_t>(split) * p.rows + static_cast<size_t>(bh) * p.Nq + row;
      float4* const orow = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
      for (int i = 0; i < D / 4; ++i) orow[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.lse_part[prow] = NEG_INF;
    }
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

// Merge of split-KV partial results, one warp per query row: with slice
// results (O_s, L_s) where O_s is normalised and L_s = log2 of its sum of
// 2^(scaled logit), the row's O = sum_s 2^(L_s - L) O_s and L = log2 sum_s 2^L_s.
// This is the order-insensitive merge of (m, l, O) states of the online
// softmax (page "llm-infra-atlas / FlashAttention 01", section 2).
template <int D>
__global__ void __launch_bounds__(256) fa_splitkv_combine_kernel(const float* __restrict__ o_part,
                                                                 const float* __restrict__ lse_part, void* o,
                                                                 float* lse, long long rows, int n_splits) {
  constexpr int kPer = D / 32;  // elements per lane
  // launched as a programmatic dependent of the sliced forward: wait until that
  // grid has completed and its partial results are visible (a no-op otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float NEG_INF = -__int_as_float(0x7f800000);
  float mx = NEG_INF;
  for (int s = 0; s < n_splits; ++s) mx = fmaxf(mx, lse_part[static_cast<size_t>(s) * rows + row]);
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  if (mx != NEG_INF) {
    for (int s = 0; s < n_splits; ++s) {
      const size_t prow = static_cast<size_t>(s) * rows + row;
      const float w = ex2(lse_part[prow] - mx);
      wsum += w;
      const float* src = o_part + prow * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  uint16_t* orow = static_cast<uint16_t*>(o) + static_cast<size_t>(row) * D + lane * kPer;
  if constexpr (kPer == 4)
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv));
  else
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16(acc[0] * inv, acc[1] * inv);
  if (lane == 0) lse[row] = (wsum > 0.f) ? (mx + __log2f(wsum)) * 0.69314718055994530942f : NEG_INF;
}

}  // namespace fa
