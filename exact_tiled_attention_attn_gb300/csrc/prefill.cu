// prefill.cu - exact tiled attention forward pass on 5th-generation tensor cores (sm_103a).
//
// What it computes ("FlashAttention: attention without the n x n matrix", section
// "Forward pass of FlashAttention"; "Module 07: Fused operators and FlashAttention",
// sections "Online softmax: derivation" and "FlashAttention-2"): for a block of
// 128 query rows, walk the key/value blocks of 128 keys, keep per row the running
// maximum m, the running sum l and the unnormalised output O, rescale l and O by
// 2^(m_old - m_new) when the maximum moves, and divide once at the end. Key blocks
// entirely above the diagonal are never visited when causal; the element mask is
// applied only on blocks that cross the diagonal or the end of the keys.
//
// How it maps onto the GPU (a work unit is two 128-row query tiles that share one K/V
// stream: two query heads of the same K/V group at the same rows, or, when the group
// size is odd, two consecutive row tiles of one head; each persistent CTA runs its units
// one after another):
//   warp 1      TMA producer: Q tiles once, then K and V tiles into one ring of slots
//               (128-byte swizzled boxes of 64 columns x 128 rows).
//   warp 0      MMA issuer (one thread issues): S_q = Q_q K^T into TMEM (fp32), then
//               O_q += P_q V with P read from TMEM (bf16) and V from shared memory.
//               The whole warp runs the issue loop in step and only lane 0's MMAs are
//               issued (a guard predicate), so it never diverges and reconverges around
//               them (3-5 % faster than branching on lane 0). It is warp 0 so that it does
//               not lose issue slots to the softmax warps on its scheduler (measured:
//               warp 9 -> 0 made the d = 64 kernel 1.8 % faster).
//   warp 2      waits for the issuer: it sits in the shared-memory barrier waits for
//               Q and each key block's K/V and hands each "go" to warp 0 through a
//               hardware named barrier (with an acknowledgement, so the two stay in
//               step). One thread's tcgen05 queue holds about one MMA, so every wait
//               the issuer did itself (~150+ clocks under load) would be tensor idle
//               time; a named-barrier handoff costs tens of clocks.
//   warps 3-6   softmax for query tile 0, warps 7-10 for tile 1 (warp w reads TMEM lanes
//               32 (w % 4) .. 32 (w % 4) + 31, so each tile's four warps cover all 128): one thread owns one
//               row (TMEM lane), so row max and row sum need no shuffles; P is
//               written back into the TMEM columns of S and its readiness goes to
//               warp 0 through a named barrier shared by the tile's four warps and the
//               issuer; O is rescaled in TMEM. At the end of a unit they write O with
//               32-byte stores, lane pairs swapping halves so that each store covers 64
//               contiguous bytes of a row.
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [256+d,256+2d);
// P_q aliases the first 64 columns of S_q.
//
// Work distribution: one persistent CTA per SM walks the units in rounds (snake order; causal
// units heaviest first, non-causal ones (batch, head)-major). A non-causal launch whose last
// round would be only partly filled runs that round's units as pieces over consecutive key
// blocks instead, and attn_fwd_merge_kernel combines each unit's pieces (the online-softmax
// merge).
//
// The maximum used as the exponent base is only moved when the new block maximum
// exceeds it by more than 2^8 (in base 2); the normalised result does not depend on
// which finite base is subtracted ("Module 07", section "Online softmax: derivation":
// the factor exp(m - c) cancels between numerator and denominator), and the bound
// keeps every p <= 256, far inside fp32 and bf16 range.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "common.cuh"

namespace gb300 {

constexpr uint64_t kPrefillWaitTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr float kRescaleThreshold = 8.0f;                   // log2 of the allowed growth of p
constexpr int kIterRing = 8;  // per-key-block barriers in flight (kv_ready, iter_done)
// hardware named barriers (0 is __syncthreads) and their thread counts
constexpr uint32_t kBarData = 1, kBarDataAck = 2, kBarP0 = 3;  // kBarP0 + 1 for tile 1
constexpr uint32_t kPair = 64;                // helper warp + issuer warp
constexpr uint32_t kSoftmaxAndIssuer = 160;   // 4 softmax warps + issuer warp
constexpr int kWarpIssuer = 0, kWarpProducer = 1, kWarpHelper = 2, kFirstSoftmaxWarp = 3;

template <int D>
struct PrefillCfg {
  static constexpr int kBM = 128;                  // query rows per tile
  static constexpr int kBN = 128;                  // keys per tile
  // One ring of K/V slots: item 2j holds K(j), item 2j+1 holds V(j), slot = item % kSlots.
  // An odd slot count lets V(j) reuse the slot of K(j-2), freed as soon as S(j-2) is done.
  static constexpr int kSlots = (D == 64) ? 11 : 5;
  static constexpr int kBoxBytes = 128 * 128;      // 128 rows x 64 bf16 columns
  static constexpr int kNumBox = D / 64;
  static constexpr int kTileBytes = kNumBox * kBoxBytes;
  static constexpr int kSmemBytes = (2 + kSlots) * kTileBytes + 1024;
  static constexpr int kTmS0 = 0, kTmS1 = 128, kTmO0 = 256, kTmO1 = 256 + D;
  static constexpr int kThreads = 352;
  static constexpr uint32_t kIdescQK = make_idesc_bf16_f32(128, 128, false);
  static constexpr uint32_t kIdescPV = make_idesc_bf16_f32(128, D, true);
  // The producer runs up to about kSlots / 2 key blocks ahead of the MMA thread; the
  // per-block barrier rings must be deeper than that, or a barrier would be re-armed for
  // block j + kIterRing before block j's phase was consumed.
  static_assert(kIterRing >= (kSlots + 1) / 2 + 2, "per-block barrier ring too shallow for the K/V ring");
};

struct PrefillParams {
  __nv_bfloat16* o;
  float* lse;
  int B, Hq, Hkv, Tq, Tk, g;
  int causal;
  int pair_heads;  // 1: tiles are heads (2p, 2p+1) at the same rows; 0: row tiles (2p, 2p+1) of one head
  int n_qt;        // number of query tiles of 128 rows
  int units;       // work units (pairs of query tiles), heaviest first when causal
  int rank_div, rank_mod, rest_div, rest_mod;  // unit -> (row-tile rank, batch-head rest); decode_unit
  // Key-split tail (see decode_item): units [0, full_units) run whole; each later unit runs as
  // `split` pieces over consecutive ranges of its key blocks, whose partial results go to
  // part_o / part_lse2 and are merged by attn_fwd_merge_kernel. items = the work items.
  int full_units, split, items;
  float* part_o;     // [piece][tile 2][row 128][D] fp32, O of the piece normalised by its own l
  float* part_lse2;  // [piece][tile 2][row 128] fp32, m + log2 l of the piece (base 2, scaled scores)
  float c;           // scale * log2(e)
  int o_v8;          // O is 32-byte aligned: the epilogue writes it with 32-byte stores
};

struct UnitInfo {
  int b, kvh;
  int head[2];
  int row0[2];
  int nkv[2];  // key tiles to visit per query tile (0 = tile inactive)
  int kb0;     // first key block (0 unless the item is a piece of a split unit)
  int part;    // piece index into part_o / part_lse2, or -1 for a whole unit
};

__device__ __forceinline__ int kv_tiles_for(const PrefillParams& p, int row0) {
  if (row0 >= p.Tq) return 0;
  const int all = (p.Tk + 127) / 128;
  if (!p.causal) return all;
  const int last_row = min(row0 + 127, p.Tq - 1);
  return min(all, last_row / 128 + 1);
}

// Unit order. Causal: by query-tile rank, heaviest (last rows) first, then (batch, head), so
// that the snake order balances the CTAs. Non-causal (all units equally long): (batch, head)
// major and the row tile fastest, so that the units running at one time cover few heads and
// their K/V blocks are read from L2 rather than DRAM.
__device__ __forceinline__ UnitInfo decode_unit(const PrefillParams& p, int unit) {
  UnitInfo u;
  // rank = (unit / rank_div) % rank_mod and rest = (unit / rest_div) % rest_mod, with the
  // divisors set on the host for the order above (no branch: fewer live registers)
  const int rank = (unit / p.rank_div) % p.rank_mod;
  const int rest = (unit / p.rest_div) % p.rest_mod;
  if (p.pair_heads) {
    const int hp_count = p.Hq / 2;
    const int hp = rest % hp_count;
    u.b = rest / hp_count;
    const int qt = p.causal ? (p.n_qt - 1 - rank) : rank;  // heaviest tiles first when causal
    u.head[0] = 2 * hp;
    u.head[1] = 2 * hp + 1;
    u.row0[0] = u.row0[1] = qt * 128;
  } else {
    const int n_pairs = (p.n_qt + 1) / 2;
    const int h = rest % p.Hq;
    u.b = rest / p.Hq;
    const int tp = p.causal ? (n_pairs - 1 - rank) : rank;
    u.head[0] = u.head[1] = h;
    u.row0[0] = 2 * tp * 128;
    u.row0[1] = (2 * tp + 1) * 128;
  }
  u.kvh = u.head[0] / p.g;
  u.nkv[0] = kv_tiles_for(p, u.row0[0]);
  u.nkv[1] = kv_tiles_for(p, u.row0[1]);
  return u;
}

// Work item -> unit or piece of a unit. A piece covers key blocks [kb0, kb1) of its unit, a
// share of the unit's n blocks; only units whose two tiles visit the same blocks (non-causal)
// are split, so both tiles of a piece visit all of its blocks (or tile 1 none, past Tq).
// kSplit = false: the launch has no split units, so every item is a whole unit.
template <bool kSplit>
__device__ __forceinline__ UnitInfo decode_item(const PrefillParams& p, int item) {
  if (!kSplit) {
    UnitInfo u = decode_unit(p, item);
    u.kb0 = 0;
    u.part = -1;
    return u;
  }
  // one straight-line path for whole units (one piece of all n blocks) and pieces (measured:
  // the branchy form made the compiler spill registers in the softmax warps)
  const bool whole = item < p.full_units;
  const int t = item - p.full_units;
  const int s = whole ? 1 : p.split;
  const int pc = whole ? 0 : t % p.split;
  UnitInfo u = decode_unit(p, whole ? item : p.full_units + t / p.split);
  const int n = max(u.nkv[0], u.nkv[1]);
  const int kb0 = pc * n / s, kb1 = (pc + 1) * n / s;
#pragma unroll
  for (int q = 0; q < 2; ++q) u.nkv[q] = max(0, min(u.nkv[q], kb1) - kb0);
  u.kb0 = kb0;
  u.part = whole ? -1 : t;
  return u;
}

// Key block j has MMA work iff some tile issues S_q(j) (j < nkv_q) or PV_q(j-1) (0 < j <= nkv_q).
__device__ __forceinline__ bool block_has_work(const UnitInfo& u, int j) {
  const int n = max(u.nkv[0], u.nkv[1]);
  return j <= n && (j < n || j > 0);
}

// The CTAs are persistent: CTA c takes units in rounds of gridDim.x, in a snake order
// (c in even rounds, gridDim.x - 1 - c in odd ones), so with the units sorted heaviest
// first the CTAs' total work stays balanced without any shared counter.
__device__ __forceinline__ int unit_index(int round) {
  const int base = round * static_cast<int>(gridDim.x);
  return (round & 1) ? base + static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                     : base + static_cast<int>(blockIdx.x);
}

template <int D, bool kSplit>
__global__ void __launch_bounds__(352, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using Cfg = PrefillCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                           // [2][tile]
  uint8_t* sKV = smem + 2 * Cfg::kTileBytes;                    // [slots][tile]

  __shared__ uint64_t q_full;
  // kv_ready[j % kIterRing]: the data of key block j is in shared memory: K(j) (j < n_iter) and
  // V(j-1) (j > 0) both complete on it, so the MMA thread waits once per block.
  __shared__ uint64_t kv_ready[kIterRing];
  // s_full1: S_1(j) done (one phase per S_1 block; tile 1 may be inactive in a unit).
  // iter_done[j % kIterRing]: the last MMA of key block j done (S_0(j) when j < nkv_0), which
  // also releases K(j) and V(j-1): the tensor pipe completes one thread's MMAs in issue
  // order, so a commit covers everything issued before it.
  __shared__ uint64_t s_full1, iter_done[kIterRing], o_done[2];
  __shared__ uint64_t mma_drain;
  __shared__ uint32_t tmem_base_holder;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 1);
    for (int r = 0; r < kIterRing; ++r) mbar_init(&kv_ready[r], 1);
    for (int r = 0; r < kIterRing; ++r) mbar_init(&iter_done[r], 1);
    mbar_init(&s_full1, 1);
    for (int q = 0; q < 2; ++q) {
      mbar_init(&o_done[q], 1);
    }
    mbar_init(&mma_drain, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpIssuer) {
    tmem_alloc(&tmem_base_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_holder;
  volatile int* abort_p = &abort_flag;

  // Every role walks the same work items (whole units, or pieces of the split units) in the
  // same order and keeps the barrier phases running across them: G = index of the item's key
  // block 0 in this CTA's sequence of key blocks (an item with n = max(nkv) has blocks 0..n,
  // so G grows by n + 1 per item).
  if (warp == kWarpProducer) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      // Q is read once per unit: evict it first, so that L2 keeps the K/V blocks the other
      // CTAs of the head group still read.
      const uint64_t q_policy = l2_policy_evict_first();
      int G = 0, U = 0;
      int slot = 0;        // slot of the next item
      int filled = 0;      // items loaded so far (saturates at kSlots)
      int rel[Cfg::kSlots];  // block whose last MMA releases the item now in each slot
      // Blocks complete in order (one thread issues all MMAs and commits), so a block at or
      // below the last one seen complete needs no wait. Skipping those waits also keeps every
      // wait less than kIterRing phases behind the ring: without it, a slot last used many
      // one-block units ago would be waited on after its barrier had wrapped twice.
      int done_upto = -1;
      auto wait_block = [&](int r) -> bool {
        if (r <= done_upto) return true;
        if (!mbar_wait(&iter_done[r % kIterRing], static_cast<uint32_t>(r / kIterRing) & 1u, abort_p,
                       kPrefillWaitTimeoutNs))
          return false;
        done_upto = r;
        return true;
      };
      bool alive = true;
      for (int round = 0; alive && round * static_cast<int>(gridDim.x) < p.items; ++round) {
        const int idx = unit_index(round);
        if (idx >= p.items) continue;
        const UnitInfo u = decode_item<kSplit>(p, idx);
        const int n_iter = max(u.nkv[0], u.nkv[1]);
        // this unit's Q overwrites the previous one's: wait for its last S MMAs (block G - 2)
        if (U > 0 && !wait_block(G - 2)) break;
        const int nq = (u.nkv[0] > 0) + (u.nkv[1] > 0);
        mbar_arrive_expect_tx(&q_full, nq * Cfg::kTileBytes);
        for (int q = 0; q < 2; ++q) {
          if (u.nkv[q] == 0) continue;
          for (int kb = 0; kb < Cfg::kNumBox; ++kb)
            tma_load_3d_hint(sQ + q * Cfg::kTileBytes + kb * Cfg::kBoxBytes, &tmQ, &q_full, kb * 64, u.row0[q],
                             u.b * p.Hq + u.head[q], q_policy);
        }
        const int zkv = u.b * p.Hkv + u.kvh;
        const int n_items = 2 * n_iter;  // item 2j = K(j), item 2j + 1 = V(j)
        for (int i = 0; i < n_items; ++i) {
          if (filled == Cfg::kSlots) {
            if (!wait_block(rel[slot])) {  // the slot's previous item is free once its block is done
              alive = false;
              break;
            }
          } else {
            ++filled;
          }
          // item i belongs to key block it = (i + 1) / 2: K(j) is read in block j, V(j) in block j + 1
          const int it = (i + 1) >> 1;
          rel[slot] = G + it;
          uint64_t* rb = &kv_ready[(G + it) % kIterRing];
          if (i == 0 || (i & 1)) {  // first item of block `it`: arm the barrier with the bytes of both tiles
            const int ntiles = (it >= 1 ? 1 : 0) + (it < n_iter ? 1 : 0);
            mbar_arrive_expect_tx(rb, ntiles * Cfg::kTileBytes);
          }
          const CUtensorMap* map = (i & 1) ? &tmV : &tmK;
          for (int kb = 0; kb < Cfg::kNumBox; ++kb)
            tma_load_3d(sKV + slot * Cfg::kTileBytes + kb * Cfg::kBoxBytes, map, rb, kb * 64,
                        (u.kb0 + (i >> 1)) * 128, zkv);
          if (++slot == Cfg::kSlots) slot = 0;
        }
        G += n_iter + 1;
        ++U;
      }
      if (*abort_p) {
        // Give the copies still in flight time to land before the CTA exits (a few microseconds
        // suffice; wait 1 ms of wall time).
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpIssuer || warp == kWarpHelper) {
    // Handoffs to the issuer go through hardware named barriers (bar.sync cannot time
    // out, so every arrival sequence below runs to the end even after an abort, and each
    // one matches the issuer's syncs one for one):
    //  * data of key block j (when any tile has work in it): the helper arrives on kBarData,
    //    the issuer syncs and acknowledges on kBarDataAck, the helper syncs on the ack;
    //  * P_q(j) written: the 128 softmax threads of tile q arrive on kBarP0 + q and the
    //    issuer syncs before PV_q(j). An arrival for P_q(j + 1) needs S_q(j + 1), which
    //    the issuer only issues after its sync for P_q(j), so arrivals never run ahead.
    if (warp == kWarpHelper) {
      // ------------------------------ wait helper ------------------------------
      // Waits until the unit's Q and block j's K/V data are in shared memory, then hands
      // them to the issuer (kBarData) and waits for the issuer's acknowledgement
      // (kBarDataAck) before looking at block j + 1, so the two warps stay in lockstep. All 32
      // lanes wait, so the warp reaches its named barriers converged (measured: 0.6 % faster at
      // d = 64 than a lane-0 wait followed by __syncwarp).
      int G = 0, U = 0;
      for (int round = 0; round * static_cast<int>(gridDim.x) < p.items; ++round) {
        const int idx = unit_index(round);
        if (idx >= p.items) continue;
        const UnitInfo u = decode_item<kSplit>(p, idx);
        const int n_iter = max(u.nkv[0], u.nkv[1]);
        mbar_wait(&q_full, static_cast<uint32_t>(U) & 1u, abort_p, kPrefillWaitTimeoutNs);
        for (int j = 0; j <= n_iter; ++j) {
          if (!block_has_work(u, j)) continue;
          if (!*abort_p)
            mbar_wait(&kv_ready[(G + j) % kIterRing], static_cast<uint32_t>((G + j) / kIterRing) & 1u, abort_p,
                      kPrefillWaitTimeoutNs);
          __syncwarp();
          named_bar_arrive(kBarData, kPair);
          named_bar_sync(kBarDataAck, kPair);
        }
        G += n_iter + 1;
        ++U;
      }
    } else {
      // ------------------------------ MMA issuer ------------------------------
      // Issue order per key block j: PV_1(j-1), S_1(j), PV_0(j-1), S_0(j). The tensor pipe
      // runs one thread's MMAs in issue order, so S_q(j) may overwrite the TMEM columns
      // that PV_q(j-1) reads P_q(j-1) from, and softmax q gets S_q(j) two GEMMs after it
      // handed over P_q(j-1) while the other tile's GEMMs keep the tensor core busy. The
      // next unit's PV_q(0) overwrites O_q only after the P_q(0) handoff, which the softmax
      // warps of tile q give after they have read O_q for the previous unit.
      // Tile 0 (active in every unit, nkv_0 >= max(nkv) - 1) learns of S_0(j) from the
      // per-block ring, whose parity waits stay sound because its waits never skip more
      // than a few blocks; tile 1, which may be inactive for a whole unit, has a barrier
      // of its own with one phase per S_1 block.
      // Descriptors advance by adding (byte offset >> 4) to the start-address field: every
      // operand lies in this CTA's shared memory window (< 256 KB), so no field overflows.
      constexpr uint32_t kTile16 = Cfg::kTileBytes >> 4, kRing16 = Cfg::kSlots * kTile16;
      const uint64_t dQ = make_sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK = make_sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t dV = make_sdesc_sw128(smem_u32(sKV), Cfg::kBoxBytes, 1024);
      uint32_t k16 = 0;                  // slot of K(j), in 16-byte units
      uint32_t v16 = kRing16 - kTile16;  // slot of V(j-1), used only when j > 0
      // The whole warp walks the loop in step; only lane 0's MMAs and commits are issued
      // (a guard predicate in the instruction), so the warp never diverges and every named
      // barrier is met by a converged warp.
      const uint32_t lead = lane == 0 ? 1u : 0u;
      bool any_mma = false;
      int G = 0;
      for (int round = 0; round * static_cast<int>(gridDim.x) < p.items; ++round) {
        const int idx = unit_index(round);
        if (idx >= p.items) continue;
        const UnitInfo u = decode_item<kSplit>(p, idx);
        const int n_iter = max(u.nkv[0], u.nkv[1]);
        const int nkv0 = u.nkv[0], nkv1 = u.nkv[1];
        for (int j = 0; j <= n_iter; ++j) {
          if (block_has_work(u, j)) {
            named_bar_sync(kBarData, kPair);
            named_bar_arrive(kBarDataAck, kPair);
          }
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {
            const int q = 1 - qq;
            const int nkv_q = q ? nkv1 : nkv0;
            const bool do_s = j < nkv_q, do_pv = j > 0 && j - 1 < nkv_q;
            if (!do_s && !do_pv) continue;
            if (do_pv) named_bar_sync(kBarP0 + q, kSoftmaxAndIssuer);
            // No abort check here (a shared-memory load would stall the issue stream): after an
            // abort the MMAs still only touch this CTA's buffers, and every waiter gives up.
            tc_fence_after();
            const uint32_t d_s = tmem + (q ? Cfg::kTmS1 : Cfg::kTmS0);
            if (do_pv) {
              const uint32_t d_o = tmem + (q ? Cfg::kTmO1 : Cfg::kTmO0);
#pragma unroll
              for (int kk = 0; kk < 128 / 16; ++kk)  // 16 keys = 2048 bytes of V per step
                umma_ts_if(lead, d_o, d_s + kk * 8, dV + v16 + kk * 128, Cfg::kIdescPV, (j > 1 || kk > 0) ? 1u : 0u);
              if (j == nkv_q) umma_commit_if(lead, &o_done[q]);  // last block of this tile: O is final
            }
            if (do_s) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off16 = ((kk >> 2) * Cfg::kBoxBytes + (kk & 3) * 32) >> 4;
                umma_ss_if(lead, d_s, dQ + q * kTile16 + off16, dK + k16 + off16, Cfg::kIdescQK, kk > 0 ? 1u : 0u);
              }
              if (q == 1) umma_commit_if(lead, &s_full1);
            }
            any_mma = true;
          }
          umma_commit_if(lead, &iter_done[(G + j) % kIterRing]);
          if (j < n_iter) {  // the unit's 2 n_iter items: K(j) and V(j) for j < n_iter
            v16 = k16 + kTile16;  // V(j) sits in the slot after K(j)
            if (v16 >= kRing16) v16 -= kRing16;
            k16 += 2 * kTile16;
            if (k16 >= kRing16) k16 -= kRing16;
          }
        }
        G += n_iter + 1;
      }
      if (lane == 0 && any_mma) {  // every MMA has finished before TMEM is released
        umma_commit(&mma_drain);
        mbar_wait(&mma_drain, 0, abort_p, kPrefillWaitTimeoutNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------ softmax warps ------------------------------
    const int q = (warp - kFirstSoftmaxWarp) >> 2;
    const int wq = warp & 3;
    const int row_in_tile = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + (q ? Cfg::kTmS1 : Cfg::kTmS0);
    const uint32_t t_o = tmem + lane_off + (q ? Cfg::kTmO1 : Cfg::kTmO0);
    const float c = p.c;
    bool ok = true;
    int G = 0;
    int s1_count = 0;  // S_1 blocks committed in earlier units (phases of s_full1)
    int o_count = 0;   // earlier units in which this tile was active (phases of o_done[q])
    for (int round = 0; round * static_cast<int>(gridDim.x) < p.items; ++round) {
    const int idx = unit_index(round);
    if (idx >= p.items) continue;
    const UnitInfo u = decode_item<kSplit>(p, idx);
    const int n_iter = max(u.nkv[0], u.nkv[1]);
    const int nkv = q ? u.nkv[1] : u.nkv[0];
    const int row0 = q ? u.row0[1] : u.row0[0];
    const int head = q ? u.head[1] : u.head[0];
    const int row = row0 + row_in_tile;
    float m_run = -INFINITY;
    float l_run = 0.f;

    // j runs over the absolute key blocks jb .. jb + nkv - 1 of the item; the barrier rings
    // count the item's blocks from G (and s1_count), so they are indexed with j - jb.
    const int jb = kSplit ? u.kb0 : 0;
    const int g_j = G - jb, s1_j = s1_count - jb;
    for (int j = jb; j < jb + nkv; ++j) {
      // S_q(j) ready: tile 1 on s_full1, tile 0 on the per-block barrier that follows S_0(j).
      // After a failed wait the warp skips the work but still arrives on the named barrier
      // below, once per block, so the issuer's syncs always complete.
      if (ok) {
        const bool w = (q == 1) ? mbar_wait(&s_full1, static_cast<uint32_t>(s1_j + j) & 1u, abort_p,
                                            kPrefillWaitTimeoutNs)
                                : mbar_wait(&iter_done[(g_j + j) % kIterRing],
                                            static_cast<uint32_t>((g_j + j) / kIterRing) & 1u, abort_p,
                                            kPrefillWaitTimeoutNs);
        ok = __all_sync(0xFFFFFFFFu, w);
      }
      if (ok) {
      tc_fence_after();
      uint32_t sr[128];
      const int j0 = j * 128;
      // blocks past the diagonal or the end of the keys need the element mask before the
      // maximum; every other block takes the row maximum from the reducing TMEM load
      // (split launches are never causal: kSplit drops the causal terms at compile time)
      const bool causal = !kSplit && p.causal;
      const bool need_mask = (j0 + 128 > p.Tk) || (causal && j0 + 127 > row0);
      float m_raw;
      if (!need_mask) {
        m_raw = tmem_ld128_max(t_s, sr);
      } else {
        tmem_ld128(t_s, sr);
        const int lim = causal ? min(p.Tk - 1, row) : (p.Tk - 1);  // last visible key of this row
#pragma unroll
        for (int k = 0; k < 128; ++k)
          if (j0 + k > lim) sr[k] = __float_as_uint(-INFINITY);
        // row max over columns 0..127: 8 independent chains of 3-input max, merged at the end
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmaxf(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
#pragma unroll
        for (int k = 16; k < 128; k += 16) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            mx[i] = fmax3(mx[i], __uint_as_float(sr[k + 2 * i]), __uint_as_float(sr[k + 2 * i + 1]));
        }
        m_raw = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      }
      const float m_blk = m_raw * c;
      const float m_cand = fmaxf(m_run, m_blk);
      const bool grow = m_cand > m_run + kRescaleThreshold;
      float corr = 1.f;
      if (grow) {
        corr = ex2_approx(m_run - m_cand);  // 0 when m_run = -inf
        m_run = m_cand;
      }
      const float base = (m_run == -INFINITY) ? 0.f : m_run;

      // p = 2^(s*c - base): packed fp32x2 FMA, one ex2 per element, packed row sums
      const float2 c2 = make_float2(c, c);
      const float2 nb2 = make_float2(-base, -base);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sr[cc * 32 + 2 * k]), __uint_as_float(sr[cc * 32 + 2 * k + 1])), c2, nb2);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          acc[k & 3] = __fadd2_rn(acc[k & 3], pp);
          pk[k] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st16(t_s + cc * 16, pk);
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]);
      const float2 a23 = __fadd2_rn(acc[2], acc[3]);
      l_run = l_run * corr + ((a01.x + a01.y) + (a23.x + a23.y));
      if (j > jb && __any_sync(0xFFFFFFFFu, grow)) {
        // O holds the sum up to block j-1 relative to the old base; PV_q(j-1) was issued before
        // S_q(j), so it has completed by now. Rescale in TMEM (after P is written, so the
        // registers of S are free).
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          tmem_ld32(t_o + cc * 32, ov);
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * corr);
          tmem_st32(t_o + cc * 32, ov);
        }
      }
      }  // ok

      tmem_st_wait();
      tc_fence_before();
      named_bar_arrive(kBarP0 + q, kSoftmaxAndIssuer);  // P_q(j) (and any O rescale) is in TMEM
    }

    if (ok && nkv > 0) {
      // warp-uniform: the next unit's waits run under __all_sync
      ok = __all_sync(0xFFFFFFFFu,
                      mbar_wait(&o_done[q], static_cast<uint32_t>(o_count) & 1u, abort_p, kPrefillWaitTimeoutNs));
      tc_fence_after();
      if (kSplit && ok && unit_index(round) >= p.full_units) {
        // A piece of a split unit: O / l of the piece in fp32 and m + log2 l, for the merge.
        // (The item index is recomputed from the round rather than kept live across the loop.)
        const float inv_l = 1.f / l_run;
        const size_t prow = (static_cast<size_t>(unit_index(round) - p.full_units) * 2 + q) * 128 + row_in_tile;
        float4* dst = reinterpret_cast<float4*>(p.part_o + prow * D);
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          tmem_ld32(t_o + cc * 32, ov);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[cc * 8 + v] = make_float4(__uint_as_float(ov[4 * v]) * inv_l, __uint_as_float(ov[4 * v + 1]) * inv_l,
                                          __uint_as_float(ov[4 * v + 2]) * inv_l,
                                          __uint_as_float(ov[4 * v + 3]) * inv_l);
        }
        p.part_lse2[prow] = m_run + log2f(l_run);
      } else if (ok) {
        const uint64_t o_policy = l2_policy_evict_first();  // O is written once and not read here
        const float inv_l = 1.f / l_run;
        const bool store = row < p.Tq;
        const size_t orow = (static_cast<size_t>(u.b) * p.Hq + head) * p.Tq + row;
        // Each thread owns one row, so a plain store of a warp covers 32 rows. When O is 32-byte
        // aligned, lanes 2i and 2i + 1 (rows 2i, 2i + 1) swap one 32-byte half of each 64-byte
        // chunk (one shuffle per word) and each 32-byte store then writes 64 contiguous bytes of
        // one row from the pair. The O stores sit on the softmax warps' path from a unit's last
        // block to the next unit's first P; measured on causal GQA B2 Hq32 T8192: 16-byte stores
        // 1625-1650 TFLOP/s, 32-byte stores 1671-1692, with the swap 1692-1697 (B1 Hq16 T4096:
        // 1185 -> 1228).
        const bool odd = (lane & 1) != 0;
        const int row_e = row0 + (row_in_tile & ~1);  // the pair's even row
        const bool st_e = row_e < p.Tq, st_o = row_e + 1 < p.Tq;
        const size_t orow_e = (static_cast<size_t>(u.b) * p.Hq + head) * p.Tq + row_e;
        // the epilogue's loops (and the O rescale's) stay rolled: they run once per unit (or
        // rarely), and unrolled they made the kernel's code larger and the softmax role spill
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          tmem_ld32(t_o + cc * 32, ov);
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pk[k] = pack_bf16x2(__uint_as_float(ov[2 * k]) * inv_l, __uint_as_float(ov[2 * k + 1]) * inv_l);
          if (p.o_v8) {
            // after the swap pk[0..7] is this lane's 32 bytes of the even row, pk[8..15] its 32
            // bytes of the odd row (the even lane holds both rows' first halves, the odd lane
            // both second halves)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t r = __shfl_xor_sync(0xFFFFFFFFu, odd ? pk[k] : pk[8 + k], 1);
              if (odd) pk[k] = r; else pk[8 + k] = r;
            }
            uint32_t* base = reinterpret_cast<uint32_t*>(p.o + orow_e * D + cc * 32) + (odd ? 8 : 0);
            if (st_e) st_global_v8_hint(base, pk, o_policy);
            if (st_o) st_global_v8_hint(base + D / 2, pk + 8, o_policy);
          } else if (store) {
            uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D + cc * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              st_global_v4_hint(dst + v, make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]),
                                o_policy);
          }
        }
        if (store && p.lse != nullptr) p.lse[orow] = (m_run + log2f(l_run)) * 0.69314718055994530942f;
      }
    }
    s1_count += u.nkv[1];
    o_count += (nkv > 0) ? 1 : 0;
    G += n_iter + 1;
    }  // units
    tc_fence_before();
  }

  __syncthreads();
  if (warp == kWarpIssuer) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of the pieces of the split units. The pieces of a unit cover disjoint key ranges, so
// the row's result is their weighted mean with weights l_p 2^(m_p - M) ("Module 07", section
// "Online softmax: derivation": partial sums over key blocks combine after rescaling to a
// common base; the same merge as flash-decoding's): O = sum_p w_p O_p / sum_p w_p with
// w_p = 2^(lse2_p - M), M = max_p lse2_p, and the row's log-sum-exp (M + log2 sum_p w_p) ln 2.
// One warp per query row of a split unit: lane p reads piece p's log-sum-exp (32 pieces at a
// time), the maximum and the weights' sum are reduced across the warp (a fixed tree), and the
// weighted sum of the pieces' rows runs in piece order with lane e holding D/32 consecutive
// columns. Up to kMergeBatch pieces, every load of the row is issued before the first is used
// (the kernel is bound by load latency, not bandwidth). Launched as a programmatic dependent
// of the prefill kernel.
constexpr int kMergeBatch = 16;  // pieces whose rows one warp loads at once

template <int D>
__global__ void __launch_bounds__(256) attn_fwd_merge_kernel(const PrefillParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the pieces' results are complete
  constexpr int E = D / 32;
  const int wg = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int t = wg >> 8;  // split unit, 256 rows (2 tiles x 128) each
  const int q = (wg >> 7) & 1;
  const int i = wg & 127;
  if (t >= p.units - p.full_units) return;
  const UnitInfo u = decode_unit(p, p.full_units + t);
  const int row = (q ? u.row0[1] : u.row0[0]) + i;  // selects, not a runtime index into u
  const int head = q ? u.head[1] : u.head[0];
  if ((q ? u.nkv[1] : u.nkv[0]) == 0 || row >= p.Tq) return;
  // piece pc of unit t is part t * split + pc: its row i of tile q is at ((part * 2 + q) * 128 + i)
  const size_t row_p0 = (static_cast<size_t>(t) * p.split * 2 + q) * 128 + i;
  const float* lse2 = p.part_lse2 + row_p0;
  const float* src = p.part_o + row_p0 * D + lane * E;
  using VecE = typename std::conditional<E == 2, float2, float4>::type;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float mx = -INFINITY, wsum = 0.f;
  auto fma_row = [&](float w, const VecE& x) {
    acc[0] = fmaf(w, x.x, acc[0]);
    acc[1] = fmaf(w, x.y, acc[1]);
    if constexpr (E == 4) {
      acc[2] = fmaf(w, reinterpret_cast<const float4&>(x).z, acc[2]);
      acc[3] = fmaf(w, reinterpret_cast<const float4&>(x).w, acc[3]);
    }
  };
  if (p.split <= kMergeBatch) {
    // every load issued before any is used: one memory latency for the whole row
    const float l_lane = lane < p.split ? lse2[static_cast<size_t>(lane) * 256] : -INFINITY;
    VecE x[kMergeBatch];
#pragma unroll
    for (int pc = 0; pc < kMergeBatch; ++pc)
      if (pc < p.split) x[pc] = *reinterpret_cast<const VecE*>(src + static_cast<size_t>(pc) * 256 * D);
    mx = l_lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    const float w_lane = lane < p.split ? ex2_approx(l_lane - mx) : 0.f;
    wsum = w_lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xFFFFFFFFu, wsum, o);
#pragma unroll
    for (int pc = 0; pc < kMergeBatch; ++pc)
      if (pc < p.split) fma_row(__shfl_sync(0xFFFFFFFFu, w_lane, pc), x[pc]);
  } else {
    for (int c = 0; c < p.split; c += 32)
      if (c + lane < p.split) mx = fmaxf(mx, lse2[static_cast<size_t>(c + lane) * 256]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    for (int c = 0; c < p.split; c += 32) {
      const int n = min(32, p.split - c);
      const float w_lane = lane < n ? ex2_approx(lse2[static_cast<size_t>(c + lane) * 256] - mx) : 0.f;
      float ws = w_lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xFFFFFFFFu, ws, o);
      wsum += ws;
#pragma unroll 4
      for (int pc = 0; pc < n; ++pc)
        fma_row(__shfl_sync(0xFFFFFFFFu, w_lane, pc),
                *reinterpret_cast<const VecE*>(src + static_cast<size_t>(c + pc) * 256 * D));
    }
  }
  const float inv = 1.f / wsum;
  const size_t orow = (static_cast<size_t>(u.b) * p.Hq + head) * p.Tq + row;
  __nv_bfloat16* dst = p.o + orow * D + lane * E;
  if constexpr (E == 2) {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  } else {
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
  }
  if (lane == 0 && p.lse != nullptr) p.lse[orow] = (mx + log2f(wsum)) * 0.69314718055994530942f;
}

// --------------------------------------------------------------------------------------
// Host side: tensor maps and launch
// --------------------------------------------------------------------------------------
// Streaming multiprocessors of the current device (queried once per device).
static int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) {
    int n = 0;
    return cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess ? n : 0;
  }
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// Persistent CTAs for the forward kernel: one per SM (the shared memory allows one), or fewer
// when the environment variable GB300_ATTN_PREFILL_CTAS gives a smaller positive count (a
// scheduling knob; the tests use it to reach the split tail on small problems).
static int prefill_ctas() {
  const int sms = sm_count();
  const char* e = std::getenv("GB300_ATTN_PREFILL_CTAS");
  if (e != nullptr) {
    const int cap = std::atoi(e);
    if (cap > 0 && cap < sms) return cap;
  }
  return sms;
}

// Scratch for the split tail with `ctas` persistent CTAs: at most ctas pieces of 2 x 128 rows,
// each row d fp32 values of O and one base-2 log-sum-exp.
static size_t split_scratch_bytes(int ctas, int d) {
  return static_cast<size_t>(ctas) * 256 * (static_cast<size_t>(d) + 1) * sizeof(float);
}

size_t prefill_workspace_bytes(int d) { return split_scratch_bytes(sm_count(), d); }

// The forward kernel on `grid` persistent CTAs, then, when units are split, the merge kernel.
template <int D>
static cudaError_t launch_fwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                const PrefillParams& p, int grid, cudaStream_t stream, int* launched) {
  using Cfg = PrefillCfg<D>;
  const bool split = p.full_units != p.units;
  auto kern = split ? attn_fwd_kernel<D, true> : attn_fwd_kernel<D, false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(mq, mk, mv, p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  *launched = 1;
  if (!split) return cudaSuccess;
  // The merge is a programmatic dependent: its grid is set up while the forward grid drains,
  // and griddepcontrol.wait orders its reads after the forward kernel's writes.
  const long long rows = static_cast<long long>(p.units - p.full_units) * 256;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, attn_fwd_merge_kernel<D>, p);
  if (err == cudaSuccess) err = cudaGetLastError();
  if (err == cudaSuccess) *launched = 2;
  return err;
}

cudaError_t launch_attn_fwd_pair(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                 int Hkv, int Tq, int Tk, int d, int causal, float scale, cudaStream_t stream);

// Which forward kernel runs: this file's kernel, unless the environment variable
// GB300_ATTN_PREFILL is "pair" (the CTA-pair kernel of prefill_pair.cu; both compute the same
// result; the pair kernel is the slower of the two on this part, see prefill_pair.cu).
static bool use_pair_kernel() {
  const char* e = std::getenv("GB300_ATTN_PREFILL");
  return e != nullptr && std::strcmp(e, "pair") == 0;
}

// Returns cudaErrorInvalidValue if a tensor map cannot be built (e.g. driver entry point missing).
//
// Schedule: the units run on min(units, CTAs) persistent CTAs in rounds. When a non-causal
// call's units leave the last round partly filled (r of `grid` CTAs busy) and a workspace is
// given, each of those r units is split along its key blocks into s = min(grid / r, blocks)
// pieces that run side by side, and the merge kernel combines them: the last round then takes
// about 1/s of a unit instead of a whole one (non-causal MHA B8 H12 T4096 d64: 1536 units on
// 152 CTAs, 16 in the last round, split 9 ways). Causal units are ordered heaviest first and
// the snake order already balances them, so they are never split.
static cudaError_t launch_attn_fwd_single(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                          int Hq, int Hkv, int Tq, int Tk, int d, int causal, float scale,
                                          void* workspace, size_t workspace_bytes, cudaStream_t stream,
                                          int* launched) {
  CUtensorMap mq, mk, mv;
  if (!encode_bf16_tile_map(&mq, q, d, Tq, B * Hq) || !encode_bf16_tile_map(&mk, k, d, Tk, B * Hkv) ||
      !encode_bf16_tile_map(&mv, v, d, Tk, B * Hkv))
    return cudaErrorInvalidValue;
  PrefillParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  // rows are d * 2 bytes apart (a multiple of 32): every row is 32-byte aligned iff O is
  p.o_v8 = (reinterpret_cast<uintptr_t>(o) % 32 == 0) ? 1 : 0;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Tq = Tq;
  p.Tk = Tk;
  p.g = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.pair_heads = (p.g % 2 == 0) ? 1 : 0;
  p.n_qt = (Tq + 127) / 128;
  p.c = scale * 1.4426950408889634f;
  const long long units =
      p.pair_heads ? static_cast<long long>(p.n_qt) * (Hq / 2) * B : static_cast<long long>((p.n_qt + 1) / 2) * Hq * B;
  // (the kernel forms round * gridDim.x + gridDim.x in int)
  if (units <= 0 || units > 0x3FFFFFFFLL) return cudaErrorInvalidValue;
  p.units = static_cast<int>(units);
  // unit order (decode_unit): causal rank-major, non-causal (batch, head)-major
  const int ranks = p.pair_heads ? p.n_qt : (p.n_qt + 1) / 2;
  const int rests = p.units / ranks;
  if (p.causal) {
    p.rank_div = rests;
    p.rank_mod = ranks;
    p.rest_div = 1;
    p.rest_mod = rests;
  } else {
    p.rank_div = 1;
    p.rank_mod = ranks;
    p.rest_div = ranks;
    p.rest_mod = rests;
  }
  const int ctas = prefill_ctas();
  if (ctas <= 0) return cudaErrorInvalidDevice;
  const int grid = p.units < ctas ? p.units : ctas;
  p.full_units = p.units;
  p.split = 1;
  p.part_o = nullptr;
  p.part_lse2 = nullptr;
  if (!p.causal && workspace != nullptr && grid < p.units) {
    const int r = p.units % grid;
    const int blocks = (Tk + 127) / 128;
    const int s = r > 0 ? std::min(grid / r, blocks) : 1;
    if (s >= 2 && workspace_bytes >= split_scratch_bytes(grid, d)) {
      p.full_units = p.units - r;
      p.split = s;
      p.part_o = static_cast<float*>(workspace);
      p.part_lse2 = p.part_o + static_cast<size_t>(grid) * 256 * d;
    }
  }
  p.items = p.full_units + (p.units - p.full_units) * p.split;  // <= units + grid
  return d == 64 ? launch_fwd_d<64>(mq, mk, mv, p, grid, stream, launched)
                 : launch_fwd_d<128>(mq, mk, mv, p, grid, stream, launched);
}

cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                            int Hkv, int Tq, int Tk, int d, int causal, float scale, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream, int* launched) {
  *launched = 0;
  if (use_pair_kernel()) {
    const cudaError_t err = launch_attn_fwd_pair(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale, stream);
    if (err == cudaSuccess) *launched = 1;
    if (err != cudaErrorInvalidDevice) return err;
    (void)cudaGetLastError();  // no resident pair on this device: the single-CTA kernel runs
  }
  return launch_attn_fwd_single(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale, workspace, workspace_bytes,
                                stream, launched);
}

uint32_t prefill_take_device_error() { return take_device_error_word(); }

}  // namespace gb300
