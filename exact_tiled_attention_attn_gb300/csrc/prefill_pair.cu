// prefill_pair.cu - exact tiled attention forward pass on CTA pairs (two SMs, cta_group::2).
//
// What it computes is the same as prefill.cu ("FlashAttention: attention without the n x n
// matrix", section "Forward pass of FlashAttention"; "Module 07: Fused operators and
// FlashAttention", sections "Online softmax: derivation" and "FlashAttention-2"): per query
// row a running maximum m, a running sum l and an unnormalised output O over blocks of 128
// keys, O and l rescaled by 2^(m_old - m_new) when the maximum moves, one division at the end.
//
// Why pairs. A 128x128x16 score MMA on one SM reads 8 KB of operands from shared memory in
// its 64 clocks, the port's whole rate, and the TMA writes of the K/V stream (64 KB per key
// block at d = 128) compete with it: measured on this part, the copies then get ~25 B/clock
// against the 32 the single-CTA kernel needs at full MMA rate, and ~12 against 31 at d = 64.
// Here the two SMs of a cluster issue M = 256 MMAs as one: each SM holds 128 of the rows (its
// own query tiles) and half of the B operand, so each SM reads and loads half of every K and
// V tile. The four query tiles of a pair share one K/V stream, which is fetched once:
// "Attention from the kernel's side", section "Prefill and decoding are different problems"
// (g query heads share one K/V load).
//
// Measured outcome (causal GQA B2 Hq32 Hkv8 T8192 d128): the pair kernel is correct (the same
// parity suite as prefill.cu) but slower, ~1200 TFLOP/s against ~1575 for the single-CTA
// kernel, which therefore stays the default (GB300_ATTN_PREFILL=pair selects this one). With
// the slot ping-pong both kernels use, a key block lasts about M + C, M being one slot's MMA
// group and C the time from S_q(j) landing to the issuer's go for P.V(j). The pair shortens M
// (its MMAs no longer starve the copies of the shared-memory port) but CTA 1's P must reach
// CTA 0's issuer through a remote mbarrier arrival and the helper warp; globaltimer traces of
// one pair show that hand-off at ~0.45 us (a named barrier in CTA 1, the remote arrival, the
// helper's wake-up, the named barrier to the issuer), more than M saves.
//
// Work unit = 4 query tiles, tile (r, q) in CTA r's slot q; the pair's MMA for slot q covers
// CTA 0's and CTA 1's tile q (M = 256). Which tiles form a unit depends on the group size g:
//   g % 4 == 0: heads 4p + 2r + q of one K/V group at the same 128 rows (no wasted keys);
//   g % 2 == 0: heads 2p + q at row tiles 2t + r;
//   g odd:      one head at row tiles 4s + 2r + q.
// In the last two, when causal, a slot walks the key blocks of its longer tile; the other
// tile's extra blocks lie above its diagonal and are masked to -inf (p = 0).
//
// Roles (352 threads per CTA, both CTAs):
//   warp 8      TMA producer: this CTA's Q tiles, then its halves of the K/V blocks (K: 64 of
//               the 128 keys, all d columns; V: all 128 keys, d/2 columns) into a ring of
//               slots. Every copy completes on the barrier of CTA 0 (the issuing CTA), which
//               counts both CTAs' arrivals and bytes.
//   warp 9      CTA 0: the MMA issuer (one thread), S = Q K^T and O += P V for the pair;
//               both CTAs: allocates and frees the pair's TMEM.
//   warp 10     CTA 0: waits for Q and K/V data and for CTA 1's P, and hands each "go" to
//               the issuer through hardware named barriers (the issuer itself never waits on
//               an mbarrier: under load such a wait costs it hundreds of clocks).
//   warps 0-7   softmax of slot 0 / slot 1 of this CTA, one thread per row, as in prefill.cu;
//               CTA 1 reports its P through a named barrier of its 4 warps and one arrival
//               on CTA 0's p_peer barrier.
// Completion of the pair's MMAs is signalled into both CTAs at once (tcgen05.commit with a
// CTA mask), so each CTA's softmax and producer wait on barriers in their own shared memory.
// TMEM (512 columns, the same columns in both CTAs): S0 [0,128) S1 [128,256)
// O0 [256,256+d) O1 [256+d,256+2d); P_q aliases the first 64 columns of S_q.
#include "pair.cuh"

namespace gb300 {

constexpr uint64_t kPairTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr float kPairRescaleThreshold = 8.0f;        // log2 of the allowed growth of p
// hardware named barriers (0 is __syncthreads)
constexpr uint32_t kPBarData = 1, kPBarDataAck = 2, kPBarP0 = 3;  // kPBarP0 + 1 for slot 1
constexpr uint32_t kPHandoff = 64;   // CTA 0: helper warp + issuer warp
constexpr uint32_t kPLeaderP = 192;  // CTA 0: 4 softmax warps + issuer warp + helper warp
constexpr uint32_t kPPeerP = 128;    // CTA 1: the 4 softmax warps of a slot

template <int D>
struct PairPrefillCfg {
  static constexpr int kQTileBytes = 128 * D * 2;  // 128 rows x D
  static constexpr int kQBoxBytes = 128 * 128;     // 128 rows x 64 columns, 128-byte swizzle
  static constexpr int kKBoxBytes = 64 * 128;      // 64 rows x 64 columns, 128-byte swizzle
  // One ring slot holds either half of a K tile (64 keys x D) or half of a V tile (128 keys x
  // D/2 columns): 16 KB at d = 128, 8 KB at d = 64. Item 2j = K(j), item 2j + 1 = V(j); an odd
  // slot count lets V(j) reuse the slot of K(j - 2) as soon as S(j - 2) is done.
  static constexpr int kHalfBytes = 64 * D * 2;
  static constexpr int kSlots = (D == 64) ? 21 : 9;
  static constexpr int kIterRing = (D == 64) ? 16 : 8;  // per-key-block barriers in flight
  static constexpr int kSmemBytes = 2 * kQTileBytes + kSlots * kHalfBytes + 1024;
  static constexpr int kTmS0 = 0, kTmS1 = 128, kTmO0 = 256, kTmO1 = 256 + D;
  static constexpr int kThreads = 352;
  static constexpr uint32_t kIdescQK = make_idesc_bf16_f32(256, 128, false);
  static constexpr uint32_t kIdescPV = make_idesc_bf16_f32(256, D, true);
  // V half per 16 keys, in 16-byte units: 16 rows of D/2 columns (128-byte rows at d = 128
  // with the 128-byte swizzle, 64-byte rows at d = 64 with the 64-byte swizzle)
  static constexpr uint32_t kV16PerK16 = (16 * D) >> 4;
  // The producer runs up to about kSlots / 2 key blocks ahead of the MMAs; the per-block
  // barrier rings must be deeper than that (see prefill.cu).
  static_assert(kIterRing >= (kSlots + 1) / 2 + 2, "per-block barrier ring too shallow for the K/V ring");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct PairPrefillParams {
  __nv_bfloat16* o;
  float* lse;
  int B, Hq, Hkv, Tq, Tk, g;
  int causal;
  int mode;   // 0: four heads at the same rows; 1: two heads at two row tiles; 2: one head at four row tiles
  int n_qt;   // query tiles of 128 rows
  int units;  // work units of four tiles, heaviest first when causal
  float c;    // scale * log2(e)
};

struct PairUnit {
  int b, kvh;
  int head[2];  // this CTA's two tiles
  int row0[2];
  int nkv[2];   // key blocks the pair's slot q walks (0 = slot inactive)
};

__device__ __forceinline__ int pair_kv_tiles(const PairPrefillParams& p, int row0) {
  if (row0 >= p.Tq) return 0;
  const int all = (p.Tk + 127) / 128;
  if (!p.causal) return all;
  const int last_row = min(row0 + 127, p.Tq - 1);
  return min(all, last_row / 128 + 1);
}

__device__ __forceinline__ PairUnit decode_pair_unit(const PairPrefillParams& p, int unit, int rank) {
  PairUnit u;
  if (p.mode == 0) {
    const int groups = p.Hq / 4;
    const int per_rank = groups * p.B;
    const int rk = unit / per_rank, rest = unit % per_rank;
    const int hg = rest % groups;
    u.b = rest / groups;
    const int qt = p.causal ? (p.n_qt - 1 - rk) : rk;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      u.head[q] = 4 * hg + 2 * rank + q;
      u.row0[q] = qt * 128;
      u.nkv[q] = pair_kv_tiles(p, qt * 128);
    }
  } else if (p.mode == 1) {
    const int hp_count = p.Hq / 2, n_tp = (p.n_qt + 1) / 2;
    const int per_rank = hp_count * p.B;
    const int rk = unit / per_rank, rest = unit % per_rank;
    const int hp = rest % hp_count;
    u.b = rest / hp_count;
    const int tp = p.causal ? (n_tp - 1 - rk) : rk;
    const int n = max(pair_kv_tiles(p, 2 * tp * 128), pair_kv_tiles(p, (2 * tp + 1) * 128));
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      u.head[q] = 2 * hp + q;
      u.row0[q] = (2 * tp + rank) * 128;
      u.nkv[q] = n;
    }
  } else {
    const int n_s = (p.n_qt + 3) / 4;
    const int per_rank = p.Hq * p.B;
    const int rk = unit / per_rank, rest = unit % per_rank;
    const int h = rest % p.Hq;
    u.b = rest / p.Hq;
    const int s = p.causal ? (n_s - 1 - rk) : rk;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      u.head[q] = h;
      u.row0[q] = (4 * s + 2 * rank + q) * 128;
      u.nkv[q] = max(pair_kv_tiles(p, (4 * s + q) * 128), pair_kv_tiles(p, (4 * s + 2 + q) * 128));
    }
  }
  u.kvh = u.head[0] / p.g;
  return u;
}

// Key block j has MMA work iff some slot issues S_q(j) (j < nkv_q) or PV_q(j-1) (0 < j <= nkv_q).
__device__ __forceinline__ bool pair_block_has_work(const PairUnit& u, int j) {
  const int n = max(u.nkv[0], u.nkv[1]);
  return j <= n && (j < n || j > 0);
}

// Persistent pairs: pair c takes units in rounds of (number of pairs), in a snake order.
__device__ __forceinline__ int pair_unit_index(int round, int cid, int ncl) {
  const int base = round * ncl;
  return (round & 1) ? base + ncl - 1 - cid : base + cid;
}

template <int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(352, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PairPrefillParams p) {
  using Cfg = PairPrefillCfg<D>;
  constexpr int R = Cfg::kIterRing;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                         // [2][Q tile]
  uint8_t* sKV = smem + 2 * Cfg::kQTileBytes;  // [slots][half tile]

  // CTA 0 only: q_full (both CTAs' Q tiles of a unit), kv_ready[j % R] (both CTAs' halves of
  // K(j) and V(j-1)): two arrivals (one producer per CTA, each with its bytes) per phase;
  // p_peer[q]: CTA 1 wrote P_q(j) (one arrival per block).
  __shared__ uint64_t q_full, kv_ready[R], p_peer[2];
  // Both CTAs, completed by the issuer's commits into both: s_full1 (S_1(j) done), iter_done
  // (the last MMA of key block j done; releases K(j) and V(j-1)), o_done[q] (slot q's O final).
  __shared__ uint64_t s_full1, iter_done[R], o_done[2];
  __shared__ uint64_t mma_drain;  // CTA 0: every MMA done before TMEM is freed
  __shared__ uint32_t tmem_base_holder;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    mbar_init(&q_full, 2);
    for (int r = 0; r < R; ++r) {
      mbar_init(&kv_ready[r], 2);
      mbar_init(&iter_done[r], 1);
    }
    mbar_init(&p_peer[0], 1);
    mbar_init(&p_peer[1], 1);
    mbar_init(&s_full1, 1);
    mbar_init(&o_done[0], 1);
    mbar_init(&o_done[1], 1);
    mbar_init(&mma_drain, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc_pair(&tmem_base_holder, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated before any cross-CTA traffic
  tc_fence_after();
  const uint32_t tmem = tmem_base_holder;
  volatile int* abort_p = &abort_flag;
  const uint32_t peer_abort = cluster_addr(smem_u32(&abort_flag), rank ^ 1u);
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    return pair_wait(bar, parity, abort_p, peer_abort, kPairTimeoutNs);
  };

  if (warp == 8) {
    // ------------------------------ TMA producer (both CTAs) ------------------------------
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      const uint32_t qf_cl = cluster_addr(smem_u32(&q_full), 0);
      int G = 0, U = 0;
      int slot = 0, filled = 0;
      int rel[Cfg::kSlots];  // block whose last MMA releases the item now in each slot
      int done_upto = -1;    // blocks complete in order: no wait at or below the last one seen
      auto wait_block = [&](int r) -> bool {
        if (r <= done_upto) return true;
        if (!wait(&iter_done[r % R], static_cast<uint32_t>(r / R) & 1u)) return false;
        done_upto = r;
        return true;
      };
      bool alive = true;
      for (int round = 0; alive && round * ncl < p.units; ++round) {
        const int idx = pair_unit_index(round, cid, ncl);
        if (idx >= p.units) continue;
        const PairUnit u = decode_pair_unit(p, idx, static_cast<int>(rank));
        const int n_iter = max(u.nkv[0], u.nkv[1]);
        // this unit's Q overwrites the previous one's: wait for its last S MMAs (block G - 2)
        if (U > 0 && !wait_block(G - 2)) break;
        const int nq = (u.nkv[0] > 0) + (u.nkv[1] > 0);
        mbar_arrive_expect_tx_cluster(qf_cl, nq * Cfg::kQTileBytes);
        for (int q = 0; q < 2; ++q) {
          if (u.nkv[q] == 0) continue;
          // rows past Tq (a tile of a unit at the end of the sequence) read as zero
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_3d_pair(sQ + q * Cfg::kQTileBytes + kb * Cfg::kQBoxBytes, &tmQ, qf_cl, kb * 64, u.row0[q],
                             u.b * p.Hq + u.head[q]);
        }
        const int zkv = u.b * p.Hkv + u.kvh;
        const int n_items = 2 * n_iter;  // item 2j = K(j) half, item 2j + 1 = V(j) half
        for (int i = 0; i < n_items; ++i) {
          if (filled == Cfg::kSlots) {
            if (!wait_block(rel[slot])) {
              alive = false;
              break;
            }
          } else {
            ++filled;
          }
          const int it = (i + 1) >> 1;  // K(j) is read in block j, V(j) in block j + 1
          rel[slot] = G + it;
          const uint32_t rb = cluster_addr(smem_u32(&kv_ready[(G + it) % R]), 0);
          if (i == 0 || (i & 1)) {  // first item of block `it`: this CTA's bytes of both halves
            const int ntiles = (it >= 1 ? 1 : 0) + (it < n_iter ? 1 : 0);
            mbar_arrive_expect_tx_cluster(rb, ntiles * Cfg::kHalfBytes);
          }
          uint8_t* dst = sKV + slot * Cfg::kHalfBytes;
          const int key0 = (i >> 1) * 128;
          if (i & 1) {
            // V(j): all 128 keys, this CTA's D/2 columns
            tma_load_3d_pair(dst, &tmV, rb, static_cast<int>(rank) * (D / 2), key0, zkv);
          } else {
            // K(j): this CTA's 64 keys, all D columns
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_3d_pair(dst + kb * Cfg::kKBoxBytes, &tmK, rb, kb * 64, key0 + static_cast<int>(rank) * 64, zkv);
          }
          if (++slot == Cfg::kSlots) slot = 0;
        }
        G += n_iter + 1;
        ++U;
      }
      if (*abort_p) {
        // let copies still in flight land before the CTA exits (1 ms of wall time)
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 9 || warp == 10) {
    if (rank == 0) {
      // Handoffs to the issuer go through hardware named barriers (bar.sync cannot time out,
      // so every arrival sequence runs to the end even after an abort, one for one with the
      // issuer's syncs):
      //  * data of key block j: the helper arrives on kPBarData, the issuer syncs and
      //    acknowledges on kPBarDataAck, the helper syncs on the acknowledgement;
      //  * P_q(j): this CTA's 4 softmax warps of slot q and the helper (after CTA 1's arrival
      //    on p_peer[q]) arrive on kPBarP0 + q, the issuer syncs before PV_q(j). An arrival
      //    for P_q(j + 1) needs S_q(j + 1), which is issued after the sync for P_q(j).
      if (warp == 10) {
        // ------------------------------ wait helper (CTA 0) ------------------------------
        int G = 0, U = 0;
        int pc[2] = {0, 0};  // phases of p_peer[q] consumed so far
        for (int round = 0; round * ncl < p.units; ++round) {
          const int idx = pair_unit_index(round, cid, ncl);
          if (idx >= p.units) continue;
          const PairUnit u = decode_pair_unit(p, idx, 0);
          const int n_iter = max(u.nkv[0], u.nkv[1]);
          if (lane == 0) wait(&q_full, static_cast<uint32_t>(U) & 1u);
          for (int j = 0; j <= n_iter; ++j) {
            if (pair_block_has_work(u, j)) {
              if (lane == 0 && !*abort_p)
                wait(&kv_ready[(G + j) % R], static_cast<uint32_t>((G + j) / R) & 1u);
              __syncwarp();
              named_bar_arrive(kPBarData, kPHandoff);
              named_bar_sync(kPBarDataAck, kPHandoff);
            }
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              const int q = 1 - qq;
              if (j > 0 && j - 1 < u.nkv[q]) {  // the issuer syncs for P_q(j - 1) now
                if (lane == 0 && !*abort_p) wait(&p_peer[q], static_cast<uint32_t>(pc[q]) & 1u);
                ++pc[q];
                __syncwarp();
                named_bar_arrive(kPBarP0 + q, kPLeaderP);
              }
            }
          }
          G += n_iter + 1;
          ++U;
        }
      } else {
        // ------------------------------ MMA issuer (CTA 0) ------------------------------
        // Issue order per key block j: PV_1(j-1), S_1(j), PV_0(j-1), S_0(j); the tensor pipe
        // runs one thread's MMAs in issue order (see prefill.cu for why this order is sound).
        // Descriptors advance by adding (byte offset >> 4) to the start-address field.
        constexpr uint32_t kQTile16 = Cfg::kQTileBytes >> 4;
        constexpr uint32_t kSlot16 = Cfg::kHalfBytes >> 4, kRing16 = Cfg::kSlots * kSlot16;
        const uint64_t dQ = make_sdesc(smem_u32(sQ), 16, 1024, 2);
        const uint64_t dK = make_sdesc(smem_u32(sKV), 16, 1024, 2);
        const uint64_t dV = (D == 128) ? make_sdesc(smem_u32(sKV), 16384, 1024, 2)  // MN-major, 128-byte rows
                                       : make_sdesc(smem_u32(sKV), 8192, 512, 4);    // MN-major, 64-byte rows
        uint32_t k16 = 0;                  // slot of K(j)
        uint32_t v16 = kRing16 - kSlot16;  // slot of V(j-1), used only when j > 0
        bool any_mma = false;
        int G = 0;
        for (int round = 0; round * ncl < p.units; ++round) {
          const int idx = pair_unit_index(round, cid, ncl);
          if (idx >= p.units) continue;
          const PairUnit u = decode_pair_unit(p, idx, 0);
          const int n_iter = max(u.nkv[0], u.nkv[1]);
          const int nkv0 = u.nkv[0], nkv1 = u.nkv[1];
          for (int j = 0; j <= n_iter; ++j) {
            if (pair_block_has_work(u, j)) {
              __syncwarp();
              named_bar_sync(kPBarData, kPHandoff);
              named_bar_arrive(kPBarDataAck, kPHandoff);
            }
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              const int q = 1 - qq;
              const int nkv_q = q ? nkv1 : nkv0;
              const bool do_s = j < nkv_q, do_pv = j > 0 && j - 1 < nkv_q;
              if (!do_s && !do_pv) continue;
              if (do_pv) {
                __syncwarp();
                named_bar_sync(kPBarP0 + q, kPLeaderP);
              }
              if (lane == 0) {
                tc_fence_after();
                const uint32_t d_s = tmem + (q ? Cfg::kTmS1 : Cfg::kTmS0);
                if (do_pv) {
                  const uint32_t d_o = tmem + (q ? Cfg::kTmO1 : Cfg::kTmO0);
#pragma unroll
                  for (int kk = 0; kk < 128 / 16; ++kk)
                    umma_ts_pair(d_o, d_s + kk * 8, dV + v16 + kk * Cfg::kV16PerK16, Cfg::kIdescPV,
                                 (j > 1 || kk > 0) ? 1u : 0u);
                  if (j == nkv_q) umma_commit_pair(&o_done[q], 3);  // last block of this slot: O is final
                }
                if (do_s) {
#pragma unroll
                  for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offq = ((kk >> 2) * Cfg::kQBoxBytes + (kk & 3) * 32) >> 4;
                    const uint32_t offk = ((kk >> 2) * Cfg::kKBoxBytes + (kk & 3) * 32) >> 4;
                    umma_ss_pair(d_s, dQ + q * kQTile16 + offq, dK + k16 + offk, Cfg::kIdescQK, kk > 0 ? 1u : 0u);
                  }
                  if (q == 1) umma_commit_pair(&s_full1, 3);
                }
                any_mma = true;
              }
            }
            if (lane == 0) umma_commit_pair(&iter_done[(G + j) % R], 3);
            if (j < n_iter) {
              v16 = k16 + kSlot16;  // V(j) sits in the slot after K(j)
              if (v16 >= kRing16) v16 -= kRing16;
              k16 += 2 * kSlot16;
              if (k16 >= kRing16) k16 -= kRing16;
            }
          }
          G += n_iter + 1;
        }
        if (lane == 0 && any_mma) {  // every MMA has finished before TMEM is released
          umma_commit_pair(&mma_drain, 1);
          wait(&mma_drain, 0);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------ softmax warps (both CTAs) ------------------------------
    const int q = warp >> 2;
    const int wq = warp & 3;
    const int row_in_tile = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + (q ? Cfg::kTmS1 : Cfg::kTmS0);
    const uint32_t t_o = tmem + lane_off + (q ? Cfg::kTmO1 : Cfg::kTmO0);
    const uint32_t p_peer_cl = cluster_addr(smem_u32(&p_peer[q]), 0);
    const float c = p.c;
    bool ok = true;
    int G = 0;
    int s1_count = 0;  // S_1 blocks committed in earlier units (phases of s_full1)
    int o_count = 0;   // earlier units in which this slot was active (phases of o_done[q])
    for (int round = 0; round * ncl < p.units; ++round) {
      const int idx = pair_unit_index(round, cid, ncl);
      if (idx >= p.units) continue;
      const PairUnit u = decode_pair_unit(p, idx, static_cast<int>(rank));
      const int n_iter = max(u.nkv[0], u.nkv[1]);
      const int nkv = u.nkv[q];
      const int row0 = u.row0[q];
      const int head = u.head[q];
      const int row = row0 + row_in_tile;
      float m_run = -INFINITY;
      float l_run = 0.f;

      for (int j = 0; j < nkv; ++j) {
        // S_q(j) ready: slot 1 on s_full1, slot 0 on the per-block barrier that follows S_0(j).
        // After a failed wait the warp skips the work but still reports P, once per block.
        if (ok) {
          const bool w = (q == 1) ? wait(&s_full1, static_cast<uint32_t>(s1_count + j) & 1u)
                                  : wait(&iter_done[(G + j) % R], static_cast<uint32_t>((G + j) / R) & 1u);
          ok = __all_sync(0xFFFFFFFFu, w);
        }
        if (ok) {
          tc_fence_after();
          uint32_t sr[128];
          const int j0 = j * 128;
          // blocks past the diagonal or the end of the keys need the element mask before the
          // maximum; every other block takes the row maximum from the reducing TMEM load
          const bool need_mask = (j0 + 128 > p.Tk) || (p.causal && j0 + 127 > row0);
          float m_raw;
          if (!need_mask) {
            m_raw = tmem_ld128_max(t_s, sr);
          } else {
            tmem_ld128(t_s, sr);
            const int lim = p.causal ? min(p.Tk - 1, row) : (p.Tk - 1);  // last visible key of this row
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
          const bool grow = m_cand > m_run + kPairRescaleThreshold;
          float corr = 1.f;
          if (grow) {
            corr = ex2_approx(m_run - m_cand);  // 0 when m_run = -inf
            m_run = m_cand;
          }
          const float base = (m_run == -INFINITY) ? 0.f : m_run;
          const float2 c2 = make_float2(c, c);
          const float2 nb2 = make_float2(-base, -base);
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float2 x = __ffma2_rn(
                  make_float2(__uint_as_float(sr[cc * 32 + 2 * k]), __uint_as_float(sr[cc * 32 + 2 * k + 1])), c2,
                  nb2);
              const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              acc[k & 3] = __fadd2_rn(acc[k & 3], pp);
              pk[k] = pack_bf16x2(pp.x, pp.y);
            }
            tmem_st16(t_s + cc * 16, pk);
          }
          const float2 a01 = __fadd2_rn(acc[0], acc[1]);
          const float2 a23 = __fadd2_rn(acc[2], acc[3]);
          l_run = l_run * corr + ((a01.x + a01.y) + (a23.x + a23.y));
          if (j > 0 && __any_sync(0xFFFFFFFFu, grow)) {
            // PV_q(j-1) was issued before S_q(j), so it has completed: rescale O in TMEM
#pragma unroll
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
        if (rank == 0) {
          named_bar_arrive(kPBarP0 + q, kPLeaderP);  // P_q(j) (and any O rescale) is in TMEM
        } else {
          named_bar_sync(kPBarP0 + q, kPPeerP);      // all 128 rows of this CTA's tile written
          if (wq == 0 && lane == 0) mbar_arrive_cluster(p_peer_cl);
        }
      }

      if (ok && nkv > 0) {
        ok = __all_sync(0xFFFFFFFFu, wait(&o_done[q], static_cast<uint32_t>(o_count) & 1u));
        tc_fence_after();
        if (ok) {
          const float inv_l = 1.f / l_run;
          const bool store = row < p.Tq;
          const size_t orow = (static_cast<size_t>(u.b) * p.Hq + head) * p.Tq + row;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            tmem_ld32(t_o + cc * 32, ov);
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              pk[k] = pack_bf16x2(__uint_as_float(ov[2 * k]) * inv_l, __uint_as_float(ov[2 * k + 1]) * inv_l);
            if (store) {
              uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D + cc * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
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
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs, copies or arrivals may touch it
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// --------------------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------------------
// Pairs that can be resident at once (one CTA per SM), per device and head size.
template <int D>
static int max_pairs() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    using Cfg = PairPrefillCfg<D>;
    if (cudaFuncSetAttribute(attn_fwd_pair_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::kSmemBytes) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_fwd_pair_kernel<D>, &cfg) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

template <int D>
static cudaError_t launch_pair_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                 const PairPrefillParams& p, cudaStream_t stream) {
  using Cfg = PairPrefillCfg<D>;
  const int pairs = max_pairs<D>();
  if (pairs <= 0) return cudaErrorInvalidDevice;
  const int ncl = p.units < pairs ? p.units : pairs;
  attn_fwd_pair_kernel<D><<<2 * ncl, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

// Returns cudaErrorInvalidValue if a tensor map cannot be built, cudaErrorInvalidDevice if no
// pair of CTAs can be resident.
cudaError_t launch_attn_fwd_pair(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                 int Hkv, int Tq, int Tk, int d, int causal, float scale, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const bool ok = encode_bf16_box_map(&mq, q, d, Tq, B * Hq, 64, 128, 128) &&
                  encode_bf16_box_map(&mk, k, d, Tk, B * Hkv, 64, 64, 128) &&
                  (d == 128 ? encode_bf16_box_map(&mv, v, d, Tk, B * Hkv, 64, 128, 128)
                            : encode_bf16_box_map(&mv, v, d, Tk, B * Hkv, 32, 128, 64));
  if (!ok) return cudaErrorInvalidValue;
  PairPrefillParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Tq = Tq;
  p.Tk = Tk;
  p.g = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.mode = (p.g % 4 == 0) ? 0 : ((p.g % 2 == 0) ? 1 : 2);
  p.n_qt = (Tq + 127) / 128;
  p.c = scale * 1.4426950408889634f;
  long long units;
  if (p.mode == 0)
    units = static_cast<long long>(p.n_qt) * (Hq / 4) * B;
  else if (p.mode == 1)
    units = static_cast<long long>((p.n_qt + 1) / 2) * (Hq / 2) * B;
  else
    units = static_cast<long long>((p.n_qt + 3) / 4) * Hq * B;
  if (units <= 0 || units > 0x3FFFFFFFLL) return cudaErrorInvalidValue;
  p.units = static_cast<int>(units);
  return d == 64 ? launch_pair_d<64>(mq, mk, mv, p, stream) : launch_pair_d<128>(mq, mk, mv, p, stream);
}

uint32_t prefill_pair_take_device_error() { return take_device_error_word(); }

}  // namespace gb300
