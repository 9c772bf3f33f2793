// backward.cu - the attention backward pass on 5th-generation tensor cores (sm_103a).
//
// What it computes ("FlashAttention: attention without the n x n matrix", section
// "Backward pass: recomputing is cheaper than storing"): from the forward's O and its
// per-row log-sum-exp L, the scores of each block are computed again and the
// probabilities recovered without normalisation, P_ij = exp(S_ij - L_i); then
//   dV = P^T dO,  dP = dO V^T,  dS_ij = P_ij (dP_ij - D_i) with D_i = dO_i . O_i,
//   dQ = dS K * scale,  dK = dS^T Q * scale.
// With grouped-query attention the gradients of a K/V head are the sums over the g
// query heads that read it.
//
// Three kernels, no atomics (every output is accumulated by one CTA):
//   bwd_delta_kernel   D_i = dO_i . O_i, one warp per row (HBM-bound, fp32 into the workspace).
//   bwd_dkdv_kernel    one CTA per (block of 128 keys, K/V head): walks the g query heads x
//                      the visible query blocks; per block S^T = K Q^T and dP^T = V dO^T into
//                      TMEM, 8 warps (two per key row) form P^T (phase 1, from S^T alone) and
//                      dS^T (phase 2, with dP^T) as bf16 pairs, each in place over the fp32
//                      values it came from, then dV += P^T dO and dK += dS^T Q with the A
//                      operand from TMEM; dV and dK stay in TMEM until the end.
//   bwd_dq_kernel      one CTA per (block of 128 queries, query head): walks the visible key
//                      blocks; S = Q K^T, dP = dO V^T, dS (bf16) into S's columns, dQ += dS K.
// Each kernel: warps 0-7 compute (warps w and w + 4 share TMEM lanes 32(w mod 4) .. + 31 and
// take one half of the row's 128 columns each), warp 8 issues the TMA copies (rings of 3 and 2
// tiles for the two walked operands), warp 9 issues the MMAs from one thread, warp 10 waits on
// the copies for it. The MMA warp learns of every event through hardware named barriers (see
// kBwdBarP1 below); every other wait is an mbarrier wait with a time limit. The next block's
// scores are issued while this block's gradient GEMMs are still queued, so the compute phases of
// one block overlap the tensor work of its neighbours (recomputing S and dP in the dQ kernel
// costs 2 of its 3 GEMMs; the layout keeps every output with one owner). Both grids are numbered
// longest CTA first within groups of heads (bwd_cta_order).
//
// P is rounded to bf16 for dV = P^T dO and dS to bf16 for the two gradient GEMMs; all
// accumulation is fp32 in TMEM; outputs are rounded once to bf16.
#include "common.cuh"

namespace gb300 {

constexpr uint64_t kBwdWaitTimeoutNs = 2000000000ull;  // 2 s per wait
// Hardware named barriers (0 is __syncthreads; the dK/dV kernel's compute warps use 1 among
// themselves). The MMA thread learns of every event it waits for through these, not through an
// mbarrier wait of its own: under MMA load such a wait costs it a few hundred clocks even on a
// phase that has already completed, and the tensor pipe idles meanwhile.
//  * kBwdBarP1 / kBwdBarP: the 8 compute warps arrive once per block (P^T written; dS written),
//    the MMA warp syncs (count 256 + 32). An arrival for block i + 1 needs a GEMM that is only
//    issued after the sync for block i, so arrivals never run a generation ahead.
//  * kBwdBarGo / kBwdBarAck: a helper warp waits on the mbarriers of the streamed tiles and hands
//    each completion to the MMA warp (Go), which acknowledges it (Ack) before the helper looks at
//    the next one, so the two warps stay in lockstep.
// Every arrival and sync runs once per block on every path, also after an abort (a bar.sync
// cannot time out): the counts on the two sides are equal by construction.
constexpr uint32_t kBwdBarP1 = 2, kBwdBarP = 3, kBwdBarGo = 4, kBwdBarAck = 5;
constexpr uint32_t kBwdComputeAndMma = 288, kBwdPair = 64;
constexpr float kLog2e = 1.4426950408889634f;
// CTA order of both kernels: the (batch, head) rows of the grid go in groups of this many, and
// within a group the longest CTAs come first. The group bounds the data that the running CTAs
// share through L2 (in the dK/dV kernel, a row's Q and dO: 67 MB for 4 rows of the causal GQA
// prefill workload, B2 Hq32 Hkv8 T8192 d128); longest-first keeps the last CTAs short. Ordered
// longest-first over the whole grid at once, the dK/dV kernel read 3.2x its inputs from DRAM.
constexpr int kBwdOrderGroup = 4;

// Linear CTA number -> (row of the grid in y, position along x), as above: groups of
// kBwdOrderGroup rows, position-major within a group (the last group may be smaller).
__device__ __forceinline__ void bwd_cta_order(int& row_y, int& pos_x) {
  const int lin = blockIdx.x + gridDim.x * blockIdx.y;
  const int grp = lin / (kBwdOrderGroup * static_cast<int>(gridDim.x));
  const int gsz = min(kBwdOrderGroup, static_cast<int>(gridDim.y) - grp * kBwdOrderGroup);
  const int within = lin - grp * kBwdOrderGroup * static_cast<int>(gridDim.x);
  row_y = grp * kBwdOrderGroup + within % gsz;
  pos_x = within / gsz;
}

template <int D>
struct BwdCfg {
  static constexpr int kBoxBytes = 128 * 128;            // 128 rows x 64 bf16 columns, 128-byte swizzle
  static constexpr int kNumBox = D / 64;
  static constexpr int kTileBytes = kNumBox * kBoxBytes;  // 128 rows x D
  static constexpr int kThreads = 352;                    // warps 0-7 compute, 8 TMA, 9 MMA, 10 wait helper
  // 7 tiles in both kernels (2 resident, 3 + 2 streamed; see each kernel); at least 116 KB so that
  // one CTA runs per SM (each allocates all 512 TMEM columns)
  static constexpr int kSmemBytes = (7 * kTileBytes + 1024) > 116 * 1024 ? (7 * kTileBytes + 1024) : 116 * 1024;
  // [128 x 128] = A (128 x D, K-major) . B^T (B 128 x D, K-major)
  static constexpr uint32_t kIdescS = make_idesc_bf16_f32(128, 128, false);
  // [128 x D] += A (TMEM, 128 x 128 bf16) . B (128 x D, MN-major)
  static constexpr uint32_t kIdescAcc = make_idesc_bf16_f32(128, D, true);
  // dK/dV kernel TMEM columns: region S [0, 128) (S^T, then P^T), region dP [128, 256) (dP^T, then
  // dS^T), then the fp32 accumulators dV and dK
  static constexpr uint32_t kTmAcc0 = 256, kTmAcc1 = 256 + D;
  // dQ kernel TMEM: S in [0, 128) and [128, 256) by turns, dP in [256, 384), the fp32 dQ
  // accumulator from 384
  static constexpr uint32_t kTmDp = 256, kTmDq = 384;
};

struct BwdParams {
  const float* lse;    // [B, Hq, Tq], natural log
  const float* delta;  // [B, Hq, Tq]
  __nv_bfloat16* dq;   // [B, Hq, Tq, D]
  __nv_bfloat16* dk;   // [B, Hkv, Tk, D]
  __nv_bfloat16* dv;
  int B, Hq, Hkv, Tq, Tk, g, causal;
  float c;             // scale * log2(e)
  float scale;
  int out_v8;          // dq, dk and dv are 32-byte aligned: rows are written with 32-byte stores
};

// Shared-memory descriptors of a tile at byte offset `off` from the descriptor of tile 0: the start
// address field holds address >> 4 in the low 14 bits, and no address here reaches 2^18, so adding
// off >> 4 to the whole descriptor moves the start and nothing else. The issuing thread forms each
// MMA's descriptors with one add instead of rebuilding them.
__device__ __forceinline__ uint64_t sdesc_at(uint64_t desc0, uint32_t off_bytes) { return desc0 + (off_bytes >> 4); }

// D[128 x 128] = A_tile . B_tile^T over K = D (both tiles 128 rows x D, K-major; a, b are their
// descriptors with LBO 16, SBO 1024)
template <int D>
__device__ __forceinline__ void bwd_mma_scores(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  using Cfg = BwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off16 = ((kk >> 2) * Cfg::kBoxBytes + (kk & 3) * 32) >> 4;
    umma_ss(d_tmem, a_desc + off16, b_desc + off16, Cfg::kIdescS, kk > 0 ? 1u : 0u);
  }
}

// D[128 x D] (+)= A (TMEM, 128 rows x 128 bf16) . B (128 rows x D, MN-major), with A's bf16 pairs
// in the layout the score region holds after the two compute phases: for each half h of the 128
// columns, 32 columns at region + 64 h + a_off (a_off 0: P^T, 32: dS^T).
// b_desc: the B tile's MN-major descriptor (LBO = one 64-column box, SBO 1024); each K step of 16
// rows moves it by 2048 bytes.
template <int D>
__device__ __forceinline__ void bwd_mma_accumulate_split(uint32_t d_tmem, uint32_t region, uint32_t a_off,
                                                         uint64_t b_desc, bool accumulate) {
  using Cfg = BwdCfg<D>;
#pragma unroll
  for (int kk = 0; kk < 128 / 16; ++kk)
    umma_ts(d_tmem, region + (kk >> 2) * 64 + a_off + (kk & 3) * 8, b_desc + kk * (2048 >> 4), Cfg::kIdescAcc,
            (accumulate || kk > 0) ? 1u : 0u);
}

// 32-byte global store (dst 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Half `half` (columns [half*D/2, (half+1)*D/2)) of one row (this thread's TMEM lane) of a
// [128 x D] fp32 accumulator, times `mul`, to bf16 in global. Called by every thread of the
// warp (the TMEM load and the shuffles are warp-collective); `store` says whether this thread's
// row exists. With v8 (the outputs 32-byte aligned) the two lanes of each pair (rows r, r + 1,
// the same half) swap one 32-byte half of each 64-byte chunk, so that each 32-byte store
// writes 64 contiguous bytes of one row (measured: causal GQA B2 Hq32 T8192 backward
// 2.347-2.368 -> 2.318-2.326 ms, B1 Hq16 T4096 0.181-0.183 -> 0.178 ms, bitwise equal).
template <int D>
__device__ __forceinline__ void bwd_store_row(uint32_t t_acc, float mul, bool have, bool store, __nv_bfloat16* dst,
                                              int half, bool v8) {
  const bool odd = (threadIdx.x & 1) != 0;
  // the pair's two rows: their store flags and addresses
  const bool store_p = __shfl_xor_sync(0xFFFFFFFFu, store ? 1 : 0, 1) != 0;
  const unsigned long long dst_p = __shfl_xor_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(dst), 1);
  __nv_bfloat16* dst_e = odd ? reinterpret_cast<__nv_bfloat16*>(dst_p) : dst;
  __nv_bfloat16* dst_o = odd ? dst : reinterpret_cast<__nv_bfloat16*>(dst_p);
  const bool st_e = odd ? store_p : store, st_o = odd ? store : store_p;
#pragma unroll
  for (int c2 = 0; c2 < D / 64; ++c2) {
    const int cc = half * (D / 64) + c2;
    uint32_t v[32];
    if (have) {
      tmem_ld32(t_acc + cc * 32, v);  // warp-collective: every lane runs it
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = 0u;
    }
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) pk[k] = pack_bf16x2(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul);
    if (v8) {
      // after the swap pk[0..7] is this lane's 32 bytes of the even row, pk[8..15] of the odd row
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t r = __shfl_xor_sync(0xFFFFFFFFu, odd ? pk[k] : pk[8 + k], 1);
        if (odd) pk[k] = r; else pk[8 + k] = r;
      }
      if (st_e) st_global_v8(reinterpret_cast<uint32_t*>(dst_e + cc * 32) + (odd ? 8 : 0), pk);
      if (st_o) st_global_v8(reinterpret_cast<uint32_t*>(dst_o + cc * 32) + (odd ? 8 : 0), pk + 8);
    } else if (store) {
      uint4* o = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
      for (int w = 0; w < 4; ++w) o[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
    }
  }
}

// ------------------------------------------------------------------------------------------
// D_i = dO_i . O_i
// ------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        float* __restrict__ delta, long long rows) {
  constexpr int E = D / 32;  // elements per lane (2 or 4)
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const __nv_bfloat16* orow = o + row * D + lane * E;
  const __nv_bfloat16* drow = dout + row * D + lane * E;
  float acc = 0.f;
  if constexpr (E == 4) {
    const uint2 a = *reinterpret_cast<const uint2*>(orow), b = *reinterpret_cast<const uint2*>(drow);
    acc = fmaf(bf16lo_to_f32(a.x), bf16lo_to_f32(b.x), acc);
    acc = fmaf(bf16hi_to_f32(a.x), bf16hi_to_f32(b.x), acc);
    acc = fmaf(bf16lo_to_f32(a.y), bf16lo_to_f32(b.y), acc);
    acc = fmaf(bf16hi_to_f32(a.y), bf16hi_to_f32(b.y), acc);
  } else {
    const uint32_t a = *reinterpret_cast<const uint32_t*>(orow), b = *reinterpret_cast<const uint32_t*>(drow);
    acc = fmaf(bf16lo_to_f32(a), bf16lo_to_f32(b), acc);
    acc = fmaf(bf16hi_to_f32(a), bf16hi_to_f32(b), acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (lane == 0) delta[row] = acc;
}

// ------------------------------------------------------------------------------------------
// dK, dV: one CTA per (key block, K/V head)
// ------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(352, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdParams p) {
  using Cfg = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + Cfg::kTileBytes;
  // Q(i) in tile 2 + i mod 3, dO(i) in tile 5 + i mod 2. Q(i) is read by S^T(i), issued a block
  // early, and last by dK(i) at the end of block i; a third Q tile lets the copy of Q(i + 1) start a
  // block before S^T(i + 1) needs it. dO(i) is last read by dV(i), in the middle of block i.
  __shared__ uint64_t kv_full, q_full[3], q_empty[3], do_full[2], do_empty[2], s_ready, dp_ready, acc_done;
  __shared__ __align__(16) float nl_s[128];   // -L log2(e) per query row, read as float4
  __shared__ __align__(16) float ndl_s[128];  // -D per query row
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Longest CTAs first within each group of (batch, K/V head) rows: under the causal mask key
  // block kb meets n_qb - kb query blocks, so key block 0 of each head starts first.
  int bh, kb;
  bwd_cta_order(bh, kb);
  const int b = bh / p.Hkv, kvh = bh % p.Hkv;
  const int j0 = kb * 128;
  const int n_qb = (p.Tq + 127) / 128;
  // query blocks that see any key of this block (top-left causal: query q sees key j iff j <= q)
  const int i_first = p.causal ? j0 / 128 : 0;
  const int n_i = max(0, n_qb - i_first);
  const int n_it = p.g * n_i;

  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);
    }
    mbar_init(&s_ready, 1);
    mbar_init(&dp_ready, 1);
    mbar_init(&acc_done, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  volatile int* abort_p = &abort_flag;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_it > 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmDO);
      mbar_arrive_expect_tx(&kv_full, 2 * Cfg::kTileBytes);
      for (int kb = 0; kb < Cfg::kNumBox; ++kb) {
        tma_load_3d(sK + kb * Cfg::kBoxBytes, &tmK, &kv_full, kb * 64, j0, b * p.Hkv + kvh);
        tma_load_3d(sV + kb * Cfg::kBoxBytes, &tmV, &kv_full, kb * 64, j0, b * p.Hkv + kvh);
      }
      for (int it = 0; it < n_it; ++it) {
        const int sq = it % 3, sd = it & 1;
        const int h = kvh * p.g + it / n_i;
        const int i0 = (i_first + it % n_i) * 128;
        if (it >= 3 && !mbar_wait(&q_empty[sq], static_cast<uint32_t>(it / 3 - 1) & 1u, abort_p, kBwdWaitTimeoutNs))
          break;
        uint8_t* sQ = smem + (2 + sq) * Cfg::kTileBytes;
        mbar_arrive_expect_tx(&q_full[sq], Cfg::kTileBytes);
        for (int kb = 0; kb < Cfg::kNumBox; ++kb)
          tma_load_3d(sQ + kb * Cfg::kBoxBytes, &tmQ, &q_full[sq], kb * 64, i0, b * p.Hq + h);
        if (it >= 2 && !mbar_wait(&do_empty[sd], static_cast<uint32_t>((it >> 1) - 1) & 1u, abort_p, kBwdWaitTimeoutNs))
          break;
        uint8_t* sDO = smem + (5 + sd) * Cfg::kTileBytes;
        mbar_arrive_expect_tx(&do_full[sd], Cfg::kTileBytes);
        for (int kb = 0; kb < Cfg::kNumBox; ++kb)
          tma_load_3d(sDO + kb * Cfg::kBoxBytes, &tmDO, &do_full[sd], kb * 64, i0, b * p.Hq + h);
      }
      if (*abort_p) {  // let copies still in flight land before the CTA exits
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 10) {
    // ---------------- wait helper: Q(i), dO(i) of blocks 1 .. n-1 landed -> MMA warp ----------------
    for (int it = 1; it < n_it; ++it) {
      if (lane == 0 && !*abort_p &&
          mbar_wait(&q_full[it % 3], static_cast<uint32_t>(it / 3) & 1u, abort_p, kBwdWaitTimeoutNs))
        mbar_wait(&do_full[it & 1], static_cast<uint32_t>(it >> 1) & 1u, abort_p, kBwdWaitTimeoutNs);
      __syncwarp();
      named_bar_arrive(kBwdBarGo, kBwdPair);
      named_bar_sync(kBwdBarAck, kBwdPair);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (the whole warp runs the loop for the named barriers; lane 0 issues) ----------------
    // Region S holds S^T(i), which phase 1 turns into P^T(i) in place; region dP holds dP^T(i),
    // which phase 2 turns into dS^T(i) in place. Per block the issue order is
    //   [P1] dV(i) | S^T(i + 1) | [P] dK(i) | dP^T(i + 1)
    // The tensor pipe runs one thread's MMAs in issue order, so S^T(i + 1) overwrites P^T(i) only
    // after dV(i) has read it, and dP^T(i + 1) overwrites dS^T(i) only after dK(i). S^T(i + 1)
    // does not wait for phase 2 of block i, and phase 1 of block i + 1 runs while dK(i) and
    // dP^T(i + 1) occupy the pipe.
    const uint64_t aK = make_sdesc_sw128(smem_u32(sK), 16, 1024), aV = make_sdesc_sw128(smem_u32(sV), 16, 1024);
    // descriptors of the streamed tiles: Q(i) at tile 2 + i mod 3, dO(i) at 5 + i mod 2; K-major for the
    // score GEMMs, MN-major (LBO one box) as the B operand of dV and dK
    const uint64_t q_k0 = make_sdesc_sw128(smem_u32(smem + 2 * Cfg::kTileBytes), 16, 1024);
    const uint64_t q_mn0 = make_sdesc_sw128(smem_u32(smem + 2 * Cfg::kTileBytes), Cfg::kBoxBytes, 1024);
    auto aQ_of = [&](int it) { return sdesc_at(q_k0, (it % 3) * Cfg::kTileBytes); };
    auto aDO_of = [&](int it) { return sdesc_at(q_k0, (3 + (it & 1)) * Cfg::kTileBytes); };
    auto bQ_of = [&](int it) { return sdesc_at(q_mn0, (it % 3) * Cfg::kTileBytes); };
    auto bDO_of = [&](int it) { return sdesc_at(q_mn0, (3 + (it & 1)) * Cfg::kTileBytes); };
    // K, V and the first Q, dO tiles: the issuing thread's own waits, once per CTA. After a failed
    // wait (or an abort) the handoffs below still run to the end; only the MMAs are skipped.
    bool ok = true;
    // region S (columns [0, 128)) holds S^T, then P^T; region dP ([128, 256)) holds dP^T, then dS^T
    const uint32_t r_s = tmem, r_d = tmem + 128;
    if (lane == 0 && n_it > 0) {
      ok = mbar_wait(&kv_full, 0, abort_p, kBwdWaitTimeoutNs) && mbar_wait(&q_full[0], 0, abort_p, kBwdWaitTimeoutNs) &&
           mbar_wait(&do_full[0], 0, abort_p, kBwdWaitTimeoutNs);
      if (ok) {
        tc_fence_after();
        bwd_mma_scores<D>(r_s, aK, aQ_of(0));   // S^T(0) = K Q^T
        umma_commit(&s_ready);
        bwd_mma_scores<D>(r_d, aV, aDO_of(0));  // dP^T(0) = V dO^T
        umma_commit(&dp_ready);
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
    for (int it = 0; it < n_it; ++it) {
      __syncwarp();
      named_bar_sync(kBwdBarP1, kBwdComputeAndMma);  // P^T(i) is in region S
      if (lane == 0 && ok) {
        tc_fence_after();
        bwd_mma_accumulate_split<D>(tmem + Cfg::kTmAcc0, r_s, 0, bDO_of(it), it > 0);   // dV += P^T dO
        umma_commit(&do_empty[it & 1]);  // dO(i) read for the last time
      }
      if (it + 1 < n_it) {
        // S^T(i + 1) overwrites P^T(i) after dV(i) has read it (MMAs run in issue order), while
        // phase 2 of block i still works in region dP: phase 1 of the next block starts early
        named_bar_sync(kBwdBarGo, kBwdPair);     // Q(i + 1) and dO(i + 1) are in shared memory
        named_bar_arrive(kBwdBarAck, kBwdPair);
        if (lane == 0 && ok) {
          tc_fence_after();
          bwd_mma_scores<D>(r_s, aK, aQ_of(it + 1));
          umma_commit(&s_ready);
        }
      }
      __syncwarp();
      named_bar_sync(kBwdBarP, kBwdComputeAndMma);  // dS^T(i) is in region dP
      if (lane == 0 && ok) {
        tc_fence_after();
        bwd_mma_accumulate_split<D>(tmem + Cfg::kTmAcc1, r_d, 0, bQ_of(it), it > 0);   // dK += dS^T Q
        umma_commit(&q_empty[it % 3]);  // Q(i) read for the last time
        if (it + 1 < n_it) {
          bwd_mma_scores<D>(r_d, aV, aDO_of(it + 1));  // dP^T(i + 1) over dS^T(i), after dK(i) has read it
          umma_commit(&dp_ready);
        }
      }
    }
    if (lane == 0) umma_commit(&acc_done);  // every MMA issued above has completed when this arrives
    __syncwarp();
  } else {
    // ---------------- compute warps: key row j0 + (t & 127) (TMEM lane), query half t >> 7 ----------------
    const int t = threadIdx.x;
    const int row = t & 127, half = t >> 7;
    const int key = j0 + row;
    const bool key_ok = key < p.Tk;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float2 c2 = make_float2(p.c, p.c);
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int h = kvh * p.g + it / n_i;
      const int i0 = (i_first + it % n_i) * 128;
      // every key of the block is visible to every query of the query block: no mask
      const bool unmasked = j0 + 128 <= p.Tk && (!p.causal || j0 + 127 <= i0);
      named_bar_sync(1, 256);  // the previous block's readers of nl_s / ndl_s are done
      {
        const int q = i0 + row;
        const size_t r = (static_cast<size_t>(b) * p.Hq + h) * p.Tq + q;
        if (half == 0) nl_s[row] = q < p.Tq ? -(p.lse[r] * kLog2e) : -INFINITY;  // rows past Tq: P = 0
        else ndl_s[row] = q < p.Tq ? -p.delta[r] : 0.f;
      }
      named_bar_sync(1, 256);
      const uint32_t r_s = tmem + lane_off, r_d = tmem + lane_off + 128;
      float pv[64];  // this thread's 64 probabilities, kept between the two phases
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s_ready, static_cast<uint32_t>(it) & 1u, abort_p,
                                                      kBwdWaitTimeoutNs));
      if (ok) {
        tc_fence_after();
        // phase 1: P^T from S^T alone. This half's 64 queries in two chunks of 32; chunk cc reads
        // columns [64 half + 32 cc, + 32) and writes its bf16 pairs to [64 half + 16 cc, + 16),
        // inside what this half has read
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int q0 = half * 64 + cc * 32;
          uint32_t sr[32];
          tmem_ld32(r_s + q0, sr);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            const float4 l4 = *reinterpret_cast<const float4*>(nl_s + q0 + 4 * v4);
            const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(sr[4 * v4]), __uint_as_float(sr[4 * v4 + 1])), c2,
                                          make_float2(l4.x, l4.y));
            const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(sr[4 * v4 + 2]), __uint_as_float(sr[4 * v4 + 3])),
                                          c2, make_float2(l4.z, l4.w));
            pv[cc * 32 + 4 * v4] = ex2_approx(x01.x);
            pv[cc * 32 + 4 * v4 + 1] = ex2_approx(x01.y);
            pv[cc * 32 + 4 * v4 + 2] = ex2_approx(x23.x);
            pv[cc * 32 + 4 * v4 + 3] = ex2_approx(x23.y);
          }
          if (!unmasked) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (!(key_ok && (!p.causal || key <= i0 + q0 + k))) pv[cc * 32 + k] = 0.f;
          }
          uint32_t pp[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) pp[k] = pack_bf16x2(pv[cc * 32 + 2 * k], pv[cc * 32 + 2 * k + 1]);
          tmem_st16(r_s + half * 64 + cc * 16, pp);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      named_bar_arrive(kBwdBarP1, kBwdComputeAndMma);  // P^T(i) is in TMEM (every block, also after a failed wait)
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&dp_ready, static_cast<uint32_t>(it) & 1u, abort_p,
                                                      kBwdWaitTimeoutNs));
      if (ok) {
        tc_fence_after();
        // phase 2: dS^T = P^T (dP^T - D), in place: chunk cc reads dP^T columns [64 half + 32 cc, + 32)
        // and writes its bf16 pairs to [64 half + 16 cc, + 16), inside what this half has read
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int q0 = half * 64 + cc * 32;
          uint32_t dr[32];
          tmem_ld32(r_d + q0, dr);
          uint32_t dd[16];
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            const float4 d4 = *reinterpret_cast<const float4*>(ndl_s + q0 + 4 * v4);
            const float2 g01 = __fmul2_rn(make_float2(pv[cc * 32 + 4 * v4], pv[cc * 32 + 4 * v4 + 1]),
                                          __fadd2_rn(make_float2(__uint_as_float(dr[4 * v4]), __uint_as_float(dr[4 * v4 + 1])),
                                                     make_float2(d4.x, d4.y)));
            const float2 g23 = __fmul2_rn(make_float2(pv[cc * 32 + 4 * v4 + 2], pv[cc * 32 + 4 * v4 + 3]),
                                          __fadd2_rn(make_float2(__uint_as_float(dr[4 * v4 + 2]), __uint_as_float(dr[4 * v4 + 3])),
                                                     make_float2(d4.z, d4.w)));
            dd[2 * v4] = pack_bf16x2(g01.x, g01.y);
            dd[2 * v4 + 1] = pack_bf16x2(g23.x, g23.y);
          }
          tmem_st16(r_d + half * 64 + cc * 16, dd);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      named_bar_arrive(kBwdBarP, kBwdComputeAndMma);  // dS^T(i) is in TMEM (every block, also after a failed wait)
    }
    if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&acc_done, 0, abort_p, kBwdWaitTimeoutNs));
    tc_fence_after();
    const size_t orow = (static_cast<size_t>(b) * p.Hkv + kvh) * p.Tk + key;
    const bool have = ok && n_it > 0;
    bwd_store_row<D>(tmem + lane_off + Cfg::kTmAcc0, 1.f, have, key_ok && (ok || n_it == 0), p.dv + orow * D, half,
                     p.out_v8 != 0);
    bwd_store_row<D>(tmem + lane_off + Cfg::kTmAcc1, p.scale, have, key_ok && (ok || n_it == 0), p.dk + orow * D,
                     half, p.out_v8 != 0);
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// dQ: one CTA per (query block, query head)
// ------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(352, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdParams p) {
  using Cfg = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = smem + Cfg::kTileBytes;
  // K(j) in tile 2 + j mod 3, V(j) in tile 5 + j mod 2. K is read by S(j) and, one block later, by
  // dQ(j), while S(j + 2) is already wanted: three K tiles are live at once.
  __shared__ uint64_t qd_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_ready[2], dp_ready, acc_done;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Longest CTAs first within each group of (batch, query head) rows: under the causal mask query
  // block qb meets qb + 1 key blocks, so the query blocks are counted down.
  int bh, slot;
  bwd_cta_order(bh, slot);
  const int qb = p.causal ? static_cast<int>(gridDim.x) - 1 - slot : slot;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int kvh = h / p.g;
  const int i0 = qb * 128;
  const int n_kb = (p.Tk + 127) / 128;
  const int last_row = min(i0 + 127, p.Tq - 1);
  const int n_j = p.causal ? min(n_kb, last_row / 128 + 1) : n_kb;

  if (threadIdx.x == 0) {
    mbar_init(&qd_full, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_ready[s], 1);
    }
    mbar_init(&dp_ready, 1);
    mbar_init(&acc_done, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  volatile int* abort_p = &abort_flag;

  if (warp == 8) {
    // ---------------- TMA producer: K(j) then V(j), each on its own ring ----------------
    if (lane == 0 && n_j > 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmDO);
      mbar_arrive_expect_tx(&qd_full, 2 * Cfg::kTileBytes);
      for (int kb = 0; kb < Cfg::kNumBox; ++kb) {
        tma_load_3d(sQ + kb * Cfg::kBoxBytes, &tmQ, &qd_full, kb * 64, i0, b * p.Hq + h);
        tma_load_3d(sDO + kb * Cfg::kBoxBytes, &tmDO, &qd_full, kb * 64, i0, b * p.Hq + h);
      }
      for (int j = 0; j < n_j; ++j) {
        const int sk = j % 3, sv = j & 1;
        if (j >= 3 && !mbar_wait(&k_empty[sk], static_cast<uint32_t>(j / 3 - 1) & 1u, abort_p, kBwdWaitTimeoutNs))
          break;
        uint8_t* sK = smem + (2 + sk) * Cfg::kTileBytes;
        mbar_arrive_expect_tx(&k_full[sk], Cfg::kTileBytes);
        for (int kb = 0; kb < Cfg::kNumBox; ++kb)
          tma_load_3d(sK + kb * Cfg::kBoxBytes, &tmK, &k_full[sk], kb * 64, j * 128, b * p.Hkv + kvh);
        if (j >= 2 && !mbar_wait(&v_empty[sv], static_cast<uint32_t>((j >> 1) - 1) & 1u, abort_p, kBwdWaitTimeoutNs))
          break;
        uint8_t* sV = smem + (5 + sv) * Cfg::kTileBytes;
        mbar_arrive_expect_tx(&v_full[sv], Cfg::kTileBytes);
        for (int kb = 0; kb < Cfg::kNumBox; ++kb)
          tma_load_3d(sV + kb * Cfg::kBoxBytes, &tmV, &v_full[sv], kb * 64, j * 128, b * p.Hkv + kvh);
      }
      if (*abort_p) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 10) {
    // ---------------- wait helper: V(j + 1), then K(j + 2), landed -> MMA warp, once per block j ----------------
    for (int j = 0; j < n_j; ++j) {
      if (j + 1 < n_j) {
        if (lane == 0 && !*abort_p)
          mbar_wait(&v_full[(j + 1) & 1], static_cast<uint32_t>((j + 1) >> 1) & 1u, abort_p, kBwdWaitTimeoutNs);
        __syncwarp();
        named_bar_arrive(kBwdBarGo, kBwdPair);
        named_bar_sync(kBwdBarAck, kBwdPair);
      }
      if (j + 2 < n_j) {
        if (lane == 0 && !*abort_p)
          mbar_wait(&k_full[(j + 2) % 3], static_cast<uint32_t>((j + 2) / 3) & 1u, abort_p, kBwdWaitTimeoutNs);
        __syncwarp();
        named_bar_arrive(kBwdBarGo, kBwdPair);
        named_bar_sync(kBwdBarAck, kBwdPair);
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer (the whole warp runs the loop for the named barriers; lane 0 issues) ----------------
    // S(j) goes to region j & 1 and dP(j) always to [256, 384); phase 2 writes dS(j) inside S(j)'s
    // region. Once phase 2 of block j is done: dP(j + 1) (phase 2 of block j + 1 waits for it
    // first), dQ(j) += dS(j) K(j), and S(j + 2) into S(j)'s region after dQ(j) has read it (the
    // tensor pipe runs one thread's MMAs in issue order). S(j + 1) was issued a block earlier, so
    // phase 1 of block j + 1 starts at once and the tensor pipe has work during phase 2.
    const uint64_t aQ = make_sdesc_sw128(smem_u32(sQ), 16, 1024), aDO = make_sdesc_sw128(smem_u32(sDO), 16, 1024);
    // K(j): K-major for S, MN-major (LBO one box) as the B operand of dQ; V(j): K-major for dP
    const uint64_t k_k0 = make_sdesc_sw128(smem_u32(smem + 2 * Cfg::kTileBytes), 16, 1024);
    const uint64_t k_mn0 = make_sdesc_sw128(smem_u32(smem + 2 * Cfg::kTileBytes), Cfg::kBoxBytes, 1024);
    auto aK_of = [&](int j) { return sdesc_at(k_k0, (j % 3) * Cfg::kTileBytes); };
    auto bK_of = [&](int j) { return sdesc_at(k_mn0, (j % 3) * Cfg::kTileBytes); };
    auto aV_of = [&](int j) { return sdesc_at(k_k0, (3 + (j & 1)) * Cfg::kTileBytes); };
    auto issue_s = [&](int j) {
      tc_fence_after();
      bwd_mma_scores<D>(tmem + (j & 1) * 128, aQ, aK_of(j));  // S(j) = Q K^T
      umma_commit(&s_ready[j & 1]);
    };
    auto issue_dp = [&](int j) {
      tc_fence_after();
      bwd_mma_scores<D>(tmem + Cfg::kTmDp, aDO, aV_of(j));  // dP(j) = dO V^T
      umma_commit(&dp_ready);
      umma_commit(&v_empty[j & 1]);
    };
    // Q, dO, K(0), V(0), K(1): the issuing thread's own waits, once per CTA. After a failed wait (or an
    // abort) the handoffs below still run to the end; only the MMAs are skipped.
    bool ok = true;
    if (lane == 0 && n_j > 0) {
      ok = mbar_wait(&qd_full, 0, abort_p, kBwdWaitTimeoutNs) && mbar_wait(&k_full[0], 0, abort_p, kBwdWaitTimeoutNs);
      if (ok) issue_s(0);
      ok = ok && mbar_wait(&v_full[0], 0, abort_p, kBwdWaitTimeoutNs);
      if (ok) issue_dp(0);
      if (ok && n_j > 1) {
        ok = mbar_wait(&k_full[1], 0, abort_p, kBwdWaitTimeoutNs);
        if (ok) issue_s(1);
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
    for (int j = 0; j < n_j; ++j) {
      __syncwarp();
      named_bar_sync(kBwdBarP, kBwdComputeAndMma);  // dS(j) is in TMEM, dP(j) consumed
      if (j + 1 < n_j) {
        named_bar_sync(kBwdBarGo, kBwdPair);  // V(j + 1) is in shared memory
        named_bar_arrive(kBwdBarAck, kBwdPair);
        if (lane == 0 && ok) issue_dp(j + 1);
      }
      if (lane == 0 && ok) {
        tc_fence_after();
        bwd_mma_accumulate_split<D>(tmem + Cfg::kTmDq, tmem + (j & 1) * 128, 0, bK_of(j), j > 0);  // dQ += dS K
        umma_commit(&k_empty[j % 3]);
      }
      if (j + 2 < n_j) {
        __syncwarp();
        named_bar_sync(kBwdBarGo, kBwdPair);  // K(j + 2) is in shared memory
        named_bar_arrive(kBwdBarAck, kBwdPair);
        if (lane == 0 && ok) issue_s(j + 2);
      }
    }
    if (lane == 0) umma_commit(&acc_done);
    __syncwarp();
  } else {
    // ---------------- compute warps: query row i0 + (t & 127) (TMEM lane), key half t >> 7 ----------------
    const int t = threadIdx.x;
    const int row = t & 127, half = t >> 7;
    const int q = i0 + row;
    const bool q_ok = q < p.Tq;
    const size_t r = (static_cast<size_t>(b) * p.Hq + h) * p.Tq + (q_ok ? q : 0);
    const float lse2 = q_ok ? p.lse[r] * kLog2e : INFINITY;  // rows past Tq: P = 0
    const float dl = q_ok ? p.delta[r] : 0.f;
    const float2 c2 = make_float2(p.c, p.c), nl2 = make_float2(-lse2, -lse2), ndl2 = make_float2(-dl, -dl);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t r_d = tmem + lane_off + Cfg::kTmDp;
    bool ok = true;
    for (int j = 0; j < n_j; ++j) {
      const uint32_t r_s = tmem + lane_off + (j & 1) * 128;
      // every key of the block is visible to every row of the query block: no mask
      const bool unmasked = (j + 1) * 128 <= p.Tk && (!p.causal || j * 128 + 127 <= i0);
      float pv[64];  // this thread's 64 probabilities, kept between the two phases
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s_ready[j & 1], static_cast<uint32_t>(j >> 1) & 1u, abort_p,
                                                      kBwdWaitTimeoutNs));
      if (ok) {
        tc_fence_after();
        // phase 1: P from S alone (this half's 64 keys in two chunks of 32)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int k0 = half * 64 + cc * 32;
          uint32_t sr[32];
          tmem_ld32(r_s + k0, sr);
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2, nl2);
            pv[cc * 32 + k] = ex2_approx(x.x);
            pv[cc * 32 + k + 1] = ex2_approx(x.y);
          }
          if (!unmasked) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int key = j * 128 + k0 + k;
              if (!(key < p.Tk && (!p.causal || key <= q))) pv[cc * 32 + k] = 0.f;
            }
          }
        }
      }
      if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&dp_ready, static_cast<uint32_t>(j) & 1u, abort_p,
                                                      kBwdWaitTimeoutNs));
      if (ok) {
        tc_fence_after();
        // phase 2: dS = P (dP - D) as bf16 pairs into [64 half + 16 cc, + 16) of S's region
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int k0 = half * 64 + cc * 32;
          uint32_t dr[32];
          tmem_ld32(r_d + k0, dr);
          uint32_t dd[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 g = __fmul2_rn(make_float2(pv[cc * 32 + 2 * k], pv[cc * 32 + 2 * k + 1]),
                                        __fadd2_rn(make_float2(__uint_as_float(dr[2 * k]), __uint_as_float(dr[2 * k + 1])), ndl2));
            dd[k] = pack_bf16x2(g.x, g.y);
          }
          tmem_st16(r_s + half * 64 + cc * 16, dd);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      named_bar_arrive(kBwdBarP, kBwdComputeAndMma);  // dS(j) is in TMEM (every block, also after a failed wait)
    }
    if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(&acc_done, 0, abort_p, kBwdWaitTimeoutNs));
    tc_fence_after();
    bwd_store_row<D>(tmem + lane_off + Cfg::kTmDq, p.scale, ok && n_j > 0, q_ok && (ok || n_j == 0),
                     p.dq + ((static_cast<size_t>(b) * p.Hq + h) * p.Tq + q) * D, half, p.out_v8 != 0);
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
template <int D>
static cudaError_t launch_bwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                const CUtensorMap& mdo, const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                float* delta, const BwdParams& p, cudaStream_t stream, int* launched) {
  using Cfg = BwdCfg<D>;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.Tq;
  bwd_delta_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(o, dout, delta, rows);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  *launched = 1;
  err = cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  const dim3 g_kv((p.Tk + 127) / 128, p.B * p.Hkv);
  bwd_dkdv_kernel<D><<<g_kv, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(mq, mk, mv, mdo, p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  *launched = 2;
  const dim3 g_q((p.Tq + 127) / 128, p.B * p.Hq);
  bwd_dq_kernel<D><<<g_q, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(mq, mk, mv, mdo, p);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  *launched = 3;
  return cudaSuccess;
}

cudaError_t launch_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Tq, int Tk,
                            int d, int causal, float scale, void* workspace, cudaStream_t stream, int* launched) {
  *launched = 0;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_bf16_tile_map(&mq, q, d, Tq, B * Hq) || !encode_bf16_tile_map(&mk, k, d, Tk, B * Hkv) ||
      !encode_bf16_tile_map(&mv, v, d, Tk, B * Hkv) || !encode_bf16_tile_map(&mdo, dout, d, Tq, B * Hq))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.lse = lse;
  p.delta = static_cast<float*>(workspace);
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  // rows are d * 2 bytes apart (a multiple of 32): every row is 32-byte aligned iff its array is
  p.out_v8 = ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) %
                  32 == 0)
                 ? 1
                 : 0;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Tq = Tq;
  p.Tk = Tk;
  p.g = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.c = scale * kLog2e;
  p.scale = scale;
  const __nv_bfloat16* ob = static_cast<const __nv_bfloat16*>(o);
  const __nv_bfloat16* db = static_cast<const __nv_bfloat16*>(dout);
  float* delta = static_cast<float*>(workspace);
  return d == 64 ? launch_bwd_d<64>(mq, mk, mv, mdo, ob, db, delta, p, stream, launched)
                 : launch_bwd_d<128>(mq, mk, mv, mdo, ob, db, delta, p, stream, launched);
}

uint32_t backward_take_device_error() { return take_device_error_word(); }

}  // namespace gb300
