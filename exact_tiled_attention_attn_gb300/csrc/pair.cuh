// pair.cuh - inline-PTX helpers for kernels that run as clusters of two CTAs on two SMs and
// issue tcgen05 MMAs for the pair (cta_group::2): the A operand (and the accumulator) comes
// half from each CTA, 128 rows each; the B operand is split by its N columns between the
// two CTAs' shared memories; one thread of the even CTA issues for both.
//
// Every tcgen05 instruction of such a kernel uses cta_group::2 (allocation, MMA, commit,
// deallocation); loads and stores of TMEM (tcgen05.ld/st) stay per CTA.
#pragma once

#include "common.cuh"

namespace gb300 {

__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of both CTAs (every warp converged): orders everything before it in either CTA
// before everything after it in either CTA.
__device__ __forceinline__ void cluster_sync_all() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the object at shared::cta address `saddr` in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (this CTA's or the peer's), with
// the instruction's default (CTA-scope release) semantics. The data these arrivals announce
// is TMEM written by tcgen05.st (ordered by tcgen05.wait::st and tcgen05.fence before the
// arrival) and copies that complete on the barrier themselves. Measured on this part, the
// cluster-scope release form took ~0.6 us per arrival in a loaded kernel, this one ~0.13 us.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar_cl, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(bar_cl), "r"(bytes) : "memory");
}

// try_wait (default acquire semantics) with a suspend-time hint.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Write 1 into the int at shared::cluster address `cl` (the peer's abort flag).
__device__ __forceinline__ void st_cluster_one(uint32_t cl) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(cl), "r"(1) : "memory");
}

// Bounded wait for a pair: gives up after `timeout_ns` or once this CTA's abort flag is set
// (by this CTA or by the peer); on its own timeout it sets both CTAs' flags and the device
// error word, so the peer's waits give up too. Returns true when the phase completed.
__device__ __forceinline__ bool pair_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t peer_abort_cl,
                                          uint64_t timeout_ns) {
  if (mbar_try_wait_cluster(bar, parity, 0u)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity, 100000u)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort = 1;
      st_cluster_one(peer_abort_cl);
      report_device_error(kErrTimeout);
      return false;
    }
  }
}

// 3-D tiled TMA load into this CTA's shared memory whose completion (complete_tx) goes to the
// mbarrier at shared::cluster address `bar_cl`, which may be the peer CTA's.
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cl, int c0, int c1,
                                                 int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cl), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// TMEM allocation for the pair: one warp of each of the two CTAs executes it; each CTA gets
// the same columns of its own TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem, both CTAs] (+)= A[smem, 128 rows per CTA] * B[smem, N/2 columns per CTA]
__device__ __forceinline__ void umma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem, both CTAs] (+)= A[tmem, both CTAs] * B[smem, N/2 columns per CTA]
__device__ __forceinline__ void umma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at this shared::cta offset in every CTA of `cta_mask` when all
// tcgen05 operations this thread issued so far have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Shared-memory matrix descriptor with a chosen swizzle mode (2 = 128-byte, 4 = 64-byte); the
// other fields as in make_sdesc_sw128.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                               uint32_t swizzle_mode) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle_mode) << 61;
  return d;
}

// Host: a 3-D TMA map over a [Z, rows, D] bf16 tensor with a box of box_cols x box_rows x 1
// and the given swizzle (64 or 128 bytes); rows past the end read as zero (tmap.cu).
bool encode_bf16_box_map(CUtensorMap* map, const void* base, int D, int rows, int Z, int box_cols, int box_rows,
                         int swizzle_bytes);

}  // namespace gb300
