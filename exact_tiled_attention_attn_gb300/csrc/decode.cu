// decode.cu - flash-decoding for one query token per sequence (sm_103a).
//
// "Attention from the kernel's side: FlashAttention, online softmax and fused
// dequantisation", section "Prefill and decoding are different problems":
// decoding streams the whole KV cache once per step at about 1 FLOP per byte,
// so it runs at memory speed; with grouped-query attention each K/V tile is
// loaded once and used by the g query heads of its group; flash-decoding
// splits the key sequence across thread blocks, each block computes a partial
// (m, l, o), and a last step merges the partials with the same rescaling rule
// as the online softmax ("Module 07: Fused operators and FlashAttention",
// section "Online softmax: derivation", the Step).
//
// Kernel 1 (split): one CTA per (split, K/V head, block of <= 4 query heads of
// its group, sequence). One producer thread streams the split's K and V rows
// into a ring of shared-memory stages with bulk asynchronous copies (each stage
// = 64 contiguous rows, completing on an mbarrier); four consumer warps read
// the stages with 16-byte shared loads (d/8 lanes per row, packed fp32x2 FMAs,
// a shuffle reduction per head), keep a running (m, l, o) per query
// head in registers, merge them at the end and write one fp32 partial per
// (sequence, head, split). The exponent base only moves when a block maximum
// exceeds it by more than 2^8, as in the prefill kernel: the normalised result
// does not depend on the base.
// Kernel 2 (combine): one CTA per (sequence, query head) merges the partials
// of the non-empty splits in split order and writes O (bf16) and LSE.
//
// Scores are kept in the base-2 domain: q is pre-multiplied by
// c = scale * log2(e), so p = 2^(c*s - m); LSE = (m + log2 l) * ln 2.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda_fp16.h>

#include "common.cuh"

namespace gb300 {

constexpr uint64_t kDecodeWaitTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr float kDecodeRescaleThreshold = 8.0f;           // log2 of the allowed growth of p
constexpr int kDecodeMaxHeadsPerCta = 4;                  // query heads one CTA keeps in registers

// EB = bytes per cached element: 2 for the bf16 cache, 1 for the E4M3 (FP8) cache.
// STAGES = shared-memory stages of K and V per CTA.
template <int D, int EB = 2, int STAGES = 2>
struct DecodeCfg {
  static constexpr int kLanesPerTok = D / 8;           // one chunk of 8 elements (8 * EB bytes) per lane
  static constexpr int kChunks = 1;                    // 16-byte chunks per lane per row
  static constexpr int kElems = 8 * kChunks;           // row elements per lane
  static constexpr int kTokPerPass = 32 / kLanesPerTok;
  static constexpr int kConsumerWarps = 4;
  static constexpr int kTile = 64;                     // rows (tokens) per stage; at d = 128 each lane
                                                       // group takes R = 8 of them per stage
  static constexpr int kStages = STAGES;               // FFMA kernel: two stages per CTA, three CTAs per SM
  static constexpr int kTokPerWarp = kTile / kConsumerWarps;
  static constexpr int kPasses = kTokPerWarp / kTokPerPass;
  static constexpr int kRowBytes = D * EB;
  static constexpr int kTileBytes = kTile * kRowBytes;
  static constexpr int kThreads = 32 * (kConsumerWarps + 1);
  static constexpr int kSmemBytes = kStages * 2 * kTileBytes + 1024;
};

struct DecodeParams {
  const __nv_bfloat16* q;
  const uint8_t* kc;       // [B, Hkv, Lcap, D] elements of EB bytes
  const uint8_t* vc;
  const float* k_scale;    // [B, Hkv] dequantisation scales of an E4M3 cache (nullptr for bf16)
  const float* v_scale;
  const int* seqlens;
  float* o_part;   // [B, Hq, S, D]
  float* ml_part;  // [B, Hq, S, 2]
  int Hq, Hkv, g, Lcap, S, C;
  int n_hblk;      // CTAs per K/V head (query heads of a group split in blocks of <= 4)
  int hblk;        // query heads per CTA
  float c;         // scale * log2(e)
};

// Two E4M3 codes (the low byte is the element at the lower address) -> two floats. The
// conversion to f16 is exact (every E4M3 value is an f16 value), and so is f16 -> f32.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two_codes & 0xFFFFu)));
  float lo, hi;
  asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(static_cast<unsigned short>(h2 & 0xFFFFu)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(static_cast<unsigned short>(h2 >> 16)));
  return make_float2(lo, hi);
}

// Lane layout inside a consumer warp: lane = grp * (D/8) + sub. The D/8 lanes of group
// grp share one key row per pass; lane sub holds the elements 8 sub .. 8 sub + 7 of the
// row (16 bytes of bf16 or 8 bytes of E4M3), so the lanes of a group read the row
// contiguously.
template <int D, int EB>
__device__ __forceinline__ void load_row_chunks(const uint8_t* row, int sub, float (&f)[DecodeCfg<D, EB>::kElems]) {
  static_assert(DecodeCfg<D, EB>::kChunks == 1, "one chunk of 8 elements per lane");
  if constexpr (EB == 2) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + sub * 16);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = bf16lo_to_f32(u[e]);
      f[2 * e + 1] = bf16hi_to_f32(u[e]);
    }
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(row + sub * 8);
    const uint32_t u[2] = {v.x, v.y};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const float2 a = e4m3x2_to_float2(u[w]);
      const float2 b = e4m3x2_to_float2(u[w] >> 16);
      f[4 * w] = a.x;
      f[4 * w + 1] = a.y;
      f[4 * w + 2] = b.x;
      f[4 * w + 3] = b.y;
    }
  }
}

// 3 CTAs per SM (registers capped at 136; the widest instances spill ~70 bytes, which costs less
// than the latency hiding of a third CTA gains)
template <int D, int G, int EB>
__global__ void __launch_bounds__(DecodeCfg<D, EB>::kThreads, 3)
    decode_split_kernel(const DecodeParams p) {
  using Cfg = DecodeCfg<D, EB>;
  constexpr int E = Cfg::kElems;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;                                       // [stages][tile][D] elements
  uint8_t* sV = smem + Cfg::kStages * Cfg::kTileBytes;      // [stages][tile][D] elements
  __shared__ uint64_t full_bar[Cfg::kStages];
  __shared__ uint64_t empty_bar[Cfg::kStages];
  __shared__ int abort_flag;

  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.n_hblk;
  const int hb = blockIdx.y % p.n_hblk;
  const int b = blockIdx.z;
  const int h0 = kvh * p.g + hb * p.hblk;                   // first query head of this CTA
  const int nh = min(p.hblk, (kvh + 1) * p.g - h0);         // heads of this CTA (<= G)
  int L = p.seqlens[b];
  L = L < 0 ? 0 : (L > p.Lcap ? p.Lcap : L);
  const int start = split * p.C;
  if (start >= L) return;  // empty split: the combine kernel never reads it
  const int end = min(start + p.C, L);
  const int ntiles = (end - start + Cfg::kTile - 1) / Cfg::kTile;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], Cfg::kConsumerWarps);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_p = &abort_flag;

  const size_t head_off = (static_cast<size_t>(b) * p.Hkv + kvh) * p.Lcap;  // in rows
  const uint8_t* kbase = p.kc + head_off * Cfg::kRowBytes;
  const uint8_t* vbase = p.vc + head_off * Cfg::kRowBytes;

  if (warp == Cfg::kConsumerWarps) {
    // ---------------- producer: one thread issues the bulk copies ----------------
    if (lane == 0) {
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % Cfg::kStages;
        const uint32_t ph = static_cast<uint32_t>(t / Cfg::kStages) & 1u;
        if (!mbar_wait(&empty_bar[s], ph ^ 1u, abort_p, kDecodeWaitTimeoutNs)) break;
        const int row0 = start + t * Cfg::kTile;
        const int nrows = min(Cfg::kTile, end - row0);
        const uint32_t bytes = static_cast<uint32_t>(nrows) * Cfg::kRowBytes;
        mbar_arrive_expect_tx(&full_bar[s], 2 * bytes);
        bulk_copy_g2s(sK + s * Cfg::kTileBytes, kbase + static_cast<size_t>(row0) * Cfg::kRowBytes, bytes, &full_bar[s]);
        bulk_copy_g2s(sV + s * Cfg::kTileBytes, vbase + static_cast<size_t>(row0) * Cfg::kRowBytes, bytes, &full_bar[s]);
        issued = t + 1;
      }
      // Let every copy this thread issued land before the CTA can exit.
      for (int t = max(0, issued - Cfg::kStages); t < issued; ++t) {
        const int s = t % Cfg::kStages;
        mbar_wait(&full_bar[s], static_cast<uint32_t>(t / Cfg::kStages) & 1u, abort_p, kDecodeWaitTimeoutNs);
      }
    }
    __syncwarp();
    __syncthreads();
    return;
  }

  // ---------------- consumers ----------------
  const int grp = lane / Cfg::kLanesPerTok;  // which row of a pass
  const int sub = lane % Cfg::kLanesPerTok;  // which chunk of the row

  // q is pre-multiplied by c = scale * log2(e) and, for an E4M3 cache, by the keys'
  // dequantisation scale, so the scores come out of the raw codes' values directly
  const float qmul = p.c * (p.k_scale != nullptr ? p.k_scale[static_cast<size_t>(b) * p.Hkv + kvh] : 1.f);
  float qf[G][E];
#pragma unroll
  for (int gh = 0; gh < G; ++gh) {
    const bool have = gh < nh;
    const __nv_bfloat16* qrow = p.q + (static_cast<size_t>(b) * p.Hq + (have ? h0 + gh : h0)) * D;
#pragma unroll
    for (int ch = 0; ch < Cfg::kChunks; ++ch) {
      const uint4 qv = *reinterpret_cast<const uint4*>(qrow + (sub + 8 * ch) * 8);
      const uint32_t u[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qf[gh][ch * 8 + 2 * e] = have ? bf16lo_to_f32(u[e]) * qmul : 0.f;
        qf[gh][ch * 8 + 2 * e + 1] = have ? bf16hi_to_f32(u[e]) * qmul : 0.f;
      }
    }
  }
  float m[G], l[G], o[G][E];
#pragma unroll
  for (int gh = 0; gh < G; ++gh) {
    m[gh] = -INFINITY;
    l[gh] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[gh][e] = 0.f;
  }

  // Each lane group (LPR = D/8 lanes) takes R consecutive rows of the warp's share of a
  // tile. Every lane computes its 8-element partial dot product for all R rows, then a
  // transpose-reduce over the group (each shuffle step halves the rows a lane keeps)
  // leaves the full score of row `my_row` in LPR/R lanes. The softmax runs once per row
  // owner; l is accumulated per lane (duplicated over the LPR/R owners) and reduced at the
  // end; p is broadcast back to the group for the P.V update, which every lane does for
  // its 8 output elements.
  constexpr int LPR = Cfg::kLanesPerTok;
  constexpr int R = Cfg::kTokPerWarp / Cfg::kTokPerPass;   // rows per group per tile
  constexpr int kRowLanes = LPR / R;                        // lanes holding one row's score
  static_assert(R >= 1 && (R & (R - 1)) == 0 && kRowLanes >= 1, "rows per group must be a power of two");
  int my_row = 0;  // row (0..R-1) whose score this lane ends up holding
#pragma unroll
  for (int off = LPR / 2, cnt = R / 2; cnt >= 1; off >>= 1, cnt >>= 1)
    if (sub & off) my_row += cnt;
  const int grp_lane0 = lane - sub;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % Cfg::kStages;
    if (!mbar_wait(&full_bar[s], static_cast<uint32_t>(t / Cfg::kStages) & 1u, abort_p, kDecodeWaitTimeoutNs))
      break;
    const uint8_t* kt = sK + s * Cfg::kTileBytes;
    const uint8_t* vt = sV + s * Cfg::kTileBytes;
    const int row0 = start + t * Cfg::kTile;
    const int tok0 = warp * Cfg::kTokPerWarp + grp * R;  // first row of this group in the tile

    // partial dot products of (c q) with this lane's 8 elements of each of the R rows, taken
    // in the order u ^ my_row: then at every step of the transpose-reduce below a lane keeps
    // the first half of what it holds and sends the second half
    float part[R][G];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      float kf[E];
      load_row_chunks<D, EB>(kt + (tok0 + (u ^ my_row)) * Cfg::kRowBytes, sub, kf);  // rows past `end`: masked below
#pragma unroll
      for (int gh = 0; gh < G; ++gh) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < E; e += 2)
          acc = __ffma2_rn(make_float2(qf[gh][e], qf[gh][e + 1]), make_float2(kf[e], kf[e + 1]), acc);
        part[u][gh] = acc.x + acc.y;
      }
    }
    // transpose-reduce: at lane distance `off` a lane keeps part[0 .. cnt) and receives its
    // partner's partial sums for the same rows (the partner's row order differs in that bit)
#pragma unroll
    for (int off = LPR / 2, cnt = R / 2; cnt >= 1; off >>= 1, cnt >>= 1) {
#pragma unroll
      for (int j = 0; j < cnt; ++j) {
#pragma unroll
        for (int gh = 0; gh < G; ++gh) part[j][gh] += __shfl_xor_sync(0xFFFFFFFFu, part[j + cnt][gh], off);
      }
    }
    // the lanes that share a row finish its sum
#pragma unroll
    for (int off = kRowLanes / 2; off >= 1; off >>= 1)
#pragma unroll
      for (int gh = 0; gh < G; ++gh) part[0][gh] += __shfl_xor_sync(0xFFFFFFFFu, part[0][gh], off);

    const bool my_valid = row0 + tok0 + my_row < end;
    // running (m, l) per head, uniform over the group; the base only moves when a score
    // exceeds it by more than 2^8, and only then is the block maximum over the group's rows
    // formed (with shuffles); otherwise p = 2^(s - m) <= 2^8 with the base unchanged
    float sc[G], pw[G], corr[G];
    bool need = false;
#pragma unroll
    for (int gh = 0; gh < G; ++gh) {
      sc[gh] = my_valid ? part[0][gh] : -INFINITY;
      need |= sc[gh] > m[gh] + kDecodeRescaleThreshold;
      corr[gh] = 1.f;
    }
    const bool grow_any = __any_sync(0xFFFFFFFFu, need);
    if (grow_any) {
#pragma unroll
      for (int gh = 0; gh < G; ++gh) {
        float mt = sc[gh];
#pragma unroll
        for (int off = LPR / 2; off >= kRowLanes; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, off));
        const float m_cand = fmaxf(m[gh], mt);
        if (m_cand > m[gh] + kDecodeRescaleThreshold) {
          corr[gh] = ex2_approx(m[gh] - m_cand);  // 0 when m was -inf
          m[gh] = m_cand;
        }
      }
    }
#pragma unroll
    for (int gh = 0; gh < G; ++gh) {
      const float base = (m[gh] == -INFINITY) ? 0.f : m[gh];
      pw[gh] = ex2_approx(sc[gh] - base);
      l[gh] = l[gh] * corr[gh] + pw[gh];
    }
    if (grow_any) {
#pragma unroll
      for (int gh = 0; gh < G; ++gh) {
        const float2 c2 = make_float2(corr[gh], corr[gh]);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 r = __fmul2_rn(make_float2(o[gh][e], o[gh][e + 1]), c2);
          o[gh][e] = r.x;
          o[gh][e + 1] = r.y;
        }
      }
    }
    // o += p v over the group's rows (p of row u comes from its owner lanes)
#pragma unroll
    for (int u = 0; u < R; ++u) {
      float pu[G];
#pragma unroll
      for (int gh = 0; gh < G; ++gh)
        pu[gh] = __shfl_sync(0xFFFFFFFFu, pw[gh], grp_lane0 + u * kRowLanes + (sub % kRowLanes));
      if (row0 + tok0 + u < end) {
        float vf[E];
        load_row_chunks<D, EB>(vt + (tok0 + u) * Cfg::kRowBytes, sub, vf);
#pragma unroll
        for (int gh = 0; gh < G; ++gh) {
          const float2 p2 = make_float2(pu[gh], pu[gh]);
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            const float2 r = __ffma2_rn(p2, make_float2(vf[e], vf[e + 1]), make_float2(o[gh][e], o[gh][e + 1]));
            o[gh][e] = r.x;
            o[gh][e + 1] = r.y;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
  }
  __syncwarp();

  // l: each lane summed the p of its own rows; add the group's distinct rows (the lanes
  // that differ in the row-selecting bits), so every lane of the group holds the group's l
#pragma unroll
  for (int off = LPR / 2; off >= kRowLanes; off >>= 1)
#pragma unroll
    for (int gh = 0; gh < G; ++gh) l[gh] += __shfl_xor_sync(0xFFFFFFFFu, l[gh], off);

  // merge the lane groups of this warp (same chunks `sub`, different rows)
#pragma unroll
  for (int off = Cfg::kLanesPerTok; off < 32; off <<= 1) {
#pragma unroll
    for (int gh = 0; gh < G; ++gh) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m[gh], off);
      const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l[gh], off);
      const float mn = fmaxf(m[gh], m2);
      const float base = (mn == -INFINITY) ? 0.f : mn;
      const float w1 = ex2_approx(m[gh] - base);
      const float w2 = ex2_approx(m2 - base);
      l[gh] = l[gh] * w1 + l2 * w2;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float o2 = __shfl_xor_sync(0xFFFFFFFFu, o[gh][e], off);
        o[gh][e] = o[gh][e] * w1 + o2 * w2;
      }
      m[gh] = mn;
    }
  }

  // merge the consumer warps through shared memory (the stages are free now)
  named_bar_sync(1, 32 * Cfg::kConsumerWarps);
  float* red = reinterpret_cast<float*>(smem);  // [warps][G][D + 2]
  constexpr int kRow = D + 2;
  if (grp == 0) {
#pragma unroll
    for (int gh = 0; gh < G; ++gh) {
      float* r = red + (warp * G + gh) * kRow;
#pragma unroll
      for (int ch = 0; ch < Cfg::kChunks; ++ch)
#pragma unroll
        for (int e = 0; e < 8; ++e) r[(sub + 8 * ch) * 8 + e] = o[gh][ch * 8 + e];
      if (sub == 0) {
        r[D] = m[gh];
        r[D + 1] = l[gh];
      }
    }
  }
  named_bar_sync(1, 32 * Cfg::kConsumerWarps);
  // the values' dequantisation scale multiplies the weighted sum once, here
  const float vmul = p.v_scale != nullptr ? p.v_scale[static_cast<size_t>(b) * p.Hkv + kvh] : 1.f;
  for (int idx = threadIdx.x; idx < nh * D; idx += 32 * Cfg::kConsumerWarps) {
    const int gh = idx / D;
    const int e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < Cfg::kConsumerWarps; ++w) M = fmaxf(M, red[(w * G + gh) * kRow + D]);
    const float base = (M == -INFINITY) ? 0.f : M;
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < Cfg::kConsumerWarps; ++w) {
      const float* r = red + (w * G + gh) * kRow;
      const float wt = ex2_approx(r[D] - base);
      acc += wt * r[e];
      lsum += wt * r[D + 1];
    }
    const size_t slot = (static_cast<size_t>(b) * p.Hq + h0 + gh) * p.S + split;
    p.o_part[slot * D + e] = acc * vmul;
    if (e == 0) {
      p.ml_part[slot * 2] = M;
      p.ml_part[slot * 2 + 1] = lsum;
    }
  }
  __syncthreads();
  // this CTA's partials are written: the combine grid (launched with programmatic stream
  // serialisation) may be scheduled once every CTA got here or exited; it still waits for
  // this grid's completion before reading them (griddepcontrol.wait)
  asm volatile("griddepcontrol.launch_dependents;");
}

// ---------------------------------------------------------------------------------------
// Split kernel on warp-level tensor-core MMAs (mma.sync m16n8k16, fp32 accumulation).
//
// Same CTA, producer, stages and partial format as decode_split_kernel; the consumers differ.
// Per element the FFMA kernel above spends ~4 issue slots: its dot products are repeated for
// every query head of the CTA and a shuffle tree reduces them; with an E4M3 cache each element
// also needs two conversions. Both products of the step are small dense contractions (the
// CTA's query heads against 64 keys of d elements), so here each consumer warp takes 16 keys
// of a stage and runs them through the tensor core:
//   S = Q K^T   A = Q (16 rows, the CTA's heads in rows 0..nh-1, the rest zero), B = K^T of
//               8 keys, fp32 accumulators; the d axis is permuted so each thread reads one
//               contiguous piece of its key row (a dot product does not depend on the order of
//               its terms, as long as Q and K use the same one);
//   O += P V    A = P, taken straight from S's accumulator layout (rows = heads, keys 2c,
//               2c+1 and 8+2c, 8+2c+1 of thread c), B = V of 16 keys x 8 output columns; the
//               output columns are permuted so each thread reads a contiguous piece of 4 rows.
// bf16 cache: K and V feed the MMA as they are (bf16 x bf16); P is rounded to bf16, as in the
// prefill. E4M3 cache: codes become f16 pairs (exact; cvt.rn.f16x2.e4m3x2), q becomes f16
// (exact for |q| in f16's normal range), P is rounded to f16. Scores leave the MMA unscaled and
// are multiplied by c = scale * log2(e) (and the keys' dequantisation scale) in fp32.
__device__ __forceinline__ void mma_16816_bf16(float (&d)[2], const uint32_t a0, const uint32_t a2, uint32_t b0,
                                               uint32_t b1) {
  // rows 8..15 of A are zero, so d2 and d3 stay zero: they are not kept
  [[maybe_unused]] float z2, z3;  // outputs of the instruction, unused
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %10, %10};"
      : "+f"(d[0]), "+f"(d[1]), "=f"(z2), "=f"(z3)
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void mma_16816_f16(float (&d)[2], const uint32_t a0, const uint32_t a2, uint32_t b0,
                                              uint32_t b1) {
  [[maybe_unused]] float z2, z3;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %10, %10};"
      : "+f"(d[0]), "+f"(d[1]), "=f"(z2), "=f"(z3)
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
}
template <int EB>
__device__ __forceinline__ void mma_16816(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  if constexpr (EB == 2) mma_16816_bf16(d, a0, a2, b0, b1);
  else mma_16816_f16(d, a0, a2, b0, b1);
}
// two E4M3 codes (bits 0-15 of w, the lower byte first) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(w & 0xFFFFu)));
  return h2;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---- the tensor-core consumer's building blocks (shared by the split and balanced kernels)

// Q of this thread's head (row gq of the MMA's A operand; a zero row when the CTA has fewer
// heads) as A fragments: for MMA kk, the k-slots (2c, 2c+1) and (2c+8, 2c+9) hold the elements
// QE c + 4 kk + (0, 1) and QE c + 4 kk + (2, 3) of the head's row (an E4M3 cache: as f16).
template <int D, int EB>
__device__ __forceinline__ void mma_load_q(const __nv_bfloat16* qrow_head, bool head_ok, int c,
                                           uint32_t (&qa)[D / 16][2]) {
  constexpr int QE = D / 4;
  const uint4* qrow = reinterpret_cast<const uint4*>(qrow_head + QE * c);
#pragma unroll
  for (int i = 0; i < QE / 8; ++i) {
    const uint4 v = qrow[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t x = head_ok ? w[e] : 0u;
      if constexpr (EB == 1) x = pack_f16x2(bf16lo_to_f32(x), bf16hi_to_f32(x));
      qa[(4 * i + e) >> 1][e & 1] = x;
    }
  }
}

// One consumer warp's block of 16 keys (rows of kt / vt, kRowBytes apart; rows at or past
// nvalid are masked): S = Q K^T, the online-softmax update of (m, l) and O += P V.
//  * S: key 8 nt + gq of the block is this thread's column; the d axis is permuted so that the
//    thread's k-slots of every MMA lie in one contiguous quarter of its key row (the dot
//    product does not depend on the order of its terms when Q and K use the same one).
//  * The base only moves when a score exceeds it by more than 2^8; then the block maximum is
//    formed (two xor shuffles within the 4 threads of a head).
//  * O: B of MMA j holds V rows (2c, 2c+1) and (2c+8, 2c+9) of the block at output column
//    VE gq + j; P is reused from the S accumulators (the FA-2 register reuse).
template <int D, int EB, int kRowBytes>
__device__ __forceinline__ void mma_decode_block(const uint8_t* kt, const uint8_t* vt, int nvalid,
                                                 const uint32_t (&qa)[D / 16][2], float cmul, int gq, int c,
                                                 float& m, float& l, float (&o)[D / 8][2]) {
  constexpr int NJ = D / 8;
  constexpr int QE = D / 4;
  constexpr int KW = QE * EB / 4;
  constexpr int VE = D / 8;
  constexpr int VW = VE * EB / 4;
  float sc[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const uint4* krow = reinterpret_cast<const uint4*>(kt + (8 * nt + gq) * kRowBytes + QE * EB * c);
    float acc[2] = {0.f, 0.f};
    // one 16-byte piece at a time: 2 MMAs of bf16, 4 of E4M3 codes
#pragma unroll
    for (int i = 0; i < KW / 4; ++i) {
      const uint4 v = krow[i];
      const uint32_t kw[4] = {v.x, v.y, v.z, v.w};
      if constexpr (EB == 2) {
#pragma unroll
        for (int h = 0; h < 2; ++h) mma_16816<EB>(acc, qa[2 * i + h][0], qa[2 * i + h][1], kw[2 * h], kw[2 * h + 1]);
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h)
          mma_16816<EB>(acc, qa[4 * i + h][0], qa[4 * i + h][1], e4m3x2_to_f16x2(kw[h]), e4m3x2_to_f16x2(kw[h] >> 16));
      }
    }
    // keys 8 nt + 2c and 8 nt + 2c + 1 of the block, base-2 scaled; keys past the end: -inf
    sc[nt][0] = (8 * nt + 2 * c < nvalid) ? acc[0] * cmul : -INFINITY;
    sc[nt][1] = (8 * nt + 2 * c + 1 < nvalid) ? acc[1] * cmul : -INFINITY;
  }

  const float mx = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
  float corr = 1.f;
  if (__any_sync(0xFFFFFFFFu, mx > m + kDecodeRescaleThreshold)) {
    float mt = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 2));
    const float m_cand = fmaxf(m, mt);
    if (m_cand > m + kDecodeRescaleThreshold) {
      corr = ex2_approx(m - m_cand);  // 0 when m was -inf
      m = m_cand;
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      o[j][0] *= corr;
      o[j][1] *= corr;
    }
  }
  const float base = (m == -INFINITY) ? 0.f : m;
  float pw[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    pw[nt][0] = ex2_approx(sc[nt][0] - base);
    pw[nt][1] = ex2_approx(sc[nt][1] - base);
  }
  l = l * corr + ((pw[0][0] + pw[0][1]) + (pw[1][0] + pw[1][1]));
  const uint32_t pa0 = (EB == 2) ? pack_bf16x2(pw[0][0], pw[0][1]) : pack_f16x2(pw[0][0], pw[0][1]);
  const uint32_t pa2 = (EB == 2) ? pack_bf16x2(pw[1][0], pw[1][1]) : pack_f16x2(pw[1][0], pw[1][1]);

  // Rows past the end are zeroed (their shared memory may hold anything, and 0 * NaN would
  // not be 0). In halves of the output columns (16-byte pieces of the four rows), to keep
  // registers low.
  constexpr int kHalves = (VW >= 8) ? 2 : 1;
  constexpr int HW = VW / kHalves;  // 32-bit words of a row per half
  constexpr int HJ = NJ / kHalves;  // MMAs per half
#pragma unroll
  for (int hf = 0; hf < kHalves; ++hf) {
    uint32_t vw[4][HW];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = 2 * c + (r & 1) + 8 * (r >> 1);
      const bool ok = row < nvalid;
      const uint8_t* vrow = vt + row * kRowBytes + VE * EB * gq + hf * HW * 4;
      if constexpr (HW >= 4) {
#pragma unroll
        for (int i = 0; i < HW / 4; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(vrow + i * 16);
          vw[r][4 * i] = ok ? v.x : 0u;
          vw[r][4 * i + 1] = ok ? v.y : 0u;
          vw[r][4 * i + 2] = ok ? v.z : 0u;
          vw[r][4 * i + 3] = ok ? v.w : 0u;
        }
      } else {
        const uint2 v = *reinterpret_cast<const uint2*>(vrow);
        vw[r][0] = ok ? v.x : 0u;
        vw[r][1] = ok ? v.y : 0u;
      }
    }
#pragma unroll
    for (int jj = 0; jj < HJ; ++jj) {
      const int j = hf * HJ + jj;
      uint32_t b0, b1;
      if constexpr (EB == 2) {
        // element j of rows (2c, 2c+1) into one register, likewise rows (2c+8, 2c+9)
        const uint32_t sel = (jj & 1) ? 0x7632u : 0x5410u;
        b0 = __byte_perm(vw[0][jj >> 1], vw[1][jj >> 1], sel);
        b1 = __byte_perm(vw[2][jj >> 1], vw[3][jj >> 1], sel);
      } else {
        // codes j of rows (2c, 2c+1) -> one f16 pair, likewise rows (2c+8, 2c+9)
        const uint32_t sel = (jj & 2) ? 0x7362u : 0x5140u;
        const uint32_t w01 = __byte_perm(vw[0][jj >> 2], vw[1][jj >> 2], sel);
        const uint32_t w23 = __byte_perm(vw[2][jj >> 2], vw[3][jj >> 2], sel);
        b0 = e4m3x2_to_f16x2((jj & 1) ? (w01 >> 16) : w01);
        b1 = e4m3x2_to_f16x2((jj & 1) ? (w23 >> 16) : w23);
      }
      mma_16816<EB>(o[j], pa0, pa2, b0, b1);
    }
  }
}

// Two CTAs per SM (at d = 128 this kernel needs ~168 registers per thread) and 3 stages of 64
// rows, 6 for the 1-byte rows of an E4M3 cache at d = 128 (96 KB of K and V per CTA, as with
// bf16 rows). Measured on the B16 Hq32 Hkv8 L ~ U[8192, 32768] decode: E4M3 d = 128, 6 stages
// 5205 GB/s against 5090 with 3; E4M3 d = 64, 12 stages 4008 against 4481 with 3; bf16 d = 64,
// 6 stages no faster than 3.
constexpr int kMmaCtasPerSm = 2;
template <int D, int EB>
__host__ __device__ constexpr int mma_stages() {
  return (EB == 1 && D == 128) ? 6 : 3;
}

template <int D, int EB>
__global__ void __launch_bounds__(DecodeCfg<D, EB, mma_stages<D, EB>()>::kThreads, kMmaCtasPerSm)
    decode_split_mma_kernel(const DecodeParams p) {
  using Cfg = DecodeCfg<D, EB, mma_stages<D, EB>()>;
  static_assert(Cfg::kTile == 16 * Cfg::kConsumerWarps, "one 16-key block per consumer warp per stage");
  constexpr int NJ = D / 8;           // MMAs along the output columns for O
  constexpr int VE = D / 8;           // elements of a value row one thread holds per output MMA
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + Cfg::kStages * Cfg::kTileBytes;
  __shared__ uint64_t full_bar[Cfg::kStages];
  __shared__ uint64_t empty_bar[Cfg::kStages];
  __shared__ int abort_flag;

  const int split = blockIdx.x;
  const int kvh = blockIdx.y / p.n_hblk;
  const int hb = blockIdx.y % p.n_hblk;
  const int b = blockIdx.z;
  const int h0 = kvh * p.g + hb * p.hblk;
  const int nh = min(p.hblk, (kvh + 1) * p.g - h0);
  int L = p.seqlens[b];
  L = L < 0 ? 0 : (L > p.Lcap ? p.Lcap : L);
  const int start = split * p.C;
  if (start >= L) return;  // empty split: the combine kernel never reads it
  const int end = min(start + p.C, L);
  const int ntiles = (end - start + Cfg::kTile - 1) / Cfg::kTile;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], Cfg::kConsumerWarps);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_p = &abort_flag;
  const size_t head_off = (static_cast<size_t>(b) * p.Hkv + kvh) * p.Lcap;
  const uint8_t* kbase = p.kc + head_off * Cfg::kRowBytes;
  const uint8_t* vbase = p.vc + head_off * Cfg::kRowBytes;

  if (warp == Cfg::kConsumerWarps) {
    if (lane == 0) {
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % Cfg::kStages;
        const uint32_t ph = static_cast<uint32_t>(t / Cfg::kStages) & 1u;
        if (!mbar_wait(&empty_bar[s], ph ^ 1u, abort_p, kDecodeWaitTimeoutNs)) break;
        const int row0 = start + t * Cfg::kTile;
        const int nrows = min(Cfg::kTile, end - row0);
        const uint32_t bytes = static_cast<uint32_t>(nrows) * Cfg::kRowBytes;
        mbar_arrive_expect_tx(&full_bar[s], 2 * bytes);
        bulk_copy_g2s(sK + s * Cfg::kTileBytes, kbase + static_cast<size_t>(row0) * Cfg::kRowBytes, bytes, &full_bar[s]);
        bulk_copy_g2s(sV + s * Cfg::kTileBytes, vbase + static_cast<size_t>(row0) * Cfg::kRowBytes, bytes, &full_bar[s]);
        issued = t + 1;
      }
      for (int t = max(0, issued - Cfg::kStages); t < issued; ++t) {
        const int s = t % Cfg::kStages;
        mbar_wait(&full_bar[s], static_cast<uint32_t>(t / Cfg::kStages) & 1u, abort_p, kDecodeWaitTimeoutNs);
      }
    }
    __syncwarp();
    __syncthreads();
    return;
  }

  // ---------------- consumers ----------------
  const int gq = lane >> 2;  // MMA row group: the query head (rows of A, P, O); the key / column of B
  const int c = lane & 3;    // position in the group
  const bool head_ok = gq < nh;
  uint32_t qa[D / 16][2];
  mma_load_q<D, EB>(p.q + (static_cast<size_t>(b) * p.Hq + (head_ok ? h0 + gq : h0)) * D, head_ok, c, qa);
  const float cmul = p.c * (p.k_scale != nullptr ? p.k_scale[static_cast<size_t>(b) * p.Hkv + kvh] : 1.f);
  float m = -INFINITY, l = 0.f;
  float o[NJ][2];
#pragma unroll
  for (int j = 0; j < NJ; ++j) o[j][0] = o[j][1] = 0.f;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % Cfg::kStages;
    if (!mbar_wait(&full_bar[s], static_cast<uint32_t>(t / Cfg::kStages) & 1u, abort_p, kDecodeWaitTimeoutNs))
      break;
    const uint8_t* kt = sK + s * Cfg::kTileBytes + warp * 16 * Cfg::kRowBytes;
    const uint8_t* vt = sV + s * Cfg::kTileBytes + warp * 16 * Cfg::kRowBytes;
    const int key0 = start + t * Cfg::kTile + warp * 16;  // first key of this warp's block
    mma_decode_block<D, EB, Cfg::kRowBytes>(kt, vt, end - key0, qa, cmul, gq, c, m, l, o);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
  }
  __syncwarp();

  // l: the 4 threads of a group hold disjoint keys' sums
  l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
  l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);

  // merge the consumer warps through shared memory (the stages are free now). This thread holds
  // O[head gq][VE (2c + e) + j] in o[j][e].
  named_bar_sync(1, 32 * Cfg::kConsumerWarps);
  float* red = reinterpret_cast<float*>(smem);  // [warps][8 heads][D + 2]
  constexpr int kRow = D + 2;
  {
    float* r = red + (warp * 8 + gq) * kRow;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      r[VE * (2 * c) + j] = o[j][0];
      r[VE * (2 * c + 1) + j] = o[j][1];
    }
    if (c == 0) {
      r[D] = m;
      r[D + 1] = l;
    }
  }
  named_bar_sync(1, 32 * Cfg::kConsumerWarps);
  const float vmul = p.v_scale != nullptr ? p.v_scale[static_cast<size_t>(b) * p.Hkv + kvh] : 1.f;
  for (int idx = threadIdx.x; idx < nh * D; idx += 32 * Cfg::kConsumerWarps) {
    const int gh = idx / D;
    const int e = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < Cfg::kConsumerWarps; ++w) M = fmaxf(M, red[(w * 8 + gh) * kRow + D]);
    const float base = (M == -INFINITY) ? 0.f : M;
    float acc = 0.f, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < Cfg::kConsumerWarps; ++w) {
      const float* r = red + (w * 8 + gh) * kRow;
      const float wt = ex2_approx(r[D] - base);
      acc += wt * r[e];
      lsum += wt * r[D + 1];
    }
    const size_t slot = (static_cast<size_t>(b) * p.Hq + h0 + gh) * p.S + split;
    p.o_part[slot * D + e] = acc * vmul;
    if (e == 0) {
      p.ml_part[slot * 2] = M;
      p.ml_part[slot * 2 + 1] = lsum;
    }
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;");
}

// ---------------------------------------------------------------------------------------
// Balanced schedule (num_splits = 0).
//
// The split kernel gives every (split, head block, sequence) a CTA of its own. With
// sequences of different lengths the CTAs differ in work, and the last ones run on a few SMs
// while the others idle (globaltimer traces of every CTA: B16 Hq32 Hkv8 d128 with
// L ~ U[8192, 32768] and 32 splits, the SMs fell idle from 184 us on and the kernel ended at
// 205 us; with L ~ U[1024, 2048] and 2 splits it ended at 26 us against 15 us of average work
// per SM). Here a persistent grid of kMmaCtasPerSm CTAs per SM divides the concatenated key
// stream of all (sequence, head block) segments, in 64-key tiles, into equal ranges, one per
// CTA (a stream-K partition: CTA c takes tiles [c NT / G, (c + 1) NT / G)). A CTA walks the
// pieces of its range in order: a segment that lies wholly in the range is finished there
// (O and LSE written, as the flash-decoding merge of one split); a segment cut by a range
// boundary leaves one partial (m, l, o) per piece in the workspace, which the merge kernel
// combines. Only a CTA's first piece can start inside a segment and only its last can end
// inside one, so each CTA needs two partial slots: slot 2c for a piece that ends inside its
// segment, slot 2c + 1 for one that starts inside its segment and runs to the end.
// ---------------------------------------------------------------------------------------
constexpr int kBalancedMaxB = 1024;  // sequences whose tile prefix sums fit the CTA's shared array

struct BalancedParams {
  const __nv_bfloat16* q;
  const uint8_t* kc;  // [B, Hkv, Lcap, D] elements of EB bytes
  const uint8_t* vc;
  const float* k_scale;  // [B, Hkv] scales of an E4M3 cache (nullptr for bf16)
  const float* v_scale;
  const int* seqlens;
  __nv_bfloat16* o;  // [B, Hq, D]
  float* lse;        // [B, Hq] or nullptr
  float* part;       // [2 G slots][kDecodeMaxHeadsPerCta heads][D + 2]: o, then m and l
  int* tile_pre;     // [kBalancedMaxB + 1]: the tile prefix sums of the lengths, for the merge
  int B, Hq, Hkv, g, n_hblk, hblk, Lcap;
  int Y;             // segments per sequence: Hkv * n_hblk (head blocks)
  int G;             // CTAs of the balanced kernel
  float c;           // scale * log2(e)
};

__device__ __forceinline__ int seq_len_clamped(const int* seqlens, int b, int Lcap) {
  const int L = seqlens[b];
  return L < 0 ? 0 : (L > Lcap ? Lcap : L);
}

// The partition of the NT tiles over the CTAs: equal ranges over Geff = min(G, NT) CTAs, so
// that none below Geff is empty (floor(c NT / Geff) strictly increases when NT >= Geff); CTAs
// from Geff on have no work, and no empty range lies between two CTAs that share a segment.
// (A second phase of smaller ranges for CTAs started later, meant to absorb the CTAs' speed
// differences, was slower: the GPU does not start a grid's CTAs in index order, so some
// large-range CTAs started after small ones; B16 Hq32 Hkv8 d128, L ~ U[8192, 32768]: 242 us
// against 183 us back to back.)
struct BalancedPartition {
  int NT, Geff;
  __device__ __forceinline__ BalancedPartition(int nt, int g) : NT(nt), Geff(nt < g ? nt : g) {}
  // tiles [lo, hi) of CTA c (lo == hi: no work)
  __device__ __forceinline__ void range(int c, int& lo, int& hi) const {
    lo = hi = 0;
    if (c < Geff) {
      lo = static_cast<int>(static_cast<long long>(c) * NT / Geff);
      hi = static_cast<int>(static_cast<long long>(c + 1) * NT / Geff);
    }
  }
  // the CTA whose range holds tile t (0 <= t < NT): the largest c with floor(c NT / Geff) <= t
  __device__ __forceinline__ int cta_of(int t) const {
    return static_cast<int>((static_cast<long long>(t + 1) * Geff + NT - 1) / NT - 1);
  }
};

// pre[b] = tiles of sequences 0..b-1 (pre[0] = 0), for b = 0..B, in shared memory; every
// thread of the CTA takes part. Tiles are of kTile keys.
template <int kTile>
__device__ __forceinline__ void balanced_prefix(const BalancedParams& p, int* pre) {
  for (int b = threadIdx.x; b < p.B; b += blockDim.x)
    pre[b + 1] = (seq_len_clamped(p.seqlens, b, p.Lcap) + kTile - 1) / kTile;
  if (threadIdx.x == 0) pre[0] = 0;
  __syncthreads();
  if (threadIdx.x < 32) {  // inclusive scan of pre[1..B] by warp 0, 32 entries at a time
    int carry = 0;
    for (int b0 = 1; b0 <= p.B; b0 += 32) {
      const int i = b0 + static_cast<int>(threadIdx.x);
      int v = i <= p.B ? pre[i] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (static_cast<int>(threadIdx.x) >= off) v += u;
      }
      if (i <= p.B) pre[i] = v + carry;
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
  }
  __syncthreads();
}

// One piece of a CTA's range: tiles [t0, t1) of segment (b, y), which covers tiles
// [seg0, seg0 + n) of the stream; the piece's first tile is tile t0 - seg0 of the segment.
struct DecodePiece {
  int t0, t1, seg0;
  int b, y, n;
};

// The piece that starts at tile t (< NT) and ends at min(hi, end of t's segment).
// (Tile indices fit in an int: the host checks Y * B * ceil(Lcap / 64) < 2^31.)
__device__ __forceinline__ DecodePiece balanced_piece(const BalancedParams& p, const int* pre, int t, int hi) {
  // the largest b with Y pre[b] <= t: its segment row holds t (sequences without tiles are skipped)
  int lo_b = 0, hi_b = p.B;  // invariant: Y pre[lo_b] <= t < Y pre[hi_b]
  while (hi_b - lo_b > 1) {
    const int mid = (lo_b + hi_b) >> 1;
    if (p.Y * pre[mid] <= t) lo_b = mid;
    else hi_b = mid;
  }
  DecodePiece pc;
  pc.b = lo_b;
  pc.n = pre[lo_b + 1] - pre[lo_b];
  const int row0 = p.Y * pre[lo_b];
  pc.y = (t - row0) / pc.n;
  pc.seg0 = row0 + pc.y * pc.n;
  pc.t0 = t;
  pc.t1 = min(hi, pc.seg0 + pc.n);
  return pc;
}

// Stages of the balanced kernel: 3 for a bf16 cache, 96 KB of K and V for an E4M3 cache (6 at
// d = 128, 12 at d = 64). Its CTAs live for the whole kernel, so the deep ring costs no per-CTA
// set-up. Measured on B16 Hq32 Hkv8 L ~ U[8192, 32768]: E4M3 d = 64, 12 stages 67.0 us back to
// back against 71.5 with 3; bf16 d = 64, 6 stages 104.8 against 100.6 with 3.
template <int D, int EB>
__host__ __device__ constexpr int balanced_stages() {
  return EB == 1 ? (96 * 1024) / (2 * 64 * D) : 3;
}

template <int D, int EB>
__global__ void __launch_bounds__(DecodeCfg<D, EB, balanced_stages<D, EB>()>::kThreads, kMmaCtasPerSm)
    decode_balanced_kernel(const BalancedParams p) {
  using Cfg = DecodeCfg<D, EB, balanced_stages<D, EB>()>;
  static_assert(Cfg::kTile == 16 * Cfg::kConsumerWarps, "one 16-key block per consumer warp per stage");
  constexpr int NJ = D / 8;
  constexpr int VE = D / 8;
  constexpr int kRed = D + 2;  // reduction row: o, m, l
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + Cfg::kStages * Cfg::kTileBytes;
  float* red = reinterpret_cast<float*>(smem + 2 * Cfg::kStages * Cfg::kTileBytes);  // [warps][4 heads][kRed]
  __shared__ uint64_t full_bar[Cfg::kStages];
  __shared__ uint64_t empty_bar[Cfg::kStages];
  __shared__ int abort_flag;
  __shared__ int pre[kBalancedMaxB + 1];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], Cfg::kConsumerWarps);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  // the previous kernel's writes (the cache, q, the lengths) are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  balanced_prefix<Cfg::kTile>(p, pre);  // ends with __syncthreads
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b <= p.B; b += blockDim.x) p.tile_pre[b] = pre[b];
  volatile int* abort_p = &abort_flag;
  int lo, hi;
  BalancedPartition(p.Y * pre[p.B], p.G).range(static_cast<int>(blockIdx.x), lo, hi);

  if (warp == Cfg::kConsumerWarps) {
    // ---------------- producer: every tile of every piece, in order ----------------
    if (lane == 0) {
      int T = 0;  // tiles issued by this CTA
      bool alive = true;
      for (int t = lo; alive && t < hi;) {
        const DecodePiece pc = balanced_piece(p, pre, t, hi);
        const int L = seq_len_clamped(p.seqlens, pc.b, p.Lcap);
        const int kvh = pc.y / p.n_hblk;
        const size_t head_off = (static_cast<size_t>(pc.b) * p.Hkv + kvh) * p.Lcap;
        const uint8_t* kbase = p.kc + head_off * Cfg::kRowBytes;
        const uint8_t* vbase = p.vc + head_off * Cfg::kRowBytes;
        for (int i = pc.t0; i < pc.t1; ++i, ++T) {
          const int s = T % Cfg::kStages;
          if (!mbar_wait(&empty_bar[s], (static_cast<uint32_t>(T / Cfg::kStages) & 1u) ^ 1u, abort_p,
                         kDecodeWaitTimeoutNs)) {
            alive = false;
            break;
          }
          const int row0 = (i - pc.seg0) * Cfg::kTile;
          const int nrows = min(Cfg::kTile, L - row0);
          const uint32_t bytes = static_cast<uint32_t>(nrows) * Cfg::kRowBytes;
          mbar_arrive_expect_tx(&full_bar[s], 2 * bytes);
          bulk_copy_g2s(sK + s * Cfg::kTileBytes, kbase + static_cast<size_t>(row0) * Cfg::kRowBytes, bytes,
                        &full_bar[s]);
          bulk_copy_g2s(sV + s * Cfg::kTileBytes, vbase + static_cast<size_t>(row0) * Cfg::kRowBytes, bytes,
                        &full_bar[s]);
        }
        t = pc.t1;
      }
      // the last copies land before the CTA may exit
      for (int u = max(0, T - Cfg::kStages); u < T; ++u)
        mbar_wait(&full_bar[u % Cfg::kStages], static_cast<uint32_t>(u / Cfg::kStages) & 1u, abort_p,
                  kDecodeWaitTimeoutNs);
    }
    __syncwarp();
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;");
    return;
  }

  // ---------------- consumers ----------------
  const int gq = lane >> 2;  // MMA row group: the query head
  const int c = lane & 3;
  int T = 0;  // tiles consumed by this CTA
  for (int t = lo; t < hi;) {
    int ntl, rem;  // tiles of the piece; keys of the sequence from this warp's first key on
    float cmul;
    uint32_t qa[D / 16][2];
    {
      const DecodePiece pc = balanced_piece(p, pre, t, hi);
      const int L = seq_len_clamped(p.seqlens, pc.b, p.Lcap);
      const int kvh = pc.y / p.n_hblk;
      const int h0 = kvh * p.g + (pc.y % p.n_hblk) * p.hblk;
      const bool head_ok = gq < min(p.hblk, (kvh + 1) * p.g - h0);
      mma_load_q<D, EB>(p.q + (static_cast<size_t>(pc.b) * p.Hq + (head_ok ? h0 + gq : h0)) * D, head_ok, c, qa);
      cmul = p.c * (p.k_scale != nullptr ? p.k_scale[static_cast<size_t>(pc.b) * p.Hkv + kvh] : 1.f);
      ntl = pc.t1 - pc.t0;
      rem = L - ((pc.t0 - pc.seg0) * Cfg::kTile + warp * 16);
    }
    float m = -INFINITY, l = 0.f;
    float o[NJ][2];
#pragma unroll
    for (int j = 0; j < NJ; ++j) o[j][0] = o[j][1] = 0.f;
    for (int k = 0; k < ntl; ++k, ++T, rem -= Cfg::kTile) {
      const int s = T % Cfg::kStages;
      // after a failed wait (the abort flag is set) every later wait fails at once; the warps
      // still meet at each named barrier below, so the CTA runs to its end
      if (!mbar_wait(&full_bar[s], static_cast<uint32_t>(T / Cfg::kStages) & 1u, abort_p, kDecodeWaitTimeoutNs))
        break;
      {
        const uint8_t* kt = sK + s * Cfg::kTileBytes + warp * 16 * Cfg::kRowBytes;
        const uint8_t* vt = sV + s * Cfg::kTileBytes + warp * 16 * Cfg::kRowBytes;
        mma_decode_block<D, EB, Cfg::kRowBytes>(kt, vt, rem, qa, cmul, gq, c, m, l, o);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    // l: the 4 threads of a group hold disjoint keys' sums
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);

    // the piece again (cheaper than keeping it in registers through the tile loop)
    const DecodePiece pc = balanced_piece(p, pre, t, hi);
    t = pc.t1;
    const int kvh = pc.y / p.n_hblk;
    const int h0 = kvh * p.g + (pc.y % p.n_hblk) * p.hblk;
    const int nh = min(p.hblk, (kvh + 1) * p.g - h0);
    // merge the consumer warps (the area is free: every warp read the previous piece's rows
    // before it reached this barrier)
    named_bar_sync(1, 32 * Cfg::kConsumerWarps);
    if (gq < nh) {
      float* r = red + (warp * kDecodeMaxHeadsPerCta + gq) * kRed;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        r[VE * (2 * c) + j] = o[j][0];
        r[VE * (2 * c + 1) + j] = o[j][1];
      }
      if (c == 0) {
        r[D] = m;
        r[D + 1] = l;
      }
    }
    named_bar_sync(1, 32 * Cfg::kConsumerWarps);
    const bool to_end = pc.t1 == pc.seg0 + pc.n;
    const bool whole = pc.t0 == pc.seg0 && to_end;
    // slot 2c: the piece ends inside its segment; 2c + 1: it starts inside and runs to the end
    const int slot = 2 * static_cast<int>(blockIdx.x) + (to_end ? 1 : 0);
    const float vmul = p.v_scale != nullptr ? p.v_scale[static_cast<size_t>(pc.b) * p.Hkv + kvh] : 1.f;
    for (int idx = threadIdx.x; idx < nh * D; idx += 32 * Cfg::kConsumerWarps) {
      const int gh = idx / D;
      const int e = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < Cfg::kConsumerWarps; ++w) M = fmaxf(M, red[(w * kDecodeMaxHeadsPerCta + gh) * kRed + D]);
      const float base = (M == -INFINITY) ? 0.f : M;
      float acc = 0.f, lsum = 0.f;
#pragma unroll
      for (int w = 0; w < Cfg::kConsumerWarps; ++w) {
        const float* r = red + (w * kDecodeMaxHeadsPerCta + gh) * kRed;
        const float wt = ex2_approx(r[D] - base);
        acc += wt * r[e];
        lsum += wt * r[D + 1];
      }
      if (whole) {
        const size_t row = static_cast<size_t>(pc.b) * p.Hq + h0 + gh;
        p.o[row * D + e] = __float2bfloat16_rn(acc * vmul / lsum);
        if (e == 0 && p.lse != nullptr) p.lse[row] = (M + log2f(lsum)) * 0.69314718055994530942f;
      } else {
        float* dst = p.part + (static_cast<size_t>(slot) * kDecodeMaxHeadsPerCta + gh) * kRed;
        dst[e] = acc * vmul;
        if (e == 0) {
          dst[D] = M;
          dst[D + 1] = lsum;
        }
      }
    }
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;");
}

// Merge of the segments that the balanced kernel cut: one CTA of D/64 warps per (sequence,
// query head), as decode_combine_kernel. A segment held by CTAs c_first < c_last has the
// partials of slots 2c (c_first <= c < c_last) and 2 c_last + 1, merged in CTA order; a
// segment inside one CTA was finished there; a sequence without keys gets O = 0 and
// LSE = -inf. Every CTA between c_first and c_last holds a piece of the segment (no range
// between them is empty, see BalancedPartition). Launched as a programmatic dependent of the
// balanced kernel.
template <int D>
__global__ void __launch_bounds__(D / 2) decode_balanced_merge_kernel(const BalancedParams p) {
  constexpr int kGroup = 32;
  constexpr int kRed = D + 2;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int bh = blockIdx.x;
  const int b = bh / p.Hq;
  const int h = bh % p.Hq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the balanced kernel's tile prefix sums (its CTA 0 stored them)
  const int before = p.tile_pre[b];
  const int total = p.tile_pre[p.B];
  const int e0 = warp * 64 + 2 * lane;
  __nv_bfloat16* orow = p.o + static_cast<size_t>(bh) * D + e0;
  const int n = p.tile_pre[b + 1] - before;
  if (n == 0) {  // no key: O = 0, LSE = -inf
    *reinterpret_cast<uint32_t*>(orow) = 0u;
    if (threadIdx.x == 0 && p.lse != nullptr) p.lse[bh] = -INFINITY;
    return;
  }
  const int kvh = h / p.g;
  const int within = h % p.g;
  const int y = kvh * p.n_hblk + within / p.hblk;
  const int gh = within % p.hblk;
  const BalancedPartition part(p.Y * total, p.G);  // NT >= n >= 1
  const int seg0 = p.Y * before + y * n;
  const int c_first = part.cta_of(seg0);
  const int c_last = part.cta_of(seg0 + n - 1);
  if (c_first == c_last) return;  // finished by its CTA
  const int np = c_last - c_first + 1;
  auto slot_of = [&](int k) { return (k < np - 1) ? 2 * (c_first + k) : 2 * c_last + 1; };
  float M = -INFINITY, lsum = 0.f;
  float2 acc = make_float2(0.f, 0.f);
  for (int g0 = 0; g0 < np; g0 += kGroup) {
    const int cnt = min(kGroup, np - g0);
    float2 mlv = make_float2(-INFINITY, 0.f);
    if (lane < cnt) {
      const float* r = p.part + (static_cast<size_t>(slot_of(g0 + lane)) * kDecodeMaxHeadsPerCta + gh) * kRed;
      mlv = make_float2(r[D], r[D + 1]);
    }
    float2 v[kGroup];
#pragma unroll
    for (int t = 0; t < kGroup; ++t) {
      v[t] = make_float2(0.f, 0.f);
      if (t < cnt)
        v[t] = *reinterpret_cast<const float2*>(
            p.part + (static_cast<size_t>(slot_of(g0 + t)) * kDecodeMaxHeadsPerCta + gh) * kRed + e0);
    }
    float mg = mlv.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xFFFFFFFFu, mg, off));
    const float M_new = fmaxf(M, mg);
    const float w = lane < cnt ? ex2_approx(mlv.x - M_new) : 0.f;
    float lp = w * mlv.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lp += __shfl_xor_sync(0xFFFFFFFFu, lp, off);
    const float r = ex2_approx(M - M_new);  // 0 on the first group (M = -inf)
    float2 a = make_float2(acc.x * r, acc.y * r);
#pragma unroll
    for (int t = 0; t < kGroup; ++t) {
      const float wt = __shfl_sync(0xFFFFFFFFu, w, t);
      if (t < cnt) {
        a.x = fmaf(wt, v[t].x, a.x);
        a.y = fmaf(wt, v[t].y, a.y);
      }
    }
    acc = a;
    lsum = fmaf(lsum, r, lp);
    M = M_new;
  }
  *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(acc.x / lsum, acc.y / lsum);
  if (threadIdx.x == 0 && p.lse != nullptr) p.lse[bh] = (M + log2f(lsum)) * 0.69314718055994530942f;
}

// One CTA of D/64 warps per (sequence, query head); warp w owns output elements [64 w, 64 w + 64),
// two per lane. The partials of up to 32 splits are loaded in one go, together with the sequence
// length: a split past the length was never written and is dropped by predicate (its bytes are
// inside the workspace, so reading them is harmless), which puts every load of a group in flight
// before the first result is needed. The splits are merged in split order (lane t of the warp
// owns split g0 + t's weight); with more than 32 splits each group of 32 is merged into a running
// (M, l, o) by the same rescaling rule. The result is deterministic for a given split count.
template <int D>
__global__ void __launch_bounds__(D / 2) decode_combine_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ ml_part,
                                                              const int* __restrict__ seqlens,
                                                              __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                              int Hq, int S, int C, int Lcap) {
  constexpr int kGroup = 32;
  // launched as a programmatic dependent of the split kernel: wait until that grid has
  // completed and its writes are visible (a no-op without such a dependency)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int bh = blockIdx.x;
  const int b = bh / Hq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = warp * 64 + 2 * lane;
  const float* ml = ml_part + static_cast<size_t>(bh) * S * 2;
  const float* op = o_part + static_cast<size_t>(bh) * S * D + e0;
  const int L_raw = seqlens[b];
  float M = -INFINITY, lsum = 0.f;
  float2 acc = make_float2(0.f, 0.f);
  for (int g0 = 0; g0 < S; g0 += kGroup) {
    const int cnt = min(kGroup, S - g0);  // splits of this group inside the workspace
    float2 mlv = make_float2(-INFINITY, 0.f);
    if (lane < cnt) mlv = *reinterpret_cast<const float2*>(ml + 2 * (g0 + lane));
    float2 v[kGroup];
#pragma unroll
    for (int t = 0; t < kGroup; ++t)
      v[t] = t < cnt ? *reinterpret_cast<const float2*>(op + static_cast<size_t>(g0 + t) * D) : make_float2(0.f, 0.f);
    const int L = L_raw < 0 ? 0 : (L_raw > Lcap ? Lcap : L_raw);
    const int nsplit = min(S, (L + C - 1) / C);
    if (g0 >= nsplit) break;
    const int valid = min(kGroup, nsplit - g0);  // splits of this group that were written
    const bool mine = lane < valid;
    float mg = mine ? mlv.x : -INFINITY;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xFFFFFFFFu, mg, off));
    const float M_new = fmaxf(M, mg);
    if (M_new == -INFINITY) continue;  // nothing seen yet (every written split so far was empty)
    const float w = mine ? ex2_approx(mlv.x - M_new) : 0.f;
    float lp = w * (mine ? mlv.y : 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lp += __shfl_xor_sync(0xFFFFFFFFu, lp, off);
    const float r = ex2_approx(M - M_new);  // 0 on the first group (M = -inf)
    float2 a = make_float2(acc.x * r, acc.y * r);
#pragma unroll
    for (int t = 0; t < kGroup; ++t) {
      const float wt = __shfl_sync(0xFFFFFFFFu, w, t);
      if (t < valid) {
        a.x = fmaf(wt, v[t].x, a.x);
        a.y = fmaf(wt, v[t].y, a.y);
      }
    }
    acc = a;
    lsum = fmaf(lsum, r, lp);
    M = M_new;
  }
  __nv_bfloat16* orow = o + static_cast<size_t>(bh) * D + e0;
  if (M == -INFINITY) {  // no key: O = 0, LSE = -inf
    *reinterpret_cast<uint32_t*>(orow) = 0u;
    if (threadIdx.x == 0 && lse != nullptr) lse[bh] = -INFINITY;
    return;
  }
  *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(acc.x / lsum, acc.y / lsum);
  if (threadIdx.x == 0 && lse != nullptr) lse[bh] = (M + log2f(lsum)) * 0.69314718055994530942f;
}

template <int D, int G, int EB>
static cudaError_t launch_split(const DecodeParams& p, int B, cudaStream_t stream) {
  using Cfg = DecodeCfg<D, EB>;
  auto kern = decode_split_kernel<D, G, EB>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  const dim3 grid(p.S, p.Hkv * p.n_hblk, B);
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int EB>
static cudaError_t launch_split_g(const DecodeParams& p, int B, cudaStream_t stream) {
  switch (p.hblk) {
    case 1: return launch_split<D, 1, EB>(p, B, stream);
    case 2: return launch_split<D, 2, EB>(p, B, stream);
    case 3: return launch_split<D, 3, EB>(p, B, stream);
    case 4: return launch_split<D, 4, EB>(p, B, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int D, int EB>
static cudaError_t launch_split_mma(const DecodeParams& p, int B, cudaStream_t stream) {
  using Cfg = DecodeCfg<D, EB, mma_stages<D, EB>()>;
  auto kern = decode_split_mma_kernel<D, EB>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  const dim3 grid(p.S, p.Hkv * p.n_hblk, B);
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

// Streaming multiprocessors of the current device (queried once per device).
static int decode_sm_count() {
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

// Workspace of the balanced schedule on the current device: two partial slots per CTA, each
// kDecodeMaxHeadsPerCta rows of d + 2 floats, then the tile prefix sums (kBalancedMaxB + 1 ints).
static size_t balanced_slot_bytes(int sms, int d) {
  return static_cast<size_t>(2) * kMmaCtasPerSm * sms * kDecodeMaxHeadsPerCta * (static_cast<size_t>(d) + 2) *
         sizeof(float);
}
size_t decode_balanced_workspace_bytes(int d) {
  const int sms = decode_sm_count();
  if (sms <= 0) return 0;
  return balanced_slot_bytes(sms, d) + (kBalancedMaxB + 4) * sizeof(int);
}
int decode_balanced_max_batch() { return kBalancedMaxB; }

template <int D, int EB>
static cudaError_t launch_balanced(const BalancedParams& p, cudaStream_t stream, int* launched) {
  using Cfg = DecodeCfg<D, EB, balanced_stages<D, EB>()>;
  const int smem = 2 * Cfg::kStages * Cfg::kTileBytes + 1024 +
                   Cfg::kConsumerWarps * kDecodeMaxHeadsPerCta * (D + 2) * static_cast<int>(sizeof(float));
  auto kern = decode_balanced_kernel<D, EB>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  kern<<<p.G, Cfg::kThreads, smem, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  *launched = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B) * static_cast<unsigned>(p.Hq));
  cfg.blockDim = dim3(static_cast<unsigned>(D / 2));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, decode_balanced_merge_kernel<D>, p);
  if (err == cudaSuccess) err = cudaGetLastError();
  if (err == cudaSuccess) *launched = 2;
  return err;
}

// The balanced schedule (num_splits = 0): a persistent grid of kMmaCtasPerSm CTAs per SM.
static cudaError_t launch_decode_balanced(const void* q, const void* kc, const void* vc, const float* k_scale,
                                          const float* v_scale, const int* seqlens, void* o, float* lse, int B,
                                          int Hq, int Hkv, int d, int Lcap, float scale, void* workspace,
                                          cudaStream_t stream, int* launched) {
  const int sms = decode_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  if (B > kBalancedMaxB) return cudaErrorInvalidValue;
  BalancedParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kc = static_cast<const uint8_t*>(kc);
  p.vc = static_cast<const uint8_t*>(vc);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.seqlens = seqlens;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.part = static_cast<float*>(workspace);
  p.tile_pre = reinterpret_cast<int*>(static_cast<char*>(workspace) + balanced_slot_bytes(sms, d));
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.n_hblk = (p.g + kDecodeMaxHeadsPerCta - 1) / kDecodeMaxHeadsPerCta;
  p.hblk = (p.g + p.n_hblk - 1) / p.n_hblk;
  p.Lcap = Lcap;
  p.Y = Hkv * p.n_hblk;
  p.G = kMmaCtasPerSm * sms;
  p.c = scale * 1.4426950408889634f;
  const bool fp8 = k_scale != nullptr;
  if (fp8) return (d == 64) ? launch_balanced<64, 1>(p, stream, launched) : launch_balanced<128, 1>(p, stream, launched);
  return (d == 64) ? launch_balanced<64, 2>(p, stream, launched) : launch_balanced<128, 2>(p, stream, launched);
}

// The split kernel's consumers: tensor-core MMAs (decode_split_mma_kernel), unless the
// environment variable GB300_ATTN_DECODE is "ffma" (decode_split_kernel; the same result up to
// rounding).
static bool use_mma_split() {
  const char* e = std::getenv("GB300_ATTN_DECODE");
  return !(e != nullptr && std::strcmp(e, "ffma") == 0);
}

// Returns the number of kernels launched through *launched. k_scale/v_scale non-null
// selects the E4M3 cache (one byte per element), else the cache is bf16.
cudaError_t launch_decode(const void* q, const void* kc, const void* vc, const float* k_scale, const float* v_scale,
                          const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv, int d, int Lcap,
                          float scale, int S, int C, void* workspace, cudaStream_t stream, int* launched) {
  *launched = 0;
  if (S == 0)
    return launch_decode_balanced(q, kc, vc, k_scale, v_scale, seqlens, o, lse, B, Hq, Hkv, d, Lcap, scale, workspace,
                                  stream, launched);
  const bool fp8 = k_scale != nullptr;
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kc = static_cast<const uint8_t*>(kc);
  p.vc = static_cast<const uint8_t*>(vc);
  p.k_scale = fp8 ? k_scale : nullptr;
  p.v_scale = fp8 ? v_scale : nullptr;
  p.seqlens = seqlens;
  p.o_part = static_cast<float*>(workspace);
  p.ml_part = p.o_part + static_cast<size_t>(B) * Hq * S * d;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.n_hblk = (p.g + kDecodeMaxHeadsPerCta - 1) / kDecodeMaxHeadsPerCta;
  p.hblk = (p.g + p.n_hblk - 1) / p.n_hblk;
  p.Lcap = Lcap;
  p.S = S;
  p.C = C;
  p.c = scale * 1.4426950408889634f;
  if (static_cast<long long>(Hkv) * p.n_hblk > 65535) return cudaErrorInvalidValue;
  cudaError_t err;
  if (use_mma_split())
    err = fp8 ? ((d == 64) ? launch_split_mma<64, 1>(p, B, stream) : launch_split_mma<128, 1>(p, B, stream))
              : ((d == 64) ? launch_split_mma<64, 2>(p, B, stream) : launch_split_mma<128, 2>(p, B, stream));
  else
    err = fp8 ? ((d == 64) ? launch_split_g<64, 1>(p, B, stream) : launch_split_g<128, 1>(p, B, stream))
              : ((d == 64) ? launch_split_g<64, 2>(p, B, stream) : launch_split_g<128, 2>(p, B, stream));
  if (err != cudaSuccess) return err;
  *launched = 1;
  // The combine is launched with programmatic stream serialisation: its grid can be set up
  // while the split grid drains (launch overhead hidden), and griddepcontrol.wait in the
  // kernel orders its reads after the split kernel's writes.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(Hq));
  cfg.blockDim = dim3(static_cast<unsigned>(d / 2));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
  if (d == 64) {
    err = cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, static_cast<const float*>(p.o_part),
                             static_cast<const float*>(p.ml_part), seqlens, ob, lse, Hq, S, C, Lcap);
  } else {
    err = cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, static_cast<const float*>(p.o_part),
                             static_cast<const float*>(p.ml_part), seqlens, ob, lse, Hq, S, C, Lcap);
  }
  if (err != cudaSuccess) return err;
  err = cudaGetLastError();
  if (err == cudaSuccess) *launched = 2;
  return err;
}

uint32_t decode_take_device_error() { return take_device_error_word(); }

// ---------------------------------------------------------------------------------------
// Fixed scratch for attn_decode_noalloc.
//
// Some callers cannot allocate device memory at the moment they want to decode: an
// engine that has already handed (nearly) all of HBM to its KV-cache pool, code running
// under a custom allocator or a memory budget that forbids new allocations, or a caller
// that must not trigger an allocation (and the synchronisation cudaMalloc/cudaFree can
// imply) in the middle of its step. For them the split partials live in this file-scope
// device array instead of a caller-provided workspace. It is part of the module image:
// every GPU that loads this library holds these bytes until the process exits.
// Nothing in it needs to start at zero: each call's split kernel writes every partial
// that the same call's combine kernel reads. All calls share it, so two such calls that
// can run at the same time on the GPU (different streams, or different host threads)
// race on it and must be serialised by the caller.
// ---------------------------------------------------------------------------------------
constexpr size_t kDecodeNoAllocScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeNoAllocScratchBytes];

size_t decode_noalloc_capacity() { return kDecodeNoAllocScratchBytes; }

// Device address of g_decode_scratch on the current device. In host code the symbol is
// only a host-side stand-in, so its device address is looked up with that device current.
// Outside a stream capture it is looked up on every call (cheap once the module is loaded),
// so a device reset or a reloaded module never leaves a stale address behind; during a
// capture the address cached by the last lookup on that device is used, since the first
// lookup on a device may load this library's device code there. Neither path calls
// cudaMalloc.
cudaError_t decode_noalloc_scratch(cudaStream_t stream, void** ptr) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  err = cudaStreamIsCapturing(stream, &cap);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  if (cap == cudaStreamCaptureStatusNone || addr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (err != cudaSuccess) return err;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

}  // namespace gb300
