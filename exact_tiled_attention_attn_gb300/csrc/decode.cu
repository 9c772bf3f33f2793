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
// Kernel 1 (split): one CTA per (split, KV head, sequence). One producer
// thread streams the split's K and V rows into a ring of shared-memory stages
// with bulk asynchronous copies (each stage = TILE contiguous rows, completing
// on an mbarrier); four consumer warps read the stages with 16-byte shared
// loads, keep a running (m, l, o) per query head of the group in registers,
// merge them at the end and write one fp32 partial per (sequence, head, split).
// Kernel 2 (combine): one CTA per (sequence, query head) merges the partials
// of the non-empty splits in split order and writes O (bf16) and LSE.
//
// Scores are kept in the base-2 domain: q is pre-multiplied by
// c = scale * log2(e), so p = 2^(c*s - m); LSE = (m + log2 l) * ln 2.
#include <mutex>

#include "common.cuh"

namespace gb300 {

constexpr uint64_t kDecodeWaitTimeoutNs = 2000000000ull;  // 2 s per wait

template <int D>
struct DecodeCfg {
  static constexpr int kLanesPerTok = D / 8;          // 16-byte slice per lane
  static constexpr int kTokPerPass = 32 / kLanesPerTok;
  static constexpr int kConsumerWarps = 4;
  static constexpr int kTile = 32;                    // rows (tokens) per stage
  static constexpr int kStages = 4;
  static constexpr int kTokPerWarp = kTile / kConsumerWarps;
  static constexpr int kPasses = kTokPerWarp / kTokPerPass;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kThreads = 32 * (kConsumerWarps + 1);
  static constexpr int kSmemBytes = kStages * 2 * kTileBytes + 1024;
};

struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const int* seqlens;
  float* o_part;   // [B, Hq, S, D]
  float* ml_part;  // [B, Hq, S, 2]
  int Hq, Hkv, g, Lcap, S, C;
  float c;         // scale * log2(e)
};

template <int D, int G>
__global__ void __launch_bounds__(DecodeCfg<D>::kThreads)
    decode_split_kernel(const DecodeParams p) {
  using Cfg = DecodeCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;                                       // [stages][tile][D] bf16
  uint8_t* sV = smem + Cfg::kStages * Cfg::kTileBytes;      // [stages][tile][D] bf16
  __shared__ uint64_t full_bar[Cfg::kStages];
  __shared__ uint64_t empty_bar[Cfg::kStages];
  __shared__ int abort_flag;

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
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
  const __nv_bfloat16* kbase = p.kc + head_off * D;
  const __nv_bfloat16* vbase = p.vc + head_off * D;

  if (warp == Cfg::kConsumerWarps) {
    // ---------------- producer: one thread issues the bulk copies ----------------
    if (lane == 0) {
      for (int t = 0; t < ntiles; ++t) {
        const int s = t % Cfg::kStages;
        const uint32_t ph = static_cast<uint32_t>(t / Cfg::kStages) & 1u;
        if (!mbar_wait(&empty_bar[s], ph ^ 1u, abort_p, kDecodeWaitTimeoutNs)) break;
        const int row0 = start + t * Cfg::kTile;
        const int nrows = min(Cfg::kTile, end - row0);
        const uint32_t bytes = static_cast<uint32_t>(nrows) * D * 2;
        mbar_arrive_expect_tx(&full_bar[s], 2 * bytes);
        bulk_copy_g2s(sK + s * Cfg::kTileBytes, kbase + static_cast<size_t>(row0) * D, bytes, &full_bar[s]);
        bulk_copy_g2s(sV + s * Cfg::kTileBytes, vbase + static_cast<size_t>(row0) * D, bytes, &full_bar[s]);
      }
      // Let every copy this thread issued land before the CTA can exit.
      for (int t = max(0, ntiles - Cfg::kStages); t < ntiles; ++t) {
        const int s = t % Cfg::kStages;
        mbar_wait(&full_bar[s], static_cast<uint32_t>(t / Cfg::kStages) & 1u, abort_p, kDecodeWaitTimeoutNs);
      }
    }
    __syncwarp();
    __syncthreads();
    return;
  }

  // ---------------- consumers ----------------
  const int grp = lane / Cfg::kLanesPerTok;   // which token of a pass
  const int sub = lane % Cfg::kLanesPerTok;   // which 8-element slice of the row

  float qf[G][8];
#pragma unroll
  for (int gh = 0; gh < G; ++gh) {
    const int h = kvh * p.g + gh;
    const uint4 qv = *reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * p.Hq + h) * D + sub * 8);
    const uint32_t u[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qf[gh][2 * e] = bf16lo_to_f32(u[e]) * p.c;
      qf[gh][2 * e + 1] = bf16hi_to_f32(u[e]) * p.c;
    }
  }
  float m[G], l[G], o[G][8];
#pragma unroll
  for (int gh = 0; gh < G; ++gh) {
    m[gh] = -INFINITY;
    l[gh] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[gh][e] = 0.f;
  }

  for (int t = 0; t < ntiles; ++t) {
    const int s = t % Cfg::kStages;
    if (!mbar_wait(&full_bar[s], static_cast<uint32_t>(t / Cfg::kStages) & 1u, abort_p, kDecodeWaitTimeoutNs))
      break;
    const uint8_t* kt = sK + s * Cfg::kTileBytes;
    const uint8_t* vt = sV + s * Cfg::kTileBytes;
    const int row0 = start + t * Cfg::kTile;

    float sc[Cfg::kPasses][G];
#pragma unroll
    for (int u = 0; u < Cfg::kPasses; ++u) {
      const int tok = warp * Cfg::kTokPerWarp + u * Cfg::kTokPerPass + grp;
      const bool valid = row0 + tok < end;
      float kf[8];
      const uint4 kv = valid ? *reinterpret_cast<const uint4*>(kt + tok * D * 2 + sub * 16) : make_uint4(0, 0, 0, 0);
      const uint32_t ku[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kf[2 * e] = bf16lo_to_f32(ku[e]);
        kf[2 * e + 1] = bf16hi_to_f32(ku[e]);
      }
#pragma unroll
      for (int gh = 0; gh < G; ++gh) {
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) part = fmaf(qf[gh][e], kf[e], part);
#pragma unroll
        for (int off = Cfg::kLanesPerTok / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
        sc[u][gh] = valid ? part : -INFINITY;
      }
    }
    // block update of the running (m, l, o) of this lane group, per head
    float pw[Cfg::kPasses][G];
#pragma unroll
    for (int gh = 0; gh < G; ++gh) {
      float mt = sc[0][gh];
#pragma unroll
      for (int u = 1; u < Cfg::kPasses; ++u) mt = fmaxf(mt, sc[u][gh]);
      const float mn = fmaxf(m[gh], mt);
      const float base = (mn == -INFINITY) ? 0.f : mn;
      const float corr = ex2_approx(m[gh] - base);
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < Cfg::kPasses; ++u) {
        pw[u][gh] = ex2_approx(sc[u][gh] - base);
        sum += pw[u][gh];
      }
      l[gh] = l[gh] * corr + sum;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[gh][e] *= corr;
      m[gh] = mn;
    }
#pragma unroll
    for (int u = 0; u < Cfg::kPasses; ++u) {
      const int tok = warp * Cfg::kTokPerWarp + u * Cfg::kTokPerPass + grp;
      if (row0 + tok < end) {
        const uint4 vv = *reinterpret_cast<const uint4*>(vt + tok * D * 2 + sub * 16);
        const uint32_t vu[4] = {vv.x, vv.y, vv.z, vv.w};
        float vf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          vf[2 * e] = bf16lo_to_f32(vu[e]);
          vf[2 * e + 1] = bf16hi_to_f32(vu[e]);
        }
#pragma unroll
        for (int gh = 0; gh < G; ++gh) {
#pragma unroll
          for (int e = 0; e < 8; ++e) o[gh][e] = fmaf(pw[u][gh], vf[e], o[gh][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
  }
  __syncwarp();

  // merge the lane groups of this warp (same slice `sub`, different tokens)
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
      for (int e = 0; e < 8; ++e) {
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
      for (int e = 0; e < 8; ++e) r[sub * 8 + e] = o[gh][e];
      if (sub == 0) {
        r[D] = m[gh];
        r[D + 1] = l[gh];
      }
    }
  }
  named_bar_sync(1, 32 * Cfg::kConsumerWarps);
  for (int idx = threadIdx.x; idx < G * D; idx += 32 * Cfg::kConsumerWarps) {
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
    const int h = kvh * p.g + gh;
    const size_t slot = (static_cast<size_t>(b) * p.Hq + h) * p.S + split;
    p.o_part[slot * D + e] = acc;
    if (e == 0) {
      p.ml_part[slot * 2] = M;
      p.ml_part[slot * 2 + 1] = lsum;
    }
  }
  __syncthreads();
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ o_part,
                                                          const float* __restrict__ ml_part,
                                                          const int* __restrict__ seqlens,
                                                          __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                          int Hq, int S, int C, int Lcap) {
  const int bh = blockIdx.x;
  const int b = bh / Hq;
  int L = seqlens[b];
  L = L < 0 ? 0 : (L > Lcap ? Lcap : L);
  const int nsplit = min(S, (L + C - 1) / C);
  const int e = threadIdx.x;
  const float* ml = ml_part + static_cast<size_t>(bh) * S * 2;
  const float* op = o_part + static_cast<size_t>(bh) * S * D;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ml[2 * s]);
  if (nsplit == 0 || M == -INFINITY) {
    o[static_cast<size_t>(bh) * D + e] = __float2bfloat16_rn(0.f);
    if (e == 0 && lse != nullptr) lse[bh] = -INFINITY;
    return;
  }
  float lsum = 0.f, acc = 0.f;
  for (int s = 0; s < nsplit; ++s) {  // fixed split order: deterministic
    const float w = ex2_approx(ml[2 * s] - M);
    lsum = fmaf(w, ml[2 * s + 1], lsum);
    acc = fmaf(w, op[static_cast<size_t>(s) * D + e], acc);
  }
  o[static_cast<size_t>(bh) * D + e] = __float2bfloat16_rn(acc / lsum);
  if (e == 0 && lse != nullptr) lse[bh] = (M + log2f(lsum)) * 0.69314718055994530942f;
}

template <int D, int G>
static cudaError_t launch_split(const DecodeParams& p, int B, cudaStream_t stream) {
  using Cfg = DecodeCfg<D>;
  auto kern = decode_split_kernel<D, G>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (err != cudaSuccess) return err;
  const dim3 grid(p.S, p.Hkv, B);
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_split_g(const DecodeParams& p, int B, cudaStream_t stream) {
  switch (p.g) {
    case 1: return launch_split<D, 1>(p, B, stream);
    case 2: return launch_split<D, 2>(p, B, stream);
    case 3: return launch_split<D, 3>(p, B, stream);
    case 4: return launch_split<D, 4>(p, B, stream);
    case 5: return launch_split<D, 5>(p, B, stream);
    case 6: return launch_split<D, 6>(p, B, stream);
    case 7: return launch_split<D, 7>(p, B, stream);
    case 8: return launch_split<D, 8>(p, B, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Returns the number of kernels launched through *launched.
cudaError_t launch_decode(const void* q, const void* kc, const void* vc, const int* seqlens, void* o, float* lse,
                          int B, int Hq, int Hkv, int d, int Lcap, float scale, int S, int C, void* workspace,
                          cudaStream_t stream, int* launched) {
  *launched = 0;
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kc = static_cast<const __nv_bfloat16*>(kc);
  p.vc = static_cast<const __nv_bfloat16*>(vc);
  p.seqlens = seqlens;
  p.o_part = static_cast<float*>(workspace);
  p.ml_part = p.o_part + static_cast<size_t>(B) * Hq * S * d;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.Lcap = Lcap;
  p.S = S;
  p.C = C;
  p.c = scale * 1.4426950408889634f;
  cudaError_t err = (d == 64) ? launch_split_g<64>(p, B, stream) : launch_split_g<128>(p, B, stream);
  if (err != cudaSuccess) return err;
  *launched = 1;
  if (d == 64) {
    decode_combine_kernel<64><<<B * Hq, 64, 0, stream>>>(p.o_part, p.ml_part, seqlens,
                                                         static_cast<__nv_bfloat16*>(o), lse, Hq, S, C, Lcap);
  } else {
    decode_combine_kernel<128><<<B * Hq, 128, 0, stream>>>(p.o_part, p.ml_part, seqlens,
                                                           static_cast<__nv_bfloat16*>(o), lse, Hq, S, C, Lcap);
  }
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
// only a host-side stand-in, so its device address is looked up once per device (with
// that device current) and cached. The first lookup on a device may load this library's
// device code there; it does not call cudaMalloc.
cudaError_t decode_noalloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
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
