// rmsnorm.cu - fused one-pass RMSNorm, and the residual-add form, with one fixed order of
// the sum of squares for every batch size (sm_103a).
//
// y[t, j] = x[t, j] / sqrt(mean_j x[t, j]^2 + eps) * w[j]
// "Module 07: Fused operators and FlashAttention", section "Fused RMSNorm": the sum of
// squares stays in registers (no x^2 tensor) and the row is held on chip, so the second
// use of x does not go back to memory; the end of its RMSNorm assignment folds in the
// residual add, rms_norm(x + residual), one more pass saved. Here the residual form
// writes h = bf16(x + r) (the new residual stream) and normalises that stored h, the
// rounding the unfused pair of operators would do ("Chapter 5. Operators and runtime",
// section 5.4.3: a fused program keeps the rounding of the original one).
//
// Batch invariance ("Chapter 5", section 5.2.4): splitting a row's sum of squares into
// more pieces when there are few rows (decode) changes the floating-point result unless
// the pieces and the order they are combined in are fixed. Every launch here uses one
// canonical order that depends only on D:
//   * 8 segments of D/8 elements when D % 64 == 0, else 1 segment (the whole row);
//   * in a segment, 16 virtual lanes: virtual lane v sums the squares of the segment's
//     16-byte vectors v, v + 16, v + 32, ... element by element (fmaf, in memory order);
//     then an xor butterfly over the 16 (distances 8, 4, 2, 1);
//   * row sum = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7)).
// Two launch shapes compute exactly this: a warp per row (lanes 0-15 and 16-31 each take
// one segment per round; used for many rows) and a block of 4 warps per row (each warp's
// half-warps take one segment each, the sums meet in shared memory; used for few rows,
// where a warp per row would leave most SMs idle). A row's output is bitwise the same in
// both, so it does not depend on how many rows are normalised together.
#include "common.cuh"

namespace gb300 {

constexpr int kNormSegLanes = 16;
constexpr int kNormSplitWarps = 4;     // warps per row in the block-per-row shape
constexpr int kNormSplitMaxRows = 512; // up to this many rows use the block-per-row shape

__device__ __forceinline__ float sumsq8(const uint4 v, float acc) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = bf16lo_to_f32(u[e]);
    const float b = bf16hi_to_f32(u[e]);
    acc = fmaf(a, a, acc);
    acc = fmaf(b, b, acc);
  }
  return acc;
}

__device__ __forceinline__ uint4 add_bf16x8(const uint4 a, const uint4 b) {
  const uint32_t ua[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    o[e] = pack_bf16x2(bf16lo_to_f32(ua[e]) + bf16lo_to_f32(ub[e]), bf16hi_to_f32(ua[e]) + bf16hi_to_f32(ub[e]));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 scale_bf16x8(const uint4 xv, const uint4 wv, float r) {
  const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    o[e] = pack_bf16x2(bf16lo_to_f32(xu[e]) * r * bf16lo_to_f32(wu[e]), bf16hi_to_f32(xu[e]) * r * bf16hi_to_f32(wu[e]));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One segment's vectors for one virtual lane: VPL vectors vl, vl + 16, ... (zero past the
// segment's end), with the residual added when RES. Loads only: every load of a row is
// issued before any reduction, so the row's DRAM latency is paid once.
template <int VPL, bool RES>
__device__ __forceinline__ void load_segment(const uint4* __restrict__ xs, const uint4* __restrict__ rs, int seg_vecs,
                                             int vl, uint4 (&v)[VPL]) {
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int k = vl + kNormSegLanes * i;
    if constexpr (RES)
      v[i] = (k < seg_vecs) ? add_bf16x8(__ldcs(xs + k), __ldcs(rs + k)) : make_uint4(0, 0, 0, 0);
    else
      v[i] = (k < seg_vecs) ? __ldcs(xs + k) : make_uint4(0, 0, 0, 0);
  }
}

// The segment's sum of squares in the canonical order: each virtual lane over its vectors
// in index order (the zero vectors past the end add exact zeros), then the butterfly over
// the 16 virtual lanes of the segment (a half-warp).
template <int VPL>
__device__ __forceinline__ float segment_sumsq(const uint4 (&v)[VPL]) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) ss = sumsq8(v[i], ss);
#pragma unroll
  for (int off = kNormSegLanes / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  return ss;
}

template <int VPL, bool RES>
__device__ __forceinline__ void store_segment(const uint4 (&v)[VPL], const uint4* __restrict__ ws,
                                              uint4* __restrict__ ys, uint4* __restrict__ hs, int seg_vecs, int vl,
                                              float r) {
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int k = vl + kNormSegLanes * i;
    if (k < seg_vecs) {
      if constexpr (RES) __stcs(hs + k, v[i]);
      __stcs(ys + k, scale_bf16x8(v[i], __ldg(ws + k), r));
    }
  }
}

// Start pulling `bytes` at `src` into L2 (an asynchronous bulk prefetch: no data returns to the
// SM, nothing waits for it).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ float combine8(const float (&s)[8]) {
  return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

// A warp per row. NSEG = 8 or 1 segments; each lane holds NSEG/2 segments' vectors (8 segments)
// or its half of the row's one segment (lanes 16-31 idle).
template <int NSEG, int VPL, bool RES>
__global__ void __launch_bounds__(256) rmsnorm_warp_kernel(const uint4* __restrict__ x, const uint4* __restrict__ res,
                                                           const uint4* __restrict__ w, uint4* __restrict__ y,
                                                           uint4* __restrict__ h, int T, int D, float eps) {
  // Launched with programmatic stream serialisation (see launch_shape). The row is first
  // prefetched into L2, which may overlap the previous kernel's end: L2 is where the previous
  // kernel's writes land, so this cannot make the loads below see old data. Then wait until the
  // previous kernel has completed and its writes are visible, and let the next launch be set up.
  constexpr int kRounds = NSEG == 8 ? 4 : 1;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nvec = D >> 3;
  if (lane == 0 && row < T) {
    prefetch_l2(x + static_cast<size_t>(row) * nvec, static_cast<uint32_t>(D) * 2);
    if (RES) prefetch_l2(res + static_cast<size_t>(row) * nvec, static_cast<uint32_t>(D) * 2);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (row >= T) return;
  const int seg_vecs = nvec / NSEG;
  const int half = lane >> 4, vl = lane & 15;
  const size_t off = static_cast<size_t>(row) * nvec;
  uint4 v[kRounds][VPL];
  float s[8];
#pragma unroll
  for (int k = 0; k < kRounds; ++k) {
    const int seg = (NSEG == 8) ? 2 * k + half : 0;
    const bool active = (NSEG == 8) || half == 0;
    load_segment<VPL, RES>(x + off + seg * seg_vecs, RES ? res + off + seg * seg_vecs : nullptr, active ? seg_vecs : 0,
                           vl, v[k]);
  }
#pragma unroll
  for (int k = 0; k < kRounds; ++k) {
    const float ss = segment_sumsq<VPL>(v[k]);
    // both half-warps' sums to every lane: s[2k] from lanes 0-15, s[2k + 1] from lanes 16-31
    const float other = __shfl_xor_sync(0xFFFFFFFFu, ss, 16);
    s[2 * k] = half ? other : ss;
    s[2 * k + 1] = half ? ss : other;
  }
  float total;
  if constexpr (NSEG == 8) {
    total = combine8(s);
  } else {
    total = s[0];
  }
  const float r = rsqrtf(total / static_cast<float>(D) + eps);
#pragma unroll
  for (int k = 0; k < kRounds; ++k) {
    const int seg = (NSEG == 8) ? 2 * k + half : 0;
    const bool active = (NSEG == 8) || half == 0;
    store_segment<VPL, RES>(v[k], w + seg * seg_vecs, y + off + seg * seg_vecs, RES ? h + off + seg * seg_vecs : nullptr,
                            active ? seg_vecs : 0, vl, r);
  }
}

// A block of kNormSplitWarps warps per row: half-warp j of warp i takes segment 2i + j.
template <int NSEG, int VPL, bool RES>
__global__ void __launch_bounds__(32 * kNormSplitWarps) rmsnorm_split_kernel(
    const uint4* __restrict__ x, const uint4* __restrict__ res, const uint4* __restrict__ w, uint4* __restrict__ y,
    uint4* __restrict__ h, int D, float eps) {
  // launched with programmatic stream serialisation: the row is prefetched into L2 first, as in
  // rmsnorm_warp_kernel, then the kernel waits for the previous one
  __shared__ float seg_sum[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x;
  const int nvec = D >> 3;
  if (threadIdx.x == 0) {
    prefetch_l2(x + static_cast<size_t>(row) * nvec, static_cast<uint32_t>(D) * 2);
    if (RES) prefetch_l2(res + static_cast<size_t>(row) * nvec, static_cast<uint32_t>(D) * 2);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int seg_vecs = nvec / NSEG;
  const int half = lane >> 4, vl = lane & 15;
  const int seg = 2 * warp + half;
  const bool active = seg < NSEG;
  const size_t off = static_cast<size_t>(row) * nvec;
  const int segc = active ? seg : 0;
  uint4 v[VPL];
  load_segment<VPL, RES>(x + off + segc * seg_vecs, RES ? res + off + segc * seg_vecs : nullptr, active ? seg_vecs : 0,
                         vl, v);
  const float ss = segment_sumsq<VPL>(v);
  if (active && vl == 0) seg_sum[seg] = ss;
  __syncthreads();
  float total;
  if constexpr (NSEG == 8) {
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = seg_sum[i];
    total = combine8(s);
  } else {
    total = seg_sum[0];
  }
  const float r = rsqrtf(total / static_cast<float>(D) + eps);
  store_segment<VPL, RES>(v, w + segc * seg_vecs, y + off + segc * seg_vecs, RES ? h + off + segc * seg_vecs : nullptr,
                          active ? seg_vecs : 0, vl, r);
}

template <int NSEG, int VPL, bool RES>
static cudaError_t launch_shape(const void* x, const void* r, const void* w, void* y, void* h, int T, int D, float eps,
                                cudaStream_t s) {
  const uint4* xp = static_cast<const uint4*>(x);
  const uint4* rp = static_cast<const uint4*>(r);
  const uint4* wp = static_cast<const uint4*>(w);
  uint4* yp = static_cast<uint4*>(y);
  uint4* hp = static_cast<uint4*>(h);
  // Programmatic stream serialisation: the grid's CTAs may be placed while the previous kernel on
  // the stream drains (griddepcontrol.wait in the kernel orders every read after its completion),
  // which hides most of the launch gap of this short, latency-bound kernel.
  cudaLaunchConfig_t cfg = {};
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err;
  if (T <= kNormSplitMaxRows) {
    cfg.gridDim = dim3(static_cast<unsigned>(T));
    cfg.blockDim = dim3(32 * kNormSplitWarps);
    err = cudaLaunchKernelEx(&cfg, rmsnorm_split_kernel<NSEG, VPL, RES>, xp, rp, wp, yp, hp, D, eps);
  } else {
    const int rows_per_block = 8;
    cfg.gridDim = dim3(static_cast<unsigned>((T + rows_per_block - 1) / rows_per_block));
    cfg.blockDim = dim3(32 * rows_per_block);
    err = cudaLaunchKernelEx(&cfg, rmsnorm_warp_kernel<NSEG, VPL, RES>, xp, rp, wp, yp, hp, T, D, eps);
  }
  return err != cudaSuccess ? err : cudaGetLastError();
}

// VPL = vectors per virtual lane per segment, rounded up to a power of two.
template <int NSEG, bool RES>
static cudaError_t launch_nseg(const void* x, const void* r, const void* w, void* y, void* h, int T, int D, float eps,
                               cudaStream_t s) {
  const int seg_vecs = (D / 8) / NSEG;
  const int vpl = (seg_vecs + kNormSegLanes - 1) / kNormSegLanes;
  if (vpl <= 1) return launch_shape<NSEG, 1, RES>(x, r, w, y, h, T, D, eps, s);
  if (vpl <= 2) return launch_shape<NSEG, 2, RES>(x, r, w, y, h, T, D, eps, s);
  if (vpl <= 4) return launch_shape<NSEG, 4, RES>(x, r, w, y, h, T, D, eps, s);
  if (vpl <= 8) return launch_shape<NSEG, 8, RES>(x, r, w, y, h, T, D, eps, s);
  if constexpr (NSEG == 8) {
    return cudaErrorInvalidValue;  // D <= 8192 keeps vpl <= 8 with 8 segments
  } else {
    if (vpl <= 16) return launch_shape<NSEG, 16, RES>(x, r, w, y, h, T, D, eps, s);
    if (vpl <= 32) return launch_shape<NSEG, 32, RES>(x, r, w, y, h, T, D, eps, s);
    return cudaErrorInvalidValue;
  }
}

// Segments of the canonical order for a row of D elements (0: D not supported).
int rmsnorm_segments(int D) {
  if (D < 8 || D % 8 != 0 || D > 8192) return 0;
  if (D % 64 == 0) return 8;
  return D <= 4096 ? 1 : 0;
}

// r/h == nullptr: plain RMSNorm; else h = bf16(x + r) and y = RMSNorm(h) * w.
cudaError_t launch_rmsnorm(const void* x, const void* r, const void* w, void* y, void* h, int T, int D, float eps,
                           cudaStream_t s) {
  const int nseg = rmsnorm_segments(D);
  const bool res = r != nullptr;
  if (nseg == 8) return res ? launch_nseg<8, true>(x, r, w, y, h, T, D, eps, s) : launch_nseg<8, false>(x, r, w, y, h, T, D, eps, s);
  if (nseg == 1) return res ? launch_nseg<1, true>(x, r, w, y, h, T, D, eps, s) : launch_nseg<1, false>(x, r, w, y, h, T, D, eps, s);
  return cudaErrorInvalidValue;
}

uint32_t rmsnorm_take_device_error() { return take_device_error_word(); }

}  // namespace gb300
