// rmsnorm.cu - fused one-pass RMSNorm, one row per warp (sm_103a).
//
// y[t, j] = x[t, j] / sqrt(mean_j x[t, j]^2 + eps) * w[j]
// "Module 07: Fused operators and FlashAttention", section "Fused RMSNorm":
// the sum of squares stays in registers (no x^2 tensor), and a row of
// D = 1024 bf16 values (2 KB) is held by one warp, so the second use of x does
// not go back to memory. Traffic is the 4D bytes per row of the fused form
// (read x, write y) plus w, which stays in L2/L1.
#include "common.cuh"

namespace gb300 {

// NV = 16-byte vectors per lane (each vector = 8 bf16). Lane l of the warp
// owns vectors l, l + 32, l + 64, ... of its row, so every load instruction of
// the warp reads 512 contiguous bytes.
template <int NV>
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const uint4* __restrict__ x, const uint4* __restrict__ w,
                                                           uint4* __restrict__ y, int T, int D, float eps) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= T) return;
  const int nvec = D >> 3;
  const uint4* xr = x + static_cast<size_t>(row) * nvec;
  uint4* yr = y + static_cast<size_t>(row) * nvec;

  uint4 xv[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = lane + 32 * i;
    xv[i] = (v < nvec) ? __ldcs(xr + v) : make_uint4(0, 0, 0, 0);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const uint32_t u[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16lo_to_f32(u[e]);
      const float b = bf16hi_to_f32(u[e]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
  const float r = rsqrtf(ss / static_cast<float>(D) + eps);

#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = lane + 32 * i;
    if (v < nvec) {
      const uint4 wv = __ldg(w + v);
      const uint32_t xu[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
      const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
      uint32_t out[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = bf16lo_to_f32(xu[e]) * r * bf16lo_to_f32(wu[e]);
        const float hi = bf16hi_to_f32(xu[e]) * r * bf16hi_to_f32(wu[e]);
        out[e] = pack_bf16x2(lo, hi);
      }
      __stcs(yr + v, make_uint4(out[0], out[1], out[2], out[3]));
    }
  }
}

template <int NV>
static cudaError_t launch_nv(const void* x, const void* w, void* y, int T, int D, float eps, cudaStream_t s) {
  const int rows_per_block = 8;
  const dim3 grid((T + rows_per_block - 1) / rows_per_block);
  rmsnorm_rows_kernel<NV><<<grid, 32 * rows_per_block, 0, s>>>(
      static_cast<const uint4*>(x), static_cast<const uint4*>(w), static_cast<uint4*>(y), T, D, eps);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* x, const void* w, void* y, int T, int D, float eps, cudaStream_t s) {
  const int nvec = D / 8;
  const int per_lane = (nvec + 31) / 32;
  if (per_lane <= 1) return launch_nv<1>(x, w, y, T, D, eps, s);
  if (per_lane <= 2) return launch_nv<2>(x, w, y, T, D, eps, s);
  if (per_lane <= 4) return launch_nv<4>(x, w, y, T, D, eps, s);
  if (per_lane <= 8) return launch_nv<8>(x, w, y, T, D, eps, s);
  if (per_lane <= 16) return launch_nv<16>(x, w, y, T, D, eps, s);
  return launch_nv<32>(x, w, y, T, D, eps, s);
}

uint32_t rmsnorm_take_device_error() { return take_device_error_word(); }

}  // namespace gb300
