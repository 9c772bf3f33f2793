// kvquant.cu - writes a bf16 KV cache as E4M3 (FP8) codes with one scale per (sequence, head).
//
// "Chapter 5. Operators and runtime", section 5.4.3, example 5-7: the E4M3 format (one sign,
// four exponent and three mantissa bits, largest finite value 448); a scale maps the largest
// magnitude of the block it covers onto 448, each element is divided by the scale and
// rounded to a representable value, and multiplying the code's value by the scale gives the
// element back. "How does FlashAttention-3 work mathematically", section 6: E4M3 for K and V.
//
// Here one scale covers the whole [L, d] block of one (sequence, K/V head):
//   scale = amax / 448   (one correctly rounded fp32 division; 1 for an all-zero block)
//   code  = RNE(x / scale), saturated at +-448   (cvt.rn.satfinite.e4m3x2.f32)
// Four launches on the caller's stream: zero the scale array; per-head amax (each CTA
// reduces its chunk and combines with atomicMax on the float's bits, which order like the
// values for non-negative floats); the codes (every CTA derives the scale from the amax);
// amax -> scale in place. The result does not depend on the order the CTAs run in.
#include "common.cuh"

namespace gb300 {

constexpr int kQuantThreads = 256;
constexpr int kQuantVecPerThread = 2;                                        // 16-byte vectors of 8 bf16
constexpr int kQuantChunk = kQuantThreads * kQuantVecPerThread * 8;          // elements per CTA
constexpr float kE4M3Max = 448.0f;

__global__ void kv_scale_zero_kernel(float* __restrict__ scale, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) scale[i] = 0.f;
}

__global__ void __launch_bounds__(kQuantThreads) kv_amax_kernel(const uint4* __restrict__ x, float* __restrict__ amax,
                                                                long long per_head) {
  __shared__ float red[kQuantThreads / 32];
  const int bh = blockIdx.y;
  const uint4* xh = x + static_cast<long long>(bh) * (per_head / 8);
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < kQuantVecPerThread; ++k) {
    const long long v = static_cast<long long>(blockIdx.x) * (kQuantChunk / 8) + k * kQuantThreads + threadIdx.x;
    if (v < per_head / 8) {
      const uint4 u = __ldcs(xh + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) m = fmax3(m, fabsf(bf16lo_to_f32(w[e])), fabsf(bf16hi_to_f32(w[e])));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
#pragma unroll
    for (int w = 0; w < kQuantThreads / 32; ++w) b = fmaxf(b, red[w]);
    atomicMax(reinterpret_cast<unsigned int*>(amax) + bh, __float_as_uint(b));
  }
}

__device__ __forceinline__ float scale_of(float amax) { return amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.f; }

// Two floats -> two E4M3 codes, the first in the low byte (the lower address).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float first, float second) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}

__global__ void __launch_bounds__(kQuantThreads) kv_quant_kernel(const uint4* __restrict__ x, uint2* __restrict__ codes,
                                                                 const float* __restrict__ amax, long long per_head) {
  const int bh = blockIdx.y;
  const float sc = scale_of(amax[bh]);
  const uint4* xh = x + static_cast<long long>(bh) * (per_head / 8);
  uint2* ch = codes + static_cast<long long>(bh) * (per_head / 8);
#pragma unroll
  for (int k = 0; k < kQuantVecPerThread; ++k) {
    const long long v = static_cast<long long>(blockIdx.x) * (kQuantChunk / 8) + k * kQuantThreads + threadIdx.x;
    if (v < per_head / 8) {
      const uint4 u = __ldcs(xh + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t c[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        c[e] = f32x2_to_e4m3x2(__fdiv_rn(bf16lo_to_f32(w[e]), sc), __fdiv_rn(bf16hi_to_f32(w[e]), sc));
      ch[v] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
  }
}

__global__ void kv_scale_finalize_kernel(float* __restrict__ scale, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) scale[i] = scale_of(scale[i]);
}

// x: bf16 [BH, per_head] (per_head a multiple of 8), codes: [BH, per_head] bytes, scale: fp32 [BH].
cudaError_t launch_kv_quantize_fp8(const void* x, void* codes, float* scale, int BH, long long per_head,
                                   cudaStream_t stream, int* launched) {
  *launched = 0;
  const long long chunks = (per_head + kQuantChunk - 1) / kQuantChunk;
  if (BH <= 0 || BH > 65535 || chunks <= 0 || chunks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const int small = (BH + 255) / 256;
  kv_scale_zero_kernel<<<small, 256, 0, stream>>>(scale, BH);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  *launched = 1;
  const dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(BH));
  kv_amax_kernel<<<grid, kQuantThreads, 0, stream>>>(static_cast<const uint4*>(x), scale, per_head);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  *launched = 2;
  kv_quant_kernel<<<grid, kQuantThreads, 0, stream>>>(static_cast<const uint4*>(x), static_cast<uint2*>(codes), scale,
                                                      per_head);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  *launched = 3;
  kv_scale_finalize_kernel<<<small, 256, 0, stream>>>(scale, BH);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  *launched = 4;
  return cudaSuccess;
}

}  // namespace gb300
