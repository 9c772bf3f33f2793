// api.cu - the library's C ABI (include/attn.h): argument validation, dispatch to the
// kernels, device error reporting and the launch counter.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/attn.h"
#include "common.cuh"

namespace gb300 {
cudaError_t launch_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                            int Tq, int Tk, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream, int* launched);
size_t prefill_workspace_bytes(int d);
cudaError_t launch_decode(const void* q, const void* kc, const void* vc, const float* k_scale, const float* v_scale,
                          const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv, int d, int Lcap,
                          float scale, int S, int C, void* workspace, cudaStream_t stream, int* launched);
cudaError_t launch_kv_quantize_fp8(const void* x, void* codes, float* scale, int BH, long long per_head,
                                   cudaStream_t stream, int* launched);
cudaError_t launch_rmsnorm(const void* x, const void* r, const void* w, void* y, void* h, int T, int D, float eps,
                           cudaStream_t s);
int rmsnorm_segments(int D);
size_t decode_noalloc_capacity();
size_t decode_balanced_workspace_bytes(int d);
int decode_balanced_max_batch();
cudaError_t decode_noalloc_scratch(cudaStream_t stream, void** ptr);
cudaError_t launch_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Tq, int Tk,
                            int d, int causal, float scale, void* workspace, cudaStream_t stream, int* launched);
uint32_t backward_take_device_error();
uint32_t prefill_take_device_error();
uint32_t prefill_pair_take_device_error();
uint32_t decode_take_device_error();
uint32_t rmsnorm_take_device_error();

static std::atomic<unsigned long long> g_launches{0};

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by the decode entry points (everything but the workspace).
static attn_status check_decode_args(const void* q, const void* kcache, const void* vcache, const int* seqlens,
                                     const void* o, const float* lse, int B, int Hq, int Hkv, int d, int Lcap,
                                     float scale, int num_splits) {
  if (q == nullptr || kcache == nullptr || vcache == nullptr || seqlens == nullptr || o == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lcap < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  // 0 selects the balanced schedule; otherwise splits of at least 16 keys
  if (num_splits < 0 || num_splits > (Lcap + 15) / 16) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (Hq / Hkv > 8) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  if (static_cast<long long>(num_splits) > 65535 || static_cast<long long>(Hkv) > 65535 || B > 65535)
    return ATTN_ERR_UNSUPPORTED;
  if (num_splits == 0) {
    // the balanced schedule keeps the tile prefix sums of all sequences in shared memory and
    // counts tiles (64 keys) of all (sequence, head block) segments in an int
    const long long blocks = (Hq / Hkv + 3) / 4;  // head blocks per K/V head
    if (B > decode_balanced_max_batch()) return ATTN_ERR_UNSUPPORTED;
    if (static_cast<long long>(Hkv) * blocks * B * ((static_cast<long long>(Lcap) + 63) / 64) >= 0x7FFFFFFFLL)
      return ATTN_ERR_UNSUPPORTED;
  }
  return ATTN_OK;
}

static int decode_chunk(int Lcap, int num_splits) {
  if (num_splits == 0) return 0;  // balanced schedule: no fixed chunks
  const long long c = (static_cast<long long>(Lcap) + num_splits - 1) / num_splits;
  return static_cast<int>((c + 15) / 16 * 16);
}

// One thread waits on a barrier that nothing completes; the bounded wait gives up.
__global__ void selftest_wait_kernel(uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, timeout_ns);
  __syncthreads();
}

}  // namespace gb300

using namespace gb300;

extern "C" {

size_t attn_fwd_workspace_size(int d) {
  if (d != 64 && d != 128) return 0;
  return prefill_workspace_bytes(d);
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Tq, int Tk, int d, int causal, float scale, cudaStream_t stream) {
  return attn_fwd_ws(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale, nullptr, 0, stream);
}

attn_status attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Tq, int Tk, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  if (static_cast<long long>(B) * Hq > 0x7FFFFFFFLL || static_cast<long long>(B) * Hkv > 0x7FFFFFFFLL)
    return ATTN_ERR_INVALID_ARG;
  if (workspace == nullptr && workspace_bytes != 0) return ATTN_ERR_WORKSPACE;
  if (workspace != nullptr) {
    if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
    if (workspace_bytes < attn_fwd_workspace_size(d)) return ATTN_ERR_WORKSPACE;
  }
  int launched = 0;
  const cudaError_t err = launch_attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, scale, workspace,
                                          workspace_bytes, stream, &launched);
  g_launches.fetch_add(static_cast<unsigned long long>(launched));
  if (err != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

size_t attn_decode_workspace_size(int B, int Hq, int d, int num_splits) {
  if (B < 1 || Hq < 1 || d < 1 || num_splits < 0) return 0;
  if (num_splits == 0) return (d == 64 || d == 128) ? decode_balanced_workspace_bytes(d) : 0;
  return static_cast<size_t>(B) * Hq * num_splits * (static_cast<size_t>(d) + 2) * sizeof(float);
}

int attn_decode_default_splits(int B, int Hkv, int Lcap) {
  if (B < 1 || Hkv < 1 || Lcap < 1) return 1;
  // Chunks of about 1024 keys (measured best at 32 splits for 16 sequences of up to 32768 keys);
  // at least enough splits for ~2 thread blocks per SM of a 152-SM part when the batch is small
  // (the split kernel runs 2 per SM; measured, B16 Hkv8 d128, Lcap 2048: 2 splits 7 % faster
  // than 4).
  int s = (Lcap + 1023) / 1024;
  const long long want = (2LL * 152 + static_cast<long long>(B) * Hkv - 1) / (static_cast<long long>(B) * Hkv);
  if (s < want) s = want > (1 << 20) ? (1 << 20) : static_cast<int>(want);
  // Rounded down to a power of two: with a power-of-two cache length every chunk is then a whole
  // number of the kernel's 64-row stages (measured with the earlier FFMA split kernel, B16 Hkv8
  // d128: Lcap 2048, 4 splits 23.7 us per step vs 28.3 us with 5; Lcap 8192, 8 splits 75.3 vs
  // 90.6 with 6).
  int p2 = 1;
  while (p2 <= s / 2) p2 *= 2;
  s = p2;
  const int smax = (Lcap + 15) / 16;
  if (s > smax) s = smax;
  return s < 1 ? 1 : s;
}

size_t attn_bwd_workspace_size(int B, int Hq, int Tq) {
  if (B < 1 || Hq < 1 || Tq < 1) return 0;
  const size_t bytes = static_cast<size_t>(B) * Hq * Tq * sizeof(float);
  return (bytes + 255) / 256 * 256;
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                     float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || lse == nullptr || dout == nullptr ||
      dq == nullptr || dk == nullptr || dv == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > 65535 || static_cast<long long>(B) * Hkv > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  if (workspace == nullptr || workspace_bytes < attn_bwd_workspace_size(B, Hq, Tq)) return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  int launched = 0;
  const cudaError_t err = launch_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d, causal, scale,
                                          workspace, stream, &launched);
  g_launches.fetch_add(static_cast<unsigned long long>(launched));
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_decode(const void* q, const void* kcache, const void* vcache, const int* seqlens, void* o,
                        float* lse, int B, int Hq, int Hkv, int d, int Lcap, float scale, int num_splits,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const attn_status st =
      check_decode_args(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, d, Lcap, scale, num_splits);
  if (st != ATTN_OK) return st;
  if (workspace == nullptr || workspace_bytes < attn_decode_workspace_size(B, Hq, d, num_splits))
    return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  const int C = decode_chunk(Lcap, num_splits);
  int launched = 0;
  const cudaError_t err = launch_decode(q, kcache, vcache, nullptr, nullptr, seqlens, o, lse, B, Hq, Hkv, d, Lcap,
                                        scale, num_splits, C, workspace, stream, &launched);
  g_launches.fetch_add(static_cast<unsigned long long>(launched));
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_decode_fp8(const void* q, const void* kcache, const void* vcache, const float* k_scale,
                            const float* v_scale, const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                            int d, int Lcap, float scale, int num_splits, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  const attn_status st =
      check_decode_args(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, d, Lcap, scale, num_splits);
  if (st != ATTN_OK) return st;
  if (k_scale == nullptr || v_scale == nullptr) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_scale) & 3u) != 0 || (reinterpret_cast<uintptr_t>(v_scale) & 3u) != 0)
    return ATTN_ERR_MISALIGNED;
  if (workspace == nullptr || workspace_bytes < attn_decode_workspace_size(B, Hq, d, num_splits))
    return ATTN_ERR_WORKSPACE;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  const int C = decode_chunk(Lcap, num_splits);
  int launched = 0;
  const cudaError_t err = launch_decode(q, kcache, vcache, k_scale, v_scale, seqlens, o, lse, B, Hq, Hkv, d, Lcap,
                                        scale, num_splits, C, workspace, stream, &launched);
  g_launches.fetch_add(static_cast<unsigned long long>(launched));
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_kv_quantize_fp8(const void* x, void* codes, float* scale, int B, int H, int L, int d,
                                 cudaStream_t stream) {
  if (x == nullptr || codes == nullptr || scale == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || L < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
  if (d % 8 != 0) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 7u) != 0 || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
    return ATTN_ERR_MISALIGNED;
  int launched = 0;
  const cudaError_t err = launch_kv_quantize_fp8(x, codes, scale, B * H, static_cast<long long>(L) * d, stream,
                                                 &launched);
  g_launches.fetch_add(static_cast<unsigned long long>(launched));
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_decode_noalloc(const void* q, const void* kcache, const void* vcache, const int* seqlens,
                                void* o, float* lse, int B, int Hq, int Hkv, int d, int Lcap, float scale,
                                int num_splits, cudaStream_t stream) {
  const attn_status st =
      check_decode_args(q, kcache, vcache, seqlens, o, lse, B, Hq, Hkv, d, Lcap, scale, num_splits);
  if (st != ATTN_OK) return st;
  // The partials must fit the library's fixed scratch; refuse before touching the device.
  if (attn_decode_workspace_size(B, Hq, d, num_splits) > decode_noalloc_capacity()) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (decode_noalloc_scratch(stream, &scratch) != cudaSuccess) return ATTN_ERR_CUDA;
  const int C = decode_chunk(Lcap, num_splits);
  int launched = 0;
  const cudaError_t err = launch_decode(q, kcache, vcache, nullptr, nullptr, seqlens, o, lse, B, Hq, Hkv, d, Lcap,
                                        scale, num_splits, C, scratch, stream, &launched);
  g_launches.fetch_add(static_cast<unsigned long long>(launched));
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status rmsnorm_fwd(const void* x, const void* w, void* y, int T, int D, float eps, cudaStream_t stream) {
  if (x == nullptr || w == nullptr || y == nullptr) return ATTN_ERR_INVALID_ARG;
  if (T < 1 || D < 8 || D % 8 != 0) return ATTN_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return ATTN_ERR_INVALID_ARG;
  if (rmsnorm_segments(D) == 0) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return ATTN_ERR_MISALIGNED;
  const cudaError_t err = launch_rmsnorm(x, nullptr, w, y, nullptr, T, D, eps, stream);
  if (err != cudaSuccess) return ATTN_ERR_CUDA;
  g_launches.fetch_add(1);
  return ATTN_OK;
}

attn_status rmsnorm_residual_fwd(const void* x, const void* r, const void* w, void* y, void* h, int T, int D,
                                 float eps, cudaStream_t stream) {
  if (x == nullptr || r == nullptr || w == nullptr || y == nullptr || h == nullptr) return ATTN_ERR_INVALID_ARG;
  if (T < 1 || D < 8 || D % 8 != 0) return ATTN_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return ATTN_ERR_INVALID_ARG;
  if (y == x || y == r || y == h) return ATTN_ERR_INVALID_ARG;
  if (rmsnorm_segments(D) == 0) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(r) || !aligned16(w) || !aligned16(y) || !aligned16(h)) return ATTN_ERR_MISALIGNED;
  const cudaError_t err = launch_rmsnorm(x, r, w, y, h, T, D, eps, stream);
  if (err != cudaSuccess) return ATTN_ERR_CUDA;
  g_launches.fetch_add(1);
  return ATTN_OK;
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "pointer not aligned";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

attn_status attn_last_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  const uint32_t e = prefill_take_device_error() | prefill_pair_take_device_error() | decode_take_device_error() |
                     rmsnorm_take_device_error() |
                     backward_take_device_error() | take_device_error_word();
  if (e == 0xFFFFFFFFu) return ATTN_ERR_CUDA;
  if (e & kErrTimeout) return ATTN_ERR_TIMEOUT;
  return ATTN_OK;
}

unsigned long long attn_kernel_launches(void) { return g_launches.load(); }

attn_status attn_selftest_wait_timeout(int timeout_us, cudaStream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return ATTN_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(timeout_us) * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  g_launches.fetch_add(1);
  return ATTN_OK;
}

}  // extern "C"
