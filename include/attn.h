/*
 * attn.h - C ABI of the GB300 (sm_103a) exact tiled attention library.
 *
 * Three operations, each a plain-pointer call that launches hand-written
 * CUDA kernels on the caller's stream:
 *
 *   attn_fwd     exact attention O = softmax(scale * Q K^T + causal mask) V for
 *                many queries (prefill), with grouped-query heads, computed
 *                tile by tile with the online-softmax recurrence so the score
 *                matrix never reaches global memory.
 *   attn_decode  the same for one query per sequence over a KV cache
 *                (flash-decoding: the key range is split across thread blocks,
 *                each writes a partial (m, l, o), a second kernel merges them).
 *   rmsnorm_fwd  fused one-pass RMSNorm, one row per warp.
 *
 * Conventions shared by every entry point
 * - All tensor pointers are DEVICE pointers to memory the caller owns; the
 *   library never allocates, frees or keeps them. "bf16" means IEEE bfloat16
 *   bit patterns (2 bytes, e.g. __nv_bfloat16 / torch.bfloat16).
 * - Layouts are dense row-major with the last dimension contiguous.
 * - Every call is asynchronous on `stream` (NULL = legacy default stream).
 *   The return value reports argument validation and launch errors only;
 *   inputs are never modified. Errors detected on the device (a bounded wait
 *   that timed out) are reported by attn_last_device_error().
 * - On any non-OK return nothing has been launched, except ATTN_ERR_CUDA,
 *   which may follow a failed launch.
 */
#ifndef GB300_ATTN_H_
#define GB300_ATTN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* NULL pointer, non-positive size, bad ratio, bad scale */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented here (e.g. head dim not 64/128) */
  ATTN_ERR_MISALIGNED = 3,   /* pointer not 16-byte aligned */
  ATTN_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than attn_decode_workspace_size() */
  ATTN_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  ATTN_ERR_TIMEOUT = 6       /* a device-side bounded wait expired (reported by attn_last_device_error) */
} attn_status;

/*
 * attn_fwd - exact scaled-dot-product attention for a batch of sequences.
 *
 * Defined by: "FlashAttention: attention without the n x n matrix", section
 * "Forward pass of FlashAttention" (block update of m, l and the accumulator,
 * O = A / l once at the end, and L = m + log l kept per row); "Module 07:
 * Fused operators and FlashAttention", sections "Online softmax: derivation"
 * and "FlashAttention-2" (query-block outer loop, causal block skipping);
 * grouped-query heads as in "Attention from the kernel's side", section
 * "Prefill and decoding are different problems".
 *
 *   q    bf16 [B, Hq,  Tq, d]      queries
 *   k    bf16 [B, Hkv, Tk, d]      keys;   query head h reads K/V head h / (Hq/Hkv)
 *   v    bf16 [B, Hkv, Tk, d]      values
 *   o    bf16 [B, Hq,  Tq, d]      output (written)
 *   lse  fp32 [B, Hq,  Tq] or NULL natural-log log-sum-exp of the scaled scores
 *                                  of each row: ln sum_j exp(scale * q_i . k_j)
 *   d      64 or 128 (else ATTN_ERR_UNSUPPORTED); Hq % Hkv == 0
 *   causal 0: every key is visible; 1: key j is visible to query i iff j <= i
 *          (aligned at the top-left corner when Tq != Tk)
 *   scale  > 0 and finite (1/sqrt(d) for standard attention)
 * Arithmetic: bf16 inputs, fp32 scores and running statistics, P rounded to
 * bf16 for the P.V product, fp32 accumulation, O rounded once to bf16.
 * q, k, v, o must be 16-byte aligned; lse 4-byte aligned. An o that is 32-byte aligned
 * is written with 32-byte stores (faster; the result is the same either way).
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Tq, int Tk, int d,
                     int causal, float scale, cudaStream_t stream);

/*
 * attn_fwd_workspace_size - bytes of scratch attn_fwd_ws can use on the current
 * device for head dimension d: 256 rows x (d + 1) fp32 values per streaming
 * multiprocessor. Returns 0 when d is not 64 or 128.
 */
size_t attn_fwd_workspace_size(int d);

/*
 * attn_fwd_ws - attn_fwd with a scratch buffer, which lets a non-causal call
 * balance its last round of work.
 *
 * The forward kernel runs its work units (two 128-row query tiles that share
 * one K/V stream) on persistent thread blocks, one per SM, in rounds. When a
 * non-causal call leaves the last round partly filled, the units of that round
 * are split along the keys into pieces that run side by side. Each piece keeps
 * its own (m, l, O), and a second kernel merges them in a fixed order with the
 * online-softmax rescaling of "Module 07: Fused operators and FlashAttention",
 * section "Online softmax: derivation" (the merge flash-decoding uses; "Attention
 * from the kernel's side", section "Prefill and decoding are different
 * problems"). Causal calls are never split. The rows of the split units agree
 * with attn_fwd to rounding, not bit for bit; every other row is identical.
 *
 *   workspace        device memory of at least attn_fwd_workspace_size(d)
 *                    bytes, 16-byte aligned, owned by the caller and not read
 *                    or written by anything else until the call's work on
 *                    `stream` has finished; or NULL with workspace_bytes 0,
 *                    which makes the call exactly attn_fwd.
 *   everything else  as attn_fwd.
 * Errors: as attn_fwd; ATTN_ERR_WORKSPACE when workspace is NULL with a non-zero
 * size or smaller than attn_fwd_workspace_size(d); ATTN_ERR_MISALIGNED when it
 * is not 16-byte aligned.
 */
attn_status attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int Hq, int Hkv, int Tq, int Tk, int d,
                        int causal, float scale, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/*
 * attn_decode_workspace_size - bytes of scratch attn_decode needs.
 * Returns 0 for invalid arguments. The workspace holds one fp32 partial
 * (m, l, o[d]) per (sequence, query head, split); for num_splits = 0 (the
 * balanced schedule) two partials of up to 4 query heads per thread block of
 * the current device (2 per SM), whatever B and Hq are.
 */
size_t attn_decode_workspace_size(int B, int Hq, int d, int num_splits);

/*
 * attn_decode_default_splits - a split count that fills the GPU for the given
 * shape (enough thread blocks for every SM several times over). Any value in
 * [1, Lcap/16] is valid, and so is 0 (the balanced schedule, see attn_decode);
 * results differ between split counts by rounding only.
 */
int attn_decode_default_splits(int B, int Hkv, int Lcap);

/*
 * attn_bwd - gradients of attn_fwd with respect to q, k and v, by recomputation
 * from the forward's O and LSE.
 *
 * Defined by: "FlashAttention: attention without the n x n matrix", section
 * "Backward pass: recomputing is cheaper than storing": the block scores are
 * computed again, P_ij = exp(S_ij - L_i) without normalisation, then
 * dV = P^T dO, dP = dO V^T, dS_ij = P_ij (dP_ij - D_i) with D_i = dO_i . O_i,
 * dQ = dS K * scale, dK = dS^T Q * scale. With Hq > Hkv the gradients of a
 * K/V head are the sums over the Hq/Hkv query heads that read it.
 *
 *   q, o, dout  bf16 [B, Hq, Tq, d]; k, v bf16 [B, Hkv, Tk, d]
 *   lse         fp32 [B, Hq, Tq]: the natural log-sum-exp attn_fwd returned
 *   dq          bf16 [B, Hq, Tq, d] (written); dk, dv bf16 [B, Hkv, Tk, d] (written)
 *   causal, scale, d, Hq % Hkv: as attn_fwd (the same causal rule, key j seen by
 *   query i iff j <= i). B*Hq <= 65535.
 *   workspace   device scratch of attn_bwd_workspace_size(B, Hq, Tq) bytes,
 *               16-byte aligned, owned by the caller (holds D_i).
 * All pointers 16-byte aligned; when dq, dk and dv are all 32-byte aligned the
 * gradients are written with 32-byte stores (faster; the same result).
 * Arithmetic: P and dS rounded to bf16 for the tensor-core products, fp32
 * accumulation, outputs rounded once to bf16. Three kernel launches; the
 * result does not depend on their timing (no atomics).
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Tq);
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv,
                     int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal, float scale,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_decode - one query token per sequence against a bf16 KV cache
 * (flash-decoding).
 *
 * Defined by: "Attention from the kernel's side: FlashAttention, online
 * softmax and fused dequantisation", section "Prefill and decoding are
 * different problems" (one query per sequence streams the whole cache; GQA
 * loads each K/V tile once for g query heads; flash-decoding splits the key
 * sequence across thread blocks, each computes a partial (m, l, o) and a
 * last step merges them with the same rescaling rule). The merge rule is the
 * step of "Module 07: Fused operators and FlashAttention", section "Online
 * softmax: derivation".
 *
 *   q        bf16 [B, Hq, d]
 *   kcache   bf16 [B, Hkv, Lcap, d]
 *   vcache   bf16 [B, Hkv, Lcap, d]
 *   seqlens  int32 [B] (device)  keys 0 .. seqlens[b]-1 of sequence b take part;
 *            precondition 1 <= seqlens[b] <= Lcap. A value outside that range
 *            is clamped on the device (0 or less gives O = 0, LSE = -inf).
 *   o        bf16 [B, Hq, d]    output (written)
 *   lse      fp32 [B, Hq] or NULL
 *   d 64 or 128, Hq % Hkv == 0, Hq / Hkv <= 8, scale > 0 and finite
 *   num_splits   1 .. ceil(Lcap / 16): split s covers keys [s*C, (s+1)*C)
 *                with C = ceil(Lcap / num_splits) rounded up to a multiple of
 *                16, one thread block per (split, head block, sequence);
 *                splits are merged in a fixed order, so the result is
 *                deterministic for a given num_splits.
 *                0: the balanced schedule. One persistent thread block per
 *                resident slot (2 per SM) takes an equal share of the 64-key
 *                tiles of all (sequence, K/V head block) pairs, cut at tile
 *                boundaries; a pair that one block holds whole is finished
 *                there, a pair that share boundaries cut is merged from one
 *                partial per block in block order (the same rule), so the
 *                result is deterministic for a given device. For batches of
 *                very different lengths it avoids the last thread blocks of
 *                the split schedule running alone. Needs B <= 1024 and fewer
 *                than 2^31 tiles over all pairs (else ATTN_ERR_UNSUPPORTED).
 *   workspace    device scratch of at least
 *                attn_decode_workspace_size(B, Hq, d, num_splits) bytes, 16-byte
 *                aligned, owned by the caller; it must not be used by another
 *                call that can run at the same time. For num_splits = 0 its
 *                size depends only on d and the current device's SM count.
 */
attn_status attn_decode(const void* q, const void* kcache, const void* vcache,
                        const int* seqlens, void* o, float* lse,
                        int B, int Hq, int Hkv, int d, int Lcap, float scale,
                        int num_splits, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);

/*
 * attn_decode_noalloc - attn_decode for callers that cannot allocate device memory.
 *
 * The source pages have no counterpart to this entry point; it exists for
 * callers that cannot provide attn_decode's workspace: an engine whose KV-cache
 * pool already owns (nearly) all device memory, code running under an allocator
 * or memory budget that forbids new allocations, or a step that must not call
 * cudaMalloc/cudaFree (and the synchronisation they can imply) while it runs.
 * It computes exactly what attn_decode computes, with the same kernels, and takes
 * the same arguments except the workspace: the per-split partials go to a fixed
 * device array inside the library (32 MiB, 256-byte aligned). That array is part
 * of the library's device image, so every GPU that loads the library holds the
 * 32 MiB until the process exits. This call never calls cudaMalloc, cudaFree or
 * any allocating library routine.
 *
 *   Size limit: attn_decode_workspace_size(B, Hq, d, num_splits) must be
 *   <= 32 MiB (33554432 bytes); larger requests return ATTN_ERR_WORKSPACE before
 *   anything runs (use fewer splits, or attn_decode with your own workspace).
 *   Device address: outside a stream capture every call looks the array's
 *   address up on the current device (cudaGetSymbolAddress), so a device
 *   reset or a reloaded module is picked up; inside a capture the address
 *   found by the last uncaptured call on that device is used. The first call
 *   on a device may load the library's device code there: make it before any
 *   stream capture on that device.
 *   Sharing: every call uses the same array, which keeps the previous call's
 *   contents (nothing in it needs to start at zero). Calls that can overlap on
 *   the GPU (other streams, other host threads) race on it: serialise them.
 * Other arguments, layouts, alignment and errors: as attn_decode.
 */
attn_status attn_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                                const int* seqlens, void* o, float* lse,
                                int B, int Hq, int Hkv, int d, int Lcap, float scale,
                                int num_splits, cudaStream_t stream);

/*
 * attn_kv_quantize_fp8 - a bf16 KV cache written as E4M3 (FP8) codes with one
 * scale per (sequence, head).
 *
 * Defined by: "Chapter 5. Operators and runtime", section 5.4.3, example 5-7
 * (the E4M3 format: one sign, four exponent and three mantissa bits, largest
 * finite value 448; a scale maps the largest magnitude of the block it covers
 * onto 448, elements are divided by it and rounded to a representable value,
 * code value x scale gives the element back) and "How does FlashAttention-3
 * work mathematically", section 6 (E4M3 for K and V). The block a scale covers
 * is the whole [L, d] slice of one (sequence, head).
 *
 *   x      bf16 [B, H, L, d], 16-byte aligned (device)
 *   codes  uint8 [B, H, L, d] (written), 8-byte aligned: code = RNE(x / scale)
 *          in E4M3, magnitudes above 448 saturated to 448
 *   scale  fp32 [B, H] (written): amax / 448 as one correctly rounded fp32
 *          division over the slice's largest magnitude; 1 for an all-zero slice
 *   d a multiple of 8; B * H <= 65535. NaN inputs are outside the contract.
 * Four kernel launches on `stream`; the result does not depend on their timing.
 */
attn_status attn_kv_quantize_fp8(const void* x, void* codes, float* scale, int B, int H, int L, int d,
                                 cudaStream_t stream);

/*
 * attn_decode_fp8 - attn_decode over an E4M3 (FP8) KV cache, dequantised in
 * registers as the tiles are read.
 *
 * Defined by: "Attention from the kernel's side: FlashAttention, online
 * softmax and fused dequantisation", section "Why a quantised cache needs a
 * fused kernel" (read the low-precision bytes straight into the kernel and
 * turn them into values in registers: the traffic is the quantised cache and
 * nothing more), with the format of attn_kv_quantize_fp8. The result is the
 * attention of attn_decode over the dequantised keys and values
 * code_value x scale.
 *
 *   kcache, vcache  uint8 E4M3 codes [B, Hkv, Lcap, d], 16-byte aligned
 *   k_scale, v_scale  fp32 [B, Hkv] (device), the per-(sequence, head) scales
 * Everything else (q, seqlens, o, lse, shapes, num_splits, the workspace and
 * its size attn_decode_workspace_size, errors) as attn_decode.
 */
attn_status attn_decode_fp8(const void* q, const void* kcache, const void* vcache,
                            const float* k_scale, const float* v_scale, const int* seqlens,
                            void* o, float* lse, int B, int Hq, int Hkv, int d, int Lcap, float scale,
                            int num_splits, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * rmsnorm_fwd - y = x / sqrt(mean_j x_j^2 + eps) * w for every row, one pass.
 *
 * Defined by: "Module 07: Fused operators and FlashAttention", section
 * "Fused RMSNorm" (the formula; sum of squares kept in registers, the row
 * held on chip, no x^2 tensor) and section "Assignment 07.1:
 * fused_rms_norm" (eps under the root, mean over D).
 *
 *   x  bf16 [T, D], w bf16 [D], y bf16 [T, D] (written; may not alias x)
 *   D  a multiple of 8, 8 <= D <= 8192, and a multiple of 64 when D > 4096;
 *   T >= 1; eps >= 0 and finite. All pointers 16-byte aligned.
 * Arithmetic: fp32 sum of squares and scaling, y rounded once to bf16. The
 * sum of squares follows one fixed order that depends only on D (8 segments
 * of D/8 elements when D % 64 == 0, combined in a fixed tree; "Chapter 5.
 * Operators and runtime", section 5.2.4), whatever T is and however the rows
 * are spread over the GPU, so a row's y is bitwise independent of the batch
 * it is normalised in.
 */
attn_status rmsnorm_fwd(const void* x, const void* w, void* y, int T, int D, float eps,
                        cudaStream_t stream);

/*
 * rmsnorm_residual_fwd - the residual add fused into RMSNorm:
 *   h = bf16(x + r)             (the new residual stream, written)
 *   y = h / sqrt(mean_j h_j^2 + eps) * w
 *
 * Defined by: "Module 07: Fused operators and FlashAttention", end of the
 * RMSNorm assignment (the kernel also folds in the residual add,
 * rms_norm(x + residual), saving a pass). The norm reads the stored (bf16)
 * h, as the unfused add-then-normalise pair would ("Chapter 5. Operators and
 * runtime", section 5.4.3: fusion keeps the original rounding).
 *
 *   x, r  bf16 [T, D]; w bf16 [D]; y, h bf16 [T, D] (written)
 *   h may alias x or r (in-place update of the residual stream); y must not
 *   alias x, r or h. D, T, eps, alignment and the fixed order of the sum of
 *   squares as rmsnorm_fwd.
 */
attn_status rmsnorm_residual_fwd(const void* x, const void* r, const void* w, void* y, void* h,
                                 int T, int D, float eps, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* attn_status_string(attn_status s);

/*
 * attn_last_device_error - synchronise `stream`, then report and clear the
 * library's device error word: ATTN_ERR_TIMEOUT if a kernel gave up on a
 * bounded wait since the last call, ATTN_ERR_CUDA if the stream reported a
 * CUDA error, else ATTN_OK.
 */
attn_status attn_last_device_error(cudaStream_t stream);

/*
 * attn_kernel_launches - number of kernels this library has launched in this
 * process (all devices, all streams). Used to count launches in a timed region.
 */
unsigned long long attn_kernel_launches(void);

/*
 * attn_selftest_wait_timeout - launch one block whose thread waits on a
 * shared-memory barrier that nothing completes, with a bound of
 * `timeout_us` microseconds (1 .. 1000000). The wait gives up, records
 * ATTN_ERR_TIMEOUT in the device error word and the kernel returns; read it
 * back with attn_last_device_error(). This exercises the same bounded-wait
 * routine the attention kernels use, without hanging the GPU.
 */
attn_status attn_selftest_wait_timeout(int timeout_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H_ */
