// tmap.cu - the TMA tensor maps of the prefill and backward kernels (host side only).
//
// The bf16 operand tiles those kernels stream are boxes of a [Z, rows, D] tensor (Z = batch x
// heads): 128 rows x 64 columns with the 128-byte swizzle for the single-CTA kernels; for the
// CTA-pair prefill also 64 rows x 64 columns (half a K tile) and 128 rows x 32 columns with the
// 64-byte swizzle (half a V tile at d = 64). The swizzle is the one the tcgen05 shared-memory
// descriptors name; rows past the end of a head read as zero (the kernels mask them).
#include "pair.cuh"

namespace gb300 {

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime (no link-time
// dependency on libcuda).
static PFN_encodeTiled get_encode_fn() {
  static PFN_encodeTiled fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(ptr);
  }
  return fn;
}

bool encode_bf16_box_map(CUtensorMap* map, const void* base, int D, int rows, int Z, int box_cols, int box_rows,
                         int swizzle_bytes) {
  PFN_encodeTiled enc = get_encode_fn();
  if (enc == nullptr) return false;
  if (swizzle_bytes != 64 && swizzle_bytes != 128) return false;
  if (box_cols * 2 > swizzle_bytes) return false;  // the inner box extent must fit the swizzle span
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(Z)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_tile_map(CUtensorMap* map, const void* base, int D, int rows, int Z) {
  return encode_bf16_box_map(map, base, D, rows, Z, 64, 128, 128);
}

}  // namespace gb300
