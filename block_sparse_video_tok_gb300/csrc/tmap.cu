// tmap.cu -- TMA tensor maps of the operands the two tensor-core kernels load and the dQ
// accumulator the backward reduces into.  Maps are encoded per call on the host (nothing is
// cached between calls), through the driver entry point of cuTensorMapEncodeTiled.
// Every map uses 128-byte rows of 64 two-byte elements in the 128-byte swizzle that the UMMA
// shared-memory descriptors of the kernels expect, except the dQ accumulator's (fp32, no
// swizzle), which only the TMA reduce-add touches.
#include <cudaTypedefs.h>

#include "vsa_internal.cuh"

namespace vsa {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

CUtensorMapDataType two_byte_type(bool bf16) {
  return bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

}  // namespace

cudaError_t make_tmap_tiles_t(CUtensorMap* map, const void* ptr, long rows, int tiles) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {64u, static_cast<cuuint64_t>(rows) * 2u};
  const cuuint64_t gstride[1] = {64u * sizeof(__half)};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(HEAD_DIM * tiles)};
  const cuuint32_t estride[2] = {1u, 1u};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), gdim,
                      gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_rows128_f32(CUtensorMap* map, const void* ptr, long rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(HEAD_DIM), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(HEAD_DIM) * sizeof(float)};
  const cuuint32_t box[2] = {32u, 64u};
  const cuuint32_t estride[2] = {1u, 1u};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), gdim,
                      gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_rows128_f16(CUtensorMap* map, const void* ptr, long rows, bool bf16) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(HEAD_DIM), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(HEAD_DIM) * sizeof(__half)};
  const cuuint32_t box[2] = {64u, 64u};
  const cuuint32_t estride[2] = {1u, 1u};
  CUresult r = encode(map, two_byte_type(bf16), 2, const_cast<void*>(ptr), gdim, gstride, box,
                      estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_rows128_f16_halves(CUtensorMap* map, const void* ptr, long rows,
                                         int box_rows, bool bf16) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t gdim[3] = {64u, static_cast<cuuint64_t>(rows), 2u};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(HEAD_DIM) * sizeof(__half),
                                 64u * sizeof(__half)};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 2u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  CUresult r = encode(map, two_byte_type(bf16), 3, const_cast<void*>(ptr), gdim, gstride, box,
                      estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace vsa
