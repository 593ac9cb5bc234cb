// tmap.h -- host-side TMA tensor-map encoding (driver entry point fetched at
// run time, so the library links only the CUDA runtime).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace pa {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A 2-D bf16 tensor of `rows` rows x `inner` elements, rows `pitch` elements
// apart (pitch >= inner, pitch * 2 a multiple of 16), read in boxes of
// box_rows x 64 elements (128 bytes) with the 128-byte swizzle. Elements past
// `inner` or `rows` read as zero.
inline bool tmap_bf16_2d_sw128_pitch(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                                     uint64_t pitch, uint32_t box_rows) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A 2-D bf16 tensor of `rows` rows x `inner` contiguous elements, read in
// boxes of box_rows x 64 elements (128 bytes) with the 128-byte swizzle.
inline bool tmap_bf16_2d_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                               uint32_t box_rows) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A (B, H, N, D) bf16 tensor whose element (b, h, n, c) sits at element
// offset b*s_b + h*s_h + n*s_n + c (D contiguous; every stride * 2 a multiple
// of 16), as a 4-D map {D, N, H, B}, read in boxes of 128 tokens x 64
// elements (128 bytes) of one (b, h) with the 128-byte swizzle. Elements past
// D read as zero and are dropped from stores.
inline bool tmap_bf16_bhnd_sw128(CUtensorMap* m, const void* base, uint64_t D, uint64_t N, uint64_t H, uint64_t B,
                                 int64_t s_n, int64_t s_h, int64_t s_b) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {D, N, H, B};
  cuuint64_t strides[3] = {(cuuint64_t)s_n * 2, (cuuint64_t)s_h * 2, (cuuint64_t)s_b * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace pa
