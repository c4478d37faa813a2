// Host-side creation of TMA tensor maps (bf16, 128-byte swizzle) through the driver entry point,
// so the library needs no link-time dependency on libcuda.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor of bf16 rows of 128 elements: dims (128, d1[, d2]) with byte strides s1[, s2];
// box (64, b1[, b2]) lands in shared memory as b1*b2 rows x 128 bytes, 128-byte swizzled.
inline bool make_tmap_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                         const_cast<void*>(base), (const cuuint64_t*)dims,
                         (const cuuint64_t*)strides_bytes, (const cuuint32_t*)box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor of fp32 rows of 128 elements, unswizzled (for TMA reductions from row-major staging):
// dims (128, d1, d2) with byte strides s1, s2; box (b0, b1, b2).
inline bool make_tmap_f32(CUtensorMap* m, const void* base, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base),
                         (const cuuint64_t*)dims, (const cuuint64_t*)strides_bytes,
                         (const cuuint32_t*)box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace msa
