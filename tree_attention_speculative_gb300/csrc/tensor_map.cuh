// Host-side encoding of TMA tensor maps (CUtensorMap) for bf16 and fp32
// tensors with 128-byte swizzle.  The driver entry point is looked up at run time, so the
// library does not link against libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>

namespace ts {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A rank-`rank` tensor map with 128-byte swizzle.  dims[0] is the innermost
// (contiguous) extent; strides_bytes[i] is the byte stride of dimension i+1.
// The box is box[0] x ... elements; box[0] times the element size must be 128
// bytes for the 128-byte swizzle.
inline bool encode_sw128(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank,
                         const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  std::memset(map, 0, sizeof(*map));
  cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, type, (cuuint32_t)rank, const_cast<void*>(base), reinterpret_cast<const cuuint64_t*>(dims),
                  reinterpret_cast<const cuuint64_t*>(strides_bytes), reinterpret_cast<const cuuint32_t*>(box),
                  elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline bool encode_bf16_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                              const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_sw128(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, box);
}

inline bool encode_f32_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                             const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_sw128(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, rank, dims, strides_bytes, box);
}

}  // namespace ts
