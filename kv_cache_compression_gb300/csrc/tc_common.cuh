// Helpers shared by the tensor-core score/vote kernels (sm_103a). Not part of the public ABI.
#pragma once

#include <cudaTypedefs.h>
#include <stdint.h>

#include "sm100_ptx.cuh"

namespace snapkv {
namespace tc {

// Butterfly reduce-transpose of C per-lane values over the 32 lanes of a warp (max or sum):
// afterwards lane l holds the warp-wide result of row l (C == 32) or of row l/2 (C == 16) in v[0].
template <int C, int O>
__device__ __forceinline__ void butterfly_max(float* v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (C >= 2) {
      constexpr int H = C / 2;
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const float send = upper ? v[k] : v[k + H];
        const float keep = upper ? v[k + H] : v[k];
        v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, O));
      }
      butterfly_max<H, O / 2>(v, lane);
    } else {
      v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], O));
      butterfly_max<1, O / 2>(v, lane);
    }
  }
}

template <int C, int O>
__device__ __forceinline__ void butterfly_sum(float* v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (C >= 2) {
      constexpr int H = C / 2;
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const float send = upper ? v[k] : v[k + H];
        const float keep = upper ? v[k + H] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      butterfly_sum<H, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      butterfly_sum<1, O / 2>(v, lane);
    }
  }
}

// Tiled tensor map of a [heads][rows][d] bf16 tensor: boxes of 64 elements x box_rows rows x 1 head,
// 128-byte swizzle (the layout tcgen05's K-major SW128 descriptors read).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// `stride_rows` (>= rows) is the distance between heads in rows (0: rows).
inline bool make_map(CUtensorMap* map, const void* ptr, int d, int64_t rows, int64_t heads, int box_rows,
                     int64_t stride_rows = 0) {
  if (stride_rows <= 0) stride_rows = rows;
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)stride_rows * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace snapkv
