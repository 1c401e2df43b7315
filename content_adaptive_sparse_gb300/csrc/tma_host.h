// Host-side TMA descriptor encoding for bf16 tensors with layout [batch, tokens, heads, d]
// (d contiguous, other strides arbitrary multiples of 16 bytes).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sa {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Map over a 4-D bf16 tensor (d, heads, tokens, batch) with element strides
// (1, s_head, s_token, s_batch). The box is (box_d, 1, box_rows, 1); the smem image of
// one box is box_rows rows of box_d elements, swizzled with `swz`.
// Returns false if the driver rejects the description.
inline bool encode_bhnd_map(CUtensorMap* map, const void* base, int64_t batch, int64_t tokens, int64_t heads,
                            int64_t d, int64_t s_batch, int64_t s_token, int64_t s_head, uint32_t box_d,
                            uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = get_encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)tokens, (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)(s_head * 2), (cuuint64_t)(s_token * 2), (cuuint64_t)(s_batch * 2)};
  cuuint32_t box[4] = {box_d, 1, box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace sa
