// Declarations shared by the translation units of libsa.so (not part of the ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_api.h"

namespace sa {

// Device error bits (one error word per translation unit that can raise them).
constexpr unsigned int kErrTimeout = 1u;     // a bounded wait expired
constexpr unsigned int kErrBadIndex = 2u;    // CSR column index out of range (skipped)

constexpr int kMaxMaskBlocks = 4096;         // nb limit of the mask builder
constexpr int kMaxRandomBlocks = 64;

// mask_build.cu
int launch_build_mask(const sa_mask_params& p, const float* d_ratio, int32_t* d_row_ptr, int32_t* d_col_idx,
                      cudaStream_t stream);

// attn_fwd.cu
constexpr int kMaxMasks = 8;       // CSRs per call (head groups)
constexpr int kMaxHeadMap = 256;   // heads with a per-head CSR choice
struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int64_t q_strides[3];
  int64_t kv_strides[3];
  int64_t o_strides[3];
  int32_t batch, n_tokens, heads, kv_heads, head_dim, block, causal, csr_shared;
  int32_t n_masks;
  const int32_t* row_ptr[kMaxMasks];
  const int32_t* col_idx[kMaxMasks];
  uint8_t head_mask[kMaxHeadMap];    // query head -> CSR
  float softmax_scale;
};
int launch_attn_fwd(const AttnArgs& a, cudaStream_t stream);
unsigned int attn_read_and_clear_error(cudaStream_t stream);

// offset_attn.cu
constexpr int kMaxOffsets = 64;
constexpr int kMaxWindow = 64;
struct OffsetArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int64_t q_strides[3];
  int64_t kv_strides[3];
  int64_t o_strides[3];
  int32_t batch, n_tokens, heads, kv_heads, head_dim, window, n_offsets;
  int32_t offsets[kMaxOffsets];
  float softmax_scale;
};
int launch_offset_attn_fwd(const OffsetArgs& a, cudaStream_t stream);
unsigned int offset_read_and_clear_error(cudaStream_t stream);

}  // namespace sa
