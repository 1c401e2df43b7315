// Declarations shared by the translation units of libsa.so (not part of the ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_api.h"

namespace sa {

// Device error bits (one error word per translation unit that can raise them).
constexpr unsigned int kErrTimeout = 1u;     // a bounded wait expired
constexpr unsigned int kErrBadIndex = 2u;    // CSR column index out of range (skipped)
constexpr unsigned int kErrCapacity = 4u;    // a device-sized output did not fit its buffer

constexpr int kMaxMaskBlocks = 4096;         // nb limit of the mask builder
constexpr int kMaxRandomBlocks = 64;

// Streaming multiprocessors of the current device (queried per call: a process may drive
// several devices).
inline int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0)
    n = 1;
  return n;
}

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
  void* workspace;                   // caller-owned, 256-byte aligned
  size_t workspace_bytes;
};
int launch_attn_fwd(const AttnArgs& a, cudaStream_t stream);
// Workspace bytes of the forward with room for kFwdDefaultSlots split parts (split-row combine).
constexpr int kFwdDefaultSlots = 608;
size_t attn_fwd_workspace_bytes(int64_t batch, int64_t n_tokens, int64_t heads, int head_dim, int64_t csr_batches,
                                int64_t n_masks);
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

// offset_interp.cu
constexpr int kMaxInterpRungs = 64;
struct InterpArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int64_t q_strides[3];
  int64_t kv_strides[3];
  int64_t o_strides[3];
  int32_t batch, n_tokens, heads, kv_heads, head_dim, window, n_rungs;
  int32_t lo[kMaxInterpRungs];   // floor of the rung distance
  float t[kMaxInterpRungs];      // weight of the farther row
  float softmax_scale;
};
int launch_offset_interp_fwd(const InterpArgs& a, cudaStream_t stream);
unsigned int interp_read_and_clear_error(cudaStream_t stream);

// attn_bwd.cu
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* d_o;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int64_t q_strides[3];    // q and dq
  int64_t kv_strides[3];   // k, v, dk and dv
  int64_t o_strides[3];    // o and d_o
  int32_t batch, n_tokens, heads, kv_heads, head_dim, block, causal, csr_shared;
  int32_t n_masks;                       // CSRs (head groups); query head h uses head_mask[h]
  const int32_t* row_ptr[kMaxMasks];
  const int32_t* col_idx[kMaxMasks];
  int64_t col_capacity[kMaxMasks];       // entries each CSR may hold (n_masks > 1)
  uint8_t head_mask[kMaxHeadMap];
  float softmax_scale;
  void* workspace;
  size_t workspace_bytes;
};
// Workspace layout of the backward: D = rowsum(dO * O) fp32 [batch][heads][n_tokens],
// the transposed CSRs' col_ptr int32 [n_masks][csr_batches][nb + 1] (csr_batches below counts
// all masks) and row_idx int32 [rest], mask m's entries after those of masks < m.
struct BwdWorkspace {
  size_t dvec_off, col_ptr_off, row_idx_off, bytes;
  int64_t row_idx_capacity;
};
BwdWorkspace bwd_workspace_layout(int64_t batch, int64_t n_tokens, int64_t heads, int64_t block,
                                  int64_t csr_batches, int64_t col_capacity);
int launch_attn_bwd(const BwdArgs& a, cudaStream_t stream);
// Device address of the library's own backward scratch (kBwdStaticScratchBytes, 256-byte
// aligned), used by sa_attn_bwd_noalloc.
constexpr size_t kBwdStaticScratchBytes = size_t(16) << 20;
int bwd_static_scratch(void** ptr);
unsigned int bwd_read_and_clear_error(cudaStream_t stream);

}  // namespace sa
