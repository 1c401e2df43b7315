/* Plain C client of the library that runs the hot path on the GPU: compiled and run by
 * tests/test_c_abi.py (marked gpu). It reads a problem file written by the test (shape,
 * mask parameters, per-block ratios and the bf16 bits of q, k, v), allocates device memory
 * with the CUDA runtime, calls sa_build_mask and sa_attn_fwd through include/sa_api.h,
 * and writes the CSR, O and LSE to a result file that the test compares with the oracle.
 *
 * Problem file (little-endian): int32 batch, n_tokens, heads, kv_heads, head_dim, block,
 * window_blocks, global_blocks, topk; float32 ratio[batch][nb]; uint16 q[batch][n][heads][d],
 * k and v [batch][n][kv_heads][d].
 * Result file: int32 row_ptr[batch][nb + 1]; int32 nnz; int32 col_idx[nnz];
 * uint16 o[batch][n][heads][d]; float32 lse[batch][heads][n]. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#include <cuda_runtime_api.h>

#include "sa_api.h"

#define TRY(call)                                                         \
  do {                                                                    \
    if ((call) != 0) {                                                    \
      fprintf(stderr, "failed: %s (line %d)\n", #call, __LINE__);         \
      return 1;                                                           \
    }                                                                     \
  } while (0)

static int read_all(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes ? 0 : 1; }
static int write_all(FILE* f, const void* src, size_t bytes) { return fwrite(src, 1, bytes, f) == bytes ? 0 : 1; }

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: abi_gpu problem.bin result.bin\n");
    return 2;
  }
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 2;
  int32_t hdr[9];
  TRY(read_all(in, hdr, sizeof(hdr)));
  const int32_t batch = hdr[0], n = hdr[1], heads = hdr[2], kv_heads = hdr[3], d = hdr[4], b = hdr[5];
  const int32_t nb = n / b;
  const size_t nq = (size_t)batch * n * heads * d, nkv = (size_t)batch * n * kv_heads * d;
  float* h_ratio = (float*)malloc(sizeof(float) * batch * nb);
  uint16_t* h_q = (uint16_t*)malloc(2 * nq);
  uint16_t* h_k = (uint16_t*)malloc(2 * nkv);
  uint16_t* h_v = (uint16_t*)malloc(2 * nkv);
  if (!h_ratio || !h_q || !h_k || !h_v) return 2;
  TRY(read_all(in, h_ratio, sizeof(float) * batch * nb));
  TRY(read_all(in, h_q, 2 * nq));
  TRY(read_all(in, h_k, 2 * nkv));
  TRY(read_all(in, h_v, 2 * nkv));
  fclose(in);

  sa_mask_params p;
  memset(&p, 0, sizeof(p));
  p.mode = SA_MASK_TOPK;
  p.block = b;
  p.n_tokens = n;
  p.batch = batch;
  p.causal = 1;
  p.window_blocks = hdr[6];
  p.global_blocks = hdr[7];
  p.topk = hdr[8];
  int64_t cap = 0;
  TRY(sa_mask_nnz_bound(&p, &cap));

  float *d_ratio = NULL, *d_lse = NULL;
  int32_t *d_row_ptr = NULL, *d_col_idx = NULL;
  void *d_q = NULL, *d_k = NULL, *d_v = NULL, *d_o = NULL, *d_ws = NULL;
  size_t ws_bytes = 0;
  TRY(sa_attn_fwd_workspace_size(batch, n, heads, d, b, batch, 1, &ws_bytes));
  TRY(cudaMalloc(&d_ws, ws_bytes));
  TRY(cudaMalloc((void**)&d_ratio, sizeof(float) * batch * nb));
  TRY(cudaMalloc((void**)&d_row_ptr, sizeof(int32_t) * batch * (nb + 1)));
  TRY(cudaMalloc((void**)&d_col_idx, sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1)));
  TRY(cudaMalloc(&d_q, 2 * nq));
  TRY(cudaMalloc(&d_k, 2 * nkv));
  TRY(cudaMalloc(&d_v, 2 * nkv));
  TRY(cudaMalloc(&d_o, 2 * nq));
  TRY(cudaMalloc((void**)&d_lse, sizeof(float) * batch * heads * n));
  cudaStream_t stream;
  TRY(cudaStreamCreate(&stream));
  TRY(cudaMemcpyAsync(d_ratio, h_ratio, sizeof(float) * batch * nb, cudaMemcpyHostToDevice, stream));
  TRY(cudaMemcpyAsync(d_q, h_q, 2 * nq, cudaMemcpyHostToDevice, stream));
  TRY(cudaMemcpyAsync(d_k, h_k, 2 * nkv, cudaMemcpyHostToDevice, stream));
  TRY(cudaMemcpyAsync(d_v, h_v, 2 * nkv, cudaMemcpyHostToDevice, stream));

  TRY(sa_build_mask(&p, d_ratio, d_row_ptr, d_col_idx, cap, stream));
  const int64_t qs[3] = {(int64_t)n * heads * d, (int64_t)heads * d, d};
  const int64_t kvs[3] = {(int64_t)n * kv_heads * d, (int64_t)kv_heads * d, d};
  TRY(sa_attn_fwd(d_q, d_k, d_v, qs, kvs, qs, batch, n, heads, kv_heads, d, b, 1, d_row_ptr, d_col_idx, 0,
                  1.0f / sqrtf((float)d), d_o, d_lse, d_ws, ws_bytes, stream));
  TRY(sa_device_status(stream));

  int32_t* h_row_ptr = (int32_t*)malloc(sizeof(int32_t) * batch * (nb + 1));
  int32_t* h_col_idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1));
  uint16_t* h_o = (uint16_t*)malloc(2 * nq);
  float* h_lse = (float*)malloc(sizeof(float) * batch * heads * n);
  if (!h_row_ptr || !h_col_idx || !h_o || !h_lse) return 2;
  TRY(cudaMemcpyAsync(h_row_ptr, d_row_ptr, sizeof(int32_t) * batch * (nb + 1), cudaMemcpyDeviceToHost, stream));
  TRY(cudaMemcpyAsync(h_col_idx, d_col_idx, sizeof(int32_t) * (size_t)cap, cudaMemcpyDeviceToHost, stream));
  TRY(cudaMemcpyAsync(h_o, d_o, 2 * nq, cudaMemcpyDeviceToHost, stream));
  TRY(cudaMemcpyAsync(h_lse, d_lse, sizeof(float) * batch * heads * n, cudaMemcpyDeviceToHost, stream));
  TRY(cudaStreamSynchronize(stream));

  FILE* out = fopen(argv[2], "wb");
  if (!out) return 2;
  const int32_t nnz = h_row_ptr[batch * (nb + 1) - 1];
  TRY(write_all(out, h_row_ptr, sizeof(int32_t) * batch * (nb + 1)));
  TRY(write_all(out, &nnz, sizeof(nnz)));
  TRY(write_all(out, h_col_idx, sizeof(int32_t) * (size_t)nnz));
  TRY(write_all(out, h_o, 2 * nq));
  TRY(write_all(out, h_lse, sizeof(float) * batch * heads * n));
  fclose(out);
  cudaFree(d_ratio);
  cudaFree(d_row_ptr);
  cudaFree(d_col_idx);
  cudaFree(d_q);
  cudaFree(d_k);
  cudaFree(d_v);
  cudaFree(d_o);
  cudaFree(d_lse);
  cudaFree(d_ws);
  cudaStreamDestroy(stream);
  printf("c gpu ok\n");
  return 0;
}
