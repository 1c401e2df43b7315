/*
 * sa_api.h - C ABI of the GB300 (sm_103a) sparse-graph attention library (libsa.so).
 *
 * The library computes attention restricted to a sparse key graph:
 *   - block graphs given as a CSR list of key blocks per query block, built on the GPU
 *     from per-block compression ratios ("Parameter-free Adaptive Sparse Attention via
 *     Compression-Based Content Selection", section 3.1 Eq. 1-2, section 3.2 Eq. 3,
 *     Appendix B Algorithm 1) or from the BigBird window/global/random pattern
 *     ("BigBird", section 2 "Derivation");
 *   - token-granular graphs made of a dense window plus alpha-scaled Fibonacci offsets
 *     ("Depth-Staggered Fibonacci Spacing for Sparse Attention", section 2 "Method").
 *
 * Conventions (all entry points):
 *   - Device pointers are marked d_*, host pointers h_*; q/k/v/o/lse are device memory.
 *   - The caller owns all memory. The library allocates no device memory; its only
 *     device state is static arrays in the module: the device error words (see
 *     sa_device_status) and the 16 MiB scratch of sa_attn_bwd_noalloc. Calls that need
 *     scratch take a caller workspace (sa_attn_fwd, sa_attn_bwd).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). Argument errors are returned synchronously before anything is launched.
 *   - Tensors q, k, v, o are bf16 with layout [batch, tokens, heads, head_dim]:
 *     head_dim contiguous, and strides[3] = {batch, token, head} strides in ELEMENTS.
 *     Every stride times 2 bytes and every base pointer must be a multiple of 16 bytes.
 *     LSE is fp32 [batch, heads, tokens], contiguous, natural logarithm.
 *   - Attention: s_ij = softmax_scale * <q_i, k_j> over the allowed keys j of query i;
 *     LSE_i = ln sum_j exp(s_ij); O_i = sum_j exp(s_ij - LSE_i) v_j. A query with no
 *     allowed key gets O_i = 0 and LSE_i = -inf. Query head h reads key/value head
 *     h / (heads / kv_heads) (grouped-query attention).
 *   - There is no CPU fallback: without a usable sm_103a device every compute entry
 *     point returns SA_ERR_CUDA or SA_ERR_UNSUPPORTED.
 */
#ifndef SA_API_H
#define SA_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = -1, /* null pointer, negative size, inconsistent shapes        */
  SA_ERR_UNSUPPORTED = -2, /* valid request outside the supported shapes / modes      */
  SA_ERR_CAPACITY = -3,    /* caller buffer too small (e.g. col_idx capacity)         */
  SA_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed             */
  SA_ERR_TIMEOUT = -5,     /* a bounded device-side wait expired (sa_device_status)   */
  SA_ERR_DEVICE = -6       /* a kernel found invalid data, e.g. an out-of-range CSR   */
} sa_status;

typedef enum {
  /* Compression-guided, causal. Row I = window W(I) = [max(0, I-w+1), I] (w blocks
   * counting the diagonal) u global key blocks {J < g, J <= I} u the top-k blocks of
   * C(I) = [0, I] minus window and globals, ordered by ratio descending then block
   * index ascending. The top-k rule is the workload's reading of "literal" blocks;
   * the page's own rule is SA_MASK_LITERAL_MEAN. */
  SA_MASK_TOPK = 0,
  /* BigBird, bidirectional ("BigBird", section 2): global rows I < g attend to every
   * block; other rows attend to window [I - w/2, I - w/2 + w - 1], the g global
   * blocks, and r random blocks drawn without replacement from the remaining blocks
   * with the Philox4x64-10 stream (Salmon et al., SC'11) keyed by `seed`: draw t of
   * row I takes word p = I*r + t of the stream
   *   word(p) = Philox4x64_10(counter = (p/4 + 1, 0, 0, 0), key = (seed, 0))[p % 4]
   * and picks index ((word >> 32) * |A|) >> 32 of the ascending remaining list A. */
  SA_MASK_BIGBIRD = 1,
  /* Every block J <= I (causal) or every block (bidirectional). */
  SA_MASK_FULL = 2,
  /* "Parameter-free Adaptive Sparse Attention ...", Eq. 2-3 / Algorithm 1: block i is
   * literal iff r_i > mean(r); M = {|I-J| <= w} u identity u {literal I and J,
   * |I-J| > w}; causal keeps J <= I. global_blocks must be 0. sa_mask_params.components
   * keeps a part of M (Appendix B "Head-specific mask distribution"). */
  SA_MASK_LITERAL_MEAN = 3
} sa_mask_mode;

/* Parts of the LITERAL_MEAN mask besides the identity (bit flags; 0 = both = full M):
 * local heads use M_local u I, long-range heads M_lit u I, hybrid heads the full M. */
enum { SA_LITERAL_LOCAL = 1, SA_LITERAL_PAIRS = 2 };

typedef struct {
  int32_t mode;          /* sa_mask_mode                                               */
  int32_t block;         /* b: 32, 64 or 128 tokens per block                           */
  int32_t n_tokens;      /* N, a multiple of b; nb = N / b <= 4096                      */
  int32_t batch;         /* number of sequences (one CSR per sequence)                  */
  int32_t causal;        /* 1 = causal (TOPK requires 1, BIGBIRD requires 0)            */
  int32_t window_blocks; /* w (meaning per mode, see sa_mask_mode)                      */
  int32_t global_blocks; /* g                                                           */
  int32_t topk;          /* k (TOPK)                                                    */
  int32_t random_blocks; /* r (BIGBIRD), <= 64                                          */
  int32_t components;    /* LITERAL_MEAN: SA_LITERAL_* flags, 0 = all; other modes: 0   */
  uint64_t seed;         /* Philox key (BIGBIRD)                                        */
} sa_mask_params;

/* Upper bound on the number of CSR entries sa_build_mask writes for these parameters
 * (exact for TOPK, BIGBIRD, FULL and the LOCAL part of LITERAL_MEAN, whose row lengths
 * do not depend on the ratios; the all-literal worst case for the other LITERAL_MEAN
 * parts). Host only; no device work. */
int sa_mask_nnz_bound(const sa_mask_params* params, int64_t* h_nnz);

/* Build the block CSR of every sequence on the GPU.
 *   d_ratio   : fp32 [batch][nb] per-block compression ratios (Eq. 1); finite values.
 *               Read by TOPK and LITERAL_MEAN, may be NULL for the other modes.
 *   d_row_ptr : int32 [batch][nb + 1], written. Offsets are absolute into d_col_idx:
 *               sequence s occupies [row_ptr[s][0], row_ptr[s][nb]), and
 *               row_ptr[s][0] == row_ptr[s-1][nb].
 *   d_col_idx : int32 [col_capacity], written; each row ascending and duplicate-free.
 * Returns SA_ERR_CAPACITY (nothing launched) if col_capacity < sa_mask_nnz_bound.
 * The output is a pure function of (params, ratios): bit-identical on every run. */
int sa_build_mask(const sa_mask_params* params, const float* d_ratio, int32_t* d_row_ptr, int32_t* d_col_idx,
                  int64_t col_capacity, void* stream);

/* Workspace bytes of sa_attn_fwd / sa_attn_fwd_heads for these shapes: the launch's work
 * counter, the split plan and room for 608 partial results of split items (about 33 KB each
 * at head_dim 64, 66 KB at 128). csr_batches is 1 for a shared CSR, else batch; n_masks is
 * the number of CSRs (1 for sa_attn_fwd). Host only. */
int sa_attn_fwd_workspace_size(int32_t batch, int32_t n_tokens, int32_t heads, int32_t head_dim, int32_t block,
                               int32_t csr_batches, int32_t n_masks, size_t* h_bytes);

/* Block-sparse attention forward over a block CSR (tcgen05 / TMEM / TMA kernel).
 * Token pair (i, j) is attended iff blk(j) is in row(blk(i)) and, if causal, j <= i
 * ("Parameter-free Adaptive Sparse Attention ...", section 3.4 "Block-to-token
 * expansion"; "BigBird", section 3: a production kernel gathers the selected keys
 * instead of masking N x N scores).
 *   q [batch, n_tokens, heads, head_dim], k/v [batch, n_tokens, kv_heads, head_dim]
 *   q_strides / kv_strides / o_strides : element strides {batch, token, head}
 *   head_dim in {32, 64, 128}; block in {32, 64, 128}; n_tokens % block == 0;
 *   heads % kv_heads == 0.
 *   d_row_ptr / d_col_idx : CSR as written by sa_build_mask. If csr_shared != 0 every
 *   sequence uses the CSR of sequence 0, else sequence s uses row_ptr[s][*].
 *   Column indices must lie in [0, nb); rows must be ascending without duplicates.
 *   An out-of-range index is skipped and reported as SA_ERR_DEVICE by
 *   sa_device_status.
 *   o : bf16 output, lse : fp32 [batch, heads, n_tokens].
 *   workspace : caller-owned device memory, 256-byte aligned, at least 256 bytes; its
 *   contents on entry do not matter. It holds the launch's work counter, so launches in
 *   flight at the same time need separate workspaces. With
 *   sa_attn_fwd_workspace_size bytes, a launch with few work items (128-row query tiles
 *   x heads x sequences: fewer than four per SM at head_dim 32 or 64, fewer than one per SM
 *   at 128) whose longest key list exceeds 1.25x an even share splits the items whose key
 *   lists are longest into parts of equal key-tile counts, writes each part's O and LSE to
 *   the workspace and merges them (LSE = ln sum exp LSE_p, O = sum exp(LSE_p - LSE) O_p), so
 *   that a few long rows do not leave SMs idle; a smaller workspace (>= 256 bytes) never
 *   splits. */
int sa_attn_fwd(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch, int32_t n_tokens,
                int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t block, int32_t causal,
                const int32_t* d_row_ptr, const int32_t* d_col_idx, int32_t csr_shared, float softmax_scale,
                void* o, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* sa_attn_fwd with one block CSR per head group ("Parameter-free Adaptive Sparse
 * Attention ...", Appendix B "Head-specific mask distribution": local, long-range and
 * hybrid heads read different parts of the block mask).
 *   n_masks      : number of CSRs, 1 .. 8.
 *   h_row_ptrs   : host array [n_masks] of device pointers, each a row_ptr as written
 *                  by sa_build_mask for the same batch, n_tokens and block.
 *   h_col_idxs   : host array [n_masks] of the matching device col_idx pointers.
 *   h_head_mask  : host int32 [heads]; query head h uses CSR h_head_mask[h], in
 *                  [0, n_masks). heads <= 256.
 * The host arrays are read before the call returns. Every other argument is as in
 * sa_attn_fwd (csr_shared applies to every CSR; the workspace size query takes n_masks). */
int sa_attn_fwd_heads(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                      const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch, int32_t n_tokens,
                      int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t block, int32_t causal,
                      int32_t n_masks, const int32_t* const* h_row_ptrs, const int32_t* const* h_col_idxs,
                      const int32_t* h_head_mask, int32_t csr_shared, float softmax_scale, void* o, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of sa_attn_bwd: D = rowsum(dO * O) (fp32 [batch][heads][n_tokens])
 * and the transposed CSR (int32 [csr_batches][nb + 1] plus col_capacity indices, where
 * col_capacity >= the number of CSR entries, e.g. sa_mask_nnz_bound). csr_batches is
 * 1 for a shared CSR, else batch. Host only. */
int sa_attn_bwd_workspace_size(int32_t batch, int32_t n_tokens, int32_t heads, int32_t block, int32_t csr_batches,
                               int64_t col_capacity, size_t* h_bytes);

/* Block-sparse attention backward over the block CSR of sa_attn_fwd: the gradients of
 * sum(dO * O) with respect to q, k and v. With P_ij = exp(s_ij - LSE_i) over the visible
 * keys and D_i = sum_d dO_id O_id:
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (<dO_i, v_j> - D_i),
 *   dQ_i = softmax_scale * sum_j dS_ij k_j,  dK_j = softmax_scale * sum_i dS_ij q_i
 * (dK / dV of a key/value head sum over its query heads). The pages train through these
 * masks ("Parameter-free Adaptive Sparse Attention ...", section 4.1; "Depth-Staggered
 * Fibonacci Spacing ...", section 3).
 *   o, lse : the forward's outputs for the same inputs (o with o_strides, lse contiguous
 *            [batch][heads][n_tokens], 16-byte aligned).
 *   d_o    : upstream gradient, bf16, layout and strides of o.
 *   dq     : bf16 with q_strides; dk, dv : bf16 with kv_strides; all written.
 *   workspace : device memory of at least sa_attn_bwd_workspace_size bytes, 256-byte
 *            aligned, owned by the caller; its contents on entry do not matter.
 * Shapes, CSR and error behaviour as in sa_attn_fwd; a CSR with more entries than the
 * workspace holds is reported by sa_device_status as SA_ERR_CAPACITY. */
int sa_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
                const int64_t q_strides[3], const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch,
                int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t block, int32_t causal,
                const int32_t* d_row_ptr, const int32_t* d_col_idx, int32_t csr_shared, float softmax_scale,
                void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream);

/* sa_attn_bwd with one block CSR per head group, the backward of sa_attn_fwd_heads.
 *   n_masks, h_row_ptrs, h_col_idxs, h_head_mask : as in sa_attn_fwd_heads.
 *   h_col_capacities : host int64 [n_masks], entries each CSR may hold (its col_idx size);
 *                      read only when n_masks > 1.
 * The workspace is sa_attn_bwd_workspace_size(batch, n_tokens, heads, block,
 * csr_batches * n_masks, sum of h_col_capacities) bytes. Every other argument is as in
 * sa_attn_bwd, which is this call with one CSR. */
int sa_attn_bwd_heads(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
                      const int64_t q_strides[3], const int64_t kv_strides[3], const int64_t o_strides[3],
                      int32_t batch, int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim,
                      int32_t block, int32_t causal, int32_t n_masks, const int32_t* const* h_row_ptrs,
                      const int32_t* const* h_col_idxs, const int64_t* h_col_capacities,
                      const int32_t* h_head_mask, int32_t csr_shared, float softmax_scale, void* dq, void* dk,
                      void* dv, void* workspace, size_t workspace_bytes, void* stream);

/* sa_attn_bwd for callers that cannot allocate device memory. The pages have no
 * counterpart of this call; it exists for the library's users. Some callers must not call
 * cudaMalloc at this point: a plugin whose host application owns every device allocation,
 * a service that allocates only at start-up so that its memory use stays fixed, or a
 * latency-bound caller for whom cudaMalloc's implicit device synchronisation is too costly.
 * This call needs no workspace from them: its scratch (D and the transposed CSR) is a
 * 16 MiB array inside the library, of which every device that loads the library holds one
 * copy until the process exits. The call itself allocates nothing.
 *   col_capacity : entries the CSR may hold, as in sa_attn_bwd_workspace_size. If the
 *                  scratch for these shapes exceeds 16 MiB the call returns
 *                  SA_ERR_CAPACITY before any launch. A col_capacity below the CSR's real
 *                  entry count is not seen on the host: the kernels clamp the transposed
 *                  lists to it (dK and dV are then incomplete) and only sa_device_status
 *                  reports it, as SA_ERR_CAPACITY.
 *   The first call on a device looks up that device's copy of the array (with the device
 *   current) and keeps its address; make that first call before any stream capture.
 *   Every call shares the one array, which keeps the previous call's contents (the call
 *   rewrites every part it reads). Calls that overlap on the GPU race on it: serialise
 *   them on one stream, or synchronise between streams.
 * Every other argument, and the outputs, as in sa_attn_bwd. */
int sa_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
                        const int64_t q_strides[3], const int64_t kv_strides[3], const int64_t o_strides[3],
                        int32_t batch, int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim,
                        int32_t block, int32_t causal, const int32_t* d_row_ptr, const int32_t* d_col_idx,
                        int64_t col_capacity, int32_t csr_shared, float softmax_scale, void* dq, void* dk, void* dv,
                        void* stream);

/* Token-granular window-plus-Fibonacci-offset attention forward ("Depth-Staggered
 * Fibonacci Spacing for Sparse Attention", section 2 "Method" and "Attended set"): query i
 * attends to keys
 *   { i - delta : delta in {0, ..., window} u D, i - delta >= 0 }   (a set),
 * where D = { round_half_even(alpha * f_k) } over the Fibonacci rungs f = 1, 2, 3, 5, ...
 * (the first n_rungs of them; n_rungs == 0: every f_k <= n_tokens; the page uses 15) and
 * alpha = alpha_num / alpha_den > 0 is the layer's scale as an exact fraction (the page's
 * per-layer linear stagger, see sa_layer_alpha). D is computed on the host exactly as
 * sa_fib_offsets returns it.
 *   head_dim 32, 64 or 128 (the page's model: 8 heads of 64); window in [0, 64]; at most 64
 *   distinct offsets beyond the window; n_tokens <= 65535 * 64 and batch * heads < 2^31
 *   (else SA_ERR_UNSUPPORTED); other arguments as in sa_attn_fwd. The kernel's copy waits
 *   are bounded: an expired wait leaves O and LSE incomplete and is reported by
 *   sa_device_status as SA_ERR_TIMEOUT. */
int sa_offset_attn_fwd(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                       const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch, int32_t n_tokens,
                       int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t window, int32_t alpha_num,
                       int32_t alpha_den, int32_t n_rungs, float softmax_scale, void* o, float* lse, void* stream);

/* sa_offset_attn_fwd over an explicit offset set (any ladder, e.g. sa_pow2_offsets):
 * query i attends to { i - delta : delta in {0, ..., window} u h_offsets, i - delta >= 0 }.
 *   h_offsets : host int32[n_offsets], strictly ascending, each > window and
 *               < n_tokens; n_offsets <= 64. Read before the call returns.
 * Every other argument, limit and error as in sa_offset_attn_fwd. */
int sa_offset_attn_fwd_list(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                            const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch,
                            int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t window,
                            const int32_t* h_offsets, int32_t n_offsets, float softmax_scale, void* o, float* lse,
                            void* stream);

/* Window plus interpolated-rung attention forward ("Depth-Staggered Fibonacci Spacing ...",
 * section 2 "Attended set"; the interpolated gather of a continuous alpha). Rung k has the
 * distance d_k = alpha * f_k (IEEE double product) over the Fibonacci rungs (ladder 0) or
 * the power-of-2 rungs (ladder 1), the first n_rungs of them (n_rungs > 0) or every rung
 * f_k <= n_tokens (n_rungs == 0). With lo = floor(d_k) and t = d_k - lo, query i sees
 *   the window rows i - delta, delta = 0..window, i - delta >= 0, and
 *   for every rung with i - d_k >= 0 the key (1 - t) k[i - lo] + t k[i - lo - 1] and the
 *   value (1 - t) v[i - lo] + t v[i - lo - 1]
 * (a rung with an integer distance inside the window is the window row itself and is not
 * counted twice). head_dim 32, 64 or 128; window in [0, 64]; at most 64 rungs remain;
 * n_tokens <= 65535 * 64; other arguments, size limits and the bounded-wait report as in
 * sa_offset_attn_fwd. alpha must be finite and > 0. */
int sa_offset_attn_interp_fwd(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                              const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch,
                              int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t window,
                              double alpha, int32_t n_rungs, int32_t ladder, float softmax_scale, void* o, float* lse,
                              void* stream);

/* Distinct offsets d_k = round_half_even(alpha * f_k), alpha = alpha_num / alpha_den > 0,
 * over Fibonacci rungs f = 1, 2, 3, 5, 8, ... ("Depth-Staggered Fibonacci Spacing ...",
 * section 2: K = 15 rungs up to 987). n_rungs > 0 takes the first n_rungs rungs;
 * n_rungs == 0 takes every rung f_k <= n_tokens. Only offsets with
 * window < d < n_tokens are returned (the window already covers the others), ascending,
 * in h_out[0 .. *h_count). Host only. Returns SA_ERR_CAPACITY if capacity is short. */
int sa_fib_offsets(int32_t alpha_num, int32_t alpha_den, int32_t n_rungs, int32_t window, int32_t n_tokens,
                   int32_t* h_out, int32_t capacity, int32_t* h_count);

/* sa_fib_offsets over the power-of-2 control base f = 1, 2, 4, 8, ... (same section,
 * "Control base": reach-matched to the Fibonacci base, 11 rungs up to 1024). */
int sa_pow2_offsets(int32_t alpha_num, int32_t alpha_den, int32_t n_rungs, int32_t window, int32_t n_tokens,
                    int32_t* h_out, int32_t capacity, int32_t* h_count);

/* Per-layer scale of the staggered schedules (same page, section 2 "The per-layer
 * scalar"): the linear ramp a_i = lo + (hi - lo) * i / (layers - 1), lo = lo_num/lo_den,
 * hi = hi_num/hi_den; layer `layer` takes a_i with i = (stride * layer) mod layers
 * (stride 1: linear stagger; stride 7 with 16 layers: the coprime stagger). Writes the
 * reduced fraction to *h_num / *h_den. stride must be >= 1 and coprime to layers.
 * Host only. */
int sa_layer_alpha(int32_t layer, int32_t layers, int32_t lo_num, int32_t lo_den, int32_t hi_num, int32_t hi_den,
                   int32_t stride, int32_t* h_num, int32_t* h_den);

/* Per-block compression ratios r_i = |zlib(x[i*b:(i+1)*b], level)| / b of a host byte
 * array h_bytes [batch][n_tokens] ("Parameter-free Adaptive Sparse Attention ...",
 * section 3.1 Eq. 1; zlib framing instead of gzip shifts every length by the same
 * constant). Writes h_ratio fp32 [batch][n_tokens / block]. Runs on up to n_threads
 * host threads (0 = hardware concurrency). Uses the system zlib (libz.so.1) loaded at
 * run time; returns SA_ERR_UNSUPPORTED if it cannot be loaded. Host only. */
int sa_block_ratios(const uint8_t* h_bytes, int32_t batch, int32_t n_tokens, int32_t block, int32_t level,
                    float* h_ratio, int32_t n_threads);

/* The whole mask step of one batch from host bytes ("Parameter-free Adaptive Sparse
 * Attention ...", section 3.1 Eq. 1 and section 3.4: the ratios of one 8192-byte sequence
 * take well under a millisecond on the host): the per-block ratios of h_bytes
 * [batch][n_tokens] are computed on up to n_threads host threads (0 = hardware
 * concurrency) into h_ratio [batch][nb] (as sa_block_ratios), then the upload of h_ratio
 * into d_ratio and the mask build (as sa_build_mask) are enqueued on `stream`.
 * The host part runs in the calling thread before the call returns, so GPU work that the
 * caller enqueued earlier (for example the uploads of Q, K and V on another stream, or the
 * previous batch's attention) overlaps it. TOPK and LITERAL_MEAN modes only (the modes
 * that read ratios). h_ratio must stay unchanged until the upload has run (use pinned
 * memory for an asynchronous copy; a pageable buffer is copied before the call returns).
 * Errors as in sa_block_ratios and sa_build_mask. */
int sa_build_mask_from_bytes(const sa_mask_params* params, const uint8_t* h_bytes, int32_t zlib_level,
                             int32_t n_threads, float* h_ratio, float* d_ratio, int32_t* d_row_ptr,
                             int32_t* d_col_idx, int64_t col_capacity, void* stream);

/* Synchronises `stream`, then reads and clears the library's device error words.
 * Returns SA_OK, SA_ERR_TIMEOUT (a bounded wait expired; the kernel unwound and its
 * outputs are undefined), SA_ERR_DEVICE (invalid CSR data was skipped) or
 * SA_ERR_CAPACITY (a device-sized structure did not fit the caller's workspace).
 * The error words belong to the current device, not to a stream: every launch on any
 * stream of the device sets them, and this call clears them. To attribute an error to
 * the right calls, synchronise every stream that launched library work before calling
 * it. */
int sa_device_status(void* stream);

/* Self-test of the failure path: launches a one-thread kernel that waits on a barrier
 * nothing completes. The wait gives up after the library's wait limit (1 s), records a
 * timeout and the kernel exits; the next sa_device_status returns SA_ERR_TIMEOUT, and the
 * context stays usable. No memory is touched. */
int sa_selftest_bounded_wait(void* stream);

/* Human-readable name of a status code (static string). */
const char* sa_status_string(int status);

/* Library ABI version, currently 1. */
int sa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SA_API_H */
