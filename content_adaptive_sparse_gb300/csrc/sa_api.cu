// Host side of the C ABI declared in include/sa_api.h: argument validation, the
// closed-form CSR size bound, Fibonacci offsets, host zlib ratios and kernel dispatch.
#include <dlfcn.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <numeric>
#include <atomic>
#include <condition_variable>
#include <functional>
#include <memory>
#include <mutex>
#include <thread>
#include <vector>

#include <cuda_runtime.h>

#include "sa_api.h"
#include "ptx_sm100.cuh"
#include "sa_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool strides_ok(const int64_t s[3]) {
  for (int i = 0; i < 3; ++i)
    if (s[i] <= 0 || (s[i] * 2) % 16 != 0) return false;
  return true;
}

// The kernels are built for sm_103a only (GB300); refuse any other device up front.
bool device_ok() {
  static int cached[64] = {0};   // 0 unknown, 1 ok, 2 not ok
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
  if (dev < 64 && cached[dev]) return cached[dev] == 1;
  int major = 0, minor = 0;
  const bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
                  major == 10 && minor == 3;
  if (dev < 64) cached[dev] = ok ? 1 : 2;
  return ok;
}

int64_t nnz_bound(const sa_mask_params& p) {
  const int64_t nb = p.n_tokens / p.block;
  int64_t per_seq = 0;
  for (int64_t I = 0; I < nb; ++I) {
    switch (p.mode) {
      case SA_MASK_TOPK: {
        const int64_t n_w = std::min<int64_t>(p.window_blocks, I + 1);
        const int64_t n_g = std::max<int64_t>(0, std::min<int64_t>(p.global_blocks, I - p.window_blocks + 1));
        const int64_t n_c = std::max<int64_t>(0, I - p.window_blocks + 1 - p.global_blocks);
        per_seq += n_w + n_g + std::min<int64_t>(p.topk, n_c);
        break;
      }
      case SA_MASK_FULL:
        per_seq += p.causal ? I + 1 : nb;
        break;
      case SA_MASK_BIGBIRD: {
        if (I < p.global_blocks) {
          per_seq += nb;
          break;
        }
        const int64_t g = std::min<int64_t>(p.global_blocks, nb);
        const int64_t wlo_raw = I - p.window_blocks / 2;
        const int64_t lo = std::max<int64_t>(0, wlo_raw), hi = std::min<int64_t>(nb - 1, wlo_raw + p.window_blocks - 1);
        const int64_t n_w = std::max<int64_t>(0, hi - lo + 1);
        const int64_t n_wg = std::max<int64_t>(0, std::min<int64_t>(hi, g - 1) - lo + 1);
        const int64_t n_union = n_w + g - n_wg;
        per_seq += n_union + std::min<int64_t>(p.random_blocks, nb - n_union);
        break;
      }
      case SA_MASK_LITERAL_MEAN:
        if (p.components == SA_LITERAL_LOCAL)   // the band alone
          per_seq += (p.causal ? I : std::min<int64_t>(nb - 1, I + p.window_blocks)) -
                     std::max<int64_t>(0, I - p.window_blocks) + 1;
        else
          per_seq += p.causal ? I + 1 : nb;     // every block literal
        break;
    }
  }
  return per_seq * p.batch;
}

int check_mask_params(const sa_mask_params* p) {
  if (!p) return SA_ERR_INVALID_ARG;
  if (p->mode < SA_MASK_TOPK || p->mode > SA_MASK_LITERAL_MEAN) return SA_ERR_INVALID_ARG;
  if (p->block <= 0 || p->n_tokens <= 0 || p->batch <= 0 || p->n_tokens % p->block != 0) return SA_ERR_INVALID_ARG;
  if (p->window_blocks < 0 || p->global_blocks < 0 || p->topk < 0 || p->random_blocks < 0) return SA_ERR_INVALID_ARG;
  if (p->components < 0 || p->components > (SA_LITERAL_LOCAL | SA_LITERAL_PAIRS)) return SA_ERR_INVALID_ARG;
  if (p->components != 0 && p->mode != SA_MASK_LITERAL_MEAN) return SA_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return SA_ERR_INVALID_ARG;
  if (p->n_tokens / p->block > sa::kMaxMaskBlocks) return SA_ERR_UNSUPPORTED;
  if (p->mode == SA_MASK_TOPK && !p->causal) return SA_ERR_UNSUPPORTED;
  if (p->mode == SA_MASK_BIGBIRD && p->causal) return SA_ERR_UNSUPPORTED;
  if (p->mode == SA_MASK_BIGBIRD && p->random_blocks > sa::kMaxRandomBlocks) return SA_ERR_UNSUPPORTED;
  if (p->mode == SA_MASK_LITERAL_MEAN && p->global_blocks != 0) return SA_ERR_UNSUPPORTED;
  return SA_OK;
}

// Self-test of the bounded waits: one thread waits on an mbarrier that nothing arrives on.
// After the wait limit the wait gives up, sets the CTA's abort flag and the timeout bit.
__device__ unsigned int g_selftest_err;

__global__ void bounded_wait_selftest_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sa::mbar_init(&bar, 1);
    abort_flag = 0;
    sa::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) sa::mbar_wait(&bar, 0, &abort_flag, &g_selftest_err, sa::kErrTimeout);
}

int check_attn_common(const void* q, const void* k, const void* v, const int64_t qs[3], const int64_t kvs[3],
                      const int64_t os[3], int32_t batch, int32_t n_tokens, int32_t heads, int32_t kv_heads, void* o,
                      float* lse) {
  if (!q || !k || !v || !qs || !kvs || !os || !o || !lse) return SA_ERR_INVALID_ARG;
  if (batch <= 0 || n_tokens <= 0 || heads <= 0 || kv_heads <= 0 || heads % kv_heads != 0) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SA_ERR_UNSUPPORTED;
  if (!strides_ok(qs) || !strides_ok(kvs) || !strides_ok(os)) return SA_ERR_UNSUPPORTED;
  return SA_OK;
}

// ---------------------------------------------------------------- zlib (loaded at run time)

// The public zlib stream record (zlib.h's z_stream, LP64 layout); declared here so that the
// library builds where only the zlib run-time library is installed.
struct ZStream {
  const unsigned char* next_in;
  unsigned int avail_in;
  unsigned long total_in;
  unsigned char* next_out;
  unsigned int avail_out;
  unsigned long total_out;
  const char* msg;
  void* state;
  void* zalloc;
  void* zfree;
  void* opaque;
  int data_type;
  unsigned long adler;
  unsigned long reserved;
};

typedef unsigned long (*compress_bound_fn)(unsigned long);
typedef const char* (*zlib_version_fn)(void);
typedef int (*deflate_init2_fn)(ZStream*, int, int, int, int, int, const char*, int);
typedef int (*deflate_fn)(ZStream*, int);
typedef int (*deflate_reset_fn)(ZStream*);
typedef int (*deflate_end_fn)(ZStream*);

struct Zlib {
  compress_bound_fn bound = nullptr;
  zlib_version_fn version = nullptr;
  deflate_init2_fn init2 = nullptr;
  deflate_fn deflate = nullptr;
  deflate_reset_fn reset = nullptr;
  deflate_end_fn end = nullptr;
  bool ok() const { return bound && version && init2 && deflate && reset && end; }
};

const Zlib& zlib() {
  static const Zlib z = [] {
    Zlib r;
    void* h = dlopen("libz.so.1", RTLD_NOW | RTLD_LOCAL);
    if (!h) h = dlopen("libz.so", RTLD_NOW | RTLD_LOCAL);
    if (h) {
      r.bound = reinterpret_cast<compress_bound_fn>(dlsym(h, "compressBound"));
      r.version = reinterpret_cast<zlib_version_fn>(dlsym(h, "zlibVersion"));
      r.init2 = reinterpret_cast<deflate_init2_fn>(dlsym(h, "deflateInit2_"));
      r.deflate = reinterpret_cast<deflate_fn>(dlsym(h, "deflate"));
      r.reset = reinterpret_cast<deflate_reset_fn>(dlsym(h, "deflateReset"));
      r.end = reinterpret_cast<deflate_end_fn>(dlsym(h, "deflateEnd"));
    }
    return r;
  }();
  return z;
}

// One worker's deflate stream with the parameters of zlib's one-shot compress2 (method 8 =
// deflate, 15 window bits, memory level 8, default strategy). deflateReset returns the stream to
// the state a fresh init leaves, so each block's output is byte for byte compress2's; reusing
// the stream saves the per-call allocation of its ~256 KB of tables.
class Deflater {
 public:
  Deflater(const Zlib& z, int level) : z_(z) {
    memset(&s_, 0, sizeof(s_));
    ok_ = z_.init2(&s_, level, 8, 15, 8, 0, z_.version(), (int)sizeof(ZStream)) == 0;
  }
  ~Deflater() {
    if (ok_) z_.end(&s_);
  }
  // Compressed length of src[0, n) (zlib framing), or -1 on error.
  long length(const unsigned char* src, unsigned int n, unsigned char* buf, unsigned int cap) {
    if (!ok_ || z_.reset(&s_) != 0) return -1;
    s_.next_in = src;
    s_.avail_in = n;
    s_.next_out = buf;
    s_.avail_out = cap;
    if (z_.deflate(&s_, 4 /* finish */) != 1 /* stream end */) return -1;
    return (long)(cap - s_.avail_out);
  }

 private:
  const Zlib& z_;
  ZStream s_;
  bool ok_ = false;
};

// Deflate stream of the calling thread for `level`, created on first use and kept for the
// thread's lifetime (a stream zlib could not set up reports -1 for every block).
Deflater* thread_deflater(const Zlib& z, int level) {
  thread_local std::unique_ptr<Deflater> per_level[10];
  std::unique_ptr<Deflater>& d = per_level[level];
  if (!d) d.reset(new Deflater(z, level));
  return d.get();
}

// Persistent host workers for the ratio pass. A call's blocks are handed out in chunks through
// an atomic counter to the calling thread and up to (limit - 1) workers; workers sleep on a
// condition variable between calls, so a call pays a wake-up instead of creating threads (and
// their allocator state) each time. Calls are serialised by the pool.
class HostPool {
 public:
  explicit HostPool(int n_workers) : workers_(n_workers) {
    for (int i = 0; i < n_workers; ++i) std::thread([this] { worker(); }).detach();
  }
  int workers() const { return workers_; }

  // Runs fn(begin, end) over [0, total) in chunks of `chunk` on the caller and up to
  // limit - 1 workers; returns when every chunk is done and no worker still holds the job.
  void run(int64_t total, int64_t chunk, int limit, const std::function<void(int64_t, int64_t)>& fn) {
    std::lock_guard<std::mutex> call(call_mu_);
    {
      std::lock_guard<std::mutex> g(mu_);
      fn_ = &fn;
      total_ = total;
      chunk_ = chunk;
      next_.store(0);
      seats_ = limit - 1;
      open_ = true;
      ++generation_;
    }
    cv_.notify_all();
    drain();
    std::unique_lock<std::mutex> g(mu_);
    open_ = false;                               // no worker joins the job after this point
    done_cv_.wait(g, [this] { return inside_ == 0; });
    fn_ = nullptr;
  }

 private:
  void drain() {
    for (;;) {
      const int64_t b = next_.fetch_add(chunk_);
      if (b >= total_) return;
      (*fn_)(b, std::min(total_, b + chunk_));
    }
  }
  void worker() {
    uint64_t seen = 0;
    for (;;) {
      {
        std::unique_lock<std::mutex> g(mu_);
        cv_.wait(g, [&] { return generation_ != seen; });
        seen = generation_;
        if (!open_ || seats_ <= 0) continue;
        --seats_;
        ++inside_;
      }
      drain();
      {
        std::lock_guard<std::mutex> g(mu_);
        if (--inside_ == 0) done_cv_.notify_all();
      }
    }
  }

  const int workers_;
  std::mutex call_mu_, mu_;
  std::condition_variable cv_, done_cv_;
  const std::function<void(int64_t, int64_t)>* fn_ = nullptr;
  int64_t total_ = 0, chunk_ = 1;
  std::atomic<int64_t> next_{0};
  int seats_ = 0, inside_ = 0;
  bool open_ = false;
  uint64_t generation_ = 0;
};

// The process's pool (hardware concurrency - 1 workers), created on first use. A forked child
// has none of the parent's workers: the fork handler drops the pointer (the parent's pool object
// is left alone) and re-initialises the creation lock, so the child builds a pool of its own.
pthread_mutex_t g_pool_mu = PTHREAD_MUTEX_INITIALIZER;
HostPool* g_pool = nullptr;
bool g_pool_hooked = false;

void pool_after_fork_in_child() {
  g_pool = nullptr;
  pthread_mutex_init(&g_pool_mu, nullptr);
}

HostPool& host_pool() {
  pthread_mutex_lock(&g_pool_mu);
  if (g_pool == nullptr) {
    if (!g_pool_hooked) {
      pthread_atfork(nullptr, nullptr, pool_after_fork_in_child);
      g_pool_hooked = true;
    }
    const int hw = (int)std::max(1u, std::thread::hardware_concurrency());
    g_pool = new HostPool(std::min(hw, 256) - 1);
  }
  HostPool* p = g_pool;
  pthread_mutex_unlock(&g_pool_mu);
  return *p;
}

}  // namespace

extern "C" {

int sa_version(void) { return 1; }

const char* sa_status_string(int status) {
  switch (status) {
    case SA_OK: return "SA_OK";
    case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG";
    case SA_ERR_UNSUPPORTED: return "SA_ERR_UNSUPPORTED";
    case SA_ERR_CAPACITY: return "SA_ERR_CAPACITY";
    case SA_ERR_CUDA: return "SA_ERR_CUDA";
    case SA_ERR_TIMEOUT: return "SA_ERR_TIMEOUT";
    case SA_ERR_DEVICE: return "SA_ERR_DEVICE";
  }
  return "SA_ERR_UNKNOWN";
}

int sa_mask_nnz_bound(const sa_mask_params* params, int64_t* h_nnz) {
  const int st = check_mask_params(params);
  if (st != SA_OK) return st;
  if (!h_nnz) return SA_ERR_INVALID_ARG;
  *h_nnz = nnz_bound(*params);
  return SA_OK;
}

int sa_build_mask(const sa_mask_params* params, const float* d_ratio, int32_t* d_row_ptr, int32_t* d_col_idx,
                  int64_t col_capacity, void* stream) {
  const int st = check_mask_params(params);
  if (st != SA_OK) return st;
  if (!d_row_ptr || !d_col_idx) return SA_ERR_INVALID_ARG;
  const bool needs_ratio = params->mode == SA_MASK_TOPK || params->mode == SA_MASK_LITERAL_MEAN;
  if (needs_ratio && !d_ratio) return SA_ERR_INVALID_ARG;
  const int64_t need = nnz_bound(*params);
  if (need > INT32_MAX) return SA_ERR_UNSUPPORTED;
  if (col_capacity < need) return SA_ERR_CAPACITY;
  if (!device_ok()) return SA_ERR_CUDA;
  return sa::launch_build_mask(*params, d_ratio, d_row_ptr, d_col_idx, static_cast<cudaStream_t>(stream));
}

int sa_attn_fwd_heads(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                      const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch, int32_t n_tokens,
                      int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t block, int32_t causal,
                      int32_t n_masks, const int32_t* const* h_row_ptrs, const int32_t* const* h_col_idxs,
                      const int32_t* h_head_mask, int32_t csr_shared, float softmax_scale, void* o, float* lse,
                      void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_attn_common(q, k, v, q_strides, kv_strides, o_strides, batch, n_tokens, heads, kv_heads, o, lse);
  if (st != SA_OK) return st;
  if (n_masks < 1 || !h_row_ptrs || !h_col_idxs || (n_masks > 1 && !h_head_mask)) return SA_ERR_INVALID_ARG;
  if (n_masks > sa::kMaxMasks || (n_masks > 1 && heads > sa::kMaxHeadMap)) return SA_ERR_UNSUPPORTED;
  for (int m = 0; m < n_masks; ++m)
    if (!h_row_ptrs[m] || !h_col_idxs[m]) return SA_ERR_INVALID_ARG;
  if (n_masks > 1)
    for (int h = 0; h < heads; ++h)
      if (h_head_mask[h] < 0 || h_head_mask[h] >= n_masks) return SA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return SA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f)) return SA_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return SA_ERR_UNSUPPORTED;
  if (block != 32 && block != 64 && block != 128) return SA_ERR_UNSUPPORTED;
  if (n_tokens % block != 0) return SA_ERR_UNSUPPORTED;
  if (n_tokens / block > sa::kMaxMaskBlocks) return SA_ERR_UNSUPPORTED;
  if ((int64_t)batch * heads > 65535 * 32 || (n_tokens + 127) / 128 > 65535) return SA_ERR_UNSUPPORTED;
  if (!workspace) return SA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SA_ERR_UNSUPPORTED;
  if (workspace_bytes < 256) return SA_ERR_CAPACITY;
  if (!device_ok()) return SA_ERR_CUDA;
  sa::AttnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  for (int i = 0; i < 3; ++i) {
    a.q_strides[i] = q_strides[i];
    a.kv_strides[i] = kv_strides[i];
    a.o_strides[i] = o_strides[i];
  }
  a.batch = batch;
  a.n_tokens = n_tokens;
  a.heads = heads;
  a.kv_heads = kv_heads;
  a.head_dim = head_dim;
  a.block = block;
  a.causal = causal;
  a.csr_shared = csr_shared != 0;
  a.n_masks = n_masks;
  for (int m = 0; m < sa::kMaxMasks; ++m) {
    a.row_ptr[m] = m < n_masks ? h_row_ptrs[m] : nullptr;
    a.col_idx[m] = m < n_masks ? h_col_idxs[m] : nullptr;
  }
  for (int h = 0; h < sa::kMaxHeadMap; ++h)
    a.head_mask[h] = (n_masks > 1 && h < heads) ? (uint8_t)h_head_mask[h] : 0;
  a.softmax_scale = softmax_scale;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return sa::launch_attn_fwd(a, static_cast<cudaStream_t>(stream));
}

int sa_attn_fwd(const void* q, const void* k, const void* v, const int64_t q_strides[3], const int64_t kv_strides[3],
                const int64_t o_strides[3], int32_t batch, int32_t n_tokens, int32_t heads, int32_t kv_heads,
                int32_t head_dim, int32_t block, int32_t causal, const int32_t* d_row_ptr, const int32_t* d_col_idx,
                int32_t csr_shared, float softmax_scale, void* o, float* lse, void* workspace,
                size_t workspace_bytes, void* stream) {
  if (!d_row_ptr || !d_col_idx) return SA_ERR_INVALID_ARG;
  return sa_attn_fwd_heads(q, k, v, q_strides, kv_strides, o_strides, batch, n_tokens, heads, kv_heads, head_dim,
                           block, causal, 1, &d_row_ptr, &d_col_idx, nullptr, csr_shared, softmax_scale, o, lse,
                           workspace, workspace_bytes, stream);
}

int sa_attn_fwd_workspace_size(int32_t batch, int32_t n_tokens, int32_t heads, int32_t head_dim, int32_t block,
                               int32_t csr_batches, int32_t n_masks, size_t* h_bytes) {
  if (batch <= 0 || n_tokens <= 0 || heads <= 0 || block <= 0 || n_tokens % block != 0 || csr_batches <= 0 ||
      n_masks <= 0 || !h_bytes)
    return SA_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return SA_ERR_UNSUPPORTED;
  *h_bytes = sa::attn_fwd_workspace_bytes(batch, n_tokens, heads, head_dim, csr_batches, n_masks);
  return SA_OK;
}

int sa_attn_bwd_workspace_size(int32_t batch, int32_t n_tokens, int32_t heads, int32_t block, int32_t csr_batches,
                               int64_t col_capacity, size_t* h_bytes) {
  if (batch <= 0 || n_tokens <= 0 || heads <= 0 || block <= 0 || n_tokens % block != 0 || csr_batches <= 0 ||
      col_capacity < 0 || !h_bytes)
    return SA_ERR_INVALID_ARG;
  *h_bytes = sa::bwd_workspace_layout(batch, n_tokens, heads, block, csr_batches, col_capacity).bytes;
  return SA_OK;
}

int sa_attn_bwd_heads(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
                      const int64_t q_strides[3], const int64_t kv_strides[3], const int64_t o_strides[3],
                      int32_t batch, int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim,
                      int32_t block, int32_t causal, int32_t n_masks, const int32_t* const* h_row_ptrs,
                      const int32_t* const* h_col_idxs, const int64_t* h_col_capacities,
                      const int32_t* h_head_mask, int32_t csr_shared, float softmax_scale, void* dq, void* dk,
                      void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  if (!o || !d_o || !lse || !dk || !dv || !workspace || !h_row_ptrs || !h_col_idxs) return SA_ERR_INVALID_ARG;
  if (n_masks < 1 || (n_masks > 1 && (!h_head_mask || !h_col_capacities))) return SA_ERR_INVALID_ARG;
  if (n_masks > sa::kMaxMasks || (n_masks > 1 && heads > sa::kMaxHeadMap)) return SA_ERR_UNSUPPORTED;
  for (int m = 0; m < n_masks; ++m) {
    if (!h_row_ptrs[m] || !h_col_idxs[m]) return SA_ERR_INVALID_ARG;
    if (n_masks > 1 && h_col_capacities[m] < 0) return SA_ERR_INVALID_ARG;
  }
  if (n_masks > 1)
    for (int h = 0; h < heads; ++h)
      if (h_head_mask[h] < 0 || h_head_mask[h] >= n_masks) return SA_ERR_INVALID_ARG;
  const int st = check_attn_common(q, k, v, q_strides, kv_strides, o_strides, batch, n_tokens, heads, kv_heads, dq,
                                   const_cast<float*>(lse));
  if (st != SA_OK) return st;
  if (!aligned16(o) || !aligned16(d_o) || !aligned16(dk) || !aligned16(dv) || !aligned16(lse)) return SA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SA_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return SA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f)) return SA_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return SA_ERR_UNSUPPORTED;
  if (block != 32 && block != 64 && block != 128) return SA_ERR_UNSUPPORTED;
  if (n_tokens % block != 0) return SA_ERR_UNSUPPORTED;
  if (n_tokens / block > sa::kMaxMaskBlocks) return SA_ERR_UNSUPPORTED;
  if ((int64_t)batch * heads * ((n_tokens + 127) / 128) > INT32_MAX) return SA_ERR_UNSUPPORTED;
  const int64_t csr_batches = csr_shared ? 1 : batch;
  int64_t cap_total = 0;
  for (int m = 0; m < n_masks; ++m) cap_total += n_masks > 1 ? h_col_capacities[m] : 0;
  if (workspace_bytes <
      sa::bwd_workspace_layout(batch, n_tokens, heads, block, csr_batches * n_masks, cap_total).bytes)
    return SA_ERR_CAPACITY;
  if (!device_ok()) return SA_ERR_CUDA;
  sa::BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.d_o = d_o;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  for (int i = 0; i < 3; ++i) {
    a.q_strides[i] = q_strides[i];
    a.kv_strides[i] = kv_strides[i];
    a.o_strides[i] = o_strides[i];
  }
  a.batch = batch;
  a.n_tokens = n_tokens;
  a.heads = heads;
  a.kv_heads = kv_heads;
  a.head_dim = head_dim;
  a.block = block;
  a.causal = causal;
  a.csr_shared = csr_shared != 0;
  a.n_masks = n_masks;
  for (int m = 0; m < sa::kMaxMasks; ++m) {
    a.row_ptr[m] = m < n_masks ? h_row_ptrs[m] : nullptr;
    a.col_idx[m] = m < n_masks ? h_col_idxs[m] : nullptr;
    a.col_capacity[m] = (m < n_masks && n_masks > 1) ? h_col_capacities[m] : 0;
  }
  for (int h = 0; h < sa::kMaxHeadMap; ++h) a.head_mask[h] = (n_masks > 1 && h < heads) ? (uint8_t)h_head_mask[h] : 0;
  a.softmax_scale = softmax_scale;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return sa::launch_attn_bwd(a, static_cast<cudaStream_t>(stream));
}

int sa_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
                const int64_t q_strides[3], const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch,
                int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t block, int32_t causal,
                const int32_t* d_row_ptr, const int32_t* d_col_idx, int32_t csr_shared, float softmax_scale,
                void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  if (!d_row_ptr || !d_col_idx) return SA_ERR_INVALID_ARG;
  return sa_attn_bwd_heads(q, k, v, o, d_o, lse, q_strides, kv_strides, o_strides, batch, n_tokens, heads, kv_heads,
                           head_dim, block, causal, 1, &d_row_ptr, &d_col_idx, nullptr, nullptr, csr_shared,
                           softmax_scale, dq, dk, dv, workspace, workspace_bytes, stream);
}

int sa_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse,
                        const int64_t q_strides[3], const int64_t kv_strides[3], const int64_t o_strides[3],
                        int32_t batch, int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim,
                        int32_t block, int32_t causal, const int32_t* d_row_ptr, const int32_t* d_col_idx,
                        int64_t col_capacity, int32_t csr_shared, float softmax_scale, void* dq, void* dk, void* dv,
                        void* stream) {
  if (batch <= 0 || n_tokens <= 0 || heads <= 0 || block <= 0 || n_tokens % block != 0 || col_capacity < 0)
    return SA_ERR_INVALID_ARG;
  const int64_t csr_batches = csr_shared ? 1 : batch;
  const size_t need = sa::bwd_workspace_layout(batch, n_tokens, heads, block, csr_batches, col_capacity).bytes;
  if (need > sa::kBwdStaticScratchBytes) return SA_ERR_CAPACITY;
  if (!device_ok()) return SA_ERR_CUDA;
  void* scratch = nullptr;
  if (sa::bwd_static_scratch(&scratch) != SA_OK) return SA_ERR_CUDA;
  return sa_attn_bwd(q, k, v, o, d_o, lse, q_strides, kv_strides, o_strides, batch, n_tokens, heads, kv_heads,
                     head_dim, block, causal, d_row_ptr, d_col_idx, csr_shared, softmax_scale, dq, dk, dv, scratch,
                     need, stream);
}

int sa_offset_attn_fwd_list(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                            const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch,
                            int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t window,
                            const int32_t* h_offsets, int32_t n_offsets, float softmax_scale, void* o, float* lse,
                            void* stream) {
  int st = check_attn_common(q, k, v, q_strides, kv_strides, o_strides, batch, n_tokens, heads, kv_heads, o, lse);
  if (st != SA_OK) return st;
  if (n_offsets < 0 || (n_offsets > 0 && !h_offsets)) return SA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f)) return SA_ERR_INVALID_ARG;
  if (window < 0) return SA_ERR_INVALID_ARG;
  if (window > sa::kMaxWindow || n_offsets > sa::kMaxOffsets) return SA_ERR_UNSUPPORTED;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return SA_ERR_UNSUPPORTED;
  for (int i = 0; i < n_offsets; ++i) {
    if (h_offsets[i] <= window || h_offsets[i] >= n_tokens) return SA_ERR_INVALID_ARG;
    if (i > 0 && h_offsets[i] <= h_offsets[i - 1]) return SA_ERR_INVALID_ARG;
  }
  // grid: (batch x heads, query tiles of 128, or 64 at head dimension 128)
  if ((int64_t)batch * heads > 0x7fffffff || (n_tokens + 63) / 64 > 65535) return SA_ERR_UNSUPPORTED;
  if (!device_ok()) return SA_ERR_CUDA;
  sa::OffsetArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  for (int i = 0; i < 3; ++i) {
    a.q_strides[i] = q_strides[i];
    a.kv_strides[i] = kv_strides[i];
    a.o_strides[i] = o_strides[i];
  }
  a.batch = batch;
  a.n_tokens = n_tokens;
  a.heads = heads;
  a.kv_heads = kv_heads;
  a.head_dim = head_dim;
  a.window = window;
  a.n_offsets = n_offsets;
  for (int i = 0; i < sa::kMaxOffsets; ++i) a.offsets[i] = i < n_offsets ? h_offsets[i] : 0;
  a.softmax_scale = softmax_scale;
  return sa::launch_offset_attn_fwd(a, static_cast<cudaStream_t>(stream));
}

int sa_offset_attn_fwd(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                       const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch, int32_t n_tokens,
                       int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t window, int32_t alpha_num,
                       int32_t alpha_den, int32_t n_rungs, float softmax_scale, void* o, float* lse, void* stream) {
  int32_t offs[sa::kMaxOffsets];
  int32_t count = 0;
  const int st = sa_fib_offsets(alpha_num, alpha_den, n_rungs, window, n_tokens, offs, sa::kMaxOffsets, &count);
  if (st == SA_ERR_CAPACITY) return SA_ERR_UNSUPPORTED;   // more distinct offsets than the kernel takes
  if (st != SA_OK) return st;
  return sa_offset_attn_fwd_list(q, k, v, q_strides, kv_strides, o_strides, batch, n_tokens, heads, kv_heads,
                                 head_dim, window, offs, count, softmax_scale, o, lse, stream);
}

}  // extern "C"

namespace {

// Distinct round_half_even(alpha * f) over a rung ladder, kept if window < d < n_tokens.
// ladder 0: Fibonacci 1, 2, 3, 5, ...; ladder 1: powers of two.
int ladder_offsets(int ladder, int32_t alpha_num, int32_t alpha_den, int32_t n_rungs, int32_t window,
                   int32_t n_tokens, int32_t* h_out, int32_t capacity, int32_t* h_count) {
  if (alpha_num <= 0 || alpha_den <= 0 || n_rungs < 0 || window < 0 || n_tokens <= 0 || !h_count ||
      capacity < 0 || (capacity > 0 && !h_out))
    return SA_ERR_INVALID_ARG;
  std::vector<int64_t> out;
  int64_t a = 1, b = 2;
  for (int k = 0;; ++k) {
    if (n_rungs > 0 ? k >= n_rungs : a > n_tokens) break;
    // round_half_even(alpha_num * f / alpha_den) in integer arithmetic
    const int64_t num = 2 * (int64_t)alpha_num * a + alpha_den;
    const int64_t den2 = 2 * (int64_t)alpha_den;
    int64_t q = num / den2;
    if (num % den2 == 0 && (q & 1)) --q;   // exact tie: go to the even neighbour
    if (q > window && q < n_tokens && std::find(out.begin(), out.end(), q) == out.end()) out.push_back(q);
    if (ladder == 0) {
      const int64_t nxt = a + b;
      a = b;
      b = nxt;
    } else {
      a *= 2;
    }
    if (a > (int64_t)1 << 40) break;
  }
  std::sort(out.begin(), out.end());
  *h_count = (int32_t)out.size();
  if ((int64_t)out.size() > capacity) return SA_ERR_CAPACITY;
  for (size_t i = 0; i < out.size(); ++i) h_out[i] = (int32_t)out[i];
  return SA_OK;
}

}  // namespace

extern "C" {

int sa_offset_attn_interp_fwd(const void* q, const void* k, const void* v, const int64_t q_strides[3],
                              const int64_t kv_strides[3], const int64_t o_strides[3], int32_t batch,
                              int32_t n_tokens, int32_t heads, int32_t kv_heads, int32_t head_dim, int32_t window,
                              double alpha, int32_t n_rungs, int32_t ladder, float softmax_scale, void* o, float* lse,
                              void* stream) {
  int st = check_attn_common(q, k, v, q_strides, kv_strides, o_strides, batch, n_tokens, heads, kv_heads, o, lse);
  if (st != SA_OK) return st;
  if (!(softmax_scale > 0.f) || !(alpha > 0.0) || !std::isfinite(alpha)) return SA_ERR_INVALID_ARG;
  if (window < 0 || n_rungs < 0 || (ladder != 0 && ladder != 1)) return SA_ERR_INVALID_ARG;
  if (window > sa::kMaxWindow) return SA_ERR_UNSUPPORTED;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return SA_ERR_UNSUPPORTED;
  sa::InterpArgs a;
  a.n_rungs = 0;
  int64_t f = 1, g = 2;   // rung ladder
  for (int r = 0;; ++r) {
    if (n_rungs > 0 ? r >= n_rungs : f > n_tokens) break;
    const double d = alpha * (double)f;
    if (d >= (double)n_tokens) {                 // never reached by any query
    } else {
      const double lo = std::floor(d);
      const double t = d - lo;
      if (!(t == 0.0 && lo <= (double)window)) {
        if (a.n_rungs >= sa::kMaxInterpRungs) return SA_ERR_UNSUPPORTED;
        a.lo[a.n_rungs] = (int32_t)lo;
        a.t[a.n_rungs] = (float)t;
        ++a.n_rungs;
      }
    }
    if (ladder == 0) {
      const int64_t nxt = f + g;
      f = g;
      g = nxt;
    } else {
      f *= 2;
    }
    if (f > ((int64_t)1 << 40)) break;
  }
  // grid: (batch x heads, 64-query tiles)
  if ((int64_t)batch * heads > 0x7fffffff || (n_tokens + 63) / 64 > 65535) return SA_ERR_UNSUPPORTED;
  if (!device_ok()) return SA_ERR_CUDA;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  for (int i = 0; i < 3; ++i) {
    a.q_strides[i] = q_strides[i];
    a.kv_strides[i] = kv_strides[i];
    a.o_strides[i] = o_strides[i];
  }
  a.batch = batch;
  a.n_tokens = n_tokens;
  a.heads = heads;
  a.kv_heads = kv_heads;
  a.head_dim = head_dim;
  a.window = window;
  a.softmax_scale = softmax_scale;
  return sa::launch_offset_interp_fwd(a, static_cast<cudaStream_t>(stream));
}

int sa_fib_offsets(int32_t alpha_num, int32_t alpha_den, int32_t n_rungs, int32_t window, int32_t n_tokens,
                   int32_t* h_out, int32_t capacity, int32_t* h_count) {
  return ladder_offsets(0, alpha_num, alpha_den, n_rungs, window, n_tokens, h_out, capacity, h_count);
}

int sa_pow2_offsets(int32_t alpha_num, int32_t alpha_den, int32_t n_rungs, int32_t window, int32_t n_tokens,
                    int32_t* h_out, int32_t capacity, int32_t* h_count) {
  return ladder_offsets(1, alpha_num, alpha_den, n_rungs, window, n_tokens, h_out, capacity, h_count);
}

int sa_layer_alpha(int32_t layer, int32_t layers, int32_t lo_num, int32_t lo_den, int32_t hi_num, int32_t hi_den,
                   int32_t stride, int32_t* h_num, int32_t* h_den) {
  if (layers <= 0 || layer < 0 || layer >= layers || lo_den <= 0 || hi_den <= 0 || stride <= 0 || !h_num ||
      !h_den)
    return SA_ERR_INVALID_ARG;
  if (std::gcd(stride, layers) != 1) return SA_ERR_INVALID_ARG;
  const int64_t i = ((int64_t)stride * layer) % layers;
  // lo + (hi - lo) * i / (L - 1) = (lo_num hi_den (L-1) + (hi_num lo_den - lo_num hi_den) i) / (lo_den hi_den (L-1))
  const int64_t span = layers > 1 ? layers - 1 : 1;
  int64_t num = (int64_t)lo_num * hi_den * span + ((int64_t)hi_num * lo_den - (int64_t)lo_num * hi_den) * i;
  int64_t den = (int64_t)lo_den * hi_den * span;
  const int64_t g = std::gcd(num < 0 ? -num : num, den);
  if (g > 1) {
    num /= g;
    den /= g;
  }
  if (num <= 0 || num > INT32_MAX || den > INT32_MAX) return SA_ERR_UNSUPPORTED;
  *h_num = (int32_t)num;
  *h_den = (int32_t)den;
  return SA_OK;
}

int sa_block_ratios(const uint8_t* h_bytes, int32_t batch, int32_t n_tokens, int32_t block, int32_t level,
                    float* h_ratio, int32_t n_threads) {
  if (!h_bytes || !h_ratio || batch <= 0 || n_tokens <= 0 || block <= 0 || n_tokens % block != 0 || level < 0 ||
      level > 9 || n_threads < 0)
    return SA_ERR_INVALID_ARG;
  const Zlib& z = zlib();
  if (!z.ok()) return SA_ERR_UNSUPPORTED;
  const int64_t nb = n_tokens / block;
  const int64_t total = nb * batch;
  const int hw = (int)std::max(1u, std::thread::hardware_concurrency());
  // at least 8 blocks per participating thread
  const int threads = (int)std::min<int64_t>(n_threads > 0 ? n_threads : hw, std::max<int64_t>(1, total / 8));
  std::atomic<int> failed{0};
  const std::function<void(int64_t, int64_t)> work = [&](int64_t begin, int64_t end) {
    std::vector<unsigned char> buf(z.bound((unsigned long)block));
    Deflater* dfl = thread_deflater(z, level);
    for (int64_t idx = begin; idx < end; ++idx) {
      const int64_t s = idx / nb, i = idx % nb;
      const long len = dfl->length(h_bytes + s * (int64_t)n_tokens + i * block, (unsigned int)block, buf.data(),
                                   (unsigned int)buf.size());
      if (len < 0) {
        failed = 1;
        return;
      }
      h_ratio[idx] = (float)((double)len / (double)block);
    }
  };
  if (threads <= 1) {
    work(0, total);
  } else {
    HostPool& pool = host_pool();
    const int limit = std::min(threads, pool.workers() + 1);
    pool.run(total, std::max<int64_t>(1, std::min<int64_t>(8, total / (4 * limit))), limit, work);
  }
  return failed ? SA_ERR_UNSUPPORTED : SA_OK;
}

int sa_build_mask_from_bytes(const sa_mask_params* params, const uint8_t* h_bytes, int32_t zlib_level,
                             int32_t n_threads, float* h_ratio, float* d_ratio, int32_t* d_row_ptr,
                             int32_t* d_col_idx, int64_t col_capacity, void* stream) {
  const int st = check_mask_params(params);
  if (st != SA_OK) return st;
  if (params->mode != SA_MASK_TOPK && params->mode != SA_MASK_LITERAL_MEAN) return SA_ERR_INVALID_ARG;
  if (!h_bytes || !h_ratio || !d_ratio || !d_row_ptr || !d_col_idx) return SA_ERR_INVALID_ARG;
  const int64_t need = nnz_bound(*params);
  if (need > INT32_MAX) return SA_ERR_UNSUPPORTED;
  if (col_capacity < need) return SA_ERR_CAPACITY;
  if (!device_ok()) return SA_ERR_CUDA;
  // host part: the ratios, on host threads, while the GPU works through what the caller
  // enqueued before this call (e.g. the Q/K/V uploads and the previous step's attention)
  const int r = sa_block_ratios(h_bytes, params->batch, params->n_tokens, params->block, zlib_level, h_ratio,
                                n_threads);
  if (r != SA_OK) return r;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = sizeof(float) * (size_t)params->batch * (size_t)(params->n_tokens / params->block);
  if (cudaMemcpyAsync(d_ratio, h_ratio, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return SA_ERR_CUDA;
  return sa::launch_build_mask(*params, d_ratio, d_row_ptr, d_col_idx, s);
}

int sa_selftest_bounded_wait(void* stream) {
  if (!device_ok()) return SA_ERR_CUDA;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

int sa_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SA_ERR_CUDA;
  unsigned int self = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&self, g_selftest_err, sizeof(self), 0, cudaMemcpyDeviceToHost, s);
  cudaMemcpyToSymbolAsync(g_selftest_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
  const unsigned int e = sa::attn_read_and_clear_error(s) | sa::offset_read_and_clear_error(s) |
                         sa::interp_read_and_clear_error(s) | sa::bwd_read_and_clear_error(s) | self;
  if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
  if (e & sa::kErrTimeout) return SA_ERR_TIMEOUT;
  if (e & sa::kErrBadIndex) return SA_ERR_DEVICE;
  if (e & sa::kErrCapacity) return SA_ERR_CAPACITY;
  return SA_OK;
}

}  // extern "C"
