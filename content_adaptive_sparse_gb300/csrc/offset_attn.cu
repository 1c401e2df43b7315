// Token-granular window-plus-offset attention forward for sm_103a.
//
// "Depth-Staggered Fibonacci Spacing for Sparse Attention", section 2 "Attended set":
// query i attends to keys i - delta, delta in {0..W} u D (D = distinct scaled Fibonacci
// offsets > W). Offsets are shared by all queries, so for a tile of 128 consecutive
// queries every delta needs one contiguous slab of 128 key/value rows (the window
// needs one slab of 128 + W rows). The kernel streams those slabs into shared memory
// with TMA (128-byte swizzle, so the per-thread row reads are bank-conflict free) and
// each thread owns one query: fp32 dot products with packed f32x2 FMAs, an online
// softmax with a lazily rescaled running max, and an fp32 output accumulator.
//
// Work item: one CTA of 128 threads per (sequence, head, 128-query tile).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx_sm100.cuh"
#include "sa_internal.h"
#include "tma_host.h"

namespace sa {
namespace {

__device__ unsigned int g_offset_err;

constexpr int kQ = 128;              // queries per CTA
constexpr int kD = 64;               // head dim supported by this kernel
constexpr int kRowBytes = kD * 2;    // 128 B per K/V row
constexpr int kSlabBytes = kQ * kRowBytes;

struct OffParams {
  int n_tokens, heads, heads_per_kv, window, n_offsets, ntiles;
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  int64_t q_sb, q_sn, q_sh, o_sb, o_sn, o_sh;
  float scale_log2;
  int offsets[kMaxOffsets];
};

// Byte offset of 16-byte chunk c of row r in a 128B-swizzled tile of 128-byte rows.
__device__ __forceinline__ uint32_t swz_off(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float* f) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xffff0000u);
  f[4] = __uint_as_float(u.z << 16);
  f[5] = __uint_as_float(u.z & 0xffff0000u);
  f[6] = __uint_as_float(u.w << 16);
  f[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

struct Acc {
  uint64_t o[kD / 2];   // packed f32 pairs of the output accumulator
  float m, l;
};

// One key: score, lazy max update, accumulate p * v. `krow`/`vrow` point at the
// swizzled shared-memory row.
__device__ __forceinline__ void visit_key(const uint64_t* q2, const uint8_t* kt, const uint8_t* vt, int r, Acc& a) {
  uint64_t s2a = 0, s2b = 0;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 u = *reinterpret_cast<const uint4*>(kt + swz_off(r, c));
    float f[8];
    bf16x8_to_f32(u, f);
    s2a = f2_fma(q2[4 * c + 0], f2_pack(f[0], f[1]), s2a);
    s2b = f2_fma(q2[4 * c + 1], f2_pack(f[2], f[3]), s2b);
    s2a = f2_fma(q2[4 * c + 2], f2_pack(f[4], f[5]), s2a);
    s2b = f2_fma(q2[4 * c + 3], f2_pack(f[6], f[7]), s2b);
  }
  float x0, x1, y0, y1;
  f2_unpack(s2a, x0, x1);
  f2_unpack(s2b, y0, y1);
  const float s = (x0 + x1) + (y0 + y1);          // already in log2 units (q pre-scaled)
  if (s > a.m + 8.0f) {                            // rare: rescale the accumulator
    const float alpha = ex2_approx(a.m - s);       // 0 on the first key
    const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
    for (int i = 0; i < kD / 2; ++i) a.o[i] = f2_mul(a.o[i], al2);
    a.l *= alpha;
    a.m = s;
  }
  const float p = ex2_approx(s - a.m);
  a.l += p;
  const uint64_t p2 = f2_pack(p, p);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 u = *reinterpret_cast<const uint4*>(vt + swz_off(r, c));
    float f[8];
    bf16x8_to_f32(u, f);
    a.o[4 * c + 0] = f2_fma(p2, f2_pack(f[0], f[1]), a.o[4 * c + 0]);
    a.o[4 * c + 1] = f2_fma(p2, f2_pack(f[2], f[3]), a.o[4 * c + 1]);
    a.o[4 * c + 2] = f2_fma(p2, f2_pack(f[4], f[5]), a.o[4 * c + 2]);
    a.o[4 * c + 3] = f2_fma(p2, f2_pack(f[6], f[7]), a.o[4 * c + 3]);
  }
}

__global__ void __launch_bounds__(kQ) offset_attn_kernel(const __grid_constant__ CUtensorMap tk_win,
                                                          const __grid_constant__ CUtensorMap tv_win,
                                                          const __grid_constant__ CUtensorMap tk_slab,
                                                          const __grid_constant__ CUtensorMap tv_slab,
                                                          const OffParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int win_rows = kQ + p.window;
  const int win_bytes = ((win_rows * kRowBytes) + 1023) & ~1023;
  uint8_t* sKw = sm;
  uint8_t* sVw = sKw + win_bytes;
  uint8_t* sSlab = sVw + win_bytes;   // [2 buffers][K slab, V slab]
  __shared__ uint64_t bar_win, bar_slab[2];
  __shared__ int abort_flag;
  int last_issued[2] = {-1, -1};   // slab index last loaded into each buffer (thread 0)

  const int t = threadIdx.x;
  const int h = blockIdx.x % p.heads;
  const int s = blockIdx.x / p.heads;
  const int tile = p.ntiles - 1 - (int)blockIdx.y;   // later tiles reach more offsets: start them first
  const int q0 = tile * kQ;
  const int hk = h / p.heads_per_kv;
  const int i = q0 + t;
  // offsets that reach at least one query of this tile: delta <= q0 + kQ - 1
  int n_off = 0;
  while (n_off < p.n_offsets && p.offsets[n_off] <= q0 + kQ - 1) ++n_off;

  if (t == 0) {
    mbar_init(&bar_win, 1);
    mbar_init(&bar_slab[0], 1);
    mbar_init(&bar_slab[1], 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar_win, 2u * win_rows * kRowBytes);
    tma_load_4d(sKw, &tk_win, &bar_win, 0, hk, q0 - p.window, s);
    tma_load_4d(sVw, &tv_win, &bar_win, 0, hk, q0 - p.window, s);
    for (int k = 0; k < 2 && k < n_off; ++k) {
      last_issued[k] = k;
      mbar_arrive_expect_tx(&bar_slab[k], 2u * kSlabBytes);
      tma_load_4d(sSlab + k * 2 * kSlabBytes, &tk_slab, &bar_slab[k], 0, hk, q0 - p.offsets[k], s);
      tma_load_4d(sSlab + k * 2 * kSlabBytes + kSlabBytes, &tv_slab, &bar_slab[k], 0, hk, q0 - p.offsets[k], s);
    }
  }

  // query row, pre-scaled by softmax_scale * log2(e)
  uint64_t q2[kD / 2];
  {
    const int iq = i < p.n_tokens ? i : p.n_tokens - 1;
    const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (int64_t)s * p.q_sb + (int64_t)iq * p.q_sn +
                                                       (int64_t)h * p.q_sh);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float f[8];
      bf16x8_to_f32(qrow[c], f);
#pragma unroll
      for (int e = 0; e < 8; e += 2) q2[4 * c + e / 2] = f2_pack(f[e] * p.scale_log2, f[e + 1] * p.scale_log2);
    }
  }
  Acc a;
#pragma unroll
  for (int k = 0; k < kD / 2; ++k) a.o[k] = 0ull;
  a.m = __int_as_float(0xff800000);
  a.l = 0.f;
  __syncthreads();

  bool ok = mbar_wait(&bar_win, 0, &abort_flag, &g_offset_err, kErrTimeout);
  __syncthreads();
  ok = ok && !abort_flag;   // every thread takes the same path below
  if (ok) {
    // window: keys i - delta, delta = 0..W; slab row of key i - delta is t + W - delta
    for (int d = 0; d <= p.window; ++d)
      if (i - d >= 0) visit_key(q2, sKw, sVw, t + p.window - d, a);
  }
  for (int k = 0; k < n_off && ok; ++k) {
    const int buf = k & 1;
    ok = mbar_wait(&bar_slab[buf], (k >> 1) & 1, &abort_flag, &g_offset_err, kErrTimeout);
    if (ok && i - p.offsets[k] >= 0) {
      const uint8_t* kt = sSlab + buf * 2 * kSlabBytes;
      visit_key(q2, kt, kt + kSlabBytes, t, a);
    }
    __syncthreads();
    if (t == 0 && ok && k + 2 < n_off) {
      last_issued[buf] = k + 2;
      mbar_arrive_expect_tx(&bar_slab[buf], 2u * kSlabBytes);
      tma_load_4d(sSlab + buf * 2 * kSlabBytes, &tk_slab, &bar_slab[buf], 0, hk, q0 - p.offsets[k + 2], s);
      tma_load_4d(sSlab + buf * 2 * kSlabBytes + kSlabBytes, &tv_slab, &bar_slab[buf], 0, hk,
                  q0 - p.offsets[k + 2], s);
    }
    ok = !abort_flag && ok;
  }
  if (!ok) {
    // drain this CTA's own copies before exit
    if (t == 0) {
      int never = 0;
      mbar_wait(&bar_win, 0, &never, &g_offset_err, kErrTimeout);
      for (int b = 0; b < 2; ++b)
        if (last_issued[b] >= 0) mbar_wait(&bar_slab[b], (last_issued[b] >> 1) & 1, &never, &g_offset_err, kErrTimeout);
    }
    __syncthreads();
    return;
  }
  if (i < p.n_tokens) {
    const float inv = a.l > 0.f ? 1.f / a.l : 0.f;
    uint4* orow = reinterpret_cast<uint4*>(p.o + (int64_t)s * p.o_sb + (int64_t)i * p.o_sn + (int64_t)h * p.o_sh);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float f[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) f2_unpack(a.o[4 * c + e], f[2 * e], f[2 * e + 1]);
      orow[c] = make_uint4(pack_bf16x2(f[0] * inv, f[1] * inv), pack_bf16x2(f[2] * inv, f[3] * inv),
                           pack_bf16x2(f[4] * inv, f[5] * inv), pack_bf16x2(f[6] * inv, f[7] * inv));
    }
    p.lse[((int64_t)s * p.heads + h) * p.n_tokens + i] =
        a.l > 0.f ? (a.m + __log2f(a.l)) * 0.69314718055994531f : __int_as_float(0xff800000);
  }
}

}  // namespace

int launch_offset_attn_fwd(const OffsetArgs& a, cudaStream_t stream) {
  if (a.head_dim != kD) return SA_ERR_UNSUPPORTED;
  CUtensorMap kw, vw, ks, vs;
  const uint32_t win_rows = (uint32_t)(kQ + a.window);
  if (!encode_bhnd_map(&kw, a.k, a.batch, a.n_tokens, a.kv_heads, kD, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], kD, win_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_bhnd_map(&vw, a.v, a.batch, a.n_tokens, a.kv_heads, kD, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], kD, win_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_bhnd_map(&ks, a.k, a.batch, a.n_tokens, a.kv_heads, kD, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], kD, kQ, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_bhnd_map(&vs, a.v, a.batch, a.n_tokens, a.kv_heads, kD, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], kD, kQ, CU_TENSOR_MAP_SWIZZLE_128B))
    return SA_ERR_UNSUPPORTED;
  OffParams p;
  p.n_tokens = a.n_tokens;
  p.heads = a.heads;
  p.heads_per_kv = a.heads / a.kv_heads;
  p.window = a.window;
  p.n_offsets = a.n_offsets;
  p.ntiles = (a.n_tokens + kQ - 1) / kQ;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.q_sb = a.q_strides[0];
  p.q_sn = a.q_strides[1];
  p.q_sh = a.q_strides[2];
  p.o_sb = a.o_strides[0];
  p.o_sn = a.o_strides[1];
  p.o_sh = a.o_strides[2];
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  for (int k = 0; k < kMaxOffsets; ++k) p.offsets[k] = k < a.n_offsets ? a.offsets[k] : 0;
  const int win_bytes = (((kQ + a.window) * kRowBytes) + 1023) & ~1023;
  const size_t smem = 1024 + 2 * (size_t)win_bytes + 4 * (size_t)kSlabBytes;
  if (cudaFuncSetAttribute(offset_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SA_ERR_CUDA;
  dim3 grid((unsigned)(a.batch * a.heads), (unsigned)p.ntiles);
  offset_attn_kernel<<<grid, kQ, smem, stream>>>(kw, vw, ks, vs, p);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

unsigned int offset_read_and_clear_error(cudaStream_t stream) {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_offset_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
  cudaMemcpyToSymbolAsync(g_offset_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  return v;
}

}  // namespace sa
