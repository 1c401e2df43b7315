// Window plus interpolated-rung attention forward for sm_103a ("Depth-Staggered Fibonacci
// Spacing for Sparse Attention", section 2 "Attended set": the gather at the continuous
// distance d_k = alpha f_k interpolates between rows i - floor(d_k) and i - floor(d_k) - 1).
//
// Entries of query i: window rows i - delta (delta = 0..W) and, for each rung (lo, t) with
// i - lo - t >= 0, the interpolated key / value (1 - t) x[i - lo] + t x[i - lo - 1]. Since
// the score is linear in the key, the rung's score is (1 - t) s_lo + t s_lo+1, and its
// value enters O with weights p (1 - t) and p t.
//
// The work per entry is a 64-wide dot product and a 64-wide update of O, so the kernel runs
// on the CUDA cores (paired f32x2 FMAs): four lanes per query row (each lane holds 16 of the
// 64 head-dimension elements of q and O; two shuffles complete a dot product), 8 consecutive
// queries of one (sequence, head) per warp, so that the lanes of a warp read neighbouring
// rows at the same offset. The running max is rescaled lazily (only when it grows by more
// than 2^8). The rung table (floor distance, weight) is computed on the host from alpha.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kD = 64;
constexpr int kLanesPerQuery = 4;                   // lanes sharing one query row (8 measured slower)
constexpr int kHalf = kD / kLanesPerQuery;          // head-dimension elements per lane
constexpr int kQueriesPerWarp = 32 / kLanesPerQuery;
constexpr int kWarpsPerBlock = 4;

struct InterpParams {
  int batch, n_tokens, heads, heads_per_kv, window, n_rungs;
  int lo[kMaxInterpRungs];
  float t[kMaxInterpRungs];
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  int64_t q_sb, q_sn, q_sh, kv_sb, kv_sn, kv_sh, o_sb, o_sn, o_sh;
  float scale_log2;
  int tiles;                       // 16-query tiles per (sequence, head)
};

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
// bf16 pair (low element first) -> two floats, exactly
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t x) {
  return f2_pack(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// <q, row> over this lane's half of the head dimension (q held as 16 float pairs), then
// completed with the partner lane's half
__device__ __forceinline__ float row_dot(const uint64_t (&q2)[kHalf / 2], const __nv_bfloat16* half_row) {
  const uint4* r4 = reinterpret_cast<const uint4*>(half_row);
  uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
  for (int c = 0; c < kHalf / 8; ++c) {
    const uint4 w = __ldg(r4 + c);
    acc0 = f2_fma(q2[4 * c + 0], bf2_to_f2(w.x), acc0);
    acc1 = f2_fma(q2[4 * c + 1], bf2_to_f2(w.y), acc1);
    acc0 = f2_fma(q2[4 * c + 2], bf2_to_f2(w.z), acc0);
    acc1 = f2_fma(q2[4 * c + 3], bf2_to_f2(w.w), acc1);
  }
  float a, b, c2, d;
  f2_unpack(acc0, a, b);
  f2_unpack(acc1, c2, d);
  float part = (a + b) + (c2 + d);
#pragma unroll
  for (int o = 1; o < kLanesPerQuery; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  return part;
}

// o += w * row over this lane's half of the head dimension
__device__ __forceinline__ void row_axpy(uint64_t (&o2)[kHalf / 2], float w, const __nv_bfloat16* half_row) {
  const uint4* r4 = reinterpret_cast<const uint4*>(half_row);
  const uint64_t w2 = f2_pack(w, w);
#pragma unroll
  for (int c = 0; c < kHalf / 8; ++c) {
    const uint4 x = __ldg(r4 + c);
    o2[4 * c + 0] = f2_fma(w2, bf2_to_f2(x.x), o2[4 * c + 0]);
    o2[4 * c + 1] = f2_fma(w2, bf2_to_f2(x.y), o2[4 * c + 1]);
    o2[4 * c + 2] = f2_fma(w2, bf2_to_f2(x.z), o2[4 * c + 2]);
    o2[4 * c + 3] = f2_fma(w2, bf2_to_f2(x.w), o2[4 * c + 3]);
  }
}

__global__ void __launch_bounds__(32 * kWarpsPerBlock) offset_interp_kernel(const __grid_constant__ InterpParams p) {
  const int warp_global = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int part = lane % kLanesPerQuery;          // which part of the head dimension
  const int per_seq = p.heads * p.tiles;
  if (warp_global >= p.batch * per_seq) return;    // whole warp
  const int s = warp_global / per_seq;
  const int rem = warp_global % per_seq;
  const int h = rem / p.tiles;
  const int i_raw = (rem % p.tiles) * kQueriesPerWarp + lane / kLanesPerQuery;
  // rows past the end repeat the last query (the shuffles need every lane of a group);
  // they are not stored
  const bool store = i_raw < p.n_tokens;
  const int i = store ? i_raw : p.n_tokens - 1;
  const int hk = h / p.heads_per_kv;
  const __nv_bfloat16* kb = p.k + (int64_t)s * p.kv_sb + (int64_t)hk * p.kv_sh + kHalf * part;
  const __nv_bfloat16* vb = p.v + (int64_t)s * p.kv_sb + (int64_t)hk * p.kv_sh + kHalf * part;

  // q pre-scaled by softmax_scale * log2(e): scores come out in log2 units
  uint64_t q2[kHalf / 2];
  {
    const uint4* qr = reinterpret_cast<const uint4*>(p.q + (int64_t)s * p.q_sb + (int64_t)i * p.q_sn +
                                                     (int64_t)h * p.q_sh + kHalf * part);
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
    for (int c = 0; c < kHalf / 8; ++c) {
      const uint4 w = __ldg(qr + c);
      q2[4 * c + 0] = f2_mul(bf2_to_f2(w.x), sc2);
      q2[4 * c + 1] = f2_mul(bf2_to_f2(w.y), sc2);
      q2[4 * c + 2] = f2_mul(bf2_to_f2(w.z), sc2);
      q2[4 * c + 3] = f2_mul(bf2_to_f2(w.w), sc2);
    }
  }
  uint64_t o2[kHalf / 2];
#pragma unroll
  for (int c = 0; c < kHalf / 2; ++c) o2[c] = 0ull;
  float m = __int_as_float(0xff800000);   // reference max (log2 units), equal in both lanes
  float l = 0.f;

  // One entry with score x (log2 units): lazily rescaled online softmax.
  auto enter = [&](float x) -> float {
    if (x > m + 8.f) {
      const float a = ex2_approx(m - x);    // 0 when m = -inf
      const uint64_t a2 = f2_pack(a, a);
#pragma unroll
      for (int c = 0; c < kHalf / 2; ++c) o2[c] = f2_mul(o2[c], a2);
      l *= a;
      m = x;
    }
    const float pe = ex2_approx(x - m);
    l += pe;
    return pe;
  };

  // The pair shuffle in row_dot names the whole warp, so every lane must reach it together:
  // both loops below have warp-uniform trip counts, and entries out of a query's range are
  // computed on a valid row and then skipped.
  // window rows i - delta, delta = 0..W (uniform count W + 1; rows below 0 skipped)
  for (int delta = 0; delta <= p.window; ++delta) {
    const int j = i - delta;
    const bool ok = j >= 0;
    const int jj = ok ? j : 0;
    const float x = row_dot(q2, kb + (int64_t)jj * p.kv_sn);
    if (ok) {
      const float pe = enter(x);
      row_axpy(o2, pe, vb + (int64_t)jj * p.kv_sn);
    }
  }
  // interpolated rungs
  for (int r = 0; r < p.n_rungs; ++r) {
    const int lo = p.lo[r];
    const float t = p.t[r];
    const int far = t > 0.f ? lo + 1 : lo;            // both rows exist iff i >= far
    const bool ok = i >= far;
    if (!__any_sync(0xffffffffu, ok)) continue;       // no query of the warp reaches this rung
    const int64_t r0 = (int64_t)(ok ? i - lo : 0) * p.kv_sn;
    if (t > 0.f) {
      const int64_t r1 = (int64_t)(ok ? i - lo - 1 : 0) * p.kv_sn;
      const float x = (1.f - t) * row_dot(q2, kb + r0) + t * row_dot(q2, kb + r1);
      if (ok) {
        const float pe = enter(x);
        row_axpy(o2, pe * (1.f - t), vb + r0);
        row_axpy(o2, pe * t, vb + r1);
      }
    } else {
      const float x = row_dot(q2, kb + r0);
      if (ok) {
        const float pe = enter(x);
        row_axpy(o2, pe, vb + r0);
      }
    }
  }

  // the self row is always an entry, so l > 0
  const float inv = 1.f / l;
  uint32_t pk[kHalf / 2];
#pragma unroll
  for (int c = 0; c < kHalf / 2; ++c) {
    float a, b;
    f2_unpack(o2[c], a, b);
    __nv_bfloat162 hv = __floats2bfloat162_rn(a * inv, b * inv);
    pk[c] = *reinterpret_cast<uint32_t*>(&hv);
  }
  if (!store) return;
  uint4* orow = reinterpret_cast<uint4*>(p.o + (int64_t)s * p.o_sb + (int64_t)i * p.o_sn + (int64_t)h * p.o_sh +
                                         kHalf * part);
#pragma unroll
  for (int c = 0; c < kHalf / 8; ++c) orow[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
  if (part == 0) p.lse[((int64_t)s * p.heads + h) * p.n_tokens + i] = (m + __log2f(l)) * 0.69314718055994531f;
}

}  // namespace

int launch_offset_interp_fwd(const InterpArgs& a, cudaStream_t stream) {
  InterpParams p;
  p.batch = a.batch;
  p.n_tokens = a.n_tokens;
  p.heads = a.heads;
  p.heads_per_kv = a.heads / a.kv_heads;
  p.window = a.window;
  p.n_rungs = a.n_rungs;
  for (int r = 0; r < kMaxInterpRungs; ++r) {
    p.lo[r] = r < a.n_rungs ? a.lo[r] : 0;
    p.t[r] = r < a.n_rungs ? a.t[r] : 0.f;
  }
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.q_sb = a.q_strides[0];
  p.q_sn = a.q_strides[1];
  p.q_sh = a.q_strides[2];
  p.kv_sb = a.kv_strides[0];
  p.kv_sn = a.kv_strides[1];
  p.kv_sh = a.kv_strides[2];
  p.o_sb = a.o_strides[0];
  p.o_sn = a.o_strides[1];
  p.o_sh = a.o_strides[2];
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  p.tiles = (a.n_tokens + kQueriesPerWarp - 1) / kQueriesPerWarp;
  const int64_t warps = (int64_t)a.batch * a.heads * p.tiles;
  const int64_t blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > INT32_MAX) return SA_ERR_UNSUPPORTED;
  offset_interp_kernel<<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
