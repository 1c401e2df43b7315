// Token-granular window-plus-offset attention forward for sm_103a.
//
// "Depth-Staggered Fibonacci Spacing for Sparse Attention", section 2 "Attended set":
// query i attends to keys i - delta, delta in {0..W} u D (D = distinct scaled Fibonacci
// offsets > W). Offsets are shared by all queries, so the key set of 16 consecutive
// queries is a band plus a few diagonals:
//   * band: every delta <= 64 (the window and the small offsets). For queries
//     [i0, i0+16) the keys [i0 - Dr, i0 + 16) (Dr = the largest such delta rounded up to
//     16) form a dense 16 x (16 + Dr) score block; a per-lane bit mask (built on the host)
//     keeps the distances that belong to the set. Computed with mma.sync m16n8k16
//     (bf16 -> f32); the row sums come from one more MMA against a ones matrix.
//   * each larger offset delta: keys [i0 - delta, i0 + 16 - delta], of which query i0+r
//     uses only key r: the diagonal of a 16 x 16 block. Computed with 8 mma.sync for QK
//     and 8 for PV; the zero off-diagonal P entries cost tensor work, not memory traffic.
//
// Work item: one CTA of 4 warps per (sequence, head, query tile); warp w owns 16 * MT
// consecutive queries as MT 16-query m-tiles (MT = 2 at head dimension 32 and 64, 1 at 128,
// which keeps the O fragments at 64 registers) and takes every key of them (band steps and
// offsets), so no two warps merge softmax states. The band (K/V rows [q0 - 64, q0 + 64 MT))
// arrives by TMA once per CTA and is shared by the four warps. Once every warp is past the
// band, its memory becomes four per-warp slab rings of two buffers: a warp streams the 16 * MT
// K and V rows of each larger offset that its own queries use two offsets ahead, and waits on
// nothing but its own copies (no cross-warp release of a buffer, no CTA barrier between
// offsets). At head dimension 64: 128-query CTAs, 65 KB of shared memory, <= 168 registers,
// three CTAs (12 warps, 384 queries in flight) per SM. K/V rows in shared memory follow the
// layouts of mma_frag.cuh (head dimension 128: two 64-dimension column chunks per tile, each
// loaded by its own TMA box).
// Softmax: exact max over the band part, then the offsets with a lazily rescaled running
// max (threshold 2^8).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mma_frag.cuh"
#include "ptx_sm100.cuh"
#include "sa_internal.h"
#include "tma_host.h"

namespace sa {
namespace {

using namespace frag;

__device__ unsigned int g_offset_err;

// Sizes at head dimension D (layouts as in mma_frag.cuh).
template <int D>
struct OffCfg {
  static constexpr int MT = D == 128 ? 1 : 2;                // 16-query m-tiles per warp
  static constexpr int WARPS = 4;
  static constexpr int Q = 16 * MT * WARPS;                   // queries per CTA
  static constexpr int BAND_MAX = 64;                         // deltas up to this go through the band
  static constexpr int BAND_ROWS = Q + BAND_MAX;              // band rows [q0 - 64, q0 + Q)
  static constexpr int SLAB_ROWS = 16 * MT;                   // K (then V) rows of one warp's slab
  static constexpr int ROW_BYTES = 2 * D;
  static constexpr int BOX_D = D < 64 ? D : 64;               // TMA box columns (one column chunk)
  static constexpr int CHUNKS = D / BOX_D;
  static constexpr int BAND_BYTES = BAND_ROWS * ROW_BYTES;    // one of K, V
  static constexpr int SLAB_BYTES = SLAB_ROWS * ROW_BYTES;    // one of K, V
  static constexpr int WARP_SLAB_BYTES = 2 * SLAB_BYTES;      // K rows, then V rows
  static constexpr int RING = 2;                              // slab buffers per warp
  static constexpr int RING_BYTES = WARPS * RING * WARP_SLAB_BYTES;
  static constexpr int SMEM = 2 * BAND_BYTES > RING_BYTES ? 2 * BAND_BYTES : RING_BYTES;
  static constexpr int CTAS_PER_SM = 3;
  // column chunks (D = 128) must keep the 1024-byte alignment of the swizzled layout
  static_assert(CHUNKS == 1 || ((BAND_ROWS * 128) % 1024 == 0 && (SLAB_ROWS * 128) % 1024 == 0), "chunk alignment");
  static_assert(BAND_ROWS <= 256 && SLAB_ROWS <= 256, "TMA box rows");
  static_assert(CTAS_PER_SM * (1024 + SMEM) <= 227 * 1024, "shared memory per SM");
};
constexpr int kBandMax = 64;
constexpr int kMaxLarge = kMaxOffsets;

struct OffParams {
  int n_tokens, heads, heads_per_kv, ntiles;
  int dr;                       // band reach Dr (multiple of 16, <= 64)
  int n_large;                  // offsets > 64, ascending
  int large[kMaxLarge];
  // per lane: bit 4*nt + e set if score fragment element e of band n-tile nt is at a
  // distance in the key set (the same for every warp and tile)
  unsigned long long keep[32];
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  int64_t q_sb, q_sn, q_sh, o_sb, o_sn, o_sh;
  float scale_log2;
};

// One CTA's TMA loads of `rows` K or V rows starting at token `row0` into dst (column chunks
// of a head dimension 128 tile cstride bytes apart); completion on bar.
template <int D>
__device__ __forceinline__ void load_rows(uint8_t* dst, uint32_t cstride, const CUtensorMap* map, uint64_t* bar,
                                          int hk, int row0, int s) {
  using C = OffCfg<D>;
#pragma unroll
  for (int c = 0; c < C::CHUNKS; ++c) tma_load_4d(dst + c * cstride, map, bar, c * C::BOX_D, hk, row0, s);
}

template <int D, int NKT>
__global__ void __launch_bounds__(128, 3)
    offset_attn_kernel(const __grid_constant__ CUtensorMap tk_band, const __grid_constant__ CUtensorMap tv_band,
                       const __grid_constant__ CUtensorMap tk_slab, const __grid_constant__ CUtensorMap tv_slab,
                       const __grid_constant__ OffParams p) {
  using C = OffCfg<D>;
  using F = Frag<D>;
  constexpr int kMT = C::MT;
  constexpr int kRing = C::RING;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKb = sm;                        // band K
  uint8_t* sVb = sKb + C::BAND_BYTES;       // band V
  constexpr uint32_t kBandCstride = C::BAND_ROWS * 128;   // head dimension 128: second column chunk
  constexpr uint32_t kSlabCstride = C::SLAB_ROWS * 128;
  // once every warp is past the band, warp w's slab ring occupies its own kRing slabs of the
  // same memory: buffer b at + b * WARP_SLAB_BYTES, K rows first, then V rows
  __shared__ uint64_t bar_band, bar_slab[C::WARPS][kRing];
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wq = warp;
  const int h = blockIdx.x % p.heads;
  const int s = blockIdx.x / p.heads;
  const int tile = p.ntiles - 1 - (int)blockIdx.y;   // later tiles reach more offsets: start them first
  const int q0 = tile * C::Q;
  const int hk = h / p.heads_per_kv;
  // larger offsets that reach at least one query of this warp
  const int qw = q0 + C::SLAB_ROWS * wq;     // first query of this warp (m-tile m: qw + 16 m)
  int n_off = 0;
  while (n_off < p.n_large && p.large[n_off] <= qw + C::SLAB_ROWS - 1) ++n_off;

  if (tid == 0) {
    mbar_init(&bar_band, 1);
#pragma unroll
    for (int w = 0; w < C::WARPS; ++w)
#pragma unroll
      for (int b = 0; b < kRing; ++b) mbar_init(&bar_slab[w][b], 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar_band, (uint32_t)(2 * C::BAND_BYTES));
  }
  __syncthreads();
  if (lane == 0) {
    if (warp == 0) load_rows<D>(sKb, kBandCstride, &tk_band, &bar_band, hk, q0 - kBandMax, s);
    if (warp == 1) load_rows<D>(sVb, kBandCstride, &tv_band, &bar_band, hk, q0 - kBandMax, s);
  }

  const int g = lane >> 2, t = lane & 3;     // mma fragment coordinates: rows g, g+8; cols 2t, 2t+1
  const float c = p.scale_log2;
  const float kNegInf = __int_as_float(0xff800000);

  // Q operands straight from global memory (rows past the end read the last row; never stored)
  uint32_t qa[kMT][F::KS][4];
#pragma unroll
  for (int m = 0; m < kMT; ++m) {
    const int qm = qw + 16 * m;
    const int last = p.n_tokens - 1;
    const int i_lo = qm + g < last ? qm + g : last, i_hi = qm + g + 8 < last ? qm + g + 8 : last;
    const __nv_bfloat16* base = p.q + (int64_t)s * p.q_sb + (int64_t)h * p.q_sh;
    load_qfrag<D>(base + (int64_t)i_lo * p.q_sn, base + (int64_t)i_hi * p.q_sn, t, qa[m]);
  }

  // warp-uniform wait results: the fragment code below uses full-warp shuffles
  bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_band, 0, &abort_flag, &g_offset_err, kErrTimeout));

  float o[kMT][F::NT][4];                    // O fragments per m-tile: D / 8 n-tiles
#pragma unroll
  for (int m = 0; m < kMT; ++m)
#pragma unroll
    for (int nt = 0; nt < F::NT; ++nt) o[m][nt][0] = o[m][nt][1] = o[m][nt][2] = o[m][nt][3] = 0.f;
  // running max of rows g, g+8 of each m-tile (log2 units) and the row sums
  float m_lo[kMT], m_hi[kMT], l_lo[kMT], l_hi[kMT];
#pragma unroll
  for (int m = 0; m < kMT; ++m) {
    m_lo[m] = m_hi[m] = kNegInf;
    l_lo[m] = l_hi[m] = 0.f;
  }

  if (ok) {
    const KV kb_tile{smem_u32(sKb), kBandCstride}, vb_tile{smem_u32(sVb), kBandCstride};
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      // ---------------- band: keys [qm - Dr, qm + 16), band slab row = key - (q0 - 64)
      const int qm = qw + 16 * m;
      uint64_t keep = p.keep[lane];
      const int lim = p.dr - qm;             // band columns below lim are keys < 0 (first tile only)
      if (lim > 0) {
#pragma unroll
        for (int nt = 0; nt < 2 * NKT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (8 * nt + 2 * t + (e & 1) < lim) keep &= ~(1ull << (4 * nt + e));
      }
      const int row0 = qm - q0 + kBandMax - p.dr;
      float sb[2 * NKT][4];
      float mx_lo = kNegInf, mx_hi = kNegInf;
#pragma unroll
      for (int nt = 0; nt < 2 * NKT; ++nt) {
        uint32_t u[2 * F::KS];
        load_kfrag<D>(kb_tile, row0 + 8 * nt + g, t, u);
        sb[nt][0] = sb[nt][1] = sb[nt][2] = sb[nt][3] = 0.f;
        qk_ntile<D>(sb[nt], qa[m], u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float v = (keep >> (4 * nt + e)) & 1ull ? sb[nt][e] : kNegInf;
          sb[nt][e] = v;
          if (e < 2) mx_lo = fmaxf(mx_lo, v);
          else mx_hi = fmaxf(mx_hi, v);
        }
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      m_lo[m] = mx_lo * c;                   // finite: distance 0 is always kept
      m_hi[m] = mx_hi * c;
      // P = exp2(s c - m); row sums of the bf16 P the PV product uses come from one more
      // MMA against a ones matrix
      float lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NKT; ++j) {
        uint32_t pa[4];
        pa[0] = pack_bf16x2(ex2_approx(fmaf(sb[2 * j][0], c, -m_lo[m])), ex2_approx(fmaf(sb[2 * j][1], c, -m_lo[m])));
        pa[1] = pack_bf16x2(ex2_approx(fmaf(sb[2 * j][2], c, -m_hi[m])), ex2_approx(fmaf(sb[2 * j][3], c, -m_hi[m])));
        pa[2] = pack_bf16x2(ex2_approx(fmaf(sb[2 * j + 1][0], c, -m_lo[m])),
                            ex2_approx(fmaf(sb[2 * j + 1][1], c, -m_lo[m])));
        pa[3] = pack_bf16x2(ex2_approx(fmaf(sb[2 * j + 1][2], c, -m_hi[m])),
                            ex2_approx(fmaf(sb[2 * j + 1][3], c, -m_hi[m])));
        mma16816(lsum, pa, kOnesBf16x2, kOnesBf16x2);
        uint32_t vb[D / 16][4];
        load_v16<D>(vb_tile, row0 + 16 * j, lane, vb);
        pv_16<D>(o[m], pa, vb);
      }
      l_lo[m] = lsum[0];
      l_hi[m] = lsum[2];
    }
  }

  // The band is read: its memory becomes the warps' slab rings. Each warp streams the
  // SLAB_ROWS key and value rows of each larger offset that its own queries use, two slabs
  // ahead, and waits on nothing but its own copies.
  __syncthreads();
  uint8_t* ring = sm + wq * (kRing * C::WARP_SLAB_BYTES);
  int issued = 0;
  if (lane == 0 && !abort_flag) {
    for (; issued < kRing && issued < n_off; ++issued) {
      uint8_t* dst = ring + issued * C::WARP_SLAB_BYTES;
      mbar_arrive_expect_tx(&bar_slab[wq][issued], (uint32_t)C::WARP_SLAB_BYTES);
      load_rows<D>(dst, kSlabCstride, &tk_slab, &bar_slab[wq][issued], hk, qw - p.large[issued], s);
      load_rows<D>(dst + C::SLAB_BYTES, kSlabCstride, &tv_slab, &bar_slab[wq][issued], hk, qw - p.large[issued], s);
    }
  }
  ok = ok && !abort_flag;

  // ---------------- larger offsets: per m-tile, one diagonal 16 x 16 block of the slab
  const int hl = (lane & ~3) | (g >> 1);     // lane of this quad that holds the diagonal
  const bool holder = (t == (g >> 1));
  const int e_sel = g & 1;                   // which of the two fragment columns is diagonal
  for (int k = 0; k < n_off && ok; ++k) {
    const int b = k % kRing;
    ok = __all_sync(0xffffffffu, mbar_wait(&bar_slab[wq][b], (uint32_t)(k / kRing) & 1u, &abort_flag,
                                           &g_offset_err, kErrTimeout));
    if (!ok) break;
    const KV kt{smem_u32(ring + b * C::WARP_SLAB_BYTES), kSlabCstride};
    const KV vt{kt.base + C::SLAB_BYTES, kSlabCstride};
    const int delta = p.large[k];
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      const int qm = qw + 16 * m;
      float s_lo, s_hi;
      diag_scores<D>(kt, 16 * m, g, t, hl, e_sel, qa[m], s_lo, s_hi);
      if (qm + g - delta < 0) s_lo = kNegInf;
      if (qm + g + 8 - delta < 0) s_hi = kNegInf;
      // lazy running max (log2 units): rescale only when a score passes the max by 2^8
      const float x_lo = s_lo * c, x_hi = s_hi * c;
      float a_lo = 1.f, a_hi = 1.f;
      if (x_lo > m_lo[m] + 8.f) { a_lo = ex2_approx(m_lo[m] - x_lo); m_lo[m] = x_lo; }
      if (x_hi > m_hi[m] + 8.f) { a_hi = ex2_approx(m_hi[m] - x_hi); m_hi[m] = x_hi; }
      if (__any_sync(0xffffffffu, a_lo != 1.f || a_hi != 1.f)) {
#pragma unroll
        for (int nt = 0; nt < F::NT; ++nt) {
          o[m][nt][0] *= a_lo;
          o[m][nt][1] *= a_lo;
          o[m][nt][2] *= a_hi;
          o[m][nt][3] *= a_hi;
        }
        l_lo[m] *= a_lo;
        l_hi[m] *= a_hi;
      }
      const uint32_t pb = pack_bf16x2(ex2_approx(fmaf(s_lo, c, -m_lo[m])), ex2_approx(fmaf(s_hi, c, -m_hi[m])));
      l_lo[m] += __uint_as_float(pb << 16);
      l_hi[m] += __uint_as_float(pb & 0xffff0000u);
      diag_pv<D>(vt, 16 * m, lane, holder, e_sel, pb, o[m]);
    }
    // every lane has read the buffer: refill it with the slab kRing ahead
    __syncwarp();
    if (lane == 0 && issued < n_off && !abort_flag) {
      uint8_t* dst = ring + b * C::WARP_SLAB_BYTES;
      mbar_arrive_expect_tx(&bar_slab[wq][b], (uint32_t)C::WARP_SLAB_BYTES);
      load_rows<D>(dst, kSlabCstride, &tk_slab, &bar_slab[wq][b], hk, qw - p.large[issued], s);
      load_rows<D>(dst + C::SLAB_BYTES, kSlabCstride, &tv_slab, &bar_slab[wq][b], hk, qw - p.large[issued], s);
      ++issued;
    }
  }

  if (ok && !abort_flag) {
    // ---------------- epilogue: O / l (bf16) and LSE
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      const float inv_lo = 1.f / l_lo[m], inv_hi = 1.f / l_hi[m];   // l > 0: every query keeps itself
      const int i_lo = qw + 16 * m + g, i_hi = qw + 16 * m + g + 8;
      __nv_bfloat16* orow_lo = p.o + (int64_t)s * p.o_sb + (int64_t)i_lo * p.o_sn + (int64_t)h * p.o_sh;
      __nv_bfloat16* orow_hi = p.o + (int64_t)s * p.o_sb + (int64_t)i_hi * p.o_sn + (int64_t)h * p.o_sh;
#pragma unroll
      for (int nt = 0; nt < F::NT; ++nt) {
        const int col = 8 * nt + 2 * t;
        if (i_lo < p.n_tokens)
          *reinterpret_cast<uint32_t*>(orow_lo + col) = pack_bf16x2(o[m][nt][0] * inv_lo, o[m][nt][1] * inv_lo);
        if (i_hi < p.n_tokens)
          *reinterpret_cast<uint32_t*>(orow_hi + col) = pack_bf16x2(o[m][nt][2] * inv_hi, o[m][nt][3] * inv_hi);
      }
      if (t == 0) {
        float* lrow = p.lse + ((int64_t)s * p.heads + h) * p.n_tokens;
        if (i_lo < p.n_tokens) lrow[i_lo] = (m_lo[m] + __log2f(l_lo[m])) * 0.69314718055994531f;
        if (i_hi < p.n_tokens) lrow[i_hi] = (m_hi[m] + __log2f(l_hi[m])) * 0.69314718055994531f;
      }
    }
  }
  // A CTA leaves only with none of its copies in flight: after an abort each warp drains
  // the slabs it issued and has not waited for, warp 0 the band.
  __syncthreads();
  if (abort_flag && lane == 0) {
    int never = 0;
    if (warp == 0) mbar_wait(&bar_band, 0, &never, &g_offset_err, kErrTimeout);
    for (int j = issued - kRing < 0 ? 0 : issued - kRing; j < issued; ++j)
      mbar_wait(&bar_slab[wq][j % kRing], (uint32_t)(j / kRing) & 1u, &never, &g_offset_err, kErrTimeout);
  }
}

template <int D, int NKT>
int launch_nkt(const CUtensorMap& kb, const CUtensorMap& vb, const CUtensorMap& ks, const CUtensorMap& vs,
               const OffParams& p, int batch, cudaStream_t stream) {
  using C = OffCfg<D>;
  const size_t smem = 1024 + (size_t)C::SMEM;
  if (cudaFuncSetAttribute(offset_attn_kernel<D, NKT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SA_ERR_CUDA;
  dim3 grid((unsigned)(batch * p.heads), (unsigned)p.ntiles);
  offset_attn_kernel<D, NKT><<<grid, C::WARPS * 32, smem, stream>>>(kb, vb, ks, vs, p);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

template <int D>
int launch_d(const OffsetArgs& a, OffParams& p, cudaStream_t stream) {
  using C = OffCfg<D>;
  const CUtensorMapSwizzle swz = D == 32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap kb, vb, ks, vs;
  if (!encode_bhnd_map(&kb, a.k, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::BOX_D, C::BAND_ROWS, swz) ||
      !encode_bhnd_map(&vb, a.v, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::BOX_D, C::BAND_ROWS, swz) ||
      !encode_bhnd_map(&ks, a.k, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::BOX_D, C::SLAB_ROWS, swz) ||
      !encode_bhnd_map(&vs, a.v, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::BOX_D, C::SLAB_ROWS, swz))
    return SA_ERR_UNSUPPORTED;
  p.ntiles = (a.n_tokens + C::Q - 1) / C::Q;
  if (p.ntiles > 65535) return SA_ERR_UNSUPPORTED;
  switch ((16 + p.dr) / 16) {
    case 1: return launch_nkt<D, 1>(kb, vb, ks, vs, p, a.batch, stream);
    case 2: return launch_nkt<D, 2>(kb, vb, ks, vs, p, a.batch, stream);
    case 3: return launch_nkt<D, 3>(kb, vb, ks, vs, p, a.batch, stream);
    case 4: return launch_nkt<D, 4>(kb, vb, ks, vs, p, a.batch, stream);
    default: return launch_nkt<D, 5>(kb, vb, ks, vs, p, a.batch, stream);
  }
}

}  // namespace

int launch_offset_attn_fwd(const OffsetArgs& a, cudaStream_t stream) {
  if (a.head_dim != 32 && a.head_dim != 64 && a.head_dim != 128) return SA_ERR_UNSUPPORTED;
  OffParams p;
  p.n_tokens = a.n_tokens;
  p.heads = a.heads;
  p.heads_per_kv = a.heads / a.kv_heads;
  // band: the window and every offset <= 64; distances 0..95 as a bit set
  uint32_t dist_mask[3] = {0u, 0u, 0u};
  int dmax = a.window;
  for (int d = 0; d <= a.window; ++d) dist_mask[d >> 5] |= 1u << (d & 31);
  p.n_large = 0;
  for (int i = 0; i < a.n_offsets; ++i) {
    const int d = a.offsets[i];
    if (d <= kBandMax) {
      dist_mask[d >> 5] |= 1u << (d & 31);
      dmax = dmax > d ? dmax : d;
    } else {
      p.large[p.n_large++] = d;
    }
  }
  for (int i = p.n_large; i < kMaxLarge; ++i) p.large[i] = 0;
  p.dr = (dmax + 15) / 16 * 16;
  const int nkt = (16 + p.dr) / 16;
  // lane (g, t) holds score elements (row g + 8(e>>1), band column 8 nt + 2t + (e&1));
  // band column col of row rr is at distance rr + Dr - col
  for (int lane = 0; lane < 32; ++lane) {
    const int g = lane >> 2, t = lane & 3;
    unsigned long long bits = 0ull;
    for (int nt = 0; nt < 2 * nkt; ++nt)
      for (int e = 0; e < 4; ++e) {
        const int rr = g + 8 * (e >> 1), col = 8 * nt + 2 * t + (e & 1);
        const int dist = rr + p.dr - col;
        if (dist >= 0 && dist < 96 && ((dist_mask[dist >> 5] >> (dist & 31)) & 1u)) bits |= 1ull << (4 * nt + e);
      }
    p.keep[lane] = bits;
  }
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
  switch (a.head_dim) {
    case 32: return launch_d<32>(a, p, stream);
    case 64: return launch_d<64>(a, p, stream);
    default: return launch_d<128>(a, p, stream);
  }
}

unsigned int offset_read_and_clear_error(cudaStream_t stream) {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_offset_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
  cudaMemcpyToSymbolAsync(g_offset_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  return v;
}

}  // namespace sa
