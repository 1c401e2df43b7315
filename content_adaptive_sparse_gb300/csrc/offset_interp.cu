// Window plus interpolated-rung attention forward for sm_103a ("Depth-Staggered Fibonacci
// Spacing for Sparse Attention", section 2 "Attended set": the gather at the continuous
// distance d_k = alpha f_k interpolates between rows i - floor(d_k) and i - floor(d_k) - 1).
//
// Entries of query i: window rows i - delta (delta = 0..W) and, for each rung (lo, t) with
// i >= lo + t, the interpolated key / value (1 - t) x[i - lo] + t x[i - lo - 1]. The score is
// linear in the key, so a rung's score is (1 - t) s_lo + t s_lo+1 with s_delta = q_i . k_{i-delta},
// and its value enters O with the weights p (1 - t) and p t.
//
// For 16 consecutive queries each distance is the diagonal of a 16 x 16 block, so the kernel
// is the integer-offset kernel's design with two diagonals per rung (mma.sync m16n8k16,
// bf16 -> f32):
//   * window: the dense 16 x (16 + Dr) block of keys [i0 - Dr, i0 + 16) (Dr = W rounded up
//     to 16) with a per-lane bit mask of the window distances, from a band of K/V rows
//     [q0 - 64, q0 + 64) that one TMA load brings in per CTA;
//   * rungs with lo + 1 <= 64: both diagonals read straight from the band;
//   * farther rungs: a 17-row K/V slab per warp (rows i0 - lo - 1 .. i0 - lo + 15; query r
//     takes rows r + 1 and r), streamed by TMA through a two-buffer ring per warp that
//     reuses the band's memory once every warp is past the band.
// One CTA of 4 warps per (sequence, head, 64-query tile); warp w owns queries q0 + 16w ..
// q0 + 16w + 15 and waits on nothing but the band and its own slabs. Softmax: exact max over
// the window block, then the rungs with a lazily rescaled running max (threshold 2^8).
// Head dimensions 32, 64 and 128; K/V rows in shared memory follow the layouts of
// mma_frag.cuh (head dimension 128: two 64-dimension column chunks per tile or slot).
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

__device__ unsigned int g_interp_err;

constexpr int kQ = 64;                     // queries per CTA
constexpr int kWarps = 4;                  // 16 queries per warp
constexpr int kBandMax = 64;               // rungs with lo + 1 <= 64 are read from the band
constexpr int kBandRows = kQ + kBandMax;   // band rows [q0 - 64, q0 + 64)
constexpr int kSlabRows = 17;              // rows i0 - lo - 1 .. i0 - lo + 15
constexpr int kSlotRows = 24;              // a rung pair's 16 x 24 score block reads 24 rows
constexpr int kRing = 2;                   // slab buffers per warp

// Sizes at head dimension D (layouts as in mma_frag.cuh).
template <int D>
struct InterpCfg {
  static constexpr int ROW_BYTES = 2 * D;
  static constexpr int BOX_D = D < 64 ? D : 64;                 // TMA box columns (one column chunk)
  static constexpr int CHUNKS = D / BOX_D;
  static constexpr int BAND_BYTES = kBandRows * ROW_BYTES;      // one of K, V
  static constexpr int BAND_CSTRIDE = kBandRows * 128;          // D = 128: second column chunk
  static constexpr int CHUNK_SLOT = D == 32 ? 2048 : 3072;      // 24 rows of one column chunk, 1 KB aligned
  static constexpr int SLOT_BYTES = CHUNKS * CHUNK_SLOT;        // one 17-row K or V slab
  static constexpr int BUF_BYTES = 2 * SLOT_BYTES;              // K slot, then V slot
  static constexpr int RINGS_BYTES = kWarps * kRing * BUF_BYTES;
  static constexpr int SMEM = RINGS_BYTES > 2 * BAND_BYTES ? RINGS_BYTES : 2 * BAND_BYTES;
  static constexpr int CTAS_PER_SM = D == 128 ? 2 : 4;
  static constexpr int SLAB_TX = 2 * kSlabRows * ROW_BYTES;     // bytes of one K + V slab load
  static_assert(kSlotRows * (ROW_BYTES < 128 ? ROW_BYTES : 128) <= CHUNK_SLOT && CHUNK_SLOT % 1024 == 0,
                "slab slots");
  // the 16 x 24 score block of a rung pair reads key rows r0 .. r0 + 23: inside a slot, and at
  // most 7 rows past the end of a K band column chunk (into the next chunk or the V band)
  static_assert((D == 128 ? BAND_CSTRIDE + (kBandRows + 7) * 128 : (kBandRows + 7) * ROW_BYTES) <= 2 * BAND_BYTES,
                "rung pair rows");
  static_assert(D != 128 || BAND_CSTRIDE % 1024 == 0, "chunk alignment");
  static_assert(CTAS_PER_SM * (1024 + SMEM) <= 227 * 1024, "shared memory per SM");
};

struct InterpParams {
  int n_tokens, heads, heads_per_kv, ntiles;
  int dr;                          // window reach Dr (multiple of 16, <= 64)
  int n_small;                     // rungs [0, n_small) have lo + 1 <= 64
  int n_rungs;                     // rungs by ascending distance
  int lo[kMaxInterpRungs];         // floor of the rung distance
  float t[kMaxInterpRungs];        // weight of the farther row
  // per lane: bit 4*nt + e set if score fragment element e of window n-tile nt is at a
  // distance 0..W (the same for every warp and tile)
  unsigned long long keep[32];
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* lse;
  int64_t q_sb, q_sn, q_sh, o_sb, o_sn, o_sh;
  float scale_log2;
};

// Raw scores of both distances of a rung for query rows g and g + 8 from one 16 x 24 block:
// key rows r0 .. r0 + 23 of a swizzled tile, where r0 + r is distance lo + 1 of query r (the
// diagonal, sb) and r0 + r + 1 distance lo (the superdiagonal, sa). Three 8-key n-tiles, 12
// mma.sync, instead of two 16 x 16 blocks (16); of the third n-tile only column 0 (query 15's
// distance lo) is read, so its other rows may hold anything. All lanes of a quad receive the
// scores of their rows.
template <int D>
__device__ __forceinline__ void diag_scores_pair(KV kt, int r0, int g, int t, const uint32_t (&qa)[Frag<D>::KS][4],
                                                 float& sa_lo, float& sa_hi, float& sb_lo, float& sb_hi) {
  uint32_t u0[2 * Frag<D>::KS], u1[2 * Frag<D>::KS], u2[2 * Frag<D>::KS];
  load_kfrag<D>(kt, r0 + g, t, u0);
  load_kfrag<D>(kt, r0 + 8 + g, t, u1);
  load_kfrag<D>(kt, r0 + 16 + g, t, u2);
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
  qk_ntile<D>(d0, qa, u0);
  qk_ntile<D>(d1, qa, u1);
  qk_ntile<D>(d2, qa, u2);
  // fragment (row R, column C) of an n-tile: lane 4 (R % 8) + C / 2, element 2 (R / 8) + C % 2.
  // Diagonal of query row g: column g of n-tile 0 (row g) / n-tile 1 (row g + 8). Superdiagonal:
  // column g + 1, which for g = 7 is column 0 of the next n-tile. The lane holding either value
  // has the same g as the lane asking for it, so each lane offers the elements its g selects.
  const int e_a = g & 1, e_b = (g + 1) & 1;
  const float diag_lo = e_a ? d0[1] : d0[0], diag_hi = e_a ? d1[3] : d1[2];
  const float sup_lo = g < 7 ? (e_b ? d0[1] : d0[0]) : d1[0];
  const float sup_hi = g < 7 ? (e_b ? d1[3] : d1[2]) : d2[2];
  const int src_diag = 4 * g + (g >> 1);
  const int src_sup = g < 7 ? 4 * g + ((g + 1) >> 1) : 28;
  sb_lo = __shfl_sync(0xffffffffu, diag_lo, src_diag);
  sb_hi = __shfl_sync(0xffffffffu, diag_hi, src_diag);
  sa_lo = __shfl_sync(0xffffffffu, sup_lo, src_sup);
  sa_hi = __shfl_sync(0xffffffffu, sup_hi, src_sup);
}

// Online-softmax state of one warp: O fragments, running max (log2 units) and row sums of
// query rows g and g + 8.
template <int D>
struct RungState {
  float o[Frag<D>::NT][4];
  float m_lo, m_hi, l_lo, l_hi;
};

// Softmax and PV of one rung from the raw diagonal scores (sa: distance lo, sb: lo + 1) of
// query rows g and g + 8; va / vb = the value rows of query row 0 at distance lo / lo + 1 in
// the swizzled tile vt; ok_* = the rung reaches the row.
template <int D>
__device__ __forceinline__ void enter_rung(RungState<D>& st, float sa_lo, float sa_hi, float sb_lo, float sb_hi,
                                           float t, bool two, bool ok_lo, bool ok_hi, float c, KV vt,
                                           int va, int vb, int lane, bool holder, int e_sel) {
  const float kNegInf = __int_as_float(0xff800000);
  const float x_lo = ok_lo ? ((1.f - t) * sa_lo + t * sb_lo) * c : kNegInf;
  const float x_hi = ok_hi ? ((1.f - t) * sa_hi + t * sb_hi) * c : kNegInf;
  // lazy running max (log2 units): rescale only when a score passes the max by 2^8
  float a_lo = 1.f, a_hi = 1.f;
  if (x_lo > st.m_lo + 8.f) { a_lo = ex2_approx(st.m_lo - x_lo); st.m_lo = x_lo; }
  if (x_hi > st.m_hi + 8.f) { a_hi = ex2_approx(st.m_hi - x_hi); st.m_hi = x_hi; }
  if (__any_sync(0xffffffffu, a_lo != 1.f || a_hi != 1.f)) {
#pragma unroll
    for (int nt = 0; nt < Frag<D>::NT; ++nt) {
      st.o[nt][0] *= a_lo;
      st.o[nt][1] *= a_lo;
      st.o[nt][2] *= a_hi;
      st.o[nt][3] *= a_hi;
    }
    st.l_lo *= a_lo;
    st.l_hi *= a_hi;
  }
  const float p_lo = ex2_approx(x_lo - st.m_lo), p_hi = ex2_approx(x_hi - st.m_hi);
  const uint32_t wa = pack_bf16x2(p_lo * (1.f - t), p_hi * (1.f - t));
  st.l_lo += __uint_as_float(wa << 16);
  st.l_hi += __uint_as_float(wa & 0xffff0000u);
  diag_pv<D>(vt, va, lane, holder, e_sel, wa, st.o);
  if (two) {
    const uint32_t wb = pack_bf16x2(p_lo * t, p_hi * t);
    st.l_lo += __uint_as_float(wb << 16);
    st.l_hi += __uint_as_float(wb & 0xffff0000u);
    diag_pv<D>(vt, vb, lane, holder, e_sel, wb, st.o);
  }
}

// One warp's (or CTA's) TMA loads of rows starting at token `row0` into dst (column chunks of
// a head dimension 128 tile cstride bytes apart); completion on bar.
template <int D>
__device__ __forceinline__ void load_rows(uint8_t* dst, uint32_t cstride, const CUtensorMap* map, uint64_t* bar,
                                          int hk, int row0, int s) {
  using C = InterpCfg<D>;
#pragma unroll
  for (int c = 0; c < C::CHUNKS; ++c) tma_load_4d(dst + c * cstride, map, bar, c * C::BOX_D, hk, row0, s);
}

template <int D, int NKT>
__global__ void __launch_bounds__(kWarps * 32, InterpCfg<D>::CTAS_PER_SM)
    offset_interp_kernel(const __grid_constant__ CUtensorMap tk_band, const __grid_constant__ CUtensorMap tv_band,
                         const __grid_constant__ CUtensorMap tk_slab, const __grid_constant__ CUtensorMap tv_slab,
                         const __grid_constant__ InterpParams p) {
  using C = InterpCfg<D>;
  using F = Frag<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sKb = sm;                        // band K
  uint8_t* sVb = sKb + C::BAND_BYTES;       // band V
  // once every warp is past the band, warp w's slab ring occupies [w * 2 BUF, (w + 1) * 2 BUF):
  // buffer b at + b * BUF_BYTES, K slot at + 0, V slot at + SLOT_BYTES
  __shared__ uint64_t bar_band, bar_slab[kWarps][kRing];
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wq = warp;
  const int h = blockIdx.x % p.heads;
  const int s = blockIdx.x / p.heads;
  const int tile = p.ntiles - 1 - (int)blockIdx.y;   // later tiles reach more rungs: start them first
  const int q0 = tile * kQ;
  const int hk = h / p.heads_per_kv;
  const int qw = q0 + 16 * wq;               // first query of this warp
  // rungs that reach at least one query of this warp (query i needs i >= lo + t, i.e.
  // i >= lo + 1 when t > 0); the reach is nondecreasing along the ascending rung list
  int n_reach = 0;
  while (n_reach < p.n_rungs && p.lo[n_reach] + (p.t[n_reach] > 0.f ? 1 : 0) <= qw + 15) ++n_reach;
  const int n_small = n_reach < p.n_small ? n_reach : p.n_small;
  const int n_large = n_reach - n_small;     // slabs of this warp: rungs n_small .. n_reach - 1

  if (tid == 0) {
    mbar_init(&bar_band, 1);
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
#pragma unroll
      for (int b = 0; b < kRing; ++b) mbar_init(&bar_slab[w][b], 1);
    abort_flag = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar_band, (uint32_t)(2 * C::BAND_BYTES));
  }
  __syncthreads();
  if (lane == 0) {
    if (warp == 0) load_rows<D>(sKb, C::BAND_CSTRIDE, &tk_band, &bar_band, hk, q0 - kBandMax, s);
    if (warp == 1) load_rows<D>(sVb, C::BAND_CSTRIDE, &tv_band, &bar_band, hk, q0 - kBandMax, s);
  }

  const int g = lane >> 2, t4 = lane & 3;    // mma fragment coordinates: rows g, g+8; cols 2t, 2t+1
  const float c = p.scale_log2;
  const float kNegInf = __int_as_float(0xff800000);

  // Q operand straight from global memory (rows past the end read the last row; never stored)
  uint32_t qa[F::KS][4];
  {
    const int last = p.n_tokens - 1;
    const int i_lo = qw + g < last ? qw + g : last, i_hi = qw + g + 8 < last ? qw + g + 8 : last;
    const __nv_bfloat16* base = p.q + (int64_t)s * p.q_sb + (int64_t)h * p.q_sh;
    load_qfrag<D>(base + (int64_t)i_lo * p.q_sn, base + (int64_t)i_hi * p.q_sn, t4, qa);
  }

  // warp-uniform wait results: the fragment code below uses full-warp shuffles
  bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_band, 0, &abort_flag, &g_interp_err, kErrTimeout));

  RungState<D> st;
#pragma unroll
  for (int nt = 0; nt < F::NT; ++nt) st.o[nt][0] = st.o[nt][1] = st.o[nt][2] = st.o[nt][3] = 0.f;
  st.m_lo = st.m_hi = kNegInf;
  st.l_lo = st.l_hi = 0.f;
  const int hl = (lane & ~3) | (g >> 1);     // lane of this quad that holds the diagonal
  const bool holder = (t4 == (g >> 1));
  const int e_sel = g & 1;                   // which of the two fragment columns is diagonal
  const int i_lo = qw + g, i_hi = qw + g + 8;

  if (ok) {
    // ---------------- window: keys [qw - Dr, qw + 16), band row = key - (q0 - 64)
    uint64_t keep = p.keep[lane];
    const int lim = p.dr - qw;               // window columns below lim are keys < 0 (first tile only)
    if (lim > 0) {
#pragma unroll
      for (int nt = 0; nt < 2 * NKT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (8 * nt + 2 * t4 + (e & 1) < lim) keep &= ~(1ull << (4 * nt + e));
    }
    const int row0 = 16 * wq + kBandMax - p.dr;
    const KV kb_tile{smem_u32(sKb), (uint32_t)C::BAND_CSTRIDE}, vb_tile{smem_u32(sVb), (uint32_t)C::BAND_CSTRIDE};
    float sb[2 * NKT][4];
    float mx_lo = kNegInf, mx_hi = kNegInf;
#pragma unroll
    for (int nt = 0; nt < 2 * NKT; ++nt) {
      uint32_t u[2 * F::KS];
      load_kfrag<D>(kb_tile, row0 + 8 * nt + g, t4, u);
      sb[nt][0] = sb[nt][1] = sb[nt][2] = sb[nt][3] = 0.f;
      qk_ntile<D>(sb[nt], qa, u);
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
    st.m_lo = mx_lo * c;                     // finite: distance 0 is always kept
    st.m_hi = mx_hi * c;
    // P = exp2(s c - m); row sums of the bf16 P come from one more MMA against a ones matrix
    float lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < NKT; ++j) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(ex2_approx(fmaf(sb[2 * j][0], c, -st.m_lo)), ex2_approx(fmaf(sb[2 * j][1], c, -st.m_lo)));
      pa[1] = pack_bf16x2(ex2_approx(fmaf(sb[2 * j][2], c, -st.m_hi)), ex2_approx(fmaf(sb[2 * j][3], c, -st.m_hi)));
      pa[2] = pack_bf16x2(ex2_approx(fmaf(sb[2 * j + 1][0], c, -st.m_lo)),
                          ex2_approx(fmaf(sb[2 * j + 1][1], c, -st.m_lo)));
      pa[3] = pack_bf16x2(ex2_approx(fmaf(sb[2 * j + 1][2], c, -st.m_hi)),
                          ex2_approx(fmaf(sb[2 * j + 1][3], c, -st.m_hi)));
      mma16816(lsum, pa, kOnesBf16x2, kOnesBf16x2);
      uint32_t vbf[D / 16][4];
      load_v16<D>(vb_tile, row0 + 16 * j, lane, vbf);
      pv_16<D>(st.o, pa, vbf);
    }
    st.l_lo = lsum[0];
    st.l_hi = lsum[2];

    // ---------------- near rungs: both rows in the band (query r: band rows ra + r, ra - 1 + r)
    for (int k = 0; k < n_small; ++k) {
      const int lo = p.lo[k];
      const float t = p.t[k];
      const bool two = t > 0.f;                // warp-uniform
      const int far = lo + (two ? 1 : 0);
      const int ra = 16 * wq + kBandMax - lo;  // >= 1 since lo <= 63
      float sa_lo, sa_hi, sb_lo = 0.f, sb_hi = 0.f;
      // (the pair's block reads up to 7 rows past the K band, into the V band: unused values)
      if (two) diag_scores_pair<D>(kb_tile, ra - 1, g, t4, qa, sa_lo, sa_hi, sb_lo, sb_hi);
      else diag_scores<D>(kb_tile, ra, g, t4, hl, e_sel, qa, sa_lo, sa_hi);
      enter_rung<D>(st, sa_lo, sa_hi, sb_lo, sb_hi, t, two, i_lo >= far, i_hi >= far, c, vb_tile, ra, ra - 1, lane,
                 holder, e_sel);
    }
  }

  // The band is read: its memory becomes the warps' slab rings.
  __syncthreads();
  uint8_t* ring = sm + wq * (kRing * C::BUF_BYTES);
  int issued = 0;
  if (lane == 0 && !abort_flag) {
    for (; issued < kRing && issued < n_large; ++issued) {
      const int lo = p.lo[n_small + issued];
      uint8_t* dst = ring + issued * C::BUF_BYTES;
      mbar_arrive_expect_tx(&bar_slab[wq][issued], (uint32_t)C::SLAB_TX);
      load_rows<D>(dst, C::CHUNK_SLOT, &tk_slab, &bar_slab[wq][issued], hk, qw - lo - 1, s);
      load_rows<D>(dst + C::SLOT_BYTES, C::CHUNK_SLOT, &tv_slab, &bar_slab[wq][issued], hk, qw - lo - 1, s);
    }
  }
  ok = ok && !abort_flag;

  // ---------------- far rungs: slab row r + 1 is distance lo of query r, slab row r distance lo + 1
  for (int j = 0; j < n_large && ok; ++j) {
    const int b = j % kRing;
    ok = __all_sync(0xffffffffu, mbar_wait(&bar_slab[wq][b], (uint32_t)(j / kRing) & 1u, &abort_flag,
                                           &g_interp_err, kErrTimeout));
    if (!ok) break;
    const int k = n_small + j;
    const int lo = p.lo[k];
    const float t = p.t[k];
    const bool two = t > 0.f;
    const int far = lo + (two ? 1 : 0);
    const KV kt{smem_u32(ring + b * C::BUF_BYTES), (uint32_t)C::CHUNK_SLOT};
    const KV vt{kt.base + C::SLOT_BYTES, (uint32_t)C::CHUNK_SLOT};
    float sa_lo, sa_hi, sb_lo = 0.f, sb_hi = 0.f;
    // (the pair's block reads rows 17 .. 23 of the 24-row slot: unused values)
    if (two) diag_scores_pair<D>(kt, 0, g, t4, qa, sa_lo, sa_hi, sb_lo, sb_hi);
    else diag_scores<D>(kt, 1, g, t4, hl, e_sel, qa, sa_lo, sa_hi);
    enter_rung<D>(st, sa_lo, sa_hi, sb_lo, sb_hi, t, two, i_lo >= far, i_hi >= far, c, vt, 1, 0, lane, holder,
                  e_sel);
    // every lane has read the buffer: refill it with the slab kRing ahead
    __syncwarp();
    if (lane == 0 && issued < n_large && !abort_flag) {
      const int lo2 = p.lo[n_small + issued];
      uint8_t* dst = ring + b * C::BUF_BYTES;
      mbar_arrive_expect_tx(&bar_slab[wq][b], (uint32_t)C::SLAB_TX);
      load_rows<D>(dst, C::CHUNK_SLOT, &tk_slab, &bar_slab[wq][b], hk, qw - lo2 - 1, s);
      load_rows<D>(dst + C::SLOT_BYTES, C::CHUNK_SLOT, &tv_slab, &bar_slab[wq][b], hk, qw - lo2 - 1, s);
      ++issued;
    }
  }

  if (ok && !abort_flag) {
    // ---------------- epilogue: O / l (bf16) and LSE
    const float inv_lo = 1.f / st.l_lo, inv_hi = 1.f / st.l_hi;   // l > 0: every query keeps itself
    __nv_bfloat16* orow_lo = p.o + (int64_t)s * p.o_sb + (int64_t)i_lo * p.o_sn + (int64_t)h * p.o_sh;
    __nv_bfloat16* orow_hi = p.o + (int64_t)s * p.o_sb + (int64_t)i_hi * p.o_sn + (int64_t)h * p.o_sh;
#pragma unroll
    for (int nt = 0; nt < F::NT; ++nt) {
      const int col = 8 * nt + 2 * t4;
      if (i_lo < p.n_tokens)
        *reinterpret_cast<uint32_t*>(orow_lo + col) = pack_bf16x2(st.o[nt][0] * inv_lo, st.o[nt][1] * inv_lo);
      if (i_hi < p.n_tokens)
        *reinterpret_cast<uint32_t*>(orow_hi + col) = pack_bf16x2(st.o[nt][2] * inv_hi, st.o[nt][3] * inv_hi);
    }
    if (t4 == 0) {
      float* lrow = p.lse + ((int64_t)s * p.heads + h) * p.n_tokens;
      if (i_lo < p.n_tokens) lrow[i_lo] = (st.m_lo + __log2f(st.l_lo)) * 0.69314718055994531f;
      if (i_hi < p.n_tokens) lrow[i_hi] = (st.m_hi + __log2f(st.l_hi)) * 0.69314718055994531f;
    }
  }
  // A CTA leaves only with none of its copies in flight: after an abort each warp drains
  // the slabs it issued and has not waited for, warp 0 the band.
  __syncthreads();
  if (abort_flag && lane == 0) {
    int never = 0;
    if (warp == 0) mbar_wait(&bar_band, 0, &never, &g_interp_err, kErrTimeout);
    for (int j = issued - kRing < 0 ? 0 : issued - kRing; j < issued; ++j)
      mbar_wait(&bar_slab[wq][j % kRing], (uint32_t)(j / kRing) & 1u, &never, &g_interp_err, kErrTimeout);
  }
}

template <int D, int NKT>
int launch_nkt(const CUtensorMap& kb, const CUtensorMap& vb, const CUtensorMap& ks, const CUtensorMap& vs,
               const InterpParams& p, int batch, cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)InterpCfg<D>::SMEM;
  if (cudaFuncSetAttribute(offset_interp_kernel<D, NKT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SA_ERR_CUDA;
  dim3 grid((unsigned)(batch * p.heads), (unsigned)p.ntiles);
  offset_interp_kernel<D, NKT><<<grid, kWarps * 32, smem, stream>>>(kb, vb, ks, vs, p);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

template <int D>
int launch_d(const InterpArgs& a, const InterpParams& p, cudaStream_t stream) {
  using C = InterpCfg<D>;
  const CUtensorMapSwizzle swz = D == 32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap kb, vb, ks, vs;
  if (!encode_bhnd_map(&kb, a.k, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::BOX_D, kBandRows, swz) ||
      !encode_bhnd_map(&vb, a.v, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::BOX_D, kBandRows, swz) ||
      !encode_bhnd_map(&ks, a.k, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::BOX_D, kSlabRows, swz) ||
      !encode_bhnd_map(&vs, a.v, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::BOX_D, kSlabRows, swz))
    return SA_ERR_UNSUPPORTED;
  switch ((16 + p.dr) / 16) {
    case 1: return launch_nkt<D, 1>(kb, vb, ks, vs, p, a.batch, stream);
    case 2: return launch_nkt<D, 2>(kb, vb, ks, vs, p, a.batch, stream);
    case 3: return launch_nkt<D, 3>(kb, vb, ks, vs, p, a.batch, stream);
    case 4: return launch_nkt<D, 4>(kb, vb, ks, vs, p, a.batch, stream);
    default: return launch_nkt<D, 5>(kb, vb, ks, vs, p, a.batch, stream);
  }
}

}  // namespace

int launch_offset_interp_fwd(const InterpArgs& a, cudaStream_t stream) {
  if (a.head_dim != 32 && a.head_dim != 64 && a.head_dim != 128) return SA_ERR_UNSUPPORTED;
  if (a.window < 0 || a.window > kBandMax || a.n_rungs < 0 || a.n_rungs > kMaxInterpRungs) return SA_ERR_UNSUPPORTED;
  if ((int64_t)a.batch * a.heads > 0x7fffffff || (a.n_tokens + kQ - 1) / kQ > 65535) return SA_ERR_UNSUPPORTED;
  InterpParams p;
  p.n_tokens = a.n_tokens;
  p.heads = a.heads;
  p.heads_per_kv = a.heads / a.kv_heads;
  p.ntiles = (a.n_tokens + kQ - 1) / kQ;
  p.dr = (a.window + 15) / 16 * 16;
  const int nkt = (16 + p.dr) / 16;
  // rungs: ascending distance, the near ones (lo + 1 <= 64) first
  p.n_rungs = a.n_rungs;
  p.n_small = 0;
  for (int r = 0; r < kMaxInterpRungs; ++r) {
    p.lo[r] = r < a.n_rungs ? a.lo[r] : 0;
    p.t[r] = r < a.n_rungs ? a.t[r] : 0.f;
  }
  for (int r = 0; r < a.n_rungs; ++r) {
    if (r > 0 && (a.lo[r] < a.lo[r - 1] || (a.lo[r] == a.lo[r - 1] && a.t[r] < a.t[r - 1]))) return SA_ERR_UNSUPPORTED;
    if (a.lo[r] < 0 || !(a.t[r] >= 0.f && a.t[r] <= 1.f)) return SA_ERR_INVALID_ARG;
    if (a.lo[r] + 1 <= kBandMax) p.n_small = r + 1;
  }
  // lane (g, t) holds score elements (row g + 8(e>>1), window column 8 nt + 2t + (e&1));
  // window column col of row rr is at distance rr + Dr - col
  for (int lane = 0; lane < 32; ++lane) {
    const int g = lane >> 2, t = lane & 3;
    unsigned long long bits = 0ull;
    for (int nt = 0; nt < 2 * nkt; ++nt)
      for (int e = 0; e < 4; ++e) {
        const int rr = g + 8 * (e >> 1), col = 8 * nt + 2 * t + (e & 1);
        const int dist = rr + p.dr - col;
        if (dist >= 0 && dist <= a.window) bits |= 1ull << (4 * nt + e);
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

unsigned int interp_read_and_clear_error(cudaStream_t stream) {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_interp_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
  cudaMemcpyToSymbolAsync(g_interp_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  return v;
}

}  // namespace sa
