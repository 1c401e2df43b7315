// Block-sparse attention forward at head dimension 128: one item stream per CTA (included by
// attn_fwd.cu after the shared parts in attn_fwd_common.cuh).
//
// At d = 128 two pipelines per SM do not fit in TMEM without writing P over S, which makes
// each pipeline's QK, softmax and PV strictly serial. Here one stream of items per CTA keeps
// two score buffers and two P buffers beside one O:
//
// TMEM (512 columns): S_0 [0, 128), S_1 [128, 256), P_0 [256, 320), P_1 [320, 384) (bf16
// pairs), O [384, 512). Key tile j uses S_(j%2) and P_(j%2): the QK of tile j+1 runs while the
// softmax works on tile j, and the PV of tile j runs while the softmax works on tile j+1.
//
// Warp roles (512 threads, 16 warps; warp w runs on SM sub-partition w % 4):
//   warps 0-7   softmax: warp w reads TMEM lane quarter w % 4 (query rows 32(w%4) ..) and
//               key columns 64(w/4) .. 64(w/4)+63 of each tile; the two warps of a lane
//               quarter exchange their half-row maxima through shared memory once per tile,
//               so both use the same running maximum. At an item's end they hand its rows'
//               max and sums to the epilogue warps and go on with the next item.
//   warp 8      lane 0 loads Q, K and V by TMA as the batches arrive (V one tile behind K)
//   warp 9      lane 0 issues the QK MMAs  S_(j%2) = Q K_j^T  (N = keys of the tile)
//   warp 10     lane 0 issues the PV MMAs  O += P_(j%2) V_j   (A = P from TMEM, B = V MN-major)
//               Two issuing threads: one thread's dependent tcgen05.mma costs about 67 cycles
//               whatever N <= 128 is, so the QK and PV streams run side by side.
//   warp 11     planner: claims items, builds the key-block union, publishes the item's key
//               tiles into a ring of two batches
//   warps 12-15 epilogue: once an item's last PV has completed, O / l and the LSE of its rows
//               (warp w: TMEM lane quarter w % 4); the next item's first PV waits for it.
#pragma once
#include "attn_fwd_common.cuh"

namespace sa {
namespace {

constexpr uint32_t kColS = 0, kColP = 256, kColO = 384;
constexpr int kStreamSoftmaxWarps = 8;   // two per TMEM lane quarter (one per half of the key tile)
constexpr int kEpilogueWarps = 4;        // one per TMEM lane quarter
constexpr int kStreamConsumers = 3 + kStreamSoftmaxWarps;   // loader, QK thread, PV thread, softmax warps
static_assert(kColO + 128 <= kTmemCols, "TMEM columns");

struct StreamBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kMaxStages], k_empty[kMaxStages], v_full[kMaxStages], v_empty[kMaxStages];
  uint64_t m_full[kMetaRing], m_empty[kMetaRing];     // batch ring
  uint64_t s_full[2];         // QK_j has written S_(j%2) (phase j / 2)
  uint64_t s_free[2];         // the softmax warps have loaded S_(j%2) (phase j / 2)
  uint64_t p_full[2];         // the softmax warps have stored P_(j%2) (phase j / 2)
  uint64_t pair[4];           // the two softmax warps of a lane quarter: row max exchange
  uint64_t o_full;            // the last PV of an item with key tiles has completed (phase: the item)
  uint64_t o_free;            // the epilogue warps have read that item's O
  uint64_t epi_full[2];       // the softmax warps have written epilogue entry e (an item's max and sums)
  uint64_t epi_empty[2];      // the epilogue warps have read entry e
  uint64_t drain_qk, drain_pv;
};

// What the softmax warps hand to the epilogue warps for one finished item.
struct EpiEntry {
  int item;                   // work item (-1: the launch is done)
  int slot;                   // partial-result slot of a split item's part (-1: write O and LSE)
  int has_tiles;              // the item had key tiles: its output is in O
  int pad;
  float m[kTile];             // running reference max per row (log2 units)
  float l[2][kTile];          // row sums of the two key halves
};

// S_(g%2) = Q K_g^T for every key tile g, as soon as its K has landed and the softmax has
// loaded S_(g-2) from the same buffer.
template <int D>
__device__ void qk_issuer(StreamBars& bars, const Batch* ring, uint8_t* sQ, uint8_t* sK, uint32_t tmem,
                          volatile int* abort_flag) {
  using C = Cfg<D>;
  const uint64_t qdesc = make_smem_desc(smem_u32(sQ), 16, C::ATOM, C::SWZ);
  const uint64_t kdesc0 = make_smem_desc(smem_u32(sK), 16, C::ATOM, C::SWZ);
  int g = 0;                // key tiles whose QK is issued
  int item_local = -1;
  int qb = 0;
  uint64_t a0 = qdesc;
  bool ok = true;
  for (int mt = 0;; ++mt) {
    int4 hdr;
    if (!(ok = wait_batch(bars, ring, mt, hdr, abort_flag))) break;
    const Batch& e = ring[mt % kMetaRing];
    if (hdr.x == kKindDone) {
      mbar_arrive(&bars.m_empty[mt % kMetaRing]);
      break;
    }
    if (hdr.w & kFirst) {
      ++item_local;
      qb = item_local % C::QB;
      if (!(ok = wait_bar(&bars.q_full[qb], (item_local / C::QB) & 1, abort_flag))) break;
      a0 = qdesc + (uint64_t)((qb * C::Q_BYTES) >> 4);
    }
    const uint4 ncw = ld_shared_u4(&e.nch[0]);
    for (int i = 0; i < hdr.y; ++i) {
      const int nkeys = 32 * (int)((word_of(ncw, i >> 2) >> (8 * (i & 3))) & 0xffu);
      const int stage = g % C::KS;
      const int b = g & 1;
      if (!(ok = wait_bar(&bars.k_full[stage], (uint32_t)(g / C::KS) & 1u, abort_flag))) break;
      if (g >= 2 && !(ok = wait_bar(&bars.s_free[b], (uint32_t)((g - 2) >> 1) & 1u, abort_flag))) break;
      tc_fence_after();
      const uint32_t idesc = make_idesc_bf16(128, (uint32_t)nkeys, 0, 0);
      const uint64_t b0 = kdesc0 + (uint64_t)((stage * C::KV_BYTES) >> 4);
      const uint32_t tS = tmem + kColS + 128u * b;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tS, a0 + kmajor_step<D>(ks, C::Q_CHUNK), b0 + kmajor_step<D>(ks, C::KV_CHUNK), idesc,
                    ks > 0 ? 1u : 0u);
      mma_commit(&bars.k_empty[stage]);   // frees the K stage
      mma_commit(&bars.s_full[b]);        // S_g is ready
      ++g;
    }
    if (!ok) break;
    mbar_arrive(&bars.m_empty[mt % kMetaRing]);
    if (hdr.w & kLast) mma_commit(&bars.q_empty[qb]);   // all QKs of this item issued
  }
  // Make sure no MMA of this thread is still writing TMEM when the CTA frees it.
  mma_commit(&bars.drain_qk);
  drain_bar(&bars.drain_qk, 0);
}

// O += P_(g%2) V_g for every key tile g once the softmax has stored P_g. An item's first PV
// (accumulate = 0) waits until the epilogue warps have read the previous item's output, and the
// commit after its last PV tells them that its output is complete.
template <int D>
__device__ void pv_issuer(StreamBars& bars, const Batch* ring, uint8_t* sV, uint32_t tmem, volatile int* abort_flag) {
  using C = Cfg<D>;
  // V is the MN-major B operand of PV: N = d runs across the d-chunks (KV_CHUNK apart)
  const uint64_t vdesc0 = make_smem_desc(smem_u32(sV), C::KV_CHUNK, C::ATOM, C::SWZ);
  const uint32_t tO = tmem + kColO;
  constexpr uint32_t idesc = make_idesc_bf16(128, D, 0, 1);
  int g = 0;                // key tiles whose PV is issued
  int with_tiles = 0;       // items with key tiles seen so far
  bool ok = true;
  bool o_init = false;
  bool has_tiles = false;   // the current item has key tiles
  for (int mt = 0;; ++mt) {
    int4 hdr;
    if (!(ok = wait_batch(bars, ring, mt, hdr, abort_flag))) break;
    const Batch& e = ring[mt % kMetaRing];
    if (hdr.x == kKindDone) {
      mbar_arrive(&bars.m_empty[mt % kMetaRing]);
      break;
    }
    if (hdr.w & kFirst) {
      has_tiles = hdr.y > 0;
      if (has_tiles) {
        // the previous item's output has been read
        if (with_tiles >= 1 && !(ok = wait_bar(&bars.o_free, (uint32_t)(with_tiles - 1) & 1u, abort_flag))) break;
        ++with_tiles;
        o_init = false;
      }
    }
    const uint4 ncw = ld_shared_u4(&e.nch[0]);
    for (int i = 0; i < hdr.y; ++i) {
      const int nkeys = 32 * (int)((word_of(ncw, i >> 2) >> (8 * (i & 3))) & 0xffu);
      const int stage = g % C::VS;
      const int b = g & 1;
      if (!(ok = wait_bar(&bars.p_full[b], (uint32_t)(g >> 1) & 1u, abort_flag))) break;
      if (!(ok = wait_bar(&bars.v_full[stage], (uint32_t)(g / C::VS) & 1u, abort_flag))) break;
      tc_fence_after();
      const uint32_t tP = tmem + kColP + 64u * b;
      const uint64_t b0 = vdesc0 + (uint64_t)((stage * C::KV_BYTES) >> 4);
      if (nkeys == kKeys) {
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks)
          mma_bf16_ts(tO, tP + 8u * ks, b0 + (uint64_t)((16 * ks * C::ROWB) >> 4), idesc, (o_init || ks > 0) ? 1u : 0u);
      } else {
        for (int ks = 0; ks < nkeys / 16; ++ks)
          mma_bf16_ts(tO, tP + 8u * ks, b0 + (uint64_t)((16 * ks * C::ROWB) >> 4), idesc, (o_init || ks > 0) ? 1u : 0u);
      }
      o_init = true;
      // frees the V stage; tells the softmax that P_(g%2) is read and O holds PV_g
      mma_commit(&bars.v_empty[stage]);
      ++g;
    }
    if (!ok) break;
    mbar_arrive(&bars.m_empty[mt % kMetaRing]);
    if ((hdr.w & kLast) && has_tiles) mma_commit(&bars.o_full);   // the item's output is complete
  }
  mma_commit(&bars.drain_pv);
  drain_bar(&bars.drain_pv, 0);
}

// ------------------------------------------------------------------ softmax (warps 0-7) and epilogue (warps 12-15)

// Rare path of the online max: this warp's half of O (columns tOh .. tOh + D/2) *= alpha
// (O quiescent).
template <int D>
__device__ __forceinline__ void rescale_o_half(uint32_t tOh, float alpha) {
  const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll 1
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t ov[16];
    tmem_ld_x16(tOh + ch * 16, ov);
    tmem_ld_wait<16>(ov);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1])), al2), lo, hi);
      ov[j] = __float_as_uint(lo);
      ov[j + 1] = __float_as_uint(hi);
    }
    tmem_st_x16(tOh + ch * 16, ov);
  }
  tmem_st_wait();
}

// Exchanges one float per row with the other softmax warp of this lane quarter through
// shared memory (phase n of the quarter's pair barrier); returns the partner's value.
__device__ __forceinline__ bool pair_exchange(StreamBars& bars, float* xch, int quarter, int half, int lane, int n,
                                              float mine, float& theirs, volatile int* abort_flag) {
  float* slot = xch + (((n & 1) * 2 + half) * 4 + quarter) * 32;
  slot[lane] = mine;
  __syncwarp();                                    // every lane's value is written before the arrive
  if (lane == 0) mbar_arrive(&bars.pair[quarter]);
  const bool ok = __all_sync(0xffffffffu, wait_bar(&bars.pair[quarter], (uint32_t)n & 1u, abort_flag));
  theirs = xch[(((n & 1) * 2 + (half ^ 1)) * 4 + quarter) * 32 + lane];
  return ok;
}

// Output of one query row of a finished item (epilogue warps): O / l in bf16 and the LSE, or,
// for a part of a split item, O / l in fp32 and the LSE into the part's slot. tO addresses
// this row's TMEM lane in the item's O buffer.
template <int D>
__device__ __forceinline__ void store_row(const Params& p, uint32_t tO, const Item& it, int row, int slot, float m,
                                          float l, bool has_tiles) {
  const float kNegInf = __int_as_float(0xff800000);
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : kNegInf;
  if (slot >= 0) {
    float* po = p.partial + (size_t)slot * (kTile * (D + 1)) + (size_t)row * D;
#pragma unroll 2
    for (int ch = 0; ch < D / 16; ++ch) {
      uint32_t ov[16];
      if (has_tiles) {
        tmem_ld_x16(tO + 16 * ch, ov);
        tmem_ld_wait<16>(ov);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) ov[j] = 0u;
      }
      float4* dst = reinterpret_cast<float4*>(po + ch * 16);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = make_float4(__uint_as_float(ov[4 * j]) * inv, __uint_as_float(ov[4 * j + 1]) * inv,
                             __uint_as_float(ov[4 * j + 2]) * inv, __uint_as_float(ov[4 * j + 3]) * inv);
    }
    p.partial[(size_t)slot * (kTile * (D + 1)) + (size_t)kTile * D + row] = lse;
    return;
  }
  const int qtok = it.tile * kTile + row;
  const bool store = qtok < p.n_tokens;
  __nv_bfloat16* orow = p.o + (int64_t)it.s * p.o_sb + (int64_t)qtok * p.o_sn + (int64_t)it.h * p.o_sh;
#pragma unroll 2
  for (int ch = 0; ch < D / 16; ++ch) {
    uint32_t ov[16];
    if (has_tiles) {
      tmem_ld_x16(tO + 16 * ch, ov);
      tmem_ld_wait<16>(ov);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) ov[j] = 0u;
    }
    if (store) {
      uint32_t pk[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2)
        pk[j >> 1] = pack_bf16x2(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
      uint4* dst = reinterpret_cast<uint4*>(orow + ch * 16);
      dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
  }
  if (store) p.lse[((int64_t)it.s * p.heads + it.h) * p.n_tokens + qtok] = lse;
}

// Softmax with half rows; this warp handles query rows 32q .. 32q+31 of every item (q = its
// TMEM lane quarter) and key columns 64 half .. 64 half + 63 of every key tile (32-key chunks
// 2 half and 2 half + 1). At the end of an item it hands the rows' max and its half's sums to
// the epilogue warps and goes on with the next item.
template <int D>
__device__ void softmax_halves(const Params& p, StreamBars& bars, const Batch* ring, EpiEntry* epi, uint32_t tmem,
                               float* xch, volatile int* abort_flag) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int row = quarter * 32 + lane;               // query row within the tile
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const float kNegInf = __int_as_float(0xff800000);
  const float c = p.scale_log2;
  const uint64_t c2 = f2_pack(c, c);

  int g = 0;                // key tiles processed
  int npair = 0;            // phases of this quarter's pair barrier
  int n_done = 0;           // epilogue entries written
  bool ok = true;
  const uint32_t tOh = tmem + kColO + (uint32_t)(half * (D / 2)) + lane_base;   // this warp's half of O
  float m_use = kNegInf;    // running reference max, log2 units
  float l = 0.f;            // row sum of this warp's key columns
  int n_item = 0;           // key tiles of the current item
  int slot = -1;            // partial-result slot of a split item's part (-1: write O and LSE)
  for (int mt = 0;; ++mt) {
    int4 hdr;
    ok = __all_sync(0xffffffffu, wait_batch(bars, ring, mt, hdr, abort_flag));
    if (!ok) break;
    const Batch& e = ring[mt % kMetaRing];
    const bool done = hdr.x == kKindDone;
    if (!done) {
      if (hdr.w & kFirst) {
        m_use = kNegInf;
        l = 0.f;
        n_item = 0;
        slot = e.slot;
      }
      // this quarter's visibility bytes and the chunk counts of the batch's tiles
      const uint4 vqw = ld_shared_u4(&e.vq[quarter][0]);
      const uint4 ncw = ld_shared_u4(&e.nch[0]);
      for (int i = 0; i < hdr.y; ++i) {
        const int sh = 8 * (i & 3);
        const int vb = (int)((word_of(vqw, i >> 2) >> sh) & 0xffu);
        const int nch = (int)((word_of(ncw, i >> 2) >> sh) & 0xffu);
        // this warp's two chunks: visibility bits and the causal-diagonal chunk among them
        const int vis = (vb >> (2 * half)) & 3;
        const int dch_all = (vb >> 4) - 1;
        const int dch = (dch_all >= 2 * half && dch_all < 2 * half + 2) ? dch_all - 2 * half : -1;
        const int b = g & 1;

        // QK_g done
        ok = __all_sync(0xffffffffu, wait_bar(&bars.s_full[b], (uint32_t)(g >> 1) & 1u, abort_flag));
        if (!ok) break;
        tc_fence_after();
        uint32_t v[64];
        const uint32_t tS = tmem + kColS + 128u * b + 64u * half + lane_base;
        tmem_ld_x32(tS, v);
        tmem_ld_x32(tS + 32, v + 32);
        tmem_ld_wait<64>(v);
        // S_(g%2) may now be overwritten by QK_(g+2)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.s_free[b]);

        if (dch >= 0) {
          // the diagonal chunk starts at this warp's first query: row r sees columns 0 .. r
          const uint32_t kp = (2u << lane) - 1u;     // lane 31: all 32 columns
          if (dch == 0) mask_chunk(v, kp);
          else mask_chunk(v + 32, kp);
        }
        float cm = kNegInf;
        if (vis & 1) cm = chunk_max(v, cm);
        if (vis & 2) cm = chunk_max(v + 32, cm);
        // the row max over both halves of the key tile
        float other;
        ok = pair_exchange(bars, xch, quarter, half, lane, npair++, cm, other, abort_flag);
        if (!ok) break;
        const float mx = fmaxf(cm, other) * c;       // -inf stays -inf
        const bool need = mx > m_use + 8.0f;
        float alpha = 1.f;
        bool o_scale = false;
        if (__any_sync(0xffffffffu, need)) {
          // the running max grows by more than 2^8: rescale l now and O before this tile's PV
          alpha = need ? ex2_approx(m_use - mx) : 1.f;   // 0 when m_use = -inf
          o_scale = need && m_use != kNegInf && n_item > 0;
          l *= alpha;
          if (need) m_use = mx;
        }
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t rs[2] = {0ull, 0ull};
        uint32_t pk[32];
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          if ((vis >> ch) & 1) {
            chunk_exp(v + 32 * ch, c2, negm2, pk + 16 * ch, rs);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[16 * ch + j] = 0u;
          }
        }
        // P_(g%2) is free once PV_(g-2) is complete
        if (g >= 2) {
          ok = __all_sync(0xffffffffu,
                          wait_bar(&bars.v_empty[(g - 2) % C::VS], (uint32_t)((g - 2) / C::VS) & 1u, abort_flag));
          if (!ok) break;
        }
        if (__any_sync(0xffffffffu, o_scale)) {
          // O must hold PV_(g-1) before it is rescaled (rare: the max grew by more than 2^8)
          ok = __all_sync(0xffffffffu,
                          wait_bar(&bars.v_empty[(g - 1) % C::VS], (uint32_t)((g - 1) / C::VS) & 1u, abort_flag));
          if (!ok) break;
          tc_fence_after();
          rescale_o_half<D>(tOh, alpha);
        }
        tc_fence_after();
        const uint32_t tP = tmem + kColP + 64u * b + 32u * half + lane_base;
        if (2 * half < nch) tmem_st_x16(tP, pk);
        if (2 * half + 1 < nch) tmem_st_x16(tP + 16, pk + 16);
        {
          const uint64_t rs2 = f2_add(rs[0], rs[1]);
          float rs_lo, rs_hi;
          f2_unpack(rs2, rs_lo, rs_hi);
          l += rs_lo + rs_hi;
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[b]);
        ++g;
        ++n_item;
      }
      if (!ok) break;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.m_empty[mt % kMetaRing]);
    if (!done && !(hdr.w & kLast)) continue;

    // hand the item (or the end of the launch) to the epilogue warps
    const int ie = n_done & 1;
    if (n_done >= 2) {
      ok = __all_sync(0xffffffffu, wait_bar(&bars.epi_empty[ie], (uint32_t)((n_done >> 1) - 1) & 1u, abort_flag));
      if (!ok) break;
    }
    EpiEntry& E = epi[ie];
    if (!done) {
      if (half == 0) E.m[row] = m_use;
      E.l[half][row] = l;
    }
    if (warp == 0 && lane == 0) {
      E.item = done ? -1 : hdr.z;
      E.slot = slot;
      E.has_tiles = n_item > 0 ? 1 : 0;
    }
    __syncwarp();                                    // the lanes' values are written before the release
    if (lane == 0) mbar_arrive(&bars.epi_full[ie]);
    ++n_done;
    if (done) break;
  }
}

// Epilogue (warps 12-15, warp w reads TMEM lane quarter w % 4): for every item the softmax
// warps hand over, waits for the item's last PV, writes its rows' O / l and LSE, and frees O
// for the next item's PVs.
template <int D>
__device__ void epilogue(const Params& p, StreamBars& bars, const EpiEntry* epi, uint32_t tmem,
                         volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  int with_tiles = 0;       // items with key tiles written
  for (int n = 0;; ++n) {
    const int ie = n & 1;
    if (!__all_sync(0xffffffffu, wait_bar(&bars.epi_full[ie], (uint32_t)(n >> 1) & 1u, abort_flag))) break;
    const EpiEntry& E = epi[ie];
    const int k = E.item;
    if (k < 0) break;
    const int slot = E.slot;
    const bool has = E.has_tiles != 0;
    const float m = E.m[row];
    const float l = E.l[0][row] + E.l[1][row];
    if (has) {
      if (!__all_sync(0xffffffffu, wait_bar(&bars.o_full, (uint32_t)with_tiles & 1u, abort_flag))) break;
      tc_fence_after();
    }
    store_row<D>(p, tmem + kColO + lane_base, decode_item(p, k), row, slot, m, l, has);
    if (has) {
      // O has been read: the next item's PVs may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.o_free);
      ++with_tiles;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.epi_empty[ie]);
  }
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_wide_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                         const __grid_constant__ Params p) {
  // `to` (the output map) is not used here: the epilogue warps write O with plain stores
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  static_assert(C::WIDE, "one-stream kernel: head dimension 128");
  __shared__ StreamBars bars;
  __shared__ Batch ring[kMetaRing];
  __shared__ EpiEntry epi[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], kStreamSoftmaxWarps);
      mbar_init(&bars.p_full[i], kStreamSoftmaxWarps);
    }
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < kMetaRing; ++i) {
      mbar_init(&bars.m_full[i], 1);
      mbar_init(&bars.m_empty[i], kStreamConsumers);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars.pair[i], 2);
    mbar_init(&bars.o_full, 1);
    mbar_init(&bars.o_free, kEpilogueWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.epi_full[i], kStreamSoftmaxWarps);
      mbar_init(&bars.epi_empty[i], kEpilogueWarps);
    }
    mbar_init(&bars.drain_qk, 1);
    mbar_init(&bars.drain_pv, 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == 9) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Register split: warpgroups 0-1 (softmax) grow, warpgroups 2-3 (control) shrink, at the
  // top of their branches (the compiler budgets the code that follows by it); the sum equals
  // the launch allocation (checked on the host), so the growth always completes.
  static_assert(kSoftmaxRegs == 184 && kCtrlRegs == 72, "register split literals");

  uint8_t* sQ = sbase;
  uint8_t* sK = sQ + C::QB * C::Q_BYTES;
  uint8_t* sV = sK + C::KS * C::KV_BYTES;
  UnionSmem& un = *reinterpret_cast<UnionSmem*>(sV + C::VS * C::KV_BYTES);
  float* xch = reinterpret_cast<float*>(sV + C::VS * C::KV_BYTES + C::UNION_BYTES);

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;" ::: "memory");
    softmax_halves<D>(p, bars, ring, epi, tmem, xch, &abort_flag);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    if (warp == 8) {
      if ((threadIdx.x & 31) == 0) loader<D>(p, &tq, &tk, &tv, bars, ring, sQ, sK, sV, &abort_flag);
      __syncwarp();
    } else if (warp == 9) {
      if ((threadIdx.x & 31) == 0) qk_issuer<D>(bars, ring, sQ, sK, tmem, &abort_flag);
      __syncwarp();
    } else if (warp == 10) {
      if ((threadIdx.x & 31) == 0) pv_issuer<D>(bars, ring, sV, tmem, &abort_flag);
      __syncwarp();
    } else if (warp == 11) {
      planner<D>(p, bars, ring, un, &abort_flag);
    } else {
      epilogue<D>(p, bars, epi, tmem, &abort_flag);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace sa
