// Block-sparse flash-attention forward for sm_103a (tcgen05 + TMEM + TMA). Head dimensions
// 32 and 64 run the two-pipeline kernel below; head dimension 128 runs the one-stream kernel
// of attn_fwd_wide.cuh. Both take their work items, key tiles and TMA loads from
// attn_fwd_common.cuh, and share the split-row combine (K9) and the launch code at the end.
//
// Two-pipeline kernel (d <= 64), with 128-key score tiles and one full score row per softmax
// thread: the fixed per-step cost of the softmax (waits, arrivals, TMEM round trips, the
// online-max bookkeeping) covers 128 scores, and no two warps ever exchange a row maximum.
//
// TMEM of pipeline x (256 columns each, two pipelines per CTA): S [256x, +128), P
// [256x + 128, +64) (bf16 pairs), O [256x + 192, +d). P has columns of its own, so the QK of
// key tile j+1 may overwrite S as soon as the softmax has loaded S_j into registers; the
// exponentials of tile j then overlap with QK_{j+1}.
//
// Warp roles (512 threads, 16 warps; warp w runs on SM sub-partition w % 4):
//   warps 0-3   softmax of pipeline 0, warp w reads TMEM lane quarter w (query rows 32w ..)
//   warps 4-7   softmax of pipeline 1
//   warps 14, 15 planners of pipeline 0 / 1: claim items, build the key-block union, publish
//               the item's key tiles into a ring of two batches (up to 16 tiles per entry):
//               the next item's union is built under the current item, and a planner never
//               claims many items ahead of its pipeline
//   warps 8, 11 lane 0 loads Q, K and V of pipeline 0 / 1 by TMA as the batches arrive
//   warps 12, 13 idle (the fourth warpgroup's remainder)
//   warps 9, 10 lane 0 issues the tcgen05 MMAs of pipeline 0 / 1 in the order QK_j, PV_{j-1}:
//                 S = Q K_j^T   (N = keys of the tile, up to 128)
//                 O += P_j V_j  (A = P_j from TMEM, B = V_j MN-major; K = 16 keys per MMA)
//               the next tile's scores are requested as soon as S is free, before the previous
//               tile's probabilities are ready. The commit that frees a K stage also tells the
//               softmax that S is ready, and the one that frees a V stage tells it that P has
//               been read and O written.
#include <string.h>

#include <atomic>

#include "attn_fwd_common.cuh"
#include "attn_fwd_wide.cuh"

namespace sa {
namespace {

constexpr int kSoftmaxWarps = 4;      // per pipeline: one per TMEM lane quarter
// Register split of this kernel: softmax warpgroups 192, control warpgroups 64 (8 x 192 + 8 x 64
// = 16 x 128). Measured against 184 / 72: 8K top-16 0.1912-0.1932 -> 0.1911 ms, BigBird 16K
// 0.391-0.395 -> 0.390-0.391 ms; 200 / 56 (control code spills) no better.
constexpr int kPipeSoftmaxRegs = 192;
constexpr int kPipeCtrlRegs = 64;
static_assert(8 * kPipeSoftmaxRegs + 8 * kPipeCtrlRegs == 16 * kLaunchRegs, "register split");
// d = 64: items of at least this many key tiles store O by TMA (measured at 1, 2, 4 and 8:
// 1-4 equal within noise, 8 slower on BigBird 16K; 1 = every item with key tiles)
constexpr int kTmaStoreTiles = 1;
// Of every 16 exponential pairs, these many on the FMA pipe (exp2_fma2). Measured on the 8K
// top-16 workload at 0 / 1 / 2 / 3 / 4 pairs: 193-195 / 197-199 / 199-200 / 211 / 213-215 us:
// in this kernel the exponentials are not held up by the MUFU pipe but by issue slots and
// latency, so the polynomial's extra instructions only add time.
constexpr int kPolyPairs = 0;
constexpr int kMetaConsumers = 2 + kSoftmaxWarps;   // MMA thread, loader, softmax warps
__host__ __device__ constexpr uint32_t col_s(int x) { return 256u * x; }
__host__ __device__ constexpr uint32_t col_p(int x) { return 256u * x + 128u; }
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u * x + 192u; }

struct PipeBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kMaxStages], k_empty[kMaxStages], v_full[kMaxStages], v_empty[kMaxStages];
  uint64_t m_full[kMetaRing], m_empty[kMetaRing];     // batch ring
  uint64_t s_free;            // the softmax has loaded S_j (phase j)
  uint64_t p_full;            // the softmax has stored P_j (phase j)
  uint64_t drain;
};

// ------------------------------------------------------------------ MMA issuer (warps 9, 10, lane 0)

// O += P_j V_j for the key tile held in ring stage `stage` (its V load was the kt-th),
// after P_j is stored. `o_init` says whether O already holds this item's sum.
template <int D>
__device__ __forceinline__ bool issue_pv(PipeBars& bars, uint32_t tP, uint32_t tO, uint64_t vdesc0, int j, int stage,
                                         int vkt, int nkeys, bool& o_init, volatile int* abort_flag) {
  using C = Cfg<D>;
  if (!wait_bar(&bars.p_full, (uint32_t)j & 1u, abort_flag)) return false;
  if (!wait_bar(&bars.v_full[stage], (uint32_t)(vkt / C::VS) & 1u, abort_flag)) return false;
  tc_fence_after();
  constexpr uint32_t idesc = make_idesc_bf16(128, D, 0, 1);
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
  // frees the V stage and tells the softmax that P_j is read and O is written
  mma_commit(&bars.v_empty[stage]);
  return true;
}

template <int D>
__device__ void mma_issuer(int x, PipeBars& bars, const Batch* ring, uint8_t* sQ, uint8_t* sK, uint8_t* sV,
                           uint32_t tmem, volatile int* abort_flag) {
  using C = Cfg<D>;
  const uint64_t qdesc = make_smem_desc(smem_u32(sQ), 16, C::ATOM, C::SWZ);
  const uint64_t kdesc0 = make_smem_desc(smem_u32(sK), 16, C::ATOM, C::SWZ);
  // V is the MN-major B operand of PV: N = d runs across the d-chunks (KV_CHUNK apart)
  const uint64_t vdesc0 = make_smem_desc(smem_u32(sV), C::KV_CHUNK, C::ATOM, C::SWZ);
  const uint32_t tS = tmem + col_s(x), tP = tmem + col_p(x), tO = tmem + col_o(x);
  int g = 0;                // key tiles of this pipeline whose QK is issued (K / V ring position)
  int item_local = -1;
  int qb = 0;
  uint64_t a0 = qdesc;
  bool ok = true;
  bool o_init = false;
  bool pend = false;        // PV of the previous key tile of this item not yet issued
  int p_nkeys = 0;
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
      o_init = false;
      pend = false;
    }
    const uint4 ncw = ld_shared_u4(&e.nch[0]);
    for (int i = 0; i < hdr.y; ++i) {
      const int nkeys = 32 * (int)((word_of(ncw, i >> 2) >> (8 * (i & 3))) & 0xffu);
      const int stage = g % C::KS;
      if (!(ok = wait_bar(&bars.k_full[stage], (uint32_t)(g / C::KS) & 1u, abort_flag))) break;
      // S is free once the softmax has loaded S_{g-1}
      if (g > 0 && !(ok = wait_bar(&bars.s_free, (uint32_t)(g - 1) & 1u, abort_flag))) break;
      tc_fence_after();
      const uint32_t idesc = make_idesc_bf16(128, (uint32_t)nkeys, 0, 0);
      const uint64_t b0 = kdesc0 + (uint64_t)((stage * C::KV_BYTES) >> 4);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_bf16_ss(tS, a0 + kmajor_step<D>(ks, C::Q_CHUNK), b0 + kmajor_step<D>(ks, C::KV_CHUNK), idesc,
                    ks > 0 ? 1u : 0u);
      // frees the K stage and tells the softmax that S_g is ready
      mma_commit(&bars.k_empty[stage]);
      if (pend && !(ok = issue_pv<D>(bars, tP, tO, vdesc0, g - 1, (g - 1) % C::VS, g - 1, p_nkeys, o_init,
                                     abort_flag)))
        break;
      pend = true;
      p_nkeys = nkeys;
      ++g;
    }
    if (!ok) break;
    mbar_arrive(&bars.m_empty[mt % kMetaRing]);
    if (hdr.w & kLast) {
      mma_commit(&bars.q_empty[qb]);   // all QKs of this item issued; arrives when they are done
      // the item's last PV: its completion releases the softmax epilogue
      if (pend && !(ok = issue_pv<D>(bars, tP, tO, vdesc0, g - 1, (g - 1) % C::VS, g - 1, p_nkeys, o_init,
                                     abort_flag)))
        break;
      pend = false;
    }
  }
  // Make sure no MMA of this thread is still writing TMEM when the CTA frees it.
  mma_commit(&bars.drain);
  drain_bar(&bars.drain, 0);
}

// ------------------------------------------------------------------ softmax + epilogue (warps 0-7)

// Rare path of the online max: O *= alpha for this thread's row (O quiescent).
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
  const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll 1
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t ov[32];
    tmem_ld_x32(tO + ch * 32, ov);
    tmem_ld_wait<32>(ov);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1])), al2), lo, hi);
      ov[j] = __float_as_uint(lo);
      ov[j + 1] = __float_as_uint(hi);
    }
    tmem_st_x32(tO + ch * 32, ov);
  }
  tmem_st_wait();
}

// Softmax and epilogue of pipeline x; this warp handles query rows 32q .. 32q+31 of every
// item (q = its TMEM lane quarter) and all 128 keys of every key tile. At d = 64 (with an
// output tensor map, to) an item's O / l rows are staged, 128B-swizzled, in the item's own Q
// buffer (its QKs are complete) and written by one TMA store per warp; the Q buffer is
// released to the loader (q_empty) once that store has read it.
template <int D>
__device__ void softmax_epilogue(const Params& p, int x, PipeBars& bars, const Batch* ring, uint32_t tmem,
                                 uint8_t* sQ, const CUtensorMap* to, volatile int* abort_flag) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;               // query row within the tile
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const float kNegInf = __int_as_float(0xff800000);
  const float c = p.scale_log2;
  const uint64_t c2 = f2_pack(c, c);
  const uint32_t tS = tmem + col_s(x) + lane_base;
  const uint32_t tP = tmem + col_p(x) + lane_base;
  const uint32_t tO = tmem + col_o(x) + lane_base;

  int g = 0;                // key tiles processed by this pipeline
  int item_local = -1;      // items of this pipeline (Q buffer item_local % QB)
  bool ok = true;
  Item it;
  it.s = it.h = it.tile = 0;
  int qtok = 0;
  float m_use = kNegInf;    // running reference max, log2 units
  float l = 0.f;            // row sum
  int n_item = 0;           // key tiles of the current item
  int slot = -1;            // partial-result slot of a split item's part (-1: write O and LSE)
  for (int mt = 0;; ++mt) {
    int4 hdr;
    ok = __all_sync(0xffffffffu, wait_batch(bars, ring, mt, hdr, abort_flag));
    if (!ok) break;
    const Batch& e = ring[mt % kMetaRing];
    if (hdr.x == kKindDone) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.m_empty[mt % kMetaRing]);
      break;
    }
    if (hdr.w & kFirst) {
      ++item_local;
      it = decode_item(p, hdr.z);
      qtok = it.tile * kTile + row;
      m_use = kNegInf;
      l = 0.f;
      n_item = 0;
      slot = e.slot;
      // Items of at least kTmaStoreTiles key tiles (d = 64, whole items) stage their output in
      // their Q buffer; the others (items without key tiles, split parts, other d) give the
      // buffer up now, and its release then waits only for the item's Q and QKs.
      // An item's first batch holds min(16, its key tiles) tiles, so this test and the one at
      // the item's end, on its tile count, agree.
      if (!(D == 64 && p.o_tma && slot < 0 && hdr.y >= kTmaStoreTiles)) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.q_empty[item_local % C::QB]);
      }
    }
    // this quarter's visibility bytes and the chunk counts of the batch's tiles
    const uint4 vqw = ld_shared_u4(&e.vq[quarter][0]);
    const uint4 ncw = ld_shared_u4(&e.nch[0]);
    for (int i = 0; i < hdr.y; ++i) {
      const int sh = 8 * (i & 3);
      const int vb = (int)((word_of(vqw, i >> 2) >> sh) & 0xffu);
      const int nch = (int)((word_of(ncw, i >> 2) >> sh) & 0xffu);
      const int vis = vb & 15, dch = (vb >> 4) - 1;

      // QK_g done: its commit is the (g / KS)-th completion of K stage g % KS
      ok = __all_sync(0xffffffffu, wait_bar(&bars.k_empty[g % C::KS], (uint32_t)(g / C::KS) & 1u, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld_x32(tS + 32 * ch, v + 32 * ch);
      tmem_ld_wait<128>(v);
      // S may now be overwritten by the next QK
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.s_free);

      if (dch >= 0) {
        // the diagonal chunk starts at this warp's first query: row r sees columns 0 .. r
        const uint32_t kp = (2u << lane) - 1u;       // lane 31: all 32 columns
        switch (dch) {
          case 0: mask_chunk(v, kp); break;
          case 1: mask_chunk(v + 32, kp); break;
          case 2: mask_chunk(v + 64, kp); break;
          default: mask_chunk(v + 96, kp); break;
        }
      }
      float cm = kNegInf;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        if ((vis >> ch) & 1) cm = chunk_max(v + 32 * ch, cm);
      const float mx = cm * c;                       // -inf stays -inf
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
      // All exponentials of the tile first (P_j packed in registers; the scores' registers
      // are reused as they die): only the stores of P wait for PV_{j-1}, so the tensor
      // core's PV and the next QK run under this tile's exponentials instead of in series
      // with them.
      uint32_t pk[64];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        if ((vis >> ch) & 1) {
          chunk_exp<kPolyPairs>(v + 32 * ch, c2, negm2, pk + 16 * ch, rs);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[16 * ch + j] = 0u;
        }
      }
      // PV_{g-1} has read P and finished writing O
      if (g > 0) {
        ok = __all_sync(0xffffffffu,
                        wait_bar(&bars.v_empty[(g - 1) % C::VS], (uint32_t)((g - 1) / C::VS) & 1u, abort_flag));
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, o_scale)) rescale_o<D>(tO, alpha);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        if (ch < nch) tmem_st_x16(tP + 16 * ch, pk + 16 * ch);
      {
        const uint64_t rs2 = f2_add(rs[0], rs[1]);
        float rs_lo, rs_hi;
        f2_unpack(rs2, rs_lo, rs_hi);
        l += rs_lo + rs_hi;
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full);
      ++g;
      ++n_item;
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.m_empty[mt % kMetaRing]);
    if (!(hdr.w & kLast)) continue;

    // epilogue: O / l and LSE of this query tile's rows
    if (n_item > 0) {
      ok = __all_sync(0xffffffffu, wait_bar(&bars.v_empty[(g - 1) % C::VS], (uint32_t)((g - 1) / C::VS) & 1u, abort_flag));
      if (!ok) break;
      tc_fence_after();
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse = l > 0.f ? (m_use + __log2f(l)) * 0.69314718055994531f : kNegInf;
    if (slot >= 0) {
      // a part of a split item: O / l of its key range (fp32) and its LSE, merged later
      float* po = p.partial + (size_t)slot * (kTile * (D + 1)) + (size_t)row * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        if (n_item > 0) {
          tmem_ld_x32(tO + 32 * ch, ov);
          tmem_ld_wait<32>(ov);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = 0u;
        }
        float4* dst = reinterpret_cast<float4*>(po + ch * 32);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(__uint_as_float(ov[4 * j]) * inv, __uint_as_float(ov[4 * j + 1]) * inv,
                               __uint_as_float(ov[4 * j + 2]) * inv, __uint_as_float(ov[4 * j + 3]) * inv);
      }
      p.partial[(size_t)slot * (kTile * (D + 1)) + (size_t)kTile * D + row] = lse;
    } else if (D == 64 && p.o_tma && n_item >= kTmaStoreTiles) {
      // Staged in the item's Q buffer (its QKs are complete: the last PV has been waited for):
      // rows of this warp, 128 bytes each, 128B-swizzled (16-byte chunk c of row r at
      // r * 128 + (c ^ (r & 7)) * 16) as the output map's box expects; rows past the sequence
      // end are dropped by the TMA store
      const int qb = item_local % C::QB;
      uint8_t* stg = sQ + qb * C::Q_BYTES + quarter * 32 * 128;
      const uint32_t srow = smem_u32(stg) + (uint32_t)lane * 128u;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        if (n_item > 0) {
          tmem_ld_x32(tO + 32 * ch, ov);
          tmem_ld_wait<32>(ov);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2)
          pk[j >> 1] = pack_bf16x2(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_shared_v4(srow + (uint32_t)(((4 * ch + j) ^ (lane & 7)) << 4), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                       pk[4 * j + 3]);
      }
      fence_proxy_async_smem();                      // the staged rows are visible to the TMA store
      __syncwarp();
      if (lane == 0) {
        tma_store_4d(to, stg, 0, it.h, it.tile * kTile + quarter * 32, it.s);
        bulk_commit_group();
      }
      if (qtok < p.n_tokens) p.lse[((int64_t)it.s * p.heads + it.h) * p.n_tokens + qtok] = lse;
      // the buffer goes back to the loader once the store has read it
      if (lane == 0) bulk_wait_group_read<0>();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.q_empty[qb]);
    } else {
      const bool store = qtok < p.n_tokens;
      __nv_bfloat16* orow = p.o + (int64_t)it.s * p.o_sb + (int64_t)qtok * p.o_sn + (int64_t)it.h * p.o_sh;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        if (n_item > 0) {
          tmem_ld_x32(tO + 32 * ch, ov);
          tmem_ld_wait<32>(ov);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = 0u;
        }
        if (store) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2)
            pk[j >> 1] = pack_bf16x2(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
      if (store) p.lse[((int64_t)it.s * p.heads + it.h) * p.n_tokens + qtok] = lse;
    }
    // The next item's first P store follows these O loads in program order, and the MMA
    // thread issues that item's first PV only after the P store: O is not overwritten early.
  }
  // every TMA store of this warp has completed before the CTA may exit
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                    const __grid_constant__ Params p) {
  using C = Cfg<D>;
  static_assert(!C::WIDE && 192 + D <= 256, "two-pipeline kernel: head dimension 32 or 64");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ PipeBars bars[2];
  __shared__ Batch ring[2][kMetaRing];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      PipeBars& b = bars[x];
      for (int i = 0; i < 2; ++i) {
        mbar_init(&b.q_full[i], 1);
        // released by the MMA thread (the item's QKs are done) and the softmax warps (at the
        // item's start, or once the item's output store has read the buffer)
        mbar_init(&b.q_empty[i], 1 + kSoftmaxWarps);
      }
      for (int i = 0; i < kMaxStages; ++i) {
        mbar_init(&b.k_full[i], 1);
        mbar_init(&b.k_empty[i], 1);
        mbar_init(&b.v_full[i], 1);
        mbar_init(&b.v_empty[i], 1);
      }
      for (int i = 0; i < kMetaRing; ++i) {
        mbar_init(&b.m_full[i], 1);
        mbar_init(&b.m_empty[i], kMetaConsumers);
      }
      mbar_init(&b.s_free, kSoftmaxWarps);
      mbar_init(&b.p_full, kSoftmaxWarps);
      mbar_init(&b.drain, 1);
    }
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
  static_assert(kPipeSoftmaxRegs == 192 && kPipeCtrlRegs == 64, "register split literals");

  // pipeline 0: softmax warps 0-3, loader 8, MMA 9, planner 14;
  // pipeline 1: softmax warps 4-7, MMA 10, loader 11, planner 15; warps 12, 13 idle
  // (sub-partition w % 4: the planners share 2 and 3 with an MMA thread and a loader, not 0
  // and 1 with both; BigBird 16K 0.395-0.400 -> 0.389-0.392 ms, the rest within noise)
  const int x = warp < 8 ? (warp >> 2) : ((warp == 8 || warp == 9 || warp == 14) ? 0 : 1);
  uint8_t* sQ = sbase + x * C::PIPE_BYTES;
  uint8_t* sK = sQ + C::QB * C::Q_BYTES;
  uint8_t* sV = sK + C::KS * C::KV_BYTES;
  UnionSmem& un = *reinterpret_cast<UnionSmem*>(sV + C::VS * C::KV_BYTES);

  if (warp < 8) {
    // warpgroups 0 and 1: one setmaxnreg instruction for both
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    softmax_epilogue<D>(p, x, bars[x], ring[x], tmem, sQ, &to, &abort_flag);
  } else {
    // warpgroups 2 and 3: one setmaxnreg instruction for both, then the roles
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
    if (warp == 8 || warp == 11) {
      if ((threadIdx.x & 31) == 0) loader<D>(p, &tq, &tk, &tv, bars[x], ring[x], sQ, sK, sV, &abort_flag);
      __syncwarp();
    } else if (warp == 9 || warp == 10) {
      if ((threadIdx.x & 31) == 0) mma_issuer<D>(x, bars[x], ring[x], sQ, sK, sV, tmem, &abort_flag);
      __syncwarp();
    } else if (warp == 14 || warp == 15) {
      planner<D>(p, bars[x], ring[x], un, &abort_flag);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ split-row combine (K9)
//
// Used when a launch has few work items for the GPU's item streams (see launch_d): a few long
// key lists would then leave SMs idle. fwd_plan_kernel counts the key tiles of every query tile's
// union (one warp per (mask, CSR sequence, query tile)), fwd_schedule_kernel (one CTA) cuts the
// items whose lists are longer than T tiles into parts of T tiles, each with a slot for its
// partial result, and lists the parts first, then the other items; attn_fwd_kernel runs the
// list; fwd_merge_kernel combines the parts of each split item:
//   LSE = ln sum_p exp(LSE_p),  O = sum_p exp(LSE_p - LSE) O_p.

struct SplitHdr {
  int list_len, n_split, part_tiles, n_split_items;
};

constexpr int kPlanWarps = 8;
constexpr int kMinPartTiles = 4;

__global__ void __launch_bounds__(32 * kPlanWarps) fwd_plan_kernel(const __grid_constant__ Params p, int n_groups,
                                                                    int* tiles) {
  __shared__ uint32_t bm[kPlanWarps][kMaxMaskBlocks / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * kPlanWarps + warp;
  if (g >= n_groups) return;                         // the whole warp leaves
  const int t = g % p.tiles_per_seq;
  const int cs = (g / p.tiles_per_seq) % p.csr_batches;
  const int m = g / (p.tiles_per_seq * p.csr_batches);
  const int nb = p.nb, nw = (nb + 31) >> 5;
  const int32_t* rp = p.row_ptr[m] + (size_t)cs * (nb + 1);
  const int32_t* ci = p.col_idx[m];
  const int I0 = (t * kTile) >> p.log2b;
  const int nq = min(kTile >> p.log2b, nb - I0);
  for (int w = lane; w < nw; w += 32) bm[warp][w] = 0u;
  __syncwarp();
  for (int r = 0; r < nq; ++r) {
    const int e1 = rp[I0 + r + 1];
    for (int e = rp[I0 + r] + lane; e < e1; e += 32) {
      const int X = ci[e];
      if (X >= 0 && X < nb && (!p.causal || X <= I0 + r)) atomicOr(&bm[warp][X >> 5], 1u << (X & 31));
    }
  }
  __syncwarp();
  int cnt = 0;
  for (int w = lane; w < nw; w += 32) cnt += __popc(bm[warp][w]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) tiles[g] = (cnt * (p.block >> 5) + 3) >> 2;   // 32-key chunks, four per key tile
}

// Block-wide exclusive scan of one int per thread (1024 threads); returns the total too.
__device__ __forceinline__ int block_scan_excl(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  total = warp_sums[31];
  return (warp > 0 ? warp_sums[warp - 1] : 0) + incl - v;
}

// Key tiles of work item k (its query tile's union, from the plan).
__device__ __forceinline__ int item_tiles(const Params& p, const int* tiles, int k) {
  const Item it = decode_item(p, k);
  const int m = p.n_masks > 1 ? p.head_mask[it.h] : 0;
  const int cs = p.csr_shared ? 0 : it.s;
  return tiles[(m * p.csr_batches + cs) * p.tiles_per_seq + it.tile];
}

__global__ void __launch_bounds__(1024) fwd_schedule_kernel(const __grid_constant__ Params p, const int* tiles,
                                                             int slot_cap, int n_pipes, int2* list, int4* split_items,
                                                             SplitHdr* hdr) {
  __shared__ int warp_sums[32];
  __shared__ int s_T;
  const int n = p.n_items;
  const int per = (n + 1023) / 1024;
  const int k0 = min(n, (int)threadIdx.x * per), k1 = min(n, k0 + per);
  // total work, longest item
  long long tot = 0;
  int mx = 0;
  for (int k = k0; k < k1; ++k) {
    const int t = item_tiles(p, tiles, k);
    tot += t;
    mx = max(mx, t);
  }
  // reduce (sum as int: a launch holds far fewer than 2^31 key tiles)
  int total = 0;
  block_scan_excl((int)tot, warp_sums, total);
  int big = mx;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) big = max(big, __shfl_xor_sync(0xffffffffu, big, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = big;
  __syncthreads();
  if (threadIdx.x == 0) {
    int b = 0;
    for (int w = 0; w < 32; ++w) b = max(b, warp_sums[w]);
    // about two parts of work per item stream (n_pipes: streams of the launch); parts of at
    // least kMinPartTiles key tiles
    int T = max(kMinPartTiles, (total + 2 * n_pipes - 1) / (2 * n_pipes));
    // No split when the longest item is within 1.25x of a stream's even share: the
    // longest-first order then balances the streams about as well, without the partial
    // results and the merge.
    const int share = (total + n_pipes - 1) / n_pipes;
    if (4 * b <= 5 * share) T = max(T, b);
    s_T = T;
    warp_sums[0] = b;
  }
  __syncthreads();
  const int longest = warp_sums[0];
  int T = s_T;
  __syncthreads();
  // the smallest T (doubling) whose parts fit the slots
  for (;;) {
    int need = 0;
    for (int k = k0; k < k1; ++k) {
      const int t = item_tiles(p, tiles, k);
      if (t > T) need += (t + T - 1) / T;
    }
    int need_tot = 0;
    block_scan_excl(need, warp_sums, need_tot);
    if (need_tot <= slot_cap || T >= longest) break;
    T *= 2;
  }
  // positions: split parts first (slot = list position), then the unsplit items
  int n_parts = 0, n_whole = 0, n_si = 0;
  for (int k = k0; k < k1; ++k) {
    const int t = item_tiles(p, tiles, k);
    if (t > T) {
      n_parts += (t + T - 1) / T;
      ++n_si;
    } else {
      ++n_whole;
    }
  }
  int tot_parts = 0, tot_whole = 0, tot_si = 0;
  int pos_p = block_scan_excl(n_parts, warp_sums, tot_parts);
  int pos_w = block_scan_excl(n_whole, warp_sums, tot_whole);
  int pos_s = block_scan_excl(n_si, warp_sums, tot_si);
  pos_w += tot_parts;
  for (int k = k0; k < k1; ++k) {
    const int t = item_tiles(p, tiles, k);
    if (t > T) {
      const int parts = (t + T - 1) / T;
      split_items[pos_s++] = make_int4(k, parts, pos_p, 0);
      for (int q = 0; q < parts; ++q) list[pos_p++] = make_int2(k, q);
    } else {
      list[pos_w++] = make_int2(k, 0);
    }
  }
  if (threadIdx.x == 0) {
    hdr->list_len = tot_parts + tot_whole;
    hdr->n_split = tot_parts;
    hdr->part_tiles = T;
    hdr->n_split_items = tot_si;
  }
}

template <int D>
__global__ void __launch_bounds__(kTile) fwd_merge_kernel(const __grid_constant__ Params p, const int4* split_items,
                                                           const SplitHdr* hdr) {
  const float kNegInf = __int_as_float(0xff800000);
  const int n_si = hdr->n_split_items;
  const int r = threadIdx.x;
  for (int j = blockIdx.x; j < n_si; j += gridDim.x) {
    const int4 si = split_items[j];
    const Item it = decode_item(p, si.x);
    const int qtok = it.tile * kTile + r;
    if (qtok >= p.n_tokens) continue;
    const float* base = p.partial + (size_t)si.z * (kTile * (D + 1));
    float mx = kNegInf;
    for (int q = 0; q < si.y; ++q) mx = fmaxf(mx, base[(size_t)q * (kTile * (D + 1)) + kTile * D + r]);
    __nv_bfloat16* orow = p.o + (int64_t)it.s * p.o_sb + (int64_t)qtok * p.o_sn + (int64_t)it.h * p.o_sh;
    float lse = kNegInf;
    float acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    if (mx != kNegInf) {
      float wsum = 0.f;
      for (int q = 0; q < si.y; ++q) {
        const float* part = base + (size_t)q * (kTile * (D + 1));
        const float lq = part[kTile * D + r];
        if (lq == kNegInf) continue;
        const float w = __expf(lq - mx);
        wsum += w;
        const float4* row = reinterpret_cast<const float4*>(part + (size_t)r * D);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) {
          const float4 v = row[c];
          acc[4 * c] += w * v.x;
          acc[4 * c + 1] += w * v.y;
          acc[4 * c + 2] += w * v.z;
          acc[4 * c + 3] += w * v.w;
        }
      }
      const float inv = 1.f / wsum;
#pragma unroll
      for (int c = 0; c < D; ++c) acc[c] *= inv;
      lse = mx + __logf(wsum);
    }
    uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
    for (int c = 0; c < D / 8; ++c)
      dst[c] = make_uint4(pack_bf16x2(acc[8 * c], acc[8 * c + 1]), pack_bf16x2(acc[8 * c + 2], acc[8 * c + 3]),
                          pack_bf16x2(acc[8 * c + 4], acc[8 * c + 5]), pack_bf16x2(acc[8 * c + 6], acc[8 * c + 7]));
    p.lse[((int64_t)it.s * p.heads + it.h) * p.n_tokens + qtok] = lse;
  }
}

// Workspace of the forward: the work counter, then (split mode) the split header, the plan's
// key-tile counts, the work list, the split items and the partial-result slots, each section
// 256-byte aligned. slot_cap is the number of slots that fit in `bytes`.
struct FwdWorkspace {
  size_t counter_off, hdr_off, tiles_off, list_off, items_off, partial_off, min_bytes, slot_cap;
};

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

FwdWorkspace fwd_workspace_layout(int64_t n_items, int64_t n_groups, int d, size_t bytes) {
  FwdWorkspace w;
  w.counter_off = 0;
  w.hdr_off = 64;
  w.min_bytes = 256;
  w.tiles_off = 256;
  w.list_off = w.tiles_off + up256((size_t)n_groups * 4);
  const size_t slot_bytes = (size_t)kTile * (d + 1) * 4;
  const size_t fixed = w.list_off + up256((size_t)n_items * 8) + 3 * 256;
  // per slot: one list entry (8 B), at most one split item (16 B), the partial (slot_bytes)
  w.slot_cap = bytes > fixed ? (bytes - fixed) / (8 + 16 + slot_bytes) : 0;
  w.items_off = w.list_off + up256((size_t)(n_items + (int64_t)w.slot_cap) * 8);
  w.partial_off = w.items_off + up256(w.slot_cap * 16);
  return w;
}

// The forward kernel of head dimension D.
template <int D>
constexpr auto fwd_kernel() {
  if constexpr (Cfg<D>::WIDE) return attn_fwd_wide_kernel<D>;
  else return attn_fwd_kernel<D>;
}

template <int D>
int launch_d(const AttnArgs& a, cudaStream_t stream) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv, to;
  const uint32_t kv_rows = a.block == 32 ? 32u : 64u;
  if (!encode_bhnd_map(&tq, a.q, a.batch, a.n_tokens, a.heads, D, a.q_strides[0], a.q_strides[1], a.q_strides[2],
                       C::CH, kTile, C::TMA_SWZ) ||
      !encode_bhnd_map(&tk, a.k, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::CH, kv_rows, C::TMA_SWZ) ||
      !encode_bhnd_map(&tv, a.v, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::CH, kv_rows, C::TMA_SWZ))
    return SA_ERR_UNSUPPORTED;
  Params p;
  p.batch = a.batch;
  p.n_tokens = a.n_tokens;
  p.heads = a.heads;
  p.heads_per_kv = a.heads / a.kv_heads;
  p.block = a.block;
  p.log2b = __builtin_ctz((unsigned)a.block);
  p.nb = a.n_tokens / a.block;
  p.causal = a.causal;
  p.csr_shared = a.csr_shared;
  p.tiles_per_seq = (a.n_tokens + kTile - 1) / kTile;
  p.n_items = a.batch * a.heads * p.tiles_per_seq;
  p.n_masks = a.n_masks;
  for (int m = 0; m < kMaxMasks; ++m) {
    p.row_ptr[m] = a.row_ptr[m];
    p.col_idx[m] = a.col_idx[m];
  }
  for (int h = 0; h < kMaxHeadMap; ++h) p.head_mask[h] = a.head_mask[h];
  p.o = static_cast<__nv_bfloat16*>(a.o);
  // d = 64: O leaves through TMA stores of 32-row boxes when its layout allows a tensor map
  // (16-byte aligned base and strides); otherwise, and at other d, through plain stores
  memset(&to, 0, sizeof(to));
  p.o_tma = D == 64 && encode_bhnd_map(&to, a.o, a.batch, a.n_tokens, a.heads, D, a.o_strides[0], a.o_strides[1],
                                       a.o_strides[2], C::CH, 32, C::TMA_SWZ)
                ? 1
                : 0;
  p.lse = a.lse;
  p.o_sb = a.o_strides[0];
  p.o_sn = a.o_strides[1];
  p.o_sh = a.o_strides[2];
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  p.csr_batches = a.csr_shared ? 1 : a.batch;
  const int n_groups = a.n_masks * p.csr_batches * p.tiles_per_seq;
  const FwdWorkspace ws = fwd_workspace_layout(p.n_items, n_groups, D, a.workspace_bytes);
  if (a.workspace == nullptr || a.workspace_bytes < ws.min_bytes) return SA_ERR_CAPACITY;
  uint8_t* wsb = static_cast<uint8_t*>(a.workspace);
  p.work_counter = reinterpret_cast<unsigned int*>(wsb + ws.counter_off);
  p.work_list = nullptr;
  p.list_hdr = nullptr;
  p.partial = nullptr;
  if (cudaMemsetAsync(p.work_counter, 0, sizeof(unsigned int), stream) != cudaSuccess) return SA_ERR_CUDA;
  const int sm_count = current_sm_count();
  // d <= 64: two pipelines per CTA; d = 128: one item stream per CTA
  auto kern = fwd_kernel<D>();
  // The register split in the kernel hands out exactly the launch allocation: refuse to
  // launch a build whose per-thread register count differs from it.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return SA_ERR_CUDA;
  if (fa.numRegs != kLaunchRegs) return SA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return SA_ERR_CUDA;
  // Split mode when the items are few for the GPU's item streams and the workspace holds
  // partial-result slots: long key lists are then cut into parts (K9), about two per stream.
  // d <= 64 (two streams per SM, each at about half an SM's speed): fewer than two items per
  // stream. d = 128 (one stream per SM at a whole SM's speed, which balances a few long items
  // well in longest-first order): fewer items than SMs. The schedule kernel still keeps the
  // items whole when the longest is within 1.25x of a stream's share.
  const int per_cta = C::WIDE ? 1 : 2;
  const int n_pipes = per_cta * sm_count;
  const bool split = ws.slot_cap >= 2 && p.n_items < (C::WIDE ? 1 : 2) * n_pipes;
  int grid = (p.n_items + per_cta - 1) / per_cta < sm_count ? (p.n_items + per_cta - 1) / per_cta : sm_count;
  if (split) {
    int* tiles = reinterpret_cast<int*>(wsb + ws.tiles_off);
    int2* list = reinterpret_cast<int2*>(wsb + ws.list_off);
    int4* split_items = reinterpret_cast<int4*>(wsb + ws.items_off);
    SplitHdr* hdr = reinterpret_cast<SplitHdr*>(wsb + ws.hdr_off);
    p.partial = reinterpret_cast<float*>(wsb + ws.partial_off);
    fwd_plan_kernel<<<(n_groups + kPlanWarps - 1) / kPlanWarps, 32 * kPlanWarps, 0, stream>>>(p, n_groups, tiles);
    fwd_schedule_kernel<<<1, 1024, 0, stream>>>(p, tiles, (int)ws.slot_cap, n_pipes, list, split_items, hdr);
    if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
    p.work_list = list;
    p.list_hdr = &hdr->list_len;
    grid = sm_count;   // the list is at most n_items + slot_cap entries long
    kern<<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, to, p);
    if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
    const int mgrid = (int)(ws.slot_cap < (size_t)(2 * sm_count) ? ws.slot_cap : (size_t)(2 * sm_count));
    fwd_merge_kernel<D><<<mgrid, kTile, 0, stream>>>(p, split_items, hdr);
    return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
  }
  kern<<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace

size_t attn_fwd_workspace_bytes(int64_t batch, int64_t n_tokens, int64_t heads, int head_dim, int64_t csr_batches,
                                int64_t n_masks) {
  const int64_t tiles_per_seq = (n_tokens + kTile - 1) / kTile;
  const int64_t n_items = batch * heads * tiles_per_seq;
  const FwdWorkspace w = fwd_workspace_layout(n_items, n_masks * csr_batches * tiles_per_seq, head_dim, 0);
  const size_t slot_bytes = (size_t)kTile * (head_dim + 1) * 4;
  // room for the default number of split parts (about four per SM of a GB300)
  return w.list_off + up256((size_t)(n_items + kFwdDefaultSlots) * 8) + up256((size_t)kFwdDefaultSlots * 16) +
         (size_t)kFwdDefaultSlots * slot_bytes + 3 * 256;
}

int launch_attn_fwd(const AttnArgs& a, cudaStream_t stream) {
  switch (a.head_dim) {
    case 32: return launch_d<32>(a, stream);
    case 64: return launch_d<64>(a, stream);
    case 128: return launch_d<128>(a, stream);
  }
  return SA_ERR_UNSUPPORTED;
}

unsigned int attn_read_and_clear_error(cudaStream_t stream) {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_attn_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
  cudaMemcpyToSymbolAsync(g_attn_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  return v;
}

}  // namespace sa
