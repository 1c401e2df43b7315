// Block-sparse flash-attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// Work item: 256 consecutive query tokens of one (sequence, head) = two 128-row query
// tiles A and B, covering 256 / b query blocks. The key blocks the item visits are the
// sorted union of those blocks' CSR rows; each key block carries one membership bit per
// query block. Key blocks are packed into key tiles of up to 128 keys; a key tile is
// "active" for tile A (B) if any of A's (B's) query blocks has it in its row, and the
// tensor core and the softmax of a query tile only touch its active key tiles.
//
// The kernel is persistent: one CTA per SM walks a static list of work items ordered
// longest first (causal: last query tiles first; BigBird: the global rows first).
//
// Warp roles (352 threads, one CTA per SM):
//   warp 0      producer: merges the CSR rows (all lanes, warp-uniform), publishes key-tile
//               descriptions in a small ring, issues TMA loads of Q and of the K / V blocks.
//   warps 1, 10 lane 0 of warp 1 (tile A) and of warp 10 (tile B) issue tcgen05 MMAs:
//                 S_X = Q_X K^T          (A, B from shared memory)
//                 O_X += P_X V           (A = P_X from TMEM, B = V, MN-major, from shared memory)
//               QK_X(t+1) as soon as the softmax of X has released tile t, then PV_X(t);
//               the two query tiles never wait on each other. Warp 1 owns TMEM (512 cols).
//   warps 2-5   softmax of tile A, warps 6-9 softmax of tile B (warp w reads TMEM lane
//               quarter w % 4), running concurrently: one query row per thread. One pass over
//               S per tile, software-pipelined by 32-column chunks (the next chunk's TMEM load
//               and max overlap this chunk's exponentials); lazily rescaled running max (P
//               chunks and O are rescaled only when the max grows by more than 2^8); final
//               normalisation and the O (bf16) / LSE (fp32) stores.
// TMEM columns (Cfg::col_*): S_A [0,128), S_B [128,256); d <= 64: O_A [256,256+d),
// O_B [320,320+d), P_A [384,448), P_B [448,512); d = 128: O_A [256,384), O_B [384,512)
// and P aliases the first 64 columns of S.
//
// Token rule: key j of block J is visible to query i of block I iff J is in row(I) and
// (not causal or j <= i) ("Parameter-free Adaptive Sparse Attention via Compression-Based
// Content Selection", section 3.4 block-to-token expansion). No token mask is
// materialised: the per-row column mask comes from the membership bits and, on the
// diagonal block, from the causal compare.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx_sm100.cuh"
#include "sa_internal.h"
#include "tma_host.h"

namespace sa {
namespace {

__device__ unsigned int g_attn_err;

constexpr int kTile = 128;        // query rows per query tile, max keys per key tile
constexpr int kItemRows = 256;    // query rows per work item (tiles A and B)
constexpr int kThreads = 352;  // 11 warps: producer, MMA A, 2 x 4 softmax, MMA B
constexpr int kMetaRing = 4;
constexpr int kMaxSlots = 4;      // key blocks per key tile (128 / b, b >= 32)
constexpr int kMaxRows = 8;       // query blocks per work item (256 / b)
constexpr uint32_t kTmemCols = 512;
constexpr int kMetaConsumers = 10; // 8 softmax warps + the two MMA threads

template <int D>
struct Cfg {
  static constexpr int CH = D >= 64 ? 64 : 32;         // elements per swizzled row
  static constexpr int NCH = D / CH;                   // d-chunks
  static constexpr int ROWB = CH * 2;                  // bytes per swizzled row
  static constexpr uint32_t SWZ = ROWB == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr CUtensorMapSwizzle TMA_SWZ =
      ROWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static constexpr uint32_t ATOM = 8 * ROWB;           // swizzle atom (8 rows)
  static constexpr int CHUNK = kTile * ROWB;           // one d-chunk of a 128-row tile
  static constexpr int TILE_BYTES = NCH * CHUNK;       // 128 rows x D bf16
  static constexpr int STAGES = D == 128 ? 2 : (D == 64 ? 3 : 4);   // K and V ring depth
  static constexpr int UNION_BYTES = (kMaxRows * kMaxMaskBlocks / 32 + kMaxMaskBlocks) * 4;   // 20 KB
  static constexpr int SMEM_NEED = 1024 + TILE_BYTES * (2 + 2 * STAGES) + UNION_BYTES;
  // at least 120 KB so that only one CTA (512 TMEM columns) is resident per SM
  static constexpr int SMEM = SMEM_NEED > 120 * 1024 ? SMEM_NEED : 120 * 1024;
  static constexpr bool P_ALIAS = D > 64;              // no room for separate P columns
  __host__ __device__ static constexpr uint32_t col_s(int x) { return x ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(int x) { return x ? (D > 64 ? 384u : 320u) : 256u; }
  __host__ __device__ static constexpr uint32_t col_p(int x) {
    return P_ALIAS ? col_s(x) : (x ? 448u : 384u);
  }
};

enum : int { kKeyTile = 0, kEndItem = 1 };

struct Meta {
  int kind;
  int nslots;
  int active;                 // bit 0: tile A, bit 1: tile B
  int jblk[kMaxSlots];
  int mask[kMaxSlots];        // bit r: query block r of the item has this key block
};

// Field-wise read of a published ring entry (the producer's mbarrier arrive orders it).
__device__ __forceinline__ Meta load_meta(const Meta* src) {
  const volatile Meta* vm = src;
  Meta m;
  m.kind = vm->kind;
  m.nslots = vm->nslots;
  m.active = vm->active;
#pragma unroll
  for (int i = 0; i < kMaxSlots; ++i) {
    m.jblk[i] = vm->jblk[i];
    m.mask[i] = vm->mask[i];
  }
  return m;
}

struct Params {
  int batch, n_tokens, heads, heads_per_kv, block, log2b, nb, causal, csr_shared;
  int pairs_per_seq;          // work items per (sequence, head)
  int n_items;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  __nv_bfloat16* o;
  float* lse;
  int64_t o_sb, o_sn, o_sh;
  float scale_log2;
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t m_full[kMetaRing], m_empty[kMetaRing];
  uint64_t s_full[2], p_full[2], pv_done[2], o_empty[2];
  uint64_t drain[2];
};

struct Item {
  int s, h, pair;
};

// Work item k of the static longest-first order: all (sequence, head) pairs of one
// query-pair rank before the next rank; causal ranks run from the last query pair.
__device__ __forceinline__ Item decode_item(const Params& p, int k) {
  const int bh = k % (p.batch * p.heads);
  const int rank = k / (p.batch * p.heads);
  Item it;
  it.h = bh % p.heads;
  it.s = bh / p.heads;
  it.pair = p.causal ? (p.pairs_per_seq - 1 - rank) : rank;
  return it;
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait(bar, parity, abort_flag, &g_attn_err, kErrTimeout);
}

__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  int never = 0;
  mbar_wait(bar, parity, &never, &g_attn_err, kErrTimeout);
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
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ------------------------------------------------------------------ producer (warp 0)

// Per-item key-block union, built by the producer warp in shared memory: one bitmap of
// nb bits per query block of the item, then an ascending list of (J | membership << 16).
struct UnionSmem {
  uint32_t bm[kMaxRows][kMaxMaskBlocks / 32];   // 4 KB
  uint32_t list[kMaxMaskBlocks];                // 16 KB
};

// Builds the union of rows I0 .. I0+nq-1 into u.list; returns its length. Column indices
// outside [0, nb) are skipped and reported; under causality a block J > I0 + r is not
// attached to query block r (its keys are all in the future).
__device__ int build_union(const Params& p, UnionSmem& u, const int32_t* rp, int I0, int nq) {
  const int lane = threadIdx.x & 31;
  const int nw = (p.nb + 31) >> 5;
  for (int r = 0; r < nq; ++r)
    for (int w = lane; w < nw; w += 32) u.bm[r][w] = 0u;
  const int bnd = (lane <= nq) ? rp[I0 + lane] : 0x7fffffff;   // lane r: start of row r
  int bq[kMaxRows + 1];
#pragma unroll
  for (int q = 0; q <= kMaxRows; ++q) bq[q] = __shfl_sync(0xffffffffu, bnd, min(q, nq));
  const int e0 = bq[0];
  const int e1 = bq[kMaxRows];
  __syncwarp();
  for (int e = e0 + lane; e < e1; e += 32) {
    const int J = p.col_idx[e];
    int r = 0;
#pragma unroll
    for (int q = 1; q < kMaxRows; ++q) r += (q < nq && e >= bq[q]) ? 1 : 0;
    if (J < 0 || J >= p.nb) {
      atomicOr(&g_attn_err, kErrBadIndex);
    } else if (!p.causal || J <= I0 + r) {
      atomicOr(&u.bm[r][J >> 5], 1u << (J & 31));
    }
  }
  __syncwarp();
  int total = 0;
  for (int w0 = 0; w0 < nw; w0 += 32) {
    const int w = w0 + lane;
    uint32_t word[kMaxRows];
    uint32_t un = 0u;
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      word[r] = (r < nq && w < nw) ? u.bm[r][w] : 0u;
      un |= word[r];
    }
    const int c = __popc(un);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int pos = total + incl - c;
    while (un) {
      const int j = __ffs(un) - 1;
      un &= un - 1u;
      uint32_t mask = 0u;
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) mask |= ((word[r] >> j) & 1u) << r;
      u.list[pos++] = (uint32_t)(w * 32 + j) | (mask << 16);
    }
    total += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
  return total;
}

template <int D>
__device__ void producer(const Params& p, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                         Bars& bars, Meta* meta, UnionSmem& u, uint8_t* sQ, uint8_t* sK, uint8_t* sV,
                         volatile int* abort_flag) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const int b = p.block;
  const int rows_per_item = kItemRows >> p.log2b;
  const int slots_per_tile = kTile >> p.log2b;
  const int maskA = (1 << (kTile >> p.log2b)) - 1;   // query blocks of tile A
  int mt = 0, kt = 0, item_local = 0;
  int k_issued = 0, v_issued = 0;                    // key tiles whose K / V loads were issued
  int q_last = -1;                                   // item_local of the last Q load
  bool ok = true;

  for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++item_local) {
    const Item it = decode_item(p, k);
    const int I0 = it.pair * rows_per_item;
    const int q0 = it.pair * kItemRows;
    const int hk = it.h / p.heads_per_kv;
    const int nq = min(rows_per_item, p.nb - I0);
    const int32_t* rp = p.row_ptr + (size_t)(p.csr_shared ? 0 : it.s) * (p.nb + 1);

    // Q of both tiles (rows beyond the sequence are zero-filled by TMA)
    if (lane == 0) {
      if (item_local > 0) ok = wait_bar(&bars.q_empty, (item_local - 1) & 1, abort_flag);
      if (ok) {
        mbar_arrive_expect_tx(&bars.q_full, 2 * C::TILE_BYTES);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_4d(sQ + x * C::TILE_BYTES + c * C::CHUNK, tq, &bars.q_full, c * C::CH, it.h, q0 + x * kTile,
                        it.s);
        q_last = item_local;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) break;

    const int n_keys = build_union(p, u, rp, I0, nq);

    for (int base = 0;; base += slots_per_tile) {
      Meta m;
      m.kind = base < n_keys ? kKeyTile : kEndItem;
      m.nslots = min(slots_per_tile, n_keys - base);
      m.active = 0;
#pragma unroll
      for (int i = 0; i < kMaxSlots; ++i) {
        const uint32_t e = (i < m.nslots) ? u.list[base + i] : 0u;
        m.jblk[i] = (int)(e & 0xffffu);
        m.mask[i] = (int)(e >> 16);
        m.active |= ((m.mask[i] & maskA) ? 1 : 0) | ((m.mask[i] & ~maskA) ? 2 : 0);
      }
      if (lane == 0) {
        const int ms = mt % kMetaRing;
        ok = wait_bar(&bars.m_empty[ms], ((mt / kMetaRing) & 1) ^ 1, abort_flag);
        if (ok) {
          meta[ms] = m;
          mbar_arrive(&bars.m_full[ms]);
        }
        if (ok && m.kind == kKeyTile) {
          const int st = kt % C::STAGES;
          const uint32_t ph = (kt / C::STAGES) & 1;
          const uint32_t bytes = (uint32_t)(m.nslots * b * D * 2);
          ok = wait_bar(&bars.k_empty[st], ph ^ 1, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(&bars.k_full[st], bytes);
#pragma unroll
            for (int i = 0; i < kMaxSlots; ++i)
              if (i < m.nslots) {
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                  tma_load_4d(sK + st * C::TILE_BYTES + c * C::CHUNK + i * b * C::ROWB, tk, &bars.k_full[st],
                              c * C::CH, hk, m.jblk[i] * b, it.s);
              }
            k_issued = kt + 1;
            ok = wait_bar(&bars.v_empty[st], ph ^ 1, abort_flag);
          }
          if (ok) {
            mbar_arrive_expect_tx(&bars.v_full[st], bytes);
#pragma unroll
            for (int i = 0; i < kMaxSlots; ++i)
              if (i < m.nslots) {
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                  tma_load_4d(sV + st * C::TILE_BYTES + c * C::CHUNK + i * b * C::ROWB, tv, &bars.v_full[st],
                              c * C::CH, hk, m.jblk[i] * b, it.s);
              }
            v_issued = kt + 1;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      ++mt;
      if (m.kind == kKeyTile) ++kt;
      if (!ok || m.kind == kEndItem) break;
    }
    __syncwarp();   // the next item's union may overwrite the list
  }
  // Drain this CTA's own copies in flight before the CTA may exit.
  if (lane == 0) {
    if (q_last >= 0) drain_bar(&bars.q_full, q_last & 1);
    // the last tile that used each stage: waiting on it covers every earlier use
    for (int t = max(0, k_issued - C::STAGES); t < k_issued; ++t)
      drain_bar(&bars.k_full[t % C::STAGES], (t / C::STAGES) & 1);
    for (int t = max(0, v_issued - C::STAGES); t < v_issued; ++t)
      drain_bar(&bars.v_full[t % C::STAGES], (t / C::STAGES) & 1);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA issuer (warp 1, lane 0)

template <int D>
struct MmaState {
  uint32_t tmem;
  uint64_t qdesc[2];      // descriptors of Q_A, Q_B at k-step 0
  uint64_t kdesc0, vdesc0;  // descriptors of K / V stage 0 at k-step 0
  int kt;                 // K/V ring position of the current key tile
  int cnt[2];             // QK count per query tile (global)
  int pv[2];              // PV count per query tile (global)
};

// Byte offset (>> 4, the descriptor's address unit) of k-step ks inside a K-major tile.
template <int D>
__device__ __forceinline__ constexpr uint32_t kmajor_step(int ks) {
  using C = Cfg<D>;
  return (uint32_t)(((ks * 16) / C::CH) * C::CHUNK + ((ks * 16) % C::CH) * 2) >> 4;
}

template <int D>
__device__ __forceinline__ void issue_qk(MmaState<D>& st, int x, int stage, int nkeys) {
  using C = Cfg<D>;
  const uint32_t idesc = make_idesc_bf16(128, (uint32_t)nkeys, 0, 0);
  const uint64_t a0 = st.qdesc[x];
  const uint64_t b0 = st.kdesc0 + (uint64_t)((stage * C::TILE_BYTES) >> 4);
  const uint32_t d = st.tmem + C::col_s(x);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
    mma_bf16_ss(d, a0 + kmajor_step<D>(ks), b0 + kmajor_step<D>(ks), idesc, ks > 0 ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void issue_pv(MmaState<D>& st, int x, int stage, int nkeys, bool accumulate) {
  using C = Cfg<D>;
  const uint32_t idesc = make_idesc_bf16(128, D, 0, 1);
  const uint64_t b0 = st.vdesc0 + (uint64_t)((stage * C::TILE_BYTES) >> 4);
  const uint32_t d = st.tmem + C::col_o(x), a = st.tmem + C::col_p(x);
  const int nks = nkeys >> 4;
#pragma unroll 8
  for (int ks = 0; ks < nks; ++ks)
    mma_bf16_ts(d, a + (uint32_t)(ks * 8), b0 + (uint64_t)((ks * 16 * C::ROWB) >> 4), idesc,
                (accumulate || ks > 0) ? 1u : 0u);
}

// One MMA-issuing thread per query tile x (warp 1 lane 0: tile A, warp 10 lane 0: tile B).
// For each key tile active for x: QK_x(t) as soon as the softmax of x has released the
// previous tile (S_x read, P_x written), then PV_x of that previous tile. With P aliased
// into S (d = 128) the previous PV goes first and must complete before QK_x(t).
template <int D>
__device__ void mma_issuer(const Params& p, Bars& bars, Meta* meta, uint8_t* sQ, uint8_t* sK, uint8_t* sV,
                           uint32_t tmem, int x, volatile int* abort_flag) {
  using C = Cfg<D>;
  MmaState<D> st;
  st.tmem = tmem;
  st.qdesc[0] = make_smem_desc(smem_u32(sQ), 16, C::ATOM, C::SWZ);
  st.qdesc[1] = make_smem_desc(smem_u32(sQ) + C::TILE_BYTES, 16, C::ATOM, C::SWZ);
  st.kdesc0 = make_smem_desc(smem_u32(sK), 16, C::ATOM, C::SWZ);
  st.vdesc0 = make_smem_desc(smem_u32(sV), C::CHUNK, C::ATOM, C::SWZ);
  int mt = 0, kt = 0;
  int pvn = 0;              // PVs issued for x (global) == tiles of x released by the softmax
  bool ok = true;
  int item_local = 0;
  for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++item_local) {
    if (!(ok = wait_bar(&bars.q_full, item_local & 1, abort_flag))) break;
    bool first_pv = true;
    int pend_stage = -1, pend_keys = 0;
    uint32_t pend_ph = 0;
    auto issue_pending_pv = [&]() -> bool {
      if (!wait_bar(&bars.v_full[pend_stage], pend_ph, abort_flag)) return false;
      if (first_pv && item_local > 0 && !wait_bar(&bars.o_empty[x], (item_local - 1) & 1, abort_flag)) return false;
      tc_fence_after();
      issue_pv<D>(st, x, pend_stage, pend_keys, !first_pv);
      mma_commit(&bars.pv_done[x]);
      mma_commit(&bars.v_empty[pend_stage]);
      first_pv = false;
      ++pvn;
      pend_stage = -1;
      return true;
    };
    for (;;) {
      const int ms = mt % kMetaRing;
      if (!(ok = wait_bar(&bars.m_full[ms], (mt / kMetaRing) & 1, abort_flag))) break;
      const Meta m = load_meta(&meta[ms]);
      mbar_arrive(&bars.m_empty[ms]);
      ++mt;
      if (m.kind != kKeyTile) break;
      const int stage = kt % C::STAGES;
      const uint32_t ph = (kt / C::STAGES) & 1;
      ++kt;
      const bool act = (m.active & (1 << x)) != 0;
      if (pend_stage >= 0 && (!act || C::P_ALIAS)) {
        // resolve the pending PV first: every later release of a K/V stage by this
        // thread must be ordered after it (and with P aliased into S, so must the QK)
        if (!(ok = wait_bar(&bars.p_full[x], (pvn & 1), abort_flag))) break;
        if (!(ok = issue_pending_pv())) break;
      }
      if (!act) {
        // This query tile does not read the stage. Release it only once it has been
        // filled for this tile: mbarrier arrivals carry no phase, so a consumer must not
        // run ahead of the producer by a whole ring lap. tcgen05.commit orders the
        // release behind this thread's earlier MMAs.
        if (!(ok = wait_bar(&bars.k_full[stage], ph, abort_flag))) break;
        mma_commit(&bars.k_empty[stage]);
        if (!(ok = wait_bar(&bars.v_full[stage], ph, abort_flag))) break;
        mma_commit(&bars.v_empty[stage]);
        continue;
      }
      if (!(ok = wait_bar(&bars.k_full[stage], ph, abort_flag))) break;
      if (pend_stage >= 0) {
        // the softmax of x has read S_x and written P_x of the pending tile
        if (!(ok = wait_bar(&bars.p_full[x], (pvn & 1), abort_flag))) break;
      }
      if (C::P_ALIAS && pvn > 0) {
        // P_x lives in S_x's columns: the last PV reading it must be complete
        if (!(ok = wait_bar(&bars.pv_done[x], (pvn - 1) & 1, abort_flag))) break;
      }
      tc_fence_after();
      issue_qk<D>(st, x, stage, m.nslots * p.block);
      mma_commit(&bars.s_full[x]);
      mma_commit(&bars.k_empty[stage]);
      if (pend_stage >= 0 && !(ok = issue_pending_pv())) break;
      pend_stage = stage;
      pend_keys = m.nslots * p.block;
      pend_ph = ph;
    }
    if (!ok) break;
    if (pend_stage >= 0) {
      if (!(ok = wait_bar(&bars.p_full[x], (pvn & 1), abort_flag))) break;
      if (!(ok = issue_pending_pv())) break;
    }
    mma_commit(&bars.q_empty);   // this thread's QKs of the item have been issued; arrives when done
  }
  // Make sure no MMA of this thread is still writing TMEM when the CTA frees it.
  mma_commit(&bars.drain[x]);
  drain_bar(&bars.drain[x], 0);
}

// ------------------------------------------------------------------ softmax + epilogue (warps 2-9)

// Rare path of the online max: multiply the P chunks [0, ch) already written for this
// tile by alpha (bf16 round trip through TMEM). Kept out of line to spare registers.
__device__ __noinline__ void rescale_p_chunks(uint32_t tP, int ch, bool u0, bool u1, bool u2, float alpha) {
  tmem_st_wait();
  const bool use_pc[3] = {u0, u1, u2};
#pragma unroll
  for (int pc = 0; pc < 3; ++pc) {
    if (pc >= ch || !use_pc[pc]) continue;
    uint32_t w[16];
    tmem_ld_x16(tP + pc * 16, w);
    tmem_ld_wait<16>(w);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      w[j] = pack_bf16x2(__uint_as_float(w[j] << 16) * alpha, __uint_as_float(w[j] & 0xffff0000u) * alpha);
    tmem_st_x16(tP + pc * 16, w);
  }
}

// One key tile of query tile x for this thread's row, in a single pass over S: per
// 32-column chunk, the chunk max updates the running max lazily (only when it grows by
// more than 2^8; then the row sum, the P chunks already written for this tile and,
// at the end, O are rescaled), p = 2^(s c - m) goes to P_x as bf16. Returns false on abort.
template <int D>
__device__ __forceinline__ bool softmax_tile(const Params& p, Bars& bars, const Meta& m, int x, uint32_t tmem,
                                             uint32_t lane_base, int sub, int qblk, int rloc, float& m_use, float& l,
                                             int& cnt, int& n_item, volatile int* abort_flag) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const int b = p.block;
  const float c = p.scale_log2;
  const float kNegInf = __int_as_float(0xff800000);
  const uint32_t tS = tmem + C::col_s(x) + lane_base;
  const uint32_t tO = tmem + C::col_o(x) + lane_base;
  const uint32_t tP = tmem + C::col_p(x) + lane_base;

  if (!wait_bar(&bars.s_full[x], cnt & 1, abort_flag)) return false;
  tc_fence_after();
  const int nch = (m.nslots * b) >> 5;             // 32-column chunks holding keys

  uint32_t keep[4];
  bool use[4];
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t kp = 0u;
    if (ch < nch) {
      const int slot = (ch * 32) >> p.log2b;
      // constant-index selects keep the meta fields in registers
      const int J = slot == 0 ? m.jblk[0] : slot == 1 ? m.jblk[1] : slot == 2 ? m.jblk[2] : m.jblk[3];
      const int msk = slot == 0 ? m.mask[0] : slot == 1 ? m.mask[1] : slot == 2 ? m.mask[2] : m.mask[3];
      if ((msk >> sub) & 1) {
        if (!p.causal || J < qblk) {
          kp = 0xffffffffu;
        } else if (J == qblk) {
          const int lim = rloc - ((ch * 32) & (b - 1));   // visible columns j <= lim
          kp = lim >= 31 ? 0xffffffffu : (lim < 0 ? 0u : ((2u << lim) - 1u));
        }
      }
    }
    keep[ch] = kp;
    use[ch] = __any_sync(0xffffffffu, kp != 0u);   // warp-uniform: this chunk has visible keys
  }

  const float m_start = m_use;
  const uint64_t c2 = f2_pack(c, c);
  uint64_t rsa[4] = {0ull, 0ull, 0ull, 0ull};     // tile row sum, 4 packed accumulators

  // Software pipeline over 32-column chunks: chunk ch+1 is loaded from TMEM before the
  // exponentials of chunk ch and its max is taken while they stream through the MUFU.
  auto chunk_max = [&](const uint32_t* v, uint32_t kp) -> float {
    float acc[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
    if (kp == 0xffffffffu) {
#pragma unroll
      for (int j = 0; j < 32; j += 2)
        acc[(j >> 1) & 3] = max3(acc[(j >> 1) & 3], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j & 3] = fmaxf(acc[j & 3], ((kp >> j) & 1u) ? __uint_as_float(v[j]) : kNegInf);
    }
    return fmaxf(max3(acc[0], acc[1], acc[2]), acc[3]) * c;   // -inf stays -inf
  };
  uint32_t va[32], vb[32];
  float cm_cur = kNegInf;
  if (use[0]) {
    tmem_ld_x32(tS, va);
    tmem_ld_wait<32>(va);
    cm_cur = chunk_max(va, keep[0]);
  }
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    if (ch >= nch) break;
    uint32_t* vc = (ch & 1) ? vb : va;
    uint32_t* vn = (ch & 1) ? va : vb;
    const bool next = ch + 1 < nch && use[ch + 1];
    if (next) tmem_ld_x32(tS + (ch + 1) * 32, vn);
    uint32_t pk[16];
    if (use[ch]) {
      const uint32_t kp = keep[ch];
      const float cm = cm_cur;
      const bool need = cm > m_use + 8.0f;
      if (__any_sync(0xffffffffu, need)) {
        // rare: the running max grows; rescale the sums and this tile's P chunks so far
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m_use - cm);          // 0 when m_use = -inf
          m_use = cm;
        }
        l *= alpha;
        const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          uint64_t r;
          asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(rsa[a]), "l"(al2));
          rsa[a] = r;
        }
        if (ch > 0) rescale_p_chunks(tP, ch, use[0], use[1], use[2], alpha);
      }
      const uint64_t negm2 = f2_pack(-m_use, -m_use);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(vc[j]), __uint_as_float(vc[j + 1])), c2, negm2), x0, x1);
        if (kp != 0xffffffffu) {                   // hidden columns contribute exactly 0
          x0 = ((kp >> j) & 1u) ? x0 : kNegInf;
          x1 = ((kp >> (j + 1)) & 1u) ? x1 : kNegInf;
        }
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        rsa[(j >> 1) & 3] = f2_add(rsa[(j >> 1) & 3], f2_pack(p0, p1));
        pk[j >> 1] = pack_bf16x2(p0, p1);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[j] = 0u;
    }
    if (next) {
      float d0, d1;
      f2_unpack(rsa[0], d0, d1);
      tmem_ld_wait_after<32>(vn, d0);              // issued after this chunk's exponentials
      cm_cur = chunk_max(vn, keep[ch + 1]);
    } else {
      cm_cur = kNegInf;
    }
    if (ch == 0 && n_item > 0) {
      // P_x and O_x are free once the previous PV of this query tile has completed
      const bool ok = wait_bar(&bars.pv_done[x], (cnt - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) return false;
      tc_fence_after();
    }
    tmem_st_x16(tP + ch * 16, pk);
  }

  // O holds the previous tiles at the old max: rescale once if this tile moved it
  if (n_item > 0 && __any_sync(0xffffffffu, m_use != m_start)) {
    const float alpha = (m_use != m_start) ? ex2_approx(m_start - m_use) : 1.f;
    const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t ov[32];
      tmem_ld_x32(tO + ch * 32, ov);
      tmem_ld_wait<32>(ov);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        uint64_t r;
        asm("mul.rn.f32x2 %0, %1, %2;"
            : "=l"(r)
            : "l"(f2_pack(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1]))), "l"(al2));
        float lo, hi;
        f2_unpack(r, lo, hi);
        ov[j] = __float_as_uint(lo);
        ov[j + 1] = __float_as_uint(hi);
      }
      tmem_st_x32(tO + ch * 32, ov);
    }
  }
  const uint64_t rs2 = f2_add(f2_add(rsa[0], rsa[1]), f2_add(rsa[2], rsa[3]));
  float rs_lo, rs_hi;
  f2_unpack(rs2, rs_lo, rs_hi);
  l += rs_lo + rs_hi;
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars.p_full[x]);
  ++cnt;
  ++n_item;
  return true;
}

template <int D>
__device__ void softmax_epilogue(const Params& p, Bars& bars, Meta* meta, uint32_t tmem, volatile int* abort_flag) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int x = (warp - 2) >> 2;                     // warps 2-5: tile A, warps 6-9: tile B
  const int quarter = warp & 3;                      // TMEM lanes this warp may access
  const int row = quarter * 32 + lane;               // query row within the tile
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const int rows_per_item = kItemRows >> p.log2b;
  const int sub = (x * kTile + row) >> p.log2b;      // query block within the item
  const int rloc = row & (p.block - 1);
  const float kNegInf = __int_as_float(0xff800000);
  const uint32_t tO = tmem + C::col_o(x) + lane_base;

  int mt = 0, cnt = 0;      // meta position, processed S tiles of this query tile (global)
  bool ok = true;
  int item_local = 0;
  for (int k = blockIdx.x; k < p.n_items && ok; k += gridDim.x, ++item_local) {
    const Item it = decode_item(p, k);
    const int qblk = it.pair * rows_per_item + sub;
    float m_use = kNegInf;   // running reference max, log2 units
    float l = 0.f;
    int n_item = 0;
    for (;;) {
      const int ms = mt % kMetaRing;
      if (!(ok = wait_bar(&bars.m_full[ms], (mt / kMetaRing) & 1, abort_flag))) break;
      const Meta m = load_meta(&meta[ms]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.m_empty[ms]);
      ++mt;
      if (m.kind != kKeyTile) break;
      if (!(m.active & (1 << x))) continue;
      if (!(ok = softmax_tile<D>(p, bars, m, x, tmem, lane_base, sub, qblk, rloc, m_use, l, cnt, n_item,
                                 abort_flag)))
        break;
    }
    if (!ok) break;

    // epilogue: O / l and LSE of this query tile
    if (n_item > 0) {
      ok = wait_bar(&bars.pv_done[x], (cnt - 1) & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
    }
    const int qtok = it.pair * kItemRows + x * kTile + row;
    const bool store = qtok < p.n_tokens;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* orow = p.o + (int64_t)it.s * p.o_sb + (int64_t)qtok * p.o_sn + (int64_t)it.h * p.o_sh;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t ov[32];
      if (n_item > 0) {
        tmem_ld_x32(tO + ch * 32, ov);
        tmem_ld_wait<32>(ov);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2)
        pk[j >> 1] = pack_bf16x2(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.o_empty[x]);
    if (store) {
      const float lse = l > 0.f ? (m_use + __log2f(l)) * 0.69314718055994531f : kNegInf;
      p.lse[((int64_t)it.s * p.heads + it.h) * p.n_tokens + qtok] = lse;
    }
  }
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sQ = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sQ + 2 * C::TILE_BYTES;
  uint8_t* sV = sK + C::STAGES * C::TILE_BYTES;
  UnionSmem& un = *reinterpret_cast<UnionSmem*>(sV + C::STAGES * C::TILE_BYTES);
  __shared__ Bars bars;
  __shared__ Meta meta[kMetaRing];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 2);              // both MMA threads
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 2);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 2);
    }
    for (int i = 0; i < kMetaRing; ++i) {
      mbar_init(&bars.m_full[i], 1);
      mbar_init(&bars.m_empty[i], kMetaConsumers);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.s_full[x], 1);
      mbar_init(&bars.p_full[x], 4);
      mbar_init(&bars.pv_done[x], 1);
      mbar_init(&bars.o_empty[x], 4);
      mbar_init(&bars.drain[x], 1);
    }
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    producer<D>(p, &tq, &tk, &tv, bars, meta, un, sQ, sK, sV, &abort_flag);
  } else if (warp == 1 || warp == 10) {
    if ((threadIdx.x & 31) == 0) mma_issuer<D>(p, bars, meta, sQ, sK, sV, tmem, warp == 1 ? 0 : 1, &abort_flag);
    __syncwarp();
  } else {
    softmax_epilogue<D>(p, bars, meta, tmem, &abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
int launch_d(const AttnArgs& a, cudaStream_t stream) {
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv;
  if (!encode_bhnd_map(&tq, a.q, a.batch, a.n_tokens, a.heads, D, a.q_strides[0], a.q_strides[1], a.q_strides[2],
                       C::CH, kTile, C::TMA_SWZ) ||
      !encode_bhnd_map(&tk, a.k, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::CH, (uint32_t)a.block, C::TMA_SWZ) ||
      !encode_bhnd_map(&tv, a.v, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                       a.kv_strides[2], C::CH, (uint32_t)a.block, C::TMA_SWZ))
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
  p.pairs_per_seq = (a.n_tokens + kItemRows - 1) / kItemRows;
  p.n_items = a.batch * a.heads * p.pairs_per_seq;
  p.row_ptr = a.row_ptr;
  p.col_idx = a.col_idx;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.o_sb = a.o_strides[0];
  p.o_sn = a.o_strides[1];
  p.o_sh = a.o_strides[2];
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  static int sm_count = 0;
  if (sm_count == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (sm_count <= 0) sm_count = 148;
  }
  auto kern = attn_fwd_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return SA_ERR_CUDA;
  const int grid = p.n_items < sm_count ? p.n_items : sm_count;
  kern<<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace

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
