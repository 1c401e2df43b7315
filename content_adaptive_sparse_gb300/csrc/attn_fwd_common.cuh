// Shared parts of the block-sparse attention forward kernels (attn_fwd.cu): the work items,
// the planner that builds each item's key-tile list, the batch ring that hands the tiles to
// the other roles, and the TMA loader. Included once, by attn_fwd.cu.
//
// Work item: one 128-row query tile of one (sequence, head): the tile's key list is the
// sorted union of its query blocks' CSR rows, each key block tagged with one membership bit
// per query block. The list is cut into 32-key chunks and four consecutive chunks form one
// key tile (128 keys; the last tile of an item may be shorter).
//
// Token rule: key j of block J is visible to query i of block I iff J is in row(I) and
// (not causal or j <= i) ("Parameter-free Adaptive Sparse Attention via Compression-Based
// Content Selection", section 3.4 block-to-token expansion). No token mask is materialised.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csr_union.cuh"
#include "ptx_sm100.cuh"
#include "sa_internal.h"
#include "tma_host.h"

namespace sa {
namespace {

__device__ unsigned int g_attn_err;

constexpr int kTile = 128;            // query rows per work item
constexpr int kKeys = 128;            // keys per S tile (four 32-key chunks)
constexpr int kThreads = 512;         // 16 warps, four warpgroups
constexpr int kMetaRing = 2;          // batch entries: items claimed ahead of the consumers
constexpr uint32_t kTmemCols = 512;
// Register split (setmaxnreg): the launch gives every thread 128 registers; the two
// warpgroups of control warps drop to kCtrlRegs so that the two softmax warpgroups can hold a
// whole 128-key score row: 8 warps x 184 + 8 warps x 72 = 16 warps x 128 per thread (the
// one-stream kernel; the two-pipeline kernel splits 192 / 64).
constexpr int kLaunchRegs = 128;
constexpr int kSoftmaxRegs = 184;
constexpr int kCtrlRegs = 72;
static_assert(8 * kSoftmaxRegs + 8 * kCtrlRegs == 16 * kLaunchRegs, "register split");
constexpr int kMaxStages = 4;

// Shared-memory layout per head dimension. d <= 64 runs the two-pipeline kernel (per pipeline:
// Q buffers, K and V rings, the union scratch; two pipelines per CTA), d = 128 the one-stream
// kernel (one set of buffers and rings per CTA, plus the softmax warps' exchange slots).
template <int D>
struct Cfg {
  static_assert(D == 32 || D == 64 || D == 128, "head dimension");
  static constexpr bool WIDE = D == 128;
  static constexpr int CH = D >= 64 ? 64 : 32;         // head-dimension elements per swizzled row
  static constexpr int NCH = D / CH;                   // d-chunks of a row
  static constexpr int ROWB = CH * 2;                  // bytes per swizzled row
  static constexpr uint32_t SWZ = ROWB == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr CUtensorMapSwizzle TMA_SWZ =
      ROWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static constexpr uint32_t ATOM = 8 * ROWB;           // swizzle atom (8 rows)
  static constexpr int Q_CHUNK = kTile * ROWB;         // one d-chunk of the Q tile
  static constexpr int Q_BYTES = NCH * Q_CHUNK;
  static constexpr int KV_CHUNK = kKeys * ROWB;        // one d-chunk of a K or V tile
  static constexpr int KV_BYTES = NCH * KV_CHUNK;      // one K or V tile
  // Ring depths (per pipeline at d <= 64, per CTA at d = 128). V is loaded one key tile
  // behind K (it is needed one softmax later); the next item's Q lands in the second buffer.
  static constexpr int QB = 2;
  static constexpr int KS = D == 32 ? 4 : 2;
  static constexpr int VS = KS;
  static constexpr int UNION_BYTES = kMaxTileBlocks * (kMaxMaskBlocks / 32) * 4 + kMaxMaskBlocks * 2;
  static constexpr int XCH_FLOATS = 2 * 2 * 4 * 32;    // [phase parity][key half][lane quarter][lane]
  static constexpr int PIPE_BYTES = (QB * Q_BYTES + (KS + VS) * KV_BYTES + UNION_BYTES + 1023) & ~1023;
  static constexpr int SMEM =
      WIDE ? 1024 + ((QB * Q_BYTES + (KS + VS) * KV_BYTES + UNION_BYTES + XCH_FLOATS * 4 + 1023) & ~1023)
           : 1024 + 2 * PIPE_BYTES;
  static_assert(KS <= kMaxStages && VS <= kMaxStages, "ring size");
  static_assert(SMEM <= 225 * 1024, "shared memory");
};

// The planner hands work to the other roles through a ring of batches: each entry carries up
// to kBatch key tiles of one item, so every consumer pays one barrier round trip per batch,
// not per tile. An item is one or more consecutive entries (the first and last flagged; an
// item without key tiles is one entry with no tiles); a Done entry ends the launch.
constexpr int kBatch = 16;
enum : int { kKindItem = 0, kKindDone = 1 };
enum : int { kFirst = 1, kLast = 2 };

struct __align__(16) Batch {
  int kind;
  int ntiles;                 // key tiles in this entry (0 .. kBatch)
  int item;                   // work item index
  int flags;                  // kFirst | kLast
  int slot;                   // partial-result slot of a split item's part (-1: the whole item)
  int pad[3];
  int4 tile[kBatch];          // per key tile and 32-key chunk c (x, y, z, w): first key token
                              // << 4 | membership bits (bit r: query block r); 0 = no chunk
  uint8_t nch[kBatch];        // per key tile: 32-key chunks (1 .. 4); 16-byte aligned
  uint8_t vq[4][kBatch];      // per TMEM lane quarter and key tile: bits 0-3, chunk c visible
                              // to some row of the quarter; bits 4-6, 1 + the causal-diagonal
                              // chunk (0: none)
};

// Visibility byte of one key tile for the 32 query rows of lane quarter q (rows 32q ..
// 32q+31 of the item's query tile, first query token q_warp; query block sub). Query and key
// chunks start at multiples of 32, so under causality at most one chunk (the one starting at
// q_warp) is the diagonal, where row r sees columns 0 .. r.
__device__ __forceinline__ int quarter_vis(const int (&tm)[4], int nch, int sub, int q_warp, int causal) {
  int vis = 0, dch = -1;
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    if (ch < nch && ((tm[ch] >> sub) & 1)) {
      const int lim0 = q_warp - (tm[ch] >> 4);     // row r sees columns c <= lim0 + r
      if (!causal || lim0 >= 31) {
        vis |= 1 << ch;
      } else if (lim0 + 31 >= 0) {
        vis |= 1 << ch;
        dch = ch;
      }
    }
  }
  return vis | ((dch + 1) << 4);
}

__device__ __forceinline__ uint4 ld_shared_u4(const void* ptr) {
  uint4 r;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_u32(ptr))
               : "memory");
  return r;
}

// Word w (0 .. 3) of a 16-byte value (selects, not an indexed read: stays in registers).
__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

__device__ __forceinline__ int4 ld_shared_v4(const void* ptr) {
  int4 r;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(smem_u32(ptr))
               : "memory");
  return r;
}

// Chunks present in a key tile (they fill positions 0 .. n-1; a present chunk always has at
// least one membership bit, so its entry is nonzero).
__device__ __forceinline__ int tile_chunks(const int4& t) {
  return (t.x != 0) + (t.y != 0) + (t.z != 0) + (t.w != 0);
}

struct Params {
  int batch, n_tokens, heads, heads_per_kv, block, log2b, nb, causal, csr_shared;
  int tiles_per_seq;          // 128-row query tiles per (sequence, head)
  int n_items;
  unsigned int* work_counter;          // next work-list entry (in the workspace, zeroed before the launch)
  // Split mode (work_list != nullptr): the schedule kernel's list of (item, part) entries, split
  // parts first; entry i < n_split is part y of item x, whose key tiles [y T, (y + 1) T) go
  // to partial-result slot i. Header: list length, n_split, T.
  const int2* work_list;
  const int* list_hdr;
  float* partial;                      // slots of 128 x (d + 1) floats: O rows, then LSE
  int csr_batches;
  int n_masks;
  const int32_t* row_ptr[kMaxMasks];   // one CSR per head group
  const int32_t* col_idx[kMaxMasks];
  uint8_t head_mask[kMaxHeadMap];      // query head -> CSR (n_masks > 1)
  __nv_bfloat16* o;
  int o_tma;                           // the kernel's output tensor map describes o (TMA stores)
  float* lse;
  int64_t o_sb, o_sn, o_sh;
  float scale_log2;
};
struct Item {
  int s, h, tile;
};

// Work item k of the longest-first order: all (sequence, head) pairs of one query-tile rank
// before the next rank; causal ranks run from the last query tile.
__device__ __forceinline__ Item decode_item(const Params& p, int k) {
  const int bh = k % (p.batch * p.heads);
  const int rank = k / (p.batch * p.heads);
  Item it;
  it.h = bh % p.heads;
  it.s = bh / p.heads;
  it.tile = p.causal ? (p.tiles_per_seq - 1 - rank) : rank;
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
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Waits (one thread) until ring entry mt is published and returns its header (kind, ntiles,
// item, flags); false on abort. Bars is the kernel's barrier set (m_full / m_empty).
template <class Bars>
__device__ __forceinline__ bool wait_batch(Bars& bars, const Batch* ring, int mt, int4& hdr,
                                           volatile int* abort_flag) {
  const int ms = mt % kMetaRing;
  if (!wait_bar(&bars.m_full[ms], (uint32_t)(mt / kMetaRing) & 1u, abort_flag)) return false;
  hdr = ld_shared_v4(&ring[ms]);
  return true;
}

// ------------------------------------------------------------------ tile loads

// The TMA boxes of one key tile (b = 32: one 32-row box per chunk; b >= 64: one 64-row box
// per chunk pair) and where they go. V is loaded one key tile behind K, so the boxes of the
// tile whose V is pending are kept here: the union list may already hold the next item.
struct TileLoad {
  int t;                      // key tile index within this ring (its position)
  int nbox, rows, s, hk;
  uint32_t bytes;
  int tok[4];
};

// Lane 0: waits for ring stage t % S of (full, empty) and issues the tile's boxes into it
// (each box once per d-chunk; chunk c of a stage starts KV_CHUNK * c bytes in).
template <int D, int S>
__device__ __forceinline__ bool load_tile(const TileLoad& L, const CUtensorMap* map, uint8_t* ring, uint64_t* full,
                                          uint64_t* empty, volatile int* abort_flag) {
  using C = Cfg<D>;
  const int st = L.t % S;
  if (!wait_bar(&empty[st], ((L.t / S) & 1) ^ 1, abort_flag)) return false;
  mbar_arrive_expect_tx(&full[st], L.bytes);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (i < L.nbox)
#pragma unroll
      for (int c = 0; c < C::NCH; ++c)
        tma_load_4d(ring + st * C::KV_BYTES + c * C::KV_CHUNK + i * L.rows * C::ROWB, map, &full[st], c * C::CH,
                    L.hk, L.tok[i], L.s);
  return true;
}

// ------------------------------------------------------------------ planner (one warp per ring)

// Claims work items from the launch-wide counter, builds each item's key-block union and
// publishes the item's key tiles in batches. With two ring entries the next item's union is
// built while the consumers still work on the current one, and no more than about two items
// are claimed ahead of them.
template <int D, class Bars>
__device__ void planner(const Params& p, Bars& bars, Batch* ring, UnionSmem& u, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const int b = p.block;
  const int cpb = b >> 5;                            // 32-key chunks per key block
  const int qb_per_tile = kTile >> p.log2b;
  int mt = 0;
  bool ok = true;
  const bool split_mode = p.work_list != nullptr;
  const int list_len = split_mode ? p.list_hdr[0] : p.n_items;
  const int n_split = split_mode ? p.list_hdr[1] : 0;
  const int part_tiles = split_mode ? p.list_hdr[2] : 0;
  for (;;) {
    int idx = 0;
    if (lane == 0) idx = (int)atomicAdd(p.work_counter, 1u);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    const bool done = idx >= list_len;
    int k = idx, part = 0;
    if (split_mode && !done) {
      const int2 ent = p.work_list[idx];
      k = ent.x;
      part = ent.y;
    }
    const int slot = (split_mode && idx < n_split) ? idx : -1;
    int n_chunks = 0;
    if (!done) {
      const Item it = decode_item(p, k);
      const int I0 = (it.tile * kTile) >> p.log2b;
      const int nq = min(qb_per_tile, p.nb - I0);
      const int mi = p.n_masks > 1 ? p.head_mask[it.h] : 0;
      const int32_t* rp = p.row_ptr[mi] + (size_t)(p.csr_shared ? 0 : it.s) * (p.nb + 1);
      n_chunks = cpb * build_union(p.nb, p.causal ? kKeepLE : kKeepAll, u, rp, p.col_idx[mi], I0, nq, &g_attn_err,
                                   kErrBadIndex);
    }
    const int n_all = (n_chunks + 3) >> 2;
    // key tiles of this entry: all of the item's, or a split part's range
    const int t_begin = slot >= 0 ? min(n_all, part * part_tiles) : 0;
    const int n_tiles = slot >= 0 ? min(n_all, t_begin + part_tiles) : n_all;
    for (int t0 = t_begin;; t0 += kBatch) {
      const int ms = mt % kMetaRing;
      if (lane == 0) ok = wait_bar(&bars.m_empty[ms], ((mt / kMetaRing) & 1) ^ 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const int nt = done ? 0 : min(kBatch, n_tiles - t0);
      // lane i < nt describes key tile t0 + i
      if (lane < nt) {
        int tm[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int q = 4 * (t0 + lane) + c;         // chunk index within the item
          const uint32_t e = q < n_chunks ? u.list[q / cpb] : 0u;
          tm[c] = q < n_chunks ? ((((int)(e & 0xfffu) * b + (q % cpb) * 32) << 4) | (int)(e >> 12)) : 0;
        }
        ring[ms].tile[lane] = make_int4(tm[0], tm[1], tm[2], tm[3]);
        const int nch = min(4, n_chunks - 4 * (t0 + lane));
        ring[ms].nch[lane] = (uint8_t)nch;
        const int tile0 = decode_item(p, k).tile * kTile;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          ring[ms].vq[q][lane] = (uint8_t)quarter_vis(tm, nch, (32 * q) >> p.log2b, tile0 + 32 * q, p.causal);
      }
      if (lane == 0) {
        *reinterpret_cast<int4*>(&ring[ms]) = make_int4(done ? kKindDone : kKindItem, nt, k,
                                                        (t0 == t_begin ? kFirst : 0) | (t0 + kBatch >= n_tiles ? kLast : 0));
        ring[ms].slot = slot;
      }
      __syncwarp();                                  // every lane's entry is written before the release
      if (lane == 0) mbar_arrive(&bars.m_full[ms]);
      ++mt;
      if (done || t0 + kBatch >= n_tiles) break;
    }
    if (!ok || done) break;
    __syncwarp();   // the next item's union may overwrite the list
  }
}

// ------------------------------------------------------------------ loader (lane 0 of one warp per ring)

// Reads the batch ring and issues the TMA loads: Q at each item's start (Q_BYTES into buffer
// item % QB), K of each key tile, and V one key tile later (the V of an item's last tile at
// the item's end). Copies still in flight are drained before return.
template <int D, class Bars>
__device__ void loader(const Params& p, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       Bars& bars, const Batch* ring, uint8_t* sQ, uint8_t* sK, uint8_t* sV,
                       volatile int* abort_flag) {
  using C = Cfg<D>;
  const int rows = p.block == 32 ? 32 : 64;          // rows per TMA box
  int kt = 0, item_local = -1;
  int k_issued = 0, v_issued = 0, q_last = -1;       // loads issued (drained at the end)
  int cur_s = 0, cur_hk = 0;
  bool ok = true;
  bool v_pending = false;                            // the V of tile `pend` is not yet issued
  TileLoad pend;
  pend.t = 0;
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
      const Item it = decode_item(p, hdr.z);
      cur_s = it.s;
      cur_hk = it.h / p.heads_per_kv;
      const int qb = item_local % C::QB;
      if (item_local >= C::QB && !(ok = wait_bar(&bars.q_empty[qb], ((item_local / C::QB) - 1) & 1, abort_flag)))
        break;
      // rows beyond the sequence are zero-filled by TMA
      mbar_arrive_expect_tx(&bars.q_full[qb], C::Q_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCH; ++c)
        tma_load_4d(sQ + qb * C::Q_BYTES + c * C::Q_CHUNK, tq, &bars.q_full[qb], c * C::CH, it.h, it.tile * kTile, it.s);
      q_last = item_local;
    }
    for (int i = 0; i < hdr.y && ok; ++i) {
      const int4 tm = ld_shared_v4(&e.tile[i]);
      const int nch = tile_chunks(tm);
      TileLoad L;
      L.t = kt;
      L.rows = rows;
      L.nbox = (nch * 32 + rows - 1) / rows;
      L.s = cur_s;
      L.hk = cur_hk;
      L.bytes = (uint32_t)(nch * 32 * D * 2);
      L.tok[0] = tm.x >> 4;
      L.tok[1] = (rows == 32 ? tm.y : tm.z) >> 4;
      L.tok[2] = tm.z >> 4;
      L.tok[3] = tm.w >> 4;
      if (!(ok = load_tile<D, C::KS>(L, tk, sK, bars.k_full, bars.k_empty, abort_flag))) break;
      k_issued = ++kt;
      if (v_pending) {
        if (!(ok = load_tile<D, C::VS>(pend, tv, sV, bars.v_full, bars.v_empty, abort_flag))) break;
        v_issued = pend.t + 1;
      }
      pend = L;
      v_pending = true;
    }
    if (!ok) break;
    mbar_arrive(&bars.m_empty[mt % kMetaRing]);
    if ((hdr.w & kLast) && v_pending) {
      // end of the item: its last V cannot wait for the next item's first K
      if (!(ok = load_tile<D, C::VS>(pend, tv, sV, bars.v_full, bars.v_empty, abort_flag))) break;
      v_issued = pend.t + 1;
      v_pending = false;
    }
  }
  // Drain the copies in flight before the CTA may exit.
  for (int i = max(0, q_last - C::QB + 1); i <= q_last; ++i) drain_bar(&bars.q_full[i % C::QB], (i / C::QB) & 1);
  for (int t = max(0, k_issued - C::KS); t < k_issued; ++t) drain_bar(&bars.k_full[t % C::KS], (t / C::KS) & 1);
  for (int t = max(0, v_issued - C::VS); t < v_issued; ++t) drain_bar(&bars.v_full[t % C::VS], (t / C::VS) & 1);
}

// Descriptor offset (bytes >> 4) of k-step ks (16 head-dimension elements) inside a K-major
// tile whose d-chunks are `chunk` bytes apart.
template <int D>
__device__ __forceinline__ constexpr uint64_t kmajor_step(int ks, int chunk) {
  using C = Cfg<D>;
  return (uint64_t)((((ks * 16) / C::CH) * chunk + ((ks * 16) % C::CH) * 2) >> 4);
}

// Max of the 32 scores of one chunk, folded into acc.
__device__ __forceinline__ float chunk_max(const uint32_t* v, float acc) {
  const float kNegInf = __int_as_float(0xff800000);
  float a[4] = {acc, kNegInf, kNegInf, kNegInf};
#pragma unroll
  for (int j = 0; j < 32; j += 2)
    a[(j >> 1) & 3] = max3(a[(j >> 1) & 3], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
  return fmaxf(max3(a[0], a[1], a[2]), a[3]);
}

// Causal diagonal chunk: scores of columns this row may not see become -inf (bit j of kp:
// column j visible), so the unmasked max and exponential paths below handle the chunk.
__device__ __forceinline__ void mask_chunk(uint32_t* v, uint32_t kp) {
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = ((kp >> j) & 1u) ? v[j] : 0xff800000u;
}

// 2^x of two values on the FMA pipe: Cody-Waite range reduction 2^x = 2^n * 2^f with
// n = floor(x) (rounding x + 1.5 * 2^23 toward minus infinity leaves n in the low mantissa bits)
// and f = x - n in [0, 1), then a cubic fitted to 2^f on [0, 1] for this kernel (least squares,
// largest relative error 7.5e-5, far below the bf16 rounding of P); 2^n enters as n added to the
// exponent field. x is at most 8 here (the lazily rescaled running max); x below -126 (masked
// scores included) gives exactly 0.
__device__ __forceinline__ uint64_t exp2_fma2(uint64_t x2) {
  float a, b;
  f2_unpack(x2, a, b);
  const float ac = fmaxf(a, -127.f), bc = fmaxf(b, -127.f);
  const uint64_t x = f2_pack(ac, bc);
  const uint64_t magic = f2_pack(12582912.f, 12582912.f);
  uint64_t t, n, f;
  asm("add.rm.f32x2 %0, %1, %2;" : "=l"(t) : "l"(x), "l"(magic));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(n) : "l"(t), "l"(magic));
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(f) : "l"(x), "l"(n));
  uint64_t q = f2_fma(f, f2_pack(0.07802403f, 0.07802403f), f2_pack(0.22606707f, 0.22606707f));
  q = f2_fma(f, q, f2_pack(0.695834f, 0.695834f));
  q = f2_fma(f, q, f2_pack(0.99992514f, 0.99992514f));
  float q0, q1, t0, t1;
  f2_unpack(q, q0, q1);
  f2_unpack(t, t0, t1);
  const float r0 = a < -126.f ? 0.f : __uint_as_float(__float_as_uint(q0) + (__float_as_uint(t0) << 23));
  const float r1 = b < -126.f ? 0.f : __uint_as_float(__float_as_uint(q1) + (__float_as_uint(t1) << 23));
  return f2_pack(r0, r1);
}

// p = 2^(s c - m) of one chunk into packed bf16 (a score of -inf gives exactly 0); adds the
// row sum into rs. The first POLY of the chunk's 16 pairs take 2^x on the FMA pipe, the rest
// on the MUFU pipe (ex2.approx), so that the two pipes share the exponentials.
template <int POLY = 0>
__device__ __forceinline__ void chunk_exp(const uint32_t* v, uint64_t c2, uint64_t negm2, uint32_t* pk, uint64_t* rs) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), c2, negm2);
    float p0, p1;
    if ((j >> 1) < POLY) {
      f2_unpack(exp2_fma2(x2), p0, p1);
    } else {
      float x0, x1;
      f2_unpack(x2, x0, x1);
      p0 = ex2_approx(x0);
      p1 = ex2_approx(x1);
    }
    rs[(j >> 1) & 1] = f2_add(rs[(j >> 1) & 1], f2_pack(p0, p1));
    pk[j >> 1] = pack_bf16x2(p0, p1);
  }
}

}  // namespace
}  // namespace sa
