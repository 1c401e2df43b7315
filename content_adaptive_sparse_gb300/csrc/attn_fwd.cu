// Block-sparse flash-attention forward for sm_103a (tcgen05 + TMEM + TMA), 64-key tiles.
//
// The library runs this kernel for head dimension 128. Head dimensions 32 and 64 go to
// attn_fwd_wide.cu (128-key tiles, one full score row per softmax thread), which is faster
// there; the template below still compiles for d = 32 and 64 (split accumulators at d = 32)
// and is kept as the measured baseline of that design.
//
// Work item: one 128-row query tile of one (sequence, head), covering 128 / b query
// blocks. The key blocks the tile visits are the sorted union of those blocks' CSR rows;
// each key block carries one membership bit per query block of the tile. The union is cut
// into 32-key chunks, and consecutive chunk pairs form 64-key key tiles.
//
// One CTA per SM runs two independent pipelines x = 0, 1 (one query tile each), so the
// tensor core always has the other pipeline's work while one waits. Each pipeline has
// its own Q buffer, K/V ring, meta ring and half of TMEM. The kernel is persistent: each
// pipeline's producer takes the next query tile from a launch-wide counter over a list
// ordered longest first (causal: last query tiles first; BigBird: the global rows first),
// so a pipeline that drew a long tile takes fewer of the rest.
//
// Warp roles (640 threads):
//   warps 0, 19  producer of pipeline 0 / 1: builds the union (whole warp), publishes
//                key-tile descriptions, issues TMA loads of Q and of the K / V chunks.
//   warps 1, 18  lane 0 issues the tcgen05 MMAs of pipeline 0 / 1:
//                  S[j % NS] = Q K_j^T        (A, B from shared memory, N = 64 keys)
//                  O += P_j V_j               (A = P_j from TMEM, B = V_j, MN-major)
//                QK of the first NS key tiles up front; after each PV_j completes, QK_{j+NS}
//                into the buffer it frees. The softmax therefore always finds the next S
//                ready. Warp 1 owns TMEM (512 columns).
//   warps 2-9, 10-17  softmax of pipeline 0 / 1, two warps per TMEM lane quarter (warp w
//                reads quarter w % 4): one query row per thread, one 32-key chunk per warp.
//                The pair agrees on each tile's row max through shared memory, keeps a
//                lazily rescaled running max (O is rescaled only when the max grows by more
//                than 2^8), writes P = 2^(s c - m) in bf16 over the first 32 columns of the
//                tile's own S buffer, and finally normalises and stores its half of O (bf16)
//                and the LSE (fp32). The exponentials (MUFU, 4 cycles per warp instruction
//                on each SM sub-partition) bound this stage; four softmax warps per
//                sub-partition keep that unit busy.
// TMEM columns of pipeline x: S buffers [256x + 64i, +64), i < NS; O [256x + 64 NS, +d).
//
// Token rule: key j of block J is visible to query i of block I iff J is in row(I) and
// (not causal or j <= i) ("Parameter-free Adaptive Sparse Attention via Compression-Based
// Content Selection", section 3.4 block-to-token expansion). No token mask is
// materialised: the per-row column mask comes from the membership bits and, on the
// diagonal, from the causal compare.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "csr_union.cuh"
#include "ptx_sm100.cuh"
#include "sa_internal.h"
#include "tma_host.h"

namespace sa {
namespace {

__device__ unsigned int g_attn_err;

// Work counters of the persistent kernel: each launch takes one slot (round robin) and zeroes
// it on its stream, so up to kWorkSlots launches may be in flight at once on any streams.
constexpr int kWorkSlots = 64;
__device__ unsigned int g_work_counters[kWorkSlots];

constexpr int kTile = 128;          // query rows per work item
constexpr int kKeyTile = 64;        // keys per S tile (two 32-key chunks)
constexpr int kThreads = 640;       // 20 warps
constexpr int kMetaRing = 8;
constexpr uint32_t kTmemCols = 512;
constexpr int kSoftmaxWarps = 8;    // per pipeline: two per TMEM lane quarter (one per 32-key chunk)
constexpr int kMetaConsumers = 1 + kSoftmaxWarps;   // the MMA thread and the softmax warps
constexpr int kMaxStages = 8;
constexpr int kMaxSBuf = 3;

template <int D>
struct Cfg {
  static constexpr int CH = D >= 64 ? 64 : 32;         // elements per swizzled row
  static constexpr int NCH = D / CH;                   // d-chunks
  static constexpr int ROWB = CH * 2;                  // bytes per swizzled row
  static constexpr uint32_t SWZ = ROWB == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr CUtensorMapSwizzle TMA_SWZ =
      ROWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static constexpr uint32_t ATOM = 8 * ROWB;           // swizzle atom (8 rows)
  static constexpr int Q_CHUNK = kTile * ROWB;         // one d-chunk of the 128-row Q tile
  static constexpr int Q_BYTES = NCH * Q_CHUNK;
  static constexpr int KV_CHUNK = kKeyTile * ROWB;     // one d-chunk of a 64-key K or V tile
  static constexpr int KV_BYTES = NCH * KV_CHUNK;
  // d = 32: each 32-key chunk half of a tile has its own O accumulator (and running max),
  // so the two softmax warps of a row never synchronise per tile; d >= 64: one O, which
  // leaves TMEM for three S buffers at d = 64 (measured 4 % faster than split O with two).
  static constexpr bool SPLIT = D < 64;
  static constexpr int NO = SPLIT ? 2 : 1;             // O accumulators per pipeline
  static constexpr int NS = D <= 64 ? 3 : 2;           // S buffers per pipeline
  static constexpr int QB = D > 64 ? 1 : 2;            // Q buffers per pipeline
  static constexpr int STAGES = D == 128 ? 2 : (D == 64 ? 4 : 6);   // K and V ring depth
  static constexpr int UNION_BYTES = kMaxTileBlocks * (kMaxMaskBlocks / 32) * 4 + kMaxMaskBlocks * 2;   // 10 KB
  static constexpr int PIPE_BYTES = (QB * Q_BYTES + 2 * STAGES * KV_BYTES + UNION_BYTES + 1023) & ~1023;
  static constexpr int SMEM_NEED = 1024 + 2 * PIPE_BYTES;
  // at least 120 KB so that only one CTA (512 TMEM columns) is resident per SM
  static constexpr int SMEM = SMEM_NEED > 120 * 1024 ? SMEM_NEED : 120 * 1024;
  __host__ __device__ static constexpr uint32_t col_s(int x, int i) { return 256u * x + 64u * i; }
  __host__ __device__ static constexpr uint32_t col_o(int x, int h) { return 256u * x + 64u * NS + (SPLIT ? D * h : 0); }
  static_assert(64 * NS + NO * D <= 256, "TMEM budget of a pipeline");
  static_assert(STAGES >= NS && STAGES <= kMaxStages && NS <= kMaxSBuf, "ring sizes");
};

// Meta kinds: a key tile of the current item, the end of the item, the header of the next
// item (tok[0] = item index), no more items.
enum : int { kKindTile = 0, kKindEnd = 1, kKindItem = 2, kKindDone = 3 };

struct Meta {
  int kind;
  int nch;                    // chunks (1 or 2) in this key tile
  int tok[2];                 // first key token of each chunk
  int mask[2];                // bit r: query block r of the tile has the chunk's key block
};

// Field-wise read of a published ring entry (the producer's mbarrier arrive orders it).
__device__ __forceinline__ Meta load_meta(const Meta* src) {
  const volatile Meta* vm = src;
  Meta m;
  m.kind = vm->kind;
  m.nch = vm->nch;
  m.tok[0] = vm->tok[0];
  m.tok[1] = vm->tok[1];
  m.mask[0] = vm->mask[0];
  m.mask[1] = vm->mask[1];
  return m;
}

struct Params {
  int batch, n_tokens, heads, heads_per_kv, block, log2b, nb, causal, csr_shared;
  int tiles_per_seq;          // 128-row query tiles per (sequence, head)
  int n_items;
  unsigned int* work_counter;          // next item index (zeroed before the launch)
  int n_masks;
  const int32_t* row_ptr[kMaxMasks];   // one CSR per head group
  const int32_t* col_idx[kMaxMasks];
  uint8_t head_mask[kMaxHeadMap];      // query head -> CSR (n_masks > 1)
  __nv_bfloat16* o;
  float* lse;
  int64_t o_sb, o_sn, o_sh;
  float scale_log2;
};

struct PipeBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kMaxStages], k_empty[kMaxStages], v_full[kMaxStages], v_empty[kMaxStages];
  uint64_t m_full[kMetaRing], m_empty[kMetaRing];
  uint64_t s_full[kMaxSBuf], p_full[kMaxSBuf];
  uint64_t pv_done[2], o_empty, drain;   // pv_done[j & 1]: PV of key tile j
  // PVs of this pipeline known complete, written by the MMA thread (which waits for every
  // PV in order). The epilogue waits on this count: a parity wait on pv_done could be two
  // phases off there, and one that is a phase ahead of the barrier passes at once.
  int pv_count;
};

struct Item {
  int s, h, tile;
};

// Work item k of the static longest-first order: all (sequence, head) pairs of one
// query-tile rank before the next rank; causal ranks run from the last query tile.
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

// Bounded wait until *count >= target (a monotonic counter published with release
// semantics by another thread of the CTA).
__device__ __forceinline__ bool wait_count(const int* count, int target, volatile int* abort_flag) {
  const volatile int* c = count;
  if (*c >= target) {
    __threadfence_block();
    return true;
  }
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);                 // leave the issue slots to working warps
    if (*c >= target) {
      __threadfence_block();
      return true;
    }
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(&g_attn_err, kErrTimeout);
        return false;
      }
    }
  }
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

// ------------------------------------------------------------------ producer (warps 0, 11)

template <int D>
__device__ void producer(const Params& p, int x, const CUtensorMap* tq, const CUtensorMap* tk,
                         const CUtensorMap* tv, PipeBars& bars, Meta* meta, UnionSmem& u, uint8_t* sQ, uint8_t* sK,
                         uint8_t* sV, volatile int* abort_flag) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const int b = p.block;
  const int cpb = b >> 5;                            // 32-key chunks per key block
  const int qb_per_tile = kTile >> p.log2b;
  int mt = 0, kt = 0, item_local = 0;
  int k_issued = 0, v_issued = 0;                    // key tiles whose K / V loads were issued
  int q_last = -1;                                   // item_local of the last Q load
  bool ok = true;

  for (;; ++item_local) {
    // the next item of the launch-wide longest-first list, announced to the MMA thread and
    // the softmax warps of this pipeline through the meta ring
    int k = 0;
    if (lane == 0) k = (int)atomicAdd(p.work_counter, 1u);
    k = __shfl_sync(0xffffffffu, k, 0);
    {
      Meta hm;
      hm.kind = k < p.n_items ? kKindItem : kKindDone;
      hm.nch = 0;
      hm.tok[0] = k;
      hm.tok[1] = 0;
      hm.mask[0] = hm.mask[1] = 0;
      if (lane == 0) {
        const int ms = mt % kMetaRing;
        ok = wait_bar(&bars.m_empty[ms], ((mt / kMetaRing) & 1) ^ 1, abort_flag);
        if (ok) {
          meta[ms] = hm;
          mbar_arrive(&bars.m_full[ms]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      ++mt;
      if (!ok || hm.kind == kKindDone) break;
    }
    const Item it = decode_item(p, k);
    const int q0 = it.tile * kTile;
    const int I0 = q0 >> p.log2b;
    const int hk = it.h / p.heads_per_kv;
    const int nq = min(qb_per_tile, p.nb - I0);
    const int mi = p.n_masks > 1 ? p.head_mask[it.h] : 0;
    const int32_t* rp = p.row_ptr[mi] + (size_t)(p.csr_shared ? 0 : it.s) * (p.nb + 1);

    // Q into buffer item_local % QB (rows beyond the sequence are zero-filled by TMA)
    if (lane == 0) {
      const int qb = item_local % C::QB;
      if (item_local >= C::QB) ok = wait_bar(&bars.q_empty[qb], ((item_local / C::QB) - 1) & 1, abort_flag);
      if (ok) {
        mbar_arrive_expect_tx(&bars.q_full[qb], C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
          tma_load_4d(sQ + qb * C::Q_BYTES + c * C::Q_CHUNK, tq, &bars.q_full[qb], c * C::CH, it.h, q0, it.s);
        q_last = item_local;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) break;

    const int n_keys = build_union(p.nb, p.causal ? kKeepLE : kKeepAll, u, rp, p.col_idx[mi], I0, nq, &g_attn_err,
                                   kErrBadIndex);
    const int n_chunks = n_keys * cpb;

    for (int c0 = 0;; c0 += 2) {
      Meta m;
      m.kind = c0 < n_chunks ? kKindTile : kKindEnd;
      m.nch = min(2, n_chunks - c0);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int q = c0 + i;
        const uint32_t e = (i < m.nch) ? u.list[q / cpb] : 0u;
        m.tok[i] = (int)(e & 0xfffu) * b + (q % cpb) * 32;
        m.mask[i] = (i < m.nch) ? (int)(e >> 12) : 0;
      }
      if (lane == 0) {
        const int ms = mt % kMetaRing;
        ok = wait_bar(&bars.m_empty[ms], ((mt / kMetaRing) & 1) ^ 1, abort_flag);
        if (ok) {
          meta[ms] = m;
          mbar_arrive(&bars.m_full[ms]);
        }
        if (ok && m.kind == kKindTile) {
          const int st = kt % C::STAGES;
          const uint32_t ph = (kt / C::STAGES) & 1;
          const uint32_t bytes = (uint32_t)(m.nch * 32 * D * 2);
          // b = 32: one 32-row box per chunk; b >= 64: the two chunks are one 64-row box
          const int nbox = b == 32 ? m.nch : 1;
          ok = wait_bar(&bars.k_empty[st], ph ^ 1, abort_flag);
          if (ok) {
            mbar_arrive_expect_tx(&bars.k_full[st], bytes);
            for (int i = 0; i < nbox; ++i)
#pragma unroll
              for (int c = 0; c < C::NCH; ++c)
                tma_load_4d(sK + st * C::KV_BYTES + c * C::KV_CHUNK + i * 32 * C::ROWB, tk, &bars.k_full[st],
                            c * C::CH, hk, m.tok[i], it.s);
            k_issued = kt + 1;
            ok = wait_bar(&bars.v_empty[st], ph ^ 1, abort_flag);
          }
          if (ok) {
            mbar_arrive_expect_tx(&bars.v_full[st], bytes);
            for (int i = 0; i < nbox; ++i)
#pragma unroll
              for (int c = 0; c < C::NCH; ++c)
                tma_load_4d(sV + st * C::KV_BYTES + c * C::KV_CHUNK + i * 32 * C::ROWB, tv, &bars.v_full[st],
                            c * C::CH, hk, m.tok[i], it.s);
            v_issued = kt + 1;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      ++mt;
      if (m.kind == kKindTile) ++kt;
      if (!ok || m.kind == kKindEnd) break;
    }
    __syncwarp();   // the next tile's union may overwrite the list
  }
  // Drain this pipeline's own copies in flight before the CTA may exit.
  if (lane == 0) {
    for (int i = max(0, q_last - C::QB + 1); i <= q_last; ++i) drain_bar(&bars.q_full[i % C::QB], (i / C::QB) & 1);
    // the last tile that used each stage: waiting on it covers every earlier use
    for (int t = max(0, k_issued - C::STAGES); t < k_issued; ++t)
      drain_bar(&bars.k_full[t % C::STAGES], (t / C::STAGES) & 1);
    for (int t = max(0, v_issued - C::STAGES); t < v_issued; ++t)
      drain_bar(&bars.v_full[t % C::STAGES], (t / C::STAGES) & 1);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA issuer (warps 1, 10, lane 0)

// Byte offset (>> 4, the descriptor's address unit) of k-step ks inside a K-major tile
// whose d-chunks are `chunk` bytes apart.
template <int D>
__device__ __forceinline__ constexpr uint32_t kmajor_step(int ks, int chunk) {
  using C = Cfg<D>;
  return (uint32_t)(((ks * 16) / C::CH) * chunk + ((ks * 16) % C::CH) * 2) >> 4;
}

template <int D>
struct MmaState {
  uint32_t tmem;
  uint64_t qdesc, kdesc0, vdesc0;   // Q, K stage 0, V stage 0 at k-step 0
};

template <int D>
__device__ __forceinline__ void issue_qk(const MmaState<D>& st, int x, int qb, int buf, int stage, int nkeys) {
  using C = Cfg<D>;
  const uint32_t idesc = make_idesc_bf16(128, (uint32_t)nkeys, 0, 0);
  const uint64_t a0 = st.qdesc + (uint64_t)((qb * C::Q_BYTES) >> 4);
  const uint64_t b0 = st.kdesc0 + (uint64_t)((stage * C::KV_BYTES) >> 4);
  const uint32_t d = st.tmem + C::col_s(x, buf);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
    mma_bf16_ss(d, a0 + kmajor_step<D>(ks, C::Q_CHUNK), b0 + kmajor_step<D>(ks, C::KV_CHUNK), idesc,
                ks > 0 ? 1u : 0u);
}

// O += P V for one key tile; P of chunk h (keys 32h .. 32h+31) sits in TMEM columns
// 32h .. 32h+15 of the S buffer. With split accumulators chunk h goes to O_h; `init` says
// whether O_h already holds this query tile's sum (else it is overwritten), and is updated.
template <int D>
__device__ __forceinline__ void issue_pv(const MmaState<D>& st, int x, int buf, int stage, int nkeys, bool (&init)[2]) {
  using C = Cfg<D>;
  const uint32_t idesc = make_idesc_bf16(128, D, 0, 1);
  const uint64_t b0 = st.vdesc0 + (uint64_t)((stage * C::KV_BYTES) >> 4);
  const uint32_t a = st.tmem + C::col_s(x, buf);
  if (C::SPLIT) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (h == 1 && nkeys <= 32) break;
      const uint32_t d = st.tmem + C::col_o(x, h);
      mma_bf16_ts(d, a + 32u * h, b0 + (uint64_t)((32 * h * C::ROWB) >> 4), idesc, init[h] ? 1u : 0u);
      mma_bf16_ts(d, a + 32u * h + 8u, b0 + (uint64_t)(((32 * h + 16) * C::ROWB) >> 4), idesc, 1u);
      init[h] = true;
    }
  } else {
    const uint32_t d = st.tmem + C::col_o(x, 0);
    mma_bf16_ts(d, a, b0, idesc, init[0] ? 1u : 0u);
    mma_bf16_ts(d, a + 8u, b0 + (uint64_t)((16 * C::ROWB) >> 4), idesc, 1u);
    if (nkeys > 32) {
      mma_bf16_ts(d, a + 32u, b0 + (uint64_t)((32 * C::ROWB) >> 4), idesc, 1u);
      mma_bf16_ts(d, a + 40u, b0 + (uint64_t)((48 * C::ROWB) >> 4), idesc, 1u);
    }
    init[0] = true;
  }
}

// Per-S-buffer record of the key tiles whose QK is issued and PV pending (at most NS; kept
// in scalars selected by buffer index so nothing goes through local memory).
struct PendRing {
  int stage0, stage1, stage2, nkeys0, nkeys1, nkeys2;
  __device__ __forceinline__ void put(int buf, int stage, int nkeys) {
    if (buf == 0) { stage0 = stage; nkeys0 = nkeys; }
    else if (buf == 1) { stage1 = stage; nkeys1 = nkeys; }
    else { stage2 = stage; nkeys2 = nkeys; }
  }
  __device__ __forceinline__ void get(int buf, int& stage, int& nkeys) const {
    stage = buf == 0 ? stage0 : (buf == 1 ? stage1 : stage2);
    nkeys = buf == 0 ? nkeys0 : (buf == 1 ? nkeys1 : nkeys2);
  }
};

// The MMA-issuing thread of pipeline x. Per query tile: QK of the first NS key tiles, then
// for each key tile j: wait for P_j, PV_j, and once PV_{j+2-NS} has completed (it frees S
// buffer (j+2-NS) % NS), QK_{j+2} into that buffer. PVs are waited for in order and the
// completed count is published for the softmax epilogue.
template <int D>
__device__ void mma_issuer(const Params& p, int x, PipeBars& bars, Meta* meta, uint8_t* sQ, uint8_t* sK,
                           uint8_t* sV, uint32_t tmem, volatile int* abort_flag) {
  using C = Cfg<D>;
  MmaState<D> st;
  st.tmem = tmem;
  st.qdesc = make_smem_desc(smem_u32(sQ), 16, C::ATOM, C::SWZ);
  st.kdesc0 = make_smem_desc(smem_u32(sK), 16, C::ATOM, C::SWZ);
  st.vdesc0 = make_smem_desc(smem_u32(sV), C::KV_CHUNK, C::ATOM, C::SWZ);
  int mt = 0;               // metas read
  int kt = 0;               // key tiles read (K/V ring position)
  int g0 = 0;               // key tiles of this pipeline before the current query tile
  int pdone = 0;            // PVs of this pipeline known complete
  bool ok = true;
  int item_local = 0;
  PendRing pend{0, 0, 0, 0, 0, 0};
  for (; ok; ++item_local) {
    {
      const int ms = mt & (kMetaRing - 1);
      if (!(ok = wait_bar(&bars.m_full[ms], (uint32_t)(mt / kMetaRing) & 1u, abort_flag))) break;
      const Meta hm = load_meta(&meta[ms]);
      mbar_arrive(&bars.m_empty[ms]);
      ++mt;
      if (hm.kind == kKindDone) break;
    }
    const int qb = item_local % C::QB;
    if (!(ok = wait_bar(&bars.q_full[qb], (item_local / C::QB) & 1, abort_flag))) break;
    int qi = 0, pi = 0;
    bool end = false;
    bool o_init[2] = {false, false};   // O accumulators written in this query tile
    // Issue QKs while S buffers are free (QK_t needs PV_{t-NS} complete): read the next
    // key tile's meta, wait for its K, QK into S buffer t % NS.
    for (;;) {
      while (ok && !end && g0 + qi < pdone + C::NS) {
        const int ms = mt & (kMetaRing - 1);
        if (!(ok = wait_bar(&bars.m_full[ms], (uint32_t)(mt / kMetaRing) & 1u, abort_flag))) break;
        const Meta m = load_meta(&meta[ms]);
        mbar_arrive(&bars.m_empty[ms]);
        ++mt;
        if (m.kind != kKindTile) {
          end = true;
          break;
        }
        const int stage = kt % C::STAGES;
        const uint32_t ph = (uint32_t)(kt / C::STAGES) & 1u;
        ++kt;
        const int t = g0 + qi;
        const int buf = t % C::NS;
        if (!(ok = wait_bar(&bars.k_full[stage], ph, abort_flag))) break;
        tc_fence_after();
        issue_qk<D>(st, x, qb, buf, stage, m.nch * 32);
        mma_commit(&bars.s_full[buf]);
        mma_commit(&bars.k_empty[stage]);
        pend.put(buf, stage, m.nch * 32);
        ++qi;
      }
      if (!ok || pi == qi) break;
      // PV of the oldest pending key tile
      const int g = g0 + pi;
      const int buf = g % C::NS;
      int stage, nkeys;
      pend.get(buf, stage, nkeys);
      // the softmax has read S_j and written P_j
      if (!(ok = wait_bar(&bars.p_full[buf], (uint32_t)(g / C::NS) & 1u, abort_flag))) break;
      if (pi == 0 && item_local > 0) {
        // the previous query tile's epilogue has read O
        if (!(ok = wait_bar(&bars.o_empty, (uint32_t)(item_local - 1) & 1u, abort_flag))) break;
      }
      // V of this key tile: its ring lap is the one its K had
      const int vkt = kt - (qi - pi);
      if (!(ok = wait_bar(&bars.v_full[stage], (uint32_t)(vkt / C::STAGES) & 1u, abort_flag))) break;
      tc_fence_after();
      issue_pv<D>(st, x, buf, stage, nkeys, o_init);
      mma_commit(&bars.pv_done[g & 1]);
      mma_commit(&bars.v_empty[stage]);
      ++pi;
      // PV_{g+2-NS} completes (in order) before QK_{g+2} takes its S buffer: with two
      // buffers that is PV_g itself, with three PV_{g-1}, which had a whole key tile to
      // finish while PV_g waits in the queue.
      const int j = g + 2 - C::NS;
      if (j >= pdone) {
        if (!(ok = wait_bar(&bars.pv_done[j & 1], (uint32_t)(j >> 1) & 1u, abort_flag))) break;
        pdone = j + 1;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&bars.pv_count) = pdone;
      }
    }
    if (!ok) break;
    // the last PVs of the query tile: their completion releases the softmax epilogue
    while (pdone < g0 + pi) {
      const int j = pdone;
      if (!(ok = wait_bar(&bars.pv_done[j & 1], (uint32_t)(j >> 1) & 1u, abort_flag))) break;
      pdone = j + 1;
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&bars.pv_count) = pdone;
    }
    if (!ok) break;
    mma_commit(&bars.q_empty[qb]);   // all QKs of this query tile issued; arrives when they are done
    g0 += qi;
  }
  // Make sure no MMA of this thread is still writing TMEM when the CTA frees it.
  mma_commit(&bars.drain);
  drain_bar(&bars.drain, 0);
}

// ------------------------------------------------------------------ softmax + epilogue (warps 2-9)

// Visibility of one 32-key chunk (first key token `tok`, membership bits `mask`) for the
// 32 rows of a warp: `cls` is warp-uniform (0: no row sees a key, 1: every row sees every
// key, 2: causal diagonal, per-row mask `kp`). `q_warp` is the query token of lane 0.
__device__ __forceinline__ int chunk_class(const Params& p, int present, int tok, int mask, int sub, int q_warp,
                                          int lane, uint32_t& kp) {
  kp = 0u;
  if (!present || !((mask >> sub) & 1)) return 0;
  kp = 0xffffffffu;
  if (!p.causal) return 1;
  const int lim0 = q_warp - tok;                    // row r sees columns c <= lim0 + r
  if (lim0 >= 31) return 1;
  if (lim0 + 31 < 0) {
    kp = 0u;
    return 0;
  }
  const int lim = lim0 + lane;
  kp = lim >= 31 ? 0xffffffffu : (lim < 0 ? 0u : ((2u << lim) - 1u));
  return 2;
}

// Max of the visible entries of a 32-column chunk (raw scores; -inf if none). `full` is
// warp-uniform: every lane of the warp sees the whole chunk.
__device__ __forceinline__ float chunk_max(const uint32_t* v, uint32_t kp, bool full) {
  const float kNegInf = __int_as_float(0xff800000);
  float acc[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
  if (full) {
#pragma unroll
    for (int j = 0; j < 32; j += 2)
      acc[(j >> 1) & 3] = max3(acc[(j >> 1) & 3], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j & 3] = fmaxf(acc[j & 3], ((kp >> j) & 1u) ? __uint_as_float(v[j]) : kNegInf);
  }
  return fmaxf(max3(acc[0], acc[1], acc[2]), acc[3]);
}

// p = 2^(s c - m) of one chunk into packed bf16 (hidden columns give exactly 0); adds the
// row sum into rsa. The mask test is hoisted out of the loop (`full` is warp-uniform).
template <bool FULL>
__device__ __forceinline__ void chunk_exp_t(const uint32_t* v, uint32_t kp, uint64_t c2, uint64_t negm2, uint32_t* pk,
                                            uint64_t* rsa) {
  const float kNegInf = __int_as_float(0xff800000);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), c2, negm2), x0, x1);
    if (!FULL) {
      x0 = ((kp >> j) & 1u) ? x0 : kNegInf;
      x1 = ((kp >> (j + 1)) & 1u) ? x1 : kNegInf;
    }
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    rsa[(j >> 1) & 3] = f2_add(rsa[(j >> 1) & 3], f2_pack(p0, p1));
    pk[j >> 1] = pack_bf16x2(p0, p1);
  }
}
__device__ __forceinline__ void chunk_exp(const uint32_t* v, uint32_t kp, bool full, uint64_t c2, uint64_t negm2,
                                          uint32_t* pk, uint64_t* rsa) {
  if (full) chunk_exp_t<true>(v, kp, c2, negm2, pk, rsa);
  else chunk_exp_t<false>(v, kp, c2, negm2, pk, rsa);
}

// Rare path of the online max: O *= alpha for this thread's row (O quiescent).
template <int NC>
__device__ __noinline__ void rescale_o(uint32_t tO, float alpha) {
  const uint64_t al2 = f2_pack(alpha, alpha);
  constexpr int W = NC < 32 ? NC : 32;
#pragma unroll 1
  for (int ch = 0; ch < NC / W; ++ch) {
    uint32_t ov[32];
    if (W == 32) {
      tmem_ld_x32(tO + ch * 32, ov);
      tmem_ld_wait<32>(ov);
    } else {
      tmem_ld_x16(tO, ov);
      tmem_ld_wait<16>(ov);
    }
#pragma unroll
    for (int j = 0; j < W; j += 2) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(ov[j]), __uint_as_float(ov[j + 1])), al2), lo, hi);
      ov[j] = __float_as_uint(lo);
      ov[j + 1] = __float_as_uint(hi);
    }
    if (W == 32) tmem_st_x32(tO + ch * 32, ov);
    else tmem_st_x16(tO, ov);
  }
  tmem_st_wait();
}

// Row-max / row-sum exchange between the two warps that share a TMEM lane quarter.
struct Exchange {
  float v[2][2][2][kTile];   // [pipeline][tile parity][chunk][row]
};

__device__ __forceinline__ void pair_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

// Softmax and epilogue of pipeline x. Warp (quarter q, chunk h) handles rows 32q..32q+31
// and key columns 32h..32h+31 of every 64-key tile.
//   d = 32 (split O): the chunk half has its own running max, row sum and accumulator
//     O_h, so the two warps of a quarter work independently; their partial results are
//     merged once per query tile in the epilogue.
//   d >= 64: one O; the pair agrees on each tile's row max through `xc` (named barrier
//     1 + 4x + q) and each warp rescales its half of the O columns.
template <int D>
__device__ void softmax_epilogue(const Params& p, int x, int h, PipeBars& bars, Meta* meta, Exchange& xc,
                                 uint32_t tmem, volatile int* abort_flag) {
  using C = Cfg<D>;
  constexpr int DH = D / 2;                          // output columns this warp stores
  constexpr int RC = C::SPLIT ? D : DH;              // O columns this warp rescales
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;                      // TMEM lanes this warp may access
  const int row = quarter * 32 + lane;               // query row within the tile
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const int sub = row >> p.log2b;                    // query block within the tile (warp-uniform)
  const int bar_id = 1 + 4 * x + quarter;
  const float kNegInf = __int_as_float(0xff800000);
  const float c = p.scale_log2;
  const uint64_t c2 = f2_pack(c, c);
  // the accumulator columns this warp rescales: all of O_h (split) or its half of O
  const uint32_t tR = tmem + (C::SPLIT ? C::col_o(x, h) : C::col_o(x, 0) + (uint32_t)(DH * h)) + lane_base;

  int mt = 0, g = 0;        // meta position, key tiles processed by this pipeline (global)
  int buf = 0;              // g % NS
  uint32_t sph = 0;         // (g / NS) & 1
  bool ok = true;
  int item_local = 0;
  for (; ok; ++item_local) {
    int k;
    {
      const int ms = mt % kMetaRing;
      if (!(ok = wait_bar(&bars.m_full[ms], (mt / kMetaRing) & 1, abort_flag))) break;
      const Meta hm = load_meta(&meta[ms]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.m_empty[ms]);
      ++mt;
      if (hm.kind == kKindDone) break;
      k = hm.tok[0];
    }
    const Item it = decode_item(p, k);
    const int qtok = it.tile * kTile + row;
    const int q_warp = it.tile * kTile + quarter * 32;
    float m_use = kNegInf;   // running reference max, log2 units
    float l = 0.f;           // row sum over this warp's chunks
    int n_item = 0;
    for (;;) {
      const int ms = mt % kMetaRing;
      if (!(ok = wait_bar(&bars.m_full[ms], (mt / kMetaRing) & 1, abort_flag))) break;
      const Meta m = load_meta(&meta[ms]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.m_empty[ms]);
      ++mt;
      if (m.kind != kKindTile) break;

      // this warp's chunk of the tile (selects, not an indexed read: keeps Meta in registers)
      uint32_t kp;
      const int cls = chunk_class(p, h < m.nch, h ? m.tok[1] : m.tok[0], h ? m.mask[1] : m.mask[0], sub, q_warp,
                                  lane, kp);
      const bool u = cls != 0, f = cls == 1;
      const uint32_t tS = tmem + C::col_s(x, buf) + lane_base;
      ok = __all_sync(0xffffffffu, wait_bar(&bars.s_full[buf], sph, abort_flag));
      if (!ok) break;
      tc_fence_after();

      uint32_t va[32];
      float cm = kNegInf;
      if (u) {
        tmem_ld_x32(tS + 32 * h, va);
        tmem_ld_wait<32>(va);
        cm = chunk_max(va, kp, f);
      }
      float mx = cm * c;                             // -inf stays -inf
      if (!C::SPLIT) {
        // tile max of the row over both chunks
        xc.v[x][g & 1][h][row] = cm;
        pair_sync(bar_id);
        mx = fmaxf(cm, xc.v[x][g & 1][h ^ 1][row]) * c;
      }
      const bool need = mx > m_use + 8.0f;
      if (__any_sync(0xffffffffu, need)) {
        // the running max grows: rescale l and, if earlier tiles contributed, O
        const float alpha = need ? ex2_approx(m_use - mx) : 1.f;   // 0 when m_use = -inf
        const bool o_scale = need && m_use != kNegInf;
        if (n_item > 0 && __any_sync(0xffffffffu, o_scale)) {
          // O is quiescent once the PV of the previous key tile has completed. S_g exists,
          // so PV_{g-NS} and every PV before it have completed (QK_g waited for it): the
          // parity wait on PV_{g-1}'s barrier cannot be two phases off.
          ok = __all_sync(0xffffffffu, wait_bar(&bars.pv_done[(g - 1) & 1], (uint32_t)((g - 1) >> 1) & 1u, abort_flag));
          if (!ok) break;
          tc_fence_after();
          rescale_o<RC>(tR, alpha);
        }
        l *= alpha;
        if (need) m_use = mx;
      }
      uint32_t pk[16];
      if (u) {
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t rsa[4] = {0ull, 0ull, 0ull, 0ull};
        chunk_exp(va, kp, f, c2, negm2, pk, rsa);
        const uint64_t rs2 = f2_add(f2_add(rsa[0], rsa[1]), f2_add(rsa[2], rsa[3]));
        float rs_lo, rs_hi;
        f2_unpack(rs2, rs_lo, rs_hi);
        l += rs_lo + rs_hi;
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
      }
      // P of this chunk (bf16 pairs) over the first 16 columns of the chunk's own S
      // columns 32h..32h+31, which this warp has already read: no other warp's S is touched
      tmem_st_x16(tS + 32 * h, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[buf]);
      ++g;
      ++n_item;
      if (++buf == C::NS) {
        buf = 0;
        sph ^= 1u;
      }
    }
    if (!ok) break;

    // epilogue: O / l and LSE of this query tile (this warp: output columns DH*h .. DH*h + DH)
    float m_fin = m_use, inv = 0.f, a0 = 0.f, a1 = 0.f;
    float lt;
    if (C::SPLIT) {
      xc.v[x][0][h][row] = m_use;
      xc.v[x][1][h][row] = l;
      pair_sync(bar_id);
      const float m0 = xc.v[x][0][0][row], m1 = xc.v[x][0][1][row];
      const float l0 = xc.v[x][1][0][row], l1 = xc.v[x][1][1][row];
      pair_sync(bar_id);                             // both read before the next tile reuses xc
      m_fin = fmaxf(m0, m1);
      a0 = l0 > 0.f ? ex2_approx(m0 - m_fin) : 0.f;
      a1 = l1 > 0.f ? ex2_approx(m1 - m_fin) : 0.f;
      lt = l0 * a0 + l1 * a1;
    } else {
      xc.v[x][g & 1][h][row] = l;
      pair_sync(bar_id);
      lt = l + xc.v[x][g & 1][h ^ 1][row];
    }
    if (n_item > 0) {
      ok = __all_sync(0xffffffffu, wait_count(&bars.pv_count, g, abort_flag));
      if (!ok) break;
      tc_fence_after();
    }
    const bool store = qtok < p.n_tokens;
    inv = lt > 0.f ? 1.f / lt : 0.f;
    __nv_bfloat16* orow =
        p.o + (int64_t)it.s * p.o_sb + (int64_t)qtok * p.o_sn + (int64_t)it.h * p.o_sh + DH * h;
#pragma unroll 1
    for (int ch = 0; ch < DH / 16; ++ch) {            // 16 output columns at a time
      uint32_t ov[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) ov[j] = 0u;
      if (n_item > 0) {
#pragma unroll
        for (int part = 0; part < C::NO; ++part) {
          // split: weight each part by its max correction (a part with no visible key,
          // whose accumulator may never have been written, contributes nothing)
          const float wt = C::SPLIT ? (part ? a1 : a0) : 1.f;
          uint32_t w[16];
          tmem_ld_x16(tmem + C::col_o(x, part) + (uint32_t)(DH * h + ch * 16) + lane_base, w);
          tmem_ld_wait<16>(w);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            ov[j] = __float_as_uint(__uint_as_float(ov[j]) + (wt != 0.f ? __uint_as_float(w[j]) * wt : 0.f));
        }
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
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.o_empty);
    if (store && h == 0) {
      const float lse = lt > 0.f ? (m_fin + __log2f(lt)) * 0.69314718055994531f : kNegInf;
      p.lse[((int64_t)it.s * p.heads + it.h) * p.n_tokens + qtok] = lse;
    }
  }
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ PipeBars bars[2];
  __shared__ Meta meta[2][kMetaRing];
  __shared__ Exchange xchg;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      PipeBars& b = bars[x];
      for (int i = 0; i < 2; ++i) {
        mbar_init(&b.q_full[i], 1);
        mbar_init(&b.q_empty[i], 1);
      }
      for (int i = 0; i < C::STAGES; ++i) {
        mbar_init(&b.k_full[i], 1);
        mbar_init(&b.k_empty[i], 1);
        mbar_init(&b.v_full[i], 1);
        mbar_init(&b.v_empty[i], 1);
      }
      for (int i = 0; i < kMetaRing; ++i) {
        mbar_init(&b.m_full[i], 1);
        mbar_init(&b.m_empty[i], kMetaConsumers);
      }
      for (int i = 0; i < C::NS; ++i) {
        mbar_init(&b.s_full[i], 1);
        mbar_init(&b.p_full[i], kSoftmaxWarps);
      }
      mbar_init(&b.pv_done[0], 1);
      mbar_init(&b.pv_done[1], 1);
      mbar_init(&b.o_empty, kSoftmaxWarps);
      mbar_init(&b.drain, 1);
      b.pv_count = 0;
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

  // pipeline 0: warps 0 (producer), 1 (MMA), 2-9 (softmax); pipeline 1: warps 19, 18, 10-17
  const int x = (warp <= 9) ? 0 : 1;
  uint8_t* sQ = sbase + x * C::PIPE_BYTES;
  uint8_t* sK = sQ + C::QB * C::Q_BYTES;
  uint8_t* sV = sK + C::STAGES * C::KV_BYTES;
  UnionSmem& un = *reinterpret_cast<UnionSmem*>(sV + C::STAGES * C::KV_BYTES);

  if (warp == 0 || warp == 19) {
    producer<D>(p, x, &tq, &tk, &tv, bars[x], meta[x], un, sQ, sK, sV, &abort_flag);
  } else if (warp == 1 || warp == 18) {
    if ((threadIdx.x & 31) == 0) mma_issuer<D>(p, x, bars[x], meta[x], sQ, sK, sV, tmem, &abort_flag);
    __syncwarp();
  } else {
    // softmax warps 2 + 8x .. 9 + 8x: chunk h = 0 for the first four, 1 for the others
    const int h = ((warp - 2 - 8 * x) >> 2) & 1;
    softmax_epilogue<D>(p, x, h, bars[x], meta[x], xchg, tmem, &abort_flag);
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
  p.lse = a.lse;
  p.o_sb = a.o_strides[0];
  p.o_sn = a.o_strides[1];
  p.o_sh = a.o_strides[2];
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  // a work counter of its own for this launch: slot (ticket mod kWorkSlots), zeroed on the
  // launch's stream first (the slots' address differs per device: looked up on every call)
  unsigned int* counters = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&counters), g_work_counters) != cudaSuccess) return SA_ERR_CUDA;
  static std::atomic<unsigned int> ticket{0};
  p.work_counter = counters + (ticket.fetch_add(1u) % kWorkSlots);
  if (cudaMemsetAsync(p.work_counter, 0, sizeof(unsigned int), stream) != cudaSuccess) return SA_ERR_CUDA;
  const int sm_count = current_sm_count();
  auto kern = attn_fwd_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return SA_ERR_CUDA;
  const int want = (p.n_items + 1) / 2;
  const int grid = want < sm_count ? want : sm_count;
  kern<<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace

int launch_attn_fwd(const AttnArgs& a, cudaStream_t stream) {
  switch (a.head_dim) {
    case 32:
    case 64:
    case 128: return launch_attn_fwd_wide(a, stream);
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
