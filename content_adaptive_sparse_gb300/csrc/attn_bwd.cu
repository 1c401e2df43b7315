// Block-sparse attention backward for sm_103a (tcgen05 + TMEM + TMA).
//
// Gradients of L = sum(dO * O) for the forward of attn_fwd.cu, over the same token rule
// (key j of block J is visible to query i of block I iff J is in row(I) and, if causal,
// j <= i). With P_ij = exp(s_ij - LSE_i) and D_i = sum_d dO_id O_id (= sum_j P_ij dP_ij):
//   dP_ij = <dO_i, v_j>,  dS_ij = P_ij (dP_ij - D_i),
//   dQ_i = c sum_j dS_ij k_j,  dK_j = c sum_i dS_ij q_i,  dV_j = sum_i P_ij dO_i.
// Six launches:
//   bwd_dvec_kernel    D_i from O and dO (bandwidth bound).
//   csc_pass (count), csc_scan, csc_pass (fill)   the transposed CSR: for each key block J,
//                      the query blocks whose rows hold J (ascending; I >= J under
//                      causality).
//   bwd_dq_kernel      query-stationary: per 128-query tile, for each 64-key step of the
//                      union of its CSR rows: S = Q K^T, dP = dO V^T (tcgen05, SS), dS in
//                      the compute warps, dQ += dS K (tcgen05, A = dS from TMEM).
//   bwd_dkdv_kernel    key-stationary: per 128-key tile of a key/value head, for each query
//                      head of its group and each 64-query step of the union of its CSC
//                      rows: S^T = K Q^T, dP^T = V dO^T (SS), P^T and dS^T in the compute
//                      warps, dV += P^T dO and dK += dS^T Q (A from TMEM).
// Splitting dQ from dK / dV recomputes S and dP once more but needs no atomics: every
// gradient row is owned by exactly one work item, so the result is deterministic.
//
// Warp roles of both attention kernels (320 threads, one work item per CTA):
//   warp 0      producer: stationary tiles by TMA, the union of CSR / CSC rows, moving
//               tiles (and, for dK / dV, the step's LSE and D) into a ring of stages.
//   warp 1      owns TMEM; lane 0 issues the MMAs.
//   warps 2-9   compute: warp w reads TMEM lane quarter w % 4 (one stationary row per
//               thread) and 32-column chunk (w - 2) / 4 of each 64-row step.
// TMEM columns: S [0, 64), dP [64, 128), accumulators from 128 (dQ; or dV then dK).
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

__device__ unsigned int g_bwd_err;

constexpr int kRows = 128;            // stationary rows per work item
constexpr int kStep = 64;             // moving rows per step (two 32-row chunks)
constexpr int kThreads = 320;
constexpr int kComputeWarps = 8;
constexpr int kMetaRing = 8;
constexpr int kMetaConsumers = 1 + kComputeWarps;
constexpr int kMaxStages = 4;
constexpr uint32_t kColS = 0, kColP = 64, kColAcc = 128;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BCfg {
  static constexpr int CH = D >= 64 ? 64 : 32;         // elements per swizzled row
  static constexpr int NCH = D / CH;
  static constexpr int ROWB = CH * 2;
  static constexpr uint32_t SWZ = ROWB == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr CUtensorMapSwizzle TMA_SWZ =
      ROWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  static constexpr uint32_t ATOM = 8 * ROWB;
  static constexpr int BIG_CHUNK = kRows * ROWB;       // one d-chunk of a 128-row tile
  static constexpr int BIG_BYTES = NCH * BIG_CHUNK;
  static constexpr int STEP_CHUNK = kStep * ROWB;      // one d-chunk of a 64-row tile
  static constexpr int STEP_BYTES = NCH * STEP_CHUNK;
  static constexpr int STAGES = D == 128 ? 2 : 3;
  // stage: two 64-row tiles (+ 2 x 64 floats for dK / dV), 1 KB aligned for the swizzle
  static constexpr int STAGE_BYTES = (2 * STEP_BYTES + 512 + 1023) & ~1023;
  static constexpr int UNION_BYTES = (int)sizeof(UnionSmem);
  static constexpr int SMEM_NEED = 1024 + 2 * BIG_BYTES + STAGES * STAGE_BYTES + UNION_BYTES;
  // at least 80 KB: at most two CTAs per SM, whose TMEM (256 columns each) then always fits
  static constexpr int SMEM = SMEM_NEED > 80 * 1024 ? SMEM_NEED : 80 * 1024;
  static constexpr uint32_t TMEM_DQ = 256;
  static constexpr uint32_t TMEM_DKDV = 128 + 2 * D <= 256 ? 256 : 512;
  // Occupancy: at d <= 64 two CTAs share an SM (256 TMEM columns each). At d = 128 the dK/dV
  // kernel takes all 512 columns, and its shared memory alone already keeps a second CTA off
  // the SM, so no CTA ever waits in tcgen05.alloc for another one's columns.
  static_assert(TMEM_DKDV == 256 || 2 * SMEM > 227 * 1024, "a 512-column CTA must have the SM to itself");
  static_assert(STAGES <= kMaxStages, "ring size");
};

enum : int { kKindStep = 0, kKindEnd = 1 };

struct Meta {
  int kind;
  int nch;         // 32-row chunks in this step (1 or 2)
  int tok[2];      // first moving token of each chunk
  int mask[2];     // bit r: stationary block r of the tile meets the chunk's block
  int head;        // query head of the step (dK / dV)
};

__device__ __forceinline__ Meta load_meta(const Meta* src) {
  const volatile Meta* vm = src;
  Meta m;
  m.kind = vm->kind;
  m.nch = vm->nch;
  m.tok[0] = vm->tok[0];
  m.tok[1] = vm->tok[1];
  m.mask[0] = vm->mask[0];
  m.mask[1] = vm->mask[1];
  m.head = vm->head;
  return m;
}

struct BParams {
  int batch, n_tokens, heads, heads_per_kv, kv_heads, block, log2b, nb, causal, csr_shared;
  int tiles;                        // 128-row tiles per sequence
  int n_items;
  int n_masks;                      // head groups: query head h uses CSR head_mask[h]
  const int32_t* rp[kMaxMasks];     // CSR (dQ) or transposed CSR (dK / dV) row pointers
  const int32_t* ci[kMaxMasks];     // CSR column / transposed CSR row indices
  uint8_t head_mask[kMaxHeadMap];
  const float* lse;                 // [batch][heads][n_tokens]
  const float* dvec;                // D, same layout
  __nv_bfloat16* out0;              // dQ, or dK
  __nv_bfloat16* out1;              // dV
  int64_t os_b, os_n, os_h;         // strides of out0 / out1
  float scale;                      // softmax scale c
  float scale_log2;                 // c log2(e)
};

struct Bars {
  uint64_t fixed_full;                                   // stationary tiles landed
  uint64_t st_full[kMaxStages], st_empty[kMaxStages];
  uint64_t m_full[kMetaRing], m_empty[kMetaRing];
  uint64_t s_full, p_full, ds_used, acc_full, drain;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait(bar, parity, abort_flag, &g_bwd_err, kErrTimeout);
}
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  int never = 0;
  mbar_wait(bar, parity, &never, &g_bwd_err, kErrTimeout);
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
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Work item k, longest first. dQ: query tiles, causal ranks from the last tile. dK / dV:
// key tiles from the first (the first key blocks are seen by the most query blocks).
struct Item {
  int s, h, tile;
};
__device__ __forceinline__ Item decode_item(const BParams& p, int k, int nh, bool reverse) {
  const int bh = k % (p.batch * nh);
  const int rank = k / (p.batch * nh);
  Item it;
  it.h = bh % nh;
  it.s = bh / nh;
  it.tile = reverse ? (p.tiles - 1 - rank) : rank;
  return it;
}

// Byte offset (>> 4) of k-step ks in a K-major tile whose d-chunks are `chunk` bytes apart.
template <int D>
__device__ __forceinline__ constexpr uint32_t kstep(int ks, int chunk) {
  using C = BCfg<D>;
  return (uint32_t)(((ks * 16) / C::CH) * chunk + ((ks * 16) % C::CH) * 2) >> 4;
}

// D[tmem] (+)= A[128 x d, K-major] * B[n x d, K-major]^T over the head dimension.
template <int D>
__device__ __forceinline__ void mma_rows_x_rows(uint32_t d_tmem, uint64_t a0, uint64_t b0, int n) {
  using C = BCfg<D>;
  const uint32_t idesc = make_idesc_bf16(128, (uint32_t)n, 0, 0);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
    mma_bf16_ss(d_tmem, a0 + kstep<D>(ks, C::BIG_CHUNK), b0 + kstep<D>(ks, C::STEP_CHUNK), idesc, ks > 0 ? 1u : 0u);
}

// D[tmem] (+)= A[128 x n] (bf16 pairs in TMEM, chunk h of 32 columns at 32h .. 32h+15)
// * B[n x d] (the moving tile read MN-major).
template <int D>
__device__ __forceinline__ void mma_tmem_x_tile(uint32_t d_tmem, uint32_t a, uint64_t bmn0, int n, bool acc) {
  using C = BCfg<D>;
  const uint32_t idesc = make_idesc_bf16(128, D, 0, 1);
  mma_bf16_ts(d_tmem, a, bmn0, idesc, acc ? 1u : 0u);
  mma_bf16_ts(d_tmem, a + 8u, bmn0 + (uint64_t)((16 * C::ROWB) >> 4), idesc, 1u);
  if (n > 32) {
    mma_bf16_ts(d_tmem, a + 32u, bmn0 + (uint64_t)((32 * C::ROWB) >> 4), idesc, 1u);
    mma_bf16_ts(d_tmem, a + 40u, bmn0 + (uint64_t)((48 * C::ROWB) >> 4), idesc, 1u);
  }
}

// ------------------------------------------------------------------ shared producer pieces

// Meta of the step whose first chunk is c0 of the union list (cpb chunks per block).
__device__ __forceinline__ Meta step_meta(const UnionSmem& u, int c0, int n_chunks, int cpb, int b, int head) {
  Meta m;
  m.kind = c0 < n_chunks ? kKindStep : kKindEnd;
  m.nch = min(2, n_chunks - c0);
  m.head = head;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int q = c0 + i;
    const uint32_t e = (m.kind == kKindStep && i < m.nch) ? u.list[q / cpb] : 0u;
    m.tok[i] = (int)(e & 0xfffu) * b + (q % cpb) * 32;
    m.mask[i] = (m.kind == kKindStep && i < m.nch) ? (int)(e >> 12) : 0;
  }
  return m;
}

// TMA of the moving rows of one step (b = 32: one 32-row box per chunk; b >= 64: the two
// chunks are one 64-row box) for both moving tensors of the stage.
template <int D>
__device__ __forceinline__ void load_step_tiles(uint8_t* stage, const CUtensorMap* t0, const CUtensorMap* t1,
                                                uint64_t* bar, const Meta& m, int b, int head, int s) {
  using C = BCfg<D>;
  const int nbox = b == 32 ? m.nch : 1;
  for (int i = 0; i < nbox; ++i)
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
      tma_load_4d(stage + c * C::STEP_CHUNK + i * 32 * C::ROWB, t0, bar, c * C::CH, head, m.tok[i], s);
      tma_load_4d(stage + C::STEP_BYTES + c * C::STEP_CHUNK + i * 32 * C::ROWB, t1, bar, c * C::CH, head, m.tok[i],
                  s);
    }
}

// ------------------------------------------------------------------ dQ kernel

template <int D>
__device__ void dq_producer(const BParams& p, const Item& it, const CUtensorMap* tq, const CUtensorMap* tdo,
                            const CUtensorMap* tk, const CUtensorMap* tv, Bars& bars, Meta* meta, UnionSmem& u,
                            uint8_t* sFix, uint8_t* sStage, volatile int* abort_flag) {
  using C = BCfg<D>;
  const int lane = threadIdx.x & 31;
  const int b = p.block;
  const int cpb = b >> 5;
  const int q0 = it.tile * kRows;
  const int I0 = q0 >> p.log2b;
  const int nq = min(kRows >> p.log2b, p.nb - I0);
  const int hk = it.h / p.heads_per_kv;
  if (lane == 0) {
    mbar_arrive_expect_tx(&bars.fixed_full, 2 * C::BIG_BYTES);
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
      tma_load_4d(sFix + c * C::BIG_CHUNK, tq, &bars.fixed_full, c * C::CH, it.h, q0, it.s);
      tma_load_4d(sFix + C::BIG_BYTES + c * C::BIG_CHUNK, tdo, &bars.fixed_full, c * C::CH, it.h, q0, it.s);
    }
  }
  const int mi = p.n_masks > 1 ? p.head_mask[it.h] : 0;
  const int32_t* rp = p.rp[mi] + (size_t)(p.csr_shared ? 0 : it.s) * (p.nb + 1);
  const int n_keys =
      build_union(p.nb, p.causal ? kKeepLE : kKeepAll, u, rp, p.ci[mi], I0, nq, &g_bwd_err, kErrBadIndex);
  const int n_chunks = n_keys * cpb;
  int kt = 0;
  bool ok = true;
  for (int c0 = 0, mt = 0;; c0 += 2, ++mt) {
    const Meta m = step_meta(u, c0, n_chunks, cpb, b, it.h);
    if (lane == 0) {
      const int ms = mt % kMetaRing;
      ok = wait_bar(&bars.m_empty[ms], ((mt / kMetaRing) & 1) ^ 1, abort_flag);
      if (ok) {
        meta[ms] = m;
        mbar_arrive(&bars.m_full[ms]);
      }
      if (ok && m.kind == kKindStep) {
        const int st = kt % C::STAGES;
        ok = wait_bar(&bars.st_empty[st], ((kt / C::STAGES) & 1) ^ 1, abort_flag);
        if (ok) {
          mbar_arrive_expect_tx(&bars.st_full[st], (uint32_t)(2 * m.nch * 32 * D * 2));
          load_step_tiles<D>(sStage + st * C::STAGE_BYTES, tk, tv, &bars.st_full[st], m, b, hk, it.s);
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (m.kind == kKindStep) ++kt;
    if (!ok || m.kind == kKindEnd) break;
  }
  // every copy of this CTA has landed before it may exit
  if (lane == 0) {
    drain_bar(&bars.fixed_full, 0);
    for (int t = max(0, kt - C::STAGES); t < kt; ++t) drain_bar(&bars.st_full[t % C::STAGES], (t / C::STAGES) & 1);
  }
  __syncwarp();
}

template <int D>
__device__ void dq_mma(Bars& bars, Meta* meta, uint8_t* sFix, uint8_t* sStage, uint32_t tmem,
                       volatile int* abort_flag) {
  using C = BCfg<D>;
  const uint64_t qdesc = make_smem_desc(smem_u32(sFix), 16, C::ATOM, C::SWZ);
  const uint64_t dodesc = make_smem_desc(smem_u32(sFix + C::BIG_BYTES), 16, C::ATOM, C::SWZ);
  const uint64_t kdesc0 = make_smem_desc(smem_u32(sStage), 16, C::ATOM, C::SWZ);
  const uint64_t vdesc0 = make_smem_desc(smem_u32(sStage + C::STEP_BYTES), 16, C::ATOM, C::SWZ);
  const uint64_t kmn0 = make_smem_desc(smem_u32(sStage), C::STEP_CHUNK, C::ATOM, C::SWZ);
  bool ok = wait_bar(&bars.fixed_full, 0, abort_flag);
  int t = 0;
  for (int mt = 0; ok; ++mt) {
    const int ms = mt % kMetaRing;
    if (!(ok = wait_bar(&bars.m_full[ms], (mt / kMetaRing) & 1, abort_flag))) break;
    const Meta m = load_meta(&meta[ms]);
    mbar_arrive(&bars.m_empty[ms]);
    if (m.kind != kKindStep) break;
    const int st = t % C::STAGES;
    if (!(ok = wait_bar(&bars.st_full[st], (t / C::STAGES) & 1, abort_flag))) break;
    // S and dP are single-buffered: the previous step's dQ MMA has read dS
    if (t > 0 && !(ok = wait_bar(&bars.ds_used, (t - 1) & 1, abort_flag))) break;
    tc_fence_after();
    const uint64_t so = (uint64_t)((st * C::STAGE_BYTES) >> 4);
    const int n = m.nch * 32;
    mma_rows_x_rows<D>(tmem + kColS, qdesc, kdesc0 + so, n);
    mma_rows_x_rows<D>(tmem + kColP, dodesc, vdesc0 + so, n);
    mma_commit(&bars.s_full);
    if (!(ok = wait_bar(&bars.p_full, t & 1, abort_flag))) break;
    tc_fence_after();
    mma_tmem_x_tile<D>(tmem + kColAcc, tmem + kColS, kmn0 + so, n, t > 0);
    mma_commit(&bars.st_empty[st]);
    mma_commit(&bars.ds_used);
    ++t;
  }
  // arrives once every MMA issued above is complete (at once if there was none)
  mma_commit(&bars.acc_full);
  mma_commit(&bars.drain);
  drain_bar(&bars.drain, 0);
}

// Visibility of one 32-key chunk for the 32 query rows of a warp (warp-uniform class:
// 0 none, 1 all, 2 causal diagonal with per-row mask kp); q_warp = query token of lane 0.
__device__ __forceinline__ int chunk_class(int causal, int present, int tok, int mask, int sub, int q_warp, int lane,
                                          uint32_t& kp) {
  kp = 0u;
  if (!present || !((mask >> sub) & 1)) return 0;
  kp = 0xffffffffu;
  if (!causal) return 1;
  const int lim0 = q_warp - tok;
  if (lim0 >= 31) return 1;
  if (lim0 + 31 < 0) {
    kp = 0u;
    return 0;
  }
  const int lim = lim0 + lane;
  kp = lim >= 31 ? 0xffffffffu : (lim < 0 ? 0u : ((2u << lim) - 1u));
  return 2;
}

template <int D>
__device__ void dq_compute(const BParams& p, const Item& it, int h, Bars& bars, Meta* meta, uint32_t tmem,
                           volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const int qtok = it.tile * kRows + row;
  const int q_warp = it.tile * kRows + quarter * 32;
  const int sub = row >> p.log2b;
  const bool valid = qtok < p.n_tokens;
  const float kNegInf = __int_as_float(0xff800000);
  const int64_t vi = ((int64_t)it.s * p.heads + it.h) * p.n_tokens + qtok;
  const float lse = valid ? p.lse[vi] : kNegInf;
  const float dval = valid ? p.dvec[vi] : 0.f;
  // x = s c log2(e) - LSE log2(e); a row without keys (LSE = -inf) gets p = 0
  const float nl2 = lse == kNegInf ? kNegInf : -lse * kLog2e;
  const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
  const uint64_t nl22 = f2_pack(nl2, nl2);
  const uint64_t negd2 = f2_pack(-dval, -dval);
  const uint32_t tS = tmem + kColS + 32u * h + lane_base;
  const uint32_t tP = tmem + kColP + 32u * h + lane_base;
  bool ok = true;
  int t = 0;
  for (int mt = 0;; ++mt) {
    const int ms = mt % kMetaRing;
    if (!(ok = wait_bar(&bars.m_full[ms], (mt / kMetaRing) & 1, abort_flag))) break;
    const Meta m = load_meta(&meta[ms]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.m_empty[ms]);
    if (m.kind != kKindStep) break;
    uint32_t kp;
    const int cls = chunk_class(p.causal, h < m.nch, h ? m.tok[1] : m.tok[0], h ? m.mask[1] : m.mask[0], sub,
                                q_warp, lane, kp);
    ok = __all_sync(0xffffffffu, wait_bar(&bars.s_full, t & 1, abort_flag));
    if (!ok) break;
    tc_fence_after();
    if (cls != 0) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[16], dv[16], pk[8];
        tmem_ld_x16(tS + 16 * half, sv);
        tmem_ld_x16(tP + 16 * half, dv);
        tmem_ld_wait<16>(sv);
        tmem_ld_wait<16>(dv);
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])), c2, nl22), x0, x1);
          const int cj = 16 * half + j;
          if (cls == 2) {
            x0 = ((kp >> cj) & 1u) ? x0 : kNegInf;
            x1 = ((kp >> (cj + 1)) & 1u) ? x1 : kNegInf;
          }
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          float d0, d1;
          f2_unpack(f2_mul(f2_pack(p0, p1), f2_add(f2_pack(__uint_as_float(dv[j]), __uint_as_float(dv[j + 1])), negd2)),
                    d0, d1);
          pk[j >> 1] = pack_bf16x2(d0, d1);
        }
        // dS (bf16 pairs) of this half over columns 8 half .. 8 half + 7 of the warp's own
        // S chunk (already read; the S columns of half 1 are not among them)
        tmem_st_x8(tS + 8 * half, pk);
      }
    } else {
      uint32_t z[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) z[j] = 0u;
      tmem_st_x16(tS, z);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.p_full);
    ++t;
  }
  if (!ok) return;
  ok = __all_sync(0xffffffffu, wait_bar(&bars.acc_full, 0, abort_flag));
  if (!ok) return;
  tc_fence_after();
  constexpr int DH = D / 2;
  __nv_bfloat16* orow = p.out0 + (int64_t)it.s * p.os_b + (int64_t)qtok * p.os_n + (int64_t)it.h * p.os_h + DH * h;
#pragma unroll 1
  for (int ch = 0; ch < DH / 16; ++ch) {
    uint32_t w[16];
    tmem_ld_x16(tmem + kColAcc + (uint32_t)(DH * h + 16 * ch) + lane_base, w);
    tmem_ld_wait<16>(w);
    if (valid) {
      uint32_t pkd[8];
#pragma unroll
      for (int j = 0; j < 16; j += 2)
        pkd[j >> 1] = t > 0 ? pack_bf16x2(__uint_as_float(w[j]) * p.scale, __uint_as_float(w[j + 1]) * p.scale) : 0u;
      uint4* dst = reinterpret_cast<uint4*>(orow + 16 * ch);
      dst[0] = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
      dst[1] = make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const __grid_constant__ BParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bars;
  __shared__ Meta meta[kMetaRing];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bars.fixed_full, 1);
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&bars.st_full[i], 1);
      mbar_init(&bars.st_empty[i], 1);
    }
    for (int i = 0; i < kMetaRing; ++i) {
      mbar_init(&bars.m_full[i], 1);
      mbar_init(&bars.m_empty[i], kMetaConsumers);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_full, kComputeWarps);
    mbar_init(&bars.ds_used, 1);
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.drain, 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TMEM_DQ);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const Item it = decode_item(p, blockIdx.x, p.heads, p.causal != 0);
  uint8_t* sFix = sbase;
  uint8_t* sStage = sFix + 2 * C::BIG_BYTES;
  UnionSmem& un = *reinterpret_cast<UnionSmem*>(sStage + C::STAGES * C::STAGE_BYTES);
  if (warp == 0) {
    dq_producer<D>(p, it, &tq, &tdo, &tk, &tv, bars, meta, un, sFix, sStage, &abort_flag);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) dq_mma<D>(bars, meta, sFix, sStage, tmem, &abort_flag);
    __syncwarp();
  } else {
    dq_compute<D>(p, it, (warp - 2) >> 2, bars, meta, tmem, &abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_DQ);
  }
}

// ------------------------------------------------------------------ dK / dV kernel

template <int D>
__device__ void dkdv_producer(const BParams& p, const Item& it, const CUtensorMap* tk, const CUtensorMap* tv,
                              const CUtensorMap* tq, const CUtensorMap* tdo, Bars& bars, Meta* meta, UnionSmem& u,
                              uint8_t* sFix, uint8_t* sStage, volatile int* abort_flag) {
  using C = BCfg<D>;
  const int lane = threadIdx.x & 31;
  const int b = p.block;
  const int cpb = b >> 5;
  const int k0 = it.tile * kRows;
  const int J0 = k0 >> p.log2b;
  const int nk = min(kRows >> p.log2b, p.nb - J0);
  if (lane == 0) {
    mbar_arrive_expect_tx(&bars.fixed_full, 2 * C::BIG_BYTES);
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) {
      tma_load_4d(sFix + c * C::BIG_CHUNK, tk, &bars.fixed_full, c * C::CH, it.h, k0, it.s);
      tma_load_4d(sFix + C::BIG_BYTES + c * C::BIG_CHUNK, tv, &bars.fixed_full, c * C::CH, it.h, k0, it.s);
    }
  }
  int cur_mask = -1, n_chunks = 0;
  int kt = 0, mt = 0;
  bool ok = true;
  // every query head of the group, then the end marker; the union of the transposed CSR's
  // rows is rebuilt when the head's CSR differs from the previous head's
  for (int hh = 0; hh <= p.heads_per_kv && ok; ++hh) {
    const int head = it.h * p.heads_per_kv + hh;
    if (hh < p.heads_per_kv) {
      const int mi = p.n_masks > 1 ? p.head_mask[head] : 0;
      if (mi != cur_mask) {
        const int32_t* rp = p.rp[mi] + (size_t)(p.csr_shared ? 0 : it.s) * (p.nb + 1);
        const int n_q =
            build_union(p.nb, p.causal ? kKeepGE : kKeepAll, u, rp, p.ci[mi], J0, nk, &g_bwd_err, kErrBadIndex);
        n_chunks = n_q * cpb;
        cur_mask = mi;
      }
    }
    for (int c0 = (hh < p.heads_per_kv ? 0 : n_chunks);; c0 += 2, ++mt) {
      const Meta m = step_meta(u, c0, n_chunks, cpb, b, head);
      if (m.kind == kKindEnd && hh < p.heads_per_kv) break;   // next head
      if (lane == 0) {
        const int ms = mt % kMetaRing;
        ok = wait_bar(&bars.m_empty[ms], ((mt / kMetaRing) & 1) ^ 1, abort_flag);
        if (ok) {
          meta[ms] = m;
          mbar_arrive(&bars.m_full[ms]);
        }
        if (ok && m.kind == kKindStep) {
          const int st = kt % C::STAGES;
          ok = wait_bar(&bars.st_empty[st], ((kt / C::STAGES) & 1) ^ 1, abort_flag);
          if (ok) {
            uint8_t* stage = sStage + st * C::STAGE_BYTES;
            float* vec = reinterpret_cast<float*>(stage + 2 * C::STEP_BYTES);   // LSE [64], D [64]
            mbar_arrive_expect_tx(&bars.st_full[st], (uint32_t)(2 * m.nch * 32 * D * 2 + 2 * m.nch * 128));
            load_step_tiles<D>(stage, tq, tdo, &bars.st_full[st], m, b, head, it.s);
            const int64_t base = ((int64_t)it.s * p.heads + head) * p.n_tokens;
            for (int i = 0; i < m.nch; ++i) {
              bulk_load(vec + 32 * i, p.lse + base + m.tok[i], 128, &bars.st_full[st]);
              bulk_load(vec + 64 + 32 * i, p.dvec + base + m.tok[i], 128, &bars.st_full[st]);
            }
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (m.kind == kKindStep) ++kt;
      if (!ok || m.kind == kKindEnd) break;
    }
  }
  if (lane == 0) {
    drain_bar(&bars.fixed_full, 0);
    for (int t = max(0, kt - C::STAGES); t < kt; ++t) drain_bar(&bars.st_full[t % C::STAGES], (t / C::STAGES) & 1);
  }
  __syncwarp();
}

template <int D>
__device__ void dkdv_mma(Bars& bars, Meta* meta, uint8_t* sFix, uint8_t* sStage, uint32_t tmem,
                         volatile int* abort_flag) {
  using C = BCfg<D>;
  const uint64_t kdesc = make_smem_desc(smem_u32(sFix), 16, C::ATOM, C::SWZ);
  const uint64_t vdesc = make_smem_desc(smem_u32(sFix + C::BIG_BYTES), 16, C::ATOM, C::SWZ);
  const uint64_t qk0 = make_smem_desc(smem_u32(sStage), 16, C::ATOM, C::SWZ);
  const uint64_t dok0 = make_smem_desc(smem_u32(sStage + C::STEP_BYTES), 16, C::ATOM, C::SWZ);
  const uint64_t qmn0 = make_smem_desc(smem_u32(sStage), C::STEP_CHUNK, C::ATOM, C::SWZ);
  const uint64_t domn0 = make_smem_desc(smem_u32(sStage + C::STEP_BYTES), C::STEP_CHUNK, C::ATOM, C::SWZ);
  const uint32_t col_dv = kColAcc, col_dk = kColAcc + D;
  bool ok = wait_bar(&bars.fixed_full, 0, abort_flag);
  int t = 0;
  for (int mt = 0; ok; ++mt) {
    const int ms = mt % kMetaRing;
    if (!(ok = wait_bar(&bars.m_full[ms], (mt / kMetaRing) & 1, abort_flag))) break;
    const Meta m = load_meta(&meta[ms]);
    mbar_arrive(&bars.m_empty[ms]);
    if (m.kind != kKindStep) break;
    const int st = t % C::STAGES;
    if (!(ok = wait_bar(&bars.st_full[st], (t / C::STAGES) & 1, abort_flag))) break;
    if (t > 0 && !(ok = wait_bar(&bars.ds_used, (t - 1) & 1, abort_flag))) break;
    tc_fence_after();
    const uint64_t so = (uint64_t)((st * C::STAGE_BYTES) >> 4);
    const int n = m.nch * 32;
    mma_rows_x_rows<D>(tmem + kColS, kdesc, qk0 + so, n);    // S^T = K Q^T
    mma_rows_x_rows<D>(tmem + kColP, vdesc, dok0 + so, n);   // dP^T = V dO^T
    mma_commit(&bars.s_full);
    if (!(ok = wait_bar(&bars.p_full, t & 1, abort_flag))) break;
    tc_fence_after();
    mma_tmem_x_tile<D>(tmem + col_dv, tmem + kColS, domn0 + so, n, t > 0);   // dV += P^T dO
    mma_tmem_x_tile<D>(tmem + col_dk, tmem + kColP, qmn0 + so, n, t > 0);    // dK += dS^T Q
    mma_commit(&bars.st_empty[st]);
    mma_commit(&bars.ds_used);
    ++t;
  }
  mma_commit(&bars.acc_full);
  mma_commit(&bars.drain);
  drain_bar(&bars.drain, 0);
}

template <int D>
__device__ void dkdv_compute(const BParams& p, const Item& it, int h, Bars& bars, Meta* meta, uint8_t* sStage,
                             uint32_t tmem, volatile int* abort_flag) {
  using C = BCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const int ktok = it.tile * kRows + row;
  const int jl = row >> p.log2b;                       // key block within the tile
  const bool valid = ktok < p.n_tokens;
  const float kNegInf = __int_as_float(0xff800000);
  const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
  const uint64_t neg_log2e2 = f2_pack(-kLog2e, -kLog2e);
  const uint64_t minus_one2 = f2_pack(-1.f, -1.f);
  const uint32_t tS = tmem + kColS + 32u * h + lane_base;
  const uint32_t tP = tmem + kColP + 32u * h + lane_base;
  bool ok = true;
  int t = 0;
  for (int mt = 0;; ++mt) {
    const int ms = mt % kMetaRing;
    if (!(ok = wait_bar(&bars.m_full[ms], (mt / kMetaRing) & 1, abort_flag))) break;
    const Meta m = load_meta(&meta[ms]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.m_empty[ms]);
    if (m.kind != kKindStep) break;
    const int st = t % C::STAGES;
    // visible query columns of this key row: the block pair is in the graph and, under
    // causality, query token >= key token
    const int tok = h ? m.tok[1] : m.tok[0];
    const bool member = h < m.nch && ((((h ? m.mask[1] : m.mask[0]) >> jl) & 1) != 0);
    uint32_t kp = 0u;
    if (member) {
      const int lim = ktok - tok;                      // first visible column
      kp = (!p.causal || lim <= 0) ? 0xffffffffu : (lim >= 32 ? 0u : (0xffffffffu << lim));
    }
    const bool any = __any_sync(0xffffffffu, kp != 0u);
    const bool full = __all_sync(0xffffffffu, kp == 0xffffffffu);   // no masked column in the warp
    ok = __all_sync(0xffffffffu, wait_bar(&bars.s_full, t & 1, abort_flag));
    if (!ok) break;
    tc_fence_after();
    if (any) {
      // LSE and D of the step's query rows (landed with the stage; this wait is complete)
      ok = __all_sync(0xffffffffu, wait_bar(&bars.st_full[st], (t / C::STAGES) & 1, abort_flag));
      if (!ok) break;
      const float* vec = reinterpret_cast<const float*>(sStage + st * C::STAGE_BYTES + 2 * C::STEP_BYTES);
      const float4* lse4 = reinterpret_cast<const float4*>(vec + 32 * h);
      const float4* d4 = reinterpret_cast<const float4*>(vec + 64 + 32 * h);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[16], dv[16], pp[8], pd[8];
        tmem_ld_x16(tS + 16 * half, sv);
        tmem_ld_x16(tP + 16 * half, dv);
        tmem_ld_wait<16>(sv);
        tmem_ld_wait<16>(dv);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 L = lse4[4 * half + q4];
          const float4 Dq = d4[4 * half + q4];
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int j = 4 * q4 + e;                  // column within this half
            const int cj = 16 * half + j;              // column within the chunk
            // x = s c - LSE log2(e); p = 2^x; dS = p (dP - D), two columns at a time
            const uint64_t nl2 = f2_mul(e ? f2_pack(L.z, L.w) : f2_pack(L.x, L.y), neg_log2e2);
            const uint64_t d2 = e ? f2_pack(Dq.z, Dq.w) : f2_pack(Dq.x, Dq.y);
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[j]), __uint_as_float(sv[j + 1])), c2, nl2), x0, x1);
            if (!full) {
              x0 = ((kp >> cj) & 1u) ? x0 : kNegInf;
              x1 = ((kp >> (cj + 1)) & 1u) ? x1 : kNegInf;
            }
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const uint64_t p2 = f2_pack(p0, p1);
            const uint64_t t2 = f2_fma(d2, minus_one2, f2_pack(__uint_as_float(dv[j]), __uint_as_float(dv[j + 1])));
            float d0, d1;
            f2_unpack(f2_mul(p2, t2), d0, d1);
            pp[j >> 1] = pack_bf16x2(p0, p1);
            pd[j >> 1] = pack_bf16x2(d0, d1);
          }
        }
        // P^T over this warp's S^T chunk, dS^T over its dP^T chunk: the 8 columns of this
        // half (the S / dP columns of half 1 are not among them)
        tmem_st_x8(tS + 8 * half, pp);
        tmem_st_x8(tP + 8 * half, pd);
      }
    } else {
      uint32_t z[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) z[j] = 0u;
      tmem_st_x16(tS, z);
      tmem_st_x16(tP, z);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.p_full);
    ++t;
  }
  if (!ok) return;
  ok = __all_sync(0xffffffffu, wait_bar(&bars.acc_full, 0, abort_flag));
  if (!ok) return;
  tc_fence_after();
  constexpr int DH = D / 2;
  const int64_t roff = (int64_t)it.s * p.os_b + (int64_t)ktok * p.os_n + (int64_t)it.h * p.os_h + DH * h;
#pragma unroll 1
  for (int part = 0; part < 2; ++part) {               // 0: dV, 1: dK (times the scale)
    const float f = part ? p.scale : 1.f;
    __nv_bfloat16* orow = (part ? p.out0 : p.out1) + roff;
#pragma unroll 1
    for (int ch = 0; ch < DH / 16; ++ch) {
      uint32_t w[16];
      tmem_ld_x16(tmem + kColAcc + (uint32_t)(part * D + DH * h + 16 * ch) + lane_base, w);
      tmem_ld_wait<16>(w);
      if (valid) {
        uint32_t pkd[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2)
          pkd[j >> 1] = t > 0 ? pack_bf16x2(__uint_as_float(w[j]) * f, __uint_as_float(w[j + 1]) * f) : 0u;
        uint4* dst = reinterpret_cast<uint4*>(orow + 16 * ch);
        dst[0] = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
        dst[1] = make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ BParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bars;
  __shared__ Meta meta[kMetaRing];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bars.fixed_full, 1);
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&bars.st_full[i], 1);
      mbar_init(&bars.st_empty[i], 1);
    }
    for (int i = 0; i < kMetaRing; ++i) {
      mbar_init(&bars.m_full[i], 1);
      mbar_init(&bars.m_empty[i], kMetaConsumers);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_full, kComputeWarps);
    mbar_init(&bars.ds_used, 1);
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.drain, 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tdo);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TMEM_DKDV);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const Item it = decode_item(p, blockIdx.x, p.kv_heads, false);
  uint8_t* sFix = sbase;
  uint8_t* sStage = sFix + 2 * C::BIG_BYTES;
  UnionSmem& un = *reinterpret_cast<UnionSmem*>(sStage + C::STAGES * C::STAGE_BYTES);
  if (warp == 0) {
    dkdv_producer<D>(p, it, &tk, &tv, &tq, &tdo, bars, meta, un, sFix, sStage, &abort_flag);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) dkdv_mma<D>(bars, meta, sFix, sStage, tmem, &abort_flag);
    __syncwarp();
  } else {
    dkdv_compute<D>(p, it, (warp - 2) >> 2, bars, meta, sStage, tmem, &abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_DKDV);
  }
}

// ------------------------------------------------------------------ D = rowsum(dO * O)

// One group of D/8 consecutive threads per (sequence, token, head) row; each thread
// takes 8 elements (16 bytes) of O and dO.
template <int D>
__global__ void __launch_bounds__(256) bwd_dvec_kernel(const __nv_bfloat16* o, const __nv_bfloat16* d_o, int64_t sb,
                                                       int64_t sn, int64_t sh, int batch, int n_tokens, int heads,
                                                       float* dvec) {
  constexpr int G = D / 8;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t rowid = gid / G;
  const int part = (int)(gid % G);
  const int64_t n_rows = (int64_t)batch * n_tokens * heads;
  float acc = 0.f;
  int h = 0, i = 0, s = 0;
  if (rowid < n_rows) {
    h = (int)(rowid % heads);
    const int64_t si = rowid / heads;
    i = (int)(si % n_tokens);
    s = (int)(si / n_tokens);
    const int64_t off = (int64_t)s * sb + (int64_t)i * sn + (int64_t)h * sh + 8 * part;
    const uint4 a = *reinterpret_cast<const uint4*>(o + off);
    const uint4 g = *reinterpret_cast<const uint4*>(d_o + off);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[e]));
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int o2 = G / 2; o2 > 0; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2, G);
  if (rowid < n_rows && part == 0) dvec[((int64_t)s * heads + h) * n_tokens + i] = acc;
}

// ------------------------------------------------------------------ transposed CSR

// Row I of sequence s contains block J (rows are ascending): binary search.
__device__ __forceinline__ bool row_has(const int32_t* ci, int lo, int hi, int J) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int v = ci[mid];
    if (v == J) return true;
    if (v < J) lo = mid + 1;
    else hi = mid;
  }
  return false;
}

// One warp per key block J: count (fill == false) or list (fill == true) the query blocks
// I whose row holds J, ascending; under causality only I >= J.
__global__ void __launch_bounds__(256) csc_pass_kernel(const int32_t* rp_all, const int32_t* ci, int nb, int causal,
                                                       int32_t* col_ptr, int32_t* row_idx, int64_t capacity,
                                                       int fill) {
  const int s = blockIdx.y;
  const int J = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (J >= nb) return;
  const int32_t* rp = rp_all + (size_t)s * (nb + 1);
  int32_t* cp = col_ptr + (size_t)s * (nb + 1);
  int pos = fill ? cp[J] : 0;
  int count = 0;
  for (int I0 = causal ? J : 0; I0 < nb; I0 += 32) {
    const int I = I0 + lane;
    const bool hit = I < nb && row_has(ci, rp[I], rp[I + 1], J);
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (fill && hit) {
      const int64_t at = (int64_t)pos + __popc(m & ((1u << lane) - 1u));
      if (at < capacity) row_idx[at] = I;
      else atomicOr(&g_bwd_err, kErrCapacity);
    }
    pos += __popc(m);
    count += __popc(m);
  }
  if (!fill && lane == 0) cp[J + 1] = count;   // counts, turned into offsets by csc_scan
}

// In-place scan of one sequence's counts: cp[J] = rp[0] + sum of counts of blocks < J.
// Each thread owns at most 4 consecutive blocks (nb <= 4096) and keeps their counts in
// registers, so no count is read after a neighbour has overwritten it. Offsets are
// clamped to the index buffer's capacity (an overflow is reported), so every list that
// is read later lies inside the buffer.
__global__ void __launch_bounds__(1024) csc_scan_kernel(const int32_t* rp_all, int nb, int32_t* col_ptr,
                                                        int64_t capacity) {
  __shared__ int part[32];
  const int s = blockIdx.x;
  const int32_t* rp = rp_all + (size_t)s * (nb + 1);
  int32_t* cp = col_ptr + (size_t)s * (nb + 1);
  const int per = (nb + 1023) / 1024;                // <= 4
  const int lo = min(nb, (int)threadIdx.x * per), hi = min(nb, lo + per);
  int cnt[4];
  int sum = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    cnt[e] = (lo + e < hi) ? cp[lo + e + 1] : 0;
    sum += cnt[e];
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) part[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = part[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    part[lane] = v;
  }
  __syncthreads();
  int64_t run = (int64_t)rp[0] + (w > 0 ? part[w - 1] : 0) + incl - sum;
  const int64_t cap = capacity;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (lo + e < hi) {
      cp[lo + e] = (int32_t)min(run, cap);
      run += cnt[e];
    }
  }
  if (lo < hi && hi == nb) {
    cp[nb] = (int32_t)min(run, cap);
    if (run > cap) atomicOr(&g_bwd_err, kErrCapacity);
  }
}

// ------------------------------------------------------------------ launch

template <int D>
int launch_attention(const BwdArgs& a, const BwdWorkspace& ws, const int32_t* const* csc_ptr,
                     const int32_t* const* csc_idx, cudaStream_t stream) {
  using C = BCfg<D>;
  const uint32_t mrows = a.block == 32 ? 32u : 64u;
  uint8_t* wsb = static_cast<uint8_t*>(a.workspace);
  BParams p;
  p.batch = a.batch;
  p.n_tokens = a.n_tokens;
  p.heads = a.heads;
  p.kv_heads = a.kv_heads;
  p.heads_per_kv = a.heads / a.kv_heads;
  p.block = a.block;
  p.log2b = __builtin_ctz((unsigned)a.block);
  p.nb = a.n_tokens / a.block;
  p.causal = a.causal;
  p.csr_shared = a.csr_shared;
  p.tiles = (a.n_tokens + kRows - 1) / kRows;
  p.lse = a.lse;
  p.dvec = reinterpret_cast<const float*>(wsb + ws.dvec_off);
  p.scale = a.softmax_scale;
  p.scale_log2 = a.softmax_scale * kLog2e;
  p.n_masks = a.n_masks;
  for (int h = 0; h < kMaxHeadMap; ++h) p.head_mask[h] = a.head_mask[h];

  // dQ: query-stationary over the CSR
  {
    CUtensorMap tq, tdo, tk, tv;
    if (!encode_bhnd_map(&tq, a.q, a.batch, a.n_tokens, a.heads, D, a.q_strides[0], a.q_strides[1], a.q_strides[2],
                         C::CH, kRows, C::TMA_SWZ) ||
        !encode_bhnd_map(&tdo, a.d_o, a.batch, a.n_tokens, a.heads, D, a.o_strides[0], a.o_strides[1],
                         a.o_strides[2], C::CH, kRows, C::TMA_SWZ) ||
        !encode_bhnd_map(&tk, a.k, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                         a.kv_strides[2], C::CH, mrows, C::TMA_SWZ) ||
        !encode_bhnd_map(&tv, a.v, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                         a.kv_strides[2], C::CH, mrows, C::TMA_SWZ))
      return SA_ERR_UNSUPPORTED;
    BParams pq = p;
    for (int m = 0; m < kMaxMasks; ++m) {
      pq.rp[m] = m < a.n_masks ? a.row_ptr[m] : nullptr;
      pq.ci[m] = m < a.n_masks ? a.col_idx[m] : nullptr;
    }
    pq.n_items = a.batch * a.heads * p.tiles;
    pq.out0 = static_cast<__nv_bfloat16*>(a.dq);
    pq.out1 = nullptr;
    pq.os_b = a.q_strides[0];
    pq.os_n = a.q_strides[1];
    pq.os_h = a.q_strides[2];
    auto kern = bwd_dq_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return SA_ERR_CUDA;
    kern<<<pq.n_items, kThreads, C::SMEM, stream>>>(tq, tdo, tk, tv, pq);
    if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
  }
  // dK, dV: key-stationary over the transposed CSR
  {
    CUtensorMap tk, tv, tq, tdo;
    if (!encode_bhnd_map(&tk, a.k, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                         a.kv_strides[2], C::CH, kRows, C::TMA_SWZ) ||
        !encode_bhnd_map(&tv, a.v, a.batch, a.n_tokens, a.kv_heads, D, a.kv_strides[0], a.kv_strides[1],
                         a.kv_strides[2], C::CH, kRows, C::TMA_SWZ) ||
        !encode_bhnd_map(&tq, a.q, a.batch, a.n_tokens, a.heads, D, a.q_strides[0], a.q_strides[1], a.q_strides[2],
                         C::CH, mrows, C::TMA_SWZ) ||
        !encode_bhnd_map(&tdo, a.d_o, a.batch, a.n_tokens, a.heads, D, a.o_strides[0], a.o_strides[1],
                         a.o_strides[2], C::CH, mrows, C::TMA_SWZ))
      return SA_ERR_UNSUPPORTED;
    BParams pk = p;
    for (int m = 0; m < kMaxMasks; ++m) {
      pk.rp[m] = m < a.n_masks ? csc_ptr[m] : nullptr;
      pk.ci[m] = m < a.n_masks ? csc_idx[m] : nullptr;
    }
    pk.n_items = a.batch * a.kv_heads * p.tiles;
    pk.out0 = static_cast<__nv_bfloat16*>(a.dk);
    pk.out1 = static_cast<__nv_bfloat16*>(a.dv);
    pk.os_b = a.kv_strides[0];
    pk.os_n = a.kv_strides[1];
    pk.os_h = a.kv_strides[2];
    auto kern = bwd_dkdv_kernel<D>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return SA_ERR_CUDA;
    kern<<<pk.n_items, kThreads, C::SMEM, stream>>>(tk, tv, tq, tdo, pk);
    if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
  }
  return SA_OK;
}

}  // namespace

BwdWorkspace bwd_workspace_layout(int64_t batch, int64_t n_tokens, int64_t heads, int64_t block,
                                  int64_t csr_batches, int64_t col_capacity) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  BwdWorkspace w;
  const int64_t nb = n_tokens / block;
  w.dvec_off = 0;
  w.col_ptr_off = up((size_t)(batch * heads * n_tokens) * 4);
  w.row_idx_off = w.col_ptr_off + up((size_t)(csr_batches * (nb + 1)) * 4);
  w.row_idx_capacity = col_capacity;
  w.bytes = w.row_idx_off + up((size_t)col_capacity * 4);
  return w;
}

int launch_attn_bwd(const BwdArgs& a, cudaStream_t stream) {
  const int csr_batches = a.csr_shared ? 1 : a.batch;
  const int nb = a.n_tokens / a.block;
  // one transposed CSR per mask: col_ptr regions of csr_batches x (nb + 1), row_idx regions of
  // each mask's capacity (one mask: whatever the workspace holds after the fixed parts)
  int64_t cap_total = 0;
  for (int m = 0; m < a.n_masks; ++m) cap_total += a.n_masks > 1 ? a.col_capacity[m] : 0;
  BwdWorkspace ws =
      bwd_workspace_layout(a.batch, a.n_tokens, a.heads, a.block, (int64_t)csr_batches * a.n_masks, cap_total);
  if (a.workspace_bytes < ws.bytes) return SA_ERR_CAPACITY;
  ws.row_idx_capacity = (int64_t)((a.workspace_bytes - ws.row_idx_off) / 4);
  uint8_t* wsb = static_cast<uint8_t*>(a.workspace);
  float* dvec = reinterpret_cast<float*>(wsb + ws.dvec_off);
  int32_t* col_ptr = reinterpret_cast<int32_t*>(wsb + ws.col_ptr_off);
  int32_t* row_idx = reinterpret_cast<int32_t*>(wsb + ws.row_idx_off);

  // D = rowsum(dO * O)
  {
    const int64_t threads = (int64_t)a.batch * a.n_tokens * a.heads * (a.head_dim / 8);
    const int64_t blocks = (threads + 255) / 256;
    const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(a.o);
    const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(a.d_o);
    switch (a.head_dim) {
      case 32: bwd_dvec_kernel<32><<<(unsigned)blocks, 256, 0, stream>>>(o, g, a.o_strides[0], a.o_strides[1],
                                                                       a.o_strides[2], a.batch, a.n_tokens, a.heads, dvec);
        break;
      case 64: bwd_dvec_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(o, g, a.o_strides[0], a.o_strides[1],
                                                                       a.o_strides[2], a.batch, a.n_tokens, a.heads, dvec);
        break;
      default: bwd_dvec_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(o, g, a.o_strides[0], a.o_strides[1],
                                                                        a.o_strides[2], a.batch, a.n_tokens, a.heads, dvec);
    }
    if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
  }
  // transposed CSRs
  const int32_t* csc_ptr[kMaxMasks];
  const int32_t* csc_idx[kMaxMasks];
  int64_t base = 0;
  for (int m = 0; m < a.n_masks; ++m) {
    int32_t* cp = col_ptr + (size_t)m * csr_batches * (nb + 1);
    int32_t* ri = row_idx + base;
    const int64_t cap = a.n_masks > 1 ? a.col_capacity[m] : ws.row_idx_capacity;
    base += cap;
    const dim3 grid((unsigned)((nb + 7) / 8), (unsigned)csr_batches);
    csc_pass_kernel<<<grid, 256, 0, stream>>>(a.row_ptr[m], a.col_idx[m], nb, a.causal, cp, ri, cap, 0);
    csc_scan_kernel<<<csr_batches, 1024, 0, stream>>>(a.row_ptr[m], nb, cp, cap);
    csc_pass_kernel<<<grid, 256, 0, stream>>>(a.row_ptr[m], a.col_idx[m], nb, a.causal, cp, ri, cap, 1);
    if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
    csc_ptr[m] = cp;
    csc_idx[m] = ri;
  }
  switch (a.head_dim) {
    case 32: return launch_attention<32>(a, ws, csc_ptr, csc_idx, stream);
    case 64: return launch_attention<64>(a, ws, csc_ptr, csc_idx, stream);
    case 128: return launch_attention<128>(a, ws, csc_ptr, csc_idx, stream);
  }
  return SA_ERR_UNSUPPORTED;
}

// Scratch of the no-allocation entry point: D and the transposed CSR of one call at a time.
// Every device that loads the library holds one copy of it until the process exits.
static __device__ __align__(256) uint8_t g_bwd_static_scratch[kBwdStaticScratchBytes];

// The array's name is only a host-side stand-in for it; the device address of each device's
// copy is looked up once, by the first call made with that device current, and kept here.
constexpr int kMaxScratchDevices = 64;
std::atomic<void*> g_bwd_scratch_addr[kMaxScratchDevices];

int bwd_static_scratch(void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return SA_ERR_CUDA;
  void* addr = g_bwd_scratch_addr[dev].load(std::memory_order_acquire);
  if (addr == nullptr) {
    if (cudaGetSymbolAddress(&addr, g_bwd_static_scratch) != cudaSuccess || addr == nullptr) return SA_ERR_CUDA;
    g_bwd_scratch_addr[dev].store(addr, std::memory_order_release);
  }
  *ptr = addr;
  return SA_OK;
}

unsigned int bwd_read_and_clear_error(cudaStream_t stream) {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_bwd_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
  cudaMemcpyToSymbolAsync(g_bwd_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  return v;
}

}  // namespace sa
