// Block-sparse flash-attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// Work item: one CTA per (sequence, head, query tile of 128 tokens). The query tile
// covers 128 / b query blocks; the key blocks it visits are the sorted union of their
// CSR rows, each tagged with the set of query blocks whose row contains it. Key blocks
// are packed into key tiles of up to 128 keys and visited once.
//
// Warp roles (192 threads):
//   warp 0     producer: merges the CSR rows (all lanes, warp-uniform), publishes the
//              key-tile descriptions and issues the TMA loads of Q, K and V tiles.
//   warp 1     TMEM owner; lane 0 issues the tensor-core MMAs:
//                S = Q K^T      (A, B from shared memory, accumulator in TMEM)
//                O += P V       (A = P from TMEM, B = V from shared memory)
//   warps 2-5  softmax: one query row per thread (its TMEM lane); online softmax with
//              a lazily rescaled running max, P written back to TMEM as bf16, final
//              normalisation and the O / LSE stores.
// TMEM (256 columns, two CTAs per SM): S in columns [0,128) with P aliased over its
// first 64 columns, O in columns [128, 128 + d).
//
// The token-level rule is: key j of block J is visible to query i of block I iff J is
// in row(I) and (not causal or j <= i) ("Parameter-free Adaptive Sparse Attention via
// Compression-Based Content Selection", section 3.4 block-to-token expansion). The
// kernel never materialises a token mask; it derives the per-row column mask from the
// row membership bits and, on the diagonal block, from the causal compare.
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

constexpr int kTile = 128;       // query rows per CTA and max keys per key tile
constexpr int kThreads = 192;
constexpr int kMetaRing = 4;
constexpr int kMaxSlots = 4;     // key blocks per key tile (128 / b, b >= 32)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;

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
  static constexpr int STAGES = D == 128 ? 1 : 2;      // K and V ring depth
  // at least 80 KB so that no more than two CTAs (2 x 256 TMEM columns) share an SM
  static constexpr int SMEM_NEED = 1024 + TILE_BYTES * (1 + 2 * STAGES);
  static constexpr int SMEM = SMEM_NEED > 80 * 1024 ? SMEM_NEED : 80 * 1024;
};

struct Meta {
  int nslots;
  int jblk[kMaxSlots];
  int mask[kMaxSlots];
};

struct Params {
  int batch, n_tokens, heads, heads_per_kv, block, log2b, nb, causal, csr_shared, ntiles;
  const int32_t* row_ptr;
  const int32_t* col_idx;
  __nv_bfloat16* o;
  float* lse;
  int64_t o_sb, o_sn, o_sh;
  float scale_log2;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t m_full[kMetaRing], m_empty[kMetaRing];
  uint64_t s_full, p_full, pv_done, drain;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  return mbar_wait(bar, parity, abort_flag, &g_attn_err, kErrTimeout);
}

// Wait that ignores the abort flag (used to drain this CTA's own copies before exit).
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity) {
  int never = 0;
  mbar_wait(bar, parity, &never, &g_attn_err, kErrTimeout);
}

// ------------------------------------------------------------------ producer (warp 0)

template <int D>
__device__ void producer(const Params& p, const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                         Bars& bars, Meta* meta, uint8_t* sQ, uint8_t* sK, uint8_t* sV, volatile int* abort_flag,
                         int s, int h, int hk, int I0, int q0) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const int b = p.block;
  const int nq = min(kTile / b, p.nb - I0);
  const int slots_per_tile = kTile / b;
  const int32_t* rp = p.row_ptr + (size_t)(p.csr_shared ? 0 : s) * (p.nb + 1);

  if (lane == 0) {
    mbar_arrive_expect_tx(&bars.q_full, C::TILE_BYTES);
#pragma unroll
    for (int c = 0; c < C::NCH; ++c) tma_load_4d(sQ + c * C::CHUNK, tq, &bars.q_full, c * C::CH, h, q0, s);
  }

  // Row cursors (warp-uniform). Lane i caches col_idx[base[r] + i] of row r.
  const int rpv = (lane <= nq) ? rp[I0 + lane] : 0;
  int head[kMaxSlots], endp[kMaxSlots], base[kMaxSlots], prev[kMaxSlots], cache[kMaxSlots];
#pragma unroll
  for (int r = 0; r < kMaxSlots; ++r) {
    const int hh = __shfl_sync(0xffffffffu, rpv, min(r, nq));
    const int ee = __shfl_sync(0xffffffffu, rpv, min(r + 1, nq));
    head[r] = hh;
    endp[r] = (r < nq) ? ee : hh;
    base[r] = hh;
    prev[r] = -1;
    cache[r] = (hh + lane < endp[r]) ? p.col_idx[hh + lane] : 0;
  }
  auto current = [&](int r) -> int {
    // next valid column of row r (validates range and strict ascent), or INT_MAX
    while (head[r] < endp[r]) {
      if (head[r] - base[r] >= 32) {
        base[r] = head[r];
        cache[r] = (base[r] + lane < endp[r]) ? p.col_idx[base[r] + lane] : 0;
      }
      const int J = __shfl_sync(0xffffffffu, cache[r], head[r] - base[r]);
      if (J >= 0 && J < p.nb && J > prev[r]) return J;
      if (lane == 0) atomicOr(&g_attn_err, kErrBadIndex);
      ++head[r];
    }
    return 0x7fffffff;
  };
  int cur[kMaxSlots];
#pragma unroll
  for (int r = 0; r < kMaxSlots; ++r) cur[r] = current(r);

  int k_issued[2] = {-1, -1}, v_issued[2] = {-1, -1};
  for (int t = 0;; ++t) {
    Meta m;
    m.nslots = 0;
    while (m.nslots < slots_per_tile) {
      int J = 0x7fffffff;
#pragma unroll
      for (int r = 0; r < kMaxSlots; ++r) J = min(J, cur[r]);
      if (J == 0x7fffffff) break;
      int mask = 0;
#pragma unroll
      for (int r = 0; r < kMaxSlots; ++r) {
        if (cur[r] == J) {
          mask |= 1 << r;
          prev[r] = J;
          ++head[r];
          cur[r] = current(r);
        }
      }
      if (p.causal) {
#pragma unroll
        for (int r = 0; r < kMaxSlots; ++r)
          if (J > I0 + r) mask &= ~(1 << r);
      }
      if (mask == 0) continue;
      m.jblk[m.nslots] = J;
      m.mask[m.nslots] = mask;
      ++m.nslots;
    }
    bool ok = true;
    if (lane == 0) {
      const int ms = t % kMetaRing;
      ok = wait_bar(&bars.m_empty[ms], ((t / kMetaRing) & 1) ^ 1, abort_flag);
      if (ok) {
        meta[ms] = m;
        mbar_arrive(&bars.m_full[ms]);
      }
      if (ok && m.nslots > 0) {
        const int st = t % C::STAGES;
        const uint32_t ph = (t / C::STAGES) & 1;
        const uint32_t bytes = (uint32_t)(m.nslots * b * D * 2);
        ok = wait_bar(&bars.k_empty[st], ph ^ 1, abort_flag);
        if (ok) {
          mbar_arrive_expect_tx(&bars.k_full[st], bytes);
          for (int i = 0; i < m.nslots; ++i)
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
              tma_load_4d(sK + st * C::TILE_BYTES + c * C::CHUNK + i * b * C::ROWB, tk, &bars.k_full[st],
                          c * C::CH, hk, m.jblk[i] * b, s);
          k_issued[st] = t;
          ok = wait_bar(&bars.v_empty[st], ph ^ 1, abort_flag);
        }
        if (ok) {
          mbar_arrive_expect_tx(&bars.v_full[st], bytes);
          for (int i = 0; i < m.nslots; ++i)
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
              tma_load_4d(sV + st * C::TILE_BYTES + c * C::CHUNK + i * b * C::ROWB, tv, &bars.v_full[st],
                          c * C::CH, hk, m.jblk[i] * b, s);
          v_issued[st] = t;
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok || m.nslots == 0) break;
  }
  // Drain this CTA's own copies in flight before the CTA may exit.
  if (lane == 0) {
    drain_bar(&bars.q_full, 0);
    for (int st = 0; st < C::STAGES; ++st) {
      if (k_issued[st] >= 0) drain_bar(&bars.k_full[st], (k_issued[st] / C::STAGES) & 1);
      if (v_issued[st] >= 0) drain_bar(&bars.v_full[st], (v_issued[st] / C::STAGES) & 1);
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA issuer (warp 1, lane 0)

template <int D>
__device__ void mma_issuer(const Params& p, Bars& bars, Meta* meta, uint8_t* sQ, uint8_t* sK, uint8_t* sV,
                           uint32_t tmem, volatile int* abort_flag) {
  using C = Cfg<D>;
  const uint32_t tS = tmem + kColS, tO = tmem + kColO;
  const uint32_t idesc_pv = make_idesc_bf16(128, D, 0, 1);
  const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
  for (int t = 0;; ++t) {
    const int ms = t % kMetaRing;
    if (!wait_bar(&bars.m_full[ms], (t / kMetaRing) & 1, abort_flag)) break;
    const int nslots = *reinterpret_cast<volatile int*>(&meta[ms].nslots);
    if (nslots == 0) break;
    const int st = t % C::STAGES;
    const uint32_t ph = (t / C::STAGES) & 1;
    if (t == 0 && !wait_bar(&bars.q_full, 0, abort_flag)) break;
    if (!wait_bar(&bars.k_full[st], ph, abort_flag)) break;
    if (t > 0 && !wait_bar(&bars.pv_done, (t - 1) & 1, abort_flag)) break;   // P (aliases S) consumed
    tc_fence_after();
    const int N = nslots * p.block;
    const uint32_t idesc_qk = make_idesc_bf16(128, (uint32_t)N, 0, 0);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int c = (ks * 16) / C::CH, koff = (ks * 16) % C::CH;
      const uint64_t a = make_smem_desc(q_addr + c * C::CHUNK + koff * 2, 16, C::ATOM, C::SWZ);
      const uint64_t bd =
          make_smem_desc(k_addr + st * C::TILE_BYTES + c * C::CHUNK + koff * 2, 16, C::ATOM, C::SWZ);
      mma_bf16_ss(tS, a, bd, idesc_qk, ks > 0 ? 1u : 0u);
    }
    mma_commit(&bars.s_full);
    mma_commit(&bars.k_empty[st]);
    if (!wait_bar(&bars.p_full, t & 1, abort_flag)) break;
    if (!wait_bar(&bars.v_full[st], ph, abort_flag)) break;
    tc_fence_after();
    for (int ks = 0; ks < N / 16; ++ks) {
      const uint64_t bd = make_smem_desc(v_addr + st * C::TILE_BYTES + ks * 16 * C::ROWB, C::CHUNK, C::ATOM, C::SWZ);
      mma_bf16_ts(tO, tS + (uint32_t)(ks * 8), bd, idesc_pv, (t > 0 || ks > 0) ? 1u : 0u);
    }
    mma_commit(&bars.pv_done);
    mma_commit(&bars.v_empty[st]);
  }
  // Make sure no MMA is still writing TMEM when the CTA frees it.
  mma_commit(&bars.drain);
  drain_bar(&bars.drain, 0);
}

// ------------------------------------------------------------------ softmax + epilogue (warps 2-5)

template <int D>
__device__ void softmax_epilogue(const Params& p, Bars& bars, Meta* meta, uint32_t tmem, volatile int* abort_flag,
                                 int s, int h, int I0, int q0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;                      // TMEM lanes this warp may access
  const int row = quarter * 32 + lane;               // query row within the tile
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const uint32_t tS = tmem + kColS + lane_base, tO = tmem + kColO + lane_base;
  const int b = p.block;
  const int sub = row >> p.log2b;                    // query block within the tile
  const int qblk = I0 + sub;
  const int rloc = row & (b - 1);
  const float c = p.scale_log2;
  const float kNegInf = __int_as_float(0xff800000);

  float m_use = kNegInf;   // running reference max, log2 units
  float l = 0.f;
  bool ok = true;
  int t = 0;
  for (;; ++t) {
    const int ms = t % kMetaRing;
    if (!wait_bar(&bars.m_full[ms], (t / kMetaRing) & 1, abort_flag)) { ok = false; break; }
    Meta m;
    {
      volatile Meta* vm = &meta[ms];
      m.nslots = vm->nslots;
#pragma unroll
      for (int i = 0; i < kMaxSlots; ++i) { m.jblk[i] = vm->jblk[i]; m.mask[i] = vm->mask[i]; }
    }
    if (m.nslots == 0) break;
    if (!wait_bar(&bars.s_full, t & 1, abort_flag)) { ok = false; break; }
    tc_fence_after();
    const int nch = (m.nslots * b) >> 5;             // 32-column chunks holding keys

    uint32_t sv[128];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
      if (ch < nch) tmem_ld_x32(tS + ch * 32, sv + ch * 32);
    tmem_ld_wait<128>(sv);

    uint32_t keep[4];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t kp = 0u;
      if (ch < nch) {
        const int slot = (ch * 32) >> p.log2b;
        const int J = m.jblk[slot];
        if ((m.mask[slot] >> sub) & 1) {
          if (!p.causal || J < qblk) {
            kp = 0xffffffffu;
          } else if (J == qblk) {
            const int lim = rloc - ((ch * 32) & (b - 1));   // visible columns j <= lim
            kp = lim >= 31 ? 0xffffffffu : (lim < 0 ? 0u : ((2u << lim) - 1u));
          }
        }
      }
      keep[ch] = kp;
    }

    float mx = kNegInf;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      if (keep[ch] == 0xffffffffu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(sv[ch * 32 + j]));
      } else if (keep[ch] != 0u) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if ((keep[ch] >> j) & 1u) mx = fmaxf(mx, __uint_as_float(sv[ch * 32 + j]));
      }
    }
    const float m_tile = mx * c;                     // -inf stays -inf (c > 0)
    const float m_new = fmaxf(m_use, m_tile);
    const bool need = m_new > m_use + 8.0f;          // rescale only when the max grew by > 2^8
    float alpha = 1.f;
    if (need) {
      alpha = ex2_approx(m_use - m_new);             // 0 when m_use = -inf
      m_use = m_new;
    }

    float rs = 0.f;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      if (ch < nch) {
        uint32_t pk[16];
        const uint32_t kp = keep[ch];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = ((kp >> j) & 1u) ? ex2_approx(fmaf(__uint_as_float(sv[ch * 32 + j]), c, -m_use)) : 0.f;
          const float p1 =
              ((kp >> (j + 1)) & 1u) ? ex2_approx(fmaf(__uint_as_float(sv[ch * 32 + j + 1]), c, -m_use)) : 0.f;
          rs += p0 + p1;
          pk[j >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st_x16(tS + ch * 16, pk);
      }
    }
    l = l * alpha + rs;

    if (__any_sync(0xffffffffu, need && t > 0)) {
      if (!wait_bar(&bars.pv_done, (t - 1) & 1, abort_flag)) ok = false;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        tmem_ld_x32(tO + ch * 32, ov);
        tmem_ld_wait<32>(ov);
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
        tmem_st_x32(tO + ch * 32, ov);
      }
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(&bars.p_full);
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.m_empty[ms]);
  }
  const int T = t;
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) return;
  if (T > 0) {
    ok = wait_bar(&bars.pv_done, (T - 1) & 1, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return;
    tc_fence_after();
  }
  const int qtok = q0 + row;
  const bool store = qtok < p.n_tokens;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  __nv_bfloat16* orow = p.o + (int64_t)s * p.o_sb + (int64_t)qtok * p.o_sn + (int64_t)h * p.o_sh;
#pragma unroll
  for (int ch = 0; ch < D / 32; ++ch) {
    uint32_t ov[32];
    if (T > 0) {
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
  if (store) {
    const float lse = l > 0.f ? (m_use + __log2f(l)) * 0.69314718055994531f : kNegInf;
    p.lse[((int64_t)s * p.heads + h) * p.n_tokens + qtok] = lse;
  }
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sQ = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sQ + C::TILE_BYTES;
  uint8_t* sV = sK + C::STAGES * C::TILE_BYTES;
  __shared__ Bars bars;
  __shared__ Meta meta[kMetaRing];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.x % p.heads;
  const int s = blockIdx.x / p.heads;
  const int tile = p.causal ? (p.ntiles - 1 - (int)blockIdx.y) : (int)blockIdx.y;
  const int I0 = tile * (kTile >> p.log2b);
  const int q0 = tile * kTile;
  const int hk = h / p.heads_per_kv;

  if (threadIdx.x == 0) {
    mbar_init(&bars.q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < kMetaRing; ++i) {
      mbar_init(&bars.m_full[i], 1);
      mbar_init(&bars.m_empty[i], 4);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_full, 128);
    mbar_init(&bars.pv_done, 1);
    mbar_init(&bars.drain, 1);
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
    producer<D>(p, &tq, &tk, &tv, bars, meta, sQ, sK, sV, &abort_flag, s, h, hk, I0, q0);
  } else if (warp == 1) {
    if ((threadIdx.x & 31) == 0) mma_issuer<D>(p, bars, meta, sQ, sK, sV, tmem, &abort_flag);
    __syncwarp();
  } else {
    softmax_epilogue<D>(p, bars, meta, tmem, &abort_flag, s, h, I0, q0);
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
  p.ntiles = (a.n_tokens + kTile - 1) / kTile;
  p.row_ptr = a.row_ptr;
  p.col_idx = a.col_idx;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.o_sb = a.o_strides[0];
  p.o_sn = a.o_strides[1];
  p.o_sh = a.o_strides[2];
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  auto kern = attn_fwd_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return SA_ERR_CUDA;
  dim3 grid((unsigned)(a.batch * a.heads), (unsigned)p.ntiles);
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
