// GPU block-CSR builder: per-block ratios and pattern parameters -> row_ptr / col_idx.
//
// CTAs of 1024 threads (256 for mean-threshold masks of up to 1024 blocks), a few per sequence
// (grid.y splits the rows). Each CTA
//   1. computes the per-sequence state the mode needs (ratio rank order for TOPK,
//      literal flags from the mean threshold for LITERAL_MEAN),
//   2. computes every row length and an exclusive scan of them (row_ptr), offset by the
//      entries of the sequences before it,
//   3. fills its share of the rows, one warp per row, in ascending block order.
// All decisions are integer or exact float compares, so the output is bit-identical
// to the definitions in include/sa_api.h on every run.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <stdint.h>

#include "sa_internal.h"

namespace sa {
namespace {

constexpr int kMaxThreads = 1024;     // CTA size for long sequences (256 when nb <= 1024)
constexpr int kMaxWarps = kMaxThreads / 32;


struct MaskArgs {
  int mode, block, nb, batch, causal, w, g, k, r;
  int local, literal;   // LITERAL_MEAN: which parts besides the identity are kept
  uint64_t seed;
  const float* ratio;
  int32_t* row_ptr;
  int32_t* col_idx;
};

// ---------------------------------------------------------------- Philox4x64-10
// Salmon, Moraes, Dror, Shaw, SC'11: two 64x64->128 multiplies per round with the
// published multipliers, key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint64_t philox_word(uint64_t seed, uint64_t p) {
  uint64_t c0 = p / 4 + 1, c1 = 0, c2 = 0, c3 = 0;
  uint64_t k0 = seed, k1 = 0;
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
    const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
    const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B97F4A7C15ull;
    k1 += 0xBB67AE8584CAA73Bull;
  }
  const uint32_t lane = static_cast<uint32_t>(p & 3u);
  return lane == 0 ? c0 : lane == 1 ? c1 : lane == 2 ? c2 : c3;
}

// ---------------------------------------------------------------- block helpers

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Sum of one int64 per thread over the CTA.
template <int T>  // threads per CTA
__device__ int64_t block_sum(int64_t v, int64_t* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  int64_t t = 0;
  for (int i = 0; i < (T / 32); ++i) t += red[i];
  __syncthreads();
  return t;
}

// In-place exclusive scan of a[0..n), n <= 4 * blockDim.x. Returns the total.
template <int T>  // threads per CTA
__device__ int block_exclusive_scan(int* a, int n, int* tmp) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (n + T - 1) / T;
  const int base = tid * per;
  int local[4];
  int s = 0;
  for (int i = 0; i < per; ++i) {
    const int idx = base + i;
    const int v = idx < n ? a[idx] : 0;
    local[i] = s;
    s += v;
  }
  int x = s;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    const int w = lane < (T / 32) ? tmp[lane] : 0;
    int wx = w;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wx, o);
      if (lane >= o) wx += y;
    }
    tmp[lane] = wx - w;
    if (lane == 31) tmp[32] = wx;
  }
  __syncthreads();
  const int excl = tmp[wid] + x - s;
  for (int i = 0; i < per; ++i) {
    const int idx = base + i;
    if (idx < n) a[idx] = excl + local[i];
  }
  const int total = tmp[32];
  __syncthreads();
  return total;
}

// ---------------------------------------------------------------- per-mode pieces

constexpr int kPriorWarps = 8;          // warps that derive earlier sequences' entry counts
constexpr int kPriorMaxBlocks = 1024;   // ... when their literal prefixes fit in shared memory

struct Smem {
  float* r;        // [nb] ratios of the current sequence
  int* order;      // [nb] TOPK: blocks by (ratio desc, index asc); LITERAL_MEAN: literal prefix [nb+1]
  int* cnt;        // [nb] row lengths, scanned in place into row offsets
  uint32_t* bm;    // [warps][words] per-warp bitmaps
  int* lscr;       // LITERAL_MEAN, nb <= kPriorMaxBlocks: [kPriorWarps][nb+1] literal prefixes of
                   // earlier sequences (nullptr: derive them one after another)
  int words;
  int64_t* red;
  double* redf;
  int* scan_tmp;   // [33]
};

template <int T>  // threads per CTA
__device__ void load_ratios(const MaskArgs& a, const Smem& s, int seq) {
  for (int j = threadIdx.x; j < a.nb; j += T) s.r[j] = a.ratio[(size_t)seq * a.nb + j];
  __syncthreads();
}

// TOPK: rank by (ratio desc, index asc) over all blocks; order[rank] = block. Eight
// consecutive lanes share a block j and count over interleaved eighths of the blocks.
template <int T>  // threads per CTA
__device__ void topk_order(const MaskArgs& a, const Smem& s) {
  const int part = threadIdx.x & 7;
  const int kGroups = T >> 3;
  const int iters = (a.nb + kGroups - 1) / kGroups;   // the same for every thread: the
  for (int it = 0; it < iters; ++it) {                // whole warp reaches the shuffles
    const int j0 = (threadIdx.x >> 3) + kGroups * it;
    const int j = j0 < a.nb ? j0 : a.nb - 1;
    const float rj = s.r[j];
    int rank = 0;
    for (int t = part; t < a.nb; t += 8) {
      const float rt = s.r[t];
      rank += (rt > rj) || (rt == rj && t < j);
    }
    rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    rank += __shfl_xor_sync(0xffffffffu, rank, 2);
    rank += __shfl_xor_sync(0xffffffffu, rank, 4);
    if (part == 0 && j0 < a.nb) s.order[rank] = j;
  }
  __syncthreads();
}

// LITERAL_MEAN: literal flag l_j = (r_j > mean r); stored as prefix counts lit[0..nb].
// Mean of one sequence's ratios (r: nb values), computed by one warp with the same arithmetic
// wherever it runs: lane-strided partial sums in double, then a butterfly over the warp (every
// lane ends with the same bits, as each step adds the same two values). Every CTA that derives
// a sequence's literal flags therefore agrees with every other on them.
__device__ double warp_seq_mean(const MaskArgs& a, const float* r) {
  const int lane = threadIdx.x & 31;
  double part = 0.0;
  for (int j = lane; j < a.nb; j += 32) part += (double)r[j];
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  return part / (double)a.nb;
}

template <int T>  // threads per CTA
__device__ void literal_prefix(const MaskArgs& a, const Smem& s) {
  if ((threadIdx.x >> 5) == 0) {
    const double m = warp_seq_mean(a, s.r);
    if (threadIdx.x == 0) s.redf[0] = m;
  }
  __syncthreads();
  const double mean = s.redf[0];
  __syncthreads();
  int* lit = s.order;
  for (int j = threadIdx.x; j < a.nb; j += T) lit[j] = ((double)s.r[j] > mean) ? 1 : 0;
  __syncthreads();
  const int total = block_exclusive_scan<T>(lit, a.nb, s.scan_tmp);
  if (threadIdx.x == 0) lit[a.nb] = total;
  __syncthreads();
}

__device__ __forceinline__ int lit_at(const int* litpre, int j) { return litpre[j + 1] - litpre[j]; }

__device__ __forceinline__ int bigbird_wlo(const MaskArgs& a, int I) { return I - a.w / 2; }

// Length of row I.
// LITERAL_MEAN row length of block row I from the literal prefix lp[0..nb].
__device__ int literal_row_len(const MaskArgs& a, const int* lp, int I) {
  int n = 1;                                                         // identity
  if (a.local) {
    const int lo = max(0, I - a.w);
    const int hi = a.causal ? I : min(a.nb - 1, I + a.w);
    n = hi - lo + 1;
  }
  if (a.literal && lit_at(lp, I)) {
    if (I - a.w - 1 >= 0) n += lp[I - a.w];                         // literals in [0, I-w-1]
    if (!a.causal && I + a.w + 1 < a.nb) n += lp[a.nb] - lp[I + a.w + 1];
  }
  return n;
}

// LITERAL_MEAN: CSR entries of the sequences before `seq`, warp w < kPriorWarps taking
// sequences w, w + kPriorWarps, ... (mean, literal prefix in its own scratch, row lengths).
template <int T>  // threads per CTA
__device__ int64_t literal_prior_entries(const MaskArgs& a, int seq, int* scratch, int64_t* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = min((T / 32), kPriorWarps);
  int64_t mine = 0;
  if (wid < nw) {
    int* lp = scratch + (size_t)wid * (a.nb + 1);
    for (int p = wid; p < seq; p += nw) {
      const float* r = a.ratio + (size_t)p * a.nb;
      const double mean = warp_seq_mean(a, r);
      int run = 0;
      for (int j0 = 0; j0 < a.nb; j0 += 32) {
        const int j = j0 + lane;
        const bool f = j < a.nb && (double)r[j] > mean;
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (j < a.nb) lp[j] = run + __popc(m & lanemask_lt());
        run += __popc(m);
      }
      if (lane == 0) lp[a.nb] = run;
      __syncwarp();
      int64_t tot = 0;
      for (int I = lane; I < a.nb; I += 32) tot += literal_row_len(a, lp, I);
      for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
      mine += tot;
      __syncwarp();                                  // lp is this warp's again for its next sequence
    }
  }
  return block_sum<T>(lane == 0 ? mine : 0, red);
}

__device__ int row_len(const MaskArgs& a, const Smem& s, int I) {
  switch (a.mode) {
    case SA_MASK_TOPK: {
      const int n_w = min(a.w, I + 1);
      const int n_g = max(0, min(a.g, I - a.w + 1));
      const int n_c = max(0, I - a.w + 1 - a.g);
      return n_w + n_g + min(a.k, n_c);
    }
    case SA_MASK_FULL:
      return a.causal ? I + 1 : a.nb;
    case SA_MASK_BIGBIRD: {
      if (I < a.g) return a.nb;
      const int g = min(a.g, a.nb);
      const int lo = max(0, bigbird_wlo(a, I)), hi = min(a.nb - 1, bigbird_wlo(a, I) + a.w - 1);
      const int n_w = max(0, hi - lo + 1);
      const int n_wg = max(0, min(hi, g - 1) - lo + 1);  // window blocks that are global
      const int n_union = n_w + g - n_wg;
      return n_union + min(a.r, a.nb - n_union);
    }
    case SA_MASK_LITERAL_MEAN:
      return literal_row_len(a, s.order, I);
  }
  return 0;
}

// Total entries of one sequence (state for that sequence already in smem).
template <int T>  // threads per CTA
__device__ int64_t seq_total(const MaskArgs& a, const Smem& s) {
  int64_t part = 0;
  for (int I = threadIdx.x; I < a.nb; I += T) part += row_len(a, s, I);
  return block_sum<T>(part, s.red);
}

// ---------------------------------------------------------------- row fills (one warp)

__device__ void fill_topk(const MaskArgs& a, const Smem& s, int I, int32_t* out, uint32_t* bm) {
  const int lane = threadIdx.x & 31;
  const int n_w = min(a.w, I + 1);
  const int n_g = max(0, min(a.g, I - a.w + 1));
  const int hi_c = I - a.w;                                  // candidates [g, hi_c]
  const int n_c = max(0, hi_c - a.g + 1);
  const int kk = min(a.k, n_c);
  for (int j = lane; j < n_g; j += 32) out[j] = j;
  if (kk == n_c) {
    for (int j = lane; j < n_c; j += 32) out[n_g + j] = a.g + j;
  } else if (kk > 0) {
    for (int wd = (a.g >> 5) + lane; wd <= (hi_c >> 5); wd += 32) bm[wd] = 0u;
    __syncwarp();
    int taken = 0;
    for (int base = 0; base < a.nb && taken < kk; base += 32) {
      const int J = (base + lane < a.nb) ? s.order[base + lane] : -1;
      const bool cand = J >= a.g && J <= hi_c;
      const unsigned m = __ballot_sync(0xffffffffu, cand);
      const int before = __popc(m & lanemask_lt());
      if (cand && taken + before < kk) atomicOr(&bm[J >> 5], 1u << (J & 31));
      taken += __popc(m);
    }
    __syncwarp();
    int pos = n_g;
    for (int base = a.g; base <= hi_c; base += 32) {
      const int J = base + lane;
      const bool sel = J <= hi_c && ((bm[J >> 5] >> (J & 31)) & 1u);
      const unsigned m = __ballot_sync(0xffffffffu, sel);
      if (sel) out[pos + __popc(m & lanemask_lt())] = J;
      pos += __popc(m);
    }
    __syncwarp();
  }
  for (int j = lane; j < n_w; j += 32) out[n_g + kk + j] = I - n_w + 1 + j;
}

__device__ void fill_literal_mean(const MaskArgs& a, const Smem& s, int I, int32_t* out) {
  const int lane = threadIdx.x & 31;
  const int* lp = s.order;
  const bool lit_i = a.literal && lit_at(lp, I) != 0;
  const int reach = a.local ? a.w : 0;                     // band kept around I
  const int lo = lit_i ? 0 : max(0, I - reach);
  const int hi = a.causal ? I : (lit_i ? a.nb - 1 : min(a.nb - 1, I + reach));
  int pos = 0;
  for (int base = lo; base <= hi; base += 32) {
    const int J = base + lane;
    bool sel = false;
    if (J <= hi) {
      const int dist = J > I ? J - I : I - J;
      sel = dist <= reach || (lit_i && lit_at(lp, J) && dist > a.w);
    }
    const unsigned m = __ballot_sync(0xffffffffu, sel);
    if (sel) out[pos + __popc(m & lanemask_lt())] = J;
    pos += __popc(m);
  }
}

__device__ void fill_bigbird(const MaskArgs& a, int I, int32_t* out, int* picks) {
  const int lane = threadIdx.x & 31;
  if (I < a.g) {
    for (int j = lane; j < a.nb; j += 32) out[j] = j;
    return;
  }
  const int g = min(a.g, a.nb);
  const int wlo = max(0, bigbird_wlo(a, I));
  const int whi = min(a.nb - 1, bigbird_wlo(a, I) + a.w - 1);
  // Interval part: [0, g) u [wlo, whi] as at most two disjoint ascending segments.
  int s0lo = 0, s0hi = g - 1, s1lo = wlo, s1hi = whi;         // inclusive bounds
  if (whi < wlo) { s1lo = 1; s1hi = 0; }                       // empty window
  if (s1lo <= s1hi && s1lo <= g) {                             // overlapping / adjacent
    s0hi = max(s0hi, s1hi);
    s1lo = 1;
    s1hi = 0;
  }
  const int n0 = max(0, s0hi - s0lo + 1), n1 = max(0, s1hi - s1lo + 1);
  const int n_int = n0 + n1;
  // Candidates A = [g, nb) minus [wlo, whi], ascending: segment a1 = [g, wlo), a2 = [max(g, whi+1), nb).
  const int a1 = max(0, wlo - g);
  const int a2start = max(g, whi + 1);
  const int a2 = max(0, a.nb - a2start);
  const int n_a = (whi < wlo) ? (a.nb - g) : a1 + a2;
  const int n_r = min(a.r, n_a);
  if (lane == 0) {
    // picks[0..n_r): chosen indices into A, kept sorted ascending.
    for (int t = 0; t < n_r; ++t) {
      const uint64_t x = philox_word(static_cast<uint64_t>(a.seed), (uint64_t)I * (uint64_t)a.r + (uint64_t)t);
      const uint64_t remaining = (uint64_t)(n_a - t);
      int j = (int)(((x >> 32) * remaining) >> 32);
      int ins = 0;
      for (; ins < t; ++ins) {
        if (picks[ins] <= j) ++j;
        else break;
      }
      for (int u = t; u > ins; --u) picks[u] = picks[u - 1];
      picks[ins] = j;
    }
    for (int t = 0; t < n_r; ++t) {                            // A-index -> block index
      const int m = picks[t];
      picks[t] = (whi < wlo) ? g + m : (m < a1 ? g + m : a2start + (m - a1));
    }
  }
  __syncwarp();
  for (int e = lane; e < n_int; e += 32) {
    const int x = e < n0 ? s0lo + e : s1lo + (e - n0);
    int below = 0;
    for (int t = 0; t < n_r; ++t) below += picks[t] < x;
    out[e + below] = x;
  }
  for (int t = lane; t < n_r; t += 32) {
    const int x = picks[t];
    const int below = max(0, min(x, s0hi + 1) - s0lo) + max(0, min(x, s1hi + 1) - s1lo);
    out[below + t] = x;
  }
  __syncwarp();
}

template <int T>  // threads per CTA: 256 or 1024
__global__ void __launch_bounds__(T) build_mask_kernel(MaskArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int64_t red[kMaxWarps];
  __shared__ double redf[kMaxWarps];
  __shared__ int scan_tmp[33];
  __shared__ int picks_all[kMaxWarps][kMaxRandomBlocks];
  const int seq = blockIdx.x;
  Smem s;
  s.words = (a.nb + 31) / 32;
  s.r = reinterpret_cast<float*>(smem_raw);
  s.order = reinterpret_cast<int*>(s.r + a.nb);
  s.cnt = s.order + (a.nb + 1);
  s.bm = reinterpret_cast<uint32_t*>(s.cnt + a.nb);
  s.lscr = (a.mode == SA_MASK_LITERAL_MEAN && a.nb <= kPriorMaxBlocks)
               ? reinterpret_cast<int*>(s.bm + (size_t)(T / 32) * s.words)
               : nullptr;
  s.red = red;
  s.redf = redf;
  s.scan_tmp = scan_tmp;

  // Entries of the sequences before this one.
  int64_t base = 0;
  if (a.mode == SA_MASK_LITERAL_MEAN) {
    if (s.lscr != nullptr) {
      base = literal_prior_entries<T>(a, seq, s.lscr, red);
    } else {
      for (int p = 0; p < seq; ++p) {
        load_ratios<T>(a, s, p);
        literal_prefix<T>(a, s);
        base += seq_total<T>(a, s);
      }
    }
  }
  const bool needs_ratio = a.mode == SA_MASK_TOPK || a.mode == SA_MASK_LITERAL_MEAN;
  if (needs_ratio) load_ratios<T>(a, s, seq);
  if (a.mode == SA_MASK_TOPK) topk_order<T>(a, s);
  if (a.mode == SA_MASK_LITERAL_MEAN) literal_prefix<T>(a, s);

  for (int I = threadIdx.x; I < a.nb; I += T) s.cnt[I] = row_len(a, s, I);
  __syncthreads();
  const int total = block_exclusive_scan<T>(s.cnt, a.nb, s.scan_tmp);
  // row lengths of the other modes do not depend on the data: every sequence has `total`
  if (a.mode != SA_MASK_LITERAL_MEAN) base = (int64_t)seq * total;
  // this CTA's share of the rows: every CTA of the sequence holds the same state and offsets
  const int per = (a.nb + gridDim.y - 1) / gridDim.y;
  const int row_lo = blockIdx.y * per, row_hi = min(a.nb, row_lo + per);
  int32_t* rp = a.row_ptr + (size_t)seq * (a.nb + 1);
  for (int I = row_lo + threadIdx.x; I < row_hi; I += T) rp[I] = (int32_t)(base + s.cnt[I]);
  if (blockIdx.y == 0 && threadIdx.x == 0) rp[a.nb] = (int32_t)(base + total);

  const int wid = threadIdx.x >> 5;
  uint32_t* bm = s.bm + (size_t)wid * s.words;
  for (int I = row_lo + wid; I < row_hi; I += (T / 32)) {
    int32_t* out = a.col_idx + base + s.cnt[I];
    switch (a.mode) {
      case SA_MASK_TOPK: fill_topk(a, s, I, out, bm); break;
      case SA_MASK_LITERAL_MEAN: fill_literal_mean(a, s, I, out); break;
      case SA_MASK_BIGBIRD: fill_bigbird(a, I, out, picks_all[wid]); break;
      case SA_MASK_FULL: {
        const int n = a.causal ? I + 1 : a.nb;
        for (int j = threadIdx.x & 31; j < n; j += 32) out[j] = j;
        break;
      }
    }
  }
}

// The kernel's dynamic shared-memory limit, raised on the current device only when a launch
// needs more than it was last raised to (the attribute call costs host time on every launch).
template <int T>
bool mask_smem_ready(size_t smem) {
  static std::atomic<size_t> raised[64];             // one table per CTA size (T)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::atomic<size_t>* r = dev >= 0 && dev < 64 ? &raised[dev] : nullptr;
  if (r != nullptr && smem <= r->load()) return true;
  if (cudaFuncSetAttribute(build_mask_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return false;
  if (r != nullptr) {
    size_t cur = r->load();
    while (cur < smem && !r->compare_exchange_weak(cur, smem)) {
    }
  }
  return true;
}

}  // namespace

int launch_build_mask(const sa_mask_params& p, const float* d_ratio, int32_t* d_row_ptr, int32_t* d_col_idx,
                      cudaStream_t stream) {
  MaskArgs a;
  a.mode = p.mode;
  a.block = p.block;
  a.nb = p.n_tokens / p.block;
  a.batch = p.batch;
  a.causal = p.causal;
  a.w = p.window_blocks;
  a.g = p.global_blocks;
  a.k = p.topk;
  a.r = p.random_blocks;
  a.seed = p.seed;
  const int comp = p.components ? p.components : (SA_LITERAL_LOCAL | SA_LITERAL_PAIRS);
  a.local = (comp & SA_LITERAL_LOCAL) != 0;
  a.literal = (comp & SA_LITERAL_PAIRS) != 0;
  a.ratio = d_ratio;
  a.row_ptr = d_row_ptr;
  a.col_idx = d_col_idx;
  const int words = (a.nb + 31) / 32;
  // LITERAL_MEAN with up to 1024 blocks: 256-thread CTAs (more, shorter CTAs; the scan's four
  // entries per thread cover the blocks). Measured on the three head-group masks of the 4 x 8K
  // workload: 200 -> 52 us (28 us with the earlier sequences' counts in parallel). The other
  // modes keep 1024 threads: the 8K top-16 mask took 12.4 us with 256 against 9.3 us with 1024
  // (ncu), and BigBird 16K was the same either way. The CTA size is a template parameter, so
  // every loop bound and stride in the kernel is a constant (with blockDim instead, the 8K
  // top-16 mask took 11.7 us).
  const int threads = (a.mode == SA_MASK_LITERAL_MEAN && a.nb <= 4 * 256) ? 256 : kMaxThreads;
  const int warps = threads / 32;
  size_t smem = (size_t)a.nb * 4 + (size_t)(a.nb + 1) * 4 + (size_t)a.nb * 4 + (size_t)warps * words * 4;
  if (a.mode == SA_MASK_LITERAL_MEAN && a.nb <= kPriorMaxBlocks) smem += (size_t)kPriorWarps * (a.nb + 1) * 4;
  if (!(threads == 256 ? mask_smem_ready<256>(smem) : mask_smem_ready<kMaxThreads>(smem))) return SA_ERR_CUDA;
  // rows of a sequence split over up to nb / warps CTAs (one row per warp), enough CTAs in
  // all to cover the GPU twice; each CTA rebuilds the sequence's state, which is cheap
  const int sm_count = current_sm_count();
  const int groups = std::max(1, std::min((a.nb + warps - 1) / warps, (2 * sm_count + a.batch - 1) / a.batch));
  const dim3 grid((unsigned)a.batch, (unsigned)groups);
  if (threads == 256)
    build_mask_kernel<256><<<grid, 256, smem, stream>>>(a);
  else
    build_mask_kernel<kMaxThreads><<<grid, kMaxThreads, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
