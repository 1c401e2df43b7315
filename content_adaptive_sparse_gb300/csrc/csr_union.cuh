// Union of a few consecutive CSR rows, built by one warp in shared memory.
//
// A 128-token tile covers nq = 128 / b consecutive blocks. Its work list is the sorted
// union of those blocks' rows, and each listed block carries one membership bit per tile
// block. The forward and dQ kernels take the union over query-block rows of the block CSR
// (key blocks J with J <= I under causality); the dK / dV kernel takes it over key-block
// rows of the transposed CSR (query blocks I with I >= J under causality).
#pragma once
#include <stdint.h>

#include "sa_internal.h"

namespace sa {

constexpr int kMaxTileBlocks = 4;   // blocks per 128-token tile (b >= 32)

struct UnionSmem {
  uint32_t bm[kMaxTileBlocks][kMaxMaskBlocks / 32];   // 2 KB
  uint16_t list[kMaxMaskBlocks];                      // 8 KB: block | membership << 12
};

// Causal filter of an entry X of tile row r (tile block T0 + r):
//   kKeepAll: none; kKeepLE: X <= T0 + r (key blocks of a query row);
//   kKeepGE: X >= T0 + r (query blocks of a key row).
enum : int { kKeepAll = 0, kKeepLE = 1, kKeepGE = 2 };

// Builds the union of rows T0 .. T0+nq-1 of (rp, ci) into u.list and returns its length.
// Entries outside [0, nb) are skipped and reported in *err (bit err_bit).
static __device__ int build_union(int nb, int keep, UnionSmem& u, const int32_t* rp, const int32_t* ci,
                                 int T0, int nq, unsigned int* err, unsigned int err_bit) {
  const int lane = threadIdx.x & 31;
  const int nw = (nb + 31) >> 5;
  for (int r = 0; r < nq; ++r)
    for (int w = lane; w < nw; w += 32) u.bm[r][w] = 0u;
  const int bnd = (lane <= nq) ? rp[T0 + lane] : 0x7fffffff;   // lane r: start of row r
  int bq[kMaxTileBlocks + 1];
#pragma unroll
  for (int q = 0; q <= kMaxTileBlocks; ++q) bq[q] = __shfl_sync(0xffffffffu, bnd, min(q, nq));
  const int e0 = bq[0];
  const int e1 = bq[kMaxTileBlocks];
  __syncwarp();
  for (int e = e0 + lane; e < e1; e += 32) {
    const int X = ci[e];
    int r = 0;
#pragma unroll
    for (int q = 1; q < kMaxTileBlocks; ++q) r += (q < nq && e >= bq[q]) ? 1 : 0;
    const bool pass = keep == kKeepAll || (keep == kKeepLE ? X <= T0 + r : X >= T0 + r);
    if (X < 0 || X >= nb) {
      atomicOr(err, err_bit);
    } else if (pass) {
      atomicOr(&u.bm[r][X >> 5], 1u << (X & 31));
    }
  }
  __syncwarp();
  int total = 0;
  for (int w0 = 0; w0 < nw; w0 += 32) {
    const int w = w0 + lane;
    uint32_t word[kMaxTileBlocks];
    uint32_t un = 0u;
#pragma unroll
    for (int r = 0; r < kMaxTileBlocks; ++r) {
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
      for (int r = 0; r < kMaxTileBlocks; ++r) mask |= ((word[r] >> j) & 1u) << r;
      u.list[pos++] = (uint16_t)((uint32_t)(w * 32 + j) | (mask << 12));
    }
    total += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
  return total;
}

}  // namespace sa
