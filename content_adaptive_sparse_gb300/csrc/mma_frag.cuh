// Warp-level mma.sync (m16n8k16, bf16 -> f32) fragment helpers for the token-granular
// offset kernels, for head dimensions D = 32, 64 and 128. One warp owns 16 query rows, lane
// (g, t) holding rows g and g + 8.
//
// K and V rows in shared memory, as TMA writes them (KV: tile base and, for D = 128, the
// distance between its two column chunks):
//   D = 64:  128-byte rows with the 128-byte swizzle (tile base 1024-byte aligned);
//   D = 128: two column chunks (dimensions 0-63, then 64-127), each a tile of 128-byte rows with
//            the 128-byte swizzle, the second `cstride` bytes after the first;
//   D = 32:  64-byte rows, no swizzle.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace sa {
namespace frag {

constexpr uint32_t kOnesBf16x2 = 0x3f803f80u;   // (1.0, 1.0) in bf16

struct KV {
  uint32_t base;      // shared-memory address of row 0
  uint32_t cstride;   // D = 128: bytes from the first column chunk to the second
};

// 128B swizzle of a tile of 128-byte rows: 16-byte chunk c of row r.
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
  return base + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Address of 16-byte unit u (dimensions 8u .. 8u + 7) of row r.
template <int D>
__device__ __forceinline__ uint32_t unit_addr(KV tile, int r, int u) {
  static_assert(D == 32 || D == 64 || D == 128, "head dimension");
  if constexpr (D == 32) {
    return tile.base + (uint32_t)(r * 64 + u * 16);
  } else if constexpr (D == 64) {
    return swz(tile.base, r, u);
  } else {
    return swz(tile.base + (uint32_t)(u >> 3) * tile.cstride, r, u & 7);
  }
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// D += A (16x16 bf16, row) * B (16x8 bf16, col), f32 accumulate.
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The QK contraction runs over the head dimension in a permuted order: in k-step ks (of D / 16),
// fragment slot j (0: k = 2t, 2t+1; 1: k = 2t+8, 2t+9) of lane (g, t) holds the physical
// dimensions t D/4 + 4ks + 2j + {0, 1}. A dot product does not depend on the order of its
// terms, and with this order every lane's Q and K operands are the D/2 contiguous bytes
// [t D/4, (t+1) D/4) of a row: plain 16-byte loads instead of ldmatrix.
template <int D>
struct Frag {
  static constexpr int KS = D / 16;       // k-steps of the QK contraction
  static constexpr int NT = D / 8;        // 8-column n-tiles of O
  static constexpr int UNITS = D / 32;    // 16-byte units of a lane's slice of a row
};

// Q operand of one 16-query m-tile from global memory: rows lo (g) and hi (g + 8), each a
// pointer to the row's dimension 0.
template <int D>
__device__ __forceinline__ void load_qfrag(const __nv_bfloat16* row_lo, const __nv_bfloat16* row_hi, int t,
                                           uint32_t (&qa)[Frag<D>::KS][4]) {
  constexpr int U = Frag<D>::UNITS;
  const uint4* lo = reinterpret_cast<const uint4*>(row_lo + t * (D / 4));
  const uint4* hi = reinterpret_cast<const uint4*>(row_hi + t * (D / 4));
  uint32_t wl[4 * U], wh[4 * U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint4 a = __ldg(lo + u), b = __ldg(hi + u);
    wl[4 * u] = a.x; wl[4 * u + 1] = a.y; wl[4 * u + 2] = a.z; wl[4 * u + 3] = a.w;
    wh[4 * u] = b.x; wh[4 * u + 1] = b.y; wh[4 * u + 2] = b.z; wh[4 * u + 3] = b.w;
  }
#pragma unroll
  for (int ks = 0; ks < Frag<D>::KS; ++ks) {
    qa[ks][0] = wl[2 * ks];
    qa[ks][1] = wh[2 * ks];
    qa[ks][2] = wl[2 * ks + 1];
    qa[ks][3] = wh[2 * ks + 1];
  }
}

// K operand of one 8-key n-tile: the lane's D/2 bytes of key row `row`.
template <int D>
__device__ __forceinline__ void load_kfrag(KV tile, int row, int t, uint32_t (&u)[2 * Frag<D>::KS]) {
  constexpr int U = Frag<D>::UNITS;
#pragma unroll
  for (int i = 0; i < U; ++i) {
    const uint4 a = lds128(unit_addr<D>(tile, row, t * U + i));
    u[4 * i] = a.x; u[4 * i + 1] = a.y; u[4 * i + 2] = a.z; u[4 * i + 3] = a.w;
  }
}

// 16 x 8 scores of one n-tile: d = Q (16 x D) . K^T (D x 8).
template <int D>
__device__ __forceinline__ void qk_ntile(float* d, const uint32_t (&qa)[Frag<D>::KS][4],
                                         const uint32_t (&u)[2 * Frag<D>::KS]) {
#pragma unroll
  for (int ks = 0; ks < Frag<D>::KS; ++ks) mma16816(d, qa[ks], u[2 * ks], u[2 * ks + 1]);
}

// B fragments (transposed) of 16 key rows x D dims of V: vb[nt2][*] covers O n-tiles 2*nt2
// and 2*nt2+1 for the 16 keys.
template <int D>
__device__ __forceinline__ void load_v16(KV tile, int row0, int lane, uint32_t (&vb)[D / 16][4]) {
  // matrices: (keys 0-7, unit c), (keys 8-15, unit c), (keys 0-7, unit c+1), (keys 8-15, unit c+1)
  const int r = row0 + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int cc = lane >> 4;
#pragma unroll
  for (int nt2 = 0; nt2 < D / 16; ++nt2)
    ldsm_x4_t(unit_addr<D>(tile, r, 2 * nt2 + cc), vb[nt2][0], vb[nt2][1], vb[nt2][2], vb[nt2][3]);
}

template <int D>
__device__ __forceinline__ void pv_16(float (&o)[Frag<D>::NT][4], const uint32_t* pa, const uint32_t (&vb)[D / 16][4]) {
#pragma unroll
  for (int nt2 = 0; nt2 < D / 16; ++nt2) {
    mma16816(o[2 * nt2], pa, vb[nt2][0], vb[nt2][1]);
    mma16816(o[2 * nt2 + 1], pa, vb[nt2][2], vb[nt2][3]);
  }
}

// Raw diagonal scores of query rows g and g+8 against key rows row0 + g and row0 + 8 + g
// of a tile (all lanes of the quad receive them).
template <int D>
__device__ __forceinline__ void diag_scores(KV kt, int row0, int g, int t, int hl, int e_sel,
                                            const uint32_t (&qa)[Frag<D>::KS][4], float& s_lo, float& s_hi) {
  uint32_t u0[2 * Frag<D>::KS], u1[2 * Frag<D>::KS];
  load_kfrag<D>(kt, row0 + g, t, u0);
  load_kfrag<D>(kt, row0 + 8 + g, t, u1);
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
  qk_ntile<D>(d0, qa, u0);
  qk_ntile<D>(d1, qa, u1);
  // query row g meets key row g at fragment column g: n-tile 0, lane t = g/2, element g%2
  s_lo = __shfl_sync(0xffffffffu, e_sel ? d0[1] : d0[0], hl);
  s_hi = __shfl_sync(0xffffffffu, e_sel ? d1[3] : d1[2], hl);
}

// O += P_diag V for the 16 value rows row0 .. row0 + 15 of a tile (query row r takes value
// row row0 + r); pb = bf16 bits (p_lo | p_hi << 16) of this quad's rows.
template <int D>
__device__ __forceinline__ void diag_pv(KV vt, int row0, int lane, bool holder, int e_sel, uint32_t pb,
                                        float (&o)[Frag<D>::NT][4]) {
  uint32_t pa[4];
  pa[0] = holder ? (e_sel ? (pb << 16) : (pb & 0xffffu)) : 0u;
  pa[1] = 0u;
  pa[2] = 0u;
  pa[3] = holder ? (e_sel ? (pb & 0xffff0000u) : (pb >> 16)) : 0u;
  uint32_t vb[D / 16][4];
  load_v16<D>(vt, row0, lane, vb);
  pv_16<D>(o, pa, vb);
}

}  // namespace frag
}  // namespace sa
