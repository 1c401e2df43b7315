// Warp-level mma.sync (m16n8k16, bf16 -> f32) fragment helpers for the token-granular
// offset kernels: K and V rows are 128-byte (64 x bf16) rows of shared-memory tiles written
// by TMA with the 128-byte swizzle (tile bases 1024-byte aligned); one warp owns 16 query
// rows, lane (g, t) holding rows g and g + 8.
#pragma once
#include <stdint.h>

namespace sa {
namespace frag {

constexpr uint32_t kOnesBf16x2 = 0x3f803f80u;   // (1.0, 1.0) in bf16

// 128B swizzle of a tile of 128-byte rows: 16-byte chunk c of row r.
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
  return base + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
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

// The QK contraction runs over the head dimension in a permuted order: in k-step ks,
// fragment slot j (0: k = 2t, 2t+1; 1: k = 2t+8, 2t+9) of lane (g, t) holds the physical
// dimensions 16t + 4ks + 2j + {0, 1}. A dot product does not depend on the order of its
// terms, and with this order every lane's Q and K operands are the 32 contiguous bytes
// [16t, 16t + 16) of a row: plain 16-byte loads instead of ldmatrix.
// K operand of one 8-key n-tile: the lane's 32 bytes of key row `row` of a swizzled tile.
__device__ __forceinline__ void load_kfrag(uint32_t tile, int row, int t, uint32_t (&u)[8]) {
  const uint4 a = lds128(swz(tile, row, 2 * t)), b = lds128(swz(tile, row, 2 * t + 1));
  u[0] = a.x; u[1] = a.y; u[2] = a.z; u[3] = a.w;
  u[4] = b.x; u[5] = b.y; u[6] = b.z; u[7] = b.w;
}

// 16 x 8 scores of one n-tile: d = Q (16 x 64) . K^T (64 x 8).
__device__ __forceinline__ void qk_ntile(float* d, const uint32_t (&qa)[4][4], const uint32_t (&u)[8]) {
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) mma16816(d, qa[ks], u[2 * ks], u[2 * ks + 1]);
}

// B fragments (transposed) of 16 key rows x 64 dims of V: vb[nt2][*] covers d n-tiles
// 2*nt2 and 2*nt2+1 for the 16 keys.
__device__ __forceinline__ void load_v16(uint32_t tile, int row0, int lane, uint32_t (&vb)[4][4]) {
  // matrices: (keys 0-7, d chunk c), (keys 8-15, d chunk c), (keys 0-7, chunk c+1), (keys 8-15, chunk c+1)
  const int r = row0 + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int cc = lane >> 4;
#pragma unroll
  for (int nt2 = 0; nt2 < 4; ++nt2) ldsm_x4_t(swz(tile, r, 2 * nt2 + cc), vb[nt2][0], vb[nt2][1], vb[nt2][2], vb[nt2][3]);
}

__device__ __forceinline__ void pv_16(float (&o)[8][4], const uint32_t* pa, const uint32_t (&vb)[4][4]) {
#pragma unroll
  for (int nt2 = 0; nt2 < 4; ++nt2) {
    mma16816(o[2 * nt2], pa, vb[nt2][0], vb[nt2][1]);
    mma16816(o[2 * nt2 + 1], pa, vb[nt2][2], vb[nt2][3]);
  }
}

// Raw diagonal scores of query rows g and g+8 against key rows row0 + g and row0 + 8 + g
// of a swizzled tile (all lanes of the quad receive them).
__device__ __forceinline__ void diag_scores(uint32_t kt, int row0, int g, int t, int hl, int e_sel,
                                            const uint32_t (&qa)[4][4], float& s_lo, float& s_hi) {
  uint32_t u0[8], u1[8];
  load_kfrag(kt, row0 + g, t, u0);
  load_kfrag(kt, row0 + 8 + g, t, u1);
  float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
  qk_ntile(d0, qa, u0);
  qk_ntile(d1, qa, u1);
  // query row g meets key row g at fragment column g: n-tile 0, lane t = g/2, element g%2
  s_lo = __shfl_sync(0xffffffffu, e_sel ? d0[1] : d0[0], hl);
  s_hi = __shfl_sync(0xffffffffu, e_sel ? d1[3] : d1[2], hl);
}

// O += P_diag V for the 16 value rows row0 .. row0 + 15 of a swizzled tile (query row r
// takes value row row0 + r); pb = bf16 bits (p_lo | p_hi << 16) of this quad's rows.
__device__ __forceinline__ void diag_pv(uint32_t vt, int row0, int lane, bool holder, int e_sel, uint32_t pb,
                                        float (&o)[8][4]) {
  uint32_t pa[4];
  pa[0] = holder ? (e_sel ? (pb << 16) : (pb & 0xffffu)) : 0u;
  pa[1] = 0u;
  pa[2] = 0u;
  pa[3] = holder ? (e_sel ? (pb & 0xffff0000u) : (pb >> 16)) : 0u;
  uint32_t vb[4][4];
  load_v16(vt, row0, lane, vb);
  pv_16(o, pa, vb);
}

}  // namespace frag
}  // namespace sa
