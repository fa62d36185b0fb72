// gdn_mma.cuh — warp-level tensor-core products for the backward kernels.
//
// One warp computes a (16 MT) x (8 NT) tile of D += A B with m16n8k16 bf16 MMAs and fp32
// accumulation. Operands are read element by element through accessor functors
// (fa(m, k), fb(k, n) -> float), so one routine serves row-major, transposed and scaled
// views of shared-memory tiles. An fp32 operand is carried as a bf16 pair hi + lo
// (about 16 significant bits) and a product takes hi*hi + hi*lo + lo*hi; an operand whose
// values are bf16 already (the raw bf16 q, k, v, dO tiles) is carried as hi alone, and the
// terms with its lo part drop out. fp16 inputs are carried as pairs too (an fp16 value is
// exactly the sum of two bf16 values).
//
// Fragment layout (lane = 4 r + c/2, r in 0..7, c in {0, 2, 4, 6}):
//   A (16 x 16): a[u] = (row r + 8 (u & 1), columns c + 8 (u >> 1) and +1)
//   B (16 x 8):  b[u] = (rows c + 8 u and +1, column r)
//   D (16 x 8):  d[e] = (row r + 8 (e >> 1), column c + (e & 1))
#pragma once

#include "gdn_common.cuh"

namespace gdn {
namespace wm {

__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ int lane_r() { return (threadIdx.x & 31) >> 2; }
__device__ __forceinline__ int lane_c() { return 2 * (threadIdx.x & 3); }

// x, y -> hi (and lo when SPLIT) as packed bf16 pairs.
template <bool SPLIT>
__device__ __forceinline__ void pack(float x, float y, uint32_t& hi, uint32_t& lo) {
  if (SPLIT) {
    split2<bf16>(x, y, hi, lo);
  } else {
    hi = pack_bf16(x, y);
    lo = 0u;
  }
}

template <bool SPLIT, class FA>
__device__ __forceinline__ void load_a(uint32_t (&hi)[4], uint32_t (&lo)[4], const FA& fa, int m0, int k0) {
  const int r = lane_r(), c = lane_c();
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int m = m0 + r + 8 * (u & 1), k = k0 + c + 8 * (u >> 1);
    pack<SPLIT>(fa(m, k), fa(m, k + 1), hi[u], lo[u]);
  }
}

template <bool SPLIT, class FB>
__device__ __forceinline__ void load_b(uint32_t (&hi)[2], uint32_t (&lo)[2], const FB& fb, int k0, int n0) {
  const int r = lane_r(), c = lane_c();
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int k = k0 + c + 8 * u, n = n0 + r;
    pack<SPLIT>(fb(k, n), fb(k + 1, n), hi[u], lo[u]);
  }
}

// acc[i][j] (the 16 x 8 tile at rows m0 + 16 i, columns n0 + 8 j) += A B over k in [k_lo, k_hi)
// (multiples of 16). AS / BS: the operand carries a lo part.
template <int MT, int NT, bool AS, bool BS, class FA, class FB>
__device__ __forceinline__ void gemm(float (&acc)[MT][NT][4], const FA& fa, const FB& fb, int m0, int n0, int k_lo,
                                     int k_hi) {
  for (int k0 = k_lo; k0 < k_hi; k0 += 16) {
    uint32_t ah[MT][4], al[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) load_a<AS>(ah[i], al[i], fa, m0 + 16 * i, k0);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint32_t bh[2], bl[2];
      load_b<BS>(bh, bl, fb, k0, n0 + 8 * j);
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        mma(acc[i][j], ah[i], bh);
        if (BS) mma(acc[i][j], ah[i], bl);
        if (AS) mma(acc[i][j], al[i], bh);
      }
    }
  }
}

template <int MT, int NT>
__device__ __forceinline__ void zero(float (&acc)[MT][NT][4]) {
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
}

// f(row, col, value&) for every accumulator element of the thread.
template <int MT, int NT, class F>
__device__ __forceinline__ void for_each(float (&acc)[MT][NT][4], int m0, int n0, const F& f) {
  const int r = lane_r(), c = lane_c();
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) f(m0 + 16 * i + r + 8 * (e >> 1), n0 + 8 * j + c + (e & 1), acc[i][j][e]);
}

// f(row, col, x0&, x1&) for the element pairs (row, col), (row, col + 1) of the thread.
template <int MT, int NT, class F>
__device__ __forceinline__ void for_each_pair(float (&acc)[MT][NT][4], int m0, int n0, const F& f) {
  const int r = lane_r(), c = lane_c();
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) f(m0 + 16 * i + r + 8 * h, n0 + 8 * j + c, acc[i][j][2 * h], acc[i][j][2 * h + 1]);
}

// ---- fragments straight from 16-bit planes in shared memory (ldmatrix). A plane holds an
// operand's bf16 values (the hi part of an fp32 operand, or its lo part) with a row pitch of
// ld elements (a multiple of 8, so that every row start is 16-byte aligned).

// A (16 x 16) at (m0, k0) from [m][k] storage.
__device__ __forceinline__ void lda(uint32_t (&a)[4], const bf16* base, int ld, int m0, int k0) {
  const int l = threadIdx.x & 31;
  const uint32_t addr = smem_u32(base + (m0 + (l & 15)) * ld + k0 + 8 * (l >> 4));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]) : "r"(addr));
}
// A (16 x 16) at (m0, k0) from [k][m] storage (A^T row-major).
__device__ __forceinline__ void lda_t(uint32_t (&a)[4], const bf16* base, int ld, int m0, int k0) {
  const int l = threadIdx.x & 31, mat = l >> 3;
  const uint32_t addr = smem_u32(base + (k0 + (l & 7) + 8 * (mat >> 1)) * ld + m0 + 8 * (mat & 1));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]) : "r"(addr));
}
// B for the two 8-column tiles n0 and n0 + 8 (b[0..1]: tile n0, b[2..3]: tile n0 + 8) at k0,
// from [n][k] storage (B^T row-major).
__device__ __forceinline__ void ldb2(uint32_t (&b)[4], const bf16* base, int ld, int k0, int n0) {
  const int l = threadIdx.x & 31, mat = l >> 3;
  const uint32_t addr = smem_u32(base + (n0 + (l & 7) + 8 * (mat >> 1)) * ld + k0 + 8 * (mat & 1));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]) : "r"(addr));
}
// The same from [k][n] storage.
__device__ __forceinline__ void ldb2_t(uint32_t (&b)[4], const bf16* base, int ld, int k0, int n0) {
  const int l = threadIdx.x & 31, mat = l >> 3;
  const uint32_t addr = smem_u32(base + (k0 + (l & 7) + 8 * (mat & 1)) * ld + n0 + 8 * (mat >> 1));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]) : "r"(addr));
}
// B for one 8-column tile n0 at k0, from [n][k] / [k][n] storage (lanes 16-31 repeat 0-15).
__device__ __forceinline__ void ldb1(uint32_t (&b)[2], const bf16* base, int ld, int k0, int n0) {
  const int l = threadIdx.x & 15;
  const uint32_t addr = smem_u32(base + (n0 + (l & 7)) * ld + k0 + 8 * (l >> 3));
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(b[0]), "=r"(b[1]) : "r"(addr));
}
__device__ __forceinline__ void ldb1_t(uint32_t (&b)[2], const bf16* base, int ld, int k0, int n0) {
  const int l = threadIdx.x & 15;
  const uint32_t addr = smem_u32(base + (k0 + l) * ld + n0);
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(b[0]), "=r"(b[1]) : "r"(addr));
}

// MMA terms of one product: hi*hi, hi*lo (B has lo), lo*hi (A has lo). bh, bl: two registers each.
template <bool AL, bool BL>
__device__ __forceinline__ void mma_terms(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                          const uint32_t* bh, const uint32_t* bl) {
  const uint32_t b0[2] = {bh[0], bh[1]};
  mma(d, ah, b0);
  if (BL) {
    const uint32_t b1[2] = {bl[0], bl[1]};
    mma(d, ah, b1);
  }
  if (AL) mma(d, al, b0);
}

// acc[i][j] (the 16 x 8 tile at rows m0 + 16 i, columns n0 + 8 j) += A B over k in [k_lo, k_hi), both
// operands from bf16 planes through ldmatrix. A: planes ah (+ al when AL) in [m][k] storage, or
// [k][m] when AKM; B: planes bh (+ bl when BL) in [n][k] storage, or [k][n] when BKN. NT even.
template <int MT, int NT, bool AKM, bool BKN, bool AL, bool BL>
__device__ __forceinline__ void pgemm(float (&acc)[MT][NT][4], const bf16* ah, const bf16* al, int lda_,
                                      const bf16* bh, const bf16* bl, int ldb_, int m0, int n0, int k_lo,
                                      int k_hi) {
  static_assert(NT % 2 == 0, "B fragments are loaded two tiles at a time");
  for (int k0 = k_lo; k0 < k_hi; k0 += 16) {
    uint32_t a_h[MT][4], a_l[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      if (AKM) lda_t(a_h[i], ah, lda_, m0 + 16 * i, k0); else lda(a_h[i], ah, lda_, m0 + 16 * i, k0);
      if (AL) {
        if (AKM) lda_t(a_l[i], al, lda_, m0 + 16 * i, k0); else lda(a_l[i], al, lda_, m0 + 16 * i, k0);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; j += 2) {
      uint32_t b_h[4], b_l[4];
      if (BKN) ldb2_t(b_h, bh, ldb_, k0, n0 + 8 * j); else ldb2(b_h, bh, ldb_, k0, n0 + 8 * j);
      if (BL) {
        if (BKN) ldb2_t(b_l, bl, ldb_, k0, n0 + 8 * j); else ldb2(b_l, bl, ldb_, k0, n0 + 8 * j);
      }
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        mma_terms<AL, BL>(acc[i][j], a_h[i], a_l[i], b_h, b_l);
        mma_terms<AL, BL>(acc[i][j + 1], a_h[i], a_l[i], b_h + 2, b_l + 2);
      }
    }
  }
}

// hi + lo of the planes at offset off (lo plane `plane` elements after hi).
__device__ __forceinline__ float plane_val(const bf16* hi, int64_t off, int64_t plane) {
  return __bfloat162float(hi[off]) + __bfloat162float(hi[off + plane]);
}

// (x0, x1) (fp32) as bf16 pairs hi + lo, stored to two planes (4-byte aligned).
__device__ __forceinline__ void store_split2(bf16* hi, bf16* lo, float x0, float x1) {
  uint32_t h, l;
  split2<bf16>(x0, x1, h, l);
  *reinterpret_cast<uint32_t*>(hi) = h;
  *reinterpret_cast<uint32_t*>(lo) = l;
}

}  // namespace wm
}  // namespace gdn
