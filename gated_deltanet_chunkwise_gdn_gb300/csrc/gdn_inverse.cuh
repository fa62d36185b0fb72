// gdn_inverse.cuh — the one triangular inverse of a 64-token WY block, shared by the forward's
// intra-chunk kernel and the backward's factor kernel.
#pragma once

#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace inv {

// The one triangular inverse: X = (I + L)^{-1} for L strictly lower 64 x 64 (fp32, pitch LDF),
// in 16 x 16 blocks ("Simple math to speed up GDN prefill", section "Save one invert": M^{-1}
// by blocked forward substitution).
//
// Diagonal blocks: X_II = (I + L_II)^{-1} by a column sweep in fp32, one lane per column, two
// blocks per warp (diag_blocks). Off-diagonal blocks by the 2 x 2 block rule on 32-row halves
// [X_A 0; X_CA X_C] with X_CA = -X_C L_CA X_A, every product on the tensor cores as warp-level
// 16 x 8 x 16 MMAs (offdiag_blocks):
//   stage 1 (warps 0, 1):    X_10 = -(X_11 L_10) X_00,   X_32 = -(X_33 L_32) X_22
//   stage 2 (warps 0-3, p, q): Y_p = sum_{m<=p} X_{2+p,2+m} L_{2+m, 0..1}   (row block p of X_C L_CA)
//                              X_{2+p,q} = -sum_{m>=q} Y_{p,m} X_{m,q}
// The left factor of each second product is the first product's accumulator, which is already
// laid out as an A operand, so the intermediates stay in registers. Each fp32 operand is split
// into bf16 hi + lo and a product takes hi*hi + hi*lo + lo*hi (about 16 bits), so the blocks
// come out with the accuracy of the fp32 substitution they replace.

// Warp-level D(16 x 8) += A(16 x 16) B(16 x 8), bf16 operands, fp32 accumulation.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A 16 x 16 operand as bf16 hi + lo fragments (lane: rows lane/4 (+8), column pairs 2(lane%4) (+8)).
struct AFrag {
  uint32_t hi[4], lo[4];
};
// B operand (16 x 16: k rows, two 8-column n tiles) as bf16 hi + lo fragments.
struct BFrag {
  uint32_t hi[2][2], lo[2][2];
};

template <int LD>
__device__ __forceinline__ AFrag load_a(const float* A) {
  const int lane = threadIdx.x & 31, r = lane >> 2, c = 2 * (lane & 3);
  AFrag f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 x = *reinterpret_cast<const float2*>(A + (r + 8 * (u & 1)) * LD + c + 8 * (u >> 1));
    split2<bf16>(x.x, x.y, f.hi[u], f.lo[u]);
  }
  return f;
}
template <int LD>
__device__ __forceinline__ BFrag load_b(const float* B) {
  const int lane = threadIdx.x & 31, n = lane >> 2, k = 2 * (lane & 3);
  BFrag f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float* b = B + (k + 8 * u) * LD + 8 * nt + n;
      split2<bf16>(b[0], b[LD], f.hi[nt][u], f.lo[nt][u]);
    }
  return f;
}
// The accumulator pair of a 16 x 16 product (n tiles 0 and 1) as the A operand of the next one.
__device__ __forceinline__ AFrag acc_as_a(const float (&d)[2][4]) {
  AFrag f;
  split2<bf16>(d[0][0], d[0][1], f.hi[0], f.lo[0]);
  split2<bf16>(d[0][2], d[0][3], f.hi[1], f.lo[1]);
  split2<bf16>(d[1][0], d[1][1], f.hi[2], f.lo[2]);
  split2<bf16>(d[1][2], d[1][3], f.hi[3], f.lo[3]);
  return f;
}
// d (16 x 16, two n tiles) += a b with the three-term split.
__device__ __forceinline__ void mma3(float (&d)[2][4], const AFrag& a, const BFrag& b) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    mma16816(d[nt], a.hi, b.hi[nt][0], b.hi[nt][1]);
    mma16816(d[nt], a.hi, b.lo[nt][0], b.lo[nt][1]);
    mma16816(d[nt], a.lo, b.hi[nt][0], b.hi[nt][1]);
  }
}
template <int LD>
__device__ __forceinline__ void store_neg(float* dst, const float (&d)[2][4]) {
  const int lane = threadIdx.x & 31, r = lane >> 2, c = 2 * (lane & 3);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    *reinterpret_cast<float2*>(dst + r * LD + 8 * nt + c) = make_float2(-d[nt][0], -d[nt][1]);
    *reinterpret_cast<float2*>(dst + (r + 8) * LD + 8 * nt + c) = make_float2(-d[nt][2], -d[nt][3]);
  }
}

// Diagonal blocks 2 w and 2 w + 1 (w = 0, 1): lanes 0-15 and 16-31 each solve one block.
template <int LDF>
__device__ __forceinline__ void diag_blocks(const float* Lf, float* Xf, int w) {
  const int lane = threadIdx.x & 31;
  const int b = 16 * (2 * w + (lane >> 4));
  const int c = lane & 15;
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = i == c ? 1.f : 0.f;
#pragma unroll
  for (int k = 0; k < 15; ++k)  // x_k is final: remove its share from the rows below
#pragma unroll
    for (int i = k + 1; i < 16; ++i) x[i] = fmaf(-Lf[(b + i) * LDF + b + k], x[k], x[i]);
#pragma unroll
  for (int i = 0; i < 16; ++i) Xf[(b + i) * LDF + b + c] = x[i];
}

// Off-diagonal blocks (warps 0-3 work, the others pass straight to the closing barrier); the
// diagonal blocks are in Xf. Ends with a block barrier.
template <int LDF>
__device__ void offdiag_blocks(const float* Lf, float* Xf) {
  const int warp = threadIdx.x >> 5;
  auto blk = [&](const float* M, int I, int J) { return M + 16 * I * LDF + 16 * J; };
  if (warp < 2) {  // stage 1: X_{I,I-1}, I = 1 + 2 warp
    const int I = 1 + 2 * warp;
    float t[2][4] = {}, x[2][4] = {};
    mma3(t, load_a<LDF>(blk(Xf, I, I)), load_b<LDF>(blk(Lf, I, I - 1)));
    mma3(x, acc_as_a(t), load_b<LDF>(blk(Xf, I - 1, I - 1)));
    store_neg<LDF>(Xf + 16 * I * LDF + 16 * (I - 1), x);
  }
  if (warp < 4) {
    tc::named_sync(4, 128);  // X_10 and X_32 are in place
    const int p = warp >> 1, q = warp & 1;
    // Y_{p,m} for m = q..1 (X_{2+p,q} needs Y_{p,q} and Y_{p,1})
    float y[2][2][4] = {};
#pragma unroll
    for (int mm = 0; mm <= p; ++mm) {
      const AFrag a = load_a<LDF>(blk(Xf, 2 + p, 2 + mm));
#pragma unroll
      for (int m = 0; m < 2; ++m)
        if (m >= q) mma3(y[m], a, load_b<LDF>(blk(Lf, 2 + mm, m)));
    }
    float x[2][4] = {};
#pragma unroll
    for (int m = 0; m < 2; ++m)
      if (m >= q) mma3(x, acc_as_a(y[m]), load_b<LDF>(blk(Xf, m, q)));
    store_neg<LDF>(Xf + 16 * (2 + p) * LDF + 16 * q, x);
  }
  __syncthreads();
}

}  // namespace inv
}  // namespace gdn
