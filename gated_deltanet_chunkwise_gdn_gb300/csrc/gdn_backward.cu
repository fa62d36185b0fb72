// gdn_backward.cu — the chunkwise backward pass of the GDN prefill.
//
// It differentiates the forward of gdn_extend_chunkwise,
//   q^ = q / sqrt(|q|^2 + eps), k^ likewise, log alpha = -exp(A_log) softplus(a + dt_bias),
//   beta = sigmoid(b), S_t = alpha_t S_{t-1} (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T,
//   o_t = scale S_t q^_t
// ("Simple math to speed up GDN prefill", section "Reminder"; pymllm page
// "pymllm.layers.attention.gdn_chunkwise", Parameters), for the scalar
//   L = sum_t <dO_t, o_t> + sum_chains <dS_final, S_final>,
// so besides the output's gradient it takes the gradient arriving at each final state, the
// incoming state gradient of the bottom-level backward in "nrm-training-kernels", section
// "Kernel". The pages print no gradient formulas: what follows is the chain rule applied to
// the chunkwise WY form of the forward (notation of gdn_common.cuh), chunk by chunk.
//
// Per chunk (rows = its C tokens), with S_in the state entering it and dS_out the gradient of
// the state leaving it:
//   forward:  U = U~ - W<- S_in^T,  O = scale (diag(e^g) Q^ S_in^T + P U),
//             S_out = e^{g_C} S_in + U^T K->,  K-> = diag(e^{g_C - g}) K^
//   reverse:  dU = scale P^T dO + K-> dS_out^T
//             dS_in = e^{g_C} dS_out + scale dO^T diag(e^g) Q^ - dU^T W<-
// and then, per chunk and independently of the others, the gradients through P, W<-, U~,
// A = (Gamma . M^{-1}) diag(beta), the one inverse M^{-1} (dM = -M^{-T} dM^{-1} M^{-T},
// kept strictly lower), the decays Gamma and e^g, the gates and the normalisation.
//
// Kernels, in launch order (after the forward's schedule and gates kernels):
//   factor   per (chunk, value head): 1/|q|, 1/|k|, M^{-1}, P, W<-, U~     (parallel)
//   state    per (chain, block of 16 state rows): S_in of every chunk, U    (sequential in chunks)
//   dstate   per (chain, block of 16 state rows): dS_out of every chunk, dU, dS_0 (sequential, reversed)
//   sgrad    per (chunk, value head, half of the key columns): scale e^g (dO S_in), -dU S_in, U dS_out,
//            e^{g_C} <dS_out, S_in>
//   local    per (chunk, value head): dv, db, da, the gradients of q^ and k^ (through the norm when no
//            value heads share a q/k head)
//   norm     per (token, q/k head), grouped heads only: the group's gradients of q^, k^ summed, through
//            the norm
//   gate_sum per value head: dA_log and ddt_bias, summed over tokens in a fixed order
// The state rows are independent in both sequential passes (the contractions run over the key
// dimension and the chunk's tokens), so their CTAs split the value dimension; in each CTA eight
// warps run the chunk step and eight fetch the next chunk's tiles and write the per-chunk
// outputs. Every product runs on the tensor cores as warp-level m16n8k16 MMAs (gdn_mma.cuh) with
// fp32 operands carried as bf16 hi + lo pairs, so the backward keeps about fp32 accuracy. The
// intermediates that later products consume are stored as such pairs (two bf16 planes in the
// bytes of fp32) and loaded by ldmatrix; the rest are fp32. Every sum is taken in a fixed order,
// so the results are deterministic.
#include <type_traits>

#include "gdn_backward.cuh"
#include "gdn_inverse.cuh"
#include "gdn_mma.cuh"

namespace gdn {

BwdLayout make_bwd_layout(int64_t T, int B, int H, int HV, int D) {
  (void)H;
  constexpr int C = 64;
  BwdLayout L{};
  const int64_t mc = T / C + B + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t per = (size_t)mc * HV;  // (chunk, value head) items
  L.max_chunks = mc;
  L.status = take(64 * sizeof(int32_t));
  L.seq_chunk_off = take((size_t)(B + 1) * sizeof(int32_t));
  L.order = take((size_t)(B > 0 ? B : 1) * sizeof(int32_t));
  L.chunk_tab = take((size_t)mc * sizeof(int4));
  L.g = take(per * C * sizeof(float));
  L.beta = take(per * C * sizeof(float));
  L.rq = take(per * C * sizeof(float));
  L.rk = take(per * C * sizeof(float));
  L.minv = take(per * C * C * sizeof(float));
  L.pm = take(per * 2 * C * C * sizeof(bf16));
  L.w = take(per * 2 * C * D * sizeof(bf16));
  L.ut = take(per * C * D * sizeof(float));
  L.s_in = take(per * D * D * sizeof(float));
  L.u = take(per * C * D * sizeof(float));
  L.ds_out = take(per * D * D * sizeof(float));
  L.du = take(per * C * D * sizeof(float));
  L.dqa = take(per * C * D * sizeof(float));
  L.dw = take(per * C * D * sizeof(float));
  L.dkr = take(per * C * D * sizeof(float));
  L.dgc = take(per * 2 * sizeof(float));
  // gradients of q^, k^ per value head: only with grouped heads (otherwise the local kernel
  // applies the normalisation's backward itself)
  const size_t per_head_grads = HV != H ? (size_t)T * HV * D * sizeof(float) : 0;
  L.dqh = take(per_head_grads);
  L.dkh = take(per_head_grads);
  L.dlala = take((size_t)T * HV * sizeof(float));
  L.total = off;
  return L;
}

namespace {

constexpr int C = 64;   // WY block (tokens per chunk)
constexpr int VB = 16;  // state rows per CTA of the sequential passes
constexpr int kSeqThreads = 256;  // 8 warps per CTA of the sequential passes
constexpr int kLocalThreads = 512;  // 16 warps per CTA of the bf16 local kernel
constexpr int NCW = 4;  // its column warps per 16-row block
constexpr int CP = C + 4;   // pitch (floats) of C x C fp32 tiles
constexpr int UP = VB + 4;  // pitch (floats) of C x VB fp32 tiles

template <typename E>
constexpr bool kSplitSrc = std::is_same<E, f16>::value;  // fp16 tiles enter the MMAs as bf16 pairs

__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(f16 x) { return __half2float(x); }

__device__ __forceinline__ void cp_async_16z(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(valid ? 16 : 0));
}

// f(i, q) for every (row i < ROWS, 16-byte piece q < PER) of a tile, spread over NTHR threads. A
// thread keeps one piece column and steps through rows NTHR / PER apart, so the loop unrolls and the
// row addresses reduce to one base plus constant strides.
template <int ROWS, int PER, int NTHR, class F>
__device__ __forceinline__ void for_pieces(int tid, const F& f) {
  static_assert(NTHR % PER == 0, "a thread keeps its piece column");
  constexpr int RP = NTHR / PER;  // rows per sweep of all threads
  const int q = tid % PER, i0 = tid / PER;
#pragma unroll
  for (int m = 0; m < (ROWS + RP - 1) / RP; ++m) {
    const int i = i0 + m * RP;
    if (ROWS % RP != 0 && i >= ROWS) break;
    f(i, q);
  }
}

// Token rows t0 .. t0 + C - 1 of a [T][heads][D] 16-bit array (head offset folded into src, row
// stride ld elements) into smem rows of pitch D + 8 elements; rows at or past len are zero-filled.
template <int D, int NTHR, typename E>
__device__ __forceinline__ void load_tokens(E* dst, const E* src, int64_t ld, int64_t t0, int len, int tid) {
  constexpr int DP = D + 8;
  const E* base = src + t0 * ld;
  for_pieces<C, D / 8, NTHR>(tid, [&](int i, int q) {
    const bool ok = i < len;
    cp_async_16z(dst + i * DP + q * 8, base + (ok ? i * ld : 0) + q * 8, ok);
  });
}
// Column block [c0, c0 + W) of the same rows (W a multiple of 8, c0 folded into src), pitch WP elements.
template <int W, int WP, int NTHR, typename E>
__device__ __forceinline__ void load_tokens_cols(E* dst, const E* src, int64_t ld, int64_t t0, int len, int tid) {
  const E* base = src + t0 * ld;
  for_pieces<C, W / 8, NTHR>(tid, [&](int i, int q) {
    const bool ok = i < len;
    cp_async_16z(dst + i * WP + q * 8, base + (ok ? i * ld : 0) + q * 8, ok);
  });
}
// ROWS x W fp32 (W a multiple of 4) from a row-major array of row stride ld floats, pitch LD.
template <int W, int LD, int ROWS, int NTHR>
__device__ __forceinline__ void load_f32(float* dst, const float* src, int64_t ld, int tid) {
  for_pieces<ROWS, W / 4, NTHR>(tid, [&](int i, int q) { cp_async_16(dst + i * LD + q * 4, src + i * ld + q * 4); });
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
// Sum over the four lanes of a fragment row (lanes 4 r .. 4 r + 3).
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}
// Sum over the eight fragment rows of a lane column (lanes c/2, c/2 + 4, ..., c/2 + 28).
__device__ __forceinline__ float col_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  x += __shfl_xor_sync(0xffffffffu, x, 16);
  return x;
}

__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

// A chunk's decay factor e^{g_i - g_c} (argument <= 0) by the SFU's base-2 exponential, relative error
// about 2^-22 (the argument is rounded once when scaled by log2(e)).
__device__ __forceinline__ float decay(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
  return y;
}

// Splits an fp16 token tile (rows x W, pitch P) in place into bf16 planes: the hi plane
// overwrites the tile, the lo plane goes to `lo` (same pitch).
template <int W, int P>
__device__ __forceinline__ void split_inplace(f16* tile, bf16* lo, int rows, int tid, int nthr) {
  for (int e = tid; e < rows * W / 2; e += nthr) {
    const int i = e / (W / 2), c = (e % (W / 2)) * 2;
    const float x0 = __half2float(tile[i * P + c]), x1 = __half2float(tile[i * P + c + 1]);
    wm::store_split2(reinterpret_cast<bf16*>(tile) + i * P + c, lo + i * P + c, x0, x1);
  }
}
template <int W, int P>
__device__ __forceinline__ void split_inplace(bf16*, bf16*, int, int, int) {}

// ----------------------------------------------------------------------------- factor

// ROWS x W bf16 plane rows (W a multiple of 8) from a row-major array of row stride ld, pitch P.
template <int W, int P, int ROWS, int NTHR>
__device__ __forceinline__ void load_rows(bf16* dst, const bf16* src, int64_t ld, int tid) {
  for_pieces<ROWS, W / 8, NTHR>(tid, [&](int i, int q) { cp_async_16(dst + i * P + q * 8, src + i * ld + q * 8); });
}

template <int D, bool XS>
struct FacSmem {
  static constexpr int DP = D + 8, PP = C + 8;
  static constexpr uint32_t TILE = C * DP * 2;
  static constexpr uint32_t PAIR = 2 * C * PP * 2;   // hi, lo planes of a C x C operand
  static constexpr uint32_t Q = 0;                   // q, k, v tiles (fp16: their hi planes after the split)
  static constexpr uint32_t K = Q + TILE;
  static constexpr uint32_t V = K + TILE;
  static constexpr uint32_t QL = V + TILE;           // fp16 only: lo planes of q, k, v
  static constexpr uint32_t L = QL + (XS ? 3 * TILE : 0);  // fp32 [C][CP] beta k^_i . k^_j (j < i); then A planes
  static constexpr uint32_t X = L + PAIR;            // fp32 [C][CP]: M^{-1}
  static constexpr uint32_t AW = X + PAIR;           // planes of A diag(e^g / |k|)
  static constexpr uint32_t VEC = AW + PAIR;         // g, beta, 1/|q|, 1/|k|, e^g/|k|
  static constexpr uint32_t bytes = VEC + 5 * C * 4;
  static_assert(C * CP * 4 <= PAIR, "the fp32 C x C tiles fit the plane-pair regions");
};

template <int D, typename E>
__global__ void __launch_bounds__(256) bwd_factor_kernel(BwdParams p) {
  constexpr bool XS = kSplitSrc<E>;
  using S = FacSmem<D, XS>;
  constexpr int DP = S::DP, PP = S::PP, PLN = C * PP;
  extern __shared__ __align__(128) unsigned char smem[];
  if (p.status[0] != GDN_OK) return;
  const int j = blockIdx.x, hv = blockIdx.y;
  if (j >= p.status[1]) return;
  const int4 ct = p.chunk_tab[j];
  const int64_t t0 = ct.y;
  const int len = ct.z;
  const int h = hv / (p.HV / p.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  E* sq = reinterpret_cast<E*>(smem + S::Q);
  E* sk = reinterpret_cast<E*>(smem + S::K);
  E* sv = reinterpret_cast<E*>(smem + S::V);
  bf16* ql = reinterpret_cast<bf16*>(smem + S::QL);
  bf16* kl = ql + C * DP;
  bf16* vl = kl + C * DP;
  float* sL = reinterpret_cast<float*>(smem + S::L);
  float* sX = reinterpret_cast<float*>(smem + S::X);
  bf16* sA = reinterpret_cast<bf16*>(smem + S::L);
  bf16* sAW = reinterpret_cast<bf16*>(smem + S::AW);
  float* vg = reinterpret_cast<float*>(smem + S::VEC);
  float* vb = vg + C;
  float* vrq = vb + C;
  float* vrk = vrq + C;
  float* vek = vrk + C;

  load_tokens<D, 256>(sq, static_cast<const E*>(p.q) + (int64_t)h * D, (int64_t)p.H * D, t0, len, tid);
  load_tokens<D, 256>(sk, static_cast<const E*>(p.k) + (int64_t)h * D, (int64_t)p.H * D, t0, len, tid);
  load_tokens<D, 256>(sv, static_cast<const E*>(p.v) + (int64_t)hv * D, (int64_t)p.HV * D, t0, len, tid);
  cp_async_commit();
  const int64_t item = (int64_t)j * p.HV + hv;
  if (tid < C) {
    vg[tid] = p.g[item * C + tid];
    vb[tid] = p.beta[item * C + tid];
  }
  cp_async_wait<0>();
  __syncthreads();
  if (XS) {
    split_inplace<D, DP>(sq, ql, C, tid, 256);
    split_inplace<D, DP>(sk, kl, C, tid, 256);
    split_inplace<D, DP>(sv, vl, C, tid, 256);
    __syncthreads();
  }
  const bf16* qh = reinterpret_cast<const bf16*>(sq);
  const bf16* kh = reinterpret_cast<const bf16*>(sk);
  const bf16* vh = reinterpret_cast<const bf16*>(sv);
  auto val = [&](const bf16* hi, const bf16* lo, int o) {
    return XS ? __bfloat162float(hi[o]) + __bfloat162float(lo[o]) : __bfloat162float(hi[o]);
  };

  for (int i = warp * 8; i < warp * 8 + 8; ++i) {  // row norms, one warp per 8 rows
    float s2q = 0.f, s2k = 0.f;
    for (int d = lane; d < D; d += 32) {
      const float x = val(qh, ql, i * DP + d), y = val(kh, kl, i * DP + d);
      s2q = fmaf(x, x, s2q);
      s2k = fmaf(y, y, s2k);
    }
    s2q = warp_sum(s2q);
    s2k = warp_sum(s2k);
    if (lane == 0) {
      vrq[i] = i < len ? 1.f / sqrtf(s2q + kNormEps) : 0.f;
      vrk[i] = i < len ? 1.f / sqrtf(s2k + kNormEps) : 0.f;
    }
  }
  __syncthreads();
  if (tid < C) {
    p.rq[item * C + tid] = vrq[tid];
    p.rk[item * C + tid] = vrk[tid];
    vek[tid] = expf(vg[tid]) * vrk[tid];
  }

  // K K^T and Q K^T (C x C): warp tile rows m0 .. m0 + 15, columns n0 .. n0 + 31
  const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
  {
    float kk[1][4][4], qk[1][4][4];
    wm::zero(kk);
    wm::zero(qk);
    wm::pgemm<1, 4, false, false, XS, XS>(kk, kh, kl, DP, kh, kl, DP, m0, n0, 0, D);
    wm::pgemm<1, 4, false, false, XS, XS>(qk, qh, ql, DP, kh, kl, DP, m0, n0, 0, D);
    wm::for_each(kk, m0, n0, [&](int i, int c, float& x) {
      sL[i * CP + c] = c < i ? vb[i] * vrk[i] * vrk[c] * x : 0.f;
    });
    bf16* P = reinterpret_cast<bf16*>(p.pm) + item * 2 * C * C;  // hi, lo planes
    wm::for_each_pair(qk, m0, n0, [&](int i, int c, float& x0, float& x1) {
      const float y0 = c <= i ? decay(vg[i] - vg[c]) * vrq[i] * vrk[c] * x0 : 0.f;
      const float y1 = c + 1 <= i ? decay(vg[i] - vg[c + 1]) * vrq[i] * vrk[c + 1] * x1 : 0.f;
      wm::store_split2(P + i * C + c, P + C * C + i * C + c, y0, y1);
    });
  }
  __syncthreads();

  // M^{-1} = (I + L)^{-1} in 16 x 16 blocks: diagonal blocks by an fp32 column sweep (warps 0, 1),
  // off-diagonal blocks on the tensor cores (warps 0-3); only the blocks on and below the diagonal
  // are written
  if (warp < 2) inv::diag_blocks<CP>(sL, sX, warp);
  __syncthreads();
  inv::offdiag_blocks<CP>(sL, sX);
  {
    // M^{-1} planes for the local kernel; A = (Gamma . M^{-1}) diag(beta) and A diag(e^g / |k|) as planes
    bf16* MI = reinterpret_cast<bf16*>(p.minv) + item * 2 * C * C;
    for (int e = tid; e < C * C / 2; e += 256) {
      const int i = e / (C / 2), c = (e % (C / 2)) * 2;
      const float m0v = c <= i ? sX[i * CP + c] : 0.f, m1v = c + 1 <= i ? sX[i * CP + c + 1] : 0.f;
      wm::store_split2(MI + i * C + c, MI + C * C + i * C + c, m0v, m1v);
      const float a0 = c <= i ? decay(vg[i] - vg[c]) * m0v * vb[c] : 0.f;
      const float a1 = c + 1 <= i ? decay(vg[i] - vg[c + 1]) * m1v * vb[c + 1] : 0.f;
      wm::store_split2(sA + i * PP + c, sA + PLN + i * PP + c, a0, a1);
      wm::store_split2(sAW + i * PP + c, sAW + PLN + i * PP + c, a0 * vek[c], a1 * vek[c + 1]);
    }
  }
  __syncthreads();

  // W<- = A diag(e^g / |k|) K and U~ = A V (C x D): rows m0.., columns nw .. nw + D/2; A is lower
  // triangular, so rows m0 .. m0 + 15 need k < m0 + 16 only.
  constexpr int NT = D / 16;
  const int nw = (D / 2) * (warp >> 2);
  {
    float acc[1][NT][4];
    wm::zero(acc);
    wm::pgemm<1, NT, false, true, true, XS>(acc, sAW, sAW + PLN, PP, kh, kl, DP, m0, nw, 0, m0 + 16);
    bf16* Wg = reinterpret_cast<bf16*>(p.w) + item * 2 * C * D;  // hi, lo planes
    wm::for_each_pair(acc, m0, nw, [&](int i, int c, float& x0, float& x1) {
      wm::store_split2(Wg + i * D + c, Wg + C * D + i * D + c, x0, x1);
    });
  }
  {
    float acc[1][NT][4];
    wm::zero(acc);
    wm::pgemm<1, NT, false, true, true, XS>(acc, sA, sA + PLN, PP, vh, vl, DP, m0, nw, 0, m0 + 16);
    float* Ug = p.ut + item * C * D;
    wm::for_each_pair(acc, m0, nw, [&](int i, int c, float& x0, float& x1) {
      *reinterpret_cast<float2*>(Ug + i * D + c) = make_float2(x0, x1);
    });
  }
}

// ----------------------------------------------------------------------------- state (forward states)
//
// The two sequential passes take every MMA operand from bf16 planes in shared memory through
// ldmatrix: an fp32 operand as two planes (hi, lo), a bf16 input tile as one. W<- and P arrive as
// planes from the factor kernel; the state (or its gradient) and the chunk's small C x VB
// operands are split into planes once per chunk. fp16 q/k/dO tiles are split into bf16 planes
// after they land (an fp16 value is exactly hi + lo).

template <int D>
struct StSmem {
  static constexpr int DP = D + 8, HP = VB + 8;
  static constexpr uint32_t TILE = C * DP * 2;       // one 16-bit C x D tile
  static constexpr uint32_t WH = 0;                  // per stage: W<- hi, lo planes [C][DP]
  static constexpr uint32_t WL = WH + TILE;
  static constexpr uint32_t K = WL + TILE;           //            k [C][DP] (the input's type)
  static constexpr uint32_t UT = K + TILE;           //            U~ columns fp32 [C][UP]
  static constexpr uint32_t VEC = UT + C * UP * 4;   //            g, 1/|k|
  static constexpr uint32_t STAGE = VEC + 2 * C * 4;
  static constexpr uint32_t SH = 2 * STAGE;          // state rows hi, lo planes [VB][DP]
  static constexpr uint32_t SL = SH + VB * DP * 2;
  static constexpr uint32_t UKH = SL + VB * DP * 2;  // diag(e^{g_C - g}/|k|) U, hi, lo planes [C][HP]
  static constexpr uint32_t UKL = UKH + C * HP * 2;
  static constexpr uint32_t UH = UKL + C * HP * 2;   // U, hi, lo planes [C][HP] (copied out by the producers)
  static constexpr uint32_t UL = UH + C * HP * 2;
  static constexpr uint32_t KL = UL + C * HP * 2;    // fp16 inputs: the lo plane of k (its hi plane
                                                     // overwrites the stage's k tile)
  static constexpr uint32_t bytes_bf16 = KL;
  static constexpr uint32_t bytes_fp16 = KL + TILE;
};

// The CTA's chain: sequence (longest first), value head, first state row.
struct ChainJob {
  int seq, hv, h, vb, c0, c1;
  int64_t slot;
};
template <int D>
__device__ __forceinline__ ChainJob chain_job(const BwdParams& p) {
  constexpr int NVB = D / VB;
  ChainJob jb;
  const int bid = blockIdx.x;
  jb.vb = (bid % NVB) * VB;
  const int chain = bid / NVB;
  jb.seq = p.order[chain / p.HV];
  jb.hv = chain % p.HV;
  jb.h = jb.hv / (p.HV / p.H);
  jb.c0 = p.seq_chunk_off[jb.seq];
  jb.c1 = p.seq_chunk_off[jb.seq + 1];
  jb.slot = p.cache_indices[jb.seq];
  return jb;
}

// rows x W bf16 plane rows (pitch P in shared memory) to a row-major global plane of row stride ld,
// 16 bytes at a time; `neg` flips the sign of every value (exact for a hi/lo pair).
template <int W, int P>
__device__ __forceinline__ void copy_rows_out(bf16* dst, const bf16* src, int64_t ld, int rows, bool neg, int tid,
                                              int nthr) {
  constexpr int PER = W / 8;
  const uint32_t flip = neg ? 0x80008000u : 0u;
  for (int e = tid; e < rows * PER; e += nthr) {
    const int i = e / PER, q = e % PER;
    uint4 x = *reinterpret_cast<const uint4*>(src + i * P + q * 8);
    x.x ^= flip;
    x.y ^= flip;
    x.z ^= flip;
    x.w ^= flip;
    *reinterpret_cast<uint4*>(dst + i * ld + q * 8) = x;
  }
}

// Warps 0-7 (consumers) run the chunk step; warps 8-15 (producers) fetch the next chunk's tiles and
// write this chunk's S_in and U planes out, so neither sits on the step's critical path.
template <int D, typename E>
__global__ void __launch_bounds__(2 * kSeqThreads) bwd_state_kernel(BwdParams p) {
  using S = StSmem<D>;
  constexpr int DP = S::DP, HP = S::HP;
  constexpr bool XS = kSplitSrc<E>;
  constexpr int NTS = D / 64;  // 8-column tiles per consumer warp of the VB x D state
  extern __shared__ __align__(128) unsigned char smem[];
  if (p.status[0] != GDN_OK) return;
  const ChainJob jb = chain_job<D>(p);
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool producer = tid >= kSeqThreads;
  const int ptid = tid - kSeqThreads;
  bf16* sSH = reinterpret_cast<bf16*>(smem + S::SH);
  bf16* sSL = reinterpret_cast<bf16*>(smem + S::SL);
  bf16* sUKH = reinterpret_cast<bf16*>(smem + S::UKH);
  bf16* sUKL = reinterpret_cast<bf16*>(smem + S::UKL);
  bf16* sUH = reinterpret_cast<bf16*>(smem + S::UH);
  bf16* sUL = reinterpret_cast<bf16*>(smem + S::UL);
  bf16* sKL = reinterpret_cast<bf16*>(smem + S::KL);
  const E* kin = static_cast<const E*>(p.k) + (int64_t)jb.h * D;

  auto issue = [&](int c, int st) {  // producers
    unsigned char* base = smem + st * S::STAGE;
    const int4 ct = p.chunk_tab[c];
    const int64_t item = (int64_t)c * p.HV + jb.hv;
    const bf16* wp = reinterpret_cast<const bf16*>(p.w) + item * 2 * C * D;
    load_tokens<D, kSeqThreads>(reinterpret_cast<bf16*>(base + S::WH), wp, D, 0, C, ptid);
    load_tokens<D, kSeqThreads>(reinterpret_cast<bf16*>(base + S::WL), wp + C * D, D, 0, C, ptid);
    load_tokens<D, kSeqThreads>(reinterpret_cast<E*>(base + S::K), kin, (int64_t)p.H * D, ct.y, ct.z, ptid);
    load_f32<VB, UP, C, kSeqThreads>(reinterpret_cast<float*>(base + S::UT), p.ut + item * C * D + jb.vb, D, ptid);
    float* vec = reinterpret_cast<float*>(base + S::VEC);
    if (ptid < 16) cp_async_16(vec + 4 * ptid, p.g + item * C + 4 * ptid);
    else if (ptid < 32) cp_async_16(vec + C + 4 * (ptid - 16), p.rk + item * C + 4 * (ptid - 16));
  };

  const float* S0 = p.state_pool + (jb.slot * p.HV + jb.hv) * (int64_t)D * D + (int64_t)jb.vb * D;
  const int ns0 = (warp & 7) * (D / 8);                         // the consumer warp's state columns
  const int mu = 16 * (warp & 3), nu = 8 * ((warp >> 2) & 1);  // its 16 x 8 tile of U (C x VB)
  float st[1][NTS][4];
  auto store_state = [&]() {
    wm::for_each_pair(st, 0, ns0, [&](int i, int c, float& x0, float& x1) {
      wm::store_split2(sSH + i * DP + c, sSL + i * DP + c, x0, x1);
    });
  };
  if (!producer) {
    wm::for_each(st, 0, ns0, [&](int i, int c, float& x) { x = S0[i * D + c]; });
    store_state();
  } else {
    if (jb.c1 > jb.c0) issue(jb.c0, 0);
    cp_async_commit();
  }

  for (int c = jb.c0; c < jb.c1; ++c) {
    const int stg = (c - jb.c0) & 1;
    if (producer) cp_async_wait<0>();
    __syncthreads();  // this chunk's tiles have landed; the state planes hold the entering state
    unsigned char* base = smem + stg * S::STAGE;
    const int64_t item = (int64_t)c * p.HV + jb.hv;
    if (producer) {
      if (c + 1 < jb.c1) issue(c + 1, stg ^ 1);
      cp_async_commit();
      bf16* Sin = reinterpret_cast<bf16*>(p.s_in) + item * 2 * D * D + (int64_t)jb.vb * D;
      copy_rows_out<D, DP>(Sin, sSH, D, VB, false, ptid, kSeqThreads);
      copy_rows_out<D, DP>(Sin + D * D, sSL, D, VB, false, ptid, kSeqThreads);
    } else {
      const bf16* sWH = reinterpret_cast<const bf16*>(base + S::WH);
      const bf16* sWL = reinterpret_cast<const bf16*>(base + S::WL);
      E* sK = reinterpret_cast<E*>(base + S::K);
      const float* sUT = reinterpret_cast<const float*>(base + S::UT);
      const float* vg = reinterpret_cast<const float*>(base + S::VEC);
      const float* vrk = vg + C;
      split_inplace<D, DP>(sK, sKL, XS ? C : 0, tid, kSeqThreads);
      // U = U~ - W<- S^T (C x VB); U and diag(e^{g_C - g}/|k|) U as planes
      float ua[4] = {0.f, 0.f, 0.f, 0.f}, ub[4] = {0.f, 0.f, 0.f, 0.f};  // even / odd k-steps
#pragma unroll
      for (int k0 = 0; k0 < D; k0 += 32) {
        uint32_t ah[4], al[4], bh[2], bl[2];
        wm::lda(ah, sWH, DP, mu, k0);
        wm::lda(al, sWL, DP, mu, k0);
        wm::ldb1(bh, sSH, DP, k0, nu);
        wm::ldb1(bl, sSL, DP, k0, nu);
        wm::mma_terms<true, true>(ua, ah, al, bh, bl);
        wm::lda(ah, sWH, DP, mu, k0 + 16);
        wm::lda(al, sWL, DP, mu, k0 + 16);
        wm::ldb1(bh, sSH, DP, k0 + 16, nu);
        wm::ldb1(bl, sSL, DP, k0 + 16, nu);
        wm::mma_terms<true, true>(ub, ah, al, bh, bl);
      }
      const float gC = vg[C - 1];
      const int r = wm::lane_r(), cl = wm::lane_c();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = mu + r + 8 * hh, cc = nu + cl;
        const float u0 = sUT[i * UP + cc] - (ua[2 * hh] + ub[2 * hh]);
        const float u1 = sUT[i * UP + cc + 1] - (ua[2 * hh + 1] + ub[2 * hh + 1]);
        wm::store_split2(sUH + i * HP + cc, sUL + i * HP + cc, u0, u1);
        const float sk = expf(gC - vg[i]) * vrk[i];
        wm::store_split2(sUKH + i * HP + cc, sUKL + i * HP + cc, sk * u0, sk * u1);
      }
    }
    __syncthreads();  // U planes complete; the producers have copied the entering state out
    if (producer) {
      bf16* Ug = reinterpret_cast<bf16*>(p.u) + item * 2 * C * D + jb.vb;
      copy_rows_out<VB, HP>(Ug, sUH, D, C, false, ptid, kSeqThreads);
      copy_rows_out<VB, HP>(Ug + C * D, sUL, D, C, false, ptid, kSeqThreads);
    } else {
      // S = e^{g_C} S + (diag(e^{g_C - g}/|k|) U)^T K
      const float* vg = reinterpret_cast<const float*>(base + S::VEC);
      const float eC = expf(vg[C - 1]);
      wm::for_each(st, 0, ns0, [&](int, int, float& x) { x *= eC; });
      const bf16* kh = reinterpret_cast<const bf16*>(base + S::K);
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 16) {
        uint32_t ah[4], al[4];
        wm::lda_t(ah, sUKH, HP, 0, k0);
        wm::lda_t(al, sUKL, HP, 0, k0);
#pragma unroll
        for (int j = 0; j < NTS; ++j) {
          uint32_t bh[2], bl[2];
          wm::ldb1_t(bh, kh, DP, k0, ns0 + 8 * j);
          if (XS) wm::ldb1_t(bl, sKL, DP, k0, ns0 + 8 * j);
          wm::mma_terms<true, XS>(st[0][j], ah, al, bh, bl);
        }
      }
      store_state();
    }
  }
}

// ----------------------------------------------------------------------------- dstate (reverse)

template <int D, bool XS>
struct DsSmem {
  static constexpr int DP = D + 8, HP = VB + 8, PP = C + 8;
  static constexpr int NST = XS ? 1 : 2;              // fp16 inputs: one stage (room for the lo planes)
  static constexpr uint32_t TILE = C * DP * 2;
  static constexpr uint32_t PH = 0;                  // per stage: P hi, lo planes [C][PP]
  static constexpr uint32_t PL = PH + C * PP * 2;
  static constexpr uint32_t DO = PL + C * PP * 2;    //            dO columns [C][HP] (input type)
  static constexpr uint32_t K = DO + C * HP * 2;     //            k [C][DP]
  static constexpr uint32_t Q = K + TILE;            //            q [C][DP]
  static constexpr uint32_t WH = Q + TILE;           //            W<- hi, lo planes [C][DP]
  static constexpr uint32_t WL = WH + TILE;
  static constexpr uint32_t VEC = WL + TILE;         //            g, 1/|q|, 1/|k|
  static constexpr uint32_t STAGE = VEC + 3 * C * 4;
  static constexpr uint32_t GH = NST * STAGE;        // gradient rows hi, lo planes [VB][DP]
  static constexpr uint32_t GL = GH + VB * DP * 2;
  static constexpr uint32_t NUH = GL + VB * DP * 2;  // -dU hi, lo planes [C][HP]
  static constexpr uint32_t NUL = NUH + C * HP * 2;
  static constexpr uint32_t OSH = NUL + C * HP * 2;  // scale diag(e^g/|q|) dO hi, lo planes [C][HP]
  static constexpr uint32_t OSL = OSH + C * HP * 2;
  static constexpr uint32_t XQL = OSL + C * HP * 2;  // fp16 inputs: lo planes of q, k, dO (their hi
  static constexpr uint32_t XKL = XQL + TILE;        // planes overwrite the stage's tiles)
  static constexpr uint32_t XOL = XKL + TILE;
  static constexpr uint32_t bytes = XS ? XOL + C * HP * 2 : XQL;
  static_assert(bytes <= 232448, "shared memory per CTA");
};

template <int D, typename E>
__global__ void __launch_bounds__(2 * kSeqThreads) bwd_dstate_kernel(BwdParams p) {
  constexpr bool XS = kSplitSrc<E>;
  using S = DsSmem<D, XS>;
  constexpr int DP = S::DP, HP = S::HP, PP = S::PP;
  constexpr int NTS = D / 64;
  extern __shared__ __align__(128) unsigned char smem[];
  if (p.status[0] != GDN_OK) return;
  const ChainJob jb = chain_job<D>(p);
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool producer = tid >= kSeqThreads;  // warps 8-15: tile fetches and the per-chunk outputs
  const int ptid = tid - kSeqThreads;
  bf16* sGH = reinterpret_cast<bf16*>(smem + S::GH);
  bf16* sGL = reinterpret_cast<bf16*>(smem + S::GL);
  bf16* sNUH = reinterpret_cast<bf16*>(smem + S::NUH);
  bf16* sNUL = reinterpret_cast<bf16*>(smem + S::NUL);
  bf16* sOSH = reinterpret_cast<bf16*>(smem + S::OSH);
  bf16* sOSL = reinterpret_cast<bf16*>(smem + S::OSL);
  bf16* xql = reinterpret_cast<bf16*>(smem + S::XQL);
  bf16* xkl = reinterpret_cast<bf16*>(smem + S::XKL);
  bf16* xol = reinterpret_cast<bf16*>(smem + S::XOL);
  const E* kin = static_cast<const E*>(p.k) + (int64_t)jb.h * D;
  const E* qin = static_cast<const E*>(p.q) + (int64_t)jb.h * D;
  const E* doin = static_cast<const E*>(p.d_out) + (int64_t)jb.hv * D + jb.vb;

  auto issue = [&](int c, int st) {  // producers
    unsigned char* base = smem + st * S::STAGE;
    const int4 ct = p.chunk_tab[c];
    const int64_t item = (int64_t)c * p.HV + jb.hv;
    const bf16* pp = reinterpret_cast<const bf16*>(p.pm) + item * 2 * C * C;
    load_tokens<C, kSeqThreads>(reinterpret_cast<bf16*>(base + S::PH), pp, C, 0, C, ptid);
    load_tokens<C, kSeqThreads>(reinterpret_cast<bf16*>(base + S::PL), pp + C * C, C, 0, C, ptid);
    load_tokens_cols<VB, HP, kSeqThreads>(reinterpret_cast<E*>(base + S::DO), doin, (int64_t)p.HV * D, ct.y, ct.z, ptid);
    load_tokens<D, kSeqThreads>(reinterpret_cast<E*>(base + S::K), kin, (int64_t)p.H * D, ct.y, ct.z, ptid);
    load_tokens<D, kSeqThreads>(reinterpret_cast<E*>(base + S::Q), qin, (int64_t)p.H * D, ct.y, ct.z, ptid);
    const bf16* wp = reinterpret_cast<const bf16*>(p.w) + item * 2 * C * D;
    load_tokens<D, kSeqThreads>(reinterpret_cast<bf16*>(base + S::WH), wp, D, 0, C, ptid);
    load_tokens<D, kSeqThreads>(reinterpret_cast<bf16*>(base + S::WL), wp + C * D, D, 0, C, ptid);
    float* vec = reinterpret_cast<float*>(base + S::VEC);
    if (ptid < 16) cp_async_16(vec + 4 * ptid, p.g + item * C + 4 * ptid);
    else if (ptid < 32) cp_async_16(vec + C + 4 * (ptid - 16), p.rq + item * C + 4 * (ptid - 16));
    else if (ptid < 48) cp_async_16(vec + 2 * C + 4 * (ptid - 32), p.rk + item * C + 4 * (ptid - 32));
  };

  const int64_t srow = (jb.slot * p.HV + jb.hv) * (int64_t)D * D + (int64_t)jb.vb * D;
  const int ns0 = (warp & 7) * (D / 8);
  const int mu = 16 * (warp & 3), nu = 8 * ((warp >> 2) & 1);
  float ds[1][NTS][4];
  auto store_grad = [&]() {
    wm::for_each_pair(ds, 0, ns0, [&](int i, int c, float& x0, float& x1) {
      wm::store_split2(sGH + i * DP + c, sGL + i * DP + c, x0, x1);
    });
  };
  if (!producer) {
    wm::for_each(ds, 0, ns0, [&](int i, int c, float& x) { x = p.d_state ? p.d_state[srow + i * D + c] : 0.f; });
    store_grad();
  } else {
    if (jb.c1 > jb.c0) issue(jb.c1 - 1, 0);
    cp_async_commit();
  }

  for (int c = jb.c1 - 1; c >= jb.c0; --c) {
    const int stg = S::NST == 2 ? (jb.c1 - 1 - c) & 1 : 0;
    if (producer) cp_async_wait<0>();
    __syncthreads();  // this chunk's tiles have landed; the gradient planes hold dS leaving this chunk
    unsigned char* base = smem + stg * S::STAGE;
    const float* vg = reinterpret_cast<const float*>(base + S::VEC);
    const int64_t item = (int64_t)c * p.HV + jb.hv;
    if (producer) {
      if (S::NST == 2 && c - 1 >= jb.c0) issue(c - 1, stg ^ 1);
      cp_async_commit();
      bf16* dSo = reinterpret_cast<bf16*>(p.ds_out) + item * 2 * D * D + (int64_t)jb.vb * D;
      copy_rows_out<D, DP>(dSo, sGH, D, VB, false, ptid, kSeqThreads);
      copy_rows_out<D, DP>(dSo + D * D, sGL, D, VB, false, ptid, kSeqThreads);
    } else {
      const bf16* sPH = reinterpret_cast<const bf16*>(base + S::PH);
      const bf16* sPL = reinterpret_cast<const bf16*>(base + S::PL);
      E* sDO = reinterpret_cast<E*>(base + S::DO);
      E* sK = reinterpret_cast<E*>(base + S::K);
      E* sQ = reinterpret_cast<E*>(base + S::Q);
      const float* vrq = vg + C;
      const float* vrk = vg + 2 * C;
      if (XS) {
        split_inplace<D, DP>(sQ, xql, C, tid, kSeqThreads);
        split_inplace<D, DP>(sK, xkl, C, tid, kSeqThreads);
        split_inplace<VB, HP>(sDO, xol, C, tid, kSeqThreads);
        tc::named_sync(1, kSeqThreads);  // consumers only
      }
      const bf16* kh = reinterpret_cast<const bf16*>(sK);
      const bf16* oh = reinterpret_cast<const bf16*>(sDO);
      // a dO value of the tile (fp16 inputs: hi + lo, exactly)
      auto dov = [&](int i, int cc) {
        return XS ? __bfloat162float(oh[i * HP + cc]) + __bfloat162float(xol[i * HP + cc]) : to_f(sDO[i * HP + cc]);
      };
      // dU = scale P^T dO + diag(e^{g_C - g}/|k|) (K dS^T)  (C x VB): the warp's 16 x 8 tile, kept as planes
      // of -dU; and the planes of scale diag(e^g/|q|) dO for the state-gradient update
      float a1[4] = {0.f, 0.f, 0.f, 0.f}, a2[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k0 = mu; k0 < C; k0 += 16) {  // P^T is upper triangular: rows mu.. need k >= mu
        uint32_t ah[4], al[4], bh[2], bl[2];
        wm::lda_t(ah, sPH, PP, mu, k0);
        wm::lda_t(al, sPL, PP, mu, k0);
        wm::ldb1_t(bh, oh, HP, k0, nu);
        if (XS) wm::ldb1_t(bl, xol, HP, k0, nu);
        wm::mma_terms<true, XS>(a1, ah, al, bh, bl);
      }
      float a3[4] = {0.f, 0.f, 0.f, 0.f};  // odd k-steps of a2
#pragma unroll
      for (int k0 = 0; k0 < D; k0 += 32) {
        uint32_t ah[4], al[4], bh[2], bl[2];
        wm::lda(ah, kh, DP, mu, k0);
        if (XS) wm::lda(al, xkl, DP, mu, k0);
        wm::ldb1(bh, sGH, DP, k0, nu);
        wm::ldb1(bl, sGL, DP, k0, nu);
        wm::mma_terms<XS, true>(a2, ah, al, bh, bl);
        wm::lda(ah, kh, DP, mu, k0 + 16);
        if (XS) wm::lda(al, xkl, DP, mu, k0 + 16);
        wm::ldb1(bh, sGH, DP, k0 + 16, nu);
        wm::ldb1(bl, sGL, DP, k0 + 16, nu);
        wm::mma_terms<XS, true>(a3, ah, al, bh, bl);
      }
      const float sc = p.scale, gC = vg[C - 1];
      const int r = wm::lane_r(), cl = wm::lane_c();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = mu + r + 8 * hh, cc = nu + cl;
        const float sk = expf(gC - vg[i]) * vrk[i];
        const float y0 = sc * a1[2 * hh] + sk * (a2[2 * hh] + a3[2 * hh]);
        const float y1 = sc * a1[2 * hh + 1] + sk * (a2[2 * hh + 1] + a3[2 * hh + 1]);
        wm::store_split2(sNUH + i * HP + cc, sNUL + i * HP + cc, -y0, -y1);
        const float sq = sc * expf(vg[i]) * vrq[i];
        wm::store_split2(sOSH + i * HP + cc, sOSL + i * HP + cc, sq * dov(i, cc), sq * dov(i, cc + 1));
      }
    }
    __syncthreads();  // -dU and the scaled dO planes complete; dS_out copied out
    if (producer) {
      bf16* dUg = reinterpret_cast<bf16*>(p.du) + item * 2 * C * D + jb.vb;  // dU = -(the -dU planes)
      copy_rows_out<VB, HP>(dUg, sNUH, D, C, true, ptid, kSeqThreads);
      copy_rows_out<VB, HP>(dUg + C * D, sNUL, D, C, true, ptid, kSeqThreads);
    } else {
      // dS = e^{g_C} dS + (scale diag(e^g/|q|) dO)^T Q - dU^T W<-   (VB x D)
      const bf16* qh = reinterpret_cast<const bf16*>(base + S::Q);
      const bf16* sWH = reinterpret_cast<const bf16*>(base + S::WH);
      const bf16* sWL = reinterpret_cast<const bf16*>(base + S::WL);
      const float eC = expf(vg[C - 1]);
      wm::for_each(ds, 0, ns0, [&](int, int, float& x) { x *= eC; });
      float dw2[1][NTS][4];  // the -dU^T W<- product, added at the end
      wm::zero(dw2);
#pragma unroll
      for (int k0 = 0; k0 < C; k0 += 16) {
        uint32_t oh4[4], ol4[4], uh4[4], ul4[4];
        wm::lda_t(oh4, sOSH, HP, 0, k0);
        wm::lda_t(ol4, sOSL, HP, 0, k0);
        wm::lda_t(uh4, sNUH, HP, 0, k0);
        wm::lda_t(ul4, sNUL, HP, 0, k0);
#pragma unroll
        for (int j = 0; j < NTS; ++j) {
          uint32_t bh[2], bl[2];
          wm::ldb1_t(bh, qh, DP, k0, ns0 + 8 * j);
          if (XS) wm::ldb1_t(bl, xql, DP, k0, ns0 + 8 * j);
          wm::mma_terms<true, XS>(ds[0][j], oh4, ol4, bh, bl);
          wm::ldb1_t(bh, sWH, DP, k0, ns0 + 8 * j);
          wm::ldb1_t(bl, sWL, DP, k0, ns0 + 8 * j);
          wm::mma_terms<true, true>(dw2[0][j], uh4, ul4, bh, bl);
        }
      }
#pragma unroll
      for (int j = 0; j < NTS; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) ds[0][j][e] += dw2[0][j][e];
      store_grad();
    }
    if (S::NST == 1 && c - 1 >= jb.c0) {  // one stage: refill it once this chunk is done with it
      __syncthreads();
      if (producer) {
        issue(c - 1, 0);
        cp_async_commit();  // committed now, so that the next iteration's wait covers it
      }
    }
  }
  if (!producer) {
    float* dS0 = p.d_state_pool + srow;
    wm::for_each_pair(ds, 0, ns0, [&](int i, int c, float& x0, float& x1) {
      *reinterpret_cast<float2*>(dS0 + i * D + c) = make_float2(x0, x1);
    });
  }
}

// ----------------------------------------------------------------------------- sgrad

// Two CTAs per (chunk, value head), each computing one half of the output columns (the key
// dimension), so that two CTAs fit on an SM and one's loads overlap the other's products. The two
// halves of an item are neighbouring blocks (blockIdx.x = 2 chunk + half), so they run at the same
// time and the second one's reads of dO, dU and U hit L2.
template <int D, bool XS>
struct SgSmem {
  static constexpr int DP = D + 8;                   // pitch of C x D tiles and planes
  static constexpr int HD = D / 2, HPD = HD + 8;     // the CTA's half of the key columns, its pitch
  static constexpr uint32_t PLS = D * HPD * 2;       // one D x D/2 plane
  static constexpr uint32_t PLC = C * DP * 2;        // one C x D plane or tile
  static constexpr uint32_t SH = 0;                  // S_in half planes, then dS_out half planes
  static constexpr uint32_t SL = SH + PLS;
  static constexpr uint32_t DO = SL + PLS;           // dO tile (fp16: its hi plane after the split)
  static constexpr uint32_t DUH = DO + PLC;          // dU planes; after the first product: U planes at DO
  static constexpr uint32_t DUL = DUH + PLC;
  static constexpr uint32_t DOL = DUL + PLC;         // fp16 only: lo plane of dO
  static constexpr uint32_t VEC = DOL + (XS ? PLC : 0);  // g; 8 warp partials
  static constexpr uint32_t bytes = VEC + C * 4 + 8 * 4;
};

template <int D, typename E>
__global__ void __launch_bounds__(256, 2) bwd_sgrad_kernel(BwdParams p) {
  constexpr bool XS = kSplitSrc<E>;
  using S = SgSmem<D, XS>;
  constexpr int DP = S::DP, HD = S::HD, HPD = S::HPD;
  extern __shared__ __align__(128) unsigned char smem[];
  if (p.status[0] != GDN_OK) return;
  const int j = blockIdx.x >> 1, hv = blockIdx.y, half = blockIdx.x & 1;
  if (j >= p.status[1]) return;
  const int4 ct = p.chunk_tab[j];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int col0 = half * HD;  // the CTA's key columns: col0 .. col0 + D/2
  bf16* sSH = reinterpret_cast<bf16*>(smem + S::SH);
  bf16* sSL = reinterpret_cast<bf16*>(smem + S::SL);
  E* sDO = reinterpret_cast<E*>(smem + S::DO);
  bf16* sDUH = reinterpret_cast<bf16*>(smem + S::DUH);
  bf16* sDUL = reinterpret_cast<bf16*>(smem + S::DUL);
  bf16* sUH = reinterpret_cast<bf16*>(smem + S::DO);  // after the first product
  bf16* sUL = sUH + C * DP;
  bf16* sDOL = reinterpret_cast<bf16*>(smem + S::DOL);
  float* vg = reinterpret_cast<float*>(smem + S::VEC);
  float* vred = vg + C;
  const int64_t item = (int64_t)j * p.HV + hv;
  const bf16* sin_g = reinterpret_cast<const bf16*>(p.s_in) + item * 2 * D * D + col0;
  const bf16* du_g = reinterpret_cast<const bf16*>(p.du) + item * 2 * C * D;
  const bf16* u_g = reinterpret_cast<const bf16*>(p.u) + item * 2 * C * D;

  load_rows<HD, HPD, D, 256>(sSH, sin_g, D, tid);
  load_rows<HD, HPD, D, 256>(sSL, sin_g + D * D, D, tid);
  load_tokens<D, 256>(sDO, static_cast<const E*>(p.d_out) + (int64_t)hv * D, (int64_t)p.HV * D, ct.y, ct.z, tid);
  load_rows<D, DP, C, 256>(sDUH, du_g, D, tid);
  load_rows<D, DP, C, 256>(sDUL, du_g + C * D, D, tid);
  if (tid < 16) cp_async_16(vg + 4 * tid, p.g + item * C + 4 * tid);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (XS) {
    split_inplace<D, DP>(sDO, sDOL, C, tid, 256);
    __syncthreads();
  }
  const bf16* doh = reinterpret_cast<const bf16*>(sDO);

  // [dO; dU] S_in[:, half]: warp tiles of 32 rows x D/4 columns; row blocks 0, 1 of dO and 0, 1 of dU
  {
    constexpr int NT = D / 32;
    const int rb = warp & 3, m0 = 32 * (rb & 1), n0 = (D / 4) * (warp >> 2);
    float acc[2][NT][4];
    wm::zero(acc);
    if (rb < 2) {
      wm::pgemm<2, NT, false, true, XS, true>(acc, doh, sDOL, DP, sSH, sSL, HPD, m0, n0, 0, D);
      float* out = p.dqa + item * C * D + col0;
      const float sc = p.scale;
      wm::for_each_pair(acc, m0, n0, [&](int i, int c, float& x0, float& x1) {
        const float f = sc * expf(vg[i]);
        *reinterpret_cast<float2*>(out + i * D + c) = make_float2(f * x0, f * x1);
      });
    } else {
      wm::pgemm<2, NT, false, true, true, true>(acc, sDUH, sDUL, DP, sSH, sSL, HPD, m0, n0, 0, D);
      bf16* out = reinterpret_cast<bf16*>(p.dw) + item * 2 * C * D + col0;  // -dU S_in as planes
      wm::for_each_pair(acc, m0, n0, [&](int i, int c, float& x0, float& x1) {
        wm::store_split2(out + i * D + c, out + C * D + i * D + c, -x0, -x1);
      });
    }
  }
  __syncthreads();
  // U planes over dO and dU; dS_out half planes over the S_in half planes, with <dS_out, S_in> on the half
  load_rows<D, DP, C, 256>(sUH, u_g, D, tid);
  load_rows<D, DP, C, 256>(sUL, u_g + C * D, D, tid);
  cp_async_commit();
  {
    const bf16* src = reinterpret_cast<const bf16*>(p.ds_out) + item * 2 * D * D + col0;
    float part = 0.f;
    constexpr int NPC = D * HD / 8 / 256;           // 16-byte pieces per thread and plane
    constexpr int BAT = NPC < 4 ? NPC : 4;          // loaded together, before any is used
    static_assert(NPC % BAT == 0, "piece batches");
    for (int e0 = 0; e0 < NPC; e0 += BAT) {
      uint4 gh[BAT], gl[BAT];
#pragma unroll
      for (int q = 0; q < BAT; ++q) {
        const int e = tid + 256 * (e0 + q), i = e / (HD / 8), c = (e % (HD / 8)) * 8;
        gh[q] = *reinterpret_cast<const uint4*>(src + i * D + c);
        gl[q] = *reinterpret_cast<const uint4*>(src + D * D + i * D + c);
      }
#pragma unroll
      for (int q = 0; q < BAT; ++q) {
        const int e = tid + 256 * (e0 + q), i = e / (HD / 8), c = (e % (HD / 8)) * 8;
        uint4* yh = reinterpret_cast<uint4*>(sSH + i * HPD + c);
        uint4* yl = reinterpret_cast<uint4*>(sSL + i * HPD + c);
        const uint4 sh = *yh, sl = *yl;
        const uint32_t a[4] = {gh[q].x, gh[q].y, gh[q].z, gh[q].w}, b[4] = {gl[q].x, gl[q].y, gl[q].z, gl[q].w};
        const uint32_t x[4] = {sh.x, sh.y, sh.z, sh.w}, y[4] = {sl.x, sl.y, sl.z, sl.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 g0 = ElemT<bf16>::unpack(a[u]), g1 = ElemT<bf16>::unpack(b[u]);
          const float2 s0 = ElemT<bf16>::unpack(x[u]), s1 = ElemT<bf16>::unpack(y[u]);
          part = fmaf(g0.x + g1.x, s0.x + s1.x, part);
          part = fmaf(g0.y + g1.y, s0.y + s1.y, part);
        }
        *yh = gh[q];
        *yl = gl[q];
      }
    }
    part = warp_sum(part);
    if (lane == 0) vred[warp] = part;
  }
  cp_async_wait<0>();
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += vred[w];
    p.dgc[item * 2 + half] = expf(vg[C - 1]) * s;  // the local kernel adds the two halves
  }
  // U dS_out[:, half] (C x D/2): warp tiles of 16 rows x D/4 columns
  {
    constexpr int NT = D / 32;
    const int m0 = 16 * (warp & 3), n0 = (D / 4) * (warp >> 2);
    float acc[1][NT][4];
    wm::zero(acc);
    wm::pgemm<1, NT, false, true, true, true>(acc, sUH, sUL, DP, sSH, sSL, HPD, m0, n0, 0, D);
    float* out = p.dkr + item * C * D + col0;
    wm::for_each_pair(acc, m0, n0, [&](int i, int c, float& x0, float& x1) {
      *reinterpret_cast<float2*>(out + i * D + c) = make_float2(x0, x1);
    });
  }
}

// ----------------------------------------------------------------------------- local

template <int D>
struct LoSmem {
  static constexpr int DP = D + 8;
  static constexpr uint32_t TOK = C * DP * 2;        // one 16-bit token tile
  static constexpr uint32_t CC = C * CP * 4;         // one fp32 C x C tile
  static constexpr uint32_t RQ = 0;                  // q, k tiles (whole kernel)
  static constexpr uint32_t RK = RQ + TOK;
  static constexpr uint32_t RX = RK + TOK;           // v, dO tiles; after their last use: X1, X2 (C x C)
  static constexpr uint32_t RXB = (2 * TOK > 2 * CC ? 2 * TOK : 2 * CC);
  static constexpr uint32_t C1 = RX + RXB;           // M^{-1}, then A
  static constexpr uint32_t C2 = C1 + CC;            // Q^K^^T, then dGamma
  static constexpr uint32_t C3 = C2 + CC;            // K^K^^T
  static constexpr uint32_t C4 = C3 + CC;            // dP
  static constexpr uint32_t PAIRD = 2 * C * DP * 2;  // hi, lo planes of a C x D operand
  static constexpr uint32_t F1 = C4 + CC;            // U, then dW (planes)
  static constexpr uint32_t F2 = F1 + PAIRD;         // dU (planes)
  static constexpr uint32_t VEC = F2 + PAIRD;        // 24 vectors of C
  static constexpr uint32_t bytes = VEC + 24 * C * 4;
  static_assert(bytes <= 232448, "shared memory per CTA");
};

// x = x^ n with n = sqrt(|x|^2 + eps): dx = dx^ / n - x (x . dx^) / n^3, for the rows of the
// accumulator tile (rows m0 .. m0 + 15 split over the two warps of a row block; `part` holds the
// two warps' partial dot products). rn = 1/n per row; raw: the 16-bit rows of x. Every thread
// of the CTA calls it (it synchronises the CTA).
template <int D, int NT, int NCW = 2, typename E>
__device__ __forceinline__ void norm_backward(float (&acc)[1][NT][4], const E* raw, const float* rn, float* part,
                                              int m0, int nd, int len, float* out, int64_t ld) {
  constexpr int DP = D + 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float pd[2] = {0.f, 0.f};
  wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
    const float y = fmaf(to_f(raw[i * DP + c]), x0, to_f(raw[i * DP + c + 1]) * x1);
    if (i - m0 < 8) pd[0] += y; else pd[1] += y;
  });
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const float sdot = quad_sum(pd[hh]);
    if ((lane & 3) == 0) part[(warp >> 2) * 64 + m0 + wm::lane_r() + 8 * hh] = sdot;
  }
  __syncthreads();
  wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
    if (i < len) {
      float dot = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; ++w) dot += part[64 * w + i];
      const float r = rn[i], f = dot * r * r * r;
      *reinterpret_cast<float2*>(out + (int64_t)i * ld + c) =
          make_float2(r * x0 - to_f(raw[i * DP + c]) * f, r * x1 - to_f(raw[i * DP + c + 1]) * f);
    }
  });
}

template <int D, typename E>
__global__ void __launch_bounds__(256, 1) bwd_local_kernel(BwdParams p) {
  using S = LoSmem<D>;
  constexpr int DP = S::DP;
  constexpr bool XS = kSplitSrc<E>;
  extern __shared__ __align__(128) unsigned char smem[];
  if (p.status[0] != GDN_OK) return;
  const int j = blockIdx.x, hv = blockIdx.y;
  if (j >= p.status[1]) return;
  const int4 ct = p.chunk_tab[j];
  const int64_t t0 = ct.y;
  const int len = ct.z;
  const int h = hv / (p.HV / p.H);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int64_t item = (int64_t)j * p.HV + hv;
  E* rq_t = reinterpret_cast<E*>(smem + S::RQ);
  E* rk_t = reinterpret_cast<E*>(smem + S::RK);
  E* rv_t = reinterpret_cast<E*>(smem + S::RX);
  E* rdo_t = reinterpret_cast<E*>(smem + S::RX + S::TOK);
  float* X1 = reinterpret_cast<float*>(smem + S::RX);
  float* X2 = reinterpret_cast<float*>(smem + S::RX + S::CC);
  float* C1 = reinterpret_cast<float*>(smem + S::C1);
  float* C2 = reinterpret_cast<float*>(smem + S::C2);
  float* C3 = reinterpret_cast<float*>(smem + S::C3);
  float* C4 = reinterpret_cast<float*>(smem + S::C4);
  bf16* F1 = reinterpret_cast<bf16*>(smem + S::F1);
  bf16* F2 = reinterpret_cast<bf16*>(smem + S::F2);
  constexpr int64_t FPL = C * DP;  // elements from a hi plane to its lo plane
  float* vg = reinterpret_cast<float*>(smem + S::VEC);
  float* vbt = vg + C;
  float* vrq = vbt + C;
  float* vrk = vrq + C;
  float* veg = vrk + C;      // e^g
  float* vdec = veg + C;     // e^{g_C - g}
  float* vdb = vdec + C;     // d beta
  float* vdg = vdb + C;      // d g
  float* vcolp = vdg + C;    // [4][C] column partials of dA . Z
  float* vrow = vcolp + 4 * C;  // row sums of dGamma . Gamma
  float* vcol = vrow + C;       // column sums of dGamma . Gamma
  float* vpA = vcol + C;        // [2][C] eg <k^, A^T dW>
  float* vpB = vpA + 2 * C;     // [2][C] dec <k^, dKr>
  float* vpC = vpB + 2 * C;     // [2][C] <dQa, q^>
  float* vnk = vpC + 2 * C;     // [2][C] <k, dk^> (normalisation backward, ungrouped heads)
  float* vnq = vnk + 2 * C;     // [2][C] <q, dq^>
  const bool fused_norm = p.HV == p.H;

  load_tokens<D, 256>(rq_t, static_cast<const E*>(p.q) + (int64_t)h * D, (int64_t)p.H * D, t0, len, tid);
  load_tokens<D, 256>(rk_t, static_cast<const E*>(p.k) + (int64_t)h * D, (int64_t)p.H * D, t0, len, tid);
  load_tokens<D, 256>(rv_t, static_cast<const E*>(p.v) + (int64_t)hv * D, (int64_t)p.HV * D, t0, len, tid);
  load_tokens<D, 256>(rdo_t, static_cast<const E*>(p.d_out) + (int64_t)hv * D, (int64_t)p.HV * D, t0, len, tid);
  const bf16* u_g = reinterpret_cast<const bf16*>(p.u) + item * 2 * C * D;
  const bf16* du_g = reinterpret_cast<const bf16*>(p.du) + item * 2 * C * D;
  load_rows<D, DP, C, 256>(F1, u_g, D, tid);
  load_rows<D, DP, C, 256>(F1 + FPL, u_g + C * D, D, tid);
  load_rows<D, DP, C, 256>(F2, du_g, D, tid);
  load_rows<D, DP, C, 256>(F2 + FPL, du_g + C * D, D, tid);
  bf16* mi_s = reinterpret_cast<bf16*>(C3);  // M^{-1} planes land in C3 (written later) and widen into C1
  load_rows<C, C, 2 * C, 256>(mi_s, reinterpret_cast<const bf16*>(p.minv) + item * 2 * C * C, C, tid);
  if (tid < 16) cp_async_16(vg + 4 * tid, p.g + item * C + 4 * tid);
  else if (tid < 32) cp_async_16(vbt + 4 * (tid - 16), p.beta + item * C + 4 * (tid - 16));
  else if (tid < 48) cp_async_16(vrq + 4 * (tid - 32), p.rq + item * C + 4 * (tid - 32));
  else if (tid < 64) cp_async_16(vrk + 4 * (tid - 48), p.rk + item * C + 4 * (tid - 48));
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (tid < C) {
    veg[tid] = expf(vg[tid]);
    vdec[tid] = expf(vg[C - 1] - vg[tid]);
  }
  for (int e = tid; e < C * C; e += 256) C1[(e / C) * CP + e % C] = wm::plane_val(mi_s, e, C * C);
  __syncthreads();

  // C x C warp tiles: rows m0 .. m0 + 15, columns n0 .. n0 + 31
  const int m0 = 16 * (warp & 3), n0 = 32 * (warp >> 2);
  float da1[1][4][4];
  {
    float qk[1][4][4], kk[1][4][4], dp[1][4][4];
    wm::zero(qk);
    wm::zero(kk);
    wm::zero(dp);
    wm::zero(da1);
    auto fq = [&](int m, int x) { return to_f(rq_t[m * DP + x]); };
    auto fk = [&](int m, int x) { return to_f(rk_t[m * DP + x]); };
    auto fkt = [&](int x, int n) { return to_f(rk_t[n * DP + x]); };
    wm::gemm<1, 4, XS, XS>(qk, fq, fkt, m0, n0, 0, D);
    wm::gemm<1, 4, XS, XS>(kk, fk, fkt, m0, n0, 0, D);
    // dP = scale tril(dO U^T)
    auto fdo = [&](int m, int x) { return to_f(rdo_t[m * DP + x]); };
    auto fut = [&](int x, int n) { return wm::plane_val(F1, n * DP + x, FPL); };
    wm::gemm<1, 4, XS, true>(dp, fdo, fut, m0, n0, 0, D);
    // dU V^T
    auto fdu = [&](int m, int x) { return wm::plane_val(F2, m * DP + x, FPL); };
    auto fvt = [&](int x, int n) { return to_f(rv_t[n * DP + x]); };
    wm::gemm<1, 4, true, XS>(da1, fdu, fvt, m0, n0, 0, D);
    const float sc = p.scale;
    wm::for_each(qk, m0, n0, [&](int i, int c, float& x) { C2[i * CP + c] = vrq[i] * vrk[c] * x; });
    wm::for_each(kk, m0, n0, [&](int i, int c, float& x) { C3[i * CP + c] = vrk[i] * vrk[c] * x; });
    wm::for_each(dp, m0, n0, [&](int i, int c, float& x) { C4[i * CP + c] = c <= i ? sc * x : 0.f; });
  }
  __syncthreads();  // U, v and dO tiles no longer read
  const bf16* dw_g = reinterpret_cast<const bf16*>(p.dw) + item * 2 * C * D;
  load_rows<D, DP, C, 256>(F1, dw_g, D, tid);
  load_rows<D, DP, C, 256>(F1 + FPL, dw_g + C * D, D, tid);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  {
    // dA = dU V^T + dW (diag(e^g/|k|) K)^T on and below the diagonal; then dZ, d beta, dGamma, dM^{-1}
    float da2[1][4][4];
    wm::zero(da2);
    auto fdw = [&](int m, int x) { return wm::plane_val(F1, m * DP + x, FPL); };
    auto fkt = [&](int x, int n) { return to_f(rk_t[n * DP + x]); };
    wm::gemm<1, 4, true, XS>(da2, fdw, fkt, m0, n0, 0, D);
    float colp[4][2];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) colp[jj][0] = colp[jj][1] = 0.f;
    const int r = wm::lane_r(), cl = wm::lane_c();
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = m0 + r + 8 * (e >> 1), c = n0 + 8 * jj + cl + (e & 1);
        float dA = da1[0][jj][e] + da2[0][jj][e] * veg[c] * vrk[c];
        float gam = 0.f, mv = 0.f;
        if (c <= i) {
          gam = expf(vg[i] - vg[c]);
          mv = C1[i * CP + c];
        } else {
          dA = 0.f;
        }
        colp[jj][e & 1] += dA * gam * mv;
        const float dZ = dA * vbt[c];
        C2[i * CP + c] = c <= i ? C4[i * CP + c] * C2[i * CP + c] + dZ * mv : 0.f;
        X1[i * CP + c] = dZ * gam;
      }
    const int lane = tid & 31;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const float s = col_sum(colp[jj][h2]);
        if (lane < 4) vcolp[(warp & 3) * C + n0 + 8 * jj + cl + h2] = s;
      }
  }
  __syncthreads();
  if (tid < C) vdb[tid] = vcolp[tid] + vcolp[C + tid] + vcolp[2 * C + tid] + vcolp[3 * C + tid];
  {
    // T1 = M^{-T} dM^{-1}  (M^{-T}[i][l] = M^{-1}[l][i], zero for l < i)
    float t1[1][4][4];
    wm::zero(t1);
    auto fa = [&](int m, int x) { return C1[x * CP + m]; };
    auto fb = [&](int x, int n) { return X1[x * CP + n]; };
    wm::gemm<1, 4, true, true>(t1, fa, fb, m0, n0, m0, C);
    wm::for_each(t1, m0, n0, [&](int i, int c, float& x) { X2[i * CP + c] = x; });
  }
  __syncthreads();
  {
    // X = -T1 M^{-T}, strictly lower  (M^{-T}[l][c] = M^{-1}[c][l], zero for l > c)
    float xx[1][4][4];
    wm::zero(xx);
    auto fa = [&](int m, int x) { return X2[m * CP + x]; };
    auto fb = [&](int x, int n) { return C1[n * CP + x]; };
    wm::gemm<1, 4, true, true>(xx, fa, fb, m0, n0, 0, n0 + 32);
    wm::for_each(xx, m0, n0, [&](int i, int c, float& x) { X1[i * CP + c] = c < i ? -x : 0.f; });
  }
  __syncthreads();
  {
    // d beta_i += sum_c X_ic (k^_i . k^_c); row and column sums of dGamma . Gamma
    const int i = tid >> 2, q4 = tid & 3;
    float sb = 0.f, sr = 0.f, scol = 0.f;
    for (int c = 16 * q4; c < 16 * q4 + 16; ++c) {
      sb = fmaf(X1[i * CP + c], C3[i * CP + c], sb);
      if (c <= i) sr = fmaf(C2[i * CP + c], expf(vg[i] - vg[c]), sr);
      if (i <= c) scol = fmaf(C2[c * CP + i], expf(vg[c] - vg[i]), scol);
    }
    sb += __shfl_xor_sync(0xffffffffu, sb, 1);
    sb += __shfl_xor_sync(0xffffffffu, sb, 2);
    sr += __shfl_xor_sync(0xffffffffu, sr, 1);
    sr += __shfl_xor_sync(0xffffffffu, sr, 2);
    scol += __shfl_xor_sync(0xffffffffu, scol, 1);
    scol += __shfl_xor_sync(0xffffffffu, scol, 2);
    if (q4 == 0) {
      vdb[i] += sb;
      vrow[i] = sr;
      vcol[i] = scol;
    }
  }
  __syncthreads();
  for (int e = tid; e < C * C; e += 256) {  // M^{-1} -> A = (Gamma . M^{-1}) diag(beta)
    const int i = e / C, c = e % C;
    C1[i * CP + c] = c <= i ? expf(vg[i] - vg[c]) * C1[i * CP + c] * vbt[c] : 0.f;
  }
  __syncthreads();

  // C x D warp tiles: rows m0 .. m0 + 15, columns nd .. nd + D/2
  constexpr int NT = D / 16;
  const int nd = (D / 2) * (warp >> 2);
  const int r = wm::lane_r();
  const int lane = tid & 31;
  auto fat = [&](int m, int x) { return C1[x * CP + m]; };  // A^T: zero for x < m
  {
    // dv = A^T dU
    float acc[1][NT][4];
    wm::zero(acc);
    auto fb = [&](int x, int n) { return wm::plane_val(F2, x * DP + n, FPL); };
    wm::gemm<1, NT, true, true>(acc, fat, fb, m0, nd, m0, C);
    wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
      if (i < len) *reinterpret_cast<float2*>(p.dv + ((t0 + i) * p.HV + hv) * D + c) = make_float2(x0, x1);
    });
  }
  {
    // dk^ = diag(e^g) A^T dW + diag(dec) dKr + (Gamma . dP)^T Q^ + diag(beta) X K^ + X^T diag(beta) K^
    float acc[1][NT][4];
    wm::zero(acc);
    auto fb = [&](int x, int n) { return wm::plane_val(F1, x * DP + n, FPL); };
    wm::gemm<1, NT, true, true>(acc, fat, fb, m0, nd, m0, C);
    const float* dkr = p.dkr + item * C * D;
    float pa[2] = {0.f, 0.f}, pb[2] = {0.f, 0.f};
    wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
      const bool lo8 = i - m0 < 8;
      const float k0 = to_f(rk_t[i * DP + c]) * vrk[i], k1 = to_f(rk_t[i * DP + c + 1]) * vrk[i];
      const float2 kr = *reinterpret_cast<const float2*>(dkr + i * D + c);
      const float ya = fmaf(k0, x0, k1 * x1), yb = fmaf(k0, kr.x, k1 * kr.y);
      if (lo8) {
        pa[0] += ya;
        pb[0] += yb;
      } else {
        pa[1] += ya;
        pb[1] += yb;
      }
      x0 = veg[i] * x0 + vdec[i] * kr.x;
      x1 = veg[i] * x1 + vdec[i] * kr.y;
    });
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float a = quad_sum(pa[hh]), b2 = quad_sum(pb[hh]);
      if ((lane & 3) == 0) {
        const int i = m0 + r + 8 * hh;
        vpA[(warp >> 2) * C + i] = veg[i] * a;
        vpB[(warp >> 2) * C + i] = vdec[i] * b2;
      }
    }
    auto fa1 = [&](int m, int x) { return x >= m ? expf(vg[x] - vg[m]) * C4[x * CP + m] * vrq[x] : 0.f; };
    auto fbq = [&](int x, int n) { return to_f(rq_t[x * DP + n]); };
    wm::gemm<1, NT, true, XS>(acc, fa1, fbq, m0, nd, m0, C);
    auto fa2 = [&](int m, int x) { return vrk[x] * (vbt[m] * X1[m * CP + x] + vbt[x] * X1[x * CP + m]); };
    auto fbk = [&](int x, int n) { return to_f(rk_t[x * DP + n]); };
    wm::gemm<1, NT, true, XS>(acc, fa2, fbk, m0, nd, 0, C);
    if (fused_norm)
      norm_backward<D, NT>(acc, rk_t, vrk, vnk, m0, nd, len, p.dk + (t0 * p.H + h) * D, (int64_t)p.H * D);
    else
      wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
        if (i < len) *reinterpret_cast<float2*>(p.dkh + ((t0 + i) * p.HV + hv) * D + c) = make_float2(x0, x1);
      });
  }
  {
    // dq^ = dQa + (Gamma . dP) diag(1/|k|) K
    float acc[1][NT][4];
    const float* dqa = p.dqa + item * C * D;
    float pc[2] = {0.f, 0.f};
    wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
      const float2 a = *reinterpret_cast<const float2*>(dqa + i * D + c);
      x0 = a.x;
      x1 = a.y;
      const float y = fmaf(to_f(rq_t[i * DP + c]), a.x, to_f(rq_t[i * DP + c + 1]) * a.y);
      if (i - m0 < 8) pc[0] += y; else pc[1] += y;
    });
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float s = quad_sum(pc[hh]);
      if ((lane & 3) == 0) {
        const int i = m0 + r + 8 * hh;
        vpC[(warp >> 2) * C + i] = vrq[i] * s;
      }
    }
    auto fa = [&](int m, int x) { return x <= m ? expf(vg[m] - vg[x]) * C4[m * CP + x] * vrk[x] : 0.f; };
    auto fbk = [&](int x, int n) { return to_f(rk_t[x * DP + n]); };
    wm::gemm<1, NT, true, XS>(acc, fa, fbk, m0, nd, 0, m0 + 16);
    if (fused_norm)
      norm_backward<D, NT>(acc, rq_t, vrq, vnq, m0, nd, len, p.dq + (t0 * p.H + h) * D, (int64_t)p.H * D);
    else
      wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
        if (i < len) *reinterpret_cast<float2*>(p.dqh + ((t0 + i) * p.HV + hv) * D + c) = make_float2(x0, x1);
      });
  }
  __syncthreads();
  if (tid < C) {
    const int i = tid;
    const float rb = vpB[i] + vpB[C + i];
    vdg[i] = (vpC[i] + vpC[C + i]) - rb + (vpA[i] + vpA[C + i]) + vrow[i] - vcol[i];
    vrow[i] = rb;  // r_i, for the chunk-end term
  }
  __syncthreads();
  if (tid == 0) {
    float sr = 0.f;
    for (int i = 0; i < C; ++i) sr += vrow[i];
    vdg[C - 1] += sr + (p.dgc[2 * item] + p.dgc[2 * item + 1]);
    float run = 0.f;  // d log alpha_i = sum_{i' >= i} dg_i'
    for (int i = C - 1; i >= 0; --i) {
      run += vdg[i];
      vdg[i] = run;
    }
  }
  __syncthreads();
  if (tid < len) {
    const int64_t t = t0 + tid;
    const float dla = vdg[tid];
    const float x = p.a[t * p.HV + hv] + p.dt_bias[hv];
    const float eA = expf(p.A_log[hv]);
    const float sig = 1.f / (1.f + expf(-x));
    const float bt = vbt[tid];
    p.da[t * p.HV + hv] = dla * (-eA) * sig;
    p.db[t * p.HV + hv] = vdb[tid] * bt * (1.f - bt);
    p.dlala[t * p.HV + hv] = dla * (-eA * softplus_f(x));
  }
}

// The local kernel for bf16 inputs: every product takes its operands from bf16 planes through
// ldmatrix. The C x C operands that the products need scaled or combined (Gamma . dP with the
// key or query norms, A, X's symmetric combination) are materialised as planes once; the
// element-wise steps run on the accumulators where the fragments already sit.
template <int D>
struct LoFastSmem {
  static constexpr int DP = D + 8, PP = C + 8;
  static constexpr uint32_t TILE = C * DP * 2;
  static constexpr uint32_t PAIR = 2 * C * PP * 2;   // hi, lo planes of a C x C operand
  static constexpr uint32_t TQ = 0;                  // q, k tiles (whole kernel)
  static constexpr uint32_t TK = TQ + TILE;
  static constexpr uint32_t R1 = TK + TILE;          // v, dO tiles; after their last use: pairs P1, P2
  static constexpr uint32_t R1B = 2 * TILE > 2 * PAIR ? 2 * TILE : 2 * PAIR;
  static constexpr uint32_t PU = R1 + R1B;           // dW planes
  static constexpr uint32_t PDU = PU + 2 * TILE;     // dU planes
  static constexpr uint32_t CM = PDU + 2 * TILE;     // M^{-1} planes, then A planes
  static constexpr uint32_t P3 = CM + PAIR;          // U planes (pitch DP, over P3 and P4) until the
  static constexpr uint32_t P4 = P3 + PAIR;          // first products; then two C x C pairs
  static_assert(2 * TILE <= 2 * PAIR, "U planes fit over P3, P4");
  static constexpr int NVEC = 40;                     // vectors of C floats (carved below, in order)
  static constexpr uint32_t VEC = P4 + PAIR;
  static constexpr uint32_t bytes = VEC + NVEC * C * 4;
  static_assert(bytes <= 232448, "shared memory per CTA");
};

template <int D>
__global__ void __launch_bounds__(kLocalThreads, 1) bwd_local_fast_kernel(BwdParams p) {
  using S = LoFastSmem<D>;
  constexpr int DP = S::DP, PP = S::PP, PLN = C * PP;
  constexpr int64_t TPL = C * DP;  // elements from a C x D hi plane to its lo plane
  extern __shared__ __align__(128) unsigned char smem[];
  if (p.status[0] != GDN_OK) return;
  const int j = blockIdx.x, hv = blockIdx.y;
  if (j >= p.status[1]) return;
  const int4 ct = p.chunk_tab[j];
  const int64_t t0 = ct.y;
  const int len = ct.z;
  const int h = hv / (p.HV / p.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t item = (int64_t)j * p.HV + hv;
  bf16* tq = reinterpret_cast<bf16*>(smem + S::TQ);
  bf16* tk = reinterpret_cast<bf16*>(smem + S::TK);
  bf16* tv = reinterpret_cast<bf16*>(smem + S::R1);
  bf16* tdo = reinterpret_cast<bf16*>(smem + S::R1 + S::TILE);
  bf16* p1 = reinterpret_cast<bf16*>(smem + S::R1);           // dM^{-1}, then X
  bf16* p2 = reinterpret_cast<bf16*>(smem + S::R1 + S::PAIR);  // (Gamma . dP) diag(1/|k|)
  bf16* pu = reinterpret_cast<bf16*>(smem + S::PU);  // dW
  bf16* pu0 = reinterpret_cast<bf16*>(smem + S::P3);  // U (first products only)
  bf16* pdu = reinterpret_cast<bf16*>(smem + S::PDU);
  bf16* cm = reinterpret_cast<bf16*>(smem + S::CM);
  bf16* p3 = reinterpret_cast<bf16*>(smem + S::P3);  // diag(1/|q|) (Gamma . dP)
  bf16* p4 = reinterpret_cast<bf16*>(smem + S::P4);  // T1, then the symmetric X combination
  float* vg = reinterpret_cast<float*>(smem + S::VEC);
  float* vbt = vg + C;
  float* vrq = vbt + C;
  float* vrk = vrq + C;
  float* veg = vrk + C;      // e^g
  float* vdec = veg + C;     // e^{g_C - g}
  float* vdb = vdec + C;     // d beta
  float* vdg = vdb + C;      // d g
  float* vcolp = vdg + C;    // [4][C] column partials (d beta, then the column sums of dGamma . Gamma)
  // row partials below come from the NCW = 4 column warps of a row block
  float* vrow = vcolp + 4 * C;      // [4][C] row sums of dGamma . Gamma
  float* vxb = vrow + NCW * C;      // [4][C] row sums of X . K^K^^T
  float* vpA = vxb + NCW * C;       // [4][C] eg <k^, A^T dW>
  float* vpB = vpA + NCW * C;       // [4][C] dec <k^, dKr>
  float* vpC = vpB + NCW * C;       // [4][C] <dQa, q^>
  float* vnk = vpC + NCW * C;       // [4][C] <k, dk^>
  float* vnq = vnk + NCW * C;       // [4][C] <q, dq^>
  static_assert(S::NVEC == 8 + 4 + 7 * NCW, "vg .. vdg single vectors, vcolp 4, the seven partial arrays NCW each");
  auto sum4 = [&](const float* a, int i) { return (a[i] + a[C + i]) + (a[2 * C + i] + a[3 * C + i]); };
  const bool fused_norm = p.HV == p.H;

  const bf16* qin = static_cast<const bf16*>(p.q) + (int64_t)h * D;
  const bf16* kin = static_cast<const bf16*>(p.k) + (int64_t)h * D;
  load_tokens<D, kLocalThreads>(tq, qin, (int64_t)p.H * D, t0, len, tid);
  load_tokens<D, kLocalThreads>(tk, kin, (int64_t)p.H * D, t0, len, tid);
  load_tokens<D, kLocalThreads>(tv, static_cast<const bf16*>(p.v) + (int64_t)hv * D, (int64_t)p.HV * D, t0, len, tid);
  load_tokens<D, kLocalThreads>(tdo, static_cast<const bf16*>(p.d_out) + (int64_t)hv * D, (int64_t)p.HV * D, t0, len, tid);
  const bf16* u_g = reinterpret_cast<const bf16*>(p.u) + item * 2 * C * D;
  const bf16* du_g = reinterpret_cast<const bf16*>(p.du) + item * 2 * C * D;
  const bf16* mi_g = reinterpret_cast<const bf16*>(p.minv) + item * 2 * C * C;
  const bf16* dw_g = reinterpret_cast<const bf16*>(p.dw) + item * 2 * C * D;
  load_rows<D, DP, C, kLocalThreads>(pu0, u_g, D, tid);
  load_rows<D, DP, C, kLocalThreads>(pu0 + TPL, u_g + C * D, D, tid);
  load_rows<D, DP, C, kLocalThreads>(pu, dw_g, D, tid);
  load_rows<D, DP, C, kLocalThreads>(pu + TPL, dw_g + C * D, D, tid);
  load_rows<D, DP, C, kLocalThreads>(pdu, du_g, D, tid);
  load_rows<D, DP, C, kLocalThreads>(pdu + TPL, du_g + C * D, D, tid);
  load_rows<C, PP, C, kLocalThreads>(cm, mi_g, C, tid);
  load_rows<C, PP, C, kLocalThreads>(cm + PLN, mi_g + C * C, C, tid);
  if (tid < 16) cp_async_16(vg + 4 * tid, p.g + item * C + 4 * tid);
  else if (tid < 32) cp_async_16(vbt + 4 * (tid - 16), p.beta + item * C + 4 * (tid - 16));
  else if (tid < 48) cp_async_16(vrq + 4 * (tid - 32), p.rq + item * C + 4 * (tid - 32));
  else if (tid < 64) cp_async_16(vrk + 4 * (tid - 48), p.rk + item * C + 4 * (tid - 48));
  cp_async_commit();
  {  // dKr and dQa (fp32, read by the C x D stage's epilogues) into L2 meanwhile: a 128-byte line per thread
    constexpr int LINES = C * D / 32;  // 128-byte lines of one C x D fp32 tile
    for (int l = tid; l < 2 * LINES; l += kLocalThreads) {
      const float* src = l < LINES ? p.dkr + item * C * D + 32 * l : p.dqa + item * C * D + 32 * (l - LINES);
      asm volatile("prefetch.global.L2 [%0];\n" ::"l"(src));
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  if (tid < C) {
    veg[tid] = expf(vg[tid]);
    vdec[tid] = expf(vg[C - 1] - vg[tid]);
  }

  // ---- C x C stage: warp tiles rows m0 .. m0 + 15, columns n0 .. n0 + 31
  const int m0 = 16 * (warp & 3), n0 = 16 * (warp >> 2);
  const int r = wm::lane_r(), cl = wm::lane_c();
  float qk[1][2][4], kk[1][2][4], dp[1][2][4], da[1][2][4];
  wm::zero(qk);
  wm::zero(kk);
  wm::zero(dp);
  wm::zero(da);
  wm::pgemm<1, 2, false, false, false, false>(qk, tq, tq, DP, tk, tk, DP, m0, n0, 0, D);
  wm::pgemm<1, 2, false, false, false, false>(kk, tk, tk, DP, tk, tk, DP, m0, n0, 0, D);
  wm::pgemm<1, 2, false, false, false, true>(dp, tdo, tdo, DP, pu0, pu0 + TPL, DP, m0, n0, 0, D);  // dO U^T
  wm::pgemm<1, 2, false, false, true, false>(da, pdu, pdu + TPL, DP, tv, tv, DP, m0, n0, 0, D);  // dU V^T
  __syncthreads();  // U, v and dO no longer read; veg, vdec visible
  {
    float da2[1][2][4];
    wm::zero(da2);
    wm::pgemm<1, 2, false, false, true, false>(da2, pu, pu + TPL, DP, tk, tk, DP, m0, n0, 0, D);  // dW K^T
    // dA (on and below the diagonal), Z = Gamma . M^{-1}, d beta (columns), dZ, dGamma (kept in qk),
    // dM^{-1} -> p1, (Gamma . dP) diag(1/|k|) -> p2, diag(1/|q|) (Gamma . dP) -> p3
    const float sc = p.scale;
    float colp[2][2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      colp[jj][0] = colp[jj][1] = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = m0 + r + 8 * hh, c = n0 + 8 * jj + cl;
        float dm[2], g1k[2], g1q[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e = 2 * hh + u, cc = c + u;
          const bool low = cc <= i;
          const float gam = low ? decay(vg[i] - vg[cc]) : 0.f;
          const float mv = wm::plane_val(cm, i * PP + cc, PLN);
          const float dA = low ? da[0][jj][e] + da2[0][jj][e] * veg[cc] * vrk[cc] : 0.f;
          const float dP = low ? sc * dp[0][jj][e] : 0.f;
          colp[jj][u] += dA * gam * mv;
          const float dZ = dA * vbt[cc];
          qk[0][jj][e] = low ? dP * qk[0][jj][e] * vrq[i] * vrk[cc] + dZ * mv : 0.f;  // dGamma
          dm[u] = dZ * gam;
          g1k[u] = gam * dP * vrk[cc];
          g1q[u] = gam * dP * vrq[i];
        }
        wm::store_split2(p1 + i * PP + c, p1 + PLN + i * PP + c, dm[0], dm[1]);
        wm::store_split2(p2 + i * PP + c, p2 + PLN + i * PP + c, g1k[0], g1k[1]);
        wm::store_split2(p3 + i * PP + c, p3 + PLN + i * PP + c, g1q[0], g1q[1]);
      }
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float s = col_sum(colp[jj][u]);
        if (lane < 4) vcolp[(warp & 3) * C + n0 + 8 * jj + cl + u] = s;
      }
  }
  __syncthreads();
  if (tid < C) vdb[tid] = vcolp[tid] + vcolp[C + tid] + vcolp[2 * C + tid] + vcolp[3 * C + tid];
  {
    // T1 = M^{-T} dM^{-1} -> p4 (M^{-T}[i][l] = M^{-1}[l][i], zero for l < i)
    float t1[1][2][4];
    wm::zero(t1);
    wm::pgemm<1, 2, true, true, true, true>(t1, cm, cm + PLN, PP, p1, p1 + PLN, PP, m0, n0, m0, C);
    wm::for_each_pair(t1, m0, n0, [&](int i, int c, float& x0, float& x1) {
      wm::store_split2(p4 + i * PP + c, p4 + PLN + i * PP + c, x0, x1);
    });
  }
  __syncthreads();
  {
    // X = -T1 M^{-T}, strictly lower (M^{-T}[l][c] = M^{-1}[c][l], zero for l > c) -> p1; with the row sums
    // of X . K^K^^T (d beta) and the row and column sums of dGamma . Gamma (d g)
    float xx[1][2][4];
    wm::zero(xx);
    wm::pgemm<1, 2, false, false, true, true>(xx, p4, p4 + PLN, PP, cm, cm + PLN, PP, m0, n0, 0, n0 + 16);
    float xb[2] = {0.f, 0.f}, wr[2] = {0.f, 0.f}, wc[2][2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      wc[jj][0] = wc[jj][1] = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int i = m0 + r + 8 * hh, c = n0 + 8 * jj + cl;
        float xv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e = 2 * hh + u, cc = c + u;
          xv[u] = cc < i ? -xx[0][jj][e] : 0.f;
          xb[hh] += xv[u] * kk[0][jj][e] * vrk[i] * vrk[cc];
          const float w = cc <= i ? qk[0][jj][e] * decay(vg[i] - vg[cc]) : 0.f;
          wr[hh] += w;
          wc[jj][u] += w;
        }
        wm::store_split2(p1 + i * PP + c, p1 + PLN + i * PP + c, xv[0], xv[1]);
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float a = quad_sum(xb[hh]), b2 = quad_sum(wr[hh]);
      if ((lane & 3) == 0) {
        vxb[(warp >> 2) * C + m0 + r + 8 * hh] = a;
        vrow[(warp >> 2) * C + m0 + r + 8 * hh] = b2;
      }
    }
    __syncthreads();  // vcolp free again (d beta read it above)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float s = col_sum(wc[jj][u]);
        if (lane < 4) vcolp[(warp & 3) * C + n0 + 8 * jj + cl + u] = s;
      }
  }
  __syncthreads();
  // A = (Gamma . M^{-1}) diag(beta) in place of M^{-1}; Y = diag(1/|k|) combination of X for the key
  // gradient: Y[i][c] = (beta_i X_ic + beta_c X_ci) / |k_c| -> p4; d beta and the row/column sums of d g
  for (int e = tid; e < C * C / 2; e += kLocalThreads) {
    const int i = e / (C / 2), c = (e % (C / 2)) * 2;
    float a2[2], y2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int cc = c + u;
      const float mv = wm::plane_val(cm, i * PP + cc, PLN);
      a2[u] = cc <= i ? decay(vg[i] - vg[cc]) * mv * vbt[cc] : 0.f;
      y2[u] = vrk[cc] * (vbt[i] * wm::plane_val(p1, i * PP + cc, PLN) + vbt[cc] * wm::plane_val(p1, cc * PP + i, PLN));
    }
    wm::store_split2(cm + i * PP + c, cm + PLN + i * PP + c, a2[0], a2[1]);
    wm::store_split2(p4 + i * PP + c, p4 + PLN + i * PP + c, y2[0], y2[1]);
  }
  if (tid < C) {
    const int i = tid;
    vdb[i] += sum4(vxb, i);
    vdg[i] = sum4(vrow, i) - sum4(vcolp, i);
  }
  __syncthreads();

  // ---- C x D stage: warp tiles rows m0 .. m0 + 15, columns nd .. nd + D/2
  constexpr int NT = D / 32;
  const int nd = (D / 4) * (warp >> 2);
  {
    // dv = A^T dU   (A^T[j][i] = A[i][j], zero for i < j)
    float acc[1][NT][4];
    wm::zero(acc);
    wm::pgemm<1, NT, true, true, true, true>(acc, cm, cm + PLN, PP, pdu, pdu + TPL, DP, m0, nd, m0, C);
    wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
      if (i < len) *reinterpret_cast<float2*>(p.dv + ((t0 + i) * p.HV + hv) * D + c) = make_float2(x0, x1);
    });
  }
  {
    // dk^ = diag(e^g) A^T dW + diag(dec) dKr + (diag(1/|q|) (Gamma . dP))^T Q + Y K
    float acc[1][NT][4];
    wm::zero(acc);
    wm::pgemm<1, NT, true, true, true, true>(acc, cm, cm + PLN, PP, pu, pu + TPL, DP, m0, nd, m0, C);
    const float* dkr = p.dkr + item * C * D;
    float pa[2] = {0.f, 0.f}, pb[2] = {0.f, 0.f};
    wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
      const bool lo8 = i - m0 < 8;
      const float k0 = __bfloat162float(tk[i * DP + c]) * vrk[i], k1 = __bfloat162float(tk[i * DP + c + 1]) * vrk[i];
      const float2 kr = *reinterpret_cast<const float2*>(dkr + i * D + c);
      const float ya = fmaf(k0, x0, k1 * x1), yb = fmaf(k0, kr.x, k1 * kr.y);
      if (lo8) {
        pa[0] += ya;
        pb[0] += yb;
      } else {
        pa[1] += ya;
        pb[1] += yb;
      }
      x0 = veg[i] * x0 + vdec[i] * kr.x;
      x1 = veg[i] * x1 + vdec[i] * kr.y;
    });
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float a = quad_sum(pa[hh]), b2 = quad_sum(pb[hh]);
      if ((lane & 3) == 0) {
        const int i = m0 + r + 8 * hh;
        vpA[(warp >> 2) * C + i] = veg[i] * a;
        vpB[(warp >> 2) * C + i] = vdec[i] * b2;
      }
    }
    wm::pgemm<1, NT, true, true, true, false>(acc, p3, p3 + PLN, PP, tq, tq, DP, m0, nd, m0, C);
    wm::pgemm<1, NT, false, true, true, false>(acc, p4, p4 + PLN, PP, tk, tk, DP, m0, nd, 0, C);
    if (fused_norm)
      norm_backward<D, NT, NCW>(acc, tk, vrk, vnk, m0, nd, len, p.dk + (t0 * p.H + h) * D, (int64_t)p.H * D);
    else
      wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
        if (i < len) *reinterpret_cast<float2*>(p.dkh + ((t0 + i) * p.HV + hv) * D + c) = make_float2(x0, x1);
      });
  }
  {
    // dq^ = dQa + ((Gamma . dP) diag(1/|k|)) K
    float acc[1][NT][4];
    const float* dqa = p.dqa + item * C * D;
    float pc[2] = {0.f, 0.f};
    wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
      const float2 a = *reinterpret_cast<const float2*>(dqa + i * D + c);
      x0 = a.x;
      x1 = a.y;
      const float y = fmaf(__bfloat162float(tq[i * DP + c]), a.x, __bfloat162float(tq[i * DP + c + 1]) * a.y);
      if (i - m0 < 8) pc[0] += y; else pc[1] += y;
    });
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float s = quad_sum(pc[hh]);
      if ((lane & 3) == 0) {
        const int i = m0 + r + 8 * hh;
        vpC[(warp >> 2) * C + i] = vrq[i] * s;
      }
    }
    wm::pgemm<1, NT, false, true, true, false>(acc, p2, p2 + PLN, PP, tk, tk, DP, m0, nd, 0, m0 + 16);
    if (fused_norm)
      norm_backward<D, NT, NCW>(acc, tq, vrq, vnq, m0, nd, len, p.dq + (t0 * p.H + h) * D, (int64_t)p.H * D);
    else
      wm::for_each_pair(acc, m0, nd, [&](int i, int c, float& x0, float& x1) {
        if (i < len) *reinterpret_cast<float2*>(p.dqh + ((t0 + i) * p.HV + hv) * D + c) = make_float2(x0, x1);
      });
  }
  __syncthreads();
  if (tid < C) {
    const int i = tid;
    const float rb = sum4(vpB, i);
    vdg[i] += sum4(vpC, i) - rb + sum4(vpA, i);
    vrow[i] = rb;  // r_i, for the chunk-end term
  }
  __syncthreads();
  if (tid == 0) {
    float sr = 0.f;
    for (int i = 0; i < C; ++i) sr += vrow[i];
    vdg[C - 1] += sr + (p.dgc[2 * item] + p.dgc[2 * item + 1]);
    float run = 0.f;  // d log alpha_i = sum_{i' >= i} dg_i'
    for (int i = C - 1; i >= 0; --i) {
      run += vdg[i];
      vdg[i] = run;
    }
  }
  __syncthreads();
  if (tid < len) {
    const int64_t t = t0 + tid;
    const float dla = vdg[tid];
    const float x = p.a[t * p.HV + hv] + p.dt_bias[hv];
    const float eA = expf(p.A_log[hv]);
    const float sig = 1.f / (1.f + expf(-x));
    const float bt = vbt[tid];
    p.da[t * p.HV + hv] = dla * (-eA) * sig;
    p.db[t * p.HV + hv] = vdb[tid] * bt * (1.f - bt);
    p.dlala[t * p.HV + hv] = dla * (-eA * softplus_f(x));
  }
}

// ----------------------------------------------------------------------------- norm, gate sums

// One warp per (token, q/k head); each lane owns 4 consecutive elements of the row (lanes past D/4
// idle), so every load is 16 bytes, and all loads of the row are issued before the reductions.
template <int D, typename E>
__global__ void __launch_bounds__(256) bwd_norm_kernel(BwdParams p) {
  if (p.status[0] != GDN_OK) return;
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= p.T * p.H) return;
  const int64_t t = wid / p.H;
  const int h = (int)(wid % p.H), r = p.HV / p.H;
  const bool on = 4 * lane < D;
  const int d0 = on ? 4 * lane : 0;
  float x[2][4], g[2][4], n2[2], dot[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const E* src = static_cast<const E*>(w == 0 ? p.q : p.k) + (t * p.H + h) * D + d0;
    const float* gh = (w == 0 ? p.dqh : p.dkh) + (t * p.HV + (int64_t)h * r) * D + d0;
    const uint2 raw = *reinterpret_cast<const uint2*>(src);  // four 16-bit values
    const float2 a = ElemT<E>::unpack(raw.x), b = ElemT<E>::unpack(raw.y);
    x[w][0] = a.x;
    x[w][1] = a.y;
    x[w][2] = b.x;
    x[w][3] = b.y;
    float4 s = *reinterpret_cast<const float4*>(gh);
    for (int e = 1; e < r; ++e) {
      const float4 y = *reinterpret_cast<const float4*>(gh + (int64_t)e * D);
      s.x += y.x;
      s.y += y.y;
      s.z += y.z;
      s.w += y.w;
    }
    g[w][0] = s.x;
    g[w][1] = s.y;
    g[w][2] = s.z;
    g[w][3] = s.w;
  }
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    n2[w] = dot[w] = 0.f;
    if (on)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        n2[w] = fmaf(x[w][u], x[w][u], n2[w]);
        dot[w] = fmaf(x[w][u], g[w][u], dot[w]);
      }
    n2[w] = warp_sum(n2[w]);
    dot[w] = warp_sum(dot[w]);
  }
  if (!on) return;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    float* out = (w == 0 ? p.dq : p.dk) + (t * p.H + h) * D + d0;
    const float n = sqrtf(n2[w] + kNormEps);
    const float inv = 1.f / n, c3 = dot[w] / (n * n * n);
    *reinterpret_cast<float4*>(out) =
        make_float4(g[w][0] * inv - x[w][0] * c3, g[w][1] * inv - x[w][1] * c3, g[w][2] * inv - x[w][2] * c3,
                    g[w][3] * inv - x[w][3] * c3);
  }
}

__global__ void __launch_bounds__(256) bwd_gate_sum_kernel(BwdParams p) {
  __shared__ float s1[256], s2[256];
  if (p.status[0] != GDN_OK) return;
  const int hv = blockIdx.x, tid = threadIdx.x;
  float a1 = 0.f, a2 = 0.f;
  for (int64_t t = tid; t < p.T; t += 256) {
    a1 += p.dlala[t * p.HV + hv];
    a2 += p.da[t * p.HV + hv];
  }
  s1[tid] = a1;
  s2[tid] = a2;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if (tid < o) {
      s1[tid] += s1[tid + o];
      s2[tid] += s2[tid + o];
    }
    __syncthreads();
  }
  if (tid == 0) {
    p.dA_log[hv] = s1[0];
    p.ddt_bias[hv] = s2[0];
  }
}

template <typename Kern>
cudaError_t set_smem(Kern k, uint32_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int D, typename E>
cudaError_t launch_all(const BwdParams& p, cudaStream_t s, int* kernels) {
  cudaError_t e;
  int n = 0;
  if (p.max_chunks > 0x3fffffff) return cudaErrorInvalidConfiguration;  // 2 blocks per chunk in x
  const dim3 items((unsigned)p.max_chunks, (unsigned)p.HV);
  const unsigned chains = (unsigned)((int64_t)p.B * p.HV * (D / VB));
  constexpr bool f16in = kSplitSrc<E>;
  if ((e = set_smem(bwd_factor_kernel<D, E>, FacSmem<D, f16in>::bytes)) != cudaSuccess) return e;
  bwd_factor_kernel<D, E><<<items, 256, FacSmem<D, f16in>::bytes, s>>>(p);
  ++n;
  if (chains > 0) {
    const uint32_t sb = f16in ? StSmem<D>::bytes_fp16 : StSmem<D>::bytes_bf16;
    const uint32_t db = DsSmem<D, f16in>::bytes;
    if ((e = set_smem(bwd_state_kernel<D, E>, sb)) != cudaSuccess) return e;
    bwd_state_kernel<D, E><<<chains, 2 * kSeqThreads, sb, s>>>(p);
    if ((e = set_smem(bwd_dstate_kernel<D, E>, db)) != cudaSuccess) return e;
    bwd_dstate_kernel<D, E><<<chains, 2 * kSeqThreads, db, s>>>(p);
    n += 2;
  }
  if ((e = set_smem(bwd_sgrad_kernel<D, E>, SgSmem<D, f16in>::bytes)) != cudaSuccess) return e;
  bwd_sgrad_kernel<D, E><<<dim3(2 * items.x, items.y), 256, SgSmem<D, f16in>::bytes, s>>>(p);
  if (f16in) {  // fp16 inputs: the generic local kernel
    if ((e = set_smem(bwd_local_kernel<D, E>, LoSmem<D>::bytes)) != cudaSuccess) return e;
    bwd_local_kernel<D, E><<<items, 256, LoSmem<D>::bytes, s>>>(p);
  } else {
    if ((e = set_smem(bwd_local_fast_kernel<D>, LoFastSmem<D>::bytes)) != cudaSuccess) return e;
    bwd_local_fast_kernel<D><<<items, kLocalThreads, LoFastSmem<D>::bytes, s>>>(p);
  }
  n += 2;
  const int64_t rows = p.T * p.H;
  if (rows > 0 && p.HV != p.H) {  // grouped heads: sum the value heads' gradients, then the norm
    bwd_norm_kernel<D, E><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(p);
    ++n;
  }
  bwd_gate_sum_kernel<<<(unsigned)p.HV, 256, 0, s>>>(p);
  ++n;
  *kernels = n;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BwdParams& p, int D, bool fp16, cudaStream_t s, int* kernels) {
  *kernels = 0;
  if (D == 64) return fp16 ? launch_all<64, f16>(p, s, kernels) : launch_all<64, bf16>(p, s, kernels);
  if (D == 128) return fp16 ? launch_all<128, f16>(p, s, kernels) : launch_all<128, bf16>(p, s, kernels);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
