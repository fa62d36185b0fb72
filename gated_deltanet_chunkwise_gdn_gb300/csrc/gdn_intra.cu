// gdn_intra.cu — K2: per-chunk Gram products, the one triangular inverse and the WY
// factors, for every chunk of every sequence in parallel, on the 5th-generation tensor
// cores (tcgen05, fp32 accumulators in TMEM) with TMA tile loads.
//
// One CTA handles one (chunk, q/k head h) and loops over the HV/H value heads that read
// head h, so K^K^^T and Q^K^^T are formed once per q/k head. With the gates g and beta of
// the gates kernel it computes, per value head (notation of gdn_common.cuh):
//   M^{-1}   for M = I + tril(diag(beta) K^K^^T, -1)   (blocked forward substitution)
//   A        = (Gamma . M^{-1}) diag(beta)             (N^{-1} B = G M^{-1} G^{-1} B,
//                                                      "Simple math to speed up GDN
//                                                      prefill", section "Save one invert")
//   W<-      = A diag(exp(g)) K^,   U~ = A V,   P = Gamma . tril(Q^K^^T)
// and stores 1/|q|, 1/|k|, W<- [C][K], U~ [C][V] and P [C][C] for the scan.
//
// For K = V = 128 the scan runs in affine-transition form and needs the per-row factor
// sk_t = exp(g_C - g_t)/|k_t| applied to the chunk's keys. It is split exactly into a
// mantissa and a power of two, sk_t = m_t 2^e_t with m_t in [0.5, 1): this kernel folds m_t
// into the rows of W<- and U~ and 1/m_t into the columns of P (so P U stays unchanged), and
// stores ks_t = 2^e_t, which the scan applies to the raw 16-bit keys without rounding.
//
// Tensor-core work (one elected thread issues, the accumulators live in TMEM):
//   MMA1  D1[128 x 128] = [K; Q] [K; Q]^T       (columns 0-63: K K^T in rows 0-63, Q K^T in rows 64-127;
//                                                the diagonal: |k|^2 and |q|^2, so no pass over the tiles)
//   MMA2  DW[128 x D]   = [A'; A] K             (rows 0-63: W<- = A' K with A' = A diag(e^g/|k|))
//   MMA3  DU[128 x D]   = [A'; A] V             (rows 64-127: U~ = A V)
// Stacking A' and A keeps every MMA at M = 128 and puts W<- and U~ rows in TMEM lanes, so
// each thread stores one contiguous output row. Normalisation and decay enter only as
// diagonal scalings of fp32 accumulators or of the C x C operand; the raw 16-bit q/k/v tiles
// feed the tensor cores as TMA wrote them (128-byte swizzle, K-major for MMA1, the same
// bytes read MN-major for MMA2/3).
#include "gdn_common.cuh"
#include "gdn_inverse.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

using inv::diag_blocks;
using inv::offdiag_blocks;

constexpr int C = 64;
constexpr int kThreads = 256;  // 8 warps; warps w and w+4 share TMEM lanes 32(w%4)..+31

template <int D>
struct IntraSmem {
  static constexpr int NB = D / 64;                     // 64-column blocks of a q/k/v row
  static constexpr uint32_t KQ = 0;                     // NB x [K block 8 KB][Q block 8 KB]
  static constexpr uint32_t V = KQ + NB * 16384;        // NB x V block 8 KB
  static constexpr uint32_t AA = V + NB * 8192;         // [A' 8 KB][A 8 KB], 128-byte swizzled
  static constexpr int LDF = 68;                        // fp32 tile pitch: conflict-free fragment loads
  static constexpr uint32_t LF = AA + 16384;            // L, fp32 64 x LDF; then the low parts of [A'; A]
  static constexpr uint32_t XF = LF + 64 * LDF * 4;     // M^{-1}, fp32 64 x LDF
  static constexpr uint32_t VEC = XF + 64 * LDF * 4;    // g, beta, 1/|q|, 1/|k|, m, 1/m, g log2(e), P's column factor (8 x 64 fp32)
  static constexpr uint32_t BAR = VEC + 8 * 64 * 4;     // 3 mbarriers + TMEM address
  static constexpr uint32_t bytes = BAR + 96;
  static constexpr uint32_t alloc = bytes + 1024;      // slack to round the base up to 1 KB
};

// TMEM columns: D1 and then DW from column 0, DU from column tmem_u<D>; D <= 128 takes 256
// columns, D = 256 all 512.
template <int D>
__host__ __device__ constexpr uint32_t tmem_u() { return D < 128 ? 128u : (uint32_t)D; }
template <int D>
__host__ __device__ constexpr uint32_t tmem_cols() { return D < 256 ? 256u : 512u; }


constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the SFU's approximation (relative error about 2^-22); e^(a - b) is ex2(a log2(e) - b log2(e)).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Gates of value head hv for the chunk (from the gates kernel), and g log2(e). All threads.
__device__ __forceinline__ void load_gates(const Params& p, int64_t jh, float* s_g, float* s_beta, float* s_g2) {
  const int tid = threadIdx.x;
  if (tid < C) {
    const float g = p.g[jh * C + tid];
    s_g[tid] = g;
    s_g2[tid] = g * kLog2e;
    s_beta[tid] = p.beta[jh * C + tid];
  }
  __syncthreads();
}

// All threads: bounded wait; every thread leaves with the same outcome.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, int32_t* status, long long budget) {
  const bool ok = tc::mbar_wait(bar, parity, budget);
  const bool all = __syncthreads_and(ok);
  if (!all && threadIdx.x == 0) set_status(status, GDN_ERR_TIMEOUT);
  return all;
}

// Persistent: each CTA takes items (item = chunk * H + q/k head) from a global counter until
// they run out. The next item's q/k/v tiles and gates are fetched by TMA while the current
// item's W<- and U~ rows are written out (for D <= 128 through shared memory and TMA stores).
template <int D, typename E>
__global__ void __launch_bounds__(kThreads, 2) intra_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                         const __grid_constant__ CUtensorMap tm_k,
                                                         const __grid_constant__ CUtensorMap tm_v,
                                                         const __grid_constant__ CUtensorMap tm_w,
                                                         const __grid_constant__ CUtensorMap tm_u, Params p) {
  using SM = IntraSmem<D>;
  constexpr int NB = SM::NB;
  constexpr int LDF = SM::LDF;
  constexpr bool kTmaStore = D <= 128;  // W<- and U~ tiles staged in the [A'; A] and L buffers
  constexpr bool kAffine = D == 128;    // rows of W<-, U~ scaled by m_t, columns of P by 1/m_t
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  if (p.status[0] != GDN_OK) return;
  const int n_items = p.status[1] * p.H;
  if ((int)blockIdx.x >= n_items) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = warp & 3;         // TMEM lane quarter of this warp
  const int half = warp >> 2;       // which half of a row's columns this warp handles
  const int row = 32 * sub + lane;  // TMEM lane / accumulator row of this thread
  const int cbase = 32 * half;      // first column of this thread's half row
  const int r_heads = p.HV / p.H;

  float* Lf = reinterpret_cast<float*>(smem + SM::LF);
  float* Xf = reinterpret_cast<float*>(smem + SM::XF);
  float* s_g = reinterpret_cast<float*>(smem + SM::VEC);
  float* s_beta = s_g + C;
  float* s_rq = s_beta + C;
  float* s_rk = s_rq + C;
  float* s_m = s_rk + C;   // K = V = 128: mantissa m_t of sk_t = exp(g_C - g_t)/|k_t| = m_t 2^e_t
  float* s_im = s_m + C;   // 1/m_t
  float* s_g2 = s_im + C;  // g log2(e)
  float* s_cf = s_g2 + C;  // column factor of P: 1/|k_t| (times 1/m_t for K = V = 128)
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SM::BAR);  // [0] q/k tiles + gates, [1] v tile, [2] MMAs
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 3);
  int4* s_ct = reinterpret_cast<int4*>(bar + 4);                // chunk record of the item being fetched
  int* s_next = reinterpret_cast<int*>(bar + 6);                 // this CTA's next item
  int4* s_ct_next = reinterpret_cast<int4*>(bar + 8);            // its chunk record

  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_init(&bar[2], 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, tmem_cols<D>());
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(32 * sub) << 16;

  // thread 0: fetch an item's k, q tiles and its first value head's gates (bar[0]) and v tile (bar[1])
  auto fetch_item = [&](int item, int4 ct) {
    const int j = item / p.H, h = item % p.H;
    const int64_t jh0 = (int64_t)j * p.HV + h * r_heads;
    *s_ct = ct;
    tc::mbar_arrive_expect_tx(&bar[0], NB * 16384 + 2 * C * 4);
    tc::bulk_load(s_g, p.g + jh0 * C, C * 4, &bar[0]);
    tc::bulk_load(s_beta, p.beta + jh0 * C, C * 4, &bar[0]);
    for (int b = 0; b < NB; ++b) {
      tc::tma_load_3d(smem + SM::KQ + b * 16384, &tm_k, 64 * b, h, ct.y, &bar[0]);
      tc::tma_load_3d(smem + SM::KQ + b * 16384 + 8192, &tm_q, 64 * b, h, ct.y, &bar[0]);
    }
    tc::mbar_arrive_expect_tx(&bar[1], NB * 8192);
    for (int b = 0; b < NB; ++b) tc::tma_load_3d(smem + SM::V + b * 8192, &tm_v, 64 * b, h * r_heads, ct.y, &bar[1]);
  };
  // Items are handed out by a counter in the status words (zeroed by the schedule kernel), so a
  // CTA that starts late simply takes fewer items.
  if (tid == 0) {
    const int first = atomicAdd(&p.status[2], 1);
    *s_next = first;
    if (first < n_items && p.stall != kStallIntra) fetch_item(first, p.chunk_tab[first / p.H]);
  }
  __syncthreads();
  int item = *s_next;

  uint32_t ph0 = 0, ph1 = 0, ph2 = 0;  // completed phases of bar[0], bar[1], bar[2]
  bool ok = true;
  while (ok && item < n_items) {
    const int j = item / p.H, h = item % p.H;
    const int hv0 = h * r_heads;

    ok = wait_all(&bar[0], ph0 & 1, p.status, p.wait_budget);
    ++ph0;
    if (!ok) break;
    const int4 ct = *s_ct;
    const int len = ct.z;
    if (tid == 0) {  // MMA1: D1 = [K; Q] [K; Q]^T (columns 0-63: K K^T and Q K^T; the diagonal: |k|^2, |q|^2)
      tc::fence_after_sync();
      constexpr uint32_t idesc1 = tc::idesc_f16(128, 128, ElemT<E>::fmt, false, false);
      const uint64_t d0 = tc::smem_desc(tc::saddr(smem + SM::KQ), 16, 1024, tc::kSwizzle128B);
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t d = d0 + ((b * 16384 + ks * 32) >> 4);
          tc::mma_f16_ss(tmem, d, d, idesc1, (b | ks) != 0);
        }
      tc::mma_commit(&bar[2]);
    }
    if (kTmaStore && tid == 0) tc::bulk_wait_read();  // the previous item's staged W<-, U~ have been read
    ok = wait_all(&bar[2], ph2 & 1, p.status, p.wait_budget);
    ++ph2;
    if (!ok) break;
    float kq[32];  // columns [32*half, 32*half+32) of this row of K K^T (rows 0-63) or Q K^T (64-127)
    tc::fence_after_sync();
    {
      uint32_t r0[16], r1[16];
      tc::tmem_ld16(tmem + lane_base + 32 * half, r0);
      tc::tmem_ld16(tmem + lane_base + 32 * half + 16, r1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        kq[u] = __uint_as_float(r0[u]);
        kq[16 + u] = __uint_as_float(r1[u]);
      }
    }
    if (tid >= 128 && tid < 128 + C) s_g2[tid - 128] = s_g[tid - 128] * kLog2e;
    if (tid < 128) {  // 1/|k| (rows 0-63) and 1/|q| (rows 64-127), 0 on padded rows, from the diagonal of
                      // D1: warp w's columns 32 w .. 32 w + 31 hold it for each lane's row (row = tid)
      float ss = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t dd[16];
        tc::tmem_ld16(tmem + lane_base + 32 * warp + 16 * hh, dd);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 16; ++u) ss = lane == 16 * hh + u ? __uint_as_float(dd[u]) : ss;
      }
      const int r64 = tid & 63;
      const float r = r64 < len ? rsqrtf(ss + kNormEps) : 0.f;
      const int64_t jq = (int64_t)j * p.H + h;
      if (tid < 64) {
        s_rk[r64] = r;
        p.rk[jq * C + r64] = r;
      } else {
        s_rq[r64] = r;
        p.rq[jq * C + r64] = r;
      }
    }
    // D1 is read: the later MMAs that overwrite its columns are issued after the barriers below
    tc::fence_before_sync();
    __syncthreads();  // 1/|k|, 1/|q| of every row are in place

    for (int ih = 0; ih < r_heads; ++ih) {
      const int hv = hv0 + ih;
      const int64_t jh = (int64_t)j * p.HV + hv;
      if (ih > 0) load_gates(p, jh, s_g, s_beta, s_g2);
      if (row < C) {  // warps 0, 1, 4, 5: L = tril(diag(beta) K^K^^T, -1), row i; diagonal blocks of M^{-1}
        const int i = row;
        const float bi = s_beta[i] * s_rk[i];
        // warp 4's part (rows 0-31, columns 32-63) is strictly upper: nothing reads it
#pragma unroll
        for (int u = 0; u < 32; u += 4) {
          if (warp == 4) break;
          const float4 rk4 = *reinterpret_cast<const float4*>(s_rk + cbase + u);
          const int nu = cbase + u;
          float4 l4;
          l4.x = nu < i ? bi * rk4.x * kq[u] : 0.f;
          l4.y = nu + 1 < i ? bi * rk4.y * kq[u + 1] : 0.f;
          l4.z = nu + 2 < i ? bi * rk4.z * kq[u + 2] : 0.f;
          l4.w = nu + 3 < i ? bi * rk4.w * kq[u + 3] : 0.f;
          *reinterpret_cast<float4*>(Lf + i * LDF + nu) = l4;
        }
        // warp 0 holds the L rows of diagonal blocks 0, 1 (rows 0-31, columns 0-31) and warp 5 those of
        // blocks 2, 3 (rows 32-63, columns 32-63): each sweeps its own two blocks
        __syncwarp();
        if (warp == 0 || warp == 5) diag_blocks<LDF>(Lf, Xf, warp == 0 ? 0 : 1);
      } else {  // warps 2, 3, 6, 7 meanwhile: P = Gamma . tril(Q^K^^T), row r, straight to global
        const int r = row - C;
        if constexpr (kAffine) {  // sk_t = m_t 2^e_t, m_t in [0.5, 1); padded rows (1/|k| = 0): m = 1, ks = 0
          if (half == 0) {
            const float sk = expf(s_g[C - 1] - s_g[r]) * s_rk[r];
            float m = 1.f, ks = 0.f;
            if (sk > 0.f) {
              int e;
              m = frexpf(sk, &e);
              ks = ldexpf(1.f, e);
            }
            s_m[r] = m;
            s_im[r] = 1.f / m;
            s_cf[r] = s_rk[r] * (1.f / m);
            p.ks[jh * C + r] = ks;
          }
          tc::named_sync(3, 128);
        }
        const float* cf = kAffine ? s_cf : s_rk;
        const float qr = s_rq[r], gr2 = s_g2[r];
        uint4* prow = reinterpret_cast<uint4*>(p.P + (jh * C + r) * C + cbase);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int n0 = cbase + 8 * c;
          if (n0 > r) {  // strictly upper: zeros (a whole warp's columns for warp 6)
            prow[c] = make_uint4(0u, 0u, 0u, 0u);
            continue;
          }
          float g8[8], c8[8];  // g log2(e) and the column factor of columns n0 .. n0+7
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            *reinterpret_cast<float4*>(g8 + 4 * q) = *reinterpret_cast<const float4*>(s_g2 + n0 + 4 * q);
            *reinterpret_cast<float4*>(c8 + 4 * q) = *reinterpret_cast<const float4*>(cf + n0 + 4 * q);
          }
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float v[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int m = 2 * u + e;
              const float x = ex2(gr2 - g8[m]) * (qr * kq[8 * c + m]) * c8[m];
              v[e] = n0 + m <= r ? x : 0.f;
            }
            w[u] = ElemT<E>::pack(v[0], v[1]);
          }
          prow[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      __syncthreads();
      offdiag_blocks<LDF>(Lf, Xf);
      // L is dead from here on: its buffer takes the low 16-bit parts of [A'; A]
      {  // A' rows (rows 0-63) and A rows (rows 64-127) as 16-bit hi + lo, 128-byte swizzled K-major.
         // Thread (i, qc) forms columns 16 qc .. 16 qc + 15 of row i of both A' and A, so each X element
         // is loaded once and the exp of A's decay factor is spread over all eight warps.
        const int i = row & 63;
        const int qc = 2 * half + (row >> 6);  // 16-column group of this thread
        const float gi = s_g[i], egi = expf(gi), gi2 = s_g2[i];
        const float mi = kAffine ? s_m[i] : 1.f;  // row scale of W<- and U~
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int n0 = 16 * qc + 8 * c;
          const uint32_t o = tc::sw128_offset(i, n0 >> 3);
          if (n0 > i) {  // strictly upper: zeros (every column of warps 4 and 6)
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(smem + SM::AA + o) = z;
            *reinterpret_cast<uint4*>(smem + SM::LF + o) = z;
            *reinterpret_cast<uint4*>(smem + SM::AA + 8192 + o) = z;
            *reinterpret_cast<uint4*>(smem + SM::LF + 8192 + o) = z;
            continue;
          }
          float x8[8], g8[8], b8[8], k8[8];  // X row i, and g log2(e), beta, 1/|k| of columns n0 .. n0+7
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            *reinterpret_cast<float4*>(x8 + 4 * q) = *reinterpret_cast<const float4*>(Xf + i * LDF + n0 + 4 * q);
            *reinterpret_cast<float4*>(g8 + 4 * q) = *reinterpret_cast<const float4*>(s_g2 + n0 + 4 * q);
            *reinterpret_cast<float4*>(b8 + 4 * q) = *reinterpret_cast<const float4*>(s_beta + n0 + 4 * q);
            *reinterpret_cast<float4*>(k8 + 4 * q) = *reinterpret_cast<const float4*>(s_rk + n0 + 4 * q);
          }
          uint32_t ah[4], al[4], bh[4], bl[4];  // A' and A, hi and lo
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float va[2], vb[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int m = 2 * u + e, nu = n0 + m;
              const float x = nu == i ? 1.f : x8[m];  // entries above the diagonal are never read
              const float xb = x * b8[m] * mi;
              va[e] = nu <= i ? egi * xb * k8[m] : 0.f;          // A'[i][nu] = e^{g_i} X beta_nu / |k_nu| m_i
              vb[e] = nu <= i ? ex2(gi2 - g8[m]) * xb : 0.f;     // A[i][nu] = e^{g_i - g_nu} X beta_nu m_i
            }
            split2<E>(va[0], va[1], ah[u], al[u]);
            split2<E>(vb[0], vb[1], bh[u], bl[u]);
          }
          *reinterpret_cast<uint4*>(smem + SM::AA + o) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
          *reinterpret_cast<uint4*>(smem + SM::LF + o) = make_uint4(al[0], al[1], al[2], al[3]);
          *reinterpret_cast<uint4*>(smem + SM::AA + 8192 + o) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
          *reinterpret_cast<uint4*>(smem + SM::LF + 8192 + o) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
        }
      }
      tc::fence_async_smem();
      ok = wait_all(&bar[1], ph1 & 1, p.status, p.wait_budget);  // its barrier also publishes [A'; A] to the MMA issuer
      ++ph1;
      if (!ok) break;
      // thread 32 claims the next item while the MMAs below run, so the atomic's round trip stays off
      // the chain of barriers (every thread read the previous claim before this item's first barrier;
      // thread 0 reads this one after the MMA barrier below, all threads at the end of the item)
      if (ih == 0 && tid == 32) {
        const int nx = atomicAdd(&p.status[2], 1);
        *s_next = nx;
        if (nx < n_items) *s_ct_next = p.chunk_tab[nx / p.H];
      }
      if (tid == 0) {  // DW = [A'; A] K (rows 0-63: W<-), DU = [A'; A] V (rows 64-127: U~), [A'; A] = hi + lo
        tc::fence_after_sync();
        constexpr uint32_t idesc2 = tc::idesc_f16(128, D, ElemT<E>::fmt, false, true);
        const uint64_t da = tc::smem_desc(tc::saddr(smem + SM::AA), 16, 1024, tc::kSwizzle128B);
        const uint64_t dk = tc::smem_desc(tc::saddr(smem + SM::KQ), 16384, 1024, tc::kSwizzle128B);
        const uint64_t dv = tc::smem_desc(tc::saddr(smem + SM::V), 8192, 1024, tc::kSwizzle128B);
        static_assert(SM::LF == SM::AA + 16384, "the low parts follow the high parts");
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)
            tc::mma_f16_ss(tmem, da + ((part * 16384 + ks * 32) >> 4), dk + ((ks * 2048) >> 4), idesc2, (part | ks) != 0);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)
            tc::mma_f16_ss(tmem + tmem_u<D>(), da + ((part * 16384 + ks * 32) >> 4), dv + ((ks * 2048) >> 4), idesc2,
                           (part | ks) != 0);
        tc::mma_commit(&bar[2]);
      }
      ok = wait_all(&bar[2], ph2 & 1, p.status, p.wait_budget);
      ++ph2;
      if (!ok) break;
      tc::fence_after_sync();
      if (tid == 0) {  // the k, q, v tiles are free: fetch what comes next
        if (ih + 1 < r_heads) {
          tc::mbar_arrive_expect_tx(&bar[1], NB * 8192);
          for (int b = 0; b < NB; ++b)
            tc::tma_load_3d(smem + SM::V + b * 8192, &tm_v, 64 * b, hv + 1, ct.y, &bar[1]);
        } else if (*s_next < n_items) {
          fetch_item(*s_next, *s_ct_next);
        }
      }
      {  // rows 0-63 of DW are W<-, rows 64-127 of DU are U~: half an output row per thread
        const bool is_u = row >= 64;
        const int mu = row & 63;
        const uint32_t col0 = (is_u ? tmem_u<D>() : 0u) + half * (D / 2);
        E* dst = reinterpret_cast<E*>(is_u ? p.U : p.W) + (jh * C + mu) * D + half * (D / 2);
        // D <= 128: 64-column block `half` of the staged tile (128-byte swizzled, the TMA box)
        unsigned char* stage = smem + (is_u ? SM::LF : SM::AA) + (D == 128 ? half * 8192 : 0);
        constexpr int NG = D / 32, GB = NG < 4 ? NG : 4;  // 16-column groups, loaded GB at a time
#pragma unroll
        for (int g0 = 0; g0 < NG; g0 += GB) {
          uint32_t r[GB][16];
#pragma unroll
          for (int c = 0; c < GB; ++c) tc::tmem_ld16(tmem + lane_base + col0 + 16 * (g0 + c), r[c]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < GB; ++c) {
            uint32_t w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) w[u] = ElemT<E>::pack(__uint_as_float(r[c][2 * u]), __uint_as_float(r[c][2 * u + 1]));
            if constexpr (kTmaStore) {
              const int ch = (D == 128 ? 0 : half * 4) + 2 * (g0 + c);  // 16-byte chunk within the 128-byte row
              *reinterpret_cast<uint4*>(stage + tc::sw128_offset(mu, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(stage + tc::sw128_offset(mu, ch + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * (g0 + c));
              d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
              d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
      }
      tc::fence_before_sync();
      if constexpr (kTmaStore) tc::fence_async_smem();
      __syncthreads();
      if (kTmaStore && tid == 0) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          tc::tma_store_2d(&tm_w, smem + SM::AA + b * 8192, 64 * b, (int)(jh * C));
          tc::tma_store_2d(&tm_u, smem + SM::LF + b * 8192, 64 * b, (int)(jh * C));
        }
        tc::bulk_commit();
        if (ih + 1 < r_heads) tc::bulk_wait_read();  // the next value head rebuilds [A'; A] in these buffers
      }
    }
    item = *s_next;
  }

  if (kTmaStore && tid == 0) tc::bulk_wait_all();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols<D>());
  }
}

template <int D, typename E>
cudaError_t launch_intra_t(const Params& p, cudaStream_t s) {
  const bool h = p.fp16 != 0;
  CUtensorMap mq, mk, mv, mw, mu;
  const int64_t rows = p.max_chunks * p.HV * C;  // rows of the W<- and U~ arrays
  if (!make_token_tile_map(&mq, p.q, D, p.H, p.T, C, h) || !make_token_tile_map(&mk, p.k, D, p.H, p.T, C, h) ||
      !make_token_tile_map(&mv, p.v, D, p.HV, p.T, C, h) || !make_2d_tile_map(&mw, p.W, D, rows, 64, C, true, h) ||
      !make_2d_tile_map(&mu, p.U, D, rows, 64, C, true, h))
    return cudaErrorInvalidValue;
  const uint32_t smem = IntraSmem<D>::alloc;
  cudaError_t e = cudaFuncSetAttribute(intra_kernel<D, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // persistent: two CTAs per SM (TMEM and shared memory allow two), never more than the items
  const int64_t items = p.max_chunks * p.H;
  const int64_t blocks = items < 2 * (int64_t)sms ? items : 2 * (int64_t)sms;
  intra_kernel<D, E><<<(unsigned)blocks, kThreads, smem, s>>>(mq, mk, mv, mw, mu, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra(const Params& p, int D, int Cc, cudaStream_t s) {
  if (Cc != C) return cudaErrorInvalidValue;
  switch (D) {
    case 64: return p.fp16 ? launch_intra_t<64, f16>(p, s) : launch_intra_t<64, bf16>(p, s);
    case 128: return p.fp16 ? launch_intra_t<128, f16>(p, s) : launch_intra_t<128, bf16>(p, s);
    case 256: return p.fp16 ? launch_intra_t<256, f16>(p, s) : launch_intra_t<256, bf16>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
