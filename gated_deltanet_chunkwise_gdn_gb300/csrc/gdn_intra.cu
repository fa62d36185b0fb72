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
// Tensor-core work (one elected thread issues, the accumulators live in TMEM):
//   MMA1  D1[128 x 64]  = [K; Q] K^T            (M=128: rows 0-63 K K^T, rows 64-127 Q K^T)
//   MMA2  DW[128 x D]   = [A'; A] K             (rows 0-63: W<- = A' K with A' = A diag(e^g/|k|))
//   MMA3  DU[128 x D]   = [A'; A] V             (rows 64-127: U~ = A V)
// Stacking A' and A keeps every MMA at M = 128 and puts W<- and U~ rows in TMEM lanes, so
// each thread stores one contiguous output row. Normalisation and decay enter only as
// diagonal scalings of fp32 accumulators or of the C x C operand; the raw bf16 q/k/v tiles
// feed the tensor cores as TMA wrote them (128-byte swizzle, K-major for MMA1, the same
// bytes read MN-major for MMA2/3).
#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int C = 64;
constexpr int kThreads = 256;  // 8 warps; warps w and w+4 share TMEM lanes 32(w%4)..+31
constexpr long long kWaitBudget = 1ll << 31;  // clock cycles before a wait gives up (~1 s)

template <int D>
struct IntraSmem {
  static constexpr int NB = D / 64;                     // 64-column blocks of a q/k/v row
  static constexpr uint32_t KQ = 0;                     // NB x [K block 8 KB][Q block 8 KB]
  static constexpr uint32_t V = KQ + NB * 16384;        // NB x V block 8 KB
  static constexpr uint32_t AA = V + NB * 8192;         // [A' 8 KB][A 8 KB], 128-byte swizzled
  static constexpr int LDF = 68;                        // fp32 tile pitch: conflict-free fragment loads
  static constexpr uint32_t LF = AA + 16384;            // L, fp32 64 x LDF; then the low parts of [A'; A]
  static constexpr uint32_t XF = LF + 64 * LDF * 4;     // M^{-1}, fp32 64 x LDF
  static constexpr uint32_t VEC = XF + 64 * LDF * 4;    // g, beta, 1/|q|, 1/|k| (4 x 64 fp32)
  static constexpr uint32_t BAR = VEC + 4 * 64 * 4;     // 3 mbarriers + TMEM address
  static constexpr uint32_t bytes = BAR + 64;
  static constexpr uint32_t alloc = bytes + 1024;      // slack to round the base up to 1 KB
};

// TMEM columns: D1 and then DW from column 0, DU from column tmem_u<D>; D <= 128 takes 256
// columns, D = 256 all 512.
template <int D>
__host__ __device__ constexpr uint32_t tmem_u() { return D < 128 ? 128u : (uint32_t)D; }
template <int D>
__host__ __device__ constexpr uint32_t tmem_cols() { return D < 256 ? 256u : 512u; }


__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
// x = hi + lo with both parts representable in tf32 (3xTF32 products keep ~fp32 accuracy).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One warp: acc (16 x 16, two 16x8 accumulator tiles) += A (16 x 16) * B (16 x 16), both
// fp32 row-major in shared memory with pitch LDF, as 3xTF32 tensor-core products.
template <int LDF>
__device__ __forceinline__ void mm16_acc(float (&acc)[2][4], const float* A, const float* B) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    uint32_t ah[4], al[4];
    split_tf32(A[g * LDF + 8 * ks + t], ah[0], al[0]);
    split_tf32(A[(g + 8) * LDF + 8 * ks + t], ah[1], al[1]);
    split_tf32(A[g * LDF + 8 * ks + t + 4], ah[2], al[2]);
    split_tf32(A[(g + 8) * LDF + 8 * ks + t + 4], ah[3], al[3]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t bh0, bl0, bh1, bl1;
      split_tf32(B[(8 * ks + t) * LDF + 8 * nt + g], bh0, bl0);
      split_tf32(B[(8 * ks + t + 4) * LDF + 8 * nt + g], bh1, bl1);
      mma_tf32_1688(acc[nt], ah, bh0, bh1);
      mma_tf32_1688(acc[nt], ah, bl0, bl1);
      mma_tf32_1688(acc[nt], al, bh0, bh1);
    }
  }
}

// Inverts the unit lower-triangular 64x64 matrix I + L (L strictly lower, in Lf) into Xf,
// by 16x16 blocks: the four diagonal blocks by forward substitution (one warp each, one
// lane per column, in registers), then block rows I = 1..3, one warp per block, with
//   X_IJ = -X_II * sum_{K=J}^{I-1} L_IK X_KJ
// formed as 3xTF32 warp-level tensor-core products (fp32 accuracy up to rounding order).
// Run by four warps (lw = 0..3 among them) that meet at named barrier 2.
template <int LDF>
__device__ void invert_unit_lower_64(const float* Lf, float* Xf, int lw) {
  const int warp = lw, lane = threadIdx.x & 31;
  {
    const int b = warp * 16;
    const int c = lane & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
      for (int kk = 0; kk < i; ++kk) acc -= Lf[(b + i) * LDF + b + kk] * x[kk];
      x[i] = acc;
    }
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) Xf[(b + i) * LDF + b + c] = x[i];
    }
  }
  tc::named_sync(2, 128);
  const int g = lane >> 2, t = lane & 3;
  for (int I = 1; I < 4; ++I) {
    if (warp < I) {
      const int J = warp;
      float acc[2][4] = {};
      for (int K = J; K < I; ++K) mm16_acc<LDF>(acc, Lf + 16 * I * LDF + 16 * K, Xf + 16 * K * LDF + 16 * J);
      float* xij = Xf + 16 * I * LDF + 16 * J;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {  // T_IJ into the X_IJ slot
        xij[g * LDF + 8 * nt + 2 * t] = acc[nt][0];
        xij[g * LDF + 8 * nt + 2 * t + 1] = acc[nt][1];
        xij[(g + 8) * LDF + 8 * nt + 2 * t] = acc[nt][2];
        xij[(g + 8) * LDF + 8 * nt + 2 * t + 1] = acc[nt][3];
      }
      __syncwarp();
      float acc2[2][4] = {};
      mm16_acc<LDF>(acc2, Xf + 16 * I * LDF + 16 * I, xij);
      __syncwarp();
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        xij[g * LDF + 8 * nt + 2 * t] = -acc2[nt][0];
        xij[g * LDF + 8 * nt + 2 * t + 1] = -acc2[nt][1];
        xij[(g + 8) * LDF + 8 * nt + 2 * t] = -acc2[nt][2];
        xij[(g + 8) * LDF + 8 * nt + 2 * t + 1] = -acc2[nt][3];
      }
    }
    tc::named_sync(2, 128);
  }
}

// Gates of value head hv for the chunk (from the gates kernel). All threads.
__device__ __forceinline__ void load_gates(const Params& p, int64_t jh, float* s_g, float* s_beta) {
  const int tid = threadIdx.x;
  if (tid < C) {
    s_g[tid] = p.g[jh * C + tid];
    s_beta[tid] = p.beta[jh * C + tid];
  }
  __syncthreads();
}

// All threads: bounded wait; every thread leaves with the same verdict.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, int32_t* status) {
  const bool ok = tc::mbar_wait(bar, parity, kWaitBudget);
  const bool all = __syncthreads_and(ok);
  if (!all && threadIdx.x == 0) set_status(status, GDN_ERR_TIMEOUT);
  return all;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) intra_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                         const __grid_constant__ CUtensorMap tm_k,
                                                         const __grid_constant__ CUtensorMap tm_v, Params p) {
  using SM = IntraSmem<D>;
  constexpr int NB = SM::NB;
  constexpr int LDF = SM::LDF;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  if (p.status[0] != GDN_OK) return;
  const int j = blockIdx.x / p.H, h = blockIdx.x % p.H;
  if (j >= p.status[1]) return;
  const int4 ct = p.chunk_tab[j];
  const int64_t t0 = ct.y;
  const int len = ct.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = warp & 3;       // TMEM lane quarter of this warp
  const int half = warp >> 2;     // which half of a row's columns this warp handles
  const int row = 32 * sub + lane;  // TMEM lane / accumulator row of this thread
  const int r_heads = p.HV / p.H;
  const int hv0 = h * r_heads;

  float* Lf = reinterpret_cast<float*>(smem + SM::LF);
  float* Xf = reinterpret_cast<float*>(smem + SM::XF);
  float* s_g = reinterpret_cast<float*>(smem + SM::VEC);
  float* s_beta = s_g + C;
  float* s_rq = s_beta + C;
  float* s_rk = s_rq + C;
  float* s_part = reinterpret_cast<float*>(smem + SM::XF);  // norm partial sums (before X is formed)
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SM::BAR);  // [0] q/k tiles, [1] v tile, [2] MMAs
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 3);

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

  if (tid == 0) {
    const int64_t jh0 = (int64_t)j * p.HV + hv0;
    tc::mbar_arrive_expect_tx(&bar[0], NB * 16384 + 2 * C * 4);
    tc::bulk_load(s_g, p.g + jh0 * C, C * 4, &bar[0]);
    tc::bulk_load(s_beta, p.beta + jh0 * C, C * 4, &bar[0]);
    for (int b = 0; b < NB; ++b) {
      tc::tma_load_3d(smem + SM::KQ + b * 16384, &tm_k, 64 * b, h, (int)t0, &bar[0]);
      tc::tma_load_3d(smem + SM::KQ + b * 16384 + 8192, &tm_q, 64 * b, h, (int)t0, &bar[0]);
    }
    tc::mbar_arrive_expect_tx(&bar[1], NB * 8192);
    for (int b = 0; b < NB; ++b) tc::tma_load_3d(smem + SM::V + b * 8192, &tm_v, 64 * b, hv0, (int)t0, &bar[1]);
  }

  bool ok = wait_all(&bar[0], 0, p.status);
  if (ok && tid == 0) {
    constexpr uint32_t idesc1 = tc::idesc_f16(128, 64, 1, false, false);
    for (int b = 0; b < NB; ++b)
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t a = tc::saddr(smem + SM::KQ + b * 16384) + ks * 32;
        const uint64_t d = tc::smem_desc(a, 16, 1024, tc::kSwizzle128B);
        tc::mma_f16_ss(tmem, d, d, idesc1, (b | ks) != 0);
      }
    tc::mma_commit(&bar[2]);
  }
  if (ok) {
    // squared row norms from the swizzled tiles: rows 0-63 k, 64-127 q; each half of the
    // threads sums half of the 16-byte chunks of the row
    const int r64 = row & 63;
    const unsigned char* base = smem + SM::KQ + (row >= 64 ? 8192 : 0);
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < 4 * NB; ++q) {
      const int cg = half * 4 * NB + q;  // chunk index over the whole row
      const uint4 v4 = *reinterpret_cast<const uint4*>(base + (cg >> 3) * 16384 + tc::sw128_offset(r64, cg & 7));
      const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(e[u]);
        ss += f.x * f.x + f.y * f.y;
      }
    }
    s_part[half * 128 + row] = ss;
  }
  __syncthreads();
  if (ok && tid < 128) {
    const int r64 = tid & 63;
    const float ss = s_part[tid] + s_part[128 + tid];
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
  if (ok) ok = wait_all(&bar[2], 0, p.status);
  float kq[32];  // columns [32*half, 32*half+32) of this row of K K^T (rows 0-63) or Q K^T (64-127)
  if (ok) {
    tc::fence_after_sync();
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t r[16];
      tc::tmem_ld16(tmem + lane_base + 32 * half + 16 * c, r);
      tc::tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 16; ++u) kq[16 * c + u] = __uint_as_float(r[u]);
    }
    tc::fence_before_sync();
  }
  __syncthreads();

  const int cbase = 32 * half;  // first column of this thread's half row
  uint32_t mma_phase = 1, v_phase = 0;
  for (int ih = 0; ok && ih < r_heads; ++ih) {
    const int hv = hv0 + ih;
    const int64_t jh = (int64_t)j * p.HV + hv;
    if (ih > 0) load_gates(p, jh, s_g, s_beta);
    if (row < C) {  // warps 0, 1, 4, 5: L = tril(diag(beta) K^K^^T, -1), row i, then M^{-1}
      const int i = row;
      const float bi = s_beta[i] * s_rk[i];
#pragma unroll
      for (int u = 0; u < 32; u += 4) {
        const float4 rk4 = *reinterpret_cast<const float4*>(s_rk + cbase + u);
        const int nu = cbase + u;
        float4 l4;
        l4.x = nu < i ? bi * rk4.x * kq[u] : 0.f;
        l4.y = nu + 1 < i ? bi * rk4.y * kq[u + 1] : 0.f;
        l4.z = nu + 2 < i ? bi * rk4.z * kq[u + 2] : 0.f;
        l4.w = nu + 3 < i ? bi * rk4.w * kq[u + 3] : 0.f;
        *reinterpret_cast<float4*>(Lf + i * LDF + nu) = l4;
      }
      tc::named_sync(2, 128);
      invert_unit_lower_64<LDF>(Lf, Xf, (warp & 1) | ((warp >> 2) << 1));
    } else {  // warps 2, 3, 6, 7 meanwhile: P = Gamma . tril(Q^K^^T), row r, straight to global
      const int r = row - C;
      const float qr = s_rq[r], gr = s_g[r];
      uint4* prow = reinterpret_cast<uint4*>(p.P + (jh * C + r) * C + cbase);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e0 = 8 * c + 2 * u, n0 = cbase + e0, n1 = n0 + 1;
          const float v0 = n0 <= r ? __expf(gr - s_g[n0]) * qr * s_rk[n0] * kq[e0] : 0.f;
          const float v1 = n1 <= r ? __expf(gr - s_g[n1]) * qr * s_rk[n1] * kq[e0 + 1] : 0.f;
          w[u] = pack_bf16(v0, v1);
        }
        prow[c] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    __syncthreads();  // L is dead from here on: its buffer takes the low bf16 parts of [A'; A]
    {  // A' rows (rows 0-63) and A rows (rows 64-127) as bf16 hi + lo, 128-byte swizzled K-major
      const int i = row & 63;
      const bool is_a = row >= 64;
      const float gi = s_g[i], egi = expf(gi);
      unsigned char* dst_hi = smem + SM::AA + (is_a ? 8192 : 0);
      unsigned char* dst_lo = smem + SM::LF + (is_a ? 8192 : 0);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int n0 = cbase + 8 * c;
        float x8[8], g8[8], b8[8], k8[8];  // X row i, and g, beta, 1/|k| of columns n0 .. n0+7
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          *reinterpret_cast<float4*>(x8 + 4 * q) = *reinterpret_cast<const float4*>(Xf + i * LDF + n0 + 4 * q);
          *reinterpret_cast<float4*>(g8 + 4 * q) = *reinterpret_cast<const float4*>(s_g + n0 + 4 * q);
          *reinterpret_cast<float4*>(b8 + 4 * q) = *reinterpret_cast<const float4*>(s_beta + n0 + 4 * q);
          *reinterpret_cast<float4*>(k8 + 4 * q) = *reinterpret_cast<const float4*>(s_rk + n0 + 4 * q);
        }
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float v2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int m = 2 * u + e, nu = n0 + m;
            const float x = nu == i ? 1.f : x8[m];  // entries above the diagonal are never read
            const float val = is_a ? __expf(gi - g8[m]) * x * b8[m] : egi * x * (b8[m] * k8[m]);
            v2[e] = nu <= i ? val : 0.f;
          }
          const __nv_bfloat162 hi = __floats2bfloat162_rn(v2[0], v2[1]);
          const float2 hf = __bfloat1622float2(hi);
          wh[u] = *reinterpret_cast<const uint32_t*>(&hi);
          wl[u] = pack_bf16(v2[0] - hf.x, v2[1] - hf.y);
        }
        *reinterpret_cast<uint4*>(dst_hi + tc::sw128_offset(i, 4 * half + c)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4*>(dst_lo + tc::sw128_offset(i, 4 * half + c)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
    }
    tc::fence_async_smem();
    __syncthreads();
    ok = wait_all(&bar[1], v_phase, p.status);
    v_phase ^= 1;
    if (!ok) break;
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idesc2 = tc::idesc_f16(128, D, 1, false, true);
      for (int part = 0; part < 2; ++part)  // [A'; A] = hi + lo
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t a = tc::smem_desc(tc::saddr(smem + (part ? SM::LF : SM::AA)) + ks * 32, 16, 1024, tc::kSwizzle128B);
          const uint64_t bk = tc::smem_desc(tc::saddr(smem + SM::KQ) + ks * 2048, 16384, 1024, tc::kSwizzle128B);
          tc::mma_f16_ss(tmem, a, bk, idesc2, (part | ks) != 0);
        }
      for (int part = 0; part < 2; ++part)
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t a = tc::smem_desc(tc::saddr(smem + (part ? SM::LF : SM::AA)) + ks * 32, 16, 1024, tc::kSwizzle128B);
          const uint64_t bv = tc::smem_desc(tc::saddr(smem + SM::V) + ks * 2048, 8192, 1024, tc::kSwizzle128B);
          tc::mma_f16_ss(tmem + tmem_u<D>(), a, bv, idesc2, (part | ks) != 0);
        }
      tc::mma_commit(&bar[2]);
    }
    ok = wait_all(&bar[2], mma_phase & 1, p.status);
    ++mma_phase;
    if (!ok) break;
    tc::fence_after_sync();
    if (tid == 0 && ih + 1 < r_heads) {  // the v tile is free: fetch the next value head's
      tc::mbar_arrive_expect_tx(&bar[1], NB * 8192);
      for (int b = 0; b < NB; ++b)
        tc::tma_load_3d(smem + SM::V + b * 8192, &tm_v, 64 * b, hv + 1, (int)t0, &bar[1]);
    }
    {  // rows 0-63 of DW are W<-, rows 64-127 of DU are U~: half an output row per thread
      const bool is_u = row >= 64;
      const int mu = row & 63;
      bf16* dst = (is_u ? p.U : p.W) + (jh * C + mu) * D + half * (D / 2);
      const uint32_t col0 = (is_u ? tmem_u<D>() : 0u) + half * (D / 2);
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
          for (int u = 0; u < 8; ++u) w[u] = pack_bf16(__uint_as_float(r[c][2 * u]), __uint_as_float(r[c][2 * u + 1]));
          uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * (g0 + c));
          d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols<D>());
  }
}

template <int D>
cudaError_t launch_intra_t(const Params& p, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  if (!make_token_tile_map(&mq, p.q, D, p.H, p.T, C) || !make_token_tile_map(&mk, p.k, D, p.H, p.T, C) ||
      !make_token_tile_map(&mv, p.v, D, p.HV, p.T, C))
    return cudaErrorInvalidValue;
  const uint32_t smem = IntraSmem<D>::alloc;
  cudaError_t e = cudaFuncSetAttribute(intra_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = p.max_chunks * p.H;
  intra_kernel<D><<<(unsigned)blocks, kThreads, smem, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra(const Params& p, int D, int Cc, cudaStream_t s) {
  if (Cc != C) return cudaErrorInvalidValue;
  switch (D) {
    case 64: return launch_intra_t<64>(p, s);
    case 128: return launch_intra_t<128>(p, s);
    case 256: return launch_intra_t<256>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
