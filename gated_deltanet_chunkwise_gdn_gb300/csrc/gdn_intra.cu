// gdn_intra.cu — K2: per-chunk gates, Gram products, the one triangular inverse and
// the WY factors, for every chunk of every sequence in parallel.
//
// One CTA handles one (chunk, q/k head h) and loops over the HV/H value heads that
// read head h, so K^K^^T and Q^K^^T are formed once per q/k head.
//
// Per value head it computes (see gdn_common.cuh for the notation):
//   log alpha = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b)   (pymllm page,
//               Parameters: raw gate inputs before softplus/exp and sigmoid)
//   g        = chunk-local inclusive cumsum of log alpha
//   M^{-1}   for M = I + tril(diag(beta) K^K^^T, -1)   (blocked forward substitution)
//   A        = (Gamma . M^{-1}) diag(beta)             (N^{-1} B = G M^{-1} G^{-1} B,
//                                                      "Simple math to speed up GDN
//                                                      prefill", section "Save one invert")
//   W<-      = A diag(exp(g)) K^,   U~ = A V,   P = Gamma . tril(Q^K^^T)
// and stores g, 1/|q|, 1/|k|, W<-, U~ and P for the scan kernel.
//
// Normalisation and decay enter only as diagonal scalings of the fp32 Gram
// accumulators or of the small C x C operand, so the raw bf16 q/k/v tiles feed the
// tensor cores unchanged.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int C = 64;
constexpr int kThreads = 128;

template <int D>
struct IntraSmem {
  static constexpr int LDT = D + 8;  // bf16 pitch of the q/k/v tiles
  static constexpr int LDA = C + 8;  // bf16 pitch of A, A'
  static constexpr int LDF = C + 1;  // fp32 pitch of L, X
  static constexpr size_t tiles = 3ull * C * LDT * sizeof(bf16);
  static constexpr size_t lx = 2ull * C * LDF * sizeof(float);
  static constexpr size_t aa = 2ull * C * LDA * sizeof(bf16);
  static constexpr size_t vec = 4ull * C * sizeof(float);
  static constexpr size_t bytes = tiles + lx + aa + vec;
};

__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

// Loads `rows` valid rows of a C x D bf16 tile (global row stride `gstride` elements)
// into smem with pitch LDT; rows >= rows are zero-filled.
template <int D, int LDT>
__device__ __forceinline__ void load_tile(bf16* s, const bf16* g, int64_t gstride, int rows) {
  constexpr int SEG = D / 8;  // 16-byte segments per row
  for (int e = threadIdx.x; e < C * SEG; e += kThreads) {
    const int r = e / SEG, c = (e % SEG) * 8;
    if (r < rows)
      cp_async_16(s + r * LDT + c, g + r * gstride + c);
    else
      *reinterpret_cast<uint4*>(s + r * LDT + c) = make_uint4(0, 0, 0, 0);
  }
}

// Inverts the unit lower-triangular 64x64 matrix I + L (L strictly lower, in Lf)
// into Xf, by 16x16 blocks: the four diagonal blocks by forward substitution (one
// warp each, one lane per column), then block rows I = 1..3 with
//   X_IJ = -X_II * sum_{K=J}^{I-1} L_IK X_KJ.
template <int LDF>
__device__ void invert_unit_lower_64(const float* Lf, float* Xf) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  __syncthreads();
  for (int I = 1; I < 4; ++I) {
    // T_IJ = sum_{K=J}^{I-1} L_IK X_KJ, written into the X_IJ slots.
    float t[6];
    const int n_ent = I * 256;
#pragma unroll
    for (int u = 0; u < 6; ++u) {
      const int e = threadIdx.x + u * kThreads;
      t[u] = 0.f;
      if (e < n_ent) {
        const int J = e >> 8, a = (e >> 4) & 15, bcol = e & 15;
        const float* lrow = Lf + (16 * I + a) * LDF;
        float acc = 0.f;
        for (int kk = 16 * J; kk < 16 * I; ++kk) acc += lrow[kk] * Xf[kk * LDF + 16 * J + bcol];
        t[u] = acc;
      }
    }
#pragma unroll
    for (int u = 0; u < 6; ++u) {
      const int e = threadIdx.x + u * kThreads;
      if (e < n_ent) {
        const int J = e >> 8, a = (e >> 4) & 15, bcol = e & 15;
        Xf[(16 * I + a) * LDF + 16 * J + bcol] = t[u];
      }
    }
    __syncthreads();
    // X_IJ = -X_II T_IJ
#pragma unroll
    for (int u = 0; u < 6; ++u) {
      const int e = threadIdx.x + u * kThreads;
      if (e < n_ent) {
        const int J = e >> 8, a = (e >> 4) & 15, bcol = e & 15;
        const float* drow = Xf + (16 * I + a) * LDF + 16 * I;
        float acc = 0.f;
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) acc += drow[cc] * Xf[(16 * I + cc) * LDF + 16 * J + bcol];
        t[u] = -acc;
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 6; ++u) {
      const int e = threadIdx.x + u * kThreads;
      if (e < n_ent) {
        const int J = e >> 8, a = (e >> 4) & 15, bcol = e & 15;
        Xf[(16 * I + a) * LDF + 16 * J + bcol] = t[u];
      }
    }
    __syncthreads();
  }
}

// Rows [16*warp, 16*warp+16) of Out(64 x D) = As(64 x 64) * Bs(64 x D), As row-major
// (pitch LDA), Bs row-major [k][n] (pitch LDT); fp32 accumulators in acc.
template <int D, int LDA, int LDT>
__device__ __forceinline__ void mma_rows_AxB(const bf16* As, const bf16* Bs, float (&acc)[D / 8][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[nt][r] = 0.f;
#pragma unroll
  for (int kk = 0; kk < C / 16; ++kk) {
    uint32_t a[4];
    ldmatrix_x4(a, As + (16 * warp + (lane & 15)) * LDA + 16 * kk + (lane >> 4) * 8);
#pragma unroll
    for (int nt = 0; nt < D / 8; nt += 2) {
      uint32_t b[4];
      const int m = lane >> 3, r = lane & 7;
      ldmatrix_x4_trans(b, Bs + (16 * kk + (m & 1) * 8 + r) * LDT + 8 * (nt + (m >> 1)));
      mma_bf16_16816(acc[nt], a, b[0], b[1]);
      mma_bf16_16816(acc[nt + 1], a, b[2], b[3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) intra_kernel(Params p) {
  using SM = IntraSmem<D>;
  constexpr int LDT = SM::LDT, LDA = SM::LDA, LDF = SM::LDF;
  extern __shared__ __align__(16) unsigned char smem[];
  bf16* Ks = reinterpret_cast<bf16*>(smem);
  bf16* Qs = Ks + C * LDT;
  bf16* Vs = Qs + C * LDT;
  float* Lf = reinterpret_cast<float*>(Vs + C * LDT);
  float* Xf = Lf + C * LDF;
  bf16* As = reinterpret_cast<bf16*>(Xf + C * LDF);
  bf16* Aw = As + C * LDA;
  float* s_g = reinterpret_cast<float*>(Aw + C * LDA);
  float* s_beta = s_g + C;
  float* s_rq = s_beta + C;
  float* s_rk = s_rq + C;

  if (p.status[0] != GDN_OK) return;
  const int j = blockIdx.x / p.H, h = blockIdx.x % p.H;
  if (j >= p.status[1]) return;
  const int4 ct = p.chunk_tab[j];
  const int64_t t0 = ct.y;
  const int len = ct.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int r_heads = p.HV / p.H;

  // q/k tiles (group 0), then v of the first value head (group 1)
  load_tile<D, LDT>(Ks, p.k + (t0 * p.H + h) * D, (int64_t)p.H * D, len);
  load_tile<D, LDT>(Qs, p.q + (t0 * p.H + h) * D, (int64_t)p.H * D, len);
  cp_async_commit();
  load_tile<D, LDT>(Vs, p.v + (t0 * p.HV + h * r_heads) * D, (int64_t)p.HV * D, len);
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();

  // inverse row norms (two threads per row)
  {
    const int row = tid >> 1, half = tid & 1;
    float sk = 0.f, sq = 0.f;
#pragma unroll 8
    for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 2) {
      const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Ks + row * LDT + c));
      const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Qs + row * LDT + c));
      sk += kf.x * kf.x + kf.y * kf.y;
      sq += qf.x * qf.x + qf.y * qf.y;
    }
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    if (half == 0) {
      const float rk = row < len ? rsqrtf(sk + kNormEps) : 0.f;
      const float rq = row < len ? rsqrtf(sq + kNormEps) : 0.f;
      s_rk[row] = rk;
      s_rq[row] = rq;
      p.rk[((int64_t)j * p.H + h) * C + row] = rk;
      p.rq[((int64_t)j * p.H + h) * C + row] = rq;
    }
  }

  // Gram products, rows [16*warp, +16): accK = K K^T, accQ = Q K^T (raw bf16 inputs)
  float accK[C / 8][4], accQ[C / 8][4];
#pragma unroll
  for (int nt = 0; nt < C / 8; ++nt)
#pragma unroll
    for (int r = 0; r < 4; ++r) accK[nt][r] = accQ[nt][r] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    uint32_t ak[4], aq[4];
    ldmatrix_x4(ak, Ks + (16 * warp + (lane & 15)) * LDT + 16 * kk + (lane >> 4) * 8);
    ldmatrix_x4(aq, Qs + (16 * warp + (lane & 15)) * LDT + 16 * kk + (lane >> 4) * 8);
#pragma unroll
    for (int nt = 0; nt < C / 8; nt += 2) {
      uint32_t b[4];
      const int m = lane >> 3, r = lane & 7;
      ldmatrix_x4(b, Ks + (8 * (nt + (m >> 1)) + r) * LDT + 16 * kk + (m & 1) * 8);
      mma_bf16_16816(accK[nt], ak, b[0], b[1]);
      mma_bf16_16816(accK[nt + 1], ak, b[2], b[3]);
      mma_bf16_16816(accQ[nt], aq, b[0], b[1]);
      mma_bf16_16816(accQ[nt + 1], aq, b[2], b[3]);
    }
  }

  for (int ih = 0; ih < r_heads; ++ih) {
    const int hv = h * r_heads + ih;
    const int64_t jh = (int64_t)j * p.HV + hv;
    // gates and the chunk-local cumulative log decay (warps 0-1, one token per thread)
    if (tid < C) {
      float la = 0.f, beta = 0.f;
      if (tid < len) {
        const int64_t t = t0 + tid;
        la = -expf(p.A_log[hv]) * softplus_f(p.a[t * p.HV + hv] + p.dt_bias[hv]);
        beta = 1.f / (1.f + expf(-p.b[t * p.HV + hv]));
      }
      float incl = la;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      s_g[tid] = incl;  // warp-local; warp 1 adds warp 0's total below
      s_beta[tid] = beta;
    }
    __syncthreads();
    if (tid >= 32 && tid < C) s_g[tid] += s_g[31];
    __syncthreads();
    if (tid < C) p.g[jh * C + tid] = s_g[tid];

    // L = tril(diag(beta) K^K^^T, -1) into Lf; P = Gamma . tril(Q^K^^T) to global
    bf16* Pg = p.P + jh * C * C;
#pragma unroll
    for (int nt = 0; nt < C / 8; ++nt) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = 16 * warp + g4 + 8 * hr;
        const int nu = 8 * nt + 2 * t4;
        const float bi = s_beta[i] * s_rk[i];
        const float l0 = nu < i ? bi * s_rk[nu] * accK[nt][2 * hr] : 0.f;
        const float l1 = nu + 1 < i ? bi * s_rk[nu + 1] * accK[nt][2 * hr + 1] : 0.f;
        Lf[i * LDF + nu] = l0;
        Lf[i * LDF + nu + 1] = l1;
        const float qi = s_rq[i], gi = s_g[i];
        const float p0 = nu <= i ? expf(gi - s_g[nu]) * qi * s_rk[nu] * accQ[nt][2 * hr] : 0.f;
        const float p1 = nu + 1 <= i ? expf(gi - s_g[nu + 1]) * qi * s_rk[nu + 1] * accQ[nt][2 * hr + 1] : 0.f;
        *reinterpret_cast<uint32_t*>(Pg + i * C + nu) = pack_bf16(p0, p1);
      }
    }
    __syncthreads();
    invert_unit_lower_64<LDF>(Lf, Xf);

    // A = (Gamma . X) diag(beta) and A' = A diag(exp(g) / |k|) (the W<- operand)
    {
      const int i = tid >> 1, c0 = (tid & 1) * 32;
      const float gi = s_g[i], egi = expf(gi);
#pragma unroll 4
      for (int c = c0; c < c0 + 32; c += 2) {
        float a0 = 0.f, a1 = 0.f, w0 = 0.f, w1 = 0.f;
        if (c <= i) {
          const float x = (c == i) ? 1.f : Xf[i * LDF + c];
          a0 = expf(gi - s_g[c]) * x * s_beta[c];
          w0 = egi * x * s_beta[c] * s_rk[c];
        }
        if (c + 1 <= i) {
          const float x = (c + 1 == i) ? 1.f : Xf[i * LDF + c + 1];
          a1 = expf(gi - s_g[c + 1]) * x * s_beta[c + 1];
          w1 = egi * x * s_beta[c + 1] * s_rk[c + 1];
        }
        *reinterpret_cast<uint32_t*>(As + i * LDA + c) = pack_bf16(a0, a1);
        *reinterpret_cast<uint32_t*>(Aw + i * LDA + c) = pack_bf16(w0, w1);
      }
    }
    cp_async_wait<0>();
    __syncthreads();

    // W<- = A' K and U~ = A V, rows [16*warp, +16)
    {
      float acc[D / 8][4];
      mma_rows_AxB<D, LDA, LDT>(Aw, Ks, acc);
      bf16* Wg = p.W + jh * C * D;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int i = 16 * warp + g4 + 8 * hr;
          *reinterpret_cast<uint32_t*>(Wg + i * D + 8 * nt + 2 * t4) = pack_bf16(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
        }
      mma_rows_AxB<D, LDA, LDT>(As, Vs, acc);
      bf16* Ug = p.U + jh * C * D;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int i = 16 * warp + g4 + 8 * hr;
          *reinterpret_cast<uint32_t*>(Ug + i * D + 8 * nt + 2 * t4) = pack_bf16(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
        }
    }
    __syncthreads();
    if (ih + 1 < r_heads) {
      load_tile<D, LDT>(Vs, p.v + (t0 * p.HV + hv + 1) * D, (int64_t)p.HV * D, len);
      cp_async_commit();
    }
  }
}

template <int D>
cudaError_t launch_intra_t(const Params& p, cudaStream_t s) {
  const size_t smem = IntraSmem<D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(intra_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = p.max_chunks * p.H;
  intra_kernel<D><<<(unsigned)blocks, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra(const Params& p, int D, int Cc, cudaStream_t s) {
  if (Cc != C) return cudaErrorInvalidValue;
  switch (D) {
    case 64: return launch_intra_t<64>(p, s);
    case 128: return launch_intra_t<128>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
