// gdn_scan.cu — K3: the sequential inter-chunk scan with the output epilogue.
//
// One CTA owns one (sequence, value head, block of VB state rows) chain. Rows of the
// state S (V x K) evolve independently — the update contracts over the key dimension
// only — so the value dimension is split across CTAs while the key dimension stays
// whole ("nrm-training-kernels", section "Kernel": the grid splits batch, heads and
// blocks of the value dimension, never the key dimension).
//
// For each chunk of the sequence, in order (pymllm page "pymllm.layers.attention.
// gdn_chunkwise": the inter-chunk propagation stays sequential, ceil(T/C) steps), with
// the state slice S (VB x K, fp32) held in registers for the whole chain:
//   U  = U~ - W<- S^T                               (the chunk's new values)
//   O  = diag(exp(g)/|q|) Q S^T + P U               (inter + masked intra part)
//   S <- exp(g_C) S + (diag(exp(g_C - g)/|k|) U)^T K
// which is "Simple math to speed up GDN prefill", section "Reminder": the chunk
// transition S_[t+1] = S-> + (U~ - W<- S^T)^T K-> with S-> = gamma_C S and
// K-> = diag(gamma_C / gamma) K^.
//
// The state is read from state_pool once at the start and written once at the end.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int C = 64;
constexpr int kThreads = 128;

template <int D, int VB>
struct ScanSmem {
  static constexpr int LDT = D + 8;   // bf16 pitch of W<-, q, k tiles and the bf16 state copy
  static constexpr int LDP = C + 8;   // bf16 pitch of P
  static constexpr int LDU = VB + 8;  // bf16 pitch of U~, U tiles
  static constexpr size_t stage_bf16 = 3ull * C * LDT + 1ull * C * LDP + 1ull * C * LDU;
  static constexpr size_t stage_bytes = stage_bf16 * sizeof(bf16) + 3ull * C * sizeof(float);
  static constexpr size_t extra_bytes = (1ull * VB * LDT + 2ull * C * LDU) * sizeof(bf16);
  static constexpr size_t bytes = 2 * stage_bytes + extra_bytes;
};

template <int W, int LD>
__device__ __forceinline__ void load_rows(bf16* s, const bf16* g, int64_t gstride, int rows) {
  constexpr int SEG = W / 8;
  for (int e = threadIdx.x; e < C * SEG; e += kThreads) {
    const int r = e / SEG, c = (e % SEG) * 8;
    if (r < rows)
      cp_async_16(s + r * LD + c, g + r * gstride + c);
    else
      *reinterpret_cast<uint4*>(s + r * LD + c) = make_uint4(0, 0, 0, 0);
  }
}

template <int D, int VB>
__global__ void __launch_bounds__(kThreads) scan_kernel(Params p) {
  using SM = ScanSmem<D, VB>;
  constexpr int LDT = SM::LDT, LDP = SM::LDP, LDU = SM::LDU;
  constexpr int NVB = D / VB;
  constexpr int MT = VB / 16;      // m-tiles of the state slice
  constexpr int NTS = D / 32;      // n-tiles of the state slice per warp
  constexpr int NTX = VB / 8;      // n-tiles of U / O
  extern __shared__ __align__(16) unsigned char smem[];

  if (p.status[0] != GDN_OK) return;
  int bid = blockIdx.x;
  const int vblk = bid % NVB;
  bid /= NVB;
  const int hv = bid % p.HV;
  const int seq = p.order[bid / p.HV];
  const int h = hv / (p.HV / p.H);
  const int c_beg = p.seq_chunk_off[seq];
  const int n_c = p.seq_chunk_off[seq + 1] - c_beg;
  if (n_c == 0) return;  // empty sequence: the slot is left as it is
  const int64_t slot = p.cache_indices[seq];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int lm = lane >> 3, lr = lane & 7;

  auto stage_ptr = [&](int st) { return smem + st * SM::stage_bytes; };
  auto Ws = [&](int st) { return reinterpret_cast<bf16*>(stage_ptr(st)); };
  auto Qs = [&](int st) { return Ws(st) + C * LDT; };
  auto Ks = [&](int st) { return Ws(st) + 2 * C * LDT; };
  auto Ps = [&](int st) { return Ws(st) + 3 * C * LDT; };
  auto Us = [&](int st) { return Ps(st) + C * LDP; };
  auto Fs = [&](int st) { return reinterpret_cast<float*>(stage_ptr(st) + SM::stage_bf16 * sizeof(bf16)); };
  bf16* Sbf = reinterpret_cast<bf16*>(smem + 2 * SM::stage_bytes);
  bf16* Vn = Sbf + VB * LDT;
  bf16* Vk = Vn + C * LDU;

  int st_t0[2], st_len[2];
  auto issue = [&](int c, int st) {
    const int j = c_beg + c;
    const int4 ct = p.chunk_tab[j];
    st_t0[st] = ct.y;
    st_len[st] = ct.z;
    const int64_t jh = (int64_t)j * p.HV + hv;
    const int64_t t0 = ct.y;
    load_rows<D, LDT>(Ws(st), p.W + jh * C * D, D, C);
    load_rows<D, LDT>(Qs(st), p.q + (t0 * p.H + h) * D, (int64_t)p.H * D, ct.z);
    load_rows<D, LDT>(Ks(st), p.k + (t0 * p.H + h) * D, (int64_t)p.H * D, ct.z);
    load_rows<C, LDP>(Ps(st), p.P + jh * C * C, C, C);
    load_rows<VB, LDU>(Us(st), p.U + jh * C * D + vblk * VB, D, C);
    float* F = Fs(st);
    const int64_t jq = (int64_t)j * p.H + h;
    if (tid < 16) cp_async_16(F + tid * 4, p.g + jh * C + tid * 4);
    else if (tid < 32) cp_async_16(F + C + (tid - 16) * 4, p.rq + jq * C + (tid - 16) * 4);
    else if (tid < 48) cp_async_16(F + 2 * C + (tid - 32) * 4, p.rk + jq * C + (tid - 32) * 4);
    cp_async_commit();
  };

  // state slice: warp w owns key columns [w*D/4, (w+1)*D/4)
  float S[MT][NTS][4];
  float* Sg = p.state_pool + ((slot * p.HV + hv) * (int64_t)D + vblk * VB) * D;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NTS; ++nt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = 16 * mt + g4 + 8 * hr, col = warp * (D / 4) + 8 * nt + 2 * t4;
        const float2 s2 = *reinterpret_cast<const float2*>(Sg + (int64_t)row * D + col);
        S[mt][nt][2 * hr] = s2.x;
        S[mt][nt][2 * hr + 1] = s2.y;
        *reinterpret_cast<uint32_t*>(Sbf + row * LDT + col) = pack_bf16(s2.x, s2.y);
      }

  issue(0, 0);
  for (int c = 0; c < n_c; ++c) {
    const int st = c & 1;
    if (c + 1 < n_c) {
      issue(c + 1, st ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float* F = Fs(st);
    const float* gs = F;
    const float* rqs = F + C;
    const float* rks = F + 2 * C;
    const float gC = gs[C - 1];

    // Step 1: X = [W<- ; Q] S^T, rows [32*warp, +32) of the 128-row stack
    float X[2][NTX][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NTX; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) X[mt][nt][r] = 0.f;
    const bf16* Abase = warp < 2 ? Ws(st) + 32 * warp * LDT : Qs(st) + 32 * (warp - 2) * LDT;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a0[4], a1[4];
      ldmatrix_x4(a0, Abase + (lane & 15) * LDT + 16 * kk + (lane >> 4) * 8);
      ldmatrix_x4(a1, Abase + (16 + (lane & 15)) * LDT + 16 * kk + (lane >> 4) * 8);
#pragma unroll
      for (int nt = 0; nt < NTX; nt += 2) {
        uint32_t b[4];
        ldmatrix_x4(b, Sbf + (8 * (nt + (lm >> 1)) + lr) * LDT + 16 * kk + (lm & 1) * 8);
        mma_bf16_16816(X[0][nt], a0, b[0], b[1]);
        mma_bf16_16816(X[0][nt + 1], a0, b[2], b[3]);
        mma_bf16_16816(X[1][nt], a1, b[0], b[1]);
        mma_bf16_16816(X[1][nt + 1], a1, b[2], b[3]);
      }
    }

    // Step 2: U = U~ - W<- S^T (warps 0-1); row-scaled inter output (warps 2-3)
    if (warp < 2) {
      const bf16* Ut = Us(st);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int mu = 32 * warp + 16 * mt + g4 + 8 * hr;
          const float sk = expf(gC - gs[mu]) * rks[mu];
#pragma unroll
          for (int nt = 0; nt < NTX; ++nt) {
            const int col = 8 * nt + 2 * t4;
            const float2 u2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Ut + mu * LDU + col));
            const float n0 = u2.x - X[mt][nt][2 * hr], n1 = u2.y - X[mt][nt][2 * hr + 1];
            *reinterpret_cast<uint32_t*>(Vn + mu * LDU + col) = pack_bf16(n0, n1);
            *reinterpret_cast<uint32_t*>(Vk + mu * LDU + col) = pack_bf16(n0 * sk, n1 * sk);
          }
        }
    } else {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = 32 * (warp - 2) + 16 * mt + g4 + 8 * hr;
          const float sq = expf(gs[r]) * rqs[r];
#pragma unroll
          for (int nt = 0; nt < NTX; ++nt) {
            X[mt][nt][2 * hr] *= sq;
            X[mt][nt][2 * hr + 1] *= sq;
          }
        }
    }
    __syncthreads();

    // Step 3a: O = inter + P U, stored (warps 2-3)
    if (warp >= 2) {
      const bf16* Pb = Ps(st) + 32 * (warp - 2) * LDP;
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk) {
        uint32_t a0[4], a1[4];
        ldmatrix_x4(a0, Pb + (lane & 15) * LDP + 16 * kk + (lane >> 4) * 8);
        ldmatrix_x4(a1, Pb + (16 + (lane & 15)) * LDP + 16 * kk + (lane >> 4) * 8);
#pragma unroll
        for (int nt = 0; nt < NTX; nt += 2) {
          uint32_t b[4];
          ldmatrix_x4_trans(b, Vn + (16 * kk + (lm & 1) * 8 + lr) * LDU + 8 * (nt + (lm >> 1)));
          mma_bf16_16816(X[0][nt], a0, b[0], b[1]);
          mma_bf16_16816(X[0][nt + 1], a0, b[2], b[3]);
          mma_bf16_16816(X[1][nt], a1, b[0], b[1]);
          mma_bf16_16816(X[1][nt + 1], a1, b[2], b[3]);
        }
      }
      const int64_t t0 = st_t0[st];
      const int len = st_len[st];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = 32 * (warp - 2) + 16 * mt + g4 + 8 * hr;
          if (r < len) {
            bf16* orow = p.out + ((t0 + r) * p.HV + hv) * (int64_t)D + vblk * VB;
#pragma unroll
            for (int nt = 0; nt < NTX; ++nt)
              *reinterpret_cast<uint32_t*>(orow + 8 * nt + 2 * t4) =
                  pack_bf16(p.scale * X[mt][nt][2 * hr], p.scale * X[mt][nt][2 * hr + 1]);
          }
        }
    }

    // Step 3b: S <- exp(g_C) S + Vk^T K (all warps, key columns of this warp)
    {
      const float eC = expf(gC);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NTS; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) S[mt][nt][r] *= eC;
      const bf16* Kt = Ks(st);
      const int cb = warp * (D / 4);
#pragma unroll
      for (int kk = 0; kk < C / 16; ++kk) {
        uint32_t a[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          ldmatrix_x4_trans(a[mt], Vk + (16 * kk + (lm >> 1) * 8 + lr) * LDU + 16 * mt + (lm & 1) * 8);
#pragma unroll
        for (int nt = 0; nt < NTS; nt += 2) {
          uint32_t b[4];
          ldmatrix_x4_trans(b, Kt + (16 * kk + (lm & 1) * 8 + lr) * LDT + cb + 8 * (nt + (lm >> 1)));
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            mma_bf16_16816(S[mt][nt], a[mt], b[0], b[1]);
            mma_bf16_16816(S[mt][nt + 1], a[mt], b[2], b[3]);
          }
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NTS; ++nt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int row = 16 * mt + g4 + 8 * hr, col = cb + 8 * nt + 2 * t4;
            *reinterpret_cast<uint32_t*>(Sbf + row * LDT + col) = pack_bf16(S[mt][nt][2 * hr], S[mt][nt][2 * hr + 1]);
          }
    }
    __syncthreads();
  }

#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NTS; ++nt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = 16 * mt + g4 + 8 * hr, col = warp * (D / 4) + 8 * nt + 2 * t4;
        *reinterpret_cast<float2*>(Sg + (int64_t)row * D + col) = make_float2(S[mt][nt][2 * hr], S[mt][nt][2 * hr + 1]);
      }
}

template <int D, int VB>
cudaError_t launch_scan_t(const Params& p, cudaStream_t s) {
  const size_t smem = ScanSmem<D, VB>::bytes;
  cudaError_t e = cudaFuncSetAttribute(scan_kernel<D, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.B * p.HV * (D / VB);
  scan_kernel<D, VB><<<(unsigned)blocks, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan(const Params& p, int D, int Cc, cudaStream_t s) {
  if (Cc != C) return cudaErrorInvalidValue;
  const int vb = D / p.nvb;
  if (D == 64 && vb == 16) return launch_scan_t<64, 16>(p, s);
  if (D == 64 && vb == 32) return launch_scan_t<64, 32>(p, s);
  if (D == 128 && vb == 16) return launch_scan_t<128, 16>(p, s);
  if (D == 128 && vb == 32) return launch_scan_t<128, 32>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
