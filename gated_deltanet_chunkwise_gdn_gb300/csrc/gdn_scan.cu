// gdn_scan.cu — K3: the sequential inter-chunk scan with the output epilogue, on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM) with TMA-fed chunk tiles.
//
// One CTA owns one (sequence, value head, block of VB = 64 state rows) chain. Rows of the
// state S (V x K) evolve independently — the update contracts over the key dimension only
// — so the value dimension is split across CTAs while the key dimension stays whole
// ("nrm-training-kernels", section "Kernel": the grid splits batch, heads and blocks of
// the value dimension, never the key dimension).
//
// For each chunk of the sequence, in order (pymllm page "pymllm.layers.attention.
// gdn_chunkwise": the inter-chunk propagation stays sequential, ceil(T/C) steps):
//   U  = U~ - W<- S^T                               (the chunk's new values)
//   O  = diag(exp(g)/|q|) Q S^T + P U               (inter + masked intra part)
//   S <- exp(g_C) S + (diag(exp(g_C - g)/|k|) U)^T K
// i.e. "Simple math to speed up GDN prefill", section "Reminder": the chunk transition
// S_[t+1] = S-> + (U~ - W<- S^T)^T K-> with S-> = gamma_C S and K-> = diag(gamma_C/gamma) K^.
//
// Per chunk, three MMAs (M = 128, issued by one thread, fp32 accumulators in TMEM):
//   MMA1  D1[128 x VB]  = [W<-; Q] S^T     rows 0-63: W<- S^T (-> U), rows 64-127: Q S^T
//   MMA3  DS[K x VB]    = K^T Uk           the state increment, Uk = diag(exp(g_C-g)/|k|) U
//   MMA2  D2[128 x VB]  = [*; P] U         rows 64-127: P U (rows 0-63 unused)
// The fp32 state slice lives in registers as S^T (thread d holds key row d), its bf16
// copy is the B operand of MMA1. U and Uk go through shared memory as the B operands of
// MMA2/MMA3. A producer warp streams W<-, Q, K, P and the gate vectors of the next chunks
// with TMA into a 3-stage ring (full/empty mbarriers, all waits bounded).
//
// The state is read from state_pool once at the start and written once at the end.
#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace {

constexpr int C = 64;
constexpr int VB = 64;
constexpr int kStages = 3;
constexpr int kConsumers = 128;  // 4 warps: thread i <-> TMEM lane i
constexpr int kThreads = kConsumers + 32;
constexpr long long kWaitBudget = 1ll << 31;  // clock cycles before a wait gives up (~1 s)
constexpr uint32_t kTmemCols = 256;           // D1 [0,64), DS [64,128), D2 [128,192)

template <int D>
struct ScanSmem {
  static constexpr int NB = D / 64;
  // one stage (offsets from the stage base; every tile 128-byte swizzled, 1 KB aligned)
  static constexpr uint32_t WQ = 0;                 // NB x [W<- block 8 KB][Q block 8 KB]
  static constexpr uint32_t K = WQ + NB * 16384;    // NB x K block 8 KB
  static constexpr uint32_t P = K + NB * 8192;      // P 8 KB (the 8 KB before it: A rows 0-63 of MMA2)
  static constexpr uint32_t F = P + 8192;           // g, 1/|q|, 1/|k| (3 x 256 B)
  static constexpr uint32_t STAGE = F + 1024;
  static constexpr uint32_t SCOPY = kStages * STAGE;  // bf16 S^T: D rows x 128 B
  static constexpr uint32_t VN = SCOPY + D * 128;     // U  [64 rows x 128 B]
  static constexpr uint32_t VK = VN + 8192;           // Uk [64 rows x 128 B]
  static constexpr uint32_t BAR = VK + 8192;          // full[3], empty[3], mma, TMEM address, flag
  static constexpr uint32_t bytes = BAR + 128;
  static constexpr uint32_t alloc = bytes + 1024;
  static constexpr uint32_t stage_tx = NB * 16384 + NB * 8192 + 8192 + 3 * 256;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    scan_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_p,
                const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, Params p) {
  using SM = ScanSmem<D>;
  constexpr int NB = SM::NB;
  constexpr int NVB = D / VB;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

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
  const int tid = threadIdx.x, warp = tid >> 5;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::BAR);
  uint64_t* empty = full + kStages;
  uint64_t* mma_bar = empty + kStages;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(mma_bar + 1);
  volatile int* s_fail = reinterpret_cast<volatile int*>(tslot + 1);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(mma_bar, 1);
    *s_fail = 0;
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------------ producer warp
    if ((tid & 31) == 0) {
      for (int c = 0; c < n_c; ++c) {
        const int s = c % kStages, use = c / kStages;
        if (use > 0 && !tc::mbar_wait(&empty[s], (use - 1) & 1, kWaitBudget)) {
          set_status(p.status, GDN_ERR_TIMEOUT);
          *s_fail = 1;
          break;
        }
        const int j = c_beg + c;
        const int4 ct = p.chunk_tab[j];
        const int t0 = ct.y;
        const int64_t jh = (int64_t)j * p.HV + hv;
        const int64_t jq = (int64_t)j * p.H + h;
        unsigned char* st = smem + s * SM::STAGE;
        reinterpret_cast<int*>(st + SM::F + 768)[0] = ct.y;  // first token and length of the chunk,
        reinterpret_cast<int*>(st + SM::F + 768)[1] = ct.z;  // published by the barrier's release
        tc::mbar_arrive_expect_tx(&full[s], SM::stage_tx);
        for (int b = 0; b < NB; ++b) {
          tc::tma_load_2d(st + SM::WQ + b * 16384, &tm_w, 64 * b, (int)(jh * C), &full[s]);
          tc::tma_load_3d(st + SM::WQ + b * 16384 + 8192, &tm_q, 64 * b, h, t0, &full[s]);
          tc::tma_load_3d(st + SM::K + b * 8192, &tm_k, 64 * b, h, t0, &full[s]);
        }
        tc::tma_load_2d(st + SM::P, &tm_p, 0, (int)(jh * C), &full[s]);
        tc::bulk_load(st + SM::F, p.g + jh * C, 256, &full[s]);
        tc::bulk_load(st + SM::F + 256, p.rq + jq * C, 256, &full[s]);
        tc::bulk_load(st + SM::F + 512, p.rk + jq * C, 256, &full[s]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ consumer warps
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const bool has_state = tid < D;      // thread d holds key row d of S^T
    const bool u_row = tid < C;          // thread mu forms row mu of U
    const bool o_row = tid >= 64;        // thread 64 + r forms output row r
    float S[VB];
    float* Sg = p.state_pool + ((slot * p.HV + hv) * (int64_t)D + vblk * VB) * D;  // S[v][d] = Sg[v*D + d]
    if (has_state) {
#pragma unroll
      for (int v = 0; v < VB; ++v) S[v] = Sg[(int64_t)v * D + tid];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) w[u] = pack_bf16(S[8 * c + 2 * u], S[8 * c + 2 * u + 1]);
        *reinterpret_cast<uint4*>(smem + SM::SCOPY + tc::sw128_offset(tid, c)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    // U~ row of the first chunk (rows of later chunks are prefetched one chunk ahead)
    uint4 ut[8];
    if (u_row) {
      const uint4* src = reinterpret_cast<const uint4*>(p.U + ((int64_t)c_beg * p.HV + hv) * C * D + (int64_t)tid * D + vblk * VB);
#pragma unroll
      for (int c = 0; c < 8; ++c) ut[c] = src[c];
    }
    tc::fence_async_smem();
    tc::named_sync(1, kConsumers);

    constexpr uint32_t idesc_x = tc::idesc_f16(128, VB, 1, false, true);  // A K-major, B MN-major
    constexpr uint32_t idesc_s = tc::idesc_f16(128, VB, 1, true, true);   // both MN-major
    uint32_t mma_phase = 0;
    bool failed = false;
    for (int c = 0; c < n_c; ++c) {
      const int s = c % kStages;
      unsigned char* st = smem + s * SM::STAGE;
      bool bad = !tc::mbar_wait(&full[s], (c / kStages) & 1, kWaitBudget) || *s_fail != 0;
      if (tc::named_sync_or(1, kConsumers, bad)) {  // the same verdict in every consumer thread
        if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT);
        failed = true;
        break;
      }
      // MMA1: D1 = [W<-; Q] S^T
      if (tid == 0) {
        tc::fence_after_sync();
        for (int b = 0; b < NB; ++b)
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t a = tc::smem_desc(tc::saddr(st + SM::WQ + b * 16384) + ks * 32, 16, 1024, tc::kSwizzle128B);
            const uint64_t bd = tc::smem_desc(tc::saddr(smem + SM::SCOPY) + b * 8192 + ks * 2048, D * 128, 1024,
                                              tc::kSwizzle128B);
            tc::mma_f16_ss(tmem, a, bd, idesc_x, (b | ks) != 0);
          }
        tc::mma_commit(mma_bar);
      }
      const float* gs = reinterpret_cast<const float*>(st + SM::F);
      const float* rqs = gs + C;
      const float* rks = gs + 2 * C;
      const float gC = gs[C - 1];
      const int ct_t0 = reinterpret_cast<const int*>(st + SM::F + 768)[0];
      const int ct_len = reinterpret_cast<const int*>(st + SM::F + 768)[1];
      const float sk_row = u_row ? expf(gC - gs[tid]) * rks[tid] : 0.f;       // Uk row scale
      const float sq_row = o_row ? expf(gs[tid - 64]) * rqs[tid - 64] * p.scale : 0.f;  // O row scale
      if (!tc::mbar_wait(mma_bar, mma_phase & 1, kWaitBudget)) {
        *s_fail = 1;
        set_status(p.status, GDN_ERR_TIMEOUT);
      }
      ++mma_phase;
      tc::fence_after_sync();
      if (u_row) {  // U = U~ - W<- S^T and Uk, row mu = tid
        const float sk = sk_row;
        uint32_t rr[VB / 16][16];
#pragma unroll
        for (int cc = 0; cc < VB / 16; ++cc) tc::tmem_ld16(tmem + lane_base + 16 * cc, rr[cc]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < VB / 16; ++cc) {
          const uint32_t* r = rr[cc];
          uint32_t wn[8], wk[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const __nv_bfloat162 u2 = reinterpret_cast<const __nv_bfloat162*>(&ut[2 * cc + (u >> 2)])[u & 3];
            const float2 uf = __bfloat1622float2(u2);
            const float n0 = uf.x - __uint_as_float(r[2 * u]), n1 = uf.y - __uint_as_float(r[2 * u + 1]);
            wn[u] = pack_bf16(n0, n1);
            wk[u] = pack_bf16(n0 * sk, n1 * sk);
          }
          *reinterpret_cast<uint4*>(smem + SM::VN + tc::sw128_offset(tid, 2 * cc)) = make_uint4(wn[0], wn[1], wn[2], wn[3]);
          *reinterpret_cast<uint4*>(smem + SM::VN + tc::sw128_offset(tid, 2 * cc + 1)) = make_uint4(wn[4], wn[5], wn[6], wn[7]);
          *reinterpret_cast<uint4*>(smem + SM::VK + tc::sw128_offset(tid, 2 * cc)) = make_uint4(wk[0], wk[1], wk[2], wk[3]);
          *reinterpret_cast<uint4*>(smem + SM::VK + tc::sw128_offset(tid, 2 * cc + 1)) = make_uint4(wk[4], wk[5], wk[6], wk[7]);
        }
        if (c + 1 < n_c) {  // prefetch the next chunk's U~ row
          const uint4* src = reinterpret_cast<const uint4*>(
              p.U + ((int64_t)(c_beg + c + 1) * p.HV + hv) * C * D + (int64_t)tid * D + vblk * VB);
#pragma unroll
          for (int q = 0; q < 8; ++q) ut[q] = src[q];
        }
      }
      tc::fence_async_smem();
      tc::fence_before_sync();
      tc::named_sync(1, kConsumers);
      // MMA3: DS = K^T Uk ; MMA2: D2 = [*; P] U
      if (tid == 0) {
        tc::fence_after_sync();
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = tc::smem_desc(tc::saddr(st + SM::K) + ks * 2048, 8192, 1024, tc::kSwizzle128B);
          const uint64_t bd = tc::smem_desc(tc::saddr(smem + SM::VK) + ks * 2048, 8192, 1024, tc::kSwizzle128B);
          tc::mma_f16_ss(tmem + 64, a, bd, idesc_s, ks > 0);
        }
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = tc::smem_desc(tc::saddr(st + SM::P - 8192) + ks * 32, 16, 1024, tc::kSwizzle128B);
          const uint64_t bd = tc::smem_desc(tc::saddr(smem + SM::VN) + ks * 2048, 8192, 1024, tc::kSwizzle128B);
          tc::mma_f16_ss(tmem + 128, a, bd, idesc_x, ks > 0);
        }
        tc::mma_commit(mma_bar);
      }
      if (!tc::mbar_wait(mma_bar, mma_phase & 1, kWaitBudget)) {
        *s_fail = 1;
        set_status(p.status, GDN_ERR_TIMEOUT);
      }
      ++mma_phase;
      tc::fence_after_sync();
      if (tid == 0) tc::mbar_arrive(&empty[s]);  // the MMAs are done with stage s; scalars are in registers
      if (has_state) {  // S <- exp(g_C) S + DS, and the bf16 copy for the next MMA1
        const float eC = expf(gC);
        uint32_t rr[VB / 16][16];
#pragma unroll
        for (int cc = 0; cc < VB / 16; ++cc) tc::tmem_ld16(tmem + lane_base + 64 + 16 * cc, rr[cc]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < VB / 16; ++cc) {
          const uint32_t* r = rr[cc];
          uint32_t w[8];
#pragma unroll
          for (int u = 0; u < 16; ++u) S[16 * cc + u] = fmaf(eC, S[16 * cc + u], __uint_as_float(r[u]));
#pragma unroll
          for (int u = 0; u < 8; ++u) w[u] = pack_bf16(S[16 * cc + 2 * u], S[16 * cc + 2 * u + 1]);
          *reinterpret_cast<uint4*>(smem + SM::SCOPY + tc::sw128_offset(tid, 2 * cc)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(smem + SM::SCOPY + tc::sw128_offset(tid, 2 * cc + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      if (o_row) {  // O row r = exp(g_r)/|q_r| (Q S^T)_r + (P U)_r
        const int r = tid - 64;
        const float sq = sq_row;
        const bool store = r < ct_len;  // padded rows are computed but not stored
        bf16* orow = p.out + (((int64_t)ct_t0 + r) * p.HV + hv) * (int64_t)D + vblk * VB;
#pragma unroll
        for (int cc = 0; cc < VB / 16; ++cc) {
          uint32_t a[16], b[16];  // tcgen05.ld is warp-collective: every lane loads
          tc::tmem_ld16(tmem + lane_base + 16 * cc, a);
          tc::tmem_ld16(tmem + lane_base + 128 + 16 * cc, b);
          tc::tmem_wait_ld();
          uint32_t w[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            w[u] = pack_bf16(sq * __uint_as_float(a[2 * u]) + p.scale * __uint_as_float(b[2 * u]),
                             sq * __uint_as_float(a[2 * u + 1]) + p.scale * __uint_as_float(b[2 * u + 1]));
          if (store) {
            uint4* d4 = reinterpret_cast<uint4*>(orow + 16 * cc);
            d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
      tc::fence_async_smem();
      tc::fence_before_sync();
      tc::named_sync(1, kConsumers);
    }
    if (has_state && !failed) {
#pragma unroll
      for (int v = 0; v < VB; ++v) Sg[(int64_t)v * D + tid] = S[v];
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_scan_t(const Params& p, cudaStream_t s) {
  using SM = ScanSmem<D>;
  const int64_t rows = p.max_chunks * p.HV * C;
  CUtensorMap mw, mp, mq, mk;
  if (!make_2d_tile_map(&mw, p.W, D, rows, 64, C, true) || !make_2d_tile_map(&mp, p.P, C, rows, 64, C, true) ||
      !make_token_tile_map(&mq, p.q, D, p.H, p.T, C) || !make_token_tile_map(&mk, p.k, D, p.H, p.T, C))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(scan_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::alloc);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.B * p.HV * (D / VB);
  scan_kernel<D><<<(unsigned)blocks, kThreads, SM::alloc, s>>>(mw, mp, mq, mk, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan(const Params& p, int D, int Cc, cudaStream_t s) {
  if (Cc != C || p.nvb != D / VB) return cudaErrorInvalidValue;
  switch (D) {
    case 64: return launch_scan_t<64>(p, s);
    case 128: return launch_scan_t<128>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
