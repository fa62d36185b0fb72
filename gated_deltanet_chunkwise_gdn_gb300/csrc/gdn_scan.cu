// gdn_scan.cu — K3: the sequential inter-chunk scan with the output epilogue, on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM) with TMA-fed chunk tiles.
//
// One CTA owns one block of VB = 64 state rows of one (sequence, value head) chain, for a
// range of chunks. Rows of the state S (V x K) evolve independently — the update contracts
// over the key dimension only — so the value dimension is split across CTAs while the key
// dimension stays whole ("nrm-training-kernels", section "Kernel": the grid splits batch,
// heads and blocks of the value dimension, never the key dimension).
//
// For each chunk, in order (pymllm page "pymllm.layers.attention.gdn_chunkwise": the
// inter-chunk propagation stays sequential):
//   U  = U~ - W<- S^T                               (the chunk's new values)
//   O  = diag(exp(g)/|q|) Q S^T + P U               (inter + masked intra part)
//   S <- exp(g_C) S + U^T K->,   K-> = diag(exp(g_C - g)/|k|) K
// i.e. "Simple math to speed up GDN prefill", section "Reminder": the chunk transition
// S_[t+1] = S-> + (U~ - W<- S^T)^T K-> with S-> = gamma_C S.
//
// Critical path per chunk (the "chain" warps 0-7; warps w and w+4 serve TMEM lanes
// 32(w%4)..+31, each taking half of the 64 columns):
//   MMA1  D1[128 x 64] = [Q; W<-] S^T          -> U = U~ - D1[64:128]; Uk = diag(exp(g_C-g)/|k|) U
//   MMA3  DS[K x 64]   = K^T (Uk_hi + Uk_lo)   -> S = exp(g_C) S + DS, 16-bit copy to smem
// Uk is carried as two 16-bit terms (hi + lo) against the exact K tile, so the state
// increment keeps about 16 bits of precision. Off the critical path:
//   MMA2  D2[128 x 64] = [P; *] U  and warps 8-9 form O from D1[0:64] and D2[0:64] one chunk
//   behind (D1, D2 double-buffered in TMEM);
//   warp 10 streams Q, W<-, K, P and the gate vectors with TMA (2-3 stage ring).
//
// Segment-parallel use (few long chains): besides a full scan over a chunk range
// (state from a buffer, outputs written), the same kernel computes the affine map of a
// chunk range — S_end = S_start T + B — as two scans without outputs: B from S_start = 0,
// and T (K x K) from the identity with U~ = 0. combine_kernel then chains the maps. For
// K = V = 128 the maps come from affine_scan_kernel (gdn_scan_affine.cu), and the factors are
// stored m-scaled (W'' = diag(m) W<-, U'' = diag(m) U~, P'' = P diag(1/m), see gdn_intra.cu):
// then U here is diag(m) U, P'' U'' = P U, and the key scale left to apply is ks = 2^e.
#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {

cudaError_t launch_combine(const Params& p, int D, int nseg, cudaStream_t s);
cudaError_t launch_affine_map_pass(const Params& p, cudaStream_t s);

namespace {

constexpr int C = 64;
constexpr int VB = 64;
// warps 0-7 chain workers (warps w and w+4 share TMEM lanes 32(w%4)..+31 and split the
// columns), warps 8-9 outputs (TMEM lanes 0-63), warp 10 TMA producer, warp 11 MMA issuer
constexpr int kChain = 256, kOut = 64;
constexpr int kThreads = 384;
constexpr int kProducerWarp = 10, kMmaWarp = 11;
constexpr uint32_t kTmemCols = 512;
// TMEM columns, per chain slot: D1 [64 slot, +64); DS [128 + 64 slot, +64) (and, for K = 256,
// keys 128-255 at [192, 256)); D2 [256 + 64 slot, +64). One chain per CTA uses slots 0/1 as a
// double buffer over chunks; two chains per CTA use slot = chain.
constexpr uint32_t kColD1 = 0, kColDS = 128, kColD2 = 256;

enum Mode : int { kFull = 0, kMapB = 1, kMapT = 2 };

// Chains (blocks of VB state rows) per CTA: for K = V = 128 one CTA runs both value blocks of
// a head, interleaved, so one block's tensor-core work overlaps the other's CUDA-core work
// and the chunk tiles are fetched once for both.
template <int D>
__host__ __device__ constexpr int chains_per_cta() { return D == 128 ? 2 : 1; }

template <int D>
struct ScanSmem {
  static constexpr int NB = D / 64;
  static constexpr int NCH = chains_per_cta<D>();
  static constexpr int STAGES = D == 64 ? 3 : (D == 128 ? 2 : 1);  // a K = 256 stage is 105 KB
  static constexpr uint32_t QW = 0;                 // NB x [Q block 8 KB][W<- block 8 KB]
  static constexpr uint32_t P = QW + NB * 16384;    // P 8 KB (A rows 64-127 of MMA2 = the 8 KB after it)
  static constexpr uint32_t K = P + 8192;           // NB x K block 8 KB (+ the 8 KB after: MMA3 rows K..127 if D = 64)
  static constexpr uint32_t F = K + NB * 8192;      // g, 1/|q|, 1/|k| (3 x 256 B), chunk t0 / len
  static constexpr uint32_t STAGE = F + 1024;
  // per chain ch at + ch * CH: 16-bit S^T (D rows x 128 B), U, Uk hi, Uk lo, U~ (64 rows x 128 B each)
  static constexpr uint32_t SCOPY = STAGES * STAGE;
  static constexpr uint32_t VN = SCOPY + D * 128;
  static constexpr uint32_t VKH = VN + 8192;
  static constexpr uint32_t VKL = VKH + 8192;
  static constexpr uint32_t UT = VKL + 8192;
  static constexpr uint32_t CH = D * 128 + 4 * 8192;
  static constexpr uint32_t BAR = SCOPY + NCH * CH;
  static constexpr uint32_t bytes = BAR + 256;
  static constexpr uint32_t alloc = bytes + 1024;
  static constexpr uint32_t tx_full = NB * 16384 + NB * 8192 + 8192 + 3 * 256;  // W, Q, K, P, F
  static constexpr uint32_t tx_map = NB * 8192 + NB * 8192 + 3 * 256;           // W, K, F
  static_assert(alloc <= 232448, "shared memory per CTA");
};

struct ScanJob {
  int mode;
  int seq, hv, vblk;  // vblk: the first of the CTA's value blocks
  int c0, c1;         // chunk range [c0, c1) within the sequence
  const float* init;  // [rows][D] start state (kFull); zeros (kMapB) / identity (kMapT) otherwise
  float* fin;         // [rows][D] where the final state goes, or nullptr
};

// Decodes this CTA's job. kind 0: whole sequences; kind 1: segment 0 (full) and the maps of
// segments 1 .. ns-2; kind 2: segments 1 .. ns-1 (full). Returns false if there is no job.
template <int D>
__device__ bool decode_job(const Params& p, int kind, int nseg, ScanJob& job) {
  constexpr int NVB = D / VB / chains_per_cta<D>();  // CTAs per state (VB x NCH rows each)
  const int B = p.B, HV = p.HV;
  const int64_t per_head = (int64_t)D * D;  // floats per (slot, value head) state
  int bid = blockIdx.x;
  job.init = nullptr;
  job.fin = nullptr;
  if (kind == 0 || (kind == 1 && bid < B * HV * NVB)) {
    job.vblk = (bid % NVB) * chains_per_cta<D>();
    bid /= NVB;
    job.seq = p.order[bid / HV];
    job.hv = bid % HV;
    const int n = p.seq_chunk_off[job.seq + 1] - p.seq_chunk_off[job.seq];
    float* pool = p.state_pool + (p.cache_indices[job.seq] * HV + job.hv) * per_head;
    job.mode = kFull;
    job.init = pool;
    if (kind == 0) {
      job.c0 = 0;
      job.c1 = n;
      job.fin = pool;
    } else {
      int ns;
      seg_range(n, nseg, p.seg_r16, 0, job.c0, job.c1, ns);
      job.fin = ns > 1 ? p.seg_state + (((int64_t)job.seq * HV + job.hv) * nseg + 1) * per_head : pool;
    }
    return job.c1 > job.c0;
  }
  if (kind == 1) {  // maps of segments 1 .. nseg-2: (B rows | T rows) x NVB blocks each
    bid -= B * HV * NVB;
    const int per_chain = (nseg - 2) * 2 * NVB;
    const int rest = bid / per_chain;
    int idx = bid % per_chain;
    job.seq = p.order[rest / HV];
    job.hv = rest % HV;
    job.vblk = (idx % NVB) * chains_per_cta<D>();
    idx /= NVB;
    const int which = idx % 2, seg = 1 + idx / 2;
    const int n = p.seq_chunk_off[job.seq + 1] - p.seq_chunk_off[job.seq];
    int ns;
    seg_range(n, nseg, p.seg_r16, seg, job.c0, job.c1, ns);
    if (seg >= ns - 1) return false;
    job.mode = which == 0 ? kMapB : kMapT;
    job.fin = p.seg_map + (((int64_t)job.seq * HV + job.hv) * nseg + seg) * 2 * per_head + (which == 0 ? 0 : per_head);
    return job.c1 > job.c0;
  }
  // kind 2: segments 1 .. nseg-1, full
  job.vblk = (bid % NVB) * chains_per_cta<D>();
  bid /= NVB;
  const int seg = 1 + bid % (nseg - 1);
  bid /= (nseg - 1);
  job.seq = p.order[bid / HV];
  job.hv = bid % HV;
  const int n = p.seq_chunk_off[job.seq + 1] - p.seq_chunk_off[job.seq];
  int ns;
  seg_range(n, nseg, p.seg_r16, seg, job.c0, job.c1, ns);
  if (seg >= ns) return false;
  job.mode = kFull;
  job.init = p.seg_state + (((int64_t)job.seq * HV + job.hv) * nseg + seg) * per_head;
  job.fin = seg == ns - 1 ? p.state_pool + (p.cache_indices[job.seq] * HV + job.hv) * per_head : nullptr;
  return job.c1 > job.c0;
}

// Bounded mbarrier wait that also gives up as soon as another role reported a failure.
__device__ __forceinline__ bool wait_or_fail(uint64_t* bar, uint32_t parity, volatile int* fail, long long budget) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (*fail || clock64() - t0 > budget) return false;
  }
  return true;
}

template <int D, typename E>
__global__ void __launch_bounds__(kThreads, 1)
    scan_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_p,
                const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, Params p, int kind,
                int nseg) {
  using SM = ScanSmem<D>;
  constexpr int NB = SM::NB, S = SM::STAGES, NCH = SM::NCH;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  if (p.status[0] != GDN_OK) return;
  ScanJob job;
  if (!decode_job<D>(p, kind, nseg, job)) return;  // uniform over the CTA
  const int mode = job.mode, hv = job.hv, vblk = job.vblk;
  const int h = hv / (p.HV / p.H);
  const int cb = p.seq_chunk_off[job.seq];
  const int nc = job.c1 - job.c0;
  const bool full_mode = mode == kFull;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::BAR);  // [S]
  uint64_t* empty = full + S;                                    // [S]
  uint64_t* mma1 = empty + S;                                    // [2] D1 of chain ch ready
  uint64_t* mma3 = mma1 + 2;                                     // [2] DS of chain ch ready
  uint64_t* mmao = mma3 + 2;                                     // [2] D2 of slot ready
  uint64_t* odone = mmao + 2;                                    // [2] O warps done with slot's D1/D2
  uint64_t* uready = odone + 2;                                  // [2] chain ch: U, Uk written, gates read
  uint64_t* sready = uready + 2;                                 // [2] chain ch: 16-bit S^T written
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sready + 2);
  volatile int* fail = reinterpret_cast<volatile int*>(tslot + 1);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], full_mode ? 2 : 1);  // the MMAs (and the output warps) release a stage
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&mma1[b], 1);
      tc::mbar_init(&mma3[b], 1);
      tc::mbar_init(&mmao[b], 1);
      tc::mbar_init(&odone[b], kOut);
      tc::mbar_init(&uready[b], kChain / 32);  // one arrival per chain warp
      tc::mbar_init(&sready[b], kChain / 32);
    }
    *fail = 0;
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
  auto report = [&]() {
    *fail = 1;
    set_status(p.status, GDN_ERR_TIMEOUT);
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer: TMA
    if (lane == 0 && p.stall != kStallScan) {
      for (int c = 0; c < nc; ++c) {
        const int s = c % S, use = c / S;
        if (use > 0 && !wait_or_fail(&empty[s], (use - 1) & 1, fail, p.wait_budget)) {
          report();
          break;
        }
        const int j = cb + job.c0 + c;
        const int4 ct = p.chunk_tab[j];
        const int64_t jh = (int64_t)j * p.HV + hv;
        const int64_t jq = (int64_t)j * p.H + h;
        unsigned char* st = smem + s * SM::STAGE;
        reinterpret_cast<int*>(st + SM::F + 768)[0] = ct.y;
        reinterpret_cast<int*>(st + SM::F + 768)[1] = ct.z;
        tc::mbar_arrive_expect_tx(&full[s], full_mode ? SM::tx_full : SM::tx_map);
        for (int b = 0; b < NB; ++b) {
          if (full_mode) tc::tma_load_3d(st + SM::QW + b * 16384, &tm_q, 64 * b, h, ct.y, &full[s]);
          tc::tma_load_2d(st + SM::QW + b * 16384 + 8192, &tm_w, 64 * b, (int)(jh * C), &full[s]);
          tc::tma_load_3d(st + SM::K + b * 8192, &tm_k, 64 * b, h, ct.y, &full[s]);
        }
        if (full_mode) tc::tma_load_2d(st + SM::P, &tm_p, 0, (int)(jh * C), &full[s]);
        tc::bulk_load(st + SM::F, p.g + jh * C, 256, &full[s]);
        tc::bulk_load(st + SM::F + 256, p.rq + jq * C, 256, &full[s]);
        // K = V = 128: the factors are stored m-scaled (see the intra kernel), the key scale is ks = 2^e
        if (D == 128) tc::bulk_load(st + SM::F + 512, p.ks + jh * C, 256, &full[s]);
        else tc::bulk_load(st + SM::F + 512, p.rk + jq * C, 256, &full[s]);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer (one thread)
    if (lane == 0) {
      constexpr int NKR = D > 128 ? 2 : 1;
      constexpr uint32_t idesc_x = tc::idesc_f16(128, VB, ElemT<E>::fmt, false, true);  // A K-major, B MN-major
      constexpr uint32_t idesc_s = tc::idesc_f16(128, VB, ElemT<E>::fmt, true, true);   // both MN-major
      // Base descriptors; an operand at byte offset o from its base is base + (o >> 4) (the
      // start-address field holds address >> 4 and shared addresses stay below 256 KB).
      const uint64_t dA1 = tc::smem_desc(tc::saddr(smem + SM::QW), 16, 1024, tc::kSwizzle128B);
      const uint64_t dB1 = tc::smem_desc(tc::saddr(smem + SM::SCOPY), D * 128, 1024, tc::kSwizzle128B);
      const uint64_t dA3 = tc::smem_desc(tc::saddr(smem + SM::K), 8192, 1024, tc::kSwizzle128B);
      const uint64_t dB3 = tc::smem_desc(tc::saddr(smem + SM::VKH), 8192, 1024, tc::kSwizzle128B);
      const uint64_t dA2 = tc::smem_desc(tc::saddr(smem + SM::P), 16, 1024, tc::kSwizzle128B);
      const uint64_t dB2 = tc::smem_desc(tc::saddr(smem + SM::VN), 8192, 1024, tc::kSwizzle128B);
      static_assert(SM::VKL == SM::VKH + 8192, "Uk lo follows Uk hi");
      bool ok = true;
      for (int c = 0; c < nc && ok; ++c) {
        const int s = c % S;
        const uint32_t so = (uint32_t)(s * SM::STAGE) >> 4;  // stage offset in descriptor units
        ok = wait_or_fail(&full[s], (c / S) & 1, fail, p.wait_budget);
        // MMA1: D1[slot] = [Q; W<-] S^T, once the chain's 16-bit S^T of chunk c-1 is written and
        // the output warps are done with the slot
        for (int ch = 0; ch < NCH && ok; ++ch) {
          const int slot = NCH == 1 ? (c & 1) : ch;
          const int use = NCH == 1 ? (c >> 1) : c;
          const uint32_t co = (uint32_t)(ch * SM::CH) >> 4;
          ok = wait_or_fail(&sready[ch], c & 1, fail, p.wait_budget);
          if (ok && full_mode && use >= 1) ok = wait_or_fail(&odone[slot], (use - 1) & 1, fail, p.wait_budget);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_f16_ss(tmem + kColD1 + 64 * slot, dA1 + so + ((b * 16384 + ks * 32) >> 4),
                             dB1 + co + ((b * 8192 + ks * 2048) >> 4), idesc_x, (b | ks) != 0);
          tc::mma_commit(&mma1[ch]);
        }
        // MMA3: DS[ch] = K^T (Uk_hi + Uk_lo) (the chain waits for this); MMA2: D2[slot] = [P; *] U
        for (int ch = 0; ch < NCH && ok; ++ch) {
          const int slot = NCH == 1 ? (c & 1) : ch;
          const uint32_t co = (uint32_t)(ch * SM::CH) >> 4;
          ok = wait_or_fail(&uready[ch], c & 1, fail, p.wait_budget);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int kr = 0; kr < NKR; ++kr)  // keys 128 kr .. 128 kr + 127: K blocks 2 kr, 2 kr + 1
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                tc::mma_f16_ss(tmem + kColDS + 64 * (ch * NKR + kr), dA3 + so + ((kr * 16384 + ks * 2048) >> 4),
                               dB3 + co + ((part * 8192 + ks * 2048) >> 4), idesc_s, (part | ks) != 0);
          tc::mma_commit(&mma3[ch]);
          if (full_mode) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_f16_ss(tmem + kColD2 + 64 * slot, dA2 + so + ((ks * 32) >> 4), dB2 + co + ((ks * 2048) >> 4),
                             idesc_x, ks > 0);
            tc::mma_commit(&mmao[slot]);
          }
        }
        // the stage is free once every MMA of chunk c is done (no later chunk reuses the last S)
        if (ok && c + S < nc) tc::mma_commit(&empty[s]);
      }
      if (!ok) report();
    }
    __syncwarp();
  } else if (warp >= kChain / 32) {
    // ------------------------------------------------------------------ outputs, one step behind
    if (full_mode) {
      const int r = tid - kChain;  // output row of the chunk (warps 8-9: TMEM lanes 0-63)
      const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
      bool bad = false;
      for (int c = 0; c < nc && !bad; ++c) {
        const int s = c % S;
        const unsigned char* st = smem + s * SM::STAGE;
        float sq = 0.f;
        int t0 = 0, len = 0;
        for (int ch = 0; ch < NCH; ++ch) {
          const int slot = NCH == 1 ? (c & 1) : ch;
          const int use = NCH == 1 ? (c >> 1) : c;
          if (!wait_or_fail(&mmao[slot], use & 1, fail, p.wait_budget)) {
            report();
            bad = true;
            break;
          }
          tc::fence_after_sync();
          if (ch == 0) {
            const float* gs = reinterpret_cast<const float*>(st + SM::F);
            sq = expf(gs[r]) * gs[C + r] * p.scale;
            t0 = reinterpret_cast<const int*>(st + SM::F + 768)[0];
            len = reinterpret_cast<const int*>(st + SM::F + 768)[1];
          }
          if (ch == NCH - 1) {  // every chain's P product is done and the gates are read
            tc::named_sync(3, kOut);
            if (tid == kChain) tc::mbar_arrive(&empty[s]);
          }
          E* orow = reinterpret_cast<E*>(p.out) + (((int64_t)t0 + r) * p.HV + hv) * (int64_t)D + (vblk + ch) * VB;
#pragma unroll
          for (int cc = 0; cc < VB / 16; ++cc) {
            uint32_t a[16], b[16];  // warp-collective TMEM loads: every lane loads
            tc::tmem_ld16(tmem + lane_base + kColD1 + 64 * slot + 16 * cc, a);
            tc::tmem_ld16(tmem + lane_base + kColD2 + 64 * slot + 16 * cc, b);
            tc::tmem_wait_ld();
            if (r < len) {
              uint32_t w[8];
#pragma unroll
              for (int u = 0; u < 8; ++u)
                w[u] = ElemT<E>::pack(sq * __uint_as_float(a[2 * u]) + p.scale * __uint_as_float(b[2 * u]),
                                 sq * __uint_as_float(a[2 * u + 1]) + p.scale * __uint_as_float(b[2 * u + 1]));
              uint4* d4 = reinterpret_cast<uint4*>(orow + 16 * cc);
              d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
              d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
          tc::fence_before_sync();
          tc::mbar_arrive(&odone[slot]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ chain workers: U, state update
    const int sub = warp & 3, half = warp >> 2;
    const int row = 32 * sub + lane;                        // TMEM lane of this thread
    const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
    const int cbase = 32 * half;                            // first of this thread's 32 columns
    constexpr int NKR = D > 128 ? 2 : 1;  // key rows per thread: row and row + 128
    const bool has_state = row < D;  // thread (row, half) holds columns cbase.. of key rows row (+128) of S^T
    const bool u_row = row >= 64;    // thread (64 + mu, half) forms half of row mu of U (TMEM lanes 64-127)
    const int mu = row - 64;         // (both flags are uniform over a warp)
    const bool use_ut = mode != kMapT;
    float S_[NCH][NKR][32];
    // 16-bit copy of the state rows this thread holds, for the next MMA1 of chain ch
    auto write_scopy = [&](int ch) {
      unsigned char* scopy = smem + SM::SCOPY + ch * SM::CH;
#pragma unroll
      for (int kr = 0; kr < NKR; ++kr) {
        const int key = row + 128 * kr;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) w[u] = ElemT<E>::pack(S_[ch][kr][8 * cc + 2 * u], S_[ch][kr][8 * cc + 2 * u + 1]);
          *reinterpret_cast<uint4*>(scopy + tc::sw128_offset(key, 4 * half + cc)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    };
    // a warp's shared-memory writes are complete and visible to the tensor cores: tell the issuer
    auto signal = [&](uint64_t* bar) {
      tc::fence_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar);
    };
    if (has_state) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const int64_t row0 = (int64_t)(vblk + ch) * VB + cbase;  // first state row held by this thread
#pragma unroll
        for (int kr = 0; kr < NKR; ++kr) {
          const int key = row + 128 * kr;
          if (mode == kFull) {
#pragma unroll
            for (int v = 0; v < 32; ++v) S_[ch][kr][v] = job.init[(row0 + v) * D + key];
          } else if (mode == kMapT) {
#pragma unroll
            for (int v = 0; v < 32; ++v) S_[ch][kr][v] = (row0 + v == key) ? 1.f : 0.f;
          } else {
#pragma unroll
            for (int v = 0; v < 32; ++v) S_[ch][kr][v] = 0.f;
          }
        }
        write_scopy(ch);
      }
    }
    // U~ rows of a chunk, fetched by the threads that use them (half a row each)
    auto fetch_ut = [&](int c) {
      const int64_t j = cb + job.c0 + c;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const E* src = reinterpret_cast<const E*>(p.U) + (j * p.HV + hv) * C * D + (int64_t)mu * D + (vblk + ch) * VB + cbase;
        unsigned char* dst = smem + SM::UT + ch * SM::CH;
#pragma unroll
        for (int q = 0; q < 4; ++q) cp_async_16(dst + tc::sw128_offset(mu, 4 * half + q), src + 8 * q);
      }
      cp_async_commit();
    };
    // bounded wait with one outcome per warp (the warp then stays converged)
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) {
      const bool ok = wait_or_fail(bar, parity, fail, p.wait_budget);
      return __all_sync(0xffffffffu, ok);
    };
    if (u_row && use_ut) fetch_ut(0);
    for (int ch = 0; ch < NCH; ++ch) signal(&sready[ch]);  // the start state is in place

    bool failed = false;
    for (int c = 0; c < nc; ++c) {
      const int s = c % S;
      const unsigned char* st = smem + s * SM::STAGE;
      if (!wait_warp(&full[s], (c / S) & 1)) {
        failed = true;
        break;
      }
      const float* gs = reinterpret_cast<const float*>(st + SM::F);
      const float gC = gs[C - 1];
      const float eC = expf(gC);
      // exp(g_C - g_mu) / |k_mu|; for K = V = 128 the rows of U~, W<- carry its mantissa m_mu (and P the
      // inverse), so U here is diag(m) U and the remaining factor is ks_mu = 2^e_mu
      const float sk = u_row ? (D == 128 ? gs[2 * C + mu] : expf(gC - gs[mu]) * gs[2 * C + mu]) : 0.f;
      if (u_row && use_ut) cp_async_wait<0>();  // this thread's U~ rows of chunk c
      for (int ch = 0; ch < NCH && !failed; ++ch) {
        if (u_row) {  // U = U~ - W<- S^T (half row mu); Uk = sk U as 16-bit hi + lo
          if (!wait_warp(&mma1[ch], c & 1)) {
            failed = true;
            break;
          }
          tc::fence_after_sync();
          const int slot = NCH == 1 ? (c & 1) : ch;
          unsigned char* cbuf = smem + ch * SM::CH;
          uint32_t rr[2][16];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) tc::tmem_ld16(tmem + lane_base + kColD1 + 64 * slot + cbase + 16 * cc, rr[cc]);
          uint4 ut[4] = {};
          if (use_ut) {
#pragma unroll
            for (int q = 0; q < 4; ++q) ut[q] = *reinterpret_cast<const uint4*>(cbuf + SM::UT + tc::sw128_offset(mu, 4 * half + q));
          }
          tc::tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t wn[8], wh[8], wl[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float2 uf = ElemT<E>::unpack(reinterpret_cast<const uint32_t*>(&ut[2 * cc + (u >> 2)])[u & 3]);
              const float n0 = uf.x - __uint_as_float(rr[cc][2 * u]), n1 = uf.y - __uint_as_float(rr[cc][2 * u + 1]);
              wn[u] = ElemT<E>::pack(n0, n1);
              split2<E>(n0 * sk, n1 * sk, wh[u], wl[u]);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t o = tc::sw128_offset(mu, 4 * half + 2 * cc + hh);
              *reinterpret_cast<uint4*>(cbuf + SM::VN + o) = make_uint4(wn[4 * hh], wn[4 * hh + 1], wn[4 * hh + 2], wn[4 * hh + 3]);
              *reinterpret_cast<uint4*>(cbuf + SM::VKH + o) = make_uint4(wh[4 * hh], wh[4 * hh + 1], wh[4 * hh + 2], wh[4 * hh + 3]);
              *reinterpret_cast<uint4*>(cbuf + SM::VKL + o) = make_uint4(wl[4 * hh], wl[4 * hh + 1], wl[4 * hh + 2], wl[4 * hh + 3]);
            }
          }
        }
        signal(&uready[ch]);  // also: this warp has read the chunk's gates
      }
      if (failed) break;
      if (u_row && use_ut && c + 1 < nc) fetch_ut(c + 1);  // every chain has read its U~ rows of chunk c
      for (int ch = 0; ch < NCH; ++ch) {
        if (!wait_warp(&mma3[ch], c & 1)) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        if (has_state) {  // S <- exp(g_C) S + DS
#pragma unroll
          for (int kr = 0; kr < NKR; ++kr) {
            uint32_t rr[2][16];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
              tc::tmem_ld16(tmem + lane_base + kColDS + 64 * (ch * NKR + kr) + cbase + 16 * cc, rr[cc]);
            tc::tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) S_[ch][kr][u] = fmaf(eC, S_[ch][kr][u], __uint_as_float(rr[u >> 4][u & 15]));
          }
          write_scopy(ch);
        }
        signal(&sready[ch]);
      }
      if (failed) break;
    }
    if (failed) report();
    if (u_row && use_ut) cp_async_wait<0>();  // no copy outlives the CTA
    if (has_state && !failed && job.fin) {
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        const int64_t row0 = (int64_t)(vblk + ch) * VB + cbase;
#pragma unroll
        for (int kr = 0; kr < NKR; ++kr)
#pragma unroll
          for (int v = 0; v < 32; ++v) job.fin[(row0 + v) * D + row + 128 * kr] = S_[ch][kr][v];
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Chains the segment maps of one (sequence, value head): S_{p+1} = S_p T_p + B_p for
// p = 1 .. ns-2, starting from S_1 (the end state of segment 0). One CTA per 16 state
// rows; fp32 on CUDA cores with T_p staged in shared memory 32 key rows at a time.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(Params p, int nseg) {
  constexpr int R = 16;   // state rows per CTA
  constexpr int KB = 32;  // key rows of T_p per staging step
  extern __shared__ float csm[];
  float* Tb = csm;         // KB x D
  float* Sr = Tb + KB * D;  // R x D
  if (p.status[0] != GDN_OK) return;
  int bid = blockIdx.x;
  const int rb = bid % (D / R);
  bid /= (D / R);
  const int hv = bid % p.HV;
  const int seq = p.order[bid / p.HV];
  const int n = p.seq_chunk_off[seq + 1] - p.seq_chunk_off[seq];
  int ns, c0_, c1_;
  seg_range(n, nseg, p.seg_r16, 0, c0_, c1_, ns);
  if (ns < 3) return;
  const int64_t per_head = (int64_t)D * D;
  const int64_t base = ((int64_t)seq * p.HV + hv) * nseg;
  const int tid = threadIdx.x;
  for (int e = tid; e < R * D; e += 256) Sr[e] = p.seg_state[(base + 1) * per_head + (int64_t)rb * R * D + e];
  const int r = tid / 16, c0 = (tid % 16) * (D / 16);  // one row, D/16 columns per thread
  for (int seg = 1; seg <= ns - 2; ++seg) {
    const float* Tg = p.seg_map + (base + seg) * 2 * per_head + per_head;  // T_p (rows: key index)
    const float* Bg = p.seg_map + (base + seg) * 2 * per_head;             // B_p (rows: value index)
    float acc[D / 16];
#pragma unroll
    for (int u = 0; u < D / 16; ++u) acc[u] = Bg[((int64_t)rb * R + r) * D + c0 + u];
    for (int k0 = 0; k0 < D; k0 += KB) {
      __syncthreads();
      for (int e = tid; e < KB * D; e += 256) Tb[e] = Tg[(int64_t)k0 * D + e];
      __syncthreads();
      for (int k = 0; k < KB; ++k) {
        const float sk = Sr[r * D + k0 + k];
#pragma unroll
        for (int u = 0; u < D / 16; ++u) acc[u] = fmaf(sk, Tb[k * D + c0 + u], acc[u]);
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < D / 16; ++u) Sr[r * D + c0 + u] = acc[u];
    __syncthreads();
    for (int e = tid; e < R * D; e += 256)
      p.seg_state[(base + seg + 1) * per_head + (int64_t)rb * R * D + e] = Sr[e];
  }
}

// The same chaining for K <= 128: one CTA of 256 threads per 16 state rows; T_p (K x K fp32,
// <= 64 KB) and the CTA's 16 rows of B_p are fetched by bulk copies one segment ahead (two
// buffers), so the loads overlap the previous segment's products. Thread (column c, row group)
// forms column c of 16 * D / 256 rows, reading T_p[k][c] once per k for all of them; the CTA's
// rows of S_p are kept transposed ([k][row], 16-byte groups XOR-swizzled by k) so that each k
// brings them in with a few broadcast vector loads.
template <int D>
__global__ void __launch_bounds__(256) combine_bulk_kernel(Params p, int nseg) {
  constexpr int R = 16;             // state rows per CTA
  constexpr int RPT = R * D / 256;  // rows per thread (8 for D = 128, 4 for D = 64)
  extern __shared__ __align__(16) float cbm[];
  float* Tb = cbm;                 // 2 x D x D
  float* Bb = Tb + 2 * D * D;      // 2 x R x D
  float* St = Bb + 2 * R * D;      // D x R: St[k][r] at k * R + swz(k, r)
  uint64_t* bar = reinterpret_cast<uint64_t*>(St + R * D);  // [2]
  if (p.status[0] != GDN_OK) return;
  int bid = blockIdx.x;
  const int rb = bid % (D / R);
  bid /= (D / R);
  const int hv = bid % p.HV;
  const int seq = p.order[bid / p.HV];
  const int n = p.seq_chunk_off[seq + 1] - p.seq_chunk_off[seq];
  int ns, c0_, c1_;
  seg_range(n, nseg, p.seg_r16, 0, c0_, c1_, ns);
  if (ns < 3) return;
  const int64_t per_head = (int64_t)D * D;
  const int64_t base = ((int64_t)seq * p.HV + hv) * nseg;
  const int tid = threadIdx.x;
  auto swz = [](int k, int r) { return ((((r >> 2) ^ k) & (R / 4 - 1)) << 2) | (r & 3); };
  auto fetch = [&](int seg) {  // thread 0: T and this CTA's rows of B of segment seg into buffer (seg - 1) & 1
    const int b = (seg - 1) & 1;
    const float* m = p.seg_map + (base + seg) * 2 * per_head;
    tc::mbar_arrive_expect_tx(&bar[b], (D * D + R * D) * 4);
    tc::bulk_load(Tb + b * D * D, m + per_head, D * D * 4, &bar[b]);
    tc::bulk_load(Bb + b * R * D, m + (int64_t)rb * R * D, R * D * 4, &bar[b]);
  };
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_fence_init();
    fetch(1);
    if (ns - 2 >= 2) fetch(2);
  }
  const float* S1 = p.seg_state + (base + 1) * per_head + (int64_t)rb * R * D;
  for (int e = tid; e < R * D; e += 256) {
    const int r = e / D, k = e % D;
    St[k * R + swz(k, r)] = S1[e];
  }
  __syncthreads();
  const int c = tid % D, r0 = (tid / D) * RPT;  // column and first row of this thread
  for (int seg = 1; seg <= ns - 2; ++seg) {
    const int b = (seg - 1) & 1;
    if (!__syncthreads_and(tc::mbar_wait(&bar[b], ((seg - 1) >> 1) & 1, p.wait_budget))) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT);
      return;
    }
    const float* T = Tb + b * D * D;
    float acc[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) acc[i] = Bb[b * R * D + (r0 + i) * D + c];
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
      const float t = T[k * D + c];
#pragma unroll
      for (int q = 0; q < RPT / 4; ++q) {
        const float4 s4 = *reinterpret_cast<const float4*>(St + k * R + swz(k, r0 + 4 * q));
        acc[4 * q] = fmaf(s4.x, t, acc[4 * q]);
        acc[4 * q + 1] = fmaf(s4.y, t, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(s4.z, t, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(s4.w, t, acc[4 * q + 3]);
      }
    }
    __syncthreads();  // every thread is done with S_p and buffer b
    if (tid == 0 && seg + 2 <= ns - 2) {
      tc::fence_async_smem();
      fetch(seg + 2);
    }
    float* dst = p.seg_state + (base + seg + 1) * per_head + (int64_t)rb * R * D;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      St[c * R + swz(c, r0 + i)] = acc[i];
      dst[(r0 + i) * D + c] = acc[i];
    }
    __syncthreads();
  }
}

template <int D, typename E>
cudaError_t launch_scan_t(const Params& p, int nseg, cudaStream_t s) {
  const bool h = p.fp16 != 0;
  using SM = ScanSmem<D>;
  constexpr int NVB = D / VB / chains_per_cta<D>();  // CTAs per state
  const int64_t rows = p.max_chunks * p.HV * C;
  CUtensorMap mw, mp, mq, mk;
  if (!make_2d_tile_map(&mw, p.W, D, rows, 64, C, true, h) || !make_2d_tile_map(&mp, p.P, C, rows, 64, C, true, h) ||
      !make_token_tile_map(&mq, p.q, D, p.H, p.T, C, h) || !make_token_tile_map(&mk, p.k, D, p.H, p.T, C, h))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(scan_kernel<D, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::alloc);
  if (e != cudaSuccess) return e;
  const int64_t chains = (int64_t)p.B * p.HV;
  if (nseg <= 1) {
    scan_kernel<D, E><<<(unsigned)(chains * NVB), kThreads, SM::alloc, s>>>(mw, mp, mq, mk, p, 0, 1);
    return cudaGetLastError();
  }
  // segment 0 and the maps of segments 1 .. nseg-2, then the combine, then segments 1 .. nseg-1.
  // K = V = 128: the first pass runs in affine-transition form (one CTA per map builds B and T
  // with a shared transition), the segment pass here.
  if constexpr (D == 128) {
    if ((e = launch_affine_map_pass(p, s)) != cudaSuccess) return e;
  } else {
    const int64_t grid1 = chains * NVB + chains * (nseg - 2) * 2 * NVB;
    scan_kernel<D, E><<<(unsigned)grid1, kThreads, SM::alloc, s>>>(mw, mp, mq, mk, p, 1, nseg);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (nseg > 2 && (e = launch_combine(p, D, nseg, s)) != cudaSuccess) return e;
  scan_kernel<D, E><<<(unsigned)(chains * (nseg - 1) * NVB), kThreads, SM::alloc, s>>>(mw, mp, mq, mk, p, 2, nseg);
  return cudaGetLastError();
}

}  // namespace

// Chains the segment maps (B, T) of every (sequence, value head): S_{p+1} = S_p T_p + B_p.
cudaError_t launch_combine(const Params& p, int D, int nseg, cudaStream_t s) {
  const int64_t chains = (int64_t)p.B * p.HV;
  cudaError_t e;
  if (D <= 128) {
    const size_t csmem = (size_t)(2 * D * D + 3 * 16 * D) * sizeof(float) + 16;
    auto kern = D == 64 ? combine_bulk_kernel<64> : combine_bulk_kernel<128>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem)) != cudaSuccess) return e;
    kern<<<(unsigned)(chains * (D / 16)), 256, csmem, s>>>(p, nseg);
  } else {
    const size_t csmem = (size_t)(32 * D + 16 * D) * sizeof(float);
    if ((e = cudaFuncSetAttribute(combine_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem)) !=
        cudaSuccess)
      return e;
    combine_kernel<256><<<(unsigned)(chains * (D / 16)), 256, csmem, s>>>(p, nseg);
  }
  return cudaGetLastError();
}

cudaError_t launch_scan(const Params& p, int D, int Cc, cudaStream_t s) {
  if (Cc != C) return cudaErrorInvalidValue;
  if (p.nvb != D / VB) return cudaErrorInvalidValue;
  switch (D) {
    case 64: return p.fp16 ? launch_scan_t<64, f16>(p, p.nseg, s) : launch_scan_t<64, bf16>(p, p.nseg, s);
    case 128: return p.fp16 ? launch_scan_t<128, f16>(p, p.nseg, s) : launch_scan_t<128, bf16>(p, p.nseg, s);
    case 256: return p.fp16 ? launch_scan_t<256, f16>(p, p.nseg, s) : launch_scan_t<256, bf16>(p, p.nseg, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
