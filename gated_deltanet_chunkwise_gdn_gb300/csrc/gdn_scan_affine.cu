// gdn_scan_affine.cu — first pass of the segmented scan for K = V = 128, in affine-transition
// form, on the 5th-generation tensor cores (tcgen05, accumulators in TMEM) with TMA-fed chunk tiles.
//
// The chunk step of "Simple math to speed up GDN prefill" (section "Reminder"),
//   S_next = exp(g_C) S + (U~ - W<- S^T)^T diag(sk) K,   sk_t = exp(g_C - g_t)/|k_t|,
// is affine in the state S (V x K):
//   S_next = exp(g_C) S - S M + B,   M = W<-^T diag(sk) K  (K x K),   B = U~^T diag(sk) K  (V x K).
// M and B do not depend on S, so each chunk's critical path is a single product S M
// (one tcgen05 group of 8 MMAs) and one fp32 update. A segment of chunks is the affine map
// S_end = S_start T + B_seg, with T the product of the (exp(g_C) I - M) and B_seg the state reached
// from S_start = 0: one CTA runs both chains with one shared M per chunk (the B chain in the chain
// warps, the T chain T <- exp(g_C) T - T M from T = I in fp32 in TMEM). combine_kernel then chains
// the maps and the second pass (scan_kernel) re-runs the segments from their start states.
// Segment 0 of each sequence runs here in full mode (outputs, its end state to the segment-state
// buffer), alongside the maps.
//
// The factor sk is split exactly as sk_t = m_t 2^e_t (m_t in [0.5, 1)): the intra kernel stored
// W'' = diag(m) W<-, U'' = diag(m) U~ and P'' = P diag(1/m), and this kernel scales the raw keys by
// ks_t = 2^e_t (exact in 16 bits): K~ = diag(ks) K, so M = W''^T K~ and B = U''^T K~ with no
// rounding beyond that of the stored factors.
//
// Outputs (full mode) use the state S entering the chunk ("nrm-training-kernels", "General
// implementation": inter-chunk part from the carried state plus the masked intra-chunk part):
//   D_O[0:64]   = Q~ S^T,  Q~ = diag(exp(g)/|q|) Q       (rows: tokens)
//   D_O[64:128] = W'' S^T  ->  U'' = U'' - D_O[64:128]   (= diag(m) U, in place)
//   D_O[0:64]  += P'' U''                                (= P U)
//   O = scale * D_O[0:64]
// Map mode keeps the 16-bit copies of S and T that feed the chain products in TMEM (the
// products read their A operand from TMEM, so only -M streams from shared memory), and the T
// chain accumulates in place: its TMEM state is pre-scaled by exp(g_C) and the MMA adds T (-M).
// One CTA per (sequence, value head, segment), 832 threads:
//   warps 0-15  chain: fp32 state rows in registers (TMEM lane quarter w%4, 32 key columns
//               each), S <- exp(g_C) S + D_S, 16-bit copy of S for the next products (shared
//               memory in full mode, TMEM in map mode);
//   warps 16-19 prep: K~ and Q~ in place in the chunk's tiles; M from TMEM to a 16-bit
//               B operand (negated);
//   warps 20-23 full mode: output rows (warps 20-21, TMEM lanes 0-63) and U'' rows formed in
//               place in the U'' tile (warps 22-23, lanes 64-127); map mode: the T chain;
//   warp 24     TMA producer (2-stage ring of the chunk tiles and gate rows);
//   warp 25     MMA issuer (one thread).
// A map-mode stage is free as soon as M and B of its chunk are formed, so the ring prefetches two
// chunks ahead.
#include "gdn_common.cuh"
#include "gdn_tc.cuh"

namespace gdn {

cudaError_t launch_combine(const Params& p, int D, int nseg, cudaStream_t s);

namespace {

constexpr int C = 64;
constexpr int D = 128;
constexpr int kThreads = 832;
constexpr int kChainWarps = 16;  // 4 per TMEM lane quarter, 32 state columns each
constexpr int kPrepWarp0 = 16, kXWarp0 = 20, kProducerWarp = 24, kMmaWarp = 25;
constexpr uint32_t kTmemCols = 512;
// TMEM columns. M accumulator [0, 128) (lanes: k_in). Full mode: D_S buffers [128, 256) and
// [256, 384) (lanes: state row), D_O [384, 512) (lanes: token rows 0-63 = outputs, 64-127 =
// W'' S^T). Map mode: D_B [128, 256); T state, fp32, also the accumulator of T (-M) [256, 384)
// (lanes: key row); 16-bit S and T as MMA A operands [384, 448) and [448, 512) (lane = row,
// two elements per column).
constexpr uint32_t kColM = 0, kColS0 = 128, kColS1 = 256, kColO = 384, kColTS = 256, kColAS = 384, kColAT = 448;

enum Mode : int { kFull = 0, kMap = 1 };

// Shared memory (offsets from a 1024-byte aligned base). Every 16-bit tile is made of
// 128-byte swizzled blocks of [rows][64 columns].
struct Smem {
  // full-mode ring stage: per 64-column block b of the key dimension, Q (Q~ in place) rows
  // then W'' rows, so that [Q~; W''] is one 128-row operand; then U'' (U'' in place), K
  // (K~ in place), P'', gate rows
  static constexpr uint32_t fQ = 0, fW = 8192, fQW_BLK = 16384, fU = 32768, fK = 49152, fP = 65536, fF = 73728;
  static constexpr uint32_t fSTAGE = 74752;
  // map-mode ring stage: W'', U'', K (K~ in place), gate rows
  static constexpr uint32_t mW = 0, mU = 16384, mK = 32768, mF = 49152;
  static constexpr uint32_t mSTAGE = 50176;
  static constexpr uint32_t MB = 151552;       // -M as B operand: [k_in][k_out], 2 column blocks of 16 KB
  static constexpr uint32_t MB1 = 2 * mSTAGE;  // map mode: second -M buffer (odd chunks), after the ring
  static constexpr uint32_t SB = MB + 32768;   // 16-bit S (or B): [row][k], 2 column blocks of 16 KB
  static constexpr uint32_t BAR = SB + 32768;
  static constexpr uint32_t bytes = BAR + 256;
  static constexpr uint32_t alloc = bytes + 1024;
  // gate rows: g [64] | 1/|q| [64] | ks [64]
  static constexpr uint32_t FG = 0, FRQ = 256, FKS = 512;
  static constexpr uint32_t tx_full = 4 * 16384 + 8192 + 3 * 256;
  static constexpr uint32_t tx_map = 3 * 16384 + 2 * 256;
  static_assert(alloc <= 232448, "shared memory per CTA");
  static_assert(2 * fSTAGE <= MB && MB1 + 32768 <= MB, "ring below the fixed tiles");
  static_assert(fSTAGE % 1024 == 0 && mSTAGE % 1024 == 0 && MB % 1024 == 0 && MB1 % 1024 == 0, "1 KB aligned tiles");
};

// Barrier indices (mbarriers at Smem::BAR).
enum Bar : int {
  kFull0 = 0,        // [2] ring stage loaded
  kEmpty0 = 2,       // [2] ring stage free (MMA commit)
  kKtReady0 = 4,     // [2] K~ formed in the stage
  kQReady0 = 6,      // [2] Q~ formed in the stage
  kMFull = 8,        // M accumulated
  kMConv = 10,       // -M written as B operand; M accumulator free
  kMbFree = 11,      // chain products done with the -M operand (map mode: buffer 0)
  kChainDone0 = 12,  // [2] D_S buffer complete
  kChainTDone = 14,  // D_T complete (map mode)
  kOutDone = 15,     // [Q~; W''] S^T complete
  kSReady = 16,      // 16-bit S (or B) copy written, D_S read
  kTReady = 17,      // 16-bit T copy written, D_T read (map mode)
  kUtReady = 18,     // U'' formed in place
  kPuDone = 19,      // output rows complete
  kOFree = 20,       // output rows read
  kMbFree1 = 21,     // map mode: chain products done with -M buffer 1
  kNumBars = 22
};
constexpr int kEcRing = 4;   // exp(g_C) of the last chunks, written by the prep warps
constexpr int kL2Ahead = 3;  // chunks between an L2 prefetch and the load into shared memory

struct Job {
  int mode;
  int seq, hv;
  int c0, c1;         // chunk range [c0, c1) within the sequence
  const float* init;  // [V][K] start state (full mode)
  float* fin;         // [V][K] final state (full mode) or B of the map, or nullptr
  float* fin_t;       // [K][K] T of the map (map mode)
};

// CTAs [0, B*HV): segment 0 of a chain in full mode; then one CTA per (chain, middle segment
// 1 .. ns-2) builds that segment's map. Returns false if this CTA has no work.
__device__ bool decode_job(const Params& p, int nseg, Job& job) {
  const int B = p.B, HV = p.HV;
  const int64_t per_head = (int64_t)D * D;
  int bid = blockIdx.x;
  job.init = nullptr;
  job.fin = nullptr;
  job.fin_t = nullptr;
  int ns = 1;
  if (bid < B * HV) {
    job.seq = p.order[bid / HV];
    job.hv = bid % HV;
    const int n = p.seq_chunk_off[job.seq + 1] - p.seq_chunk_off[job.seq];
    float* pool = p.state_pool + (p.cache_indices[job.seq] * HV + job.hv) * per_head;
    job.mode = kFull;
    job.init = pool;
    seg_range(n, nseg, p.seg_r16, 0, job.c0, job.c1, ns);
    job.fin = ns > 1 ? p.seg_state + (((int64_t)job.seq * HV + job.hv) * nseg + 1) * per_head : pool;
    return job.c1 > job.c0;
  }
  if (nseg < 3) return false;
  bid -= B * HV;
  const int seg = 1 + bid % (nseg - 2);
  const int rest = bid / (nseg - 2);
  job.seq = p.order[rest / HV];
  job.hv = rest % HV;
  const int n = p.seq_chunk_off[job.seq + 1] - p.seq_chunk_off[job.seq];
  seg_range(n, nseg, p.seg_r16, seg, job.c0, job.c1, ns);
  if (seg >= ns - 1) return false;
  job.mode = kMap;
  float* m = p.seg_map + (((int64_t)job.seq * HV + job.hv) * nseg + seg) * 2 * per_head;
  job.fin = m;
  job.fin_t = m + per_head;
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

// Scales the 8 16-bit elements of a 16-byte chunk by f (in place).
template <typename E>
__device__ __forceinline__ void scale_chunk(unsigned char* p, float f) {
  uint4 v = *reinterpret_cast<const uint4*>(p);
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 x = ElemT<E>::unpack(w[u]);
    w[u] = ElemT<E>::pack(x.x * f, x.y * f);
  }
  *reinterpret_cast<uint4*>(p) = v;
}

template <typename E>
__global__ void __launch_bounds__(kThreads, 1)
    affine_scan_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_u,
                       const __grid_constant__ CUtensorMap tm_p, const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k, Params p, int nseg) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  if (p.status[0] != GDN_OK) return;
  Job job;
  if (!decode_job(p, nseg, job)) return;  // uniform over the CTA
  const bool full = job.mode == kFull;
  const int hv = job.hv;
  const int h = hv / (p.HV / p.H);
  const int cb = p.seq_chunk_off[job.seq];
  const int nc = job.c1 - job.c0;
  const int nsb = full ? 2 : 1;  // D_S buffers
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // ring layout of this mode
  const uint32_t STG = full ? Smem::fSTAGE : Smem::mSTAGE;
  const uint32_t oW = full ? Smem::fW : Smem::mW, oU = full ? Smem::fU : Smem::mU;
  const uint32_t oK = full ? Smem::fK : Smem::mK, oF = full ? Smem::fF : Smem::mF;
  const uint32_t wblk = full ? Smem::fQW_BLK : 8192;  // distance between the 64-column blocks of W''

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* fail = reinterpret_cast<volatile int*>(tslot + 1);
  float* ec = reinterpret_cast<float*>(tslot + 2);  // [kEcRing]

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bars[kFull0 + s], 1);
      tc::mbar_init(&bars[kEmpty0 + s], 1);
      tc::mbar_init(&bars[kKtReady0 + s], 4);
      tc::mbar_init(&bars[kQReady0 + s], 4);
      tc::mbar_init(&bars[kChainDone0 + s], 1);
    }
    tc::mbar_init(&bars[kMFull], 1);
    tc::mbar_init(&bars[kMConv], 4);
    tc::mbar_init(&bars[kMbFree], 1);
    tc::mbar_init(&bars[kMbFree1], 1);
    tc::mbar_init(&bars[kChainTDone], 1);
    tc::mbar_init(&bars[kOutDone], 1);
    tc::mbar_init(&bars[kSReady], kChainWarps);
    tc::mbar_init(&bars[kTReady], 4);
    tc::mbar_init(&bars[kUtReady], 2);
    tc::mbar_init(&bars[kPuDone], 1);
    tc::mbar_init(&bars[kOFree], 2);
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
  // bounded wait with one outcome per warp (the warp then stays converged)
  auto wait_warp = [&](int b, uint32_t parity) {
    const bool ok = wait_or_fail(&bars[b], parity, fail, p.wait_budget);
    return __all_sync(0xffffffffu, ok);
  };
  // a warp's shared-memory writes (and TMEM reads) are complete: arrive on barrier b
  auto signal = [&](int b) {
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bars[b]);
  };
  auto stage = [&](int c) { return smem + (c & 1) * STG; };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer: TMA
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int c = 0; c < nc && ok && p.stall != kStallAffineScan; ++c) {
        const int s = c & 1;
        if (c >= 2 && !(ok = wait_or_fail(&bars[kEmpty0 + s], ((c >> 1) - 1) & 1, fail, p.wait_budget))) break;
        const int j = cb + job.c0 + c;
        const int4 ct = p.chunk_tab[j];
        const int64_t jh = (int64_t)j * p.HV + hv;
        const int64_t jq = (int64_t)j * p.H + h;
        unsigned char* st = stage(c);
        uint64_t* fb = &bars[kFull0 + s];
        tc::mbar_arrive_expect_tx(fb, full ? Smem::tx_full : Smem::tx_map);
        for (int b = 0; b < 2; ++b) {
          tc::tma_load_2d(st + oW + b * wblk, &tm_w, 64 * b, (int)(jh * C), fb);
          tc::tma_load_2d(st + oU + b * 8192, &tm_u, 64 * b, (int)(jh * C), fb);
          tc::tma_load_3d(st + oK + b * 8192, &tm_k, 64 * b, h, ct.y, fb);
          if (full) tc::tma_load_3d(st + Smem::fQ + b * Smem::fQW_BLK, &tm_q, 64 * b, h, ct.y, fb);
        }
        if (full) tc::tma_load_2d(st + Smem::fP, &tm_p, 0, (int)(jh * C), fb);
        tc::bulk_load(st + oF + Smem::FG, p.g + jh * C, 256, fb);
        if (full) tc::bulk_load(st + oF + Smem::FRQ, p.rq + jq * C, 256, fb);
        tc::bulk_load(st + oF + Smem::FKS, p.ks + jh * C, 256, fb);
        issued = c + 1;
        if (c + kL2Ahead < nc) {  // warm L2 with a later chunk's tiles: its load then hits L2
          const int j2 = j + kL2Ahead;
          const int64_t jh2 = (int64_t)j2 * p.HV + hv;
          const int t2 = p.chunk_tab[j2].y;
          for (int b = 0; b < 2; ++b) {
            tc::tma_prefetch_2d(&tm_w, 64 * b, (int)(jh2 * C));
            tc::tma_prefetch_2d(&tm_u, 64 * b, (int)(jh2 * C));
            tc::tma_prefetch_3d(&tm_k, 64 * b, h, t2);
            if (full) tc::tma_prefetch_3d(&tm_q, 64 * b, h, t2);
          }
          if (full) tc::tma_prefetch_2d(&tm_p, 0, (int)(jh2 * C));
        }
      }
      if (!ok) report();
      // no copy outlives the CTA: the last loads of each buffer have landed (bounded)
      for (int c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
        tc::mbar_wait(&bars[kFull0 + (c & 1)], (c >> 1) & 1, p.wait_budget);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer (one thread)
    if (lane == 0) {
      constexpr uint32_t fmt = ElemT<E>::fmt;
      constexpr uint32_t id_mb = tc::idesc_f16(128, 128, fmt, true, true);   // A, B MN-major
      constexpr uint32_t id_ch = tc::idesc_f16(128, 128, fmt, false, true);  // A K-major, B MN-major
      constexpr uint32_t id_o = tc::idesc_f16(128, 128, fmt, false, false);  // A, B K-major
      // Base descriptors; an operand at byte offset o from its base is base + (o >> 4).
      // MN-major operands of 128 rows/columns: two 64-element blocks LBO apart, 8-row groups
      // SBO = 1024 apart; K-major operands: 128-byte rows, 8-row groups 1024 apart.
      const uint64_t dW = tc::smem_desc(tc::saddr(smem + oW), wblk, 1024, tc::kSwizzle128B);
      const uint64_t dU = tc::smem_desc(tc::saddr(smem + oU), 8192, 1024, tc::kSwizzle128B);
      const uint64_t dK = tc::smem_desc(tc::saddr(smem + oK), 8192, 1024, tc::kSwizzle128B);
      const uint64_t dS = tc::smem_desc(tc::saddr(smem + Smem::SB), 16, 1024, tc::kSwizzle128B);
      const uint64_t dM = tc::smem_desc(tc::saddr(smem + Smem::MB), 16384, 1024, tc::kSwizzle128B);
      const uint64_t dM1 = tc::smem_desc(tc::saddr(smem + Smem::MB1), 16384, 1024, tc::kSwizzle128B);
      const uint64_t dQW = tc::smem_desc(tc::saddr(smem + Smem::fQ), 16, 1024, tc::kSwizzle128B);
      const uint64_t dP = tc::smem_desc(tc::saddr(smem + Smem::fP), 16, 1024, tc::kSwizzle128B);
      auto koff = [](int ks, uint32_t block) { return (uint32_t)(((ks >> 2) * block + (ks & 3) * 32) >> 4); };
      bool ok = true;
      auto W8 = [&](int b, uint32_t parity) {
        if (ok) ok = wait_or_fail(&bars[b], parity, fail, p.wait_budget);
        return ok;
      };
      auto so = [&](int c) { return (uint32_t)((c & 1) * STG) >> 4; };
      auto issue_m = [&](int c) {  // M_c = W''^T K~ into the M accumulator
        const uint32_t o = so(c);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_f16_ss(tmem + kColM, dW + o + (ks * 2048 >> 4), dK + o + (ks * 2048 >> 4), id_mb, ks > 0);
        tc::mma_commit(&bars[kMFull]);
      };
      auto issue_b = [&](int c) {  // B_c = U''^T K~ into D_S buffer c % nsb (the chain adds -S M)
        const uint32_t o = so(c);
        const uint32_t dcol = (c % nsb) ? kColS1 : kColS0;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_f16_ss(tmem + dcol, dU + o + (ks * 2048 >> 4), dK + o + (ks * 2048 >> 4), id_mb, ks > 0);
      };
      W8(kFull0, 0);
      W8(kKtReady0, 0);
      if (ok) {
        tc::fence_after_sync();
        issue_m(0);
        issue_b(0);
        if (!full) tc::mma_commit(&bars[kEmpty0]);  // map mode: the stage is done once M, B are formed
      }
      for (int c = 0; c < nc && ok; ++c) {
        const int s = c & 1;
        const int buf = c % nsb;
        // chain product: D_S[buf] += S (-M); map mode also T += T (-M)
        W8(kMConv, c & 1);
        W8(kSReady, c & 1);
        if (!full) W8(kTReady, c & 1);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t dcol = buf ? kColS1 : kColS0;
        if (full) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_f16_ss(tmem + dcol, dS + koff(ks, 16384), dM + (ks * 2048 >> 4), id_ch, 1);
          tc::mma_commit(&bars[kChainDone0 + buf]);
          tc::mma_commit(&bars[kMbFree]);
          // D_O = [Q~; W''] S^T
          W8(kQReady0 + s, (c >> 1) & 1);
          if (c >= 1) W8(kOFree, (c - 1) & 1);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_f16_ss(tmem + kColO, dQW + so(c) + koff(ks, Smem::fQW_BLK), dS + koff(ks, 16384), id_o, ks > 0);
          tc::mma_commit(&bars[kOutDone]);
          if (c + 1 < nc) {  // the next chunk's M (its accumulator is free) and B
            W8(kFull0 + ((c + 1) & 1), ((c + 1) >> 1) & 1);
            W8(kKtReady0 + ((c + 1) & 1), ((c + 1) >> 1) & 1);
            if (!ok) break;
            tc::fence_after_sync();
            issue_m(c + 1);
            issue_b(c + 1);
          }
        } else {
          // A operands from TMEM (8 columns = 16 keys per MMA), -M from buffer c & 1. M of the next
          // chunk goes between the two chain products, so that its conversion (into the other -M
          // buffer) overlaps the T product.
          const uint64_t dMc = (c & 1) ? dM1 : dM;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_f16_ts(tmem + dcol, tmem + kColAS + 8 * ks, dMc + (ks * 2048 >> 4), id_ch, 1);
          tc::mma_commit(&bars[kChainDone0 + buf]);
          if (c + 1 < nc) {
            W8(kFull0 + ((c + 1) & 1), ((c + 1) >> 1) & 1);
            W8(kKtReady0 + ((c + 1) & 1), ((c + 1) >> 1) & 1);
            if (!ok) break;
            tc::fence_after_sync();
            issue_m(c + 1);
          }
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // T state (pre-scaled by exp(g_C)) += T (-M)
            tc::mma_f16_ts(tmem + kColTS, tmem + kColAT + 8 * ks, dMc + (ks * 2048 >> 4), id_ch, 1);
          tc::mma_commit(&bars[kChainTDone]);
          tc::mma_commit(&bars[(c & 1) ? kMbFree1 : kMbFree]);
          if (c + 1 < nc) {
            if (!W8(kSReady, (c + 1) & 1)) break;  // single D_B buffer: the chain warps have read it
            issue_b(c + 1);
            tc::mma_commit(&bars[kEmpty0 + ((c + 1) & 1)]);  // the stage is done once M, B are formed
          }
        }
        if (full) {
          // D_O[0:64] += P'' U''
          W8(kUtReady, c & 1);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_f16_ss(tmem + kColO, dP + so(c) + (ks * 32 >> 4), dU + so(c) + (ks * 2048 >> 4), id_ch, 1);
          tc::mma_commit(&bars[kPuDone]);
          tc::mma_commit(&bars[kEmpty0 + s]);
        }
      }
      if (!ok) report();
    }
    __syncwarp();
  } else if (warp < kPrepWarp0) {
    // ------------------------------------------------------------------ chain: S <- exp(g_C) S + D_S
    const int quarter = warp & 3, part = warp >> 2;
    const int row = 32 * quarter + lane;  // state row (TMEM lane)
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    // this thread's 32 columns 32 part .. 32 part + 31: chunks 4 (part & 1) .. +3 of 64-column block part >> 1
    unsigned char* sblk = smem + Smem::SB + (part >> 1) * 16384;
    const int ch0 = 4 * (part & 1);
    float S_[32];
    auto write_sb = [&]() {
      if (full) {  // shared memory (B operand of D_O, A operand of the chain product)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) w[u] = ElemT<E>::pack(S_[8 * q + 2 * u], S_[8 * q + 2 * u + 1]);
          *reinterpret_cast<uint4*>(sblk + tc::sw128_offset(row, ch0 + q)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {  // TMEM A operand: keys 32 part .. 32 part + 31 in columns 16 part .. 16 part + 15
        uint32_t w[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) w[u] = ElemT<E>::pack(S_[2 * u], S_[2 * u + 1]);
        tc::tmem_st16(tmem + lane_base + kColAS + 16 * part, w);
        tc::tmem_wait_st();
      }
    };
    if (full) {
      const float4* src = reinterpret_cast<const float4*>(job.init + (int64_t)row * D + 32 * part);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = src[u];
        S_[4 * u] = x.x;
        S_[4 * u + 1] = x.y;
        S_[4 * u + 2] = x.z;
        S_[4 * u + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < 32; ++u) S_[u] = 0.f;
    }
    write_sb();
    signal(kSReady);
    bool failed = false;
    for (int c = 0; c < nc; ++c) {
      const int buf = c % nsb;
      if (!wait_warp(kMConv, c & 1) || !wait_warp(kChainDone0 + buf, (c / nsb) & 1) ||
          (full && !wait_warp(kOutDone, c & 1))) {
        failed = true;
        break;
      }
      tc::fence_after_sync();
      const float eC = ec[c % kEcRing];
      const uint32_t dcol = (buf ? kColS1 : kColS0) + 32 * part;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t rr[16];
        tc::tmem_ld16(tmem + lane_base + dcol + 16 * g, rr);
        tc::tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 16; ++u) S_[16 * g + u] = fmaf(eC, S_[16 * g + u], __uint_as_float(rr[u]));
      }
      write_sb();
      signal(kSReady);
    }
    if (failed) report();
    if (!failed && job.fin) {
      float4* dst = reinterpret_cast<float4*>(job.fin + (int64_t)row * D + 32 * part);
#pragma unroll
      for (int u = 0; u < 8; ++u) dst[u] = make_float4(S_[4 * u], S_[4 * u + 1], S_[4 * u + 2], S_[4 * u + 3]);
    }
  } else if (warp < kXWarp0) {
    // ------------------------------------------------------------------ prep: K~, Q~ in place; -M
    const int quarter = warp & 3;
    const int pt = tid - 32 * kPrepWarp0;  // 0..127
    const int r = pt & 63, blk = pt >> 6;  // tile row and 64-column block of this thread
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    const int kin = 32 * quarter + lane;   // M accumulator row of this thread
    auto form_kt = [&](int c) {  // K~ = diag(ks) K in place (exact: ks is a power of two, or 0 on padded rows)
      unsigned char* st = stage(c);
      const float* F = reinterpret_cast<const float*>(st + oF);
      const float f = F[Smem::FKS / 4 + r];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) scale_chunk<E>(st + oK + blk * 8192 + tc::sw128_offset(r, ch), f);
    };
    // exp(g_C) of chunk c into the gate ring; written before -M of chunk c - 1 is signalled, so
    // that every role that waits for that signal may read it
    auto put_ec = [&](int c) {
      if (pt == 0) ec[c % kEcRing] = expf(reinterpret_cast<const float*>(stage(c) + oF)[Smem::FG / 4 + C - 1]);
    };
    auto form_qt = [&](int c) {  // Q~ = diag(exp(g)/|q|) Q
      unsigned char* st = stage(c);
      const float* F = reinterpret_cast<const float*>(st + oF);
      const float f = expf(F[Smem::FG / 4 + r]) * F[Smem::FRQ / 4 + r];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) scale_chunk<E>(st + Smem::fQ + blk * Smem::fQW_BLK + tc::sw128_offset(r, ch), f);
    };
    bool failed = false;
    if (!wait_warp(kFull0, 0)) {
      failed = true;
    } else {
      put_ec(0);
      form_kt(0);
      signal(kKtReady0);
      if (full) {
        form_qt(0);
        signal(kQReady0);
      }
    }
    for (int c = 0; c < nc && !failed; ++c) {
      // -M of chunk c goes to buffer MB (full mode: the only one; map mode: even chunks) or MB1,
      // once the chain products of the buffer's previous chunk are done
      const bool odd = !full && (c & 1);
      const bool free_ok = full ? (c < 1 || wait_warp(kMbFree, (c - 1) & 1))
                                : (c < 2 || wait_warp(odd ? kMbFree1 : kMbFree, ((c - 2) >> 1) & 1));
      if (!wait_warp(kMFull, c & 1) || !free_ok) {
        failed = true;
        break;
      }
      // map mode: the T chain reads exp(g_C) of chunk c + 1 once -M of chunk c is signalled (its
      // stage is loaded early, as map-mode stages are released once M and B are formed)
      if (!full && c + 1 < nc) {
        if (!wait_warp(kFull0 + ((c + 1) & 1), ((c + 1) >> 1) & 1)) {
          failed = true;
          break;
        }
        put_ec(c + 1);
      }
      tc::fence_after_sync();
      // -M (row kin, 128 columns) as the B operand [k_in][k_out], 16 columns at a time
#pragma unroll 2
      for (int g = 0; g < 8; ++g) {
        uint32_t rr[16];
        tc::tmem_ld16(tmem + lane_base + kColM + 16 * g, rr);
        tc::tmem_wait_ld();
        unsigned char* dst = smem + (odd ? Smem::MB1 : Smem::MB) + (g >> 2) * 16384;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {  // 16-byte chunk 2 (g & 3) + q2 of the 128-byte row
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            w[u] = ElemT<E>::pack(-__uint_as_float(rr[8 * q2 + 2 * u]), -__uint_as_float(rr[8 * q2 + 2 * u + 1]));
          *reinterpret_cast<uint4*>(dst + tc::sw128_offset(kin, 2 * (g & 3) + q2)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      signal(kMConv);
      if (c + 1 < nc) {
        if (full) {  // full mode: the chains read it only after -M of chunk c + 1
          if (!wait_warp(kFull0 + ((c + 1) & 1), ((c + 1) >> 1) & 1)) {
            failed = true;
            break;
          }
          put_ec(c + 1);
        }
        form_kt(c + 1);
        signal(kKtReady0 + ((c + 1) & 1));
        if (full) {
          form_qt(c + 1);
          signal(kQReady0 + ((c + 1) & 1));
        }
      }
    }
    if (failed) report();
  } else if (warp < kProducerWarp) {
    const int quarter = warp & 3;
    const int lrow = 32 * quarter + lane;  // TMEM lane of this thread
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    bool failed = false;
    if (full && quarter < 2) {
      // ---------------------------------------------------------------- output rows (lanes 0-63)
      const int t = lrow;
      for (int c = 0; c < nc; ++c) {
        const int4 ct = p.chunk_tab[cb + job.c0 + c];
        if (!wait_warp(kPuDone, c & 1)) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<E*>(p.out) + (((int64_t)ct.y + t) * p.HV + hv) * D);
#pragma unroll
        for (int g2 = 0; g2 < 4; ++g2) {
          uint32_t rr[2][16];
          tc::tmem_ld16(tmem + lane_base + kColO + 32 * g2, rr[0]);
          tc::tmem_ld16(tmem + lane_base + kColO + 32 * g2 + 16, rr[1]);
          tc::tmem_wait_ld();
          if (t < ct.z) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int e = 8 * q4 + 2 * u;
                w[u] = ElemT<E>::pack(p.scale * __uint_as_float(rr[e >> 4][e & 15]),
                                      p.scale * __uint_as_float(rr[(e + 1) >> 4][(e + 1) & 15]));
              }
              orow[4 * g2 + q4] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars[kOFree]);
      }
    } else if (full) {
      // ---------------------------------------------------------------- U'' = U'' - W'' S^T in place (lanes 64-127)
      const int t = lrow - 64;
      for (int c = 0; c < nc; ++c) {
        const int s = c & 1;
        if (!wait_warp(kOutDone, c & 1) || !wait_warp(kFull0 + s, (c >> 1) & 1)) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        unsigned char* urow = stage(c) + oU;
#pragma unroll
        for (int g2 = 0; g2 < 4; ++g2) {  // value columns 32 g2 .. 32 g2 + 31
          uint32_t rr[2][16];
          tc::tmem_ld16(tmem + lane_base + kColO + 32 * g2, rr[0]);
          tc::tmem_ld16(tmem + lane_base + kColO + 32 * g2 + 16, rr[1]);
          tc::tmem_wait_ld();
          unsigned char* blk = urow + (g2 >> 1) * 8192;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4* ptr = reinterpret_cast<uint4*>(blk + tc::sw128_offset(t, (g2 & 1) * 4 + q4));
            uint4 x = *ptr;
            uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int e = 8 * q4 + 2 * u;
              const float2 f = ElemT<E>::unpack(w[u]);
              w[u] = ElemT<E>::pack(f.x - __uint_as_float(rr[e >> 4][e & 15]), f.y - __uint_as_float(rr[(e + 1) >> 4][(e + 1) & 15]));
            }
            *ptr = x;
          }
        }
        signal(kUtReady);
      }
    } else {
      // ---------------------------------------------------------------- T chain (map mode)
      // T (fp32, TMEM) holds exp(g_C) T before each chain product, which adds T (-M) in place; the
      // 16-bit copy of T is the product's A operand (TMEM). T starts as the identity.
      const int v = lrow;  // key row of T
      auto put_row = [&](int g, const uint32_t (&x)[16], float f) {  // columns 16 g .. 16 g + 15
        uint32_t w[8], y[16];
#pragma unroll
        for (int u = 0; u < 8; ++u) w[u] = ElemT<E>::pack(__uint_as_float(x[2 * u]), __uint_as_float(x[2 * u + 1]));
#pragma unroll
        for (int u = 0; u < 16; ++u) y[u] = __float_as_uint(f * __uint_as_float(x[u]));
        tc::tmem_st8(tmem + lane_base + kColAT + 8 * g, w);
        tc::tmem_st16(tmem + lane_base + kColTS + 16 * g, y);
      };
      // exp(g_C) of chunk 0 is in the gate ring once -M of chunk 0 is
      if (!wait_warp(kMConv, 0)) failed = true;
      if (!failed) {
        const float e0 = ec[0];
#pragma unroll 2
        for (int g = 0; g < 8; ++g) {
          uint32_t x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = __float_as_uint((16 * g + i == v) ? 1.f : 0.f);
          put_row(g, x, e0);
        }
        tc::tmem_wait_st();
        signal(kTReady);
      }
      for (int c = 0; c < nc && !failed; ++c) {
        // kMConv(c) also orders the prep warps' exp(g_C) of chunk c + 1 before this read
        if (!wait_warp(kMConv, c & 1) || !wait_warp(kChainTDone, c & 1)) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        if (c + 1 == nc) break;  // the final T stays unscaled in TMEM
        const float eN = ec[(c + 1) % kEcRing];
#pragma unroll 2
        for (int g = 0; g < 8; ++g) {
          uint32_t x[16];
          tc::tmem_ld16(tmem + lane_base + kColTS + 16 * g, x);
          tc::tmem_wait_ld();
          put_row(g, x, eN);
        }
        tc::tmem_wait_st();
        signal(kTReady);
      }
      if (!failed && job.fin_t) {
        float4* dst = reinterpret_cast<float4*>(job.fin_t + (int64_t)v * D);
#pragma unroll 2
        for (int g = 0; g < 8; ++g) {
          uint32_t b[16];
          tc::tmem_ld16(tmem + lane_base + kColTS + 16 * g, b);
          tc::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[4 * g + q] = make_float4(__uint_as_float(b[4 * q]), __uint_as_float(b[4 * q + 1]),
                                         __uint_as_float(b[4 * q + 2]), __uint_as_float(b[4 * q + 3]));
        }
      }
    }
    if (failed) report();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename E>
cudaError_t launch_t(const Params& p, cudaStream_t s) {
  const bool h16 = p.fp16 != 0;
  const int64_t rows = p.max_chunks * p.HV * C;
  CUtensorMap mw, mu, mp, mq, mk;
  if (!make_2d_tile_map(&mw, p.W, D, rows, 64, C, true, h16) || !make_2d_tile_map(&mu, p.U, D, rows, 64, C, true, h16) ||
      !make_2d_tile_map(&mp, p.P, C, rows, 64, C, true, h16) || !make_token_tile_map(&mq, p.q, D, p.H, p.T, C, h16) ||
      !make_token_tile_map(&mk, p.k, D, p.H, p.T, C, h16))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(affine_scan_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem::alloc);
  if (e != cudaSuccess) return e;
  const int64_t chains = (int64_t)p.B * p.HV;
  affine_scan_kernel<E><<<(unsigned)(chains * (p.nseg - 1)), kThreads, Smem::alloc, s>>>(mw, mu, mp, mq, mk, p, p.nseg);
  return cudaGetLastError();
}

}  // namespace

// First pass of a segmented scan for K = V = 128: segment 0 of every chain with outputs (its end
// state to the segment-state buffer) and the affine map (B, T) of each middle segment.
cudaError_t launch_affine_map_pass(const Params& p, cudaStream_t s) {
  if (p.nseg < 2) return cudaErrorInvalidValue;
  return p.fp16 ? launch_t<f16>(p, s) : launch_t<bf16>(p, s);
}

}  // namespace gdn
