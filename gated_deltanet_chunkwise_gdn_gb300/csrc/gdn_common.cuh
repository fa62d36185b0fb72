// gdn_common.cuh — shared definitions of the GB300 chunkwise GDN prefill kernels.
//
// Notation (per chunk of C tokens of one sequence, one value head):
//   g_i      = sum_{j<=i in chunk} log alpha_j          (chunk-local log decay, <= 0)
//   Gamma    = exp(g_mu - g_nu) for mu >= nu           ("Simple math to speed up GDN
//                                                       prefill", section "Reminder")
//   M        = I + tril(diag(beta) K^ K^^T, -1)
//   A        = (Gamma . M^{-1}) diag(beta) = N^{-1} B   (section "Save one invert")
//   W<-      = A diag(exp(g)) K^                       (C x K, decayed WY keys)
//   U~       = A V                                     (C x V, decayed WY values)
//   P        = Gamma . tril(Q^ K^^T)                   (C x C, causal intra-chunk scores)
// and the chunk step on the state S (V x K):
//   U   = U~ - W<- S^T
//   O   = diag(exp(g)) Q^ S^T + P U
//   S  <- exp(g_C) S + U^T diag(exp(g_C - g)) K^
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

using bf16 = __nv_bfloat16;
using f16 = __half;

constexpr float kNormEps = 1e-6f;  // q^ = q / sqrt(|q|^2 + eps)

// ----------------------------------------------------------------------------- workspace

// Offsets (bytes) of the workspace regions for one call. Every region starts on a
// 256-byte boundary.
struct WsLayout {
  size_t status;         // int32[64]: [0] status code, [1] number of chunks, [2] intra item counter
  size_t seq_chunk_off;  // int32[B+1]: first chunk of each sequence
  size_t order;          // int32[B]: sequences, longest first
  size_t chunk_tab;      // int4[max_chunks]: (seq, first token, length, chunk index in seq)
  size_t g;              // fp32[max_chunks][HV][C]: chunk-local cumulative log decay
  size_t beta;           // fp32[max_chunks][HV][C]: beta (0 on padded rows)
  size_t rq;             // fp32[max_chunks][H][C]: 1/|q| per row (0 on padded rows)
  size_t rk;             // fp32[max_chunks][H][C]: 1/|k| per row (0 on padded rows)
  size_t ks;             // fp32[max_chunks][HV][C]: power-of-two part of exp(g_C - g)/|k| (K = V = 128)
  size_t w;              // E[max_chunks][HV][C][K]: W<-   (E: the call's 16-bit element type)
  size_t u;              // E[max_chunks][HV][C][V]: U~
  size_t p;              // E[max_chunks][HV][C][C]: P
  size_t seg_state;      // fp32[B][HV][nseg][V][K]: start state of each segment (segmented scan)
  size_t seg_map;        // fp32[B][HV][nseg][2][K][K]: affine map (B, T) of each segment
  size_t total;
  int64_t max_chunks;
  int nseg;
};

// Segments per sequence for the scan: more than one only when there are too few
// (sequence, head, 64-row block) chains to fill the GPU and the sequences may be long.
// K = V = 128 (affine-transition scan): each pass runs ctas * (nseg - 1) CTAs, one per SM.
// Otherwise the first launch runs ctas * (1 + 2 (nseg - 2)) CTAs.
inline int choose_nseg(int64_t T, int B, int HV, int K, int V, int C) {
  const int64_t max_chunks = T / C;  // the longest sequence has at most this many chunks
  int best = 1;
  if (K == 128 && V == 128) {
    const int64_t ctas = (int64_t)B * HV;
    for (int n = 2; n <= 16; ++n)
      if (ctas * (n - 1) <= 148 && max_chunks >= 32 * n) best = n;
    return best;
  }
  const int64_t ctas = (int64_t)B * HV * (V / 64);
  for (int n = 2; n <= 8; ++n) {
    const int64_t grid1 = ctas * (1 + 2 * (n - 2));
    if (grid1 <= 148 && max_chunks >= 32 * n) best = n;
  }
  return best;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Chunk range [c0, c1) of segment `part` when a sequence of n chunks is cut into at most
// nseg segments for the segmented scan; ns = number of non-empty segments. Segment 0 is
// r16/16 times as long as the others: its CTA runs in full mode (outputs) alongside the map
// CTAs of the later segments, which do less work per chunk. The rest is split evenly.
__host__ __device__ inline void seg_range(int n, int nseg, int r16, int part, int& c0, int& c1, int& ns) {
  if (nseg <= 1 || n <= 0) {
    ns = n > 0 ? 1 : 0;
    c0 = part == 0 ? 0 : n;
    c1 = n;
    return;
  }
  const int den = (nseg - 1) * 16 + r16;
  int L0 = (int)(((int64_t)n * r16 + den - 1) / den);
  L0 = L0 < 1 ? 1 : (L0 > n ? n : L0);
  const int rest = n - L0;
  const int L1 = rest > 0 ? (rest + nseg - 2) / (nseg - 1) : 1;
  ns = 1 + (rest + L1 - 1) / L1;
  if (part == 0) {
    c0 = 0;
    c1 = L0;
  } else {
    c0 = L0 + (part - 1) * L1;
    c1 = c0 + L1;
    c0 = c0 < n ? c0 : n;
    c1 = c1 < n ? c1 : n;
  }
}

inline WsLayout make_layout(int64_t T, int B, int H, int HV, int K, int V, int C) {
  WsLayout L{};
  const int64_t mc = T / C + B + 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.max_chunks = mc;
  L.status = take(64 * sizeof(int32_t));
  L.seq_chunk_off = take((size_t)(B + 1) * sizeof(int32_t));
  L.order = take((size_t)(B > 0 ? B : 1) * sizeof(int32_t));
  L.chunk_tab = take((size_t)mc * sizeof(int4));
  L.g = take((size_t)mc * HV * C * sizeof(float));
  L.beta = take((size_t)mc * HV * C * sizeof(float));
  L.rq = take((size_t)mc * H * C * sizeof(float));
  L.rk = take((size_t)mc * H * C * sizeof(float));
  L.ks = take(K == 128 && V == 128 ? (size_t)mc * HV * C * sizeof(float) : 0);
  L.w = take((size_t)mc * HV * C * K * sizeof(bf16));
  L.u = take((size_t)mc * HV * C * V * sizeof(bf16));
  L.p = take((size_t)mc * HV * C * C * sizeof(bf16));
  L.nseg = choose_nseg(T, B, HV, K, V, C);
  const size_t per_head = (size_t)K * K * sizeof(float);
  L.seg_state = take(L.nseg > 1 ? (size_t)B * HV * L.nseg * per_head : 0);
  L.seg_map = take(L.nseg > 2 ? (size_t)B * HV * L.nseg * 2 * per_head : 0);
  L.total = off;
  return L;
}

// ----------------------------------------------------------------------------- launch params

struct Params {
  const bf16* q;  // 16-bit elements of the call's type (bf16 or fp16, see fp16)
  const bf16* k;
  const bf16* v;
  const float* a;
  const float* b;
  const float* A_log;
  const float* dt_bias;
  float* state_pool;
  const int64_t* cache_indices;
  const int64_t* cu_seqlens;
  bf16* out;
  int64_t T;
  int64_t pool_size;
  int B, H, HV;
  int nvb;  // value-dimension blocks per (sequence, value head) chain in the scan
  float scale;
  int64_t max_chunks;
  // workspace regions
  int32_t* status;
  int32_t* seq_chunk_off;
  int32_t* order;
  int4* chunk_tab;
  float* g;
  float* beta;
  float* rq;
  float* rk;
  float* ks;  // K = V = 128 only: ks[t] = 2^e with exp(g_C - g_t)/|k_t| = m_t 2^e, m_t in [0.5, 1)
  bf16* W;
  bf16* U;
  bf16* P;
  float* seg_state;
  float* seg_map;
  int nseg;  // segments per sequence in the scan (1: one pass over each whole sequence)
  int seg_r16;  // length of segment 0 relative to the others, in 16ths (see seg_range)
  int fp16;  // q, k, v, out (and the workspace factors) hold fp16 elements, else bf16
  long long wait_budget;  // clock cycles before a bounded mbarrier wait gives up
  int stall;  // test hook (gdn_test_set_stall): kernel whose CTAs withhold their tile loads, 0 = none
};

// Kernels a test can make stall (their producers issue no tile load, so every wait runs out).
enum StallKernel : int { kStallNone = 0, kStallIntra = 1, kStallScan = 2, kStallAffineScan = 3 };
constexpr long long kDefaultWaitBudget = 1ll << 31;  // about one second at the SM clock

// ----------------------------------------------------------------------------- device helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The 16-bit element type of a call (q, k, v, out, and every tensor-core operand derived
// from them: tcgen05 kind::f16 takes A and B of one type). fmt: the MMA operand format code.
template <typename E>
struct ElemT;
template <>
struct ElemT<bf16> {
  static constexpr uint32_t fmt = 1;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) { return pack_bf16(lo, hi); }
  static __device__ __forceinline__ float2 unpack(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
};
template <>
struct ElemT<f16> {
  static constexpr uint32_t fmt = 0;
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ float2 unpack(uint32_t w) { return __half22float2(*reinterpret_cast<const __half2*>(&w)); }
};
// (a, b) = hi + lo with hi and lo both in E: the pair carries about twice E's precision.
template <typename E>
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = ElemT<E>::pack(a, b);
  const float2 h = ElemT<E>::unpack(hi);
  lo = ElemT<E>::pack(a - h.x, b - h.y);
}

// Status word: the first error recorded wins.
__device__ __forceinline__ void set_status(int32_t* status, int code) {
  atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ----------------------------------------------------------------------------- kernels

// K0: validates cu_seqlens / cache_indices, builds the chunk table and the
// longest-first sequence order. One block, with schedule_smem_bytes(B) of dynamic shared
// memory. Batches up to kScheduleSortMax are checked and ordered by sorting in shared memory;
// larger ones keep their input order and have their slots checked beforehand by the
// multi-block check of the single-token step (pre_checked = 1).
constexpr int kScheduleSortMax = 8192;
size_t schedule_smem_bytes(int B);
__global__ void schedule_kernel(Params p, int C, int pre_checked);

// Host-side tensor maps (gdn_tma.cu): token tiles of a [T, heads, D] array of 16-bit
// elements (128-byte swizzled), and tiles of a row-major [rows, inner] array; fp16 selects
// fp16 elements, else bf16.
bool make_token_tile_map(CUtensorMap* map, const void* base, int D, int heads, int64_t T, int box_rows, bool fp16);
bool make_2d_tile_map(CUtensorMap* map, const void* base, int inner, int64_t rows, int box_inner, int box_rows,
                      bool swizzle128, bool fp16);

// Host-side launchers (one per translation unit, templated on head size).
cudaError_t launch_gates(const Params& p, int C, cudaStream_t s);
cudaError_t launch_intra(const Params& p, int D, int C, cudaStream_t s);
cudaError_t launch_scan(const Params& p, int D, int C, cudaStream_t s);

}  // namespace gdn
