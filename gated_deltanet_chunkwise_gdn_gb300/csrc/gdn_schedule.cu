// gdn_schedule.cu — K0: device-side validation and the varlen chunk schedule.
//
// Chunks restart at every sequence start and never span two sequences; the last
// chunk of a sequence may be partial (the sequential inter-chunk loop of the pymllm
// page "pymllm.layers.attention.gdn_chunkwise" runs ceil(T/C) steps per sequence).
// cu_seqlens and cache_indices follow that page's Parameters.
#include "gdn_common.cuh"

namespace gdn {

namespace {
constexpr int kThreads = 512;
constexpr int kOrderMaxBatch = 4096;  // above this, sequences keep their input order
}

__global__ void __launch_bounds__(kThreads) schedule_kernel(Params p, int C) {
  __shared__ int s_err;
  __shared__ int s_warp_sum[kThreads / 32];
  __shared__ int s_total;
  const int tid = threadIdx.x;
  const int B = p.B;
  if (tid == 0) s_err = 0;
  __syncthreads();

  // 1. validation: monotone cu_seqlens from 0 to T; slots in range and distinct.
  if (tid == 0 && (p.cu_seqlens[0] != 0 || p.cu_seqlens[B] != p.T)) atomicCAS(&s_err, 0, GDN_ERR_BAD_SEQLENS);
  for (int i = tid; i < B; i += kThreads) {
    if (p.cu_seqlens[i + 1] < p.cu_seqlens[i]) atomicCAS(&s_err, 0, GDN_ERR_BAD_SEQLENS);
    const int64_t slot = p.cache_indices[i];
    if (slot < 0 || slot >= p.pool_size) atomicCAS(&s_err, 0, GDN_ERR_BAD_INDEX);
    for (int j = 0; j < i; ++j)
      if (p.cache_indices[j] == slot) {
        atomicCAS(&s_err, 0, GDN_ERR_BAD_INDEX);
        break;
      }
  }
  __syncthreads();
  if (s_err != 0) {
    if (tid == 0) {
      p.status[0] = s_err;
      p.status[1] = 0;
    }
    return;
  }

  // 2. chunk offsets: each thread owns a contiguous run of sequences.
  const int per = (B + kThreads - 1) / kThreads;
  const int s0 = min(B, tid * per), s1 = min(B, s0 + per);
  int local = 0;
  for (int s = s0; s < s1; ++s) {
    const int64_t len = p.cu_seqlens[s + 1] - p.cu_seqlens[s];
    local += (int)((len + C - 1) / C);
  }
  // block exclusive scan of `local`
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int x = lane < kThreads / 32 ? s_warp_sum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane < kThreads / 32) s_warp_sum[lane] = x;  // inclusive over warps
    if (lane == kThreads / 32 - 1) s_total = x;
  }
  __syncthreads();
  int run = (warp > 0 ? s_warp_sum[warp - 1] : 0) + incl - local;
  for (int s = s0; s < s1; ++s) {
    p.seq_chunk_off[s] = run;
    const int64_t len = p.cu_seqlens[s + 1] - p.cu_seqlens[s];
    run += (int)((len + C - 1) / C);
  }
  if (tid == 0) p.seq_chunk_off[B] = s_total;
  __syncthreads();

  // 3. chunk table: chunk j -> (sequence, first token, length, index in sequence).
  const int n_chunks = s_total;
  for (int j = tid; j < n_chunks; j += kThreads) {
    int lo = 0, hi = B - 1;  // last s with seq_chunk_off[s] <= j (skips empty sequences)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.seq_chunk_off[mid] <= j) lo = mid; else hi = mid - 1;
    }
    const int c = j - p.seq_chunk_off[lo];
    const int64_t t0 = p.cu_seqlens[lo] + (int64_t)c * C;
    const int64_t len = min((int64_t)C, p.cu_seqlens[lo + 1] - t0);
    p.chunk_tab[j] = make_int4(lo, (int)t0, (int)len, c);
  }

  // 4. longest-first order of sequences (ties by index): the scan's chains start
  //    with the longest so the tail of the grid is short.
  for (int i = tid; i < B; i += kThreads) {
    if (B > kOrderMaxBatch) {
      p.order[i] = i;
      continue;
    }
    const int64_t li = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
    int rank = 0;
    for (int j = 0; j < B; ++j) {
      const int64_t lj = p.cu_seqlens[j + 1] - p.cu_seqlens[j];
      rank += (lj > li) || (lj == li && j < i);
    }
    p.order[rank] = i;
  }
  if (tid == 0) {
    p.status[1] = n_chunks;
    p.status[2] = 0;  // item counter of the intra kernel
    p.status[0] = GDN_OK;
  }
}

}  // namespace gdn
