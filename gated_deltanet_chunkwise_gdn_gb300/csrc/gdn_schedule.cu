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

// Sorts the n (a power of two, <= kScheduleSortMax) keys in shared memory ascending; every thread
// of the block takes part. Bitonic network: log2(n) (log2(n) + 1) / 2 passes of n / 2 exchanges.
__device__ void bitonic_sort(uint64_t* a, int n) {
  for (int k = 2; k <= n; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int l = i ^ j;
        if (l > i) {
          const uint64_t x = a[i], y = a[l];
          if ((x > y) == ((i & k) == 0)) {
            a[i] = y;
            a[l] = x;
          }
        }
      }
      __syncthreads();
    }
}

__host__ __device__ inline int pow2_at_least(int n) {
  int m = 1;
  while (m < n) m <<= 1;
  return m;
}
}  // namespace

size_t schedule_smem_bytes(int B) {
  return B <= kScheduleSortMax ? (size_t)pow2_at_least(B > 0 ? B : 1) * sizeof(uint64_t) : 0;
}

// pre_checked: the slots were already checked by the multi-block check (batches above
// kScheduleSortMax), which left GDN_OK or GDN_ERR_BAD_INDEX in the status word.
__global__ void __launch_bounds__(kThreads) schedule_kernel(Params p, int C, int pre_checked) {
  extern __shared__ uint64_t s_key[];  // pow2_at_least(B) sort keys (B <= kScheduleSortMax)
  __shared__ int s_err;
  __shared__ int s_warp_sum[kThreads / 32];
  __shared__ int s_total;
  const int tid = threadIdx.x;
  const int B = p.B;
  const bool sorted = B <= kScheduleSortMax;
  const int n2 = sorted ? pow2_at_least(B > 0 ? B : 1) : 0;
  if (tid == 0) s_err = pre_checked ? p.status[0] : 0;
  __syncthreads();

  // 1. validation: monotone cu_seqlens from 0 to T; slots in range and distinct (distinct: the
  //    sorted slots hold no two equal neighbours).
  if (tid == 0 && (p.cu_seqlens[0] != 0 || p.cu_seqlens[B] != p.T)) atomicCAS(&s_err, 0, GDN_ERR_BAD_SEQLENS);
  for (int i = tid; i < B; i += kThreads) {
    if (p.cu_seqlens[i + 1] < p.cu_seqlens[i]) atomicCAS(&s_err, 0, GDN_ERR_BAD_SEQLENS);
    const int64_t slot = p.cache_indices[i];
    if (slot < 0 || slot >= p.pool_size) atomicCAS(&s_err, 0, GDN_ERR_BAD_INDEX);
  }
  if (sorted) {
    for (int i = tid; i < n2; i += kThreads) s_key[i] = i < B ? (uint64_t)p.cache_indices[i] : ~0ull;
    __syncthreads();
    bitonic_sort(s_key, n2);
    for (int i = tid + 1; i < B; i += kThreads)
      if (s_key[i] == s_key[i - 1]) atomicCAS(&s_err, 0, GDN_ERR_BAD_INDEX);
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

  // 4. longest-first order of sequences (ties by index): the scan's chains start with the
  //    longest so the tail of the grid is short. Key: (INT32_MAX - length, index), sorted.
  if (sorted) {
    __syncthreads();
    for (int i = tid; i < n2; i += kThreads) {
      uint64_t key = ~0ull;
      if (i < B) {
        const int64_t len = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
        key = ((uint64_t)(INT32_MAX - len) << 32) | (uint32_t)i;
      }
      s_key[i] = key;
    }
    __syncthreads();
    bitonic_sort(s_key, n2);
    for (int r = tid; r < B; r += kThreads) p.order[r] = (int)(uint32_t)s_key[r];
  } else {
    for (int i = tid; i < B; i += kThreads) p.order[i] = i;
  }
  if (tid == 0) {
    p.status[1] = n_chunks;
    p.status[2] = 0;  // item counter of the intra kernel
    p.status[0] = GDN_OK;
  }
}

}  // namespace gdn
