// gdn_decode.cu — the single-token step (decode) of the Gated DeltaNet recurrence against the
// state pool: one new token per sequence, every value head, state read and written in place.
//
// For sequence b, value head hv (q/k head h = hv / (HV/H)), slot = cache_indices[b]:
//   q^ = q / sqrt(|q|^2 + eps),  k^ likewise
//   alpha = exp(-exp(A_log) softplus(a + dt_bias)),  beta = sigmoid(b)
//   S'  = alpha S + beta (v - alpha S k^) k^^T        (the transition of "Simple math to speed
//                                                      up GDN prefill", section "Reminder", for
//                                                      one token: S (alpha (I - beta k^ k^^T)) + beta v k^^T)
//   o   = scale S' q^ = scale (alpha S q^ + beta (v - alpha S k^) (k^ . q^))
// (the token reads the state after its own write: "nrm-training-kernels", section "General
// implementation", item 4). It is the one-token case of the chunkwise call with the same pool
// and index contract (pymllm page "pymllm.layers.attention.gdn_chunkwise", Parameters).
//
// The step is bound by HBM: each (sequence, value head) reads and writes its V x K fp32 state
// once (64 KB each way at K = V = 128) against 6 K V flops. Row v of S depends only on v_v and on
// the shared k^, q^, alpha, beta, so one CTA streams one state: each warp owns V/8 rows, loads
// them with coalesced 16-byte streaming loads (a warp reads whole 512-byte rows), forms both row
// dot products S_v k^ and S_v q^ from the same registers, and writes the updated rows back with
// streaming stores. Nothing is staged: the state never leaves registers. The update kernel is
// launched behind the slot check with programmatic dependent launch, so its launch and its
// input-only prologue (q^, k^, gates) overlap the check.
#include "gdn_decode.cuh"

namespace gdn {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kCheckTile = 256;
constexpr int kCheckOneBlock = 1024;  // batches up to this size are checked by one block

// Programmatic dependent launch: the check kernel lets the update kernel start (its grid is
// launched with programmatic stream serialization); the update kernel does its input-only
// prologue and then waits for the check kernel to finish before it reads the status.
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisite_grid() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float softplus_d(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

// cache_indices: every slot in [0, pool_size) and no slot twice, for B <= 1024 in one block of
// 32 ceil(B/32) threads: thread i compares its slot with those of every j < i (branch-free, to
// its warp's last index) and the block writes the outcome to the status word, GDN_OK included.
__global__ void __launch_bounds__(kCheckOneBlock) decode_check_one_block_kernel(const int64_t* idx, int B,
                                                                               int64_t pool_size, int32_t* status) {
  __shared__ int64_t s_idx[kCheckOneBlock];
  allow_dependent_launch();
  const int i = threadIdx.x;
  const int64_t slot = i < B ? idx[i] : -1;
  s_idx[i] = slot;
  __syncthreads();
  bool bad = i < B && (slot < 0 || slot >= pool_size);
  const int jend = min(B, (i | 31) + 1);  // the same bound for every lane of the warp
  int j = 0;
  for (; j + 4 <= jend; j += 4) {
#pragma unroll
    for (int u = 0; u < 4; ++u) bad |= (j + u < i) & (s_idx[j + u] == slot);
  }
  for (; j < jend; ++j) bad |= (j < i) & (s_idx[j] == slot);
  bad = i < B && bad;
  if (__syncthreads_or(bad)) {
    if (i == 0) *status = GDN_ERR_BAD_INDEX;
  } else if (i == 0) {
    *status = GDN_OK;
  }
}

// The same check for larger batches (the status word is zeroed before it, and only errors are
// recorded). Block x enumerates the lower triangle of 256 x 256 tiles of index pairs row by
// row: it compares the slots of tile ti with those of tile tj <= ti (pairs j < i); the diagonal
// tiles also check the range.
__global__ void __launch_bounds__(kCheckTile) decode_check_kernel(const int64_t* idx, int B, int64_t pool_size,
                                                                 int32_t* status) {
  __shared__ int64_t s_idx[kCheckTile];
  allow_dependent_launch();
  const int64_t x = blockIdx.x;
  int64_t ti = (int64_t)((sqrt(8.0 * (double)x + 1.0) - 1.0) * 0.5);
  while (ti > 0 && ti * (ti + 1) / 2 > x) --ti;
  while ((ti + 1) * (ti + 2) / 2 <= x) ++ti;
  const int64_t tj = x - ti * (ti + 1) / 2;
  const int tid = threadIdx.x;
  const int64_t j0 = tj * kCheckTile;
  if (j0 + tid < B) s_idx[tid] = idx[j0 + tid];
  __syncthreads();
  const int64_t i = ti * kCheckTile + tid;
  if (i >= B) return;
  const int64_t slot = idx[i];
  if (ti == tj && (slot < 0 || slot >= pool_size)) set_status(status, GDN_ERR_BAD_INDEX);
  const int n = ti == tj ? tid : (int)min((int64_t)kCheckTile, (int64_t)B - j0);
  for (int j = 0; j < n; ++j)
    if (s_idx[j] == slot) {
      set_status(status, GDN_ERR_BAD_INDEX);
      break;
    }
}

// Columns of a state row held by one lane: NPL = K / 32 of them, in runs of VEC = min(NPL, 4)
// consecutive columns, run c at column 32 VEC c + VEC lane (so each load instruction of a warp
// covers 32 VEC consecutive floats).
template <int K>
struct RowSplit {
  static constexpr int NPL = K / 32;
  static constexpr int VEC = NPL < 4 ? NPL : 4;
  static constexpr int RUNS = NPL / VEC;
  static __device__ __forceinline__ int col(int lane, int run) { return 32 * VEC * run + VEC * lane; }
};

template <int VEC>
__device__ __forceinline__ void load_row(float* dst, const float* src) {
  if constexpr (VEC == 4) {
    const float4 x = __ldcs(reinterpret_cast<const float4*>(src));
    dst[0] = x.x, dst[1] = x.y, dst[2] = x.z, dst[3] = x.w;
  } else {
    const float2 x = __ldcs(reinterpret_cast<const float2*>(src));
    dst[0] = x.x, dst[1] = x.y;
  }
}
template <int VEC>
__device__ __forceinline__ void store_row(float* dst, const float* src) {
  if constexpr (VEC == 4) {
    __stcs(reinterpret_cast<float4*>(dst), make_float4(src[0], src[1], src[2], src[3]));
  } else {
    __stcs(reinterpret_cast<float2*>(dst), make_float2(src[0], src[1]));
  }
}

// VEC consecutive 16-bit elements (VEC even) as floats.
template <typename E, int VEC>
__device__ __forceinline__ void load_elems(float* dst, const E* src) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(src);
#pragma unroll
  for (int u = 0; u < VEC / 2; ++u) {
    const float2 f = ElemT<E>::unpack(w[u]);
    dst[2 * u] = f.x;
    dst[2 * u + 1] = f.y;
  }
}

// One CTA per (sequence b, value head hv): blockIdx.x = b * HV + hv.
template <int K, int V, typename E>
__global__ void __launch_bounds__(kDecThreads, 2) decode_kernel(DecodeParams p) {
  using RS = RowSplit<K>;
  constexpr int NPL = RS::NPL, VEC = RS::VEC, RUNS = RS::RUNS;
  constexpr int RPW = V / kDecWarps;                          // state rows of one warp
  constexpr int RB = RPW * NPL <= 64 ? RPW : 64 / NPL;       // rows in registers at once
  static_assert(RPW <= 32 && RPW % RB == 0, "row split");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / p.HV, hv = blockIdx.x % p.HV;
  const int h = hv / (p.HV / p.H);
  const E* qrow = static_cast<const E*>(p.q) + ((int64_t)b * p.H + h) * K;
  const E* krow = static_cast<const E*>(p.k) + ((int64_t)b * p.H + h) * K;
  const int64_t bh = (int64_t)b * p.HV + hv;

  // q^, k^ on this lane's columns (every warp forms them: two 32-lane sums)
  float qh[NPL], kh[NPL];
#pragma unroll
  for (int r = 0; r < RUNS; ++r) {
    load_elems<E, VEC>(qh + VEC * r, qrow + RS::col(lane, r));
    load_elems<E, VEC>(kh + VEC * r, krow + RS::col(lane, r));
  }
  float sq = 0.f, sk = 0.f;
#pragma unroll
  for (int e = 0; e < NPL; ++e) {
    sq = fmaf(qh[e], qh[e], sq);
    sk = fmaf(kh[e], kh[e], sk);
  }
  const float rq = rsqrtf(warp_sum(sq) + kNormEps), rk = rsqrtf(warp_sum(sk) + kNormEps);
  float kq = 0.f;
#pragma unroll
  for (int e = 0; e < NPL; ++e) {
    qh[e] *= rq;
    kh[e] *= rk;
    kq = fmaf(kh[e], qh[e], kq);
  }
  kq = warp_sum(kq);
  const float alpha = expf(-expf(p.A_log[hv]) * softplus_d(p.a[bh] + p.dt_bias[hv]));
  const float beta = 1.f / (1.f + expf(-p.b[bh]));

  const int v0 = warp * RPW;                        // first row of this warp
  const E* vrow = static_cast<const E*>(p.v) + bh * V;
  float v_mine = 0.f, o_mine = 0.f;                  // lane l: v and o of row v0 + l (l < RPW)
  if (lane < RPW) v_mine = ElemT<E>::unpack((uint32_t)reinterpret_cast<const uint16_t*>(vrow)[v0 + lane]).x;

  wait_prerequisite_grid();  // the slot check has finished and its status is visible
  if (*p.status != GDN_OK) return;
  const int64_t slot = p.cache_indices[b];
  float* S = p.state_pool + (slot * p.HV + hv) * (int64_t)V * K;
#pragma unroll
  for (int r0 = 0; r0 < RPW; r0 += RB) {
    float s[RB][NPL];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
      for (int c = 0; c < RUNS; ++c) load_row<VEC>(s[r] + VEC * c, S + (int64_t)(v0 + r0 + r) * K + RS::col(lane, c));
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      float dk = 0.f, dq = 0.f;
#pragma unroll
      for (int e = 0; e < NPL; ++e) {
        dk = fmaf(s[r][e], kh[e], dk);
        dq = fmaf(s[r][e], qh[e], dq);
      }
      dk = warp_sum(dk);
      dq = warp_sum(dq);
      const float vv = __shfl_sync(0xffffffffu, v_mine, r0 + r);
      const float delta = beta * (vv - alpha * dk);  // beta (v - (alpha S) k^) for this row
#pragma unroll
      for (int e = 0; e < NPL; ++e) s[r][e] = fmaf(alpha, s[r][e], delta * kh[e]);
      const float o = p.scale * fmaf(alpha, dq, delta * kq);
      o_mine = lane == r0 + r ? o : o_mine;
#pragma unroll
      for (int c = 0; c < RUNS; ++c) store_row<VEC>(S + (int64_t)(v0 + r0 + r) * K + RS::col(lane, c), s[r] + VEC * c);
    }
  }
  if (lane < RPW) {
    const uint32_t w = ElemT<E>::pack(o_mine, 0.f);
    reinterpret_cast<uint16_t*>(static_cast<E*>(p.out) + bh * V)[v0 + lane] = (uint16_t)(w & 0xffffu);
  }
}

template <int D, typename E>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)p.B * p.HV));
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, D, E>, p);
}

}  // namespace

bool decode_check_needs_zeroed_status(int B) { return B > kCheckOneBlock; }

cudaError_t launch_decode_check(const DecodeParams& p, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  if (!decode_check_needs_zeroed_status(p.B)) {
    const unsigned threads = (unsigned)((p.B + 31) / 32 * 32);
    decode_check_one_block_kernel<<<1, threads, 0, s>>>(p.cache_indices, p.B, p.pool_size, p.status);
    return cudaGetLastError();
  }
  const int64_t nt = ((int64_t)p.B + kCheckTile - 1) / kCheckTile;
  decode_check_kernel<<<(unsigned)(nt * (nt + 1) / 2), kCheckTile, 0, s>>>(p.cache_indices, p.B, p.pool_size,
                                                                         p.status);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, int D, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  const bool h = p.fp16 != 0;
  switch (D) {
    case 64: return h ? launch_decode_t<64, f16>(p, s) : launch_decode_t<64, bf16>(p, s);
    case 128: return h ? launch_decode_t<128, f16>(p, s) : launch_decode_t<128, bf16>(p, s);
    case 256: return h ? launch_decode_t<256, f16>(p, s) : launch_decode_t<256, bf16>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
