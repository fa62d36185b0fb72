// gdn_gates.cu — K1: the gates of every chunk, for all value heads at once.
//
//   log alpha = -exp(A_log) softplus(a + dt_bias),  beta = sigmoid(b)
//               (pymllm page "pymllm.layers.attention.gdn_chunkwise", Parameters: a and b
//               are the raw gate inputs before softplus/exp and sigmoid)
//   g         = chunk-local inclusive prefix sum of log alpha  ("Simple math to speed up GDN
//               prefill", section "Reminder": g_i = sum of log alpha_j, j <= i in the chunk)
//
// One CTA per (chunk, block of up to 64 value heads). The chunk's rows of a and b are
// contiguous in memory ([T, HV] fp32), so they are read with 16-byte loads when HV allows;
// the per-head results are transposed in shared memory and written as [chunk][HV][C] rows,
// the layout the intra-chunk and scan kernels read with bulk copies. Padded rows of a
// partial chunk get log alpha = 0 and beta = 0.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int C = 64;
constexpr int HB = 64;  // value heads per CTA
constexpr int kThreads = 256;

__device__ __forceinline__ float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

__global__ void __launch_bounds__(kThreads) gates_kernel(Params p) {
  __shared__ float s_la[HB][C + 1];
  __shared__ float s_bt[HB][C + 1];
  if (p.status[0] != GDN_OK) return;
  const int j = blockIdx.x;
  if (j >= p.status[1]) return;
  const int4 ct = p.chunk_tab[j];
  const int64_t t0 = ct.y;
  const int len = ct.z;
  const int HV = p.HV;
  const int h0 = blockIdx.y * HB;
  const int nh = min(HB, HV - h0);
  const int tid = threadIdx.x;

  auto gate = [&](int t, int h, float a, float b) {
    s_la[h][t] = -expf(p.A_log[h0 + h]) * softplus_f(a + p.dt_bias[h0 + h]);
    s_bt[h][t] = 1.f / (1.f + expf(-b));
  };
  if ((HV & 3) == 0 && (nh & 3) == 0) {  // 16-byte loads: 4 heads of one token each
    const int nq = nh >> 2;
    for (int e = tid; e < len * nq; e += kThreads) {
      const int t = e / nq, h = (e % nq) * 4;
      const int64_t o = (t0 + t) * HV + h0 + h;
      const float4 a4 = *reinterpret_cast<const float4*>(p.a + o);
      const float4 b4 = *reinterpret_cast<const float4*>(p.b + o);
      gate(t, h, a4.x, b4.x);
      gate(t, h + 1, a4.y, b4.y);
      gate(t, h + 2, a4.z, b4.z);
      gate(t, h + 3, a4.w, b4.w);
    }
  } else {
    for (int e = tid; e < len * nh; e += kThreads) {
      const int t = e / nh, h = e % nh;
      const int64_t o = (t0 + t) * HV + h0 + h;
      gate(t, h, p.a[o], p.b[o]);
    }
  }
  for (int e = tid; e < (C - len) * nh; e += kThreads) {  // padded rows
    const int t = len + e / nh, h = e % nh;
    s_la[h][t] = 0.f;
    s_bt[h][t] = 0.f;
  }
  __syncthreads();

  // one warp per head: lane l owns tokens 2l, 2l+1; inclusive scan over the warp
  const int warp = tid >> 5, lane = tid & 31;
  for (int h = warp; h < nh; h += kThreads / 32) {
    const float x0 = s_la[h][2 * lane];
    const float x1 = x0 + s_la[h][2 * lane + 1];
    float incl = x1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const float excl = incl - x1;
    const int64_t row = ((int64_t)j * HV + h0 + h) * C;
    reinterpret_cast<float2*>(p.g + row)[lane] = make_float2(excl + x0, incl);
    reinterpret_cast<float2*>(p.beta + row)[lane] = make_float2(s_bt[h][2 * lane], s_bt[h][2 * lane + 1]);
  }
}

}  // namespace

cudaError_t launch_gates(const Params& p, int Cc, cudaStream_t s) {
  if (Cc != C) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)p.max_chunks, (unsigned)((p.HV + HB - 1) / HB));
  gates_kernel<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
