// gdn_backward.cuh — launch parameters and workspace layout of the chunkwise backward pass
// (gdn_backward.cu), shared with the host entry point in gdn_api.cu.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Workspace regions (byte offsets, each on a 256-byte boundary). mc = max_chunks, D = K = V.
struct BwdLayout {
  size_t status, seq_chunk_off, order, chunk_tab;  // as in the forward (schedule kernel)
  size_t g, beta;                                   // fp32 [mc][HV][C] (gates kernel)
  size_t rq, rk;                                    // fp32 [mc][HV][C]: 1/|q|, 1/|k| (0 on padded rows)
  size_t minv;                                      // bf16 [mc][HV][2][C][C]: M^{-1}, hi and lo planes
  size_t pm;                                        // bf16 [mc][HV][2][C][C]: P = Gamma . tril(Q^ K^^T), hi and lo planes
  size_t w;                                         // bf16 [mc][HV][2][C][D]: W<-, hi and lo planes
  size_t ut;                                        // fp32 [mc][HV][C][D]: U~
  size_t s_in;                                      // bf16 [mc][HV][2][D][D]: state entering each chunk (planes)
  size_t u;                                         // bf16 [mc][HV][2][C][D]: U = U~ - W<- S^T (planes)
  size_t ds_out;                                    // bf16 [mc][HV][2][D][D]: gradient of the state leaving each chunk
  size_t du;                                        // bf16 [mc][HV][2][C][D]: gradient of U (planes)
  size_t dqa, dkr;                                  // fp32 [mc][HV][C][D]: scale e^g (dO S_in), U dS_out
  size_t dw;                                        // bf16 [mc][HV][2][C][D]: -dU S_in (planes)
  size_t dgc;                                       // fp32 [mc][HV][2]: exp(g_C) <dS_out, S_in>, by key-column half
  size_t dqh, dkh;                                  // fp32 [T][HV][D]: gradients of q^, k^ per value head
  size_t dlala;                                     // fp32 [T][HV]: d log alpha * log alpha
  size_t total;
  int64_t max_chunks;
};

BwdLayout make_bwd_layout(int64_t T, int B, int H, int HV, int D);

struct BwdParams {
  const void* q;  // [T][H][D], 16-bit (bf16, or fp16 when fp16 = 1)
  const void* k;
  const void* v;      // [T][HV][D]
  const void* d_out;  // [T][HV][D], same type as v
  const float* a;     // [T][HV]
  const float* b;
  const float* A_log;  // [HV]
  const float* dt_bias;
  const float* state_pool;  // [pool][HV][D][D]: the initial states
  const float* d_state;     // [pool][HV][D][D]: gradient of the final states, or null (zero)
  const int64_t* cache_indices;
  float* dq;  // [T][H][D]
  float* dk;
  float* dv;  // [T][HV][D]
  float* da;  // [T][HV]
  float* db;
  float* dA_log;  // [HV]
  float* ddt_bias;
  float* d_state_pool;  // [pool][HV][D][D]: gradient of the initial states, written at the batch's slots
  int64_t T;
  int B, H, HV;
  float scale;
  int64_t max_chunks;
  int32_t* status;
  int32_t* seq_chunk_off;
  int32_t* order;
  int4* chunk_tab;
  float *g, *beta, *rq, *rk;
  void *minv, *pm, *w;           // bf16 hi, lo planes
  float* ut;
  void *s_in, *u, *ds_out, *du;  // bf16 hi, lo planes
  float* dqa;
  void* dw;                      // bf16 hi, lo planes
  float *dkr, *dgc, *dqh, *dkh, *dlala;
};

// Launches the backward kernels after the schedule and gates kernels of the call have run on s.
// kernels: set to the number of kernels launched.
cudaError_t launch_backward(const BwdParams& p, int D, bool fp16, cudaStream_t s, int* kernels);

}  // namespace gdn
