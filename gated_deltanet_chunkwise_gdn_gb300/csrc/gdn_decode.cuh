// gdn_decode.cuh — the single-token step (decode): its launch arguments and launchers.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

// Arguments of one single-token step (gdn_decode_step); pointers as in include/gdn.h.
struct DecodeParams {
  const void* q;  // [B, H, K] 16-bit (bf16, or fp16 when fp16 is set)
  const void* k;
  const void* v;  // [B, HV, V]
  const float* a;
  const float* b;
  const float* A_log;
  const float* dt_bias;
  float* state_pool;
  const int64_t* cache_indices;
  void* out;  // [B, HV, V], v's type
  int64_t pool_size;
  int B, H, HV;
  float scale;
  int32_t* status;  // the step's status word: set by the check kernel (zeroed first for large batches)
  int fp16;
};

// Slot check and state update. Batches above 1024 are checked by a grid that records only
// errors, so the status word must be zeroed before it.
bool decode_check_needs_zeroed_status(int B);
cudaError_t launch_decode_check(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, int D, cudaStream_t s);

}  // namespace gdn
