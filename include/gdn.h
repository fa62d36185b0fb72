/*
 * gdn.h — C ABI of the GB300 chunkwise Gated DeltaNet prefill library (libgdn_gb300.so).
 *
 * The operation
 * -------------
 * gdn_extend_chunkwise runs the Gated DeltaNet recurrence over a packed batch of
 * prompts ("extend" / prefill), reading and writing each prompt's recurrent state
 * in a pooled state buffer; gdn_decode_step advances the same states by one token
 * each (see its declaration). It follows the interface documented for
 * gdn_extend_chunkwise(q, k, v, a, b, A_log, dt_bias, state_pool, cache_indices,
 * cu_seqlens, chunk_size=64) on the pymllm page "pymllm.layers.attention.gdn_chunkwise"
 * (section "Module Contents", Parameters and Returns), and computes, for every
 * sequence b and value head hv (q/k head h = hv / (HV/H)), token by token:
 *
 *   S  = state_pool[cache_indices[b], hv]                            (V x K, fp32)
 *   q^ = q[t,h] / sqrt(|q[t,h]|^2 + 1e-6),   k^ likewise
 *   alpha = exp(-exp(A_log[hv]) * softplus(a[t,hv] + dt_bias[hv]))
 *   beta  = sigmoid(b[t,hv])
 *   S  = S (alpha (I - beta k^ k^T)) + beta v[t,hv] k^T
 *   out[t,hv] = scale * S q^
 *
 * The state transition is the one in "Simple math to speed up GDN prefill"
 * (section "Reminder"); a token reads the state after its own write
 * ("nrm-training-kernels", section "General implementation", item 4). The
 * library evaluates it chunkwise in WY form with one triangular inverse per chunk,
 * the decayed factor taken from N^{-1} = G M^{-1} G^{-1} ("Simple math to speed up
 * GDN prefill", section "Save one invert"). Results equal the recurrence up to
 * rounding; chunk_size does not change them beyond rounding.
 *
 * Memory, layout, ownership
 * -------------------------
 * Every array pointer is a DEVICE pointer, dense and row-major with the last
 * index fastest. The caller owns every buffer; the library allocates nothing
 * per call and keeps no pointer after the call returns.
 *
 * Execution
 * ---------
 * The call validates its host-side arguments, then enqueues its kernels on
 * `stream` (a cudaStream_t; NULL means the legacy default stream) and returns
 * without waiting. Errors that need device data (cu_seqlens, cache_indices) are
 * detected by the first kernel, which records a status in the workspace; all
 * later kernels of that call then do nothing, so state_pool is left untouched
 * and `out` is left unwritten. Read that status with gdn_get_device_status.
 * Calls on one stream are ordered; two calls that share a workspace must not
 * run concurrently on different streams. No exception crosses this interface.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,  /* null pointer, bad size or HV % H != 0            */
  GDN_ERR_UNSUPPORTED = 2,  /* (K, V, chunk_size) not built                       */
  GDN_ERR_BAD_INDEX = 3,    /* cache index outside [0, pool_size) or repeated     */
  GDN_ERR_WORKSPACE = 4,    /* workspace null, too small or misaligned            */
  GDN_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up                 */
  GDN_ERR_CUDA = 6,         /* a CUDA runtime call failed                         */
  GDN_ERR_BAD_SEQLENS = 7   /* cu_seqlens[0] != 0, decreasing, or last != total   */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_FP16 = 1 } gdn_dtype;

/*
 * Bytes of device workspace one gdn_extend_chunkwise call needs for these sizes.
 * Returns 0 if the sizes are invalid or not supported. The workspace must be
 * 256-byte aligned. It holds the call's status word, the chunk schedule and the
 * per-chunk WY factors; it needs no initialisation and may be reused by later
 * calls on the same stream.
 */
GDN_API size_t gdn_workspace_size(int64_t total_tokens, int32_t batch, int32_t H, int32_t HV, int32_t K,
                          int32_t V, int32_t chunk_size);

/*
 * Chunkwise GDN prefill over a packed varlen batch.
 *
 *  q, k          [total_tokens, H, K]   bf16 or fp16 (dtype); q and k are NOT pre-normalised.
 *  v             [total_tokens, HV, V]  same dtype.
 *  a             [total_tokens, HV]     fp32, raw decay-gate input (before softplus/exp).
 *  b             [total_tokens, HV]     fp32, raw update-gate input (before sigmoid).
 *  A_log, dt_bias [HV]                  fp32.
 *  state_pool    [pool_size, HV, V, K]  fp32, read and overwritten in place for the
 *                                       slots named by cache_indices; other slots untouched.
 *  cache_indices [batch]                int64, pool slot of each sequence; distinct, in range.
 *  cu_seqlens    [batch + 1]            int64, cu_seqlens[0] = 0, non-decreasing,
 *                                       cu_seqlens[batch] = total_tokens. Zero-length
 *                                       sequences are allowed and leave their slot as is.
 *  out           [total_tokens, HV, V]  same dtype as v, written (round to nearest even).
 *  H, HV         q/k heads and value heads; HV must be a multiple of H.
 *  K, V          head sizes (supported: K = V in {64, 128, 256}; otherwise
 *                GDN_ERR_UNSUPPORTED).
 *  chunk_size    64 or 128 (otherwise GDN_ERR_UNSUPPORTED). The kernels factor each chunk
 *                in 64-token WY blocks: a 128-token chunk is computed as its two halves,
 *                which gives the same result up to rounding.
 *                Size limit: (total_tokens / 64 + batch + 1) * HV * 64 < 2^31 (the rows of
 *                the per-chunk factors in the workspace); larger calls return
 *                GDN_ERR_UNSUPPORTED and gdn_workspace_size returns 0 for them.
 *  scale         multiplies every output (1.0 reads o_t = S_t q_t as written).
 *  workspace     device buffer of at least gdn_workspace_size(...) bytes, 256-byte aligned.
 *  stream        cudaStream_t to enqueue on.
 *
 * Returns GDN_OK once the work is enqueued, or an error detected on the host, in
 * which case nothing was enqueued and no buffer was touched.
 */
GDN_API gdn_status gdn_extend_chunkwise(const void *q, const void *k, const void *v, gdn_dtype dtype,
                                const float *a, const float *b, const float *A_log,
                                const float *dt_bias, float *state_pool, int64_t pool_size,
                                const int64_t *cache_indices, const int64_t *cu_seqlens,
                                int32_t batch, void *out, int64_t total_tokens, int32_t H,
                                int32_t HV, int32_t K, int32_t V, int32_t chunk_size, float scale,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * Same computation and arguments as gdn_extend_chunkwise, for callers that cannot
 * allocate device memory (for example a plugin inside a host runtime that owns all
 * device memory, or a serving loop that may not call cudaMalloc/cudaFree once running,
 * since those can synchronise the device or fail under a fixed memory budget). The pages
 * have no counterpart of this entry point: it is a deployment variant of the call above.
 *
 * Instead of a caller-provided workspace it uses a scratch array built into the library:
 * 64 MiB, reserved on every GPU that loads the library until the process exits. Calls
 * whose gdn_workspace_size(...) exceeds 64 MiB return GDN_ERR_WORKSPACE before touching
 * anything. It calls no allocator. The first call on each device looks up the scratch
 * address on that device (make it before capturing any stream); the address is kept until
 * the process exits, so after cudaDeviceReset on a device this entry point must not be
 * used there again. All calls share the scratch and it keeps the last call's contents;
 * calls that overlap on the GPU (e.g. on two streams at once) race on it and must not be
 * issued.
 *
 * device_status: optional DEVICE pointer to one int32, 4-byte aligned (else
 * GDN_ERR_INVALID_ARG). When not NULL and the call returns GDN_OK, the status the call's
 * kernels record (GDN_OK, GDN_ERR_BAD_INDEX, GDN_ERR_BAD_SEQLENS, GDN_ERR_TIMEOUT) is
 * copied there, in stream order, after the call's kernels. A call that returns an error
 * enqueues nothing and leaves *device_status unwritten.
 */
GDN_API gdn_status gdn_extend_chunkwise_noalloc(const void *q, const void *k, const void *v, gdn_dtype dtype,
                                                const float *a, const float *b, const float *A_log,
                                                const float *dt_bias, float *state_pool, int64_t pool_size,
                                                const int64_t *cache_indices, const int64_t *cu_seqlens,
                                                int32_t batch, void *out, int64_t total_tokens, int32_t H,
                                                int32_t HV, int32_t K, int32_t V, int32_t chunk_size, float scale,
                                                int32_t *device_status, void *stream);

/*
 * Single-token step (decode): one new token for each of `batch` sequences, against the
 * same state pool and index contract as gdn_extend_chunkwise. It is that call with
 * cu_seqlens = 0, 1, ..., batch (the one-token case of the recurrence above: the
 * transition of "Simple math to speed up GDN prefill", section "Reminder", and the
 * output read after the write), computed directly without chunking:
 *
 *   S' = alpha S + beta (v - alpha S k^) k^^T,   out = scale S' q^
 *
 *  q, k          [batch, H, K]   bf16 or fp16 (dtype), not pre-normalised.
 *  v             [batch, HV, V]  same dtype.
 *  a, b          [batch, HV]     fp32 raw gate inputs; A_log, dt_bias [HV] fp32.
 *  state_pool    [pool_size, HV, V, K] fp32, slots named by cache_indices read and
 *                overwritten in place; other slots untouched.
 *  cache_indices [batch] int64, distinct, in [0, pool_size).
 *  out           [batch, HV, V] same dtype as v, written.
 *  K, V          K = V in {64, 128, 256} (otherwise GDN_ERR_UNSUPPORTED).
 *  device_status DEVICE pointer to one int32 (4-byte aligned), owned by the caller. In
 *                stream order the step sets it to GDN_OK, or to GDN_ERR_BAD_INDEX if a slot
 *                is out of range or repeated, in which case the update kernel touches
 *                nothing. Read it with gdn_get_device_status(device_status, stream).
 *  stream        cudaStream_t to enqueue on.
 *
 * q, k, v, out and state_pool must be 16-byte aligned; 0 <= batch <= 2^20 and
 * batch * HV < 2^31. Host-detectable errors (null pointer, misalignment, bad sizes,
 * HV % H != 0, dtype) return before anything is enqueued; batch = 0 only resets the
 * status word. No workspace; the library allocates nothing. Launches two kernels (the
 * second with programmatic dependent launch behind the first); batches above 1024 also
 * zero the status word with one memset before them.
 */
GDN_API gdn_status gdn_decode_step(const void *q, const void *k, const void *v, gdn_dtype dtype,
                                   const float *a, const float *b, const float *A_log,
                                   const float *dt_bias, float *state_pool, int64_t pool_size,
                                   const int64_t *cache_indices, int32_t batch, void *out, int32_t H,
                                   int32_t HV, int32_t K, int32_t V, float scale,
                                   int32_t *device_status, void *stream);

/*
 * Bytes of workspace that gdn_chunkwise_backward needs for these sizes, or 0 if the
 * sizes are not supported (K != V, K not in {64, 128}, chunk_size not in {64, 128},
 * HV % H != 0, HV > 65535, total_tokens >= 2^31). About 384 KB per (64-token chunk,
 * value head) at K = V = 128 plus 1 KB per (token, value head): the per-chunk
 * intermediates of the backward are kept in fp32.
 */
GDN_API size_t gdn_backward_workspace_size(int64_t total_tokens, int32_t batch, int32_t H,
                                           int32_t HV, int32_t K, int32_t V, int32_t chunk_size);

/*
 * Backward pass of gdn_extend_chunkwise: the gradients of
 *
 *   L = sum_t <d_out_t, out_t> + sum over (sequence, value head) <d_state, S_final>
 *
 * with respect to every input of the forward call with the same arguments. The pages
 * give no backward formulas; the bottom-level GDN backward of "nrm-training-kernels",
 * section "Kernel", takes the gradient arriving at the final state besides the output's
 * (d_state here). The kernels apply the chain rule to the chunkwise WY form of
 * "Simple math to speed up GDN prefill" (sections "Reminder" and "Save one invert"):
 * a forward pass over the chunks that recomputes the state entering each chunk, a
 * reverse pass over the chunks for the state gradient, then per-chunk gradients through
 * the one inverse, the decays, the gates and the q/k normalisation.
 *
 *  q, k, v, a, b, A_log, dt_bias, cache_indices, cu_seqlens, batch, total_tokens, H, HV,
 *  K, V, chunk_size, scale, dtype: as for gdn_extend_chunkwise (DEVICE pointers).
 *  state_pool    [pool_size, HV, V, K] fp32, READ ONLY: the initial states, i.e. the
 *                pool as the forward call found it (the forward overwrites the slots it
 *                uses, so a caller that needs the backward keeps a copy).
 *  d_out         [total_tokens, HV, V] same dtype as v: gradient of out.
 *  d_state       [pool_size, HV, V, K] fp32: gradient of the final state of each
 *                sequence, read at the batch's slots; NULL means zero.
 *  dq, dk        [total_tokens, H, K] fp32, written (value heads sharing a q/k head
 *                contribute their sum).
 *  dv            [total_tokens, HV, V] fp32, written.
 *  da, db        [total_tokens, HV] fp32, written.
 *  dA_log, ddt_bias  [HV] fp32, written (sums over all tokens, in a fixed order).
 *  d_state_pool  [pool_size, HV, V, K] fp32: the gradient of the initial states is
 *                written at the batch's slots; other slots are untouched. It may be the
 *                same buffer as d_state (each slot is read before it is written).
 *  workspace     DEVICE pointer, 256-byte aligned, >= gdn_backward_workspace_size bytes,
 *                owned by the caller; no two calls in flight may share one.
 *
 * Supported: K = V in {64, 128}; chunk_size 64 or 128 (the kernels work on 64-token WY
 * blocks; the gradients do not depend on the block length in exact arithmetic).
 * q, k, v, d_out, dq, dk 16-byte aligned; dv, state_pool, d_state, d_state_pool 8-byte aligned.
 * Host-detectable errors return before anything is enqueued. Device-detected errors
 * (cu_seqlens, cache_indices: as for gdn_extend_chunkwise) are recorded in the
 * workspace's status word, read by gdn_get_device_status(workspace, stream); the
 * gradient outputs are then left unwritten. Every sum is taken in a fixed order, so
 * repeated calls give bit-identical results.
 */
GDN_API gdn_status gdn_chunkwise_backward(const void *q, const void *k, const void *v,
                                          gdn_dtype dtype, const float *a, const float *b,
                                          const float *A_log, const float *dt_bias,
                                          const float *state_pool, int64_t pool_size,
                                          const int64_t *cache_indices, const int64_t *cu_seqlens,
                                          int32_t batch, const void *d_out, const float *d_state,
                                          float *dq, float *dk, float *dv, float *da, float *db,
                                          float *dA_log, float *ddt_bias, float *d_state_pool,
                                          int64_t total_tokens, int32_t H, int32_t HV, int32_t K,
                                          int32_t V, int32_t chunk_size, float scale,
                                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * Waits for `stream`, then returns the status recorded on the device by the last
 * gdn_extend_chunkwise call that used this workspace (GDN_OK, GDN_ERR_BAD_INDEX,
 * GDN_ERR_BAD_SEQLENS or GDN_ERR_TIMEOUT), or GDN_ERR_CUDA if the stream reported
 * an error. Synchronises the host with the stream. Given the device_status word of
 * gdn_decode_step instead of a workspace, it returns that step's status.
 */
GDN_API gdn_status gdn_get_device_status(const void *workspace, void *stream);

/*
 * Where one gdn_extend_chunkwise call keeps its per-chunk intermediates in the workspace
 * (byte offsets from the workspace start), for inspection and tests; the layout belongs to
 * this library version. For chunk j of the call's chunk table (int32[4] per chunk at
 * chunk_tab: sequence, first token, length, chunk index in the sequence; chunks restart
 * at each sequence and hold `block` tokens, the last one fewer), value head hv and q/k head h:
 *   g    fp32 [.][HV][block]    chunk-local cumulative log decay at (j * HV + hv) * block
 *   beta fp32 [.][HV][block]    beta, 0 on rows past the chunk's length
 *   rq, rk fp32 [.][H][block]   1/|q|, 1/|k| at (j * H + h) * block, 0 past the length
 *   w, u 16-bit [.][HV][block][K or V]  the WY factors W<- and U~ of the chunk
 *   p    16-bit [.][HV][block][block]   the masked, decayed intra-chunk scores
 * With affine_factors = 1 (K = V = 128) row t of w and u and column t of p carry the
 * mantissa m_t of exp(g_last - g_t) / |k_t| = m_t * 2^e_t (rows times m_t, columns divided by
 * it) and ks (fp32, like g) holds 2^e_t; otherwise ks is (size_t)-1 and the factors are
 * unscaled. A scan cut into nseg > 1 segments per sequence keeps, per (sequence b, value
 * head hv, segment s), the fp32 start state [V][K] at seg_state + ((b * HV + hv) * nseg + s) * V*K*4
 * and, when nseg > 2, the segment's affine map S_end = S_start T + B0 at seg_map: B0 [V][K] then
 * T [K][K] at ((b * HV + hv) * nseg + s) * 2 * K*K*4. Returns GDN_ERR_UNSUPPORTED for sizes
 * gdn_workspace_size rejects.
 */
typedef struct {
  size_t status, chunk_tab, g, beta, rq, rk, ks, w, u, p, seg_state, seg_map, total;
  int64_t max_chunks;
  int32_t block;
  int32_t affine_factors;
  int32_t nseg;
} gdn_workspace_layout_t;
GDN_API gdn_status gdn_workspace_layout(int64_t total_tokens, int32_t batch, int32_t H, int32_t HV, int32_t K,
                                        int32_t V, int32_t chunk_size, gdn_workspace_layout_t *out);

/*
 * Test hook for the failure path of the bounded device-side waits; never needed in use.
 * kernel = 1 (the intra-chunk kernel), 2 (the chunk scan) or 3 (the first pass of the
 * segmented scan for K = V = 128) makes that kernel's CTAs issue none of their tile loads in
 * later gdn_extend_chunkwise calls, so every wait in them runs out after wait_budget_cycles
 * SM clock cycles: the call then records GDN_ERR_TIMEOUT, leaves state_pool untouched and
 * every kernel exits normally. kernel = 0 restores normal operation and the default budget
 * (2^31 cycles, about a second). Process-wide; not to be changed while calls are in flight.
 */
GDN_API gdn_status gdn_test_set_stall(int32_t kernel, int64_t wait_budget_cycles);

/* Static, human-readable name of a status. Never NULL. */
GDN_API const char *gdn_status_string(gdn_status status);

/*
 * Instrumentation. gdn_profile_start makes every later gdn_extend_chunkwise or gdn_decode_step call
 * record a pair of CUDA events around each kernel it launches, on the call's own
 * stream, for up to max_launches kernel launches in total (the events are created
 * here, on the current device). gdn_profile_stop waits for those events, adds the
 * elapsed time of each kernel kind into total_ms[id] and its launch count into
 * launches[id] for id < n_slots, frees the events and returns the number of kernel
 * kinds (ids 0 .. n-1; see gdn_kernel_name). Returns -1 if profiling was not started
 * or an event failed. Not meant to be used while another thread issues calls.
 */
GDN_API gdn_status gdn_profile_start(int32_t max_launches);
GDN_API int32_t gdn_profile_stop(double *total_ms, int64_t *launches, int32_t n_slots);

/* Name of kernel kind `id` (as used by gdn_profile_stop), or NULL if out of range. */
GDN_API const char *gdn_kernel_name(int32_t id);

/* Total number of kernels this library has launched in the process so far. */
GDN_API int64_t gdn_launch_count(void);

/* Library version as major * 10000 + minor * 100 + patch. */
GDN_API int32_t gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
