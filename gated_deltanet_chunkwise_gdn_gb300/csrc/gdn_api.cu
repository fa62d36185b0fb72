// gdn_api.cu — host side of the C ABI declared in include/gdn.h: argument checks,
// workspace carve-up and the launch sequence K0 (schedule) -> K1 (gates) -> K2 (intra) -> K3 (scan)
// of the prefill call, and the single-token step (slot check -> state update).
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "gdn_backward.cuh"
#include "gdn_common.cuh"
#include "gdn_decode.cuh"

namespace {

// ---------------------------------------------------------------- instrumentation

// An NVTX range over one entry-point call (host side: argument checks and the enqueue of its
// kernels), visible in Nsight timelines next to the kernels; a no-op unless a tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
enum KernelId {  // scan: every scan-stage launch
  kKernSchedule = 0, kKernGates = 1, kKernIntra = 2, kKernScan = 3, kKernDecodeCheck = 4, kKernDecode = 5,
  kKernBackward = 6, kKernCount = 7
};
const char* const kKernelNames[kKernCount] = {"schedule", "gates", "intra", "scan", "decode_check", "decode",
                                              "backward"};

std::atomic<int64_t> g_launches{0};

// Test hook (gdn_test_set_stall): the wait budget of every bounded device-side wait, and the
// kernel that withholds its tile loads. Read by each prefill call when it builds its launch
// arguments.
std::atomic<long long> g_wait_budget{gdn::kDefaultWaitBudget};
std::atomic<int> g_stall{gdn::kStallNone};

struct ProfRecord {
  int id;
  cudaEvent_t start, stop;
};
struct Profiler {
  std::mutex mu;
  bool on = false;
  int capacity = 0;
  std::vector<ProfRecord> recs;
  std::vector<cudaEvent_t> pool;  // created at start, 2 per allowed launch
} g_prof;

// Records the start event of kernel `id` on stream s; returns the record index or -1.
int prof_begin(int id, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.on || (int)g_prof.recs.size() >= g_prof.capacity) return -1;
  const int i = (int)g_prof.recs.size();
  ProfRecord r{id, g_prof.pool[2 * i], g_prof.pool[2 * i + 1]};
  if (cudaEventRecord(r.start, s) != cudaSuccess) return -1;
  g_prof.recs.push_back(r);
  return i;
}
void prof_end(int rec, cudaStream_t s, int kernels = 1) {
  g_launches.fetch_add(kernels, std::memory_order_relaxed);
  if (rec < 0) return;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  cudaEventRecord(g_prof.recs[rec].stop, s);
}

// The enqueue of one kernel group of a call: an NVTX range named after the group (nested in the
// call's range, closed when the scope ends, error returns included) and, while the profiler is on,
// the group's CUDA-event pair; done() records the end event and counts the group's launches.
struct LaunchScope {
  NvtxRange range;
  int rec;
  cudaStream_t s;
  LaunchScope(int id, cudaStream_t stream) : range(kKernelNames[id]), rec(prof_begin(id, stream)), s(stream) {}
  void done(int kernels = 1) { prof_end(rec, s, kernels); }
};

bool supported_shape(int K, int V, int C) {
  if (K != V) return false;
  return (K == 64 || K == 128 || K == 256) && (C == 64 || C == 128);
}

// The kernels' WY block: 64 tokens. A 128-token chunk is processed as its two 64-token
// halves, each with its own M^{-1}; in exact arithmetic the result does not depend on
// the block length (the chunkwise form equals the token recurrence for any block length).
constexpr int kWyBlock = 64;

// Value-dimension split of the scan: blocks of 64 state rows per CTA.
int choose_nvb(int V) { return V / 64; }

// The per-chunk factors W<-, U~ and P are tiles of [max_chunks * HV * 64, *] arrays that TMA
// addresses with 32-bit signed row coordinates, so the row count must stay below 2^31.
bool factor_rows_fit(const gdn::WsLayout& L, int HV) {
  return L.max_chunks * (int64_t)HV * kWyBlock <= (int64_t)INT32_MAX;
}

// The backward pass: K = V in {64, 128}; chunk_size 64 or 128 (64-token WY blocks either way).
bool supported_backward_shape(int K, int V, int C) {
  return K == V && (K == 64 || K == 128) && (C == 64 || C == 128);
}

// Largest batch of one single-token step. Above 1024 sequences the slot check runs one block
// per pair of 256-index tiles: 2^20 sequences take 8.4 M blocks, far inside the grid limit.
constexpr int32_t kMaxDecodeBatch = 1 << 20;

// K0 of a prefill or backward call: for batches above kScheduleSortMax the multi-block slot check
// first (it records errors in the zeroed status word), then schedule_kernel.
gdn_status launch_schedule(const gdn::Params& p, int32_t batch, int64_t pool_size, const int64_t* cache_indices,
                           cudaStream_t s) {
  LaunchScope ls(kKernSchedule, s);
  const bool pre_check = batch > gdn::kScheduleSortMax;
  if (pre_check) {
    gdn::DecodeParams dp{};
    dp.cache_indices = cache_indices;
    dp.pool_size = pool_size;
    dp.B = batch;
    dp.status = p.status;
    if (cudaMemsetAsync(p.status, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
    if (gdn::launch_decode_check(dp, s) != cudaSuccess) return GDN_ERR_CUDA;
  }
  const size_t sched_smem = gdn::schedule_smem_bytes(batch);
  if (sched_smem > 48 * 1024 &&
      cudaFuncSetAttribute(gdn::schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sched_smem) !=
          cudaSuccess)
    return GDN_ERR_CUDA;
  gdn::schedule_kernel<<<1, 512, sched_smem, s>>>(p, kWyBlock, pre_check ? 1 : 0);
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  ls.done(pre_check ? 2 : 1);
  return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_workspace_size(int64_t total_tokens, int32_t batch, int32_t H, int32_t HV, int32_t K, int32_t V,
                          int32_t chunk_size) {
  if (total_tokens < 0 || total_tokens >= (int64_t)INT32_MAX || batch < 0 || H <= 0 || HV <= 0 || HV % H != 0)
    return 0;
  if (!supported_shape(K, V, chunk_size)) return 0;
  const gdn::WsLayout L = gdn::make_layout(total_tokens, batch, H, HV, K, V, kWyBlock);
  return factor_rows_fit(L, HV) ? L.total : 0;
}

gdn_status gdn_extend_chunkwise(const void* q, const void* k, const void* v, gdn_dtype dtype, const float* a,
                                const float* b, const float* A_log, const float* dt_bias, float* state_pool,
                                int64_t pool_size, const int64_t* cache_indices, const int64_t* cu_seqlens,
                                int32_t batch, void* out, int64_t total_tokens, int32_t H, int32_t HV, int32_t K,
                                int32_t V, int32_t chunk_size, float scale, void* workspace, size_t workspace_bytes,
                                void* stream) {
  NvtxRange range("gdn_extend_chunkwise");
  if (batch < 0 || total_tokens < 0 || total_tokens >= (int64_t)INT32_MAX || H <= 0 || HV <= 0 || HV % H != 0 ||
      K <= 0 || V <= 0 || chunk_size <= 0)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_BF16 && dtype != GDN_FP16) return GDN_ERR_INVALID_ARG;
  if (!cu_seqlens || !A_log || !dt_bias) return GDN_ERR_INVALID_ARG;
  if (batch > 0 && (!state_pool || !cache_indices || pool_size <= 0)) return GDN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!q || !k || !v || !a || !b || !out)) return GDN_ERR_INVALID_ARG;
  if (!supported_shape(K, V, chunk_size)) return GDN_ERR_UNSUPPORTED;
  const gdn::WsLayout L = gdn::make_layout(total_tokens, batch, H, HV, K, V, kWyBlock);
  if (!factor_rows_fit(L, HV)) return GDN_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return GDN_ERR_WORKSPACE;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  gdn::Params p{};
  p.q = static_cast<const gdn::bf16*>(q);
  p.k = static_cast<const gdn::bf16*>(k);
  p.v = static_cast<const gdn::bf16*>(v);
  p.a = a;
  p.b = b;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.state_pool = state_pool;
  p.cache_indices = cache_indices;
  p.cu_seqlens = cu_seqlens;
  p.out = static_cast<gdn::bf16*>(out);
  p.T = total_tokens;
  p.pool_size = pool_size;
  p.B = batch;
  p.H = H;
  p.HV = HV;
  p.nvb = choose_nvb(V);
  p.scale = scale;
  p.max_chunks = L.max_chunks;
  p.status = reinterpret_cast<int32_t*>(ws + L.status);
  p.seq_chunk_off = reinterpret_cast<int32_t*>(ws + L.seq_chunk_off);
  p.order = reinterpret_cast<int32_t*>(ws + L.order);
  p.chunk_tab = reinterpret_cast<int4*>(ws + L.chunk_tab);
  p.g = reinterpret_cast<float*>(ws + L.g);
  p.beta = reinterpret_cast<float*>(ws + L.beta);
  p.rq = reinterpret_cast<float*>(ws + L.rq);
  p.rk = reinterpret_cast<float*>(ws + L.rk);
  p.ks = reinterpret_cast<float*>(ws + L.ks);
  p.W = reinterpret_cast<gdn::bf16*>(ws + L.w);
  p.U = reinterpret_cast<gdn::bf16*>(ws + L.u);
  p.P = reinterpret_cast<gdn::bf16*>(ws + L.p);
  p.seg_state = reinterpret_cast<float*>(ws + L.seg_state);
  p.seg_map = reinterpret_cast<float*>(ws + L.seg_map);
  p.nseg = L.nseg;
  p.seg_r16 = K == 128 ? 8 : 16;  // K = V = 128: a full-mode chunk costs about twice a map-mode chunk
  p.fp16 = dtype == GDN_FP16 ? 1 : 0;
  p.wait_budget = g_wait_budget.load(std::memory_order_relaxed);
  p.stall = g_stall.load(std::memory_order_relaxed);

  if (launch_schedule(p, batch, pool_size, cache_indices, s) != GDN_OK) return GDN_ERR_CUDA;
  if (total_tokens == 0 || batch == 0) return GDN_OK;
  {
    LaunchScope ls(kKernGates, s);
    if (gdn::launch_gates(p, kWyBlock, s) != cudaSuccess) return GDN_ERR_CUDA;
    ls.done();
  }
  {
    LaunchScope ls(kKernIntra, s);
    if (gdn::launch_intra(p, K, kWyBlock, s) != cudaSuccess) return GDN_ERR_CUDA;
    ls.done();
  }
  {
    LaunchScope ls(kKernScan, s);
    if (gdn::launch_scan(p, K, kWyBlock, s) != cudaSuccess) return GDN_ERR_CUDA;
    ls.done(p.nseg <= 1 ? 1 : (p.nseg == 2 ? 2 : 3));  // segmented: maps, combine, segments
  }
  return GDN_OK;
}

size_t gdn_backward_workspace_size(int64_t total_tokens, int32_t batch, int32_t H, int32_t HV, int32_t K,
                                   int32_t V, int32_t chunk_size) {
  if (total_tokens < 0 || total_tokens >= (int64_t)INT32_MAX || batch < 0 || H <= 0 || HV <= 0 || HV % H != 0 ||
      HV > 65535)
    return 0;
  if (!supported_backward_shape(K, V, chunk_size)) return 0;
  if ((int64_t)batch * HV * (K / 16) > (int64_t)INT32_MAX) return 0;  // grid of the sequential passes
  if ((total_tokens * H + 7) / 8 > (int64_t)INT32_MAX) return 0;       // grid of the grouped-heads norm kernel
  return gdn::make_bwd_layout(total_tokens, batch, H, HV, K).total;
}

gdn_status gdn_chunkwise_backward(const void* q, const void* k, const void* v, gdn_dtype dtype, const float* a,
                                  const float* b, const float* A_log, const float* dt_bias, const float* state_pool,
                                  int64_t pool_size, const int64_t* cache_indices, const int64_t* cu_seqlens,
                                  int32_t batch, const void* d_out, const float* d_state, float* dq, float* dk,
                                  float* dv, float* da, float* db, float* dA_log, float* ddt_bias,
                                  float* d_state_pool, int64_t total_tokens, int32_t H, int32_t HV, int32_t K,
                                  int32_t V, int32_t chunk_size, float scale, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  NvtxRange range("gdn_chunkwise_backward");
  if (batch < 0 || total_tokens < 0 || total_tokens >= (int64_t)INT32_MAX || H <= 0 || HV <= 0 || HV % H != 0 ||
      K <= 0 || V <= 0 || chunk_size <= 0)
    return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_BF16 && dtype != GDN_FP16) return GDN_ERR_INVALID_ARG;
  if (!cu_seqlens || !A_log || !dt_bias || !dA_log || !ddt_bias) return GDN_ERR_INVALID_ARG;
  if (batch > 0 && (!state_pool || !cache_indices || !d_state_pool || pool_size <= 0)) return GDN_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!q || !k || !v || !a || !b || !d_out || !dq || !dk || !dv || !da || !db))
    return GDN_ERR_INVALID_ARG;
  auto al = [](const void* x, uintptr_t n) { return (reinterpret_cast<uintptr_t>(x) & (n - 1)) == 0; };
  if (total_tokens > 0 &&
      !(al(q, 16) && al(k, 16) && al(v, 16) && al(d_out, 16) && al(dq, 16) && al(dk, 16) && al(dv, 8)))
    return GDN_ERR_INVALID_ARG;
  if (batch > 0 && !(al(state_pool, 8) && al(d_state_pool, 8) && al(d_state, 8))) return GDN_ERR_INVALID_ARG;
  const size_t need = gdn_backward_workspace_size(total_tokens, batch, H, HV, K, V, chunk_size);
  if (need == 0) return GDN_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return GDN_ERR_WORKSPACE;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const gdn::BwdLayout L = gdn::make_bwd_layout(total_tokens, batch, H, HV, K);
  // The schedule and gates kernels of the forward, on the backward's workspace.
  gdn::Params p{};
  p.a = a;
  p.b = b;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.cache_indices = cache_indices;
  p.cu_seqlens = cu_seqlens;
  p.T = total_tokens;
  p.pool_size = pool_size;
  p.B = batch;
  p.H = H;
  p.HV = HV;
  p.max_chunks = L.max_chunks;
  p.status = reinterpret_cast<int32_t*>(ws + L.status);
  p.seq_chunk_off = reinterpret_cast<int32_t*>(ws + L.seq_chunk_off);
  p.order = reinterpret_cast<int32_t*>(ws + L.order);
  p.chunk_tab = reinterpret_cast<int4*>(ws + L.chunk_tab);
  p.g = reinterpret_cast<float*>(ws + L.g);
  p.beta = reinterpret_cast<float*>(ws + L.beta);
  p.wait_budget = g_wait_budget.load(std::memory_order_relaxed);

  if (launch_schedule(p, batch, pool_size, cache_indices, s) != GDN_OK) return GDN_ERR_CUDA;
  if (batch == 0) return GDN_OK;
  if (total_tokens > 0) {
    LaunchScope ls(kKernGates, s);
    if (gdn::launch_gates(p, kWyBlock, s) != cudaSuccess) return GDN_ERR_CUDA;
    ls.done();
  }

  gdn::BwdParams bp{};
  bp.q = q;
  bp.k = k;
  bp.v = v;
  bp.d_out = d_out;
  bp.a = a;
  bp.b = b;
  bp.A_log = A_log;
  bp.dt_bias = dt_bias;
  bp.state_pool = state_pool;
  bp.d_state = d_state;
  bp.cache_indices = cache_indices;
  bp.dq = dq;
  bp.dk = dk;
  bp.dv = dv;
  bp.da = da;
  bp.db = db;
  bp.dA_log = dA_log;
  bp.ddt_bias = ddt_bias;
  bp.d_state_pool = d_state_pool;
  bp.T = total_tokens;
  bp.B = batch;
  bp.H = H;
  bp.HV = HV;
  bp.scale = scale;
  bp.max_chunks = L.max_chunks;
  bp.status = p.status;
  bp.seq_chunk_off = p.seq_chunk_off;
  bp.order = p.order;
  bp.chunk_tab = p.chunk_tab;
  auto f = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  bp.g = f(L.g);
  bp.beta = f(L.beta);
  bp.rq = f(L.rq);
  bp.rk = f(L.rk);
  bp.minv = f(L.minv);
  bp.pm = f(L.pm);
  bp.w = f(L.w);
  bp.ut = f(L.ut);
  bp.s_in = f(L.s_in);
  bp.u = f(L.u);
  bp.ds_out = f(L.ds_out);
  bp.du = f(L.du);
  bp.dqa = f(L.dqa);
  bp.dw = f(L.dw);
  bp.dkr = f(L.dkr);
  bp.dgc = f(L.dgc);
  bp.dqh = f(L.dqh);
  bp.dkh = f(L.dkh);
  bp.dlala = f(L.dlala);
  {
    LaunchScope ls(kKernBackward, s);
    int kernels = 0;
    if (gdn::launch_backward(bp, K, dtype == GDN_FP16, s, &kernels) != cudaSuccess) return GDN_ERR_CUDA;
    ls.done(kernels);
  }
  return GDN_OK;
}

gdn_status gdn_decode_step(const void* q, const void* k, const void* v, gdn_dtype dtype, const float* a,
                           const float* b, const float* A_log, const float* dt_bias, float* state_pool,
                           int64_t pool_size, const int64_t* cache_indices, int32_t batch, void* out, int32_t H,
                           int32_t HV, int32_t K, int32_t V, float scale, int32_t* device_status, void* stream) {
  NvtxRange range("gdn_decode_step");
  if (batch < 0 || batch > kMaxDecodeBatch || H <= 0 || HV <= 0 || HV % H != 0 || K <= 0 || V <= 0)
    return GDN_ERR_INVALID_ARG;
  if ((int64_t)batch * HV > (int64_t)INT32_MAX) return GDN_ERR_INVALID_ARG;
  if (dtype != GDN_BF16 && dtype != GDN_FP16) return GDN_ERR_INVALID_ARG;
  if (!device_status || (reinterpret_cast<uintptr_t>(device_status) & 3u) != 0 || !A_log || !dt_bias)
    return GDN_ERR_INVALID_ARG;
  if (batch > 0 && (!q || !k || !v || !a || !b || !out || !state_pool || !cache_indices || pool_size <= 0))
    return GDN_ERR_INVALID_ARG;
  if (K != V || (K != 64 && K != 128 && K != 256)) return GDN_ERR_UNSUPPORTED;
  auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
  if (batch > 0 && !(al16(q) && al16(k) && al16(v) && al16(out) && al16(state_pool))) return GDN_ERR_INVALID_ARG;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  gdn::DecodeParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.a = a;
  p.b = b;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.state_pool = state_pool;
  p.cache_indices = cache_indices;
  p.out = out;
  p.pool_size = pool_size;
  p.B = batch;
  p.H = H;
  p.HV = HV;
  p.scale = scale;
  p.status = device_status;
  p.fp16 = dtype == GDN_FP16 ? 1 : 0;
  if (batch == 0 || gdn::decode_check_needs_zeroed_status(batch)) {
    if (cudaMemsetAsync(device_status, 0, sizeof(int32_t), s) != cudaSuccess) return GDN_ERR_CUDA;
    if (batch == 0) return GDN_OK;
  }
  {
    LaunchScope ls(kKernDecodeCheck, s);
    if (gdn::launch_decode_check(p, s) != cudaSuccess) return GDN_ERR_CUDA;
    ls.done();
  }
  {
    LaunchScope ls(kKernDecode, s);
    if (gdn::launch_decode(p, K, s) != cudaSuccess) return GDN_ERR_CUDA;
    ls.done();
  }
  return GDN_OK;
}

gdn_status gdn_get_device_status(const void* workspace, void* stream) {
  if (!workspace) return GDN_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t st = 0;
  if (cudaMemcpyAsync(&st, workspace, sizeof st, cudaMemcpyDeviceToHost, s) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
  if (st < 0 || st > GDN_ERR_BAD_SEQLENS) return GDN_ERR_CUDA;
  return static_cast<gdn_status>(st);
}

gdn_status gdn_workspace_layout(int64_t total_tokens, int32_t batch, int32_t H, int32_t HV, int32_t K, int32_t V,
                                int32_t chunk_size, gdn_workspace_layout_t* out) {
  if (!out) return GDN_ERR_INVALID_ARG;
  if (gdn_workspace_size(total_tokens, batch, H, HV, K, V, chunk_size) == 0) return GDN_ERR_UNSUPPORTED;
  const gdn::WsLayout L = gdn::make_layout(total_tokens, batch, H, HV, K, V, kWyBlock);
  out->status = L.status;
  out->chunk_tab = L.chunk_tab;
  out->g = L.g;
  out->beta = L.beta;
  out->rq = L.rq;
  out->rk = L.rk;
  out->ks = K == 128 ? L.ks : (size_t)-1;
  out->w = L.w;
  out->u = L.u;
  out->p = L.p;
  out->seg_state = L.seg_state;
  out->seg_map = L.seg_map;
  out->total = L.total;
  out->max_chunks = L.max_chunks;
  out->block = kWyBlock;
  out->affine_factors = K == 128 ? 1 : 0;
  out->nseg = L.nseg;
  return GDN_OK;
}

gdn_status gdn_test_set_stall(int32_t kernel, int64_t wait_budget_cycles) {
  if (kernel < gdn::kStallNone || kernel > gdn::kStallAffineScan || wait_budget_cycles <= 0)
    return GDN_ERR_INVALID_ARG;
  g_wait_budget.store(kernel == gdn::kStallNone ? gdn::kDefaultWaitBudget : wait_budget_cycles,
                      std::memory_order_relaxed);
  g_stall.store(kernel, std::memory_order_relaxed);
  return GDN_OK;
}

const char* gdn_status_string(gdn_status status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null pointer, bad size or HV not a multiple of H";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: head size or chunk size not built";
    case GDN_ERR_BAD_INDEX: return "GDN_ERR_BAD_INDEX: cache index out of range or repeated";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace null, too small or not 256-byte aligned";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device-side wait gave up";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA runtime call failed";
    case GDN_ERR_BAD_SEQLENS: return "GDN_ERR_BAD_SEQLENS: cu_seqlens not 0..total_tokens non-decreasing";
  }
  return "GDN_ERR_UNKNOWN";
}

gdn_status gdn_profile_start(int32_t max_launches) {
  if (max_launches <= 0) return GDN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  for (cudaEvent_t e : g_prof.pool) cudaEventDestroy(e);
  g_prof.pool.clear();
  g_prof.recs.clear();
  g_prof.on = false;
  for (int i = 0; i < 2 * max_launches; ++i) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) {
      for (cudaEvent_t x : g_prof.pool) cudaEventDestroy(x);
      g_prof.pool.clear();
      return GDN_ERR_CUDA;
    }
    g_prof.pool.push_back(e);
  }
  g_prof.recs.reserve(max_launches);
  g_prof.capacity = max_launches;
  g_prof.on = true;
  return GDN_OK;
}

int32_t gdn_profile_stop(double* total_ms, int64_t* launches, int32_t n_slots) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.on) return -1;
  g_prof.on = false;
  int ok = 1;
  for (int i = 0; i < n_slots; ++i) {
    if (total_ms) total_ms[i] = 0.0;
    if (launches) launches[i] = 0;
  }
  for (const ProfRecord& r : g_prof.recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
      ok = 0;
      continue;
    }
    if (r.id < n_slots) {
      if (total_ms) total_ms[r.id] += ms;
      if (launches) launches[r.id] += 1;
    }
  }
  for (cudaEvent_t e : g_prof.pool) cudaEventDestroy(e);
  g_prof.pool.clear();
  g_prof.recs.clear();
  return ok ? kKernCount : -1;
}

const char* gdn_kernel_name(int32_t id) { return (id >= 0 && id < kKernCount) ? kKernelNames[id] : nullptr; }

int64_t gdn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t gdn_version(void) { return 200; }

}  // extern "C"
