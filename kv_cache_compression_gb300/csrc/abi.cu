// C ABI of the SnapKV library: argument validation, workspace layout and launch order.
// Every argument error is found here, on the host, before anything is enqueued.
#include <math.h>
#include <stdint.h>
#include <stdio.h>

#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "snapkv_common.cuh"
#include "snapkv_internal.h"

namespace snapkv {

namespace {

constexpr int kVoteChunk = 1024;   // prompt columns per CTA of the score/vote kernels
constexpr int64_t kMaxPrompt = (int64_t)1 << 30;
constexpr int kMaxObs = 128;

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// An NVTX range around an entry point's host work (validation and enqueueing), so that a profiler's
// timeline shows which library call enqueued which kernels; without a tool attached it costs a few
// nanoseconds.
struct HostRange {
  explicit HostRange(const char* name) { nvtxRangePushA(name); }
  ~HostRange() { nvtxRangePop(); }
  HostRange(const HostRange&) = delete;
  HostRange& operator=(const HostRange&) = delete;
};

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + bn && b0 < a0 + an;
}

// V may be device memory or page-locked host memory mapped into the device's address space: the
// compression reads only the kept rows and the window rows of V, so a caller whose values live on
// the host need not copy the rest over the host link. Pageable host memory is refused. The query
// runs in relaxed capture mode, so that a call being captured into a CUDA graph may make it.
snapkv_status device_view_of_values(const void* v, const void** v_dev) {
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return SNAPKV_ERR_CUDA;
  cudaPointerAttributes at{};
  const cudaError_t e = cudaPointerGetAttributes(&at, v);
  cudaThreadExchangeStreamCaptureMode(&mode);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return e == cudaErrorInvalidValue ? SNAPKV_ERR_INVALID_ARG : SNAPKV_ERR_CUDA;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    *v_dev = v;
    return SNAPKV_OK;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer && aligned16(at.devicePointer)) {
    *v_dev = at.devicePointer;
    return SNAPKV_OK;
  }
  return SNAPKV_ERR_INVALID_ARG;
}

// Validates the problem statement (q_heads query heads share the params' KV heads); on success
// fills l_prefix, k_sel and the window-query rows per KV head.
snapkv_status check_params(const snapkv_compress_params* p, int32_t q_heads, int64_t* l_prefix, int64_t* k_sel,
                           int* q_rows) {
  if (!p) return SNAPKV_ERR_INVALID_ARG;
  if (q_heads < p->heads || p->heads < 1 || q_heads % p->heads != 0) return SNAPKV_ERR_INVALID_ARG;
  if (p->batch < 1 || p->heads < 1 || p->head_dim < 1 || p->l_obs < 1 || p->pool_kernel < 1)
    return SNAPKV_ERR_INVALID_ARG;
  if (p->l_prompt <= p->l_obs || p->l_prompt > kMaxPrompt) return SNAPKV_ERR_INVALID_ARG;
  if (p->softmax_scope != SNAPKV_SCOPE_PROMPT_CAUSAL && p->softmax_scope != SNAPKV_SCOPE_PREFIX_ONLY)
    return SNAPKV_ERR_INVALID_ARG;
  if (p->dtype != SNAPKV_F32 && p->dtype != SNAPKV_BF16) return SNAPKV_ERR_INVALID_ARG;
  if (p->algo < SNAPKV_ALGO_AUTO || p->algo > SNAPKV_ALGO_TENSOR_CORE_CLUSTER)
    return SNAPKV_ERR_INVALID_ARG;
  if (p->budget <= 0 && !(p->ratio_p >= 0.0 && p->ratio_p <= 1.0)) return SNAPKV_ERR_INVALID_ARG;
  if ((int64_t)p->batch * p->heads > 65535) return SNAPKV_ERR_INVALID_ARG;  // grid.y limit
  if (p->head_dim != 64 && p->head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  if (p->pool_kernel % 2 == 0) return SNAPKV_ERR_UNSUPPORTED;
  if (p->l_obs > kMaxObs || (int64_t)(q_heads / p->heads) * p->l_obs > kMaxObs) return SNAPKV_ERR_UNSUPPORTED;
  const int64_t lp = p->l_prompt - p->l_obs;
  int64_t k;
  if (p->budget > 0)
    k = p->budget < lp ? p->budget : lp;
  else
    k = (int64_t)floor(p->ratio_p * (double)lp);
  if (k < 0) k = 0;
  if (k > lp) k = lp;
  *l_prefix = lp;
  *k_sel = k;
  *q_rows = (q_heads / p->heads) * p->l_obs;
  return SNAPKV_OK;
}

}  // namespace

CompressLayout compress_layout(int batch, int heads, int l_obs, int q_rows, int64_t l_prompt, int64_t k_sel) {
  CompressLayout L;
  const size_t bh = (size_t)batch * heads;
  const int64_t l_prefix = l_prompt - l_obs;
  L.vote_chunk = kVoteChunk;
  L.n_chunk_all = (int)((l_prompt + kVoteChunk - 1) / kVoteChunk);
  L.n_chunk_prefix = (int)((l_prefix + kVoteChunk - 1) / kVoteChunk);
  const int64_t kpi = vote_tc_keys_per_item(q_rows, l_obs);
  const int64_t tc_items = (l_prompt + kpi - 1) / kpi;
  const int64_t chunks = tc_items > L.n_chunk_all ? tc_items : L.n_chunk_all;
  L.partial = 0;
  L.c = up256(bh * chunks * q_rows * 2 * sizeof(float));
  L.p = L.c + up256(bh * l_prefix * sizeof(float));
  L.idx = L.p + up256(bh * l_prefix * sizeof(float));
  const size_t group = (size_t)(q_rows / l_obs);   // query heads per KV head
  // per-query-head votes of the tensor-core path under grouped-query attention
  L.c_q = L.idx + up256(bh * (k_sel > 0 ? k_sel : 1) * sizeof(int32_t));
  L.tc_zsum = L.c_q + (group > 1 ? up256(bh * group * l_prefix * sizeof(float)) : 0);
  L.tc_counters = L.tc_zsum + up256(bh * q_rows * sizeof(double));
  L.total = L.tc_counters + up256(bh * group * sizeof(uint32_t));
  return L;
}

}  // namespace snapkv

using namespace snapkv;

extern "C" {

int32_t snapkv_abi_version(void) { return 100; }

const char* snapkv_status_string(int32_t status) {
  switch (status) {
    case SNAPKV_OK: return "SNAPKV_OK";
    case SNAPKV_ERR_INVALID_ARG: return "SNAPKV_ERR_INVALID_ARG";
    case SNAPKV_ERR_UNSUPPORTED: return "SNAPKV_ERR_UNSUPPORTED";
    case SNAPKV_ERR_CAPACITY: return "SNAPKV_ERR_CAPACITY";
    case SNAPKV_ERR_CUDA: return "SNAPKV_ERR_CUDA";
    case SNAPKV_ERR_TIMEOUT: return "SNAPKV_ERR_TIMEOUT";
    case SNAPKV_ERR_WORKSPACE: return "SNAPKV_ERR_WORKSPACE";
    case SNAPKV_ERR_INTERNAL: return "SNAPKV_ERR_INTERNAL";
    default: break;
  }
  if (status < 0 || status > 127) return "SNAPKV_ERR_UNKNOWN";
  // Several bits: a fixed table of combinations is not worth it; name the highest-priority one.
  if (status & SNAPKV_ERR_INTERNAL) return "SNAPKV_ERR_INTERNAL|...";
  if (status & SNAPKV_ERR_TIMEOUT) return "SNAPKV_ERR_TIMEOUT|...";
  if (status & SNAPKV_ERR_CUDA) return "SNAPKV_ERR_CUDA|...";
  if (status & SNAPKV_ERR_CAPACITY) return "SNAPKV_ERR_CAPACITY|...";
  if (status & SNAPKV_ERR_WORKSPACE) return "SNAPKV_ERR_WORKSPACE|...";
  if (status & SNAPKV_ERR_UNSUPPORTED) return "SNAPKV_ERR_UNSUPPORTED|...";
  return "SNAPKV_ERR_INVALID_ARG|...";
}

int64_t snapkv_compress_kept(const snapkv_compress_params* params) {
  int64_t lp = 0, k = 0;
  int rows = 0;
  if (!params || check_params(params, params->heads, &lp, &k, &rows) != SNAPKV_OK) return -1;
  return k;
}

int64_t snapkv_compress_k(const snapkv_compress_params* params) { return snapkv_compress_kept(params); }

size_t snapkv_compress_gqa_workspace_size(const snapkv_compress_params* params, int32_t q_heads) {
  int64_t lp = 0, k = 0;
  int rows = 0;
  if (!params || check_params(params, q_heads, &lp, &k, &rows) != SNAPKV_OK) return 0;
  return compress_layout(params->batch, params->heads, params->l_obs, rows, params->l_prompt, k).total;
}

size_t snapkv_compress_workspace_size(const snapkv_compress_params* params) {
  return params ? snapkv_compress_gqa_workspace_size(params, params->heads) : 0;
}

}  // extern "C"

namespace {

// The stage kernels of one validated compression job, in stream order.
snapkv_status run_compress(const CompressJob& job, int algo) {
  const bool cl_ok = algo == SNAPKV_ALGO_TENSOR_CORE_CLUSTER && vote_cluster_eligible(job);
  const bool tc_ok = (algo == SNAPKV_ALGO_AUTO || algo == SNAPKV_ALGO_TENSOR_CORE) && vote_tc_eligible(job);
  const bool tc_only = algo == SNAPKV_ALGO_TENSOR_CORE || algo == SNAPKV_ALGO_TENSOR_CORE_CLUSTER;
  if (tc_only && !cl_ok && !tc_ok) return SNAPKV_ERR_UNSUPPORTED;
  bool voted = false;
  if (cl_ok) {
    if (launch_vote_cluster(job) == cudaSuccess) voted = true;
    else cudaGetLastError();   // a refused launch is not sticky; try the next kernel
  }
  if (!voted && tc_ok) {
    if (launch_vote_tc(job) == cudaSuccess) voted = true;
    else cudaGetLastError();
  }
  if (!voted && tc_only) return SNAPKV_ERR_CUDA;
  if (!voted && launch_vote_simt(job) != cudaSuccess) return SNAPKV_ERR_CUDA;
  bool gathered = false;
  if (launch_pool_topk(job, &gathered) != cudaSuccess) return SNAPKV_ERR_CUDA;
  if (gathered) {   // the gather stage ran inside the top-k kernel
    job.mark(2 * kStageGather);
    job.mark(2 * kStageGather + 1);
  } else if (launch_gather(job) != cudaSuccess) {
    return SNAPKV_ERR_CUDA;
  }
  return SNAPKV_OK;
}

snapkv_status compress_impl(const snapkv_compress_params* params, int32_t q_heads, const void* q_obs, const void* k,
                            const void* v, void* k_out, void* v_out, int64_t cap, int32_t* len_out, int32_t* idx_out,
                            float* vote_out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            snapkv_stream_t stream, void* const* stage_events, int32_t n_events) {
  if (n_events < 0 || (n_events > 0 && !stage_events)) return SNAPKV_ERR_INVALID_ARG;
  int64_t l_prefix = 0, k_sel = 0;
  int q_rows = 0;
  const snapkv_status st = check_params(params, q_heads, &l_prefix, &k_sel, &q_rows);
  if (st != SNAPKV_OK) return st;
  if (!q_obs || !k || !v || !k_out || !v_out || !len_out) return SNAPKV_ERR_INVALID_ARG;
  if (!aligned16(q_obs) || !aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out))
    return SNAPKV_ERR_INVALID_ARG;
  if (((uintptr_t)len_out & 3u) || ((uintptr_t)idx_out & 3u) || ((uintptr_t)vote_out & 3u) ||
      ((uintptr_t)dev_status & 3u))
    return SNAPKV_ERR_INVALID_ARG;
  if (cap < k_sel + params->l_obs || cap > kMaxPrompt) return SNAPKV_ERR_CAPACITY;
  const CompressLayout L =
      compress_layout(params->batch, params->heads, params->l_obs, q_rows, params->l_prompt, k_sel);
  if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u)) return SNAPKV_ERR_WORKSPACE;

  const size_t esize = params->dtype == SNAPKV_BF16 ? 2 : 4;
  const size_t bh = (size_t)params->batch * params->heads;
  const size_t in_bytes = bh * (size_t)params->l_prompt * params->head_dim * esize;
  const size_t out_bytes = bh * (size_t)cap * params->head_dim * esize;
  if (overlaps(k, in_bytes, k_out, out_bytes) || overlaps(k, in_bytes, v_out, out_bytes) ||
      overlaps(v, in_bytes, k_out, out_bytes) || overlaps(v, in_bytes, v_out, out_bytes) ||
      overlaps(k_out, out_bytes, v_out, out_bytes))
    return SNAPKV_ERR_INVALID_ARG;
  const snapkv_status vs = device_view_of_values(v, &v);
  if (vs != SNAPKV_OK) return vs;

  char* ws = static_cast<char*>(workspace);
  CompressJob job;
  job.batch = params->batch;
  job.heads = params->heads;
  job.head_dim = params->head_dim;
  job.l_obs = params->l_obs;
  job.q_rows = q_rows;
  job.pool_kernel = params->pool_kernel;
  job.scope = params->softmax_scope;
  job.dtype = params->dtype;
  job.l_prompt = params->l_prompt;
  job.kv_stride = params->l_prompt;
  job.l_prefix = l_prefix;
  job.k_sel = k_sel;
  job.cap = cap;
  job.q_obs = q_obs;
  job.k = k;
  job.v = v;
  job.k_out = k_out;
  job.v_out = v_out;
  job.len_out = len_out;
  job.idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + L.idx);
  job.c = vote_out ? vote_out : reinterpret_cast<float*>(ws + L.c);
  job.p = reinterpret_cast<float*>(ws + L.p);
  job.partial = reinterpret_cast<float*>(ws + L.partial);
  job.c_q = reinterpret_cast<float*>(ws + L.c_q);
  job.tc_zsum = reinterpret_cast<double*>(ws + L.tc_zsum);
  job.tc_cnt = reinterpret_cast<uint32_t*>(ws + L.tc_counters);
  job.tc_zero_bytes = L.total - L.tc_zsum;
  job.vote_chunk = L.vote_chunk;
  job.n_chunk_all = L.n_chunk_all;
  job.n_chunk_prefix = L.n_chunk_prefix;
  job.dev_status = dev_status;
  job.stream = reinterpret_cast<cudaStream_t>(stream);
  job.events = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(stage_events));
  job.n_events = n_events;

  return run_compress(job, params->algo);
}

}  // namespace

extern "C" {

snapkv_status snapkv_compress_profiled(const snapkv_compress_params* params, const void* q_obs, const void* k,
                                       const void* v, void* k_out, void* v_out, int64_t cap, int32_t* len_out,
                                       int32_t* idx_out, float* vote_out, void* workspace, size_t workspace_bytes,
                                       int32_t* dev_status, snapkv_stream_t stream, void* const* stage_events,
                                       int32_t n_events) {
  HostRange nvtx_range("snapkv_compress");
  if (!params) return SNAPKV_ERR_INVALID_ARG;
  return compress_impl(params, params->heads, q_obs, k, v, k_out, v_out, cap, len_out, idx_out, vote_out, workspace,
                       workspace_bytes, dev_status, stream, stage_events, n_events);
}

snapkv_status snapkv_compress_gqa(const snapkv_compress_params* params, int32_t q_heads, const void* q_obs,
                                  const void* k, const void* v, void* k_out, void* v_out, int64_t cap,
                                  int32_t* len_out, int32_t* idx_out, float* vote_out, void* workspace,
                                  size_t workspace_bytes, int32_t* dev_status, snapkv_stream_t stream) {
  HostRange nvtx_range("snapkv_compress_gqa");
  return compress_impl(params, q_heads, q_obs, k, v, k_out, v_out, cap, len_out, idx_out, vote_out, workspace,
                       workspace_bytes, dev_status, stream, nullptr, 0);
}

size_t snapkv_compress_varlen_workspace_size(const snapkv_compress_params* params, const int64_t* l_prompts) {
  int64_t lp = 0, k = 0;
  int rows = 0;
  if (!params || !l_prompts || check_params(params, params->heads, &lp, &k, &rows) != SNAPKV_OK) return 0;
  size_t need = 0;
  for (int32_t b = 0; b < params->batch; ++b) {
    snapkv_compress_params pb = *params;
    pb.batch = 1;
    pb.l_prompt = l_prompts[b];
    if (pb.l_prompt > params->l_prompt || check_params(&pb, pb.heads, &lp, &k, &rows) != SNAPKV_OK) return 0;
    const size_t t = compress_layout(1, pb.heads, pb.l_obs, rows, pb.l_prompt, k).total;
    if (t > need) need = t;
  }
  // One launch over the whole batch lays the batch out with the longest sequence's sizes.
  int64_t lp_max = 0, k_max = 0;
  check_params(params, params->heads, &lp_max, &k_max, &rows);
  const size_t all = compress_layout(params->batch, params->heads, params->l_obs, rows, params->l_prompt, k_max).total;
  return all > need ? all : need;
}

snapkv_status snapkv_compress_varlen(const snapkv_compress_params* params, const int64_t* l_prompts,
                                     const void* q_obs, const void* k, const void* v, void* k_out, void* v_out,
                                     int64_t cap, int32_t* len_out, int32_t* idx_out, float* vote_out,
                                     void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                     snapkv_stream_t stream) {
  HostRange nvtx_range("snapkv_compress_varlen");
  int64_t lp_max = 0, k_max = 0;
  int rows = 0;
  if (!params || !l_prompts) return SNAPKV_ERR_INVALID_ARG;
  const snapkv_status st = check_params(params, params->heads, &lp_max, &k_max, &rows);
  if (st != SNAPKV_OK) return st;
  if (!q_obs || !k || !v || !k_out || !v_out || !len_out) return SNAPKV_ERR_INVALID_ARG;
  if (!aligned16(q_obs) || !aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out))
    return SNAPKV_ERR_INVALID_ARG;
  if (((uintptr_t)len_out & 3u) || ((uintptr_t)idx_out & 3u) || ((uintptr_t)vote_out & 3u) ||
      ((uintptr_t)dev_status & 3u))
    return SNAPKV_ERR_INVALID_ARG;
  const size_t need = snapkv_compress_varlen_workspace_size(params, l_prompts);
  if (need == 0) return SNAPKV_ERR_INVALID_ARG;   // a sequence length outside [L_obs + 1, params->l_prompt]
  if (cap < k_max + params->l_obs || cap > kMaxPrompt) return SNAPKV_ERR_CAPACITY;   // k grows with L
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255u)) return SNAPKV_ERR_WORKSPACE;
  const size_t esize = params->dtype == SNAPKV_BF16 ? 2 : 4;
  const size_t H = (size_t)params->heads, d = (size_t)params->head_dim;
  const size_t in_bytes = params->batch * H * (size_t)params->l_prompt * d * esize;
  const size_t out_bytes = params->batch * H * (size_t)cap * d * esize;
  if (overlaps(k, in_bytes, k_out, out_bytes) || overlaps(k, in_bytes, v_out, out_bytes) ||
      overlaps(v, in_bytes, k_out, out_bytes) || overlaps(v, in_bytes, v_out, out_bytes) ||
      overlaps(k_out, out_bytes, v_out, out_bytes))
    return SNAPKV_ERR_INVALID_ARG;
  const snapkv_status vs = device_view_of_values(v, &v);
  if (vs != SNAPKV_OK) return vs;

  const cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);

  // The whole ragged batch in one launch of the score/vote kernel and one of the top-k kernel,
  // when the tensor-core path takes it (every sequence keeps at least one row, and the longest
  // fits the resident queue); otherwise one compression per sequence, one after another.
  std::vector<int64_t> ks((size_t)params->batch);
  for (int32_t b = 0; b < params->batch; ++b) {
    snapkv_compress_params pb = *params;
    pb.batch = 1;
    pb.l_prompt = l_prompts[b];
    int64_t lpb = 0;
    int rows_b = 0;
    check_params(&pb, pb.heads, &lpb, &ks[(size_t)b], &rows_b);   // validated above
  }
  if (params->algo == SNAPKV_ALGO_AUTO || params->algo == SNAPKV_ALGO_TENSOR_CORE) {
    const CompressLayout L = compress_layout(params->batch, params->heads, params->l_obs, rows, params->l_prompt, k_max);
    CompressJob job;
    job.batch = params->batch;
    job.heads = params->heads;
    job.head_dim = params->head_dim;
    job.l_obs = params->l_obs;
    job.q_rows = rows;
    job.pool_kernel = params->pool_kernel;
    job.scope = params->softmax_scope;
    job.dtype = params->dtype;
    job.l_prompt = params->l_prompt;
    job.kv_stride = params->l_prompt;
    job.l_prefix = lp_max;
    job.k_sel = k_max;
    job.cap = cap;
    job.q_obs = q_obs;
    job.k = k;
    job.v = v;
    job.k_out = k_out;
    job.v_out = v_out;
    job.len_out = len_out;
    job.idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + L.idx);
    job.c = vote_out ? vote_out : reinterpret_cast<float*>(ws + L.c);
    job.p = reinterpret_cast<float*>(ws + L.p);
    job.partial = reinterpret_cast<float*>(ws + L.partial);
    job.c_q = reinterpret_cast<float*>(ws + L.c_q);
    job.tc_zsum = reinterpret_cast<double*>(ws + L.tc_zsum);
    job.tc_cnt = reinterpret_cast<uint32_t*>(ws + L.tc_counters);
    job.tc_zero_bytes = L.total - L.tc_zsum;
    job.vote_chunk = L.vote_chunk;
    job.n_chunk_all = L.n_chunk_all;
    job.n_chunk_prefix = L.n_chunk_prefix;
    job.dev_status = dev_status;
    job.stream = strm;
    job.events = nullptr;
    job.n_events = 0;
    job.n_var = params->batch;
    job.var_l_prompt = l_prompts;
    job.var_k = ks.data();
    if (vote_tc_ragged_eligible(job) && pool_topk_ragged_eligible(job)) {
      if (launch_vote_tc(job) != cudaSuccess) return SNAPKV_ERR_CUDA;
      bool gathered = false;
      if (launch_pool_topk(job, &gathered) != cudaSuccess || !gathered) return SNAPKV_ERR_CUDA;
      return SNAPKV_OK;
    }
  }

  for (int32_t b = 0; b < params->batch; ++b) {
    snapkv_compress_params pb = *params;
    pb.batch = 1;
    pb.l_prompt = l_prompts[b];
    int64_t l_prefix = 0, k_sel = 0;
    int q_rows = 0;
    check_params(&pb, pb.heads, &l_prefix, &k_sel, &q_rows);   // validated above
    const CompressLayout L = compress_layout(1, pb.heads, pb.l_obs, q_rows, pb.l_prompt, k_sel);
    CompressJob job;
    job.batch = 1;
    job.heads = pb.heads;
    job.head_dim = pb.head_dim;
    job.l_obs = pb.l_obs;
    job.q_rows = q_rows;
    job.pool_kernel = pb.pool_kernel;
    job.scope = pb.softmax_scope;
    job.dtype = pb.dtype;
    job.l_prompt = pb.l_prompt;
    job.kv_stride = params->l_prompt;   // the padded batch's row stride
    job.l_prefix = l_prefix;
    job.k_sel = k_sel;
    job.cap = cap;
    job.q_obs = static_cast<const char*>(q_obs) + (size_t)b * H * pb.l_obs * d * esize;
    job.k = static_cast<const char*>(k) + (size_t)b * H * params->l_prompt * d * esize;
    job.v = static_cast<const char*>(v) + (size_t)b * H * params->l_prompt * d * esize;
    job.k_out = static_cast<char*>(k_out) + (size_t)b * H * cap * d * esize;
    job.v_out = static_cast<char*>(v_out) + (size_t)b * H * cap * d * esize;
    job.len_out = len_out + b;
    job.idx = reinterpret_cast<int32_t*>(ws + L.idx);
    job.c = reinterpret_cast<float*>(ws + L.c);
    job.p = reinterpret_cast<float*>(ws + L.p);
    job.partial = reinterpret_cast<float*>(ws + L.partial);
    job.c_q = reinterpret_cast<float*>(ws + L.c_q);
    job.tc_zsum = reinterpret_cast<double*>(ws + L.tc_zsum);
    job.tc_cnt = reinterpret_cast<uint32_t*>(ws + L.tc_counters);
    job.tc_zero_bytes = L.total - L.tc_zsum;
    job.vote_chunk = L.vote_chunk;
    job.n_chunk_all = L.n_chunk_all;
    job.n_chunk_prefix = L.n_chunk_prefix;
    job.dev_status = dev_status;
    job.stream = strm;
    job.events = nullptr;
    job.n_events = 0;
    const snapkv_status r = run_compress(job, pb.algo);
    if (r != SNAPKV_OK) return r;
    // This sequence's indices and vote into the caller's [B, H, k_max] and [B, H, L_prefix_max].
    if (idx_out && k_sel > 0 &&
        cudaMemcpy2DAsync(idx_out + (size_t)b * H * k_max, (size_t)k_max * 4, job.idx, (size_t)k_sel * 4,
                          (size_t)k_sel * 4, H, cudaMemcpyDeviceToDevice, strm) != cudaSuccess)
      return SNAPKV_ERR_CUDA;
    if (vote_out &&
        cudaMemcpy2DAsync(vote_out + (size_t)b * H * lp_max, (size_t)lp_max * 4, job.c, (size_t)l_prefix * 4,
                          (size_t)l_prefix * 4, H, cudaMemcpyDeviceToDevice, strm) != cudaSuccess)
      return SNAPKV_ERR_CUDA;
  }
  return SNAPKV_OK;
}

snapkv_status snapkv_compress(const snapkv_compress_params* params, const void* q_obs, const void* k,
                              const void* v, void* k_out, void* v_out, int64_t cap, int32_t* len_out,
                              int32_t* idx_out, float* vote_out, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, snapkv_stream_t stream) {
  return snapkv_compress_profiled(params, q_obs, k, v, k_out, v_out, cap, len_out, idx_out, vote_out, workspace,
                                  workspace_bytes, dev_status, stream, nullptr, 0);
}

snapkv_status snapkv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int64_t cap,
                            int32_t* len, int32_t batch, int32_t heads, int32_t head_dim, int32_t dtype,
                            int32_t* dev_status, snapkv_stream_t stream) {
  HostRange nvtx_range("snapkv_append");
  if (!k_new || !v_new || !k_cache || !v_cache || !len) return SNAPKV_ERR_INVALID_ARG;
  if (batch < 1 || heads < 1 || head_dim < 1 || cap < 1 || cap > kMaxPrompt) return SNAPKV_ERR_INVALID_ARG;
  if (dtype != SNAPKV_F32 && dtype != SNAPKV_BF16) return SNAPKV_ERR_INVALID_ARG;
  if ((int64_t)batch * heads > 65535) return SNAPKV_ERR_INVALID_ARG;  // grid.y limit
  if (head_dim != 64 && head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      ((uintptr_t)len & 3u) || ((uintptr_t)dev_status & 3u))
    return SNAPKV_ERR_INVALID_ARG;
  if (launch_append(k_new, v_new, k_cache, v_cache, cap, len, batch, heads, head_dim, dtype, dev_status,
                    reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SNAPKV_ERR_CUDA;
  return SNAPKV_OK;
}

size_t snapkv_decode_workspace_size(int32_t batch, int32_t heads, int32_t head_dim, int64_t cap) {
  if (batch < 1 || heads < 1 || cap < 1 || cap > kMaxPrompt) return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  return decode_layout(batch, heads, head_dim, cap).total;
}

snapkv_status snapkv_decode_attend(const void* q, const void* k_cache, const void* v_cache, int64_t cap,
                                   const int32_t* len, void* out, int32_t batch, int32_t heads, int32_t head_dim,
                                   int32_t dtype, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                   snapkv_stream_t stream) {
  HostRange nvtx_range("snapkv_decode_attend");
  if (!q || !k_cache || !v_cache || !len || !out) return SNAPKV_ERR_INVALID_ARG;
  if (batch < 1 || heads < 1 || head_dim < 1 || cap < 1 || cap > kMaxPrompt) return SNAPKV_ERR_INVALID_ARG;
  if (dtype != SNAPKV_F32 && dtype != SNAPKV_BF16) return SNAPKV_ERR_INVALID_ARG;
  if ((int64_t)batch * heads > 65535) return SNAPKV_ERR_INVALID_ARG;  // grid.y limit
  if (head_dim != 64 && head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || ((uintptr_t)len & 3u) ||
      ((uintptr_t)dev_status & 3u))
    return SNAPKV_ERR_INVALID_ARG;
  const DecodeLayout L = decode_layout(batch, heads, head_dim, cap);
  if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u)) return SNAPKV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  DecodeJob job;
  job.batch = batch;
  job.heads = heads;
  job.head_dim = head_dim;
  job.dtype = dtype;
  job.cap = cap;
  job.q = q;
  job.k_cache = k_cache;
  job.v_cache = v_cache;
  job.len = len;
  job.out = out;
  job.partial = reinterpret_cast<float*>(ws + L.partial);
  job.tickets = reinterpret_cast<uint32_t*>(ws + L.tickets);
  job.split_rows = L.split_rows;
  job.n_split = L.n_split;
  job.dev_status = dev_status;
  job.stream = reinterpret_cast<cudaStream_t>(stream);
  if (launch_decode(job) != cudaSuccess) return SNAPKV_ERR_CUDA;
  return SNAPKV_OK;
}

snapkv_status snapkv_append_decode_attend(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                          void* v_cache, int64_t cap, const int32_t* len_in, int32_t* len_out,
                                          void* out, int32_t batch, int32_t heads, int32_t head_dim, int32_t dtype,
                                          void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                          snapkv_stream_t stream) {
  HostRange nvtx_range("snapkv_append_decode_attend");
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !len_in || !len_out || !out) return SNAPKV_ERR_INVALID_ARG;
  if (batch < 1 || heads < 1 || head_dim < 1 || cap < 1 || cap > kMaxPrompt) return SNAPKV_ERR_INVALID_ARG;
  if (dtype != SNAPKV_F32 && dtype != SNAPKV_BF16) return SNAPKV_ERR_INVALID_ARG;
  if ((int64_t)batch * heads > 65535) return SNAPKV_ERR_INVALID_ARG;  // grid.y limit
  if (head_dim != 64 && head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(out) || ((uintptr_t)len_in & 3u) || ((uintptr_t)len_out & 3u) || ((uintptr_t)dev_status & 3u))
    return SNAPKV_ERR_INVALID_ARG;
  // Every head reads len_in[b] while the new lengths are written: the two arrays must not overlap.
  if (overlaps(len_in, (size_t)batch * 4, len_out, (size_t)batch * 4)) return SNAPKV_ERR_INVALID_ARG;
  const DecodeLayout L = decode_layout(batch, heads, head_dim, cap);
  if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255u)) return SNAPKV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  const cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
  DecodeJob job;
  job.batch = batch;
  job.heads = heads;
  job.head_dim = head_dim;
  job.dtype = dtype;
  job.cap = cap;
  job.q = q;
  job.k_cache = k_cache;
  job.v_cache = v_cache;
  job.len = len_in;
  job.out = out;
  job.partial = reinterpret_cast<float*>(ws + L.partial);
  job.tickets = reinterpret_cast<uint32_t*>(ws + L.tickets);
  job.split_rows = L.split_rows;
  job.n_split = L.n_split;
  job.dev_status = dev_status;
  job.stream = strm;
  if (cap <= decode_fuses_append_max_cap()) {   // one launch: the decode kernel appends first
    job.k_new = k_new;
    job.v_new = v_new;
    job.len_out = len_out;
  } else {   // longer caches: the new lengths start as a copy, the append kernel then updates them
    if (cudaMemcpyAsync(len_out, len_in, (size_t)batch * 4, cudaMemcpyDeviceToDevice, strm) != cudaSuccess)
      return SNAPKV_ERR_CUDA;
    if (launch_append(k_new, v_new, k_cache, v_cache, cap, len_out, batch, heads, head_dim, dtype, dev_status,
                      strm) != cudaSuccess)
      return SNAPKV_ERR_CUDA;
    job.len = len_out;
  }
  if (launch_decode(job) != cudaSuccess) return SNAPKV_ERR_CUDA;
  return SNAPKV_OK;
}

snapkv_status snapkv_decode_attend_noalloc(const void* q, const void* k_cache, const void* v_cache, int64_t cap,
                                           const int32_t* len, void* out, int32_t batch, int32_t heads,
                                           int32_t head_dim, int32_t dtype, int32_t* dev_status,
                                           snapkv_stream_t stream) {
  HostRange nvtx_range("snapkv_decode_attend_noalloc");
  if (!q || !k_cache || !v_cache || !len || !out) return SNAPKV_ERR_INVALID_ARG;
  if (batch < 1 || heads < 1 || head_dim < 1 || cap < 1 || cap > kMaxPrompt) return SNAPKV_ERR_INVALID_ARG;
  if (dtype != SNAPKV_F32 && dtype != SNAPKV_BF16) return SNAPKV_ERR_INVALID_ARG;
  if ((int64_t)batch * heads > 65535) return SNAPKV_ERR_INVALID_ARG;  // grid.y limit
  if (head_dim != 64 && head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || ((uintptr_t)len & 3u) ||
      ((uintptr_t)dev_status & 3u))
    return SNAPKV_ERR_INVALID_ARG;
  // Only caches longer than the cluster kernel's limit take the split kernel, which keeps partials
  // and tickets in the built-in array; shorter ones need no scratch at all.
  if (cap > decode_fuses_append_max_cap() &&
      decode_layout(batch, heads, head_dim, cap).total > kDecodeNoAllocScratchBytes)
    return SNAPKV_ERR_WORKSPACE;
  DecodeJob job;
  job.batch = batch;
  job.heads = heads;
  job.head_dim = head_dim;
  job.dtype = dtype;
  job.cap = cap;
  job.q = q;
  job.k_cache = k_cache;
  job.v_cache = v_cache;
  job.len = len;
  job.out = out;
  job.partial = nullptr;
  job.tickets = nullptr;
  job.split_rows = 0;
  job.n_split = 0;
  job.dev_status = dev_status;
  job.stream = reinterpret_cast<cudaStream_t>(stream);
  if (launch_decode_noalloc(job) != cudaSuccess) return SNAPKV_ERR_CUDA;
  return SNAPKV_OK;
}

snapkv_status snapkv_hit_rate(const void* q, const void* k_cache, int64_t cap, const int32_t* len, int64_t l_prefix,
                              const int32_t* idx, int64_t k, int32_t batch, int32_t heads, int32_t head_dim,
                              int32_t dtype, double theta, int32_t* hits, int32_t* total, int32_t* dev_status,
                              snapkv_stream_t stream) {
  HostRange nvtx_range("snapkv_hit_rate");
  if (!q || !k_cache || !len || !hits || !total || (k > 0 && !idx)) return SNAPKV_ERR_INVALID_ARG;
  if (batch < 1 || heads < 1 || cap < 1 || cap > kMaxPrompt || k < 0) return SNAPKV_ERR_INVALID_ARG;
  if ((int64_t)batch * heads > 2147483647LL) return SNAPKV_ERR_INVALID_ARG;
  if (l_prefix < 1 || l_prefix > cap || l_prefix > ((int64_t)1 << 20)) return SNAPKV_ERR_INVALID_ARG;
  if (!(theta >= 0.0)) return SNAPKV_ERR_INVALID_ARG;
  if (dtype != SNAPKV_F32 && dtype != SNAPKV_BF16) return SNAPKV_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return SNAPKV_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || ((uintptr_t)len & 3u) || ((uintptr_t)idx & 3u) ||
      ((uintptr_t)hits & 3u) || ((uintptr_t)total & 3u) || ((uintptr_t)dev_status & 3u))
    return SNAPKV_ERR_INVALID_ARG;
  HitRateJob job;
  job.batch = batch;
  job.heads = heads;
  job.head_dim = head_dim;
  job.dtype = dtype;
  job.cap = cap;
  job.l_prefix = l_prefix;
  job.k_sel = k;
  job.theta = theta;
  job.q = q;
  job.k_cache = k_cache;
  job.len = len;
  job.idx = idx;
  job.hits = hits;
  job.total = total;
  job.dev_status = dev_status;
  job.stream = reinterpret_cast<cudaStream_t>(stream);
  if (launch_hit_rate(job) != cudaSuccess) return SNAPKV_ERR_CUDA;
  return SNAPKV_OK;
}

}  // extern "C"
