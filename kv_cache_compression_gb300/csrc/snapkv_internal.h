// Internal launcher interface between the C ABI layer (abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace snapkv {

// Sequences of a ragged batch that the score/vote and top-k kernels take in one launch.
constexpr int kMaxVarSeq = 64;

// One compression call, after host-side validation.
struct CompressJob {
  int batch, heads, head_dim, l_obs, pool_kernel, scope, dtype;
  int q_rows;          // window-query rows per KV head: (query heads / KV heads) * l_obs
  int64_t l_prompt, l_prefix, k_sel, cap;
  int64_t kv_stride;   // rows between heads in k and v (>= l_prompt; larger for padded varlen batches)
  // Ragged batch in one launch (n_var > 0, at most kMaxVarSeq): sequence b has var_l_prompt[b]
  // prompt rows and keeps var_k[b] prefix rows; l_prompt, l_prefix and k_sel then hold the maxima,
  // which are also the row strides of the vote (c) and of the indices (idx).
  int n_var = 0;
  const int64_t* var_l_prompt = nullptr;   // host array [batch]
  const int64_t* var_k = nullptr;          // host array [batch]
  const void* q_obs;
  const void* k;
  const void* v;
  void* k_out;
  void* v_out;
  int32_t* len_out;
  int32_t* idx;        // kept indices (caller's buffer or workspace)
  float* c;            // vote (caller's buffer or workspace)
  float* c_q;          // per-query-head votes under grouped-query attention (workspace)
  float* p;            // pooled vote (workspace)
  float* partial;      // per-chunk row statistics (workspace)
  double* tc_zsum;     // per-(head, row) fp64 sums of 2^(logit) (workspace; zeroed per call)
  uint32_t* tc_cnt;    // per-head statistics items done (workspace, right after tc_zsum)
  size_t tc_zero_bytes;   // bytes from tc_zsum through the counters, cleared before the kernel
  int vote_chunk;      // keys per chunk of the score/vote kernels
  int n_chunk_all;     // chunks covering the whole prompt
  int n_chunk_prefix;  // chunks covering the prefix
  int32_t* dev_status;
  cudaStream_t stream;
  cudaEvent_t* events;  // optional stage events (see snapkv_compress_profiled), may be null
  int n_events;
  // Records stage event `slot`. Inside a stream capture the record becomes an event-record node of
  // the graph (an external event), so that replays of the graph time the stage too.
  void mark(int slot) const {
    if (!events || slot >= n_events || !events[slot]) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags(events[slot], stream, cudaEventRecordExternal);
    else
      cudaEventRecord(events[slot], stream);
  }
};

// Stage event slots: events[2s] before and events[2s+1] after the kernels of stage s.
enum { kStageScore = 0, kStageVote = 1, kStageTopk = 2, kStageGather = 3, kStages = 4 };

// Workspace layout of a compression call (byte offsets, each 256-aligned).
struct CompressLayout {
  size_t partial, c, p, idx, c_q, tc_zsum, tc_counters, total;
  int vote_chunk, n_chunk_all, n_chunk_prefix;
};

CompressLayout compress_layout(int batch, int heads, int l_obs, int q_rows, int64_t l_prompt, int64_t k_sel);

cudaError_t launch_vote_simt(const CompressJob& job);
// Tensor-core score + vote (bf16, d 64/128, L_obs <= 64, items per head <= 2 x SMs).
bool vote_tc_eligible(const CompressJob& job);
// The cluster-per-head tensor-core kernel (a head's keys fit 8 CTAs x 4 TMEM slots).
bool vote_cluster_eligible(const CompressJob& job);
cudaError_t launch_vote_cluster(const CompressJob& job);
int vote_tc_keys_per_item(int q_rows, int l_obs);
cudaError_t launch_vote_tc(const CompressJob& job);
// Whether a ragged batch (job.n_var > 0, maxima in l_prompt / l_prefix / k_sel) can take one
// launch of the score/vote kernel and one of the cluster top-k kernel.
bool vote_tc_ragged_eligible(const CompressJob& job);
bool pool_topk_ragged_eligible(const CompressJob& job);
// Max-pool + top-k; for prefixes the cluster kernel handles it also writes K_c, V_c and len_out
// (*gathered = true), otherwise launch_gather must follow.
cudaError_t launch_pool_topk(const CompressJob& job, bool* gathered);
cudaError_t launch_gather(const CompressJob& job);

struct DecodeJob {
  int batch, heads, head_dim, dtype;
  int64_t cap;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* len;
  void* out;
  float* partial;       // [B*H][n_split][d + 2]
  uint32_t* tickets;    // [B*H]
  int split_rows, n_split;
  int32_t* dev_status;
  cudaStream_t stream;
  // Fused append (k_new non-null; caches of at most decode_fuses_append_max_cap() rows): row
  // len[b] of every head of sequence b takes the new token's K and V (when it fits) before the
  // attention, which then covers len[b] + 1 rows, and len_out[b] receives the new length.
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  int32_t* len_out = nullptr;
};

// Largest cache (rows per head) whose decode kernel can take the append along.
int64_t decode_fuses_append_max_cap();

struct DecodeLayout {
  size_t partial, tickets, total;
  int split_rows, n_split;
};

DecodeLayout decode_layout(int batch, int heads, int head_dim, int64_t cap);

cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          int64_t cap, int32_t* len, int batch, int heads, int head_dim, int dtype,
                          int32_t* dev_status, cudaStream_t stream);
cudaError_t launch_decode(const DecodeJob& job);

// One hit-rate diagnostic call, after host-side validation.
struct HitRateJob {
  int batch, heads, head_dim, dtype;
  int64_t cap, l_prefix, k_sel;
  double theta;
  const void* q;
  const void* k_cache;
  const int32_t* len;
  const int32_t* idx;
  int32_t* hits;
  int32_t* total;
  int32_t* dev_status;
  cudaStream_t stream;
};

cudaError_t launch_hit_rate(const HitRateJob& job);

// Streaming multiprocessors of the current device (looked up once per device; 148 if the query
// fails). Launchers size their grids and cluster shapes with it.
int device_sm_count();

// Size of the built-in scratch array behind snapkv_decode_attend_noalloc.
constexpr size_t kDecodeNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB
// Decode attention with the split partials and tickets in the built-in scratch array
// (job.partial / job.tickets are ignored and replaced).
cudaError_t launch_decode_noalloc(DecodeJob job);

}  // namespace snapkv
