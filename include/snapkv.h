/*
 * snapkv.h — C ABI of the GB300 (sm_103a) SnapKV library: prefill-time KV-cache compression and
 * decode attention over the compressed cache.
 *
 * Sources (page title, section / equation):
 *   [SnapKV]  "論文解説: SnapKV — アテンションパターン観測によるKVキャッシュ圧縮" (0h-n0.github.io,
 *             posts/paper-2404-14469): プロンプトの分割 (L_prompt = L_prefix + L_obs),
 *             投票メカニズム (C = sum_i W_obs[:, i, :], I = Top_k(C, k), k = floor(p L_prefix)),
 *             クラスタリングによる文脈保持 (1D max pooling of C before top-k), アルゴリズム (the
 *             restated Algorithm 1: snap_kv_compress(query, key, value, obs_window, max_cap,
 *             kernel) -> (K_c, V_c)), 実装のポイント (per-head independent selection).
 *   [KVcache] "第22章 KV Cache" (waylandz.com, llm-transformer-book-ja/chapter-22-kv-cache),
 *             section 22.2: K_cache <- [K_cache; k_t], V_cache <- [V_cache; v_t] and
 *             o_t = softmax(q_t K_cache^T / sqrt(d_h)) V_cache.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers of the current device; the library never
 *     allocates, frees or synchronises, and keeps no state between calls. The caller owns every
 *     buffer, the workspace and the stream.
 *   - Work is enqueued asynchronously on `stream`. Argument errors are found on the host before
 *     anything is enqueued and returned; nothing is launched then.
 *   - Data-dependent errors found on the GPU (a full cache, a length beyond the capacity, a wait
 *     that gave up) are OR-ed as snapkv_status bits into *dev_status (device int32, optional:
 *     NULL disables the report), which the caller reads after synchronising the stream.
 *   - Tensors are dense, row-major, with the head dimension innermost; every device pointer must
 *     be 16-byte aligned. Q, K and V of one call share one dtype.
 */
#ifndef SNAPKV_H
#define SNAPKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SNAPKV_API __attribute__((visibility("default")))
#else
#define SNAPKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (same type); NULL is the legacy default stream. */
typedef struct CUstream_st* snapkv_stream_t;

/* Status codes; they are bits, so device-side reports can be OR-ed together. */
typedef enum {
  SNAPKV_OK = 0,
  SNAPKV_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size, misaligned pointer, bad enum       */
  SNAPKV_ERR_UNSUPPORTED = 2,   /* valid but not implemented: head_dim not 64/128, even pool  */
  SNAPKV_ERR_CAPACITY = 4,      /* cache capacity too small for k + L_obs, or cache full      */
  SNAPKV_ERR_CUDA = 8,          /* a CUDA launch failed                                       */
  SNAPKV_ERR_TIMEOUT = 16,      /* a bounded wait inside a kernel gave up (results invalid)   */
  SNAPKV_ERR_WORKSPACE = 32,    /* workspace NULL or smaller than the *_workspace_size answer */
  SNAPKV_ERR_INTERNAL = 64      /* a kernel's own consistency check failed (a library bug)    */
} snapkv_status;

typedef enum { SNAPKV_F32 = 0, SNAPKV_BF16 = 1 } snapkv_dtype;

/* Which logits enter a window row's softmax (the vote always keeps the prefix columns):
 *   PROMPT_CAUSAL: all prompt columns the window query sees, i.e. column j <= L_prefix + i for
 *                  window row i (causal inside the window). This is the default reading.
 *   PREFIX_ONLY:   the prefix columns only, as the restated Algorithm 1 listing of [SnapKV]
 *                  (アルゴリズム) normalises them. */
typedef enum { SNAPKV_SCOPE_PROMPT_CAUSAL = 0, SNAPKV_SCOPE_PREFIX_ONLY = 1 } snapkv_softmax_scope;

/* Which kernels compute the logits, softmax statistics and vote (the results agree within the
 * vote tolerance; the selection and the gathered rows are the same up to top-k boundary ties):
 *   AUTO:                the streaming tensor-core kernel when eligible (bf16, L_obs <= 64), else
 *                        the SIMT kernels;
 *   SIMT:                always the SIMT fp32 kernels (any dtype, L_obs <= 128);
 *   TENSOR_CORE:         the streaming tensor-core kernel, or SNAPKV_ERR_UNSUPPORTED when not
 *                        eligible (its row sums are fp64 atomics, so the vote's last bits can vary
 *                        from call to call);
 *   TENSOR_CORE_CLUSTER: one thread-block cluster per head (bf16, L_obs <= 64, a head's keys fit
 *                        8 CTAs x 4 TMEM slots: L_prompt <= 16384 at L_obs 17..32, 32768 at
 *                        L_obs <= 16, 8192 at L_obs 33..64), else SNAPKV_ERR_UNSUPPORTED. Every
 *                        reduction runs in a fixed order, so repeated calls give identical bits. */
typedef enum {
  SNAPKV_ALGO_AUTO = 0,
  SNAPKV_ALGO_SIMT = 1,
  SNAPKV_ALGO_TENSOR_CORE = 2,
  SNAPKV_ALGO_TENSOR_CORE_CLUSTER = 3
} snapkv_algo;

/* Problem statement of one compression call: one layer, `batch` sequences of one length. */
typedef struct {
  int32_t batch;          /* B >= 1                                                           */
  int32_t heads;          /* H >= 1 (one KV head per query head)                              */
  int32_t head_dim;       /* d: 64 or 128                                                     */
  int32_t l_obs;          /* observation window, 1 <= L_obs < L_prompt ([SnapKV] プロンプトの分割) */
  int64_t l_prompt;       /* L_prompt; L_prefix = L_prompt - L_obs                             */
  int32_t pool_kernel;    /* K_pool, odd, >= 1 (stride 1, padding K_pool/2, -inf padding)      */
  int32_t softmax_scope;  /* snapkv_softmax_scope                                              */
  double ratio_p;         /* p in [0,1]: k = floor(p * L_prefix) in IEEE double (budget <= 0)  */
  int64_t budget;         /* > 0: k = min(budget, L_prefix) (the listing's max_cap)            */
  int32_t dtype;          /* snapkv_dtype of Q, K, V and of the outputs                         */
  int32_t algo;           /* snapkv_algo (0 = automatic choice)                                 */
} snapkv_compress_params;

/* Kept prefix slots per head, k (host-side, for sizing). Returns -1 if the params are invalid. */
SNAPKV_API int64_t snapkv_compress_kept(const snapkv_compress_params* params);
/* The same value under the name the sizing step is usually called by. */
SNAPKV_API int64_t snapkv_compress_k(const snapkv_compress_params* params);

/* Workspace bytes snapkv_compress needs for these params (0 if the params are invalid). */
SNAPKV_API size_t snapkv_compress_workspace_size(const snapkv_compress_params* params);

/*
 * snapkv_compress — SnapKV prefill compression of one layer ([SnapKV] 投票メカニズム,
 * クラスタリングによる文脈保持, アルゴリズム), per (sequence, head) independently:
 *   s_ij = q_i . k_j / sqrt(d)                  window query i < L_obs, visible prompt column j
 *   w_ij = exp(s_ij - m_i) / Z_i                 fp32 row softmax (scope as above)
 *   C_j  = sum_{i < L_obs} w_ij                 j < L_prefix
 *   P_j  = max C_{j'} over |j' - j| <= K_pool/2 (clipped to the prefix)
 *   I    = the k positions of largest P, ties to the lower index, ascending
 *   K_c  = [K[I]; K[L_prefix : L_prompt]],  V_c likewise   (length R = k + L_obs)
 *
 * q_obs     device [B, H, L_obs, d]     the window's queries (prompt rows L_prefix..L_prompt-1)
 * k         device [B, H, L_prompt, d]  the layer's prompt keys (not modified)
 * v         [B, H, L_prompt, d]         the layer's prompt values (not modified): device memory, or
 *           page-locked host memory mapped into the device's address space (cudaHostAlloc, or
 *           cudaHostRegister with mapping). Only the R kept and window rows of each head are read,
 *           so values that live on the host cross the host link for those rows alone (method: the
 *           non-selected prefix values are never needed). Pageable host memory is refused with
 *           SNAPKV_ERR_INVALID_ARG; the type is looked up with cudaPointerGetAttributes, in
 *           relaxed stream-capture mode so that the call may be captured into a CUDA graph.
 * k_out     device [B, H, cap, d]        rows 0..R-1 of every head are written; the rest untouched
 * v_out     device [B, H, cap, d]
 * cap       rows per head of k_out / v_out; must be >= R, else SNAPKV_ERR_CAPACITY
 * len_out   device int32 [B]             set to R for every sequence
 * idx_out   device int32 [B, H, k]       kept prefix positions, ascending (NULL: not returned)
 * vote_out  device fp32 [B, H, L_prefix] the vote C (NULL: not returned)
 * workspace device, >= snapkv_compress_workspace_size(params) bytes, 256-byte aligned: scratch
 *           whose contents on entry do not matter (it needs no zero-fill, and one workspace can
 *           serve calls of any shape that fits it, one call at a time on the GPU)
 * dev_status device int32 (optional)     error bits OR-ed in on the GPU
 */
SNAPKV_API snapkv_status snapkv_compress(const snapkv_compress_params* params, const void* q_obs,
                              const void* k, const void* v, void* k_out, void* v_out, int64_t cap,
                              int32_t* len_out, int32_t* idx_out, float* vote_out,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              snapkv_stream_t stream);

/*
 * snapkv_compress_profiled — snapkv_compress, plus caller-created CUDA events (cudaEvent_t, cast
 * to void*) recorded on `stream` around the kernels of each stage, so that a caller can time
 * every stage on the device: stage_events[2s] is recorded just before and stage_events[2s+1]
 * just after the kernels of stage s, with s = 0 score statistics (row max and sum of every
 * window row), 1 vote, 2 max-pool + top-k, 3 gather + window append. Memsets that clear per-call
 * counters come before a stage's first marker. A fused kernel runs inside its first stage: the
 * tensor-core kernels do score and vote together (stage 0; stage 1 is empty), and for prefixes of
 * at most 8 x 24K keys the top-k kernel also gathers (stage 2; stage 3 is empty). Slots beyond n_events, or
 * NULL entries, are skipped; n_events = 0 behaves exactly like snapkv_compress. The events are
 * owned by the caller. A stage that needs no kernel for the given problem records its two
 * events back to back. When `stream` is being captured into a CUDA graph, each record is
 * captured as an event-record node (cudaEventRecordExternal), so every replay of the graph
 * records the events again.
 */
SNAPKV_API snapkv_status snapkv_compress_profiled(const snapkv_compress_params* params, const void* q_obs,
                                                  const void* k, const void* v, void* k_out, void* v_out,
                                                  int64_t cap, int32_t* len_out, int32_t* idx_out,
                                                  float* vote_out, void* workspace, size_t workspace_bytes,
                                                  int32_t* dev_status, snapkv_stream_t stream,
                                                  void* const* stage_events, int32_t n_events);

/*
 * snapkv_compress_gqa — snapkv_compress for grouped-query attention: `q_heads` query heads share
 * the params' `heads` KV heads (q_heads a multiple of heads; the G = q_heads / heads query heads of
 * KV head h are h*G .. h*G + G - 1). The pages do not cover grouped heads; the reading taken: each
 * query head votes with its own row softmax over its KV head's keys ([SnapKV] 投票メカニズム), the
 * KV head's vote is the sum of its G query heads' votes, and pooling, selection and gather run per
 * KV head. G * L_obs <= 128 (else SNAPKV_ERR_UNSUPPORTED).
 *
 * q_obs     device [B, q_heads, L_obs, d]
 * k         device [B, heads, L_prompt, d]
 * v         [B, heads, L_prompt, d], device or mapped page-locked host memory as for snapkv_compress
 * vote_out  device fp32 [B, heads, L_prefix] (the summed vote; NULL: not returned)
 * every other argument as for snapkv_compress, with heads = KV heads; the workspace size is
 * snapkv_compress_gqa_workspace_size(params, q_heads).
 */
SNAPKV_API size_t snapkv_compress_gqa_workspace_size(const snapkv_compress_params* params, int32_t q_heads);
SNAPKV_API snapkv_status snapkv_compress_gqa(const snapkv_compress_params* params, int32_t q_heads,
                                             const void* q_obs, const void* k, const void* v, void* k_out,
                                             void* v_out, int64_t cap, int32_t* len_out, int32_t* idx_out,
                                             float* vote_out, void* workspace, size_t workspace_bytes,
                                             int32_t* dev_status, snapkv_stream_t stream);

/*
 * snapkv_compress_varlen — snapkv_compress of a batch whose prompts have different lengths: sequence
 * b has l_prompts[b] rows (host array, L_obs < l_prompts[b] <= params->l_prompt), so its prefix,
 * its window (the last L_obs of its own rows) and its k = floor(p * L_prefix_b) or
 * min(budget, L_prefix_b) ([SnapKV] 投票メカニズム) are its own. Each sequence's result is what
 * snapkv_compress of that sequence alone gives, written into its slice of the shared outputs. The
 * tensor-core path takes the whole batch in one launch per kernel (up to 64 sequences, each keeping
 * at least one row); otherwise the sequences are compressed one after another on `stream`.
 *
 * q_obs     device [B, H, L_obs, d]   each sequence's window queries
 * k, v      [B, H, params->l_prompt, d], padded: sequence b's rows 0 .. l_prompts[b]-1 are read;
 *           k in device memory, v in device or mapped page-locked host memory (as for snapkv_compress)
 * k_out, v_out device [B, H, cap, d], cap >= k_max + L_obs where k_max = snapkv_compress_kept(params)
 *           (k grows with the prompt length); rows 0 .. k_b + L_obs - 1 of sequence b are written
 * len_out   device int32 [B], set to k_b + L_obs
 * idx_out   device int32 [B, H, k_max] (NULL: not returned); sequence b's heads hold k_b indices
 *           (ascending), the rest of each row is left untouched
 * vote_out  device fp32 [B, H, L_prefix_max] (NULL: not returned), L_prefix_max = params->l_prompt -
 *           L_obs; sequence b's heads hold L_prefix_b values, the rest is left untouched
 * workspace >= snapkv_compress_varlen_workspace_size(params, l_prompts) bytes, 256-byte aligned
 * A length outside (L_obs, params->l_prompt] gives SNAPKV_ERR_INVALID_ARG (and a workspace size of 0).
 */
SNAPKV_API size_t snapkv_compress_varlen_workspace_size(const snapkv_compress_params* params,
                                                        const int64_t* l_prompts);
SNAPKV_API snapkv_status snapkv_compress_varlen(const snapkv_compress_params* params, const int64_t* l_prompts,
                                                const void* q_obs, const void* k, const void* v, void* k_out,
                                                void* v_out, int64_t cap, int32_t* len_out, int32_t* idx_out,
                                                float* vote_out, void* workspace, size_t workspace_bytes,
                                                int32_t* dev_status, snapkv_stream_t stream);

/*
 * snapkv_append — one decode step's cache append ([KVcache] 22.2): for every sequence b and
 * head h, row len[b] of k_cache / v_cache receives k_new / v_new, then len[b] += 1.
 *
 * k_new, v_new      device [B, H, d]
 * k_cache, v_cache  device [B, H, cap, d]
 * len               device int32 [B], current cached rows per sequence (read, then incremented)
 * A sequence with len[b] >= cap (or < 0) is left untouched and SNAPKV_ERR_CAPACITY is reported in
 * *dev_status.
 */
SNAPKV_API snapkv_status snapkv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                            int64_t cap, int32_t* len, int32_t batch, int32_t heads,
                            int32_t head_dim, int32_t dtype, int32_t* dev_status,
                            snapkv_stream_t stream);

/* Workspace bytes snapkv_decode_attend needs (0 if the sizes are invalid). */
SNAPKV_API size_t snapkv_decode_workspace_size(int32_t batch, int32_t heads, int32_t head_dim, int64_t cap);

/*
 * snapkv_decode_attend — decode attention over each head's (compressed) cache ([KVcache] 22.2):
 *   o = softmax(q . K_cache[r]^T / sqrt(d), r < len[b]) V_cache     (fp32 math)
 * Every cached row is visible (the query is the newest position).
 *
 * q                 device [B, H, d]
 * k_cache, v_cache  device [B, H, cap, d]
 * len               device int32 [B]; rows 0..len[b]-1 are attended. len[b] > cap is clamped to
 *                   cap and reported as SNAPKV_ERR_CAPACITY; len[b] <= 0 gives o = 0.
 * out               device [B, H, d], same dtype as the cache
 * workspace         device, >= snapkv_decode_workspace_size(...) bytes, 256-byte aligned:
 *                   scratch whose contents on entry do not matter (one call at a time on the GPU)
 */
SNAPKV_API snapkv_status snapkv_decode_attend(const void* q, const void* k_cache, const void* v_cache,
                                   int64_t cap, const int32_t* len, void* out, int32_t batch,
                                   int32_t heads, int32_t head_dim, int32_t dtype, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status,
                                   snapkv_stream_t stream);

/*
 * snapkv_append_decode_attend — one whole decode step ([KVcache] 22.2: append the new token's row,
 * then attend over every cached row including it): the result of snapkv_append followed by
 * snapkv_decode_attend, in one launch for caches of up to 16384 rows per head (the decode kernel
 * writes the new row into the cache and into its own shared-memory copy of the rows before it
 * attends). Longer caches take the two kernels one after the other.
 *
 * q, k_new, v_new   device [B, H, d]
 * k_cache, v_cache  device [B, H, cap, d]; row len_in[b] of every head receives k_new / v_new
 * len_in            device int32 [B], cached rows before this step (read only)
 * len_out           device int32 [B], receives len_in[b] + 1 (len_in[b] when the row does not fit);
 *                   must not overlap len_in, so a caller alternates two length arrays
 * out               device [B, H, d], same dtype as the cache
 * workspace         as for snapkv_decode_attend (snapkv_decode_workspace_size(B, H, d, cap))
 * A sequence with len_in[b] >= cap (or < 0) is not appended, SNAPKV_ERR_CAPACITY is reported in
 * *dev_status, and the attention covers its len_in[b] rows (clamped to cap) as snapkv_decode_attend
 * would.
 */
SNAPKV_API snapkv_status snapkv_append_decode_attend(const void* q, const void* k_new, const void* v_new,
                                                     void* k_cache, void* v_cache, int64_t cap,
                                                     const int32_t* len_in, int32_t* len_out, void* out,
                                                     int32_t batch, int32_t heads, int32_t head_dim,
                                                     int32_t dtype, void* workspace, size_t workspace_bytes,
                                                     int32_t* dev_status, snapkv_stream_t stream);

/*
 * snapkv_decode_attend_noalloc — snapkv_decode_attend without a workspace argument, for callers
 * that cannot allocate device memory or hand one over: for example a plugin or custom-operator
 * interface that passes only inputs and outputs, or a latency-critical serving loop where a
 * cudaMalloc (which can synchronise the device and take a driver-wide lock) is not allowed.
 * The pages have no counterpart to this entry point; it computes exactly what
 * snapkv_decode_attend computes, with the same arguments minus the workspace.
 *
 * It allocates nothing. Caches of up to 16384 rows per head take the cluster kernel, which keeps
 * its partial results on chip and needs no scratch at all. Longer caches take the split kernel,
 * whose scratch (the split partials and the per-head tickets) is a 16 MiB array built into the
 * library, which every GPU that loads the library holds until the process exits. Such a problem
 * needing more than that — 256-byte-rounded B*H*S*(d+2)*4 bytes of partials, with S = ceil(cap/128)
 * splits (longer splits once S would pass 512), plus B*H*4 bytes of tickets — is rejected with
 * SNAPKV_ERR_WORKSPACE before anything is enqueued. The first long-cache call on a device looks up
 * the array's device address (with that device current) and caches it for the device's current
 * context, so make that first call before any stream capture; a new context on the device (for
 * example after cudaDeviceReset) makes the next call look it up again. All long-cache calls share the
 * one array and it keeps the last call's contents (the tickets are cleared on `stream` at the start
 * of each such call), so long-cache calls that overlap on the GPU — on different streams, or from
 * different host threads — race and give wrong results: serialise them. Calls on caches of up to
 * 16384 rows never touch the array and do not race.
 */
SNAPKV_API snapkv_status snapkv_decode_attend_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                      int64_t cap, const int32_t* len, void* out, int32_t batch,
                                                      int32_t heads, int32_t head_dim, int32_t dtype,
                                                      int32_t* dev_status, snapkv_stream_t stream);

/*
 * snapkv_hit_rate — the explainer's Hit Rate diagnostic ([SnapKV] Hit Rate（適中率）の定式化):
 * how much of a generation-time query's attention the kept positions cover. For every sequence b
 * and head h, A_cur = softmax(q . K_cache[r]^T / sqrt(d), r < len[b]) ([KVcache] 22.2, the
 * uncompressed cache) taken at the prefix positions j < l_prefix; then
 *   total[b,h] = #{ j : A_cur[j] > theta }                (sum of M_threshold)
 *   hits[b,h]  = #{ j in idx[b,h] : A_cur[j] > theta }    (sum of O = M_threshold AND M_vote)
 * and the hit rate is H = sum(hits) / sum(total) (the explainer uses theta = 0.05). The threshold
 * test runs in fp32 on the GPU, so a weight within a few ulps of theta may land on either side.
 *
 * q           device [B, H, d], the query of a decode step
 * k_cache     device [B, H, cap, d], the uncompressed cache (prompt rows first)
 * len         device int32 [B], cached rows (clamped to cap, reported as SNAPKV_ERR_CAPACITY)
 * l_prefix    prefix length, 1 <= l_prefix <= min(cap, 2^20)
 * idx         device int32 [B, H, k], the kept prefix positions (an index outside [0, l_prefix) is
 *             skipped and reported as SNAPKV_ERR_INVALID_ARG in *dev_status); k >= 0
 * theta       >= 0
 * hits, total device int32 [B, H]
 */
SNAPKV_API snapkv_status snapkv_hit_rate(const void* q, const void* k_cache, int64_t cap, const int32_t* len,
                                         int64_t l_prefix, const int32_t* idx, int64_t k, int32_t batch,
                                         int32_t heads, int32_t head_dim, int32_t dtype, double theta,
                                         int32_t* hits, int32_t* total, int32_t* dev_status,
                                         snapkv_stream_t stream);

/* Human-readable name of a status value (a static string; bits are listed when several). */
SNAPKV_API const char* snapkv_status_string(int32_t status);

/* ABI version of this header (major * 100 + minor). */
SNAPKV_API int32_t snapkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SNAPKV_H */
