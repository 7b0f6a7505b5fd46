// Decode-step append and split-K decode attention over the (compressed) cache.
//
// KV-cache chapter ("第22章 KV Cache"), section 22.2: K_cache <- [K_cache; k_t],
// V_cache <- [V_cache; v_t], then o_t = softmax(q_t K_cache^T / sqrt(d_h)) V_cache with every cached
// row visible. Each CTA keeps an online softmax (running max m, running sum l, unnormalised output
// o) in the log2 domain over its share of a head's rows. Two kernels:
//   * caches of up to kClusterMaxCap rows: one thread-block cluster (up to 8 CTAs) per (sequence,
//     head); the CTAs split the head's cap rows evenly (so the row loads need not wait for len; rows
//     at or past len are masked), and after one cluster barrier each CTA
//     finishes a slice of the output columns from every CTA's (m, l, o) read through distributed
//     shared memory. No workspace is touched.
//   * longer caches: splits of `split_rows` rows, one CTA each, partials in the workspace, and the
//     last CTA of the head to finish (an atomic ticket, no waiting) merges them.
// The cluster kernel can also take the step's append along (snapkv_append_decode_attend): the
// CTA whose rows hold the new row writes it into the cache and into its shared-memory copy before
// the attention reads it. The separate append kernel serves snapkv_append and longer caches.
#include <cudaTypedefs.h>

#include <mutex>

#include "sm100_ptx.cuh"
#include "snapkv_common.cuh"
#include "snapkv_internal.h"

// Built-in scratch of snapkv_decode_attend_noalloc: the split partials and the per-head tickets
// that snapkv_decode_attend otherwise takes from the caller's workspace. Every GPU that loads the
// library holds this array until the process exits; all calls of that entry point share it.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[snapkv::kDecodeNoAllocScratchBytes];

namespace snapkv {
namespace {

constexpr int kDecThreads = 128;
constexpr int kSplitRows = 128;
constexpr int kMaxSplits = 512;   // <= the floats of sm_o in every instantiation
constexpr int kClThreads = 256;
constexpr int kClMaxCtas = 8;
constexpr int64_t kClusterMaxCap = 16384;

__global__ void __launch_bounds__(256)
append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_cache,
              uint4* __restrict__ v_cache, int64_t cap, int32_t* __restrict__ len, int heads, int vpr,
              int32_t* __restrict__ dev_status) {
  const int b = blockIdx.x;
  // The new rows and the length are loaded together (one memory round trip): every thread reads
  // len[b] itself; the barrier below keeps the update after every thread's read.
  constexpr int kPer = 4;   // 16-byte pieces of K (and of V) per thread per round
  const int total = heads * vpr;
  const int64_t row0 = (int64_t)b * heads * vpr;
  const int p = len[b];
  const bool ok = p >= 0 && (int64_t)p < cap;
  for (int base = 0; base < total; base += kPer * (int)blockDim.x) {
    uint4 kv[kPer], vv[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int u = base + i * (int)blockDim.x + (int)threadIdx.x;
      if (u < total) {
        kv[i] = k_new[row0 + u];
        vv[i] = v_new[row0 + u];
      }
    }
    if (ok) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int u = base + i * (int)blockDim.x + (int)threadIdx.x;
        if (u < total) {
          const int h = u / vpr, c = u % vpr;
          const int64_t bh = (int64_t)b * heads + h;
          k_cache[(bh * cap + p) * vpr + c] = kv[i];
          v_cache[(bh * cap + p) * vpr + c] = vv[i];
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (ok)
      len[b] = p + 1;
    else
      report(dev_status, SNAPKV_ERR_CAPACITY);
  }
}

struct DecArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* len;
  void* out;
  float* partial;
  uint32_t* tickets;
  int64_t cap;
  int heads, split_rows, n_split;
  float scale_log2;
  int32_t* dev_status;
  const void* k_new;   // fused append (cluster kernel): the new token's K and V rows [B, H, d], or null
  const void* v_new;
  int32_t* len_out;    // fused append: the new lengths [B]
};

template <typename T> __device__ __forceinline__ void store_out(T* p, float x);
template <> __device__ __forceinline__ void store_out<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

template <typename T, int D>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(DecArgs a) {
  constexpr int V = Elem<T>::kVec;
  constexpr int LPR = D / V;                       // lanes per cache row
  constexpr int RPW = 32 / LPR;                    // rows per warp step
  constexpr int GROUPS = (kDecThreads / 32) * RPW; // row groups per CTA
  constexpr int UNROLL = 4;
  __shared__ float sm_m[GROUPS], sm_l[GROUPS];
  __shared__ __align__(16) float sm_o[GROUPS][D];
  __shared__ int sh_last;

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int split = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.heads);
  int n = a.len[b];
  if ((int64_t)n > a.cap) {
    if (split == 0 && tid == 0 && bh % a.heads == 0) report(a.dev_status, SNAPKV_ERR_CAPACITY);
    n = (int)a.cap;
  }
  if (n < 0) n = 0;
  const int r0 = split * a.split_rows;
  const int r1 = min(n, r0 + a.split_rows);
  const int sub = lane / LPR, cl = lane % LPR;
  const int group = warp * RPW + sub;

  const T* qp = static_cast<const T*>(a.q) + bh * D;
  float q[V];
  Elem<T>::widen(ld_nc_v4(qp + cl * V), q);
#pragma unroll
  for (int e = 0; e < V; ++e) q[e] *= a.scale_log2;

  const T* kc = static_cast<const T*>(a.k_cache) + bh * a.cap * D + cl * V;
  const T* vc = static_cast<const T*>(a.v_cache) + bh * a.cap * D + cl * V;
  float m = -INFINITY, l = 0.f, o[V];
#pragma unroll
  for (int e = 0; e < V; ++e) o[e] = 0.f;

  // The trip count depends only on the split, so every lane of a warp runs the same iterations
  // (the row reductions below shuffle across the whole warp).
  for (int base = r0; base < r1; base += GROUPS * UNROLL) {
    const int rb = base + group;
    uint4 kr[UNROLL], vr[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int r = rb + u * GROUPS;
      if (r < r1 && in_bounds(r >= 0 && r < a.cap, a.dev_status)) {
        kr[u] = ld_stream_v4(kc + (int64_t)r * D);
        vr[u] = ld_stream_v4(vc + (int64_t)r * D);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float s[UNROLL];
    float smax = -INFINITY;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float kf[V];
      Elem<T>::widen(kr[u], kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < V; ++e) dot = fmaf(q[e], kf[e], dot);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      s[u] = (rb + u * GROUPS < r1) ? dot : -INFINITY;
      smax = fmaxf(smax, s[u]);
    }
    const float m_new = fmaxf(m, smax);
    if (m_new == -INFINITY) continue;
    const float corr = ex2(m - m_new);
    l *= corr;
#pragma unroll
    for (int e = 0; e < V; ++e) o[e] *= corr;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const float p = ex2(s[u] - m_new);
      float vf[V];
      Elem<T>::widen(vr[u], vf);
      l += p;
#pragma unroll
      for (int e = 0; e < V; ++e) o[e] = fmaf(p, vf[e], o[e]);
    }
    m = m_new;
  }

  if (cl == 0) {
    sm_m[group] = m;
    sm_l[group] = l;
  }
#pragma unroll
  for (int e = 0; e < V; ++e) sm_o[group][cl * V + e] = o[e];
  __syncthreads();

  float* part = a.partial + (bh * a.n_split + split) * (D + 2);
  for (int t = tid; t < D; t += kDecThreads) {
    float M = -INFINITY;
#pragma unroll
    for (int g = 0; g < GROUPS; ++g) M = fmaxf(M, sm_m[g]);
    float ot = 0.f, lt = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int g = 0; g < GROUPS; ++g) {
        if (sm_m[g] == -INFINITY) continue;
        const float w = ex2(sm_m[g] - M);
        ot = fmaf(sm_o[g][t], w, ot);
        lt = fmaf(sm_l[g], w, lt);
      }
    }
    part[t] = ot;
    if (t == 0) {
      part[D] = M;
      part[D + 1] = lt;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t ticket = atomicAdd(a.tickets + bh, 1u);
    sh_last = ticket == (uint32_t)(a.n_split - 1);
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  // Last CTA of the head: merge the splits. The split maxima and sums are fetched in parallel
  // into shared memory (reusing sm_o), then each output column sums its splits' weighted partial
  // outputs with independent loads.
  const float* parts = a.partial + bh * a.n_split * (D + 2);
  float* sw = &sm_o[0][0];                       // [n_split] weights, then the scalar total
  float M = -INFINITY;
  for (int sp = tid; sp < a.n_split; sp += kDecThreads) M = fmaxf(M, __ldcg(parts + sp * (D + 2) + D));
  M = warp_max(M);
  if (lane == 0) sm_m[warp] = M;
  __syncthreads();
  M = sm_m[0];
#pragma unroll
  for (int w = 1; w < kDecThreads / 32; ++w) M = fmaxf(M, sm_m[w]);
  __syncthreads();
  float lsum = 0.f;
  for (int sp = tid; sp < a.n_split; sp += kDecThreads) {
    const float ms = __ldcg(parts + sp * (D + 2) + D);
    const float w = (ms == -INFINITY || M == -INFINITY) ? 0.f : ex2(ms - M);
    sw[sp] = w;
    lsum = fmaf(__ldcg(parts + sp * (D + 2) + D + 1), w, lsum);
  }
  lsum = warp_sum(lsum);
  if (lane == 0) sm_l[warp] = lsum;
  __syncthreads();
  float ltot = 0.f;
#pragma unroll
  for (int w = 0; w < kDecThreads / 32; ++w) ltot += sm_l[w];
  T* out = static_cast<T*>(a.out) + bh * D;
  for (int t = tid; t < D; t += kDecThreads) {
    float ot = 0.f;
    int sp = 0;
    for (; sp + 4 <= a.n_split; sp += 4) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcg(parts + (sp + u) * (D + 2) + t);
#pragma unroll
      for (int u = 0; u < 4; ++u) ot = fmaf(v[u], sw[sp + u], ot);
    }
    for (; sp < a.n_split; ++sp) ot = fmaf(__ldcg(parts + sp * (D + 2) + t), sw[sp], ot);
    store_out<T>(out + t, ltot > 0.f ? ot / ltot : 0.f);
  }
}

// One cluster per (sequence, head): CTA `rank` takes rows [rank * per, (rank + 1) * per) of the
// head's cap rows (those at or past len masked). The rows are contiguous in the cache, so one
// thread streams them into shared memory with bulk copies, kClBufs chunks of 16 KB of K and 16 KB
// of V in flight, and the row groups compute from shared memory.
constexpr int kClChunkBytes = 16 * 1024;
constexpr int kClBufs = 3;
constexpr long long kClWaitLimit = 4000000000LL;   // ~2 s of SM clock

// Orders this thread's generic-proxy writes to shared memory before later async-proxy (bulk copy)
// accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <typename T, int D>
__global__ void __launch_bounds__(kClThreads) decode_cluster_kernel(DecArgs a) {
  constexpr int V = Elem<T>::kVec;
  constexpr int LPR = D / V;                       // lanes per cache row
  constexpr int RPW = 32 / LPR;                    // rows per warp step
  constexpr int GROUPS = (kClThreads / 32) * RPW;  // row groups per CTA
  constexpr int ROW_BYTES = D * (int)sizeof(T);
  constexpr int CH = kClChunkBytes / ROW_BYTES;    // rows per chunk
  constexpr int UNROLL = CH / GROUPS;              // rows per group per chunk
  static_assert(CH % GROUPS == 0, "chunk rows");
  extern __shared__ __align__(128) uint8_t dsm[];  // [kClBufs][K, V][kClChunkBytes]
  __shared__ __align__(8) uint64_t bar[kClBufs];
  __shared__ int no_abort;
  __shared__ float sm_m[GROUPS], sm_l[GROUPS];
  __shared__ __align__(16) float sm_o[GROUPS][D];
  __shared__ float cta_m, cta_l;                   // this CTA's partial, read by the whole cluster
  __shared__ __align__(16) float cta_o[D];

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const uint32_t rank = ptx::cluster_rank(), csize = ptx::cluster_size();
  const int64_t bh = blockIdx.x / csize;
  const int b = (int)(bh / a.heads);
  const int cap = (int)a.cap;
  const int per = (cap + (int)csize - 1) / (int)csize;
  const int r0 = min(cap, (int)rank * per);
  const int r1 = min(cap, r0 + per);   // rows at or past n are streamed (they are inside cap) and masked
  const int nchunks = (r1 - r0 + CH - 1) / CH;
  const T* kc = static_cast<const T*>(a.k_cache) + bh * a.cap * D;
  const T* vc = static_cast<const T*>(a.v_cache) + bh * a.cap * D;
  auto issue = [&](int c) {
    const int buf = c % kClBufs;
    const int cr0 = r0 + c * CH;
    const int rows = min(CH, r1 - cr0);
    // (a chunk that fails the check copies nothing, so its barrier still completes)
    const bool ok = in_bounds(cr0 >= 0 && rows > 0 && cr0 + rows <= cap, a.dev_status);
    const uint32_t bytes = ok ? (uint32_t)(rows * ROW_BYTES) : 0u;
    ptx::mbar_arrive_expect_tx(&bar[buf], 2 * bytes);
    if (ok) {
      ptx::bulk_load(dsm + (2 * buf) * kClChunkBytes, kc + (int64_t)cr0 * D, bytes, &bar[buf]);
      ptx::bulk_load(dsm + (2 * buf + 1) * kClChunkBytes, vc + (int64_t)cr0 * D, bytes, &bar[buf]);
    }
  };
  if (tid == 0) {
    for (int i = 0; i < kClBufs; ++i) ptx::mbar_init(&bar[i], 1);
    no_abort = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int c = 0; c < nchunks && c < kClBufs; ++c) issue(c);

  int n = a.len[b];
  // Fused append ([KVcache] 22.2: the cache grows by the new token's row, then attention covers
  // it): the row goes to cache row n when n < cap, the attention then covers n + 1 rows, and the
  // first head's cluster records the new length; a full cache is reported and left unchanged.
  int new_row = -1;
  if (a.k_new) {
    const bool first = rank == 0 && tid == 0 && bh % a.heads == 0;
    if (n >= 0 && n < cap) {
      new_row = n;
      n += 1;
    } else if (first) {
      report(a.dev_status, SNAPKV_ERR_CAPACITY);
    }
    if (first) a.len_out[b] = n;
  }
  if ((int64_t)n > a.cap) {
    if (rank == 0 && tid == 0 && bh % a.heads == 0) report(a.dev_status, SNAPKV_ERR_CAPACITY);
    n = cap;
  }
  if (n < 0) n = 0;
  const int sub = lane / LPR, cl = lane % LPR;
  const int group = warp * RPW + sub;
  // The CTA whose rows hold the new row writes it into the chunk's shared-memory copy (after that
  // chunk lands, before any group reads it) and into the cache; its first 2 * PIECES threads hold
  // the row's 16-byte pieces (K, then V) from the start.
  constexpr int PIECES = ROW_BYTES / 16;
  const bool owns_new = new_row >= r0 && new_row < r1;
  const int new_chunk = owns_new ? (new_row - r0) / CH : -1;
  uint4 new_piece = make_uint4(0u, 0u, 0u, 0u);
  if (owns_new && tid < 2 * PIECES) {
    const uint4* src = static_cast<const uint4*>(tid < PIECES ? a.k_new : a.v_new) + bh * PIECES;
    new_piece = ld_nc_v4(src + tid % PIECES);
  }

  const T* qp = static_cast<const T*>(a.q) + bh * D;
  float q[V];
  Elem<T>::widen(ld_nc_v4(qp + cl * V), q);
#pragma unroll
  for (int e = 0; e < V; ++e) q[e] *= a.scale_log2;

  float m = -INFINITY, l = 0.f, o[V];
#pragma unroll
  for (int e = 0; e < V; ++e) o[e] = 0.f;
  bool timed_out = false;
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c % kClBufs;
    if (!ptx::mbar_wait(&bar[buf], (uint32_t)((c / kClBufs) & 1), &no_abort, kClWaitLimit)) timed_out = true;
    if (c == new_chunk) {   // uniform in the CTA
      if (tid < 2 * PIECES) {
        const int rr = new_row - (r0 + c * CH);
        uint8_t* srow = dsm + (2 * buf + (tid < PIECES ? 0 : 1)) * kClChunkBytes + rr * ROW_BYTES;
        *reinterpret_cast<uint4*>(srow + (tid % PIECES) * 16) = new_piece;
        // The caches of the fused entry point are writable; the chunk's copy of this row has landed.
        T* crow = const_cast<T*>(tid < PIECES ? kc : vc) + (int64_t)new_row * D;
        reinterpret_cast<uint4*>(crow)[tid % PIECES] = new_piece;
        fence_proxy_async_smem();   // before a later bulk copy refills this buffer
      }
      __syncthreads();
    }
    const uint8_t* kbuf = dsm + (2 * buf) * kClChunkBytes;
    const uint8_t* vbuf = kbuf + kClChunkBytes;
    const int cr0 = r0 + c * CH;
    float s[UNROLL];
    float smax = -INFINITY;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int rr = group + u * GROUPS;   // row within the chunk
      float kf[V];
      Elem<T>::widen(*reinterpret_cast<const uint4*>(kbuf + rr * ROW_BYTES + cl * 16), kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < V; ++e) dot = fmaf(q[e], kf[e], dot);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const int r = cr0 + rr;
      s[u] = (r < r1 && r < n) ? dot : -INFINITY;
      smax = fmaxf(smax, s[u]);
    }
    const float m_new = fmaxf(m, smax);
    if (m_new != -INFINITY) {
      const float corr = ex2(m - m_new);
      l *= corr;
#pragma unroll
      for (int e = 0; e < V; ++e) o[e] *= corr;
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const float p = ex2(s[u] - m_new);   // 0 for masked rows
        if (p != 0.f) {
          float vf[V];
          Elem<T>::widen(*reinterpret_cast<const uint4*>(vbuf + (group + u * GROUPS) * ROW_BYTES + cl * 16), vf);
          l += p;
#pragma unroll
          for (int e = 0; e < V; ++e) o[e] = fmaf(p, vf[e], o[e]);
        }
      }
      m = m_new;
    }
    __syncthreads();   // every group is done with this buffer
    if (tid == 0 && c + kClBufs < nchunks) issue(c + kClBufs);
  }
  if (timed_out && tid == 0) {
    report(a.dev_status, SNAPKV_ERR_TIMEOUT);
    // A copy whose wait gave up may still be landing: wait for it (bounded) before leaving.
    for (int c = (nchunks > kClBufs ? nchunks - kClBufs : 0); c < nchunks; ++c)
      ptx::mbar_wait(&bar[c % kClBufs], (uint32_t)((c / kClBufs) & 1), &no_abort, kClWaitLimit);
  }

  if (cl == 0) {
    sm_m[group] = m;
    sm_l[group] = l;
  }
#pragma unroll
  for (int e = 0; e < V; ++e) sm_o[group][cl * V + e] = o[e];
  __syncthreads();
  // This CTA's partial: column t combines the row groups.
  if (tid < D) {
    float M = -INFINITY;
#pragma unroll
    for (int g = 0; g < GROUPS; ++g) M = fmaxf(M, sm_m[g]);
    float ot = 0.f, lt = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int g = 0; g < GROUPS; ++g) {
        if (sm_m[g] == -INFINITY) continue;
        const float w = ex2(sm_m[g] - M);
        ot = fmaf(sm_o[g][tid], w, ot);
        lt = fmaf(sm_l[g], w, lt);
      }
    }
    cta_o[tid] = ot;
    if (tid == 0) {
      cta_m = M;
      cta_l = lt;
    }
  }
  ptx::cluster_sync();   // every CTA's partial is complete
  // Column t is finished by CTA t % csize from all the cluster's partials.
  T* out = static_cast<T*>(a.out) + bh * D;
  for (int t = (int)rank + (int)csize * tid; t < D; t += (int)csize * kClThreads) {
    float mr[kClMaxCtas];
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kClMaxCtas; ++r) {
      mr[r] = r < (int)csize ? __uint_as_float(ptx::dsmem_ld_u32(ptx::map_rank(&cta_m, (uint32_t)r))) : -INFINITY;
      M = fmaxf(M, mr[r]);
    }
    float lt = 0.f, ot = 0.f;
#pragma unroll
    for (int r = 0; r < kClMaxCtas; ++r) {
      if (r < (int)csize && mr[r] != -INFINITY) {
        const float w = ex2(mr[r] - M);
        lt = fmaf(__uint_as_float(ptx::dsmem_ld_u32(ptx::map_rank(&cta_l, (uint32_t)r))), w, lt);
        ot = fmaf(__uint_as_float(ptx::dsmem_ld_u32(ptx::map_rank(&cta_o[t], (uint32_t)r))), w, ot);
      }
    }
    store_out<T>(out + t, lt > 0.f ? ot / lt : 0.f);
  }
  ptx::cluster_sync();   // no CTA leaves while its partial may still be read
}

template <typename T, int D>
cudaError_t launch_decode_cluster(const DecodeJob& job, const DecArgs& a) {
  const int64_t bh = (int64_t)job.batch * job.heads;
  // CTAs per head: splitting a head's rows over a cluster cuts the latency of a small batch; once
  // the heads alone give about two CTAs per SM, one CTA per head streams all its rows and skips the
  // merge (2048 heads of 2208 rows: 8 CTAs per head 462 us, 1 CTA 319 us per launch; 256 heads of
  // 850 rows: 7 CTAs 45 us, 1 CTA 22 us).
  int csize = (int)((job.cap + kSplitRows - 1) / kSplitRows);
  const int64_t per_head = (int64_t)2 * device_sm_count() / (bh > 0 ? bh : 1);
  if ((int64_t)csize > per_head) csize = (int)per_head;
  if (csize > kClMaxCtas) csize = kClMaxCtas;
  if (csize < 1) csize = 1;
  cudaLaunchConfig_t cfg = {};
  static std::once_flag smem_set;   // the dynamic shared-memory attribute, once per instantiation
  static cudaError_t smem_err = cudaSuccess;
  std::call_once(smem_set, [] {
    smem_err = cudaFuncSetAttribute(decode_cluster_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    2 * kClBufs * kClChunkBytes);
  });
  if (smem_err != cudaSuccess) return smem_err;
  cfg.gridDim = dim3((unsigned)(bh * csize));
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = 2 * kClBufs * kClChunkBytes;
  cfg.stream = job.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_cluster_kernel<T, D>, a);
}

template <typename T, int D>
cudaError_t launch_decode_typed(const DecodeJob& job, const DecArgs& a) {
  const int64_t bh = (int64_t)job.batch * job.heads;
  decode_split_kernel<T, D><<<dim3(job.n_split, (unsigned)bh), kDecThreads, 0, job.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int64_t decode_fuses_append_max_cap() { return kClusterMaxCap; }

DecodeLayout decode_layout(int batch, int heads, int head_dim, int64_t cap) {
  DecodeLayout L;
  // 128-row splits, or longer ones (a multiple of 128) for caches beyond 512 splits: the merge
  // keeps one weight per split in the CTA's shared memory.
  int64_t rows = kSplitRows;
  if ((cap + rows - 1) / rows > kMaxSplits) rows = ((cap + kMaxSplits - 1) / kMaxSplits + kSplitRows - 1) / kSplitRows * kSplitRows;
  L.split_rows = (int)rows;
  L.n_split = (int)((cap + rows - 1) / rows);
  if (L.n_split < 1) L.n_split = 1;
  const size_t bh = (size_t)batch * heads;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  L.partial = 0;
  L.tickets = up(bh * L.n_split * (head_dim + 2) * sizeof(float));
  L.total = up(L.tickets + bh * sizeof(uint32_t));
  return L;
}

cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache, int64_t cap,
                          int32_t* len, int batch, int heads, int head_dim, int dtype, int32_t* dev_status,
                          cudaStream_t stream) {
  const int esize = dtype == SNAPKV_BF16 ? 2 : 4;
  const int vpr = head_dim * esize / 16;
  append_kernel<<<batch, 256, 0, stream>>>(static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                                           static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), cap, len,
                                           heads, vpr, dev_status);
  return cudaGetLastError();
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};

// Identifier of the calling thread's current context, unique for the life of the process (0 if
// the driver cannot tell). A device's context is replaced by cudaDeviceReset or by a context the
// caller makes current; the module, and with it the scratch array, is then loaded again at a new
// address, so a cached address is only reused under the context it was looked up in.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the built-in scratch for the current device and context. The array's host-side
// name is only a stand-in, never a device address: the first call on a device (and the first after
// its context changed) looks the address up with cudaGetSymbolAddress and caches it.
cudaError_t noalloc_scratch_address(void** out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_noalloc_addr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_noalloc_addr[dev] = p;
    g_noalloc_ctx[dev] = current_context_id();   // the lookup made the context current if none was
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_decode_noalloc(DecodeJob job) {
  if (job.cap <= kClusterMaxCap) {   // the cluster kernel keeps its partials on chip: no scratch
    job.partial = nullptr;
    job.tickets = nullptr;
    return launch_decode(job);
  }
  const DecodeLayout L = decode_layout(job.batch, job.heads, job.head_dim, job.cap);
  if (L.total > kDecodeNoAllocScratchBytes) return cudaErrorInvalidValue;  // rejected earlier by the ABI
  void* base = nullptr;
  cudaError_t err = noalloc_scratch_address(&base);
  if (err != cudaSuccess) return err;
  char* ws = static_cast<char*>(base);
  job.partial = reinterpret_cast<float*>(ws + L.partial);
  job.tickets = reinterpret_cast<uint32_t*>(ws + L.tickets);
  job.split_rows = L.split_rows;
  job.n_split = L.n_split;
  return launch_decode(job);
}

cudaError_t launch_decode(const DecodeJob& job) {
  DecArgs a;
  a.q = job.q;
  a.k_cache = job.k_cache;
  a.v_cache = job.v_cache;
  a.len = job.len;
  a.out = job.out;
  a.partial = job.partial;
  a.tickets = job.tickets;
  a.cap = job.cap;
  a.heads = job.heads;
  a.split_rows = job.split_rows;
  a.n_split = job.n_split;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)job.head_dim));
  a.dev_status = job.dev_status;
  a.k_new = job.k_new;
  a.v_new = job.v_new;
  a.len_out = job.len_out;
  if (job.k_new && job.cap > kClusterMaxCap) return cudaErrorInvalidValue;   // the ABI appends separately
  if (job.cap <= kClusterMaxCap) {
    if (job.dtype == SNAPKV_BF16)
      return job.head_dim == 64 ? launch_decode_cluster<__nv_bfloat16, 64>(job, a)
                                : launch_decode_cluster<__nv_bfloat16, 128>(job, a);
    return job.head_dim == 64 ? launch_decode_cluster<float, 64>(job, a) : launch_decode_cluster<float, 128>(job, a);
  }
  // The per-head tickets start at zero on every call (the workspace's contents are not trusted).
  const cudaError_t err =
      cudaMemsetAsync(job.tickets, 0, (size_t)job.batch * job.heads * sizeof(uint32_t), job.stream);
  if (err != cudaSuccess) return err;
  if (job.dtype == SNAPKV_BF16)
    return job.head_dim == 64 ? launch_decode_typed<__nv_bfloat16, 64>(job, a)
                              : launch_decode_typed<__nv_bfloat16, 128>(job, a);
  return job.head_dim == 64 ? launch_decode_typed<float, 64>(job, a) : launch_decode_typed<float, 128>(job, a);
}

}  // namespace snapkv
