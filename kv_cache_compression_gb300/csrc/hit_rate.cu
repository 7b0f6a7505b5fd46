// Hit-rate diagnostic of the vote.
//
// SnapKV explainer ("論文解説: SnapKV"), section Hit Rate（適中率）の定式化: with A_cur the attention
// of a generation-time query over the prefix positions, M_threshold = 1(A_cur > theta), M_vote the
// kept positions and O = M_threshold AND M_vote, the hit rate is H = sum(O) / sum(M_threshold).
// A_cur is the decode attention of the KV-cache chapter (section 22.2) over every row of the
// uncompressed cache, taken at the prefix positions.
//
// Caches of up to kHrClusterRows x 8 rows: one thread-block cluster of up to 8 CTAs per (sequence,
// head). CTA r streams its share of the cache rows into shared memory with bulk copies, keeps their
// logits s' (log2 domain) in shared memory and its running (max, sum of 2^(s' - max)); after one
// cluster barrier every CTA folds all (max, sum) pairs in rank order into log2 Z, counts its prefix
// rows with s' - log2 Z > log2 theta and those among them whose bit is set in its bitmap of the
// kept indices, and adds both counts into CTA 0 through distributed shared memory. Longer caches:
// one CTA per (sequence, head) that reads the keys twice.
#include "sm100_ptx.cuh"
#include "snapkv_common.cuh"
#include "snapkv_internal.h"

namespace snapkv {
namespace {

constexpr int kHrThreads = 256;
constexpr int kHrCtas = 8;
constexpr int kHrClusterRows = 16384;             // rows per CTA of the cluster kernel (64 KB of logits)
constexpr int kHrChunkBytes = 16 * 1024;
constexpr int kHrBufs = 3;
constexpr long long kHrWaitLimit = 4000000000LL;   // ~2 s of SM clock

struct HrArgs {
  const void* q;
  const void* k_cache;
  const int32_t* len;
  const int32_t* idx;
  int32_t* hits;
  int32_t* total;
  int64_t cap, l_prefix, k_sel;
  int heads;
  float scale_log2, log2_theta;
  int32_t* dev_status;
};

template <typename T, int D>
__device__ __forceinline__ float row_logit(const T* kc, int64_t r, int cl, const float* q) {
  constexpr int V = Elem<T>::kVec;
  constexpr int LPR = D / V;
  float kf[V];
  Elem<T>::widen(ld_stream_v4(kc + r * D + cl * V), kf);
  float dot = 0.f;
#pragma unroll
  for (int e = 0; e < V; ++e) dot = fmaf(q[e], kf[e], dot);
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  return dot;
}

template <typename T, int D>
__global__ void __launch_bounds__(kHrThreads) hit_rate_kernel(HrArgs a) {
  constexpr int V = Elem<T>::kVec;
  constexpr int LPR = D / V;
  constexpr int RPW = 32 / LPR;
  constexpr int GROUPS = (kHrThreads / 32) * RPW;
  extern __shared__ uint32_t kept_bits[];          // [ceil(l_prefix / 32)]
  __shared__ float sm_m[GROUPS], sm_l[GROUPS];
  __shared__ float sh_cut;
  __shared__ int sh_hits, sh_total;

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int64_t bh = blockIdx.x;
  const int b = (int)(bh / a.heads);
  int64_t n = a.len[b];
  if (n > a.cap) {
    if (tid == 0 && bh % a.heads == 0) report(a.dev_status, SNAPKV_ERR_CAPACITY);
    n = a.cap;
  }
  if (n < 0) n = 0;
  const int64_t np = n < a.l_prefix ? n : a.l_prefix;   // prefix positions present in the cache
  const int sub = lane / LPR, cl = lane % LPR;
  const int group = warp * RPW + sub;

  const int nwords = (int)((a.l_prefix + 31) / 32);
  for (int w = tid; w < nwords; w += kHrThreads) kept_bits[w] = 0u;
  if (tid == 0) {
    sh_hits = 0;
    sh_total = 0;
  }
  __syncthreads();
  const int32_t* idx = a.idx + bh * a.k_sel;
  for (int64_t t = tid; t < a.k_sel; t += kHrThreads) {
    const int32_t j = idx[t];
    if (j >= 0 && j < a.l_prefix) atomicOr(&kept_bits[j >> 5], 1u << (j & 31));
    else report(a.dev_status, SNAPKV_ERR_INVALID_ARG);
  }

  const T* qp = static_cast<const T*>(a.q) + bh * D;
  float q[V];
  Elem<T>::widen(ld_nc_v4(qp + cl * V), q);
#pragma unroll
  for (int e = 0; e < V; ++e) q[e] *= a.scale_log2;
  const T* kc = static_cast<const T*>(a.k_cache) + bh * a.cap * D;

  // Pass 1: log2 Z = M + log2(sum 2^(s' - M)) over every cached row. The trip count is the same
  // for all lanes of a warp (the dot products shuffle across the whole warp).
  float m = -INFINITY, l = 0.f;
  for (int64_t base = 0; base < n; base += GROUPS) {
    const int64_t r = base + group;
    const float dot = row_logit<T, D>(kc, r < n ? r : 0, cl, q);   // every lane shuffles
    const float s = r < n ? dot : -INFINITY;
    if (s > m) {
      l = l * ex2(m - s) + 1.f;
      m = s;
    } else if (s > -INFINITY) {
      l += ex2(s - m);
    }
  }
  if (cl == 0) {
    sm_m[group] = m;
    sm_l[group] = l;
  }
  __syncthreads();
  if (tid == 0) {
    float M = -INFINITY;
    for (int g = 0; g < GROUPS; ++g) M = fmaxf(M, sm_m[g]);
    float Z = 0.f;
    if (M > -INFINITY)
      for (int g = 0; g < GROUPS; ++g)
        if (sm_m[g] > -INFINITY) Z = fmaf(sm_l[g], ex2(sm_m[g] - M), Z);
    // A_cur[j] > theta  <=>  s'_j > log2 Z + log2 theta
    sh_cut = M > -INFINITY ? M + log2f(Z) + a.log2_theta : INFINITY;
  }
  __syncthreads();
  const float cut = sh_cut;

  // Pass 2: the prefix positions above the threshold, and those among them that were kept.
  int hits = 0, total = 0;
  for (int64_t base = 0; base < np; base += GROUPS) {
    const int64_t r = base + group;
    const float dot = row_logit<T, D>(kc, r < np ? r : 0, cl, q);   // every lane shuffles
    const float s = r < np ? dot : -INFINITY;
    if (cl == 0 && r < np && s > cut) {
      ++total;
      hits += (kept_bits[r >> 5] >> (r & 31)) & 1u;
    }
  }
  hits = __reduce_add_sync(0xffffffffu, hits);
  total = __reduce_add_sync(0xffffffffu, total);
  if (lane == 0) {
    atomicAdd(&sh_hits, hits);
    atomicAdd(&sh_total, total);
  }
  __syncthreads();
  if (tid == 0) {
    a.hits[bh] = sh_hits;
    a.total[bh] = sh_total;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kHrThreads) hit_rate_cluster_kernel(HrArgs a) {
  constexpr int V = Elem<T>::kVec;
  constexpr int LPR = D / V;
  constexpr int RPW = 32 / LPR;
  constexpr int GROUPS = (kHrThreads / 32) * RPW;
  constexpr int ROW_BYTES = D * (int)sizeof(T);
  constexpr int CH = kHrChunkBytes / ROW_BYTES;    // rows per chunk
  constexpr int UNROLL = CH / GROUPS;
  static_assert(CH % GROUPS == 0, "chunk rows");
  extern __shared__ __align__(128) uint8_t dsm[];  // [kHrBufs][chunk] keys, then per-row logits, then bits
  __shared__ __align__(8) uint64_t bar[kHrBufs];
  __shared__ int no_abort;
  __shared__ float sm_m[GROUPS], sm_l[GROUPS];
  __shared__ float cta_m, cta_l;                   // this CTA's (max, sum), read by the cluster
  __shared__ uint32_t cnt[2];                      // hits, total (CTA 0 receives the cluster's)

  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const uint32_t rank = ptx::cluster_rank(), csize = ptx::cluster_size();
  const int64_t bh = blockIdx.x / csize;
  const int b = (int)(bh / a.heads);
  const int cap = (int)a.cap;
  const int per = (cap + (int)csize - 1) / (int)csize;   // <= kHrClusterRows by the launch
  const int r0 = min(cap, (int)rank * per);
  const int r1 = min(cap, r0 + per);
  const int nchunks = (r1 - r0 + CH - 1) / CH;
  float* logit = reinterpret_cast<float*>(dsm + kHrBufs * kHrChunkBytes);   // [per]
  uint32_t* bits = reinterpret_cast<uint32_t*>(logit + per);               // [(per + 31) / 32]
  const T* kc = static_cast<const T*>(a.k_cache) + bh * a.cap * D;
  auto issue = [&](int c) {
    const int buf = c % kHrBufs;
    const int cr0 = r0 + c * CH;
    const uint32_t bytes = (uint32_t)(min(CH, r1 - cr0) * ROW_BYTES);
    ptx::mbar_arrive_expect_tx(&bar[buf], bytes);
    ptx::bulk_load(dsm + buf * kHrChunkBytes, kc + (int64_t)cr0 * D, bytes, &bar[buf]);
  };
  if (tid == 0) {
    for (int i = 0; i < kHrBufs; ++i) ptx::mbar_init(&bar[i], 1);
    no_abort = 0;
    cnt[0] = 0u;
    cnt[1] = 0u;
    ptx::fence_mbar_init();
  }
  for (int w = tid; w < (per + 31) / 32; w += kHrThreads) bits[w] = 0u;
  __syncthreads();
  if (tid == 0)
    for (int c = 0; c < nchunks && c < kHrBufs; ++c) issue(c);
  // Kept positions inside this CTA's rows.
  const int32_t* idx = a.idx + bh * a.k_sel;
  for (int64_t t = tid; t < a.k_sel; t += kHrThreads) {
    const int32_t j = idx[t];
    if (j < 0 || j >= a.l_prefix) report(a.dev_status, SNAPKV_ERR_INVALID_ARG);
    else if (j >= r0 && j < r1) atomicOr(&bits[(j - r0) >> 5], 1u << ((j - r0) & 31));
  }
  int n = a.len[b];
  if ((int64_t)n > a.cap) {
    if (rank == 0 && tid == 0 && bh % a.heads == 0) report(a.dev_status, SNAPKV_ERR_CAPACITY);
    n = cap;
  }
  if (n < 0) n = 0;
  const int sub = lane / LPR, cl = lane % LPR;
  const int group = warp * RPW + sub;
  const T* qp = static_cast<const T*>(a.q) + bh * D;
  float q[V];
  Elem<T>::widen(ld_nc_v4(qp + cl * V), q);
#pragma unroll
  for (int e = 0; e < V; ++e) q[e] *= a.scale_log2;

  float m = -INFINITY, l = 0.f;
  bool timed_out = false;
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c % kHrBufs;
    if (!ptx::mbar_wait(&bar[buf], (uint32_t)((c / kHrBufs) & 1), &no_abort, kHrWaitLimit)) timed_out = true;
    const uint8_t* kbuf = dsm + buf * kHrChunkBytes;
    const int cr0 = r0 + c * CH;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int rr = group + u * GROUPS;
      float kf[V];
      Elem<T>::widen(*reinterpret_cast<const uint4*>(kbuf + rr * ROW_BYTES + cl * 16), kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < V; ++e) dot = fmaf(q[e], kf[e], dot);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const int r = cr0 + rr;
      if (r < r1 && r < n) {
        if (cl == 0) logit[r - r0] = dot;
        if (dot > m) {
          l = l * ex2(m - dot) + 1.f;
          m = dot;
        } else {
          l += ex2(dot - m);
        }
      }
    }
    __syncthreads();   // every group is done with this buffer
    if (tid == 0 && c + kHrBufs < nchunks) issue(c + kHrBufs);
  }
  if (timed_out && tid == 0) {
    report(a.dev_status, SNAPKV_ERR_TIMEOUT);
    for (int c = (nchunks > kHrBufs ? nchunks - kHrBufs : 0); c < nchunks; ++c)
      ptx::mbar_wait(&bar[c % kHrBufs], (uint32_t)((c / kHrBufs) & 1), &no_abort, kHrWaitLimit);
  }
  if (cl == 0) {
    sm_m[group] = m;
    sm_l[group] = l;
  }
  __syncthreads();
  if (tid == 0) {
    float M = -INFINITY;
    for (int g = 0; g < GROUPS; ++g) M = fmaxf(M, sm_m[g]);
    float Z = 0.f;
    if (M > -INFINITY)
      for (int g = 0; g < GROUPS; ++g)
        if (sm_m[g] > -INFINITY) Z = fmaf(sm_l[g], ex2(sm_m[g] - M), Z);
    cta_m = M;
    cta_l = Z;
  }
  ptx::cluster_sync();   // every CTA's (max, sum) is complete
  // log2 Z of the whole cache, folded in rank order (the same value on every CTA).
  float M = -INFINITY;
  float mr[kHrCtas];
#pragma unroll
  for (int r = 0; r < kHrCtas; ++r) {
    mr[r] = r < (int)csize ? __uint_as_float(ptx::dsmem_ld_u32(ptx::map_rank(&cta_m, (uint32_t)r))) : -INFINITY;
    M = fmaxf(M, mr[r]);
  }
  float Z = 0.f;
#pragma unroll
  for (int r = 0; r < kHrCtas; ++r)
    if (r < (int)csize && mr[r] > -INFINITY)
      Z = fmaf(__uint_as_float(ptx::dsmem_ld_u32(ptx::map_rank(&cta_l, (uint32_t)r))), ex2(mr[r] - M), Z);
  // A_cur[j] > theta  <=>  s'_j > log2 Z + log2 theta
  const float cut = M > -INFINITY ? M + log2f(Z) + a.log2_theta : INFINITY;
  const int pend = min(r1, min(n, (int)a.l_prefix));   // this CTA's prefix rows present in the cache
  uint32_t hits = 0, total = 0;
  for (int r = r0 + tid; r < pend; r += kHrThreads) {
    if (logit[r - r0] > cut) {
      ++total;
      hits += (bits[(r - r0) >> 5] >> ((r - r0) & 31)) & 1u;
    }
  }
  hits = __reduce_add_sync(0xffffffffu, hits);
  total = __reduce_add_sync(0xffffffffu, total);
  if (lane == 0 && (hits | total)) {
    ptx::dsmem_add_u32(ptx::map_rank(&cnt[0], 0), hits);
    ptx::dsmem_add_u32(ptx::map_rank(&cnt[1], 0), total);
  }
  ptx::cluster_sync();   // CTA 0 holds the cluster's counts; no CTA leaves while others read it
  if (rank == 0 && tid == 0) {
    a.hits[bh] = (int32_t)cnt[0];
    a.total[bh] = (int32_t)cnt[1];
  }
}

template <typename T, int D>
cudaError_t launch_cluster(const HitRateJob& job, const HrArgs& a) {
  const int64_t bh = (int64_t)job.batch * job.heads;
  int csize = (int)((job.cap + 2047) / 2048);
  if (csize > kHrCtas) csize = kHrCtas;
  if (csize < 1) csize = 1;
  const int per = (int)((job.cap + csize - 1) / csize);
  const size_t smem = (size_t)kHrBufs * kHrChunkBytes + (size_t)per * 4 + (size_t)((per + 31) / 32) * 4;
  cudaError_t err =
      cudaFuncSetAttribute(hit_rate_cluster_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(bh * csize));
  cfg.blockDim = dim3(kHrThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = job.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, hit_rate_cluster_kernel<T, D>, a);
}

template <typename T, int D>
cudaError_t launch_typed(const HitRateJob& job, const HrArgs& a) {
  if (job.cap <= (int64_t)kHrCtas * kHrClusterRows) return launch_cluster<T, D>(job, a);
  const size_t smem = (size_t)((job.l_prefix + 31) / 32) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    const cudaError_t err =
        cudaFuncSetAttribute(hit_rate_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  hit_rate_kernel<T, D><<<(unsigned)((int64_t)job.batch * job.heads), kHrThreads, smem, job.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hit_rate(const HitRateJob& job) {
  HrArgs a;
  a.q = job.q;
  a.k_cache = job.k_cache;
  a.len = job.len;
  a.idx = job.idx;
  a.hits = job.hits;
  a.total = job.total;
  a.cap = job.cap;
  a.l_prefix = job.l_prefix;
  a.k_sel = job.k_sel;
  a.heads = job.heads;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)job.head_dim));
  a.log2_theta = (float)log2(job.theta);
  a.dev_status = job.dev_status;
  if (job.dtype == SNAPKV_BF16)
    return job.head_dim == 64 ? launch_typed<__nv_bfloat16, 64>(job, a) : launch_typed<__nv_bfloat16, 128>(job, a);
  return job.head_dim == 64 ? launch_typed<float, 64>(job, a) : launch_typed<float, 128>(job, a);
}

}  // namespace snapkv
