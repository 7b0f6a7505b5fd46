// Score + softmax + vote, SIMT fp32 (any dtype; the fp32-input path and the general fallback).
//
// SnapKV explainer ("論文解説: SnapKV"), sections 投票メカニズム and アルゴリズム: for every window
// query i the logits s_ij = q_i . k_j / sqrt(d) over the prompt columns it sees, the row softmax
// w_ij = exp(s_ij - m_i) / Z_i, and the vote C_j = sum_i w_ij over the prefix columns.
//
// Two launches per call. Pass 0 (statistics) streams every prompt column once and leaves, per
// (head, chunk of columns, window row), the partial row maximum and partial sum of exponentials.
// Pass 1 (vote) merges those partials into m_i and 1/Z_i, recomputes the logits of the prefix
// columns and writes C_j. Logits live in the log2 domain (scaled by log2(e)/sqrt(d)) so every
// exponential is one ex2. Under grouped-query attention a KV head's window rows are its query
// heads' rows one after another (rows = G * L_obs); row i sits at window position i mod L_obs, and
// the vote sums every row.
#include "snapkv_common.cuh"
#include "snapkv_internal.h"

namespace snapkv {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;                   // prompt columns per tile (one per thread of a group)
constexpr int kGroups = kThreads / kTile;   // window rows are split over 4 groups of threads

struct VoteParams {
  const void* q_obs;
  const void* k;
  float* partial;       // [B*H][n_chunk_all][rows][2] (m, z)
  float* c_out;         // [B*H][l_prefix]
  int64_t l_prompt, l_prefix, kv_stride;
  int l_obs, rows, scope, chunk, n_chunk_all;   // rows: window-query rows per head
  float scale_log2;     // log2(e) / sqrt(d)
  int32_t* dev_status;  // the bounds-checked build reports here
};

template <int D, int QG>
constexpr size_t vote_smem_floats() {
  return (size_t)D * QG * kGroups + (size_t)kTile * (D + 1) + 2 * QG * kGroups + kGroups * kTile +
         2 * (kThreads / 32) * QG;
}

template <typename T, int D, int QG>
__global__ void __launch_bounds__(kThreads) vote_simt_kernel(VoteParams a, int pass) {
  constexpr int LQ = QG * kGroups;      // padded window rows
  constexpr int V = Elem<T>::kVec;      // elements per 16-byte vector
  constexpr int VPR = D / V;            // vectors per row
  extern __shared__ __align__(16) float smem[];
  float* qT = smem;                        // [D][LQ], transposed window queries
  float* kS = qT + D * LQ;                 // [kTile][D + 1], one key tile in fp32
  float* st_m = kS + kTile * (D + 1);      // [LQ] final row max (pass 1)
  float* st_zi = st_m + LQ;                // [LQ] final 1 / Z   (pass 1)
  float* red = st_zi + LQ;                 // [kGroups][kTile] partial votes (pass 1)
  float* wred = red + kGroups * kTile;     // [warps][QG][2] warp statistics (pass 0)

  __shared__ int row_pos[LQ];   // window position of each query row (row mod L_obs)
  const int tid = threadIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t col0 = (int64_t)blockIdx.x * a.chunk;
  const int64_t col1 = min(col0 + (int64_t)a.chunk, pass == 0 ? a.l_prompt : a.l_prefix);
  const T* qg = static_cast<const T*>(a.q_obs) + bh * a.rows * D;
  const T* kg = static_cast<const T*>(a.k) + bh * a.kv_stride * D;

  for (int i = tid; i < LQ; i += kThreads) row_pos[i] = i % a.l_obs;
  for (int u = tid; u < LQ * VPR; u += kThreads) {
    const int i = u / VPR, cv = u % VPR;
    float f[V];
    if (i < a.rows) {
      Elem<T>::widen(ld_nc_v4(qg + (int64_t)i * D + cv * V), f);
    } else {
#pragma unroll
      for (int e = 0; e < V; ++e) f[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < V; ++e) qT[(cv * V + e) * LQ + i] = f[e];
  }
  if (pass == 1) {
    for (int i = tid; i < LQ; i += kThreads) {
      float m = -INFINITY, z = 0.f;
      if (i < a.rows) {
        const float* pr = a.partial + (bh * a.n_chunk_all * a.rows + i) * 2;
        for (int c = 0; c < a.n_chunk_all; ++c) m = fmaxf(m, pr[(int64_t)c * a.rows * 2]);
        for (int c = 0; c < a.n_chunk_all; ++c) {
          const float mc = pr[(int64_t)c * a.rows * 2], zc = pr[(int64_t)c * a.rows * 2 + 1];
          if (mc != -INFINITY) z += zc * ex2(mc - m);
        }
      }
      st_m[i] = (i < a.rows) ? m : 0.f;
      st_zi[i] = (i < a.rows && z > 0.f) ? 1.f / z : 0.f;
    }
  }
  __syncthreads();

  const int j = tid % kTile, g = tid / kTile;
  float m_run[QG], z_run[QG];
#pragma unroll
  for (int r = 0; r < QG; ++r) {
    m_run[r] = -INFINITY;
    z_run[r] = 0.f;
  }

  for (int64_t t0 = col0; t0 < col1; t0 += kTile) {
    for (int u = tid; u < kTile * VPR; u += kThreads) {
      const int r = u / VPR, cv = u % VPR;
      float f[V];
      if (t0 + r < col1) {
        Elem<T>::widen(ld_nc_v4(kg + (t0 + r) * D + cv * V), f);
      } else {
#pragma unroll
        for (int e = 0; e < V; ++e) f[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < V; ++e) kS[r * (D + 1) + cv * V + e] = f[e];
    }
    __syncthreads();
    float acc[QG];
#pragma unroll
    for (int r = 0; r < QG; ++r) acc[r] = 0.f;
#pragma unroll 4
    for (int c = 0; c < D; ++c) {
      const float kv = kS[j * (D + 1) + c];
      const float4* q4 = reinterpret_cast<const float4*>(qT + c * LQ + g * QG);
#pragma unroll
      for (int u = 0; u < QG / 4; ++u) {
        const float4 q = q4[u];
        acc[4 * u + 0] = fmaf(q.x, kv, acc[4 * u + 0]);
        acc[4 * u + 1] = fmaf(q.y, kv, acc[4 * u + 1]);
        acc[4 * u + 2] = fmaf(q.z, kv, acc[4 * u + 2]);
        acc[4 * u + 3] = fmaf(q.w, kv, acc[4 * u + 3]);
      }
    }
    __syncthreads();
    const int64_t col = t0 + j;
    if (pass == 0) {
#pragma unroll
      for (int r = 0; r < QG; ++r) {
        const int i = g * QG + r;
        const bool vis = col < col1 && i < a.rows &&
                         (a.scope == SNAPKV_SCOPE_PROMPT_CAUSAL ? col <= a.l_prefix + row_pos[i] : col < a.l_prefix);
        if (vis) {
          const float s = acc[r] * a.scale_log2;
          if (s > m_run[r]) {
            z_run[r] = z_run[r] * ex2(m_run[r] - s) + 1.f;
            m_run[r] = s;
          } else {
            z_run[r] += ex2(s - m_run[r]);
          }
        }
      }
    } else {
      // Every prefix column is visible to every window row in both scopes.
      float csum = 0.f;
#pragma unroll
      for (int r = 0; r < QG; ++r) {
        const int i = g * QG + r;
        if (i < a.rows) csum += ex2(acc[r] * a.scale_log2 - st_m[i]) * st_zi[i];
      }
      red[g * kTile + j] = csum;
      __syncthreads();
      if (g == 0 && col < col1) {
        float c = red[j];
#pragma unroll
        for (int q = 1; q < kGroups; ++q) c += red[q * kTile + j];
        if (in_bounds(col >= 0 && col < a.l_prefix, a.dev_status)) a.c_out[bh * a.l_prefix + col] = c;
      }
    }
  }

  if (pass == 0) {
    // Merge the running statistics of the 64 threads of each group, then of the 2 warps.
    const int warp = tid / 32, lane = tid % 32;
#pragma unroll
    for (int r = 0; r < QG; ++r) {
      const float mw = warp_max(m_run[r]);
      const float zc = (m_run[r] == -INFINITY) ? 0.f : z_run[r] * ex2(m_run[r] - mw);
      const float zw = warp_sum(zc);
      if (lane == 0) {
        wred[(warp * QG + r) * 2] = mw;
        wred[(warp * QG + r) * 2 + 1] = zw;
      }
    }
    __syncthreads();
    constexpr int kWarpsPerGroup = kTile / 32;
    for (int i = tid; i < a.rows; i += kThreads) {
      const int gg = i / QG, r = i % QG;
      float m = -INFINITY;
      for (int w = 0; w < kWarpsPerGroup; ++w) m = fmaxf(m, wred[((gg * kWarpsPerGroup + w) * QG + r) * 2]);
      float z = 0.f;
      for (int w = 0; w < kWarpsPerGroup; ++w) {
        const float mw = wred[((gg * kWarpsPerGroup + w) * QG + r) * 2];
        if (mw != -INFINITY) z += wred[((gg * kWarpsPerGroup + w) * QG + r) * 2 + 1] * ex2(mw - m);
      }
      float* out = a.partial + ((bh * a.n_chunk_all + blockIdx.x) * a.rows + i) * 2;
      out[0] = m;
      out[1] = z;
    }
  }
}

template <typename T, int D, int QG>
cudaError_t launch_typed(const CompressJob& job, const VoteParams& a) {
  const size_t smem = vote_smem_floats<D, QG>() * sizeof(float);
  auto kern = vote_simt_kernel<T, D, QG>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t bh = (int64_t)job.batch * job.heads;
  job.mark(2 * kStageScore);
  kern<<<dim3(job.n_chunk_all, (unsigned)bh), kThreads, smem, job.stream>>>(a, 0);
  job.mark(2 * kStageScore + 1);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  job.mark(2 * kStageVote);
  if (job.n_chunk_prefix > 0) {
    kern<<<dim3(job.n_chunk_prefix, (unsigned)bh), kThreads, smem, job.stream>>>(a, 1);
    err = cudaGetLastError();
  }
  job.mark(2 * kStageVote + 1);
  return err;
}

template <typename T, int D>
cudaError_t launch_d(const CompressJob& job, const VoteParams& a) {
  if (job.q_rows <= 4 * kGroups) return launch_typed<T, D, 4>(job, a);
  if (job.q_rows <= 8 * kGroups) return launch_typed<T, D, 8>(job, a);
  if (job.q_rows <= 16 * kGroups) return launch_typed<T, D, 16>(job, a);
  return launch_typed<T, D, 32>(job, a);
}

template <typename T>
cudaError_t launch_t(const CompressJob& job, const VoteParams& a) {
  return job.head_dim == 64 ? launch_d<T, 64>(job, a) : launch_d<T, 128>(job, a);
}

}  // namespace

cudaError_t launch_vote_simt(const CompressJob& job) {
  VoteParams a;
  a.q_obs = job.q_obs;
  a.k = job.k;
  a.partial = job.partial;
  a.c_out = job.c;
  a.l_prompt = job.l_prompt;
  a.kv_stride = job.kv_stride;
  a.l_prefix = job.l_prefix;
  a.l_obs = job.l_obs;
  a.rows = job.q_rows;
  a.dev_status = job.dev_status;
  a.scope = job.scope;
  a.chunk = job.vote_chunk;
  a.n_chunk_all = job.n_chunk_all;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)job.head_dim));
  return job.dtype == SNAPKV_BF16 ? launch_t<__nv_bfloat16>(job, a) : launch_t<float>(job, a);
}

}  // namespace snapkv
