// Max-pool + top-k + ascending compaction, one CTA per (sequence, head).
//
// SnapKV explainer ("論文解説: SnapKV"), sections クラスタリングによる文脈保持 and 投票メカニズム:
// P_j = max of the vote C over |j' - j| <= K_pool / 2 (clipped to the prefix, i.e. -inf padding),
// then the k positions of largest P, ties to the lower index, emitted in ascending order.
//
// Selection is exact: every P_j is >= +0, so its fp32 bit pattern read as uint32 orders like the
// value. A three-digit MSB-first radix select (11 + 11 + 10 bits) finds tau, the k-th largest
// pattern, and how many copies of tau to keep; one ordered compaction pass then keeps every
// P_j > tau and the lowest-index copies of tau, writing the indices ascending.
#include "snapkv_common.cuh"
#include "snapkv_internal.h"

namespace snapkv {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBins = 2048;

// Exclusive block-wide prefix sum of one value per thread (all threads must call).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* sh_warp, uint32_t* total) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? sh_warp[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) sh_warp[lane] = w;  // inclusive warp totals
    if (lane == kWarps - 1) *total = w;
  }
  __syncthreads();
  const uint32_t base = warp > 0 ? sh_warp[warp - 1] : 0u;
  const uint32_t out = base + x - v;
  __syncthreads();
  return out;
}

__global__ void __launch_bounds__(kThreads)
pool_topk_kernel(const float* __restrict__ c_all, float* __restrict__ p_all, int32_t* __restrict__ idx_all,
                 int64_t l_prefix, int radius, int64_t k_sel) {
  __shared__ uint32_t hist[kMaxBins];
  __shared__ uint32_t sh_warp[kWarps];
  __shared__ uint32_t sh_total;
  __shared__ uint32_t sh_digit, sh_above;

  const int tid = threadIdx.x;
  const int64_t bh = blockIdx.x;
  const float* c = c_all + bh * l_prefix;
  float* p = p_all + bh * l_prefix;
  int32_t* idx = idx_all + bh * k_sel;
  const int L = (int)l_prefix;

  for (int j = tid; j < L; j += kThreads) {
    float m = c[j];
    const int lo = max(0, j - radius), hi = min(L - 1, j + radius);
    for (int q = lo; q <= hi; ++q) m = fmaxf(m, c[q]);
    p[j] = m;
  }
  __syncthreads();
  if (k_sel <= 0) return;

  // Radix select of the k-th largest bit pattern.
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k_sel;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass], nb = 1 << widths[pass];
    for (int b = tid; b < nb; b += kThreads) hist[b] = 0u;
    __syncthreads();
    for (int j = tid; j < L; j += kThreads) {
      const uint32_t u = __float_as_uint(p[j]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & (uint32_t)(nb - 1)], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // Lane l owns bins [nb - (l+1)*per, nb - l*per), scanned from the top.
      const int per = nb / 32;
      const int top = nb - tid * per;
      uint32_t s = 0;
      for (int b = top - 1; b >= top - per; --b) s += hist[b];
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      const uint32_t before = incl - s;
      if (before < krem && krem <= incl) {
        uint32_t acc = before;
        for (int b = top - 1; b >= top - per; --b) {
          const uint32_t h = hist[b];
          if (acc + h >= krem) {
            sh_digit = (uint32_t)b;
            sh_above = acc;
            break;
          }
          acc += h;
        }
      }
    }
    __syncthreads();
    prefix |= sh_digit << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    krem -= sh_above;
    __syncthreads();
  }
  const uint32_t tau = prefix;
  const uint32_t need_eq = krem;  // copies of tau to keep, lowest index first

  // Ordered compaction over contiguous segments.
  const int seg = (L + kThreads - 1) / kThreads;
  const int j0 = min(L, tid * seg), j1 = min(L, j0 + seg);
  uint32_t gt = 0, eq = 0;
  for (int j = j0; j < j1; ++j) {
    const uint32_t u = __float_as_uint(p[j]);
    gt += u > tau;
    eq += u == tau;
  }
  const uint32_t eq_before = block_exclusive_scan(eq, sh_warp, &sh_total);
  const uint32_t take_eq = eq_before >= need_eq ? 0u : min(eq, need_eq - eq_before);
  uint32_t pos = block_exclusive_scan(gt + take_eq, sh_warp, &sh_total);
  uint32_t e = eq_before;
  for (int j = j0; j < j1; ++j) {
    const uint32_t u = __float_as_uint(p[j]);
    bool keep = u > tau;
    if (u == tau) {
      keep = e < need_eq;
      ++e;
    }
    if (keep) {
      if ((int64_t)pos < k_sel) idx[pos] = j;  // always true when the select above is exact
      ++pos;
    }
  }
}

}  // namespace

cudaError_t launch_pool_topk(const CompressJob& job) {
  const int64_t bh = (int64_t)job.batch * job.heads;
  job.mark(2 * kStageTopk);
  pool_topk_kernel<<<(unsigned)bh, kThreads, 0, job.stream>>>(job.c, job.p, job.idx, job.l_prefix,
                                                              job.pool_kernel / 2, job.k_sel);
  job.mark(2 * kStageTopk + 1);
  return cudaGetLastError();
}

}  // namespace snapkv
