// Gather of the kept prefix rows + append of the observation window, K and V together.
//
// SnapKV explainer ("論文解説: SnapKV"), section アルゴリズム (and 実装のポイント, per-head indices):
// K_c = [K[I]; K[L_prefix : L_prompt]] and V_c likewise, I ascending and different per head.
// A bit-exact copy in 16-byte vectors; one thread per 16-byte piece of an output row, so a warp
// moves contiguous 512-byte spans and every HBM sector it touches is used whole.
#include <atomic>

#include "snapkv_common.cuh"
#include "snapkv_internal.h"

namespace snapkv {
namespace {

__global__ void __launch_bounds__(256)
gather_window_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k_out,
                     uint4* __restrict__ v_out, const int32_t* __restrict__ idx, int32_t* __restrict__ len_out,
                     int batch, int heads, int64_t kv_stride, int64_t l_prompt, int64_t l_prefix, int64_t k_sel,
                     int64_t rows_out,
                     int64_t cap, int vpr, int32_t* __restrict__ dev_status) {
  const int64_t per_head = rows_out * vpr;
  const int64_t total = (int64_t)batch * heads * per_head;
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b < batch; b += blockDim.x) len_out[b] = (int32_t)rows_out;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total;
       u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bh = u / per_head;
    const int64_t rem = u - bh * per_head;
    const int64_t r = rem / vpr;
    const int c = (int)(rem - r * vpr);
    const int64_t src = r < k_sel ? (int64_t)idx[bh * k_sel + r] : l_prefix + (r - k_sel);
    if (src < 0 || src >= l_prompt) {  // never for indices from the selection kernel
      report(dev_status, SNAPKV_ERR_INTERNAL);
      continue;
    }
    const int64_t in_at = (bh * kv_stride + src) * vpr + c;
    const int64_t out_at = (bh * cap + r) * vpr + c;
    const uint4 kv = ld_stream_v4(k + in_at);
    const uint4 vv = ld_stream_v4(v + in_at);
    k_out[out_at] = kv;
    v_out[out_at] = vv;
  }
}

}  // namespace

int device_sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];   // 0: not looked up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 148;
  int sms = cache[dev].load(std::memory_order_relaxed);
  if (sms > 0) return sms;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
  cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

cudaError_t launch_gather(const CompressJob& job) {
  const int esize = job.dtype == SNAPKV_BF16 ? 2 : 4;
  const int vpr = job.head_dim * esize / 16;
  const int64_t rows_out = job.k_sel + job.l_obs;
  const int64_t total = (int64_t)job.batch * job.heads * rows_out * vpr;
  const int sms = device_sm_count();
  int64_t blocks = (total + 255) / 256;
  const int64_t cap_blocks = (int64_t)sms * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (blocks < 1) blocks = 1;
  job.mark(2 * kStageGather);
  gather_window_kernel<<<(unsigned)blocks, 256, 0, job.stream>>>(
      static_cast<const uint4*>(job.k), static_cast<const uint4*>(job.v), static_cast<uint4*>(job.k_out),
      static_cast<uint4*>(job.v_out), job.idx, job.len_out, job.batch, job.heads, job.kv_stride, job.l_prompt,
      job.l_prefix,
      job.k_sel, rows_out, job.cap, vpr, job.dev_status);
  job.mark(2 * kStageGather + 1);
  return cudaGetLastError();
}

}  // namespace snapkv
