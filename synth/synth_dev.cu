/*
 * Device side of the seeded synthetic-input generator: the same element function as
 * synth_host.c, one thread per element, so a tensor generated here is bit-identical to the
 * host copy. Used only to create inputs on the GPU (tests, benchmark); no SnapKV arithmetic.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_gen.h"

__global__ void synth_fill_kernel(void* __restrict__ out, int out_bf16, int B, int H, int rows,
                                  int d, int row0, int seq0, int head0, uint32_t layer,
                                  uint32_t tensor,
                                  uint64_t seed, const float* __restrict__ chan_scale,
                                  const uint8_t* __restrict__ plant_mask,
                                  const float* __restrict__ plant_vec) {
  const size_t total = (size_t)B * H * rows * d;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t at = (size_t)blockIdx.x * blockDim.x + threadIdx.x; at < total; at += stride) {
    const int c = (int)(at % d);
    const size_t row_flat = at / d;               /* (b*H + h)*rows + r */
    const int r = (int)(row_flat % rows);
    const size_t bh = row_flat / rows;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const uint32_t s_lo = synth_stream_lo((uint32_t)(seq0 + b), (uint32_t)(head0 + h));
    const uint32_t s_hi = synth_stream_hi(layer, tensor);
    const uint32_t counter = (uint32_t)(row0 + r) * (uint32_t)d + (uint32_t)c;
    const int planted = plant_mask ? (int)plant_mask[row_flat] : 0;
    const float scale = chan_scale ? chan_scale[bh * d + c] : 1.0f;
    const float plant = planted ? plant_vec[bh * d + c] : 0.0f;
    const float z = synth_element(seed, s_lo, s_hi, counter, chan_scale != nullptr, scale, planted,
                                  plant);
    if (out_bf16)
      reinterpret_cast<uint16_t*>(out)[at] = synth_bf16_rne(z);
    else
      reinterpret_cast<float*>(out)[at] = z;
  }
}

extern "C" int synth_fill_device(void* out, int out_bf16, int B, int H, int rows, int d, int row0,
                                 int seq0, int head0, uint32_t layer, uint32_t tensor, uint64_t seed,
                                 const float* chan_scale, const uint8_t* plant_mask,
                                 const float* plant_vec, void* stream) {
  if (!out || B < 0 || H < 0 || rows < 0 || d <= 0) return 1;
  if (plant_mask && !plant_vec) return 1;
  const size_t total = (size_t)B * H * rows * d;
  if (total == 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t blocks = (total + 255) / 256;
  const size_t cap = (size_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  synth_fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      out, out_bf16, B, H, rows, d, row0, seq0, head0, layer, tensor, seed, chan_scale, plant_mask,
      plant_vec);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
