// Internal helpers shared by the SnapKV kernels (sm_103a). Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/snapkv.h"

namespace snapkv {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x with the hardware ex2 instruction (approximate, relative error a few 2^-23; subnormal results
// flush to zero, which only drops weights below 2^-126).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void report(int32_t* dev_status, int32_t bits) {
  if (dev_status) atomicOr(dev_status, bits);
}

// Bounds-checked build (compiled with -DSNAPKV_CHECKED): the global indices a kernel computes from
// data or from its own bookkeeping are checked before the access; a violation is reported as
// SNAPKV_ERR_INTERNAL (a library bug) and the access is skipped. The regular build compiles every
// check away (the index arithmetic is correct by construction there, and the tests run the checked
// build to show it).
#ifdef SNAPKV_CHECKED
__device__ __forceinline__ bool in_bounds(bool ok, int32_t* dev_status) {
  if (!ok) report(dev_status, SNAPKV_ERR_INTERNAL);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool, int32_t*) { return true; }
#endif

// Element type traits: 16-byte vectors of 8 bf16 or 4 fp32, widened to fp32.
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kVec = 4;
  __device__ __forceinline__ static void widen(const uint4& raw, float* out) {
    out[0] = __uint_as_float(raw.x);
    out[1] = __uint_as_float(raw.y);
    out[2] = __uint_as_float(raw.z);
    out[3] = __uint_as_float(raw.w);
  }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static void widen(const uint4& raw, float* out) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Streaming 16-byte load (no L1 allocation) for data read exactly once.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace snapkv
