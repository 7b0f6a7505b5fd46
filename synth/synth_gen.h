/*
 * Seeded synthetic-input generator, shared by the host (plain C) and the device (CUDA).
 *
 * This header holds NO SnapKV arithmetic. It only turns (seed, stream, counter) into the
 * input values the tests and the benchmark feed to both the CPU oracle and the CUDA path:
 *
 *   - Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and Shaw,
 *     "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): a 128-bit counter and a
 *     64-bit key, ten rounds of two 32x32->64 multiplies, key bumped by the Weyl constants.
 *   - An approximately standard normal value built as an Irwin-Hall(12) sum of twelve
 *     16-bit uniforms: N = (sum(u_k + 1/2) - 6*2^16) * 2^-16. It is exact in fp32
 *     (|sum| < 2^20), has mean exactly 0, variance 1 - 2^-32 and tails at +-6.
 *   - A uniform in [0,1) on 24 bits, and fp32 -> bf16 round-to-nearest-even done on the
 *     bit pattern, so both sides give bit-identical values without libm.
 *
 * Every floating-point step below is a single IEEE fp32 operation (the host library is built
 * with -ffp-contract=off; the device code uses the explicitly rounded intrinsics), so the
 * host and the device produce the same bits.
 */
#ifndef SYNTH_GEN_H
#define SYNTH_GEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_HD __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

/* Tensor ids: which random stream of a (layer, sequence, head) a tensor draws from. */
enum {
  SYNTH_T_Q = 1,       /* queries (only the observation-window rows are ever drawn)   */
  SYNTH_T_K = 2,       /* keys of the prompt                                           */
  SYNTH_T_V = 3,       /* values of the prompt                                         */
  SYNTH_T_SCALE = 4,   /* per-channel key scale s_c ~ U(0.5, 2)                         */
  SYNTH_T_PLANT = 5,   /* positions of the planted keys                               */
  SYNTH_T_LEN = 6,     /* ragged prompt lengths                                       */
  SYNTH_T_QNEW = 7,    /* decode-step query                                           */
  SYNTH_T_KNEW = 8,    /* decode-step key                                             */
  SYNTH_T_VNEW = 9     /* decode-step value                                           */
};

typedef struct { uint32_t v[4]; } synth_u32x4;

SYNTH_HD synth_u32x4 synth_philox4x32_10(synth_u32x4 ctr, uint32_t k0, uint32_t k1) {
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)ctr.v[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)ctr.v[2];
    synth_u32x4 n;
    n.v[0] = (uint32_t)(p1 >> 32) ^ ctr.v[1] ^ k0;
    n.v[1] = (uint32_t)p1;
    n.v[2] = (uint32_t)(p0 >> 32) ^ ctr.v[3] ^ k1;
    n.v[3] = (uint32_t)p0;
    ctr = n;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return ctr;
}

/* Stream id of (layer, sequence, head, tensor). Distinct tuples give distinct counters. */
SYNTH_HD uint32_t synth_stream_lo(uint32_t seq, uint32_t head) { return (seq << 16) | (head & 0xFFFFu); }
SYNTH_HD uint32_t synth_stream_hi(uint32_t layer, uint32_t tensor) { return (layer << 8) | (tensor & 0xFFu); }

/* Counter layout: {element, stream_lo, stream_hi, word}. word selects one of two blocks. */
SYNTH_HD synth_u32x4 synth_block(uint64_t seed, uint32_t s_lo, uint32_t s_hi, uint32_t element,
                                 uint32_t word) {
  synth_u32x4 c;
  c.v[0] = element;
  c.v[1] = s_lo;
  c.v[2] = s_hi;
  c.v[3] = word;
  return synth_philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
}

/* Irwin-Hall(12) normal of one element: twelve 16-bit halves of six 32-bit words. */
SYNTH_HD float synth_normal(uint64_t seed, uint32_t s_lo, uint32_t s_hi, uint32_t element) {
  const synth_u32x4 a = synth_block(seed, s_lo, s_hi, element, 0u);
  const synth_u32x4 b = synth_block(seed, s_lo, s_hi, element, 1u);
  const uint32_t w[6] = {a.v[0], a.v[1], a.v[2], a.v[3], b.v[0], b.v[1]};
  int32_t sum = 0;
  for (int i = 0; i < 6; ++i) sum += (int32_t)(w[i] & 0xFFFFu) + (int32_t)(w[i] >> 16);
  /* sum(u + 1/2) - 6*2^16 = sum - 393210, scaled by 2^-16: both steps exact in fp32. */
  return (float)(sum - 393210) * (1.0f / 65536.0f);
}

/* Uniform on [0,1) with 24 random bits (exact in fp32). */
SYNTH_HD float synth_uniform(uint64_t seed, uint32_t s_lo, uint32_t s_hi, uint32_t element) {
  const synth_u32x4 a = synth_block(seed, s_lo, s_hi, element, 0u);
  return (float)(a.v[0] >> 8) * (1.0f / 16777216.0f);
}

/* Raw 32-bit draw (for integer choices made on the host). */
SYNTH_HD uint32_t synth_u32(uint64_t seed, uint32_t s_lo, uint32_t s_hi, uint32_t element) {
  return synth_block(seed, s_lo, s_hi, element, 0u).v[0];
}

#if defined(__CUDA_ARCH__)
SYNTH_HD float synth_mul(float a, float b) { return __fmul_rn(a, b); }
SYNTH_HD float synth_add(float a, float b) { return __fadd_rn(a, b); }
SYNTH_HD uint32_t synth_f32_bits(float f) { return __float_as_uint(f); }
#else
SYNTH_HD float synth_mul(float a, float b) { return a * b; }
SYNTH_HD float synth_add(float a, float b) { return a + b; }
SYNTH_HD uint32_t synth_f32_bits(float f) {
  union { float f; uint32_t u; } x;
  x.f = f;
  return x.u;
}
#endif

/* fp32 -> bf16, round to nearest, ties to even (inputs here are finite). */
SYNTH_HD uint16_t synth_bf16_rne(float f) {
  uint32_t u = synth_f32_bits(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/*
 * One element of a generated tensor, as fp32 before any storage rounding:
 *   z = normal(stream, counter)
 *   z = z * scale     if a per-channel scale is given   (one fp32 multiply)
 *   z = z + plant     if the row is planted            (one fp32 add)
 */
SYNTH_HD float synth_element(uint64_t seed, uint32_t s_lo, uint32_t s_hi, uint32_t counter,
                             int has_scale, float scale, int planted, float plant) {
  float z = synth_normal(seed, s_lo, s_hi, counter);
  if (has_scale) z = synth_mul(z, scale);
  if (planted) z = synth_add(z, plant);
  return z;
}

/* Per-channel key scale s_c = 0.5 + 1.5*u, u ~ U[0,1) (one fp32 multiply, one fp32 add). */
SYNTH_HD float synth_chan_scale(uint64_t seed, uint32_t layer, uint32_t seq, uint32_t head,
                                uint32_t channel) {
  const float u = synth_uniform(seed, synth_stream_lo(seq, head),
                                synth_stream_hi(layer, SYNTH_T_SCALE), channel);
  return synth_add(0.5f, synth_mul(1.5f, u));
}

#endif /* SYNTH_GEN_H */
