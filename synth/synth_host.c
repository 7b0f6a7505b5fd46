/*
 * Host side of the seeded synthetic-input generator (plain C, built with -ffp-contract=off).
 * Produces exactly the bits that synth_dev.cu produces on the GPU for the same arguments.
 * No SnapKV arithmetic lives here.
 */
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "synth_gen.h"

/*
 * Fill out[B][H][rows][d] (fp32 if out_bf16 == 0, else bf16 bit patterns).
 * Element (b, h, r, c) draws from stream (layer, seq0 + b, head0 + h, tensor) at counter
 * (row0 + r) * d + c.
 * chan_scale [B][H][d], plant_mask [B][H][rows], plant_vec [B][H][d] are optional (NULL).
 */
typedef struct {
  void* out;
  int out_bf16, B, H, rows, d, row0, seq0, head0;
  uint32_t layer, tensor;
  uint64_t seed;
  const float* chan_scale;
  const uint8_t* plant_mask;
  const float* plant_vec;
  int64_t row_begin, row_end; /* flattened ((b, h), r) row range of this worker */
} fill_job;

static void fill_rows(const fill_job* j) {
  const uint32_t s_hi = synth_stream_hi(j->layer, j->tensor);
  for (int64_t fr = j->row_begin; fr < j->row_end; ++fr) {
    const int64_t bh = fr / j->rows;
    const int r = (int)(fr % j->rows);
    const int b = (int)(bh / j->H), h = (int)(bh % j->H);
    const uint32_t s_lo = synth_stream_lo((uint32_t)(j->seq0 + b), (uint32_t)(j->head0 + h));
    const int planted = j->plant_mask ? (int)j->plant_mask[fr] : 0;
    for (int c = 0; c < j->d; ++c) {
      const uint32_t counter = (uint32_t)(j->row0 + r) * (uint32_t)j->d + (uint32_t)c;
      const float scale = j->chan_scale ? j->chan_scale[bh * j->d + c] : 1.0f;
      const float plant = planted ? j->plant_vec[bh * j->d + c] : 0.0f;
      const float z = synth_element(j->seed, s_lo, s_hi, counter, j->chan_scale != NULL, scale, planted,
                                    plant);
      const size_t at = (size_t)fr * (size_t)j->d + (size_t)c;
      if (j->out_bf16)
        ((uint16_t*)j->out)[at] = synth_bf16_rne(z);
      else
        ((float*)j->out)[at] = z;
    }
  }
}

static void* fill_worker(void* arg) {
  fill_rows((const fill_job*)arg);
  return NULL;
}

int synth_fill(void* out, int out_bf16, int B, int H, int rows, int d, int row0, int seq0,
               int head0, uint32_t layer, uint32_t tensor, uint64_t seed, const float* chan_scale,
               const uint8_t* plant_mask, const float* plant_vec, int threads) {
  if (!out || B < 0 || H < 0 || rows < 0 || d <= 0) return 1;
  if (plant_mask && !plant_vec) return 1;
  const int64_t total_rows = (int64_t)B * H * rows;
  if (threads < 1) threads = 1;
  if (threads > 64) threads = 64;
  if ((int64_t)threads > total_rows / 64 + 1) threads = (int)(total_rows / 64 + 1);
  fill_job jobs[64];
  pthread_t tids[64];
  for (int t = 0; t < threads; ++t) {
    fill_job j = {out, out_bf16, B, H, rows, d, row0, seq0, head0, layer, tensor, seed,
                  chan_scale, plant_mask, plant_vec,
                  total_rows * t / threads, total_rows * (t + 1) / threads};
    jobs[t] = j;
  }
  int started = 0;
  for (int t = 1; t < threads; ++t) {
    if (pthread_create(&tids[t], NULL, fill_worker, &jobs[t]) != 0) break;
    started = t;
  }
  fill_rows(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
  for (int t = started + 1; t < threads; ++t) fill_rows(&jobs[t]); /* threads that failed to start */
  return 0;
}

/* Per-channel key scales s_c of (layer, seq0 + b, h) for c < d, out[B][H][d]. */
void synth_chan_scales(float* out, int B, int H, int d, int seq0, uint32_t layer, uint64_t seed) {
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int c = 0; c < d; ++c)
        out[((size_t)b * H + h) * d + c] =
            synth_chan_scale(seed, layer, (uint32_t)(seq0 + b), (uint32_t)h, (uint32_t)c);
}

/* Raw 32-bit draws of stream (layer, seq, head, tensor) at counters [0, n). */
void synth_u32_stream(uint32_t* out, int n, uint64_t seed, uint32_t layer, uint32_t seq,
                      uint32_t head, uint32_t tensor) {
  const uint32_t s_lo = synth_stream_lo(seq, head), s_hi = synth_stream_hi(layer, tensor);
  for (int i = 0; i < n; ++i) out[i] = synth_u32(seed, s_lo, s_hi, (uint32_t)i);
}

/* One raw Philox4x32-10 block, for known-answer tests of the generator. */
void synth_philox_block(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  synth_u32x4 c;
  memcpy(c.v, ctr, sizeof c.v);
  const synth_u32x4 r = synth_philox4x32_10(c, key[0], key[1]);
  memcpy(out, r.v, sizeof r.v);
}

/*
 * m distinct integers from [0, n), chosen uniformly without replacement by Floyd's
 * algorithm (R. W. Floyd, as given by Bentley, "Programming Pearls", CACM 1987), drawing
 * from stream (layer, seq, head, tensor). Integers in [0, j] use the multiply-shift map
 * floor(u * (j + 1) / 2^32). Output is in ascending order. Returns 0 on success.
 */
int synth_floyd(int32_t* out, int32_t n, int32_t m, uint64_t seed, uint32_t layer, uint32_t seq,
                uint32_t head, uint32_t tensor, uint8_t* scratch /* n bytes, zeroed here */) {
  if (m < 0 || n < 0 || m > n) return 1;
  memset(scratch, 0, (size_t)n);
  const uint32_t s_lo = synth_stream_lo(seq, head), s_hi = synth_stream_hi(layer, tensor);
  uint32_t draw = 0;
  for (int32_t j = n - m; j < n; ++j) {
    const uint32_t u = synth_u32(seed, s_lo, s_hi, draw++);
    const int32_t t = (int32_t)(((uint64_t)u * (uint64_t)(uint32_t)(j + 1)) >> 32);
    if (scratch[t])
      scratch[j] = 1;
    else
      scratch[t] = 1;
  }
  int32_t w = 0;
  for (int32_t i = 0; i < n; ++i)
    if (scratch[i]) out[w++] = i;
  return w == m ? 0 : 2;
}
