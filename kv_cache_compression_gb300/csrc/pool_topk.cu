// Max-pool + top-k + ascending compaction (+ the gather of the kept rows), per (sequence, head).
//
// SnapKV explainer ("論文解説: SnapKV"), sections クラスタリングによる文脈保持 and 投票メカニズム:
// P_j = max of the vote C over |j' - j| <= K_pool / 2 (clipped to the prefix, i.e. -inf padding),
// then the k positions of largest P, ties to the lower index, emitted in ascending order.
//
// Selection is exact: every P_j is >= +0, so its fp32 bit pattern read as uint32 orders like the
// value. A three-digit MSB-first radix select (11 + 11 + 10 bits) finds tau, the k-th largest
// pattern, and how many copies of tau to keep; one ordered compaction pass then keeps every
// P_j > tau and the lowest-index copies of tau, writing the indices ascending.
//
// Two kernels, chosen by the prefix length:
//   * prefixes up to kClusterMaxPrefix: a cluster of up to 8 CTAs per head (fewer, down to one, when
//     the batch alone fills the GPU); each CTA holds a contiguous slice of P in shared memory; the
//     slices' histograms are summed through distributed shared memory and every CTA locates the same
//     digit; the compaction offsets of the slices are exchanged the same way. The kernel also does
//     the gather of the section アルゴリズム (K_c = [K[I]; K[L_prefix:]], V_c likewise): a CTA's kept
//     indices are a contiguous block of the ascending output, so it copies its own kept rows, and a
//     share of the window rows;
//   * longer prefixes: one CTA per head with P in global memory, followed by the separate gather
//     kernel.
#include "sm100_ptx.cuh"
#include "snapkv_common.cuh"
#include "snapkv_internal.h"

namespace snapkv {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBins = 2048;

// Histogram update aggregated over the warp: lanes holding the same digit add once, through
// their lowest lane (the pooled votes share few leading bits, so plain atomics would pile onto a
// handful of bins). Every lane of the warp must call it; `valid` masks lanes with nothing to add.
__device__ __forceinline__ void warp_hist_add(uint32_t* hist, uint32_t digit, bool valid) {
  const uint32_t active = __ballot_sync(0xffffffffu, valid);
  if (!valid) return;
  const uint32_t peers = __match_any_sync(active, digit);
  if ((threadIdx.x & 31) == (uint32_t)(__ffs(peers) - 1)) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

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
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0), nb = pass < 2 ? 2048 : 1024;   // 11 + 11 + 10 bits
    for (int b = tid; b < nb; b += kThreads) hist[b] = 0u;
    __syncthreads();
    for (int j0 = 0; j0 < L; j0 += kThreads) {   // warp-uniform trip count
      const int j = j0 + tid;
      const uint32_t u = j < L ? __float_as_uint(p[j]) : 0u;
      warp_hist_add(hist, (u >> shift) & (uint32_t)(nb - 1), j < L && (u & mask) == prefix);
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

constexpr int kCThreads = 512;
constexpr int kCWarps = kCThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int64_t kClusterMaxSlice = 24 * 1024;   // vote elements per CTA held in shared memory (x2 with P)
constexpr int64_t kClusterMaxPrefix = kMaxCluster * kClusterMaxSlice;

// Exclusive prefix sum over the CTA (all threads must call).
__device__ __forceinline__ uint32_t cta_exclusive_scan(uint32_t v, uint32_t* sh_warp) {
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
    uint32_t w = lane < kCWarps ? sh_warp[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kCWarps) sh_warp[lane] = w;
  }
  __syncthreads();
  const uint32_t out = (warp > 0 ? sh_warp[warp - 1] : 0u) + x - v;
  __syncthreads();
  return out;
}

// Shared-memory words of the cluster kernel: the pooled slice, then the vote with its halo during
// the pool (this slice's histogram afterwards), then the two cluster-histogram buffers.
constexpr int kHistWords = kMaxBins;
constexpr int kPoolChunk = 4096;   // vote values (plus the pooling halo) staged at a time
constexpr int kSumWords = 2 * kMaxBins;

__host__ __device__ constexpr int round4(int x) { return (x + 3) & ~3; }

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// Stages hn (<= kPoolChunk + 1024) vote values starting at prefix position h0 into buf, -inf outside
// [0, L): every load of the chunk is issued before the first store, so the chunk costs one memory
// round trip rather than one per value.
constexpr int kStageLoads = (kPoolChunk + 1024 + 511) / 512;
__device__ __forceinline__ void stage_vote(float* buf, const float* c, int h0, int hn, int L) {
  float x[kStageLoads];
#pragma unroll
  for (int i = 0; i < kStageLoads; ++i) {
    const int q = (int)threadIdx.x + i * (int)blockDim.x;
    const int j = h0 + q;
    x[i] = (q < hn && j >= 0 && j < L) ? __ldcg(c + j) : -INFINITY;
  }
#pragma unroll
  for (int i = 0; i < kStageLoads; ++i) {
    const int q = (int)threadIdx.x + i * (int)blockDim.x;
    if (q < hn) buf[q] = x[i];
  }
}

// Max over the staged window buf[j .. j + 2 radius] (the pool of position j); the explainer's
// presets use kernels of 5 to 13, so those take an unrolled path.
__device__ __forceinline__ float window_max(const float* buf, int j, int radius) {
  float m = buf[j];
  switch (radius) {
    case 2:
#pragma unroll
      for (int q = 1; q <= 4; ++q) m = fmaxf(m, buf[j + q]);
      break;
    case 3:
#pragma unroll
      for (int q = 1; q <= 6; ++q) m = fmaxf(m, buf[j + q]);
      break;
    case 6:
#pragma unroll
      for (int q = 1; q <= 12; ++q) m = fmaxf(m, buf[j + q]);
      break;
    default:
      for (int q = 1; q <= 2 * radius; ++q) m = fmaxf(m, buf[j + q]);
  }
  return m;
}

// One cluster per (sequence, head); CTA `rank` of the cluster owns P[rank * slice, ...).
//
// Each CTA keeps a copy of the cluster-wide histogram. In a radix pass every CTA histograms its
// slice, then adds each non-empty bin into every CTA's copy with distributed-shared-memory
// reductions; after one cluster barrier each CTA holds the whole histogram and finds the digit
// locally. The copies alternate between two buffers, and a buffer is cleared right after its pass
// so the pass after next can add into it.
// Row copies of the fused gather: K and V rows of `vpr` 16-byte pieces.
struct GatherArgs {
  const uint4* k;
  const uint4* v;
  uint4* k_out;
  uint4* v_out;
  int32_t* len_out;
  int64_t kv_stride, cap;   // rows between heads in k / v, rows per head in k_out / v_out
  int64_t c_stride, idx_stride;   // rows between heads in the vote and in the indices
  int32_t* dev_status;            // consistency failures of the gather (a library bug) are reported here
  int vpr, l_obs, heads;
  // Ragged batch (n > 0): sequence s (= head / heads) has its own prefix length and kept count;
  // the kernel's l_prefix, k_sel and slice arguments are then the maxima.
  struct {
    int n;
    int l_prefix[kMaxVarSeq];
    int k[kMaxVarSeq];
  } var;
};

// One step of the radix select: in the complete histogram `s` (nb bins) of the values that match
// the digits found so far, the bin holding the krem-th largest value, counted from the top bin.
// Writes the bin, the count of values in higher bins, whether the bin's values are all kept and the
// bin's count to the shared outputs; every thread of the CTA must call it, and a barrier must come
// before the outputs are read. Thread t holds the four bins of group t counted from the top; a
// block scan gives the values in higher groups.
__device__ __forceinline__ void find_digit(const uint32_t* s, int nb, uint32_t krem, uint32_t* sh_warp,
                                           uint32_t* sh_digit, uint32_t* sh_above, uint32_t* sh_full,
                                           uint32_t* sh_bin) {
  const int tid = threadIdx.x;
  const int ngroups = nb / 4;   // <= kCThreads
  const int grp = ngroups - 1 - tid;
  uint4 g4 = make_uint4(0, 0, 0, 0);
  if (tid < ngroups) g4 = *reinterpret_cast<const uint4*>(s + 4 * grp);
  const uint32_t cnt = g4.x + g4.y + g4.z + g4.w;
  const uint32_t above = cta_exclusive_scan(cnt, sh_warp);
  if (tid < ngroups && above < krem && krem <= above + cnt) {
    uint32_t acc = above;
    const uint32_t hb[4] = {g4.w, g4.z, g4.y, g4.x};   // bins 4 grp + 3 .. 4 grp
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (acc + hb[q] >= krem) {
        *sh_digit = (uint32_t)(4 * grp + 3 - q);
        *sh_above = acc;
        *sh_full = acc + hb[q] == krem ? 1u : 0u;   // the digit's bin is kept whole
        *sh_bin = hb[q];
        break;
      }
      acc += hb[q];
    }
  }
}

// Gather of the section アルゴリズム for one CTA's share of a head (K and V together): the CTA's kept
// prefix rows, which take cache rows p0 .. p0 + n_rows - 1, then the window rows rank, rank + csize,
// ... of the L_obs window. The kept positions are read from `kept` in shared memory when the list
// fit there, else (kept == nullptr) from the head's index row, which this CTA wrote before the
// barrier that precedes the call. 16-byte pieces, four rows' worth of loads in flight per thread; the
// destinations are recomputed for the stores rather than held in registers across the loads, which
// keeps the kernels free of spills.
__device__ __forceinline__ void gather_rows(const GatherArgs& g, int64_t bh, uint32_t rank, uint32_t csize,
                                            const uint32_t* kept, const int32_t* idx, uint32_t p0,
                                            uint32_t n_rows, int64_t l_prefix, int64_t k_sel) {
  const int tid = threadIdx.x;
  const int vpr = g.vpr;
  const uint4* kin = g.k + bh * g.kv_stride * vpr;
  const uint4* vin = g.v + bh * g.kv_stride * vpr;
  uint4* kout = g.k_out + bh * g.cap * vpr;
  uint4* vout = g.v_out + bh * g.cap * vpr;
  const int n_win = (g.l_obs - (int)rank + (int)csize - 1) / (int)csize;   // window rows of this CTA
  const int64_t items = ((int64_t)n_rows + n_win) * vpr;
  constexpr int U = 4;
  const int vsh = __ffs(vpr) - 1;   // 16-byte pieces per row: 8, 16 or 32
  for (int64_t base = tid; base < items; base += (int64_t)U * blockDim.x) {
    uint4 kv[U], vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t it = base + (int64_t)u * blockDim.x;
      if (it < items) {
        const int64_t row = it >> vsh;
        const int c = (int)(it & (vpr - 1));
        int64_t src;
        if (row < (int64_t)n_rows)
          src = kept ? (int64_t)kept[row] : (int64_t)__ldcg(idx + p0 + row);
        else
          src = l_prefix + (int64_t)rank + (row - n_rows) * csize;
        if (in_bounds(src >= 0 && src < g.kv_stride, g.dev_status)) {
          kv[u] = ld_stream_v4(kin + src * vpr + c);
          vv[u] = ld_stream_v4(vin + src * vpr + c);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t it = base + (int64_t)u * blockDim.x;
      if (it < items) {
        const int64_t row = it >> vsh;
        const int c = (int)(it & (vpr - 1));
        const int64_t out = row < (int64_t)n_rows ? (int64_t)p0 + row : k_sel + (int64_t)rank + (row - n_rows) * csize;
        if (in_bounds(out >= 0 && out < g.cap, g.dev_status)) {
          kout[out * vpr + c] = kv[u];
          vout[out * vpr + c] = vv[u];
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kCThreads, 2)   // two CTAs per SM (a 32-head layer in one wave)
pool_topk_cluster_kernel(const float* __restrict__ c_all, int32_t* __restrict__ idx_all, int64_t l_prefix,
                         int radius, int64_t k_sel, int slice, GatherArgs g) {
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* pbits = sm;                                      // [slice] pooled vote bit patterns
  uint32_t* work = sm + round4(slice);                       // 16-B aligned
  float* cbuf = reinterpret_cast<float*>(work);              // [min(slice, kPoolChunk) + 2 * radius] vote + halo
  uint32_t* hist = work;                                     // [kMaxBins] this slice's histogram
  uint32_t* sums = work + round4(max(min(slice, kPoolChunk) + 2 * radius, kHistWords));   // [2][kMaxBins] cluster histograms
  // (the layout above is sized for the largest slice; a ragged batch's shorter sequences use less)
  uint32_t* sh_warp = sums + kSumWords;                      // [32]
  uint32_t* counts = sh_warp + 32;                           // [8 + 1] packed (greater << 16 | equal) per slice
  __shared__ uint32_t sh_digit, sh_above, sh_full, sh_bin;

  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t rank = ptx::cluster_rank(), csize = ptx::cluster_size();
  const int64_t bh = blockIdx.x / csize;
  if (g.var.n > 0) {   // this head's sequence of a ragged batch
    const int sq = (int)(bh / g.heads);
    l_prefix = g.var.l_prefix[sq];
    k_sel = g.var.k[sq];
    slice = (int)((l_prefix + (int64_t)csize - 1) / (int64_t)csize);
  }
  const float* c = c_all + bh * g.c_stride;
  int32_t* idx = idx_all + bh * g.idx_stride;
  const int L = (int)l_prefix;
  const int j0 = min(L, (int)rank * slice), j1 = min(L, j0 + slice);
  const int n = j1 - j0;
  // The vote was written by the score kernel just before, but much of it has left L2 behind the
  // keys streamed since: every 128-byte line of the slice is requested at once.
  for (int q = tid * 32; q < n; q += kCThreads * 32) prefetch_l2(c + j0 + q);

  // A head on one CTA reads its own histograms and skips every cluster exchange.
  const bool alone = csize == 1;
  if (!alone) {
    for (int b = tid; b < kSumWords; b += kCThreads) sums[b] = 0u;
    ptx::cluster_arrive();   // this CTA's cluster histograms are clear (waited for before the first add)
  }

  // Max pool of the slice, kPoolChunk values at a time: the vote (L2-resident) with its halo is
  // staged in shared memory by coalesced independent loads, -inf outside the prefix; then each P_j
  // is a max over the window. (The staging buffer stays small, so that a long prefix's slices leave
  // room for two CTAs per SM.)
  for (int ch0 = 0; ch0 < n; ch0 += kPoolChunk) {
    const int cn = min(kPoolChunk, n - ch0);
    const int h0 = j0 + ch0 - radius, hn = cn + 2 * radius;
    stage_vote(cbuf, c, h0, hn, L);
    __syncthreads();
    for (int j = tid; j < cn; j += kCThreads) pbits[ch0 + j] = __float_as_uint(window_max(cbuf, j, radius));
    __syncthreads();   // the next chunk, and the histogram below, reuse the staging buffer
  }
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k_sel;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0), nb = pass < 2 ? 2048 : 1024;   // 11 + 11 + 10 bits
    uint32_t* s = sums + (pass & 1) * kMaxBins;
    for (int b = tid; b < nb; b += kCThreads) hist[b] = 0u;
    __syncthreads();
    if (pass == 0) {
      // Every value counts, and a warp's 32 neighbouring values mostly share their top digit: the
      // warp adds each distinct digit once.
      for (int jb = 0; jb < n; jb += kCThreads) {   // warp-uniform trip count
        const int j = jb + tid;
        const uint32_t u = j < n ? pbits[j] : 0u;
        warp_hist_add(hist, (u >> shift) & (uint32_t)(nb - 1), j < n);
      }
    } else {
      // Only the values in the chosen bin count (a few percent), spread over the lower digits:
      // plain shared-memory atomics (256-head layer: 62.4 -> 60.4 us per launch against the
      // warp-aggregated add).
      for (int j = tid; j < n; j += kCThreads) {
        const uint32_t u = pbits[j];
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & (uint32_t)(nb - 1)], 1u);
      }
    }
    __syncthreads();
    const uint32_t* whole = hist;   // the head's histogram
    if (!alone) {
      if (pass == 0) ptx::cluster_wait();
      for (int b = tid; b < nb; b += kCThreads) {
        const uint32_t v = hist[b];
        if (v != 0u)
          for (uint32_t r = 0; r < csize; ++r) ptx::dsmem_add_u32(ptx::map_rank(s + b, r), v);
      }
      ptx::cluster_sync();   // every slice's bins have been added into every copy
      whole = s;
    }
    find_digit(whole, nb, krem, sh_warp, &sh_digit, &sh_above, &sh_full, &sh_bin);
    __syncthreads();
    prefix |= sh_digit << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    krem -= sh_above;
    // When every value with the digits found so far is kept, the lower digits cannot change the
    // selection: stop (every CTA reads the same histogram, so all stop at the same pass).
    if (sh_full) break;
    if (pass == 0 && !alone)   // cleared before this CTA arrives at the next pass's barrier
      for (int b = tid; b < nb; b += kCThreads) s[b] = 0u;
  }
  // Selection: every value whose decided digits exceed tau's, plus the lowest-index need_eq of
  // those equal to tau's (all of them when the select stopped early).
  const uint32_t tau = prefix, need_eq = krem;

  // Ordered compaction, warp-ordered: warp w owns the contiguous segment [w * seg, (w + 1) * seg) of
  // the slice (seg a multiple of 32) and reads it 32 consecutive values at a time, so lane l reads
  // word base + l (no bank conflicts); ballots give each value's rank among the greater and equal
  // values before it. Slices are in rank order; a slice holds fewer than 2^16 values, so its
  // (greater, equal) counts travel as one packed word, and each CTA stores its total into the later
  // slices' CTAs.
  const int warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int seg = ((n + kCWarps * 32 - 1) / (kCWarps * 32)) * 32;
  const int s0 = min(n, warp * seg), s1 = min(n, s0 + seg);
  uint32_t w_gt = 0, w_eq = 0;
  for (int base = s0; base < s1; base += 32) {   // warp-uniform trip count
    const int j = base + lane;
    const uint32_t u = j < s1 ? (pbits[j] & mask) : 0u;
    w_gt += __popc(__ballot_sync(0xffffffffu, j < s1 && u > tau));
    w_eq += __popc(__ballot_sync(0xffffffffu, j < s1 && u == tau));
  }
  if (lane == 0) sh_warp[warp] = (w_gt << 16) | w_eq;
  __syncthreads();
  uint32_t packed_in = 0, cta_total = 0;   // this warp's exclusive prefix, the CTA's total
  for (int w = 0; w < kCWarps; ++w) {
    const uint32_t x = sh_warp[w];
    if (w < warp) packed_in += x;
    cta_total += x;
  }
  if (tid == 0) {
    for (uint32_t r = rank + 1; r < csize; ++r) ptx::dsmem_st_u32(ptx::map_rank(counts + rank, r), cta_total);
    counts[kMaxCluster] = cta_total;
  }
  if (alone)
    __syncthreads();
  else
    ptx::cluster_sync();   // last access to another CTA's shared memory
  const uint32_t before = (uint32_t)lane < rank ? counts[lane] : 0u;
  const uint32_t gt_before = warp_sum_u32(before >> 16), eq_before = warp_sum_u32(before & 0xffffu);
  // Output position of a kept value: every greater value before it, plus the equal values before it
  // that are kept (the lowest-index need_eq copies of tau are kept). The CTA's kept rows take the
  // output positions [p0, p0 + n_kept); `kept` (the histogram space) lists them in order.
  const uint32_t p0 = gt_before + (eq_before < need_eq ? eq_before : need_eq);
  const uint32_t eq_cta = counts[kMaxCluster] & 0xffffu;
  const uint32_t eq_end = eq_before + eq_cta;
  const uint32_t n_kept = (counts[kMaxCluster] >> 16) + (eq_end < need_eq ? eq_end : need_eq) -
                          (eq_before < need_eq ? eq_before : need_eq);
  uint32_t* kept = work;
  const int kept_cap = round4(max(min(slice, kPoolChunk) + 2 * radius, kHistWords));   // the work space
  uint32_t g_run = gt_before + (packed_in >> 16);      // greater values before this warp's next chunk
  uint32_t e_run = eq_before + (packed_in & 0xffffu);  // equal values before it
  for (int base = s0; base < s1; base += 32) {
    const int j = base + lane;
    const uint32_t u = j < s1 ? (pbits[j] & mask) : 0u;
    const bool is_gt = j < s1 && u > tau, is_eq = j < s1 && u == tau;
    const uint32_t gtb = __ballot_sync(0xffffffffu, is_gt), eqb = __ballot_sync(0xffffffffu, is_eq);
    const uint32_t e_rank = e_run + __popc(eqb & lt_mask);
    if (is_gt || (is_eq && e_rank < need_eq)) {
      const uint32_t pos = g_run + __popc(gtb & lt_mask) + (e_rank < need_eq ? e_rank : need_eq);
      if ((int64_t)pos < k_sel) {
        idx[pos] = j0 + j;
        if (pos - p0 < (uint32_t)kept_cap) kept[pos - p0] = (uint32_t)(j0 + j);
      }
    }
    g_run += __popc(gtb);
    e_run += __popc(eqb);
  }
  __syncthreads();

  // The kept rows land in [p0, p0 + n_kept) of the first k_sel cache rows, and every one of them
  // was listed above; an inconsistent count would be a library bug: reported, not followed.
  uint32_t n_rows = n_kept;
  if ((int64_t)p0 + n_kept > k_sel) {
    if (tid == 0) report(g.dev_status, SNAPKV_ERR_INTERNAL);
    n_rows = 0;
  }
  gather_rows(g, bh, rank, csize, n_kept <= (uint32_t)kept_cap ? kept : nullptr, idx, p0, n_rows, l_prefix, k_sel);
  if (rank == 0 && tid == 0 && bh % g.heads == 0) g.len_out[bh / g.heads] = (int32_t)(k_sel + g.l_obs);
}

}  // namespace

bool pool_topk_ragged_eligible(const CompressJob& job) {
  if (job.n_var < 1 || job.n_var > kMaxVarSeq) return false;
  if (!(job.l_prefix <= kClusterMaxPrefix && job.pool_kernel <= 1025)) return false;
  for (int b = 0; b < job.n_var; ++b)
    if (job.var_k[b] < 1) return false;
  return true;
}

cudaError_t launch_pool_topk(const CompressJob& job, bool* gathered) {
  const int64_t bh = (int64_t)job.batch * job.heads;
  if (gathered) *gathered = false;
  job.mark(2 * kStageTopk);
  cudaError_t err = cudaSuccess;
  if (job.k_sel <= 0) {
    // Nothing is selected: no launch.
  } else if (job.n_var > 0 && !(job.l_prefix <= kClusterMaxPrefix && job.pool_kernel <= 1025)) {
    err = cudaErrorInvalidValue;   // a ragged batch takes the cluster kernel only
  } else if (job.l_prefix <= kClusterMaxPrefix && job.pool_kernel <= 1025) {
    // CTAs per head. A head's select is latency-bound (a few radix passes, each ending in a barrier),
    // so a small batch spreads each head over up to 8 CTAs of a cluster; once the heads alone give
    // about two CTAs per SM, each head stays on one CTA (no cross-CTA exchange) and the GPU is filled
    // with heads instead (256 heads of 16K keys: 8 CTAs per head 126 us, 2: 70 us, 1: 65 us per
    // launch). The size is the largest power of two with at most about two CTAs per SM in total, at
    // least 2048 keys per CTA, and at most kClusterMaxSlice keys per CTA.
    const int64_t fill = (int64_t)2 * device_sm_count();
    int cl = 1;
    while (cl < kMaxCluster && (int64_t)(2 * cl) * bh <= fill) cl *= 2;
    const int by_keys = (int)((job.l_prefix + 2047) / 2048);
    if (cl > by_keys) cl = by_keys;
    const int need = (int)((job.l_prefix + kClusterMaxSlice - 1) / kClusterMaxSlice);
    if (cl < need) cl = need;
    if (cl > kMaxCluster) cl = kMaxCluster;
    if (cl < 1) cl = 1;
    GatherArgs g;
    g.k = static_cast<const uint4*>(job.k);
    g.v = static_cast<const uint4*>(job.v);
    g.k_out = static_cast<uint4*>(job.k_out);
    g.v_out = static_cast<uint4*>(job.v_out);
    g.len_out = job.len_out;
    g.kv_stride = job.kv_stride;
    g.cap = job.cap;
    g.vpr = job.head_dim * (job.dtype == SNAPKV_BF16 ? 2 : 4) / 16;
    g.l_obs = job.l_obs;
    g.heads = job.heads;
    g.c_stride = job.l_prefix;
    g.idx_stride = job.k_sel;
    g.dev_status = job.dev_status;
    g.var.n = 0;
    if (job.n_var > 0) {
      if (job.n_var > kMaxVarSeq) return cudaErrorInvalidValue;
      g.var.n = job.n_var;
      for (int b = 0; b < job.n_var; ++b) {
        g.var.l_prefix[b] = (int)(job.var_l_prompt[b] - job.l_obs);
        g.var.k[b] = (int)job.var_k[b];
        if (g.var.k[b] < 1) return cudaErrorInvalidValue;   // a ragged launch keeps at least one row
      }
    }
    const int radius = job.pool_kernel / 2;
    const int slice = (int)((job.l_prefix + cl - 1) / cl);
    const int work = (slice < kPoolChunk ? slice : kPoolChunk) + 2 * radius;
    const size_t smem =
        (size_t)(round4(slice) + round4(work > kHistWords ? work : kHistWords) + kSumWords + 32 + kMaxCluster + 1) *
        sizeof(uint32_t);
    err = cudaFuncSetAttribute(pool_topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(bh * cl));
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = job.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, pool_topk_cluster_kernel, (const float*)job.c, job.idx, job.l_prefix, radius,
                             job.k_sel, slice, g);
    if (gathered) *gathered = err == cudaSuccess;
  } else {
    pool_topk_kernel<<<(unsigned)bh, kThreads, 0, job.stream>>>(job.c, job.p, job.idx, job.l_prefix,
                                                                job.pool_kernel / 2, job.k_sel);
    err = cudaGetLastError();
  }
  job.mark(2 * kStageTopk + 1);
  return err;
}

}  // namespace snapkv
