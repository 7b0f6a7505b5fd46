// Score + softmax + vote with one thread-block cluster per head (bf16, d = 64 or 128, at most 128
// window-query rows per head, prompts of at most 8 CTAs x 4 TMEM slots of keys: 16K keys at 32
// rows). Under grouped-query attention a KV head's rows are its query heads' windows one after
// another (row i at window position i mod L_obs), and the vote sums every row.
//
// SnapKV explainer ("論文解説: SnapKV"), sections 投票メカニズム and アルゴリズム: logits
// s_ij = q_i . k_j / sqrt(d) of the L_obs window queries against every prompt key, the row
// softmax w_ij = exp(s_ij - m_i) / Z_i over the keys row i can see, and the vote C_j = sum_i w_ij
// over the prefix keys.
//
// One cluster of C CTAs per (sequence, head); CTA r owns the key chunks (items) 4r .. 4r + 3, each
// 128 / N tiles of 128 keys = one 128-column TMEM slot, so all of a CTA's logits stay in TMEM and
// every key is read from HBM once. Per CTA:
//   warp 0      TMA: the head's window queries once, then the CTA's key tiles through a ring of
//               shared-memory stages;
//   warp 1      MMA: one thread issues tcgen05.mma (M = 128 keys, N = padded L_obs, K = 16) of each
//               tile into its item's slot;
//   warps 2..9  epilogue, two warpgroups (items g and g + 2), one thread per key (TMEM lane):
//     statistics  per item and warp, the row maxima M_w (log2 domain) and sums z_w = sum 2^(s' - M_w);
//                 the CTA folds its (item, warp) pairs of each row into (M, Z) in shared memory;
//     exchange    after one cluster barrier, each row's (M, Z) of all C CTAs, read through
//                 distributed shared memory, give log2 Z_i of the whole head (the same fp32 value
//                 on every CTA: the fold runs in a fixed order);
//     vote        C_j = sum_i 2^(s'_ij - log2 Z_i) from the logits still in TMEM.
// A second cluster barrier keeps every CTA resident until its peers have read its (M, Z).
// Waits on mbarriers are bounded: a timeout reports SNAPKV_ERR_TIMEOUT, and the threads carry on
// along the same path (reading stale data is harmless), so every thread reaches both cluster
// barriers and the cluster exits.
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>

#include "sm100_ptx.cuh"
#include "snapkv_common.cuh"
#include "snapkv_internal.h"
#include "tc_common.cuh"

namespace snapkv {
namespace {

constexpr int kThreadsCl = 320;                  // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kTileKeys = 128;
constexpr int kItemsPerCta = 4;                  // TMEM slots of 128 columns
constexpr int kMaxCtas = 8;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimit = 4000000000LL;   // ~2 s of SM clock
constexpr long long kDrainLimit = 400000000LL;

struct ClArgs {
  int64_t l_prompt, l_prefix;
  int l_obs, rows, scope, n_items, keys_per_item, csize;   // rows: window-query rows per head
  float scale_log2;
  float* c_out;       // [BH][l_prefix]
  int32_t* dev_status;
};

template <int D, int N>
struct ClLayout {
  static constexpr int KB = D / 64;                 // 128-byte k-blocks per row
  static constexpr int TI = 128 / N;                // tiles per item
  static constexpr int A_BYTES = kTileKeys * 128;   // one k-block of a key tile
  static constexpr int STAGE_BYTES = KB * A_BYTES;
  static constexpr int QB_BYTES = N * 128;          // one k-block of the window queries
  static constexpr int Q_BYTES = KB * QB_BYTES;
  static constexpr int STAT_FLOATS = kItemsPerCta * 4 * N;   // per (item, warp, row)
  static constexpr int FIXED = Q_BYTES + 2 * STAT_FLOATS * 4 + 2 * N * 4 + N * 4 +
                               8 * (2 * 8 + 1 + kItemsPerCta * 8 + 1) + 64 + 1024;
  static constexpr int STAGES_FIT = (232448 - FIXED) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < 8 ? STAGES_FIT : 8;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_Q = OFF_K + STAGES * STAGE_BYTES;
  static constexpr int OFF_STAT = OFF_Q + Q_BYTES;                 // z then M, [item][warp][N]
  static constexpr int OFF_ROWSTAT = OFF_STAT + 2 * STAT_FLOATS * 4;   // [2][N]: this CTA's (M, Z)
  static constexpr int OFF_CV = OFF_ROWSTAT + 2 * N * 4;           // [N]: log2 Z_i of the head
  static constexpr int OFF_BAR = (OFF_CV + N * 4 + 7) & ~7;
  static constexpr int NBARS = 2 * STAGES + 1 + kItemsPerCta * TI + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  // + slack for 1024-byte alignment; at least 120 KB so that no two CTAs share an SM (each
  // allocates all 512 TMEM columns).
  static constexpr int BYTES_USED = OFF_MISC + 64 + 1024;
  static constexpr int BYTES = BYTES_USED > 120 * 1024 ? BYTES_USED : 120 * 1024;
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(128, N);
  static_assert(N % 16 == 0 && N >= 16 && N <= 128, "N");
  static_assert(kItemsPerCta * TI * N == (int)kTmemCols, "four slots fill TMEM");
  static_assert(QB_BYTES % 1024 == 0 && OFF_Q % 1024 == 0, "swizzle atoms");
  static_assert(STAGES >= 2 && BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ int item_tiles(const ClArgs& a, int item, int TI) {
  const int64_t left = a.l_prompt - (int64_t)item * a.keys_per_item;
  const int t = (int)((left + kTileKeys - 1) / kTileKeys);
  return t < TI ? t : TI;
}

// GQ: grouped-query rows, whose window position row mod L_obs comes from a table (a separate
// instantiation, so that the single-head case keeps its simpler epilogue).
template <int D, int N, bool GQ>
__global__ void __launch_bounds__(kThreadsCl, 1)
vote_cluster_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                    ClArgs a) {
  using Lay = ClLayout<D, N>;
  constexpr int TI = Lay::TI;
  constexpr int R = N < 32 ? N : 32;               // rows per register chunk
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + Lay::OFF_BAR);
  uint64_t* empty = full + Lay::STAGES;
  uint64_t* q_full = empty + Lay::STAGES;
  uint64_t* tile_full = q_full + 1;
  uint64_t* final_bar = tile_full + kItemsPerCta * TI;
  uint32_t* misc = reinterpret_cast<uint32_t*>(base + Lay::OFF_MISC);   // [0] tmem base, [1] abort
  volatile int* abort = reinterpret_cast<volatile int*>(misc + 1);
  float* st_z = reinterpret_cast<float*>(base + Lay::OFF_STAT);
  float* st_m = st_z + Lay::STAT_FLOATS;
  float* rowstat = reinterpret_cast<float*>(base + Lay::OFF_ROWSTAT);
  float* cvrow = reinterpret_cast<float*>(base + Lay::OFF_CV);
  __shared__ int no_abort;
  __shared__ int row_pos[GQ ? N : 1];   // window position of each query row (row mod L_obs)

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ptx::cluster_rank();
  const int64_t bh = blockIdx.x / a.csize;
  const int item0 = kItemsPerCta * (int)rank;
  const int n_my = min(kItemsPerCta, a.n_items - item0);   // >= 1 by the launch

  if (threadIdx.x == 0) {
    for (int i = 0; i < Lay::NBARS; ++i) ptx::mbar_init(full + i, 1);
    misc[1] = 0;
    no_abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&misc[0], kTmemCols);
    ptx::tmem_relinquish();
  }
  if (GQ)
    for (int i = threadIdx.x; i < N; i += kThreadsCl) row_pos[i] = i % a.l_obs;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = misc[0];
  auto fail = [&]() {
    report(a.dev_status, SNAPKV_ERR_TIMEOUT);
    *abort = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmap_k);
      ptx::prefetch_tensormap(&tmap_q);
      const uint64_t drop = ptx::make_policy_evict_first();   // keys are read once
      ptx::mbar_arrive_expect_tx(q_full, Lay::Q_BYTES);
#pragma unroll
      for (int kb = 0; kb < Lay::KB; ++kb)
        ptx::tma_load_3d(base + Lay::OFF_Q + kb * Lay::QB_BYTES, &tmap_q, kb * 64, 0, (int)bh, q_full);
      uint32_t g = 0;
      bool ok = true;
      for (int s = 0; s < n_my && ok; ++s) {
        const int item = item0 + s;
        const int tiles = item_tiles(a, item, TI);
        const int key0 = item * a.keys_per_item;
        for (int t = 0; t < tiles; ++t, ++g) {
          const int stage = g % Lay::STAGES;
          const uint32_t round = g / Lay::STAGES;
          if (!ptx::mbar_wait(&empty[stage], (round & 1) ^ 1, abort, kWaitLimit)) {
            fail();
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], Lay::STAGE_BYTES);
#pragma unroll
          for (int kb = 0; kb < Lay::KB; ++kb)
            ptx::tma_load_3d_hint(base + Lay::OFF_K + stage * Lay::STAGE_BYTES + kb * Lay::A_BYTES, &tmap_k,
                                  kb * 64, key0 + t * kTileKeys, (int)bh, &full[stage], drop);
        }
      }
      // Drain: every copy this thread started must land before the CTA may exit.
      for (uint32_t k = (g > (uint32_t)Lay::STAGES ? g - Lay::STAGES : 0u); k < g; ++k)
        ptx::mbar_wait(&full[k % Lay::STAGES], (k / Lay::STAGES) & 1, &no_abort, kDrainLimit);
      ptx::mbar_wait(q_full, 0, &no_abort, kDrainLimit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = ptx::mbar_wait(q_full, 0, abort, kWaitLimit);
      if (!ok) fail();
      ptx::tc_fence_after();
      const uint32_t q_addr = ptx::smem_u32(base + Lay::OFF_Q);
      uint32_t g = 0;
      for (int s = 0; s < n_my && ok; ++s) {
        const int tiles = item_tiles(a, item0 + s, TI);
        for (int t = 0; t < TI; ++t) {
          if (t < tiles && ok) {
            const int stage = g % Lay::STAGES;
            const uint32_t round = g / Lay::STAGES;
            if (!ptx::mbar_wait(&full[stage], round & 1, abort, kWaitLimit)) {
              fail();
              ok = false;
            } else {
              ptx::tc_fence_after();
              const uint32_t a_addr = ptx::smem_u32(base + Lay::OFF_K + stage * Lay::STAGE_BYTES);
              const uint32_t d_tmem = tmem_base + (uint32_t)(s * TI * N + t * N);
#pragma unroll
              for (int kb = 0; kb < Lay::KB; ++kb) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                  const uint64_t ad = ptx::smem_desc_k_sw128(a_addr + kb * Lay::A_BYTES + ks * 32);
                  const uint64_t bd = ptx::smem_desc_k_sw128(q_addr + kb * Lay::QB_BYTES + ks * 32);
                  ptx::mma_bf16(d_tmem, ad, bd, Lay::IDESC, (kb | ks) != 0);
                }
              }
              ptx::mma_commit(&empty[stage]);
              ++g;
            }
          }
          ptx::mma_commit(&tile_full[s * TI + t]);
        }
      }
      ptx::mma_commit(final_bar);
      ptx::mbar_wait(final_bar, 0, &no_abort, kDrainLimit);
    }
  }

  // ------------------------------------------------------------ epilogue (warps 2..9)
  const bool epi = warp >= 2;
  const int q4 = warp & 3;                         // TMEM lane quarter this warp may access
  const int gw = (warp - 2) & 3;                   // warp within its group
  const int grp = (warp - 2) >> 2;                 // group: items grp, grp + 2
  const int etid = threadIdx.x - 64;               // epilogue thread 0..255
  const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
  const int key_in_tile = q4 * 32 + lane;
  const int64_t lim = a.scope == SNAPKV_SCOPE_PROMPT_CAUSAL ? a.l_prefix : a.l_prefix - 1;
  auto load_rows = [&](uint32_t col, float* acc) {
    __syncwarp();
#pragma unroll
    for (int h = 0; h < R; h += 16) ptx::tmem_ld16(tmem_base + lane_addr + col + h, acc + h);
    ptx::tmem_wait_ld();
  };
  auto visible = [&](int row, int64_t key) {
    return row < a.rows && key < a.l_prompt &&
           (a.scope == SNAPKV_SCOPE_PROMPT_CAUSAL ? key <= lim + (GQ ? row_pos[row] : row) : key <= lim);
  };

  if (epi) {
    // Statistics of the group's items.
    for (int s = grp; s < kItemsPerCta; s += 2) {
      if (s >= n_my) break;
      const int item = item0 + s;
      const int tiles = item_tiles(a, item, TI);
      const int64_t item_key0 = (int64_t)item * a.keys_per_item;
      for (int t = 0; t < TI; ++t)
        if (!ptx::mbar_wait(&tile_full[s * TI + t], 0, abort, kWaitLimit)) fail();
      ptx::tc_fence_after();
#pragma unroll 1
      for (int r0 = 0; r0 < N; r0 += R) {
        float v[R];
#pragma unroll
        for (int i = 0; i < R; ++i) v[i] = -INFINITY;
        for (int t = 0; t < tiles; ++t) {
          float acc[R];
          load_rows((uint32_t)(s * TI * N + t * N + r0), acc);
          const int64_t tkey0 = item_key0 + t * kTileKeys;
          if (tkey0 + kTileKeys <= a.l_prefix) {
#pragma unroll
            for (int i = 0; i < R; ++i) v[i] = fmaxf(v[i], acc[i]);
          } else {
            const int64_t key = tkey0 + key_in_tile;
#pragma unroll
            for (int i = 0; i < R; ++i)
              if (visible(r0 + i, key)) v[i] = fmaxf(v[i], acc[i]);
          }
        }
        tc::butterfly_max<R, 16>(v, lane);
        const float mw = v[0] * a.scale_log2;   // this warp's log2-domain row maximum (or -inf)
        float mrow[R];
#pragma unroll
        for (int i = 0; i < R; ++i) mrow[i] = __shfl_sync(0xffffffffu, mw, R == 32 ? i : 2 * i);
#pragma unroll
        for (int i = 0; i < R; ++i) v[i] = 0.f;
        for (int t = 0; t < tiles; ++t) {
          float acc[R];
          load_rows((uint32_t)(s * TI * N + t * N + r0), acc);
          const int64_t tkey0 = item_key0 + t * kTileKeys;
          if (tkey0 + kTileKeys <= a.l_prefix) {
#pragma unroll
            for (int i = 0; i < R; ++i) v[i] += ex2(fmaf(acc[i], a.scale_log2, -mrow[i]));
          } else {
            const int64_t key = tkey0 + key_in_tile;
#pragma unroll
            for (int i = 0; i < R; ++i)
              if (visible(r0 + i, key)) v[i] += ex2(fmaf(acc[i], a.scale_log2, -mrow[i]));
          }
        }
        tc::butterfly_sum<R, 16>(v, lane);
        if (R == 32 || (lane & 1) == 0) {
          const int row = r0 + (R == 32 ? lane : lane >> 1);
          st_z[(s * 4 + gw) * N + row] = v[0];
          st_m[(s * 4 + gw) * N + row] = mw;
        }
      }
    }
    ptx::named_barrier(1, 256);
    // This CTA's (M, Z) of each row: its (item, warp) pairs folded in a fixed order.
    if (etid < N) {
      float M = -INFINITY;
      for (int p = 0; p < n_my * 4; ++p) M = fmaxf(M, st_m[p * N + etid]);
      float Z = 0.f;
      if (M > -INFINITY)
        for (int p = 0; p < n_my * 4; ++p) {
          const float m = st_m[p * N + etid];
          if (m > -INFINITY) Z = fmaf(st_z[p * N + etid], ex2(m - M), Z);
        }
      rowstat[etid] = M;
      rowstat[N + etid] = Z;
    }
  }
  __syncwarp();
  ptx::cluster_sync();   // every CTA's (M, Z) is complete

  if (epi) {
    // log2 Z_i of the head from all the cluster's (M, Z), folded in rank order.
    if (etid < N) {
      float mr[kMaxCtas];
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kMaxCtas; ++r) {
        mr[r] = r < a.csize ? __uint_as_float(ptx::dsmem_ld_u32(ptx::map_rank(&rowstat[etid], (uint32_t)r)))
                            : -INFINITY;
        M = fmaxf(M, mr[r]);
      }
      float Z = 0.f;
#pragma unroll
      for (int r = 0; r < kMaxCtas; ++r)
        if (r < a.csize && mr[r] > -INFINITY)
          Z = fmaf(__uint_as_float(ptx::dsmem_ld_u32(ptx::map_rank(&rowstat[N + etid], (uint32_t)r))),
                   ex2(mr[r] - M), Z);
      // rows past L_obs (zero logits) and rows with no visible key get zero weight
      cvrow[etid] = (etid < a.rows && Z > 0.f) ? M + log2f(Z) : INFINITY;
    }
  }
  __syncwarp();
  ptx::cluster_arrive();   // this CTA is done reading the peers' (M, Z)
  if (epi) {
    ptx::named_barrier(1, 256);
    constexpr int NC = N <= 32 ? N : 1;
    float cr[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) cr[i] = cvrow[i];
    for (int s = grp; s < kItemsPerCta; s += 2) {
      if (s >= n_my) break;
      const int item = item0 + s;
      const int tiles = item_tiles(a, item, TI);
      const int64_t item_key0 = (int64_t)item * a.keys_per_item;
      for (int t = 0; t < tiles; ++t) {
        const int64_t key = item_key0 + t * kTileKeys + key_in_tile;
        float csum = 0.f;
#pragma unroll
        for (int r0 = 0; r0 < N; r0 += R) {
          float acc[R];
          load_rows((uint32_t)(s * TI * N + t * N + r0), acc);
#pragma unroll
          for (int i = 0; i < R; ++i)
            csum += ex2(fmaf(acc[i], a.scale_log2, -(N <= 32 ? cr[(r0 + i) % NC] : cvrow[r0 + i])));
        }
        if (key < a.l_prefix) a.c_out[bh * a.l_prefix + key] = csum;
      }
    }
    ptx::tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
  __syncwarp();
  ptx::cluster_wait();   // no CTA leaves while its peers may still read its (M, Z)
}

template <int D, int N, bool GQ>
int cluster_smem_ready() {
  // The shared-memory attribute is set once per instantiation (0 unknown, 1 set, -1 failed).
  static std::atomic<int> state{0};
  int st = state.load(std::memory_order_acquire);
  if (st == 0) {
    st = cudaFuncSetAttribute(vote_cluster_kernel<D, N, GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              ClLayout<D, N>::BYTES) == cudaSuccess
             ? 1
             : -1;
    state.store(st, std::memory_order_release);
  }
  return st;
}

// Padded row count: 16, 32, 64 or 128 for one head's window, 64 or 128 for grouped windows.
int n_pad(int rows, int l_obs) {
  const int n = rows <= 16 ? 16 : (rows <= 32 ? 32 : (rows <= 64 ? 64 : 128));
  return (rows != l_obs && n < 64) ? 64 : n;
}

int cluster_ctas(const CompressJob& job) {
  const int kpi = (128 / n_pad(job.q_rows, job.l_obs)) * kTileKeys;
  const int64_t items = (job.l_prompt + kpi - 1) / kpi;
  return (int)((items + kItemsPerCta - 1) / kItemsPerCta);
}

template <int D, int N, bool GQ>
cudaError_t launch_cluster_typed(const CompressJob& job) {
  using Lay = ClLayout<D, N>;
  if (cluster_smem_ready<D, N, GQ>() < 0) return cudaErrorInvalidConfiguration;
  CUtensorMap mk, mq;
  const int64_t bh = (int64_t)job.batch * job.heads;
  if (!tc::make_map(&mk, job.k, D, job.l_prompt, bh, kTileKeys, job.kv_stride) ||
      !tc::make_map(&mq, job.q_obs, D, job.q_rows, bh, N))
    return cudaErrorInvalidValue;
  ClArgs a;
  a.l_prompt = job.l_prompt;
  a.l_prefix = job.l_prefix;
  a.l_obs = job.l_obs;
  a.rows = job.q_rows;
  a.scope = job.scope;
  a.keys_per_item = Lay::TI * kTileKeys;
  a.n_items = (int)((job.l_prompt + a.keys_per_item - 1) / a.keys_per_item);
  a.csize = (a.n_items + kItemsPerCta - 1) / kItemsPerCta;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)job.head_dim));
  a.c_out = job.c;
  a.dev_status = job.dev_status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(bh * a.csize));
  cfg.blockDim = dim3(kThreadsCl);
  cfg.dynamicSmemBytes = Lay::BYTES;
  cfg.stream = job.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  job.mark(2 * kStageScore);
  const cudaError_t err = cudaLaunchKernelEx(&cfg, vote_cluster_kernel<D, N, GQ>, mk, mq, a);
  job.mark(2 * kStageScore + 1);
  job.mark(2 * kStageVote);
  job.mark(2 * kStageVote + 1);
  return err;
}

}  // namespace

bool vote_cluster_eligible(const CompressJob& job) {
  if (job.dtype != SNAPKV_BF16 || job.q_rows > 128) return false;
  if (job.head_dim != 64 && job.head_dim != 128) return false;
  const int c = cluster_ctas(job);
  return c >= 1 && c <= kMaxCtas && (int64_t)job.batch * job.heads * c < ((int64_t)1 << 31);
}

cudaError_t launch_vote_cluster(const CompressJob& job) {
  const int n = n_pad(job.q_rows, job.l_obs);
  if (job.q_rows != job.l_obs) {
    if (job.head_dim == 64) return n == 64 ? launch_cluster_typed<64, 64, true>(job) : launch_cluster_typed<64, 128, true>(job);
    return n == 64 ? launch_cluster_typed<128, 64, true>(job) : launch_cluster_typed<128, 128, true>(job);
  }
  if (job.head_dim == 64) {
    if (n == 16) return launch_cluster_typed<64, 16, false>(job);
    if (n == 32) return launch_cluster_typed<64, 32, false>(job);
    if (n == 64) return launch_cluster_typed<64, 64, false>(job);
    return launch_cluster_typed<64, 128, false>(job);
  }
  if (n == 16) return launch_cluster_typed<128, 16, false>(job);
  if (n == 32) return launch_cluster_typed<128, 32, false>(job);
  if (n == 64) return launch_cluster_typed<128, 64, false>(job);
  return launch_cluster_typed<128, 128, false>(job);
}

}  // namespace snapkv
