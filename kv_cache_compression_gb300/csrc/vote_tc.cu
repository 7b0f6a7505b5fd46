// Score + softmax + vote on the 5th-generation tensor cores (bf16, d = 64 or 128, L_obs <= 128).
// Under grouped-query attention (G query heads per KV head) every query head is a head of its own
// here, reading its KV head's keys (key tiles of the G heads of a group are fetched in the same
// round of the queue, so the later ones hit in L2); its vote goes to a per-query-head buffer and a
// second kernel adds the G votes of each KV head in a fixed order.
//
// SnapKV explainer ("論文解説: SnapKV"), sections 投票メカニズム and アルゴリズム: logits
// s_ij = q_i . k_j / sqrt(d) of the L_obs window queries against every prompt key, the row
// softmax w_ij = exp(s_ij - m_i) / Z_i, and the vote C_j = sum_i w_ij over the prefix keys.
//
// Work is a queue of items, each TI = 128 / N tiles of 128 keys of one head, of two kinds:
//   A (statistics): per window row, the maximum M of the logits (log2 domain) over the item's
//     visible keys and z = sum 2^(s' - M); the item adds z * 2^M into the head's fp64 row sum
//     Z_i = sum_j 2^(s'_ij) (a fire-and-forget reduction) and then bumps the head's counter with a
//     release-ordered reduction. fp64's exponent range holds every row maximum within +-1000 in
//     log2 units; a larger one is reported as SNAPKV_ERR_UNSUPPORTED.
//   B (vote): once the head's counter shows all its A items, C_j = sum_i 2^(s'_ij - log2 Z_i) for
//     the item's prefix keys (the softmax max-subtraction cancels between numerator and Z_i).
// Resident mode (when a head has at most grid items, or, with two epilogue warpgroups or in a ragged
// batch, at most 4 x grid): the queue holds one item per key chunk; its logits stay in its TMEM slot
// after the statistics pass, and the warpgroup computes the vote from TMEM once the head is
// complete, so each key is read by the SM only once. With at most grid items per head a CTA holds
// at most one item of a head, and the vote follows its own statistics at once (every epilogue
// warpgroup holds one item, and the MMA fills the free slot ahead); otherwise it follows the
// statistics of the group's next item, so that a warpgroup never waits while holding an item
// without pass A: two warpgroups take the items, a CTA holds at most four items, two per
// warpgroup, and at most four items of one head, so the lowest unfinished head always completes.
// Longer heads take the re-read mode of items A and B above.
//
// A persistent, cooperative grid (one CTA per SM) takes queue positions round-robin. Per CTA:
//   warp 0      TMA: streams each item's key tiles (128 keys x 128 B per box, 128-byte swizzle)
//               into a ring of shared-memory stages and the head's window queries into one of two
//               buffers;
//   warp 1      MMA: one thread issues tcgen05.mma (M = 128 keys, N = padded L_obs, K = 16) for each
//               tile into the item's TMEM slot (four slots of 128 columns);
//   warps 2, 3  idle: with warps 0 and 1 they form warpgroup 0, which lowers its registers
//               (setmaxnreg) so that the epilogue warpgroups can raise theirs;
//   warps 4..   epilogue: G warpgroups (three for windows of up to 64 rows, else two), one thread
//               per key (TMEM lane); warpgroup g takes the CTA's items n = g, g + G, ..., reads
//               their logits with tcgen05.ld and gives the slot back as soon as it is done with it.
//
// Progress: A items never wait, and a B item waits only for A items that come earlier in the queue;
// every CTA takes its positions in queue order and the cooperative launch keeps all CTAs resident,
// so the lowest unfinished head always completes. All waits are bounded; on a timeout the kernel
// reports SNAPKV_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>
#include <cstdlib>

#include "sm100_ptx.cuh"
#include "snapkv_common.cuh"
#include "snapkv_internal.h"
#include "tc_common.cuh"

namespace snapkv {
namespace {

constexpr int kCtlWarps = 4;                       // warpgroup 0: TMA producer, MMA issuer, two idle
// Epilogue warpgroups and the register split (setmaxnreg) that goes with them. Windows of up to 64
// rows take three warpgroups: 16 warps give each thread 128 registers at launch, warpgroup 0 lowers
// itself to 56 and the epilogue raises itself to 136 (a 32-row chunk of logits and the vote's
// per-row factors of a 64-row window fit). Wider windows keep up to 128 per-row factors in
// registers and take two warpgroups: 12 warps, 168 registers at launch, 56 and 224. No split asks
// for more than the launch's registers (a larger request would wait for ever), and the host
// launches the kernel only if the compiler gave it that count. Fewer groups than TMEM slots is what
// the queue's progress argument needs (a group holds at most two slots, one with a vote pending).
template <int N>
struct EpiCfg {
  static constexpr int kGroups = N <= 64 ? 3 : 2;
  static constexpr int kThreads = (kCtlWarps + 4 * kGroups) * 32;
  static constexpr int kLaunchRegs = kGroups == 3 ? 128 : 168;
  static constexpr int kCtlRegs = 56;
  static constexpr int kEpiRegs = kGroups == 3 ? 136 : 224;
  static_assert(kCtlWarps * 32 * kCtlRegs + kGroups * 128 * kEpiRegs <= kThreads * kLaunchRegs, "register split");
  static_assert(kCtlRegs % 8 == 0 && kEpiRegs % 8 == 0 && kEpiRegs <= 256, "setmaxnreg counts");
};
constexpr int kMaxGroups = 3;
constexpr int kTeardownBarrier = 1 + kMaxGroups;   // named barrier of all warps before TMEM is freed
constexpr int kTileKeys = 128;
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitLimit = 4000000000LL;   // ~2 s of SM clock
constexpr long long kDrainLimit = 400000000LL;

// Per-sequence sizes of a ragged batch: the queue holds the sequences one after another, heads in
// order within a sequence, key chunks in order within a head.
struct VarSeqs {
  int n;                          // sequences (0: a uniform batch)
  int heads;                      // heads per sequence
  int item0[kMaxVarSeq + 1];      // first queue position of each sequence
  int n_chunk[kMaxVarSeq];
  int64_t l_prompt[kMaxVarSeq];
};

struct TcArgs {
  int64_t l_prompt, l_prefix;     // uniform batch (ragged: the maxima)
  int64_t c_stride;               // row stride of c_out (l_prefix, or its maximum for a ragged batch)
  int l_obs, scope, n_chunk, n_queue, keys_per_item, bh_total, delta;
  int group;         // query heads per KV head: head h reads the keys of KV head h / group
  int resident;      // 1: one item per key chunk, logits stay in TMEM from statistics to vote
  float scale_log2;
  long long wait_limit;   // SM cycles after which a bounded wait gives up (kWaitLimit unless testing)
  double* zsum;      // [BH][l_obs]: Z_i = sum_j 2^(s'_ij) over the head's visible keys (fp64)
  uint32_t* cnt;     // [BH] A items whose contribution to zsum is complete
  float* c_out;      // [BH][c_stride]
  int32_t* dev_status;
};

// Kernel parameters: a ragged batch carries its per-sequence sizes, a uniform one nothing more.
template <bool VAR>
struct TcParams : TcArgs {
  VarSeqs vs;
};
template <>
struct TcParams<false> : TcArgs {};

struct Item {
  int kind;   // 0: statistics (A), 1: vote (B)
  int head;
  int chunk;
  int l_prompt;        // the head's prompt length
};

// Queue position -> item. Blocks of n_chunk positions: A(0..delta-1), then B(h), A(h + delta)
// alternating, then the last B heads.
template <bool VAR>
__device__ __forceinline__ Item queue_item(const TcParams<VAR>& a, int p) {
  Item it;
  if constexpr (VAR) {   // ragged batch (resident mode only)
    int lo = 0, hi = a.vs.n - 1;   // the sequence s with item0[s] <= p < item0[s + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.vs.item0[mid] <= p)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int local = p - a.vs.item0[lo], nc = a.vs.n_chunk[lo];
    it.kind = 0;
    it.head = lo * a.vs.heads + local / nc;
    it.chunk = local % nc;
    it.l_prompt = (int)a.vs.l_prompt[lo];
    return it;
  }
  const int nc = a.n_chunk, H = a.bh_total, D = a.delta;
  const int blk = p / nc, off = p % nc;
  it.chunk = off;
  it.l_prompt = (int)a.l_prompt;
  if (a.resident) {   // every item is a statistics item whose vote follows from TMEM
    it.kind = 0;
    it.head = blk;
    return it;
  }
  if (blk < D) {
    it.kind = 0;
    it.head = blk;
  } else {
    const int r = blk - D;
    if (r < 2 * (H - D)) {
      it.kind = (r & 1) ? 0 : 1;
      it.head = (r & 1) ? D + (r >> 1) : (r >> 1);
    } else {
      it.kind = 1;
      it.head = (H - D) + (r - 2 * (H - D));
    }
  }
  return it;
}

constexpr int kSlots = 4;                          // TMEM item slots (128 columns each)

template <int D, int N>
struct TcLayout {
  static constexpr int KB = D / 64;                 // 128-byte k-blocks per row
  static constexpr int TI = 128 / N;                // tiles per item: one slot of 128 columns
  static constexpr int A_BYTES = kTileKeys * 128;   // one k-block of a key tile
  static constexpr int STAGE_BYTES = KB * A_BYTES;
  static constexpr int QB_BYTES = N * 128;          // one k-block of the window queries
  static constexpr int Q_BYTES = KB * QB_BYTES;
  // Everything but the key-tile ring, then at most 4 ring stages: 152 SMs x 4 x 32 KB of reads in
  // flight keep HBM busy, and a deeper ring only lengthens the memory queues that the epilogue's
  // reductions, counter updates and vote stores wait in. Measured per launch of the 256-head 16K-key
  // layer with three epilogue warpgroups: 3 stages 172.7 us, 4 stages 165.2 us, 5 stages 167.7 us
  // (with two warpgroups on the 32-head layer, 8 stages had measured 39.3 us against 34.6 us).
  static constexpr int G = EpiCfg<N>::kGroups;
  static constexpr int FIXED =
      2 * Q_BYTES + G * 4 * N * 4 + G * N * 4 + kSlots * N * 4 + 8 * (2 * 8 + 4 + 4 * 16 + 4 + 1) + 64 + 1024;
  static constexpr int STAGES_FIT = (232448 - FIXED) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < 4 ? STAGES_FIT : 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_Q = OFF_K + STAGES * STAGE_BYTES;
  static constexpr int OFF_RED = OFF_Q + 2 * Q_BYTES;        // [G groups][4 warps][N] floats
  static constexpr int OFF_ROW = OFF_RED + G * 4 * N * 4;    // [G groups][N] floats: per-row constants
  static constexpr int OFF_SMAX = OFF_ROW + G * N * 4;      // [kSlots][N] floats: an item's row maxima
  static constexpr int OFF_BAR = OFF_SMAX + kSlots * N * 4;
  static constexpr int NBAR = 2 * STAGES + 4 + kSlots * TI + kSlots + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // + slack for 1024-byte alignment; at least 120 KB so that no two CTAs share an SM (each one
  // allocates all 512 TMEM columns, and a second allocation on the same SM would block).
  static constexpr int BYTES_USED = OFF_MISC + 64 + 1024;
  static constexpr int BYTES = BYTES_USED > 120 * 1024 ? BYTES_USED : 120 * 1024;
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(128, N);
  static_assert(N % 16 == 0 && N >= 16 && N <= 128, "N");
  static_assert(kSlots * TI * N == (int)kTmemCols, "four slots fill TMEM");
  static_assert(QB_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(STAGES >= 2 && BYTES <= 232448, "shared memory");
};

struct Ctx {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* tile_full;
  uint64_t* tmem_empty;
  uint64_t* final_bar;
  uint32_t* misc;   // [0] tmem base, [1] abort
  volatile int* abort;
};

__device__ __forceinline__ void fail(const Ctx& c, int32_t* dev_status) {
  report(dev_status, SNAPKV_ERR_TIMEOUT);
  *c.abort = 1;
}

// Prompt length of an item's head: per item in a ragged batch, else the batch's.
template <bool VAR>
__device__ __forceinline__ int64_t prompt_of(const TcArgs& a, const Item& it) {
  if constexpr (VAR)
    return (int64_t)it.l_prompt;
  else
    return a.l_prompt;
}

template <bool VAR>
__device__ __forceinline__ int tiles_of(const TcArgs& a, const Item& it, int TI) {
  const int64_t key0 = (int64_t)it.chunk * a.keys_per_item;
  const int64_t left = prompt_of<VAR>(a, it) - key0;
  const int t = (int)((left + kTileKeys - 1) / kTileKeys);
  return t < TI ? t : TI;
}

template <int D, int N, bool VAR>
__global__ void __launch_bounds__(EpiCfg<N>::kThreads, 1)
vote_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
               TcParams<VAR> a) {
  using Lay = TcLayout<D, N>;
  using Epi = EpiCfg<N>;
  constexpr int TI = Lay::TI;
  constexpr int G = Epi::kGroups;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + Lay::OFF_BAR);
  Ctx c;
  c.full = bars;
  c.empty = bars + Lay::STAGES;
  c.q_full = bars + 2 * Lay::STAGES;
  c.q_empty = c.q_full + 2;
  c.tile_full = c.q_empty + 2;
  c.tmem_empty = c.tile_full + kSlots * TI;
  c.final_bar = c.tmem_empty + kSlots;
  c.misc = reinterpret_cast<uint32_t*>(base + Lay::OFF_MISC);
  c.abort = reinterpret_cast<volatile int*>(c.misc + 1);
  float* red = reinterpret_cast<float*>(base + Lay::OFF_RED);
  float* rowc = reinterpret_cast<float*>(base + Lay::OFF_ROW);
  float* slot_max = reinterpret_cast<float*>(base + Lay::OFF_SMAX);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < Lay::NBAR; ++i) ptx::mbar_init(bars + i, 1);
    for (int i = 1; i < 8; ++i) c.misc[i] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&c.misc[0], kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = c.misc[0];
  __shared__ int no_abort;
  if (threadIdx.x == 0) no_abort = 0;
  __syncthreads();
  // Every role ends here and returns: the roles' code paths never join again, so each compiles
  // within its own register share.
  auto teardown = [&]() {
    __syncwarp();   // the roles' single-lane loops have rejoined their warps
    ptx::named_barrier(kTeardownBarrier, Epi::kThreads);   // every warp is done with TMEM
    if (warp == 1) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
  };
  if (warp < kCtlWarps)   // warpgroup-uniform
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Epi::kCtlRegs));
  else
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Epi::kEpiRegs));

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tensormap(&tmap_k);
      ptx::prefetch_tensormap(&tmap_q);
      const uint64_t keep = ptx::make_policy_evict_last();
      const uint64_t drop = ptx::make_policy_evict_first();
      uint32_t g = 0;
      int n = 0;
      for (;; ++n) {
        const int p = blockIdx.x + n * gridDim.x;
        if (p >= a.n_queue || *c.abort) break;
        const Item it = queue_item<VAR>(a, p);
        const int qb = n & 1;
        if (!ptx::mbar_wait(&c.q_empty[qb], ((n >> 1) & 1) ^ 1, c.abort, a.wait_limit)) {
          fail(c, a.dev_status);
          break;
        }
        ptx::mbar_arrive_expect_tx(&c.q_full[qb], Lay::Q_BYTES);
#pragma unroll
        for (int kb = 0; kb < Lay::KB; ++kb)
          ptx::tma_load_3d(base + Lay::OFF_Q + qb * Lay::Q_BYTES + kb * Lay::QB_BYTES, &tmap_q, kb * 64, 0, it.head,
                           &c.q_full[qb]);
        const int tiles = tiles_of<VAR>(a, it, TI);
        const int key0 = it.chunk * a.keys_per_item;
        // Keys are read once, except in re-read mode where a head's vote items read its keys again
        // from L2: only those statistics loads ask L2 to keep the lines. Marking the whole stream
        // evict-last fills L2 with lines that are never read again and slows the stream (16K-key
        // layer, event-timed: 41 us per launch with every load evict-last, 38.9 us with evict-first).
        const uint64_t policy = (it.kind == 0 && !a.resident) ? keep : drop;
        bool ok = true;
        for (int t = 0; t < tiles; ++t, ++g) {
          const int stage = g % Lay::STAGES;
          const uint32_t round = g / Lay::STAGES;
          if (!ptx::mbar_wait(&c.empty[stage], (round & 1) ^ 1, c.abort, a.wait_limit)) {
            fail(c, a.dev_status);
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&c.full[stage], Lay::STAGE_BYTES);
#pragma unroll
          for (int kb = 0; kb < Lay::KB; ++kb)
            ptx::tma_load_3d_hint(base + Lay::OFF_K + stage * Lay::STAGE_BYTES + kb * Lay::A_BYTES, &tmap_k,
                                  kb * 64, key0 + t * kTileKeys, it.head / a.group, &c.full[stage], policy);
        }
        if (!ok) {
          ++n;
          break;
        }
      }
      // Drain: every copy this thread started must land before the CTA may exit.
      const uint32_t issued = g;
      for (uint32_t k = (issued > (uint32_t)Lay::STAGES ? issued - Lay::STAGES : 0u); k < issued; ++k)
        ptx::mbar_wait(&c.full[k % Lay::STAGES], (k / Lay::STAGES) & 1, &no_abort, kDrainLimit);
      for (int k = (n > 2 ? n - 2 : 0); k < n; ++k)
        ptx::mbar_wait(&c.q_full[k & 1], (k >> 1) & 1, &no_abort, kDrainLimit);
    }
    teardown();
    return;
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t g = 0;
      for (int n = 0;; ++n) {
        const int p = blockIdx.x + n * gridDim.x;
        if (p >= a.n_queue || *c.abort) break;
        const Item it = queue_item<VAR>(a, p);
        const int slot = n % kSlots, use = n / kSlots, qb = n & 1;
        if (!ptx::mbar_wait(&c.tmem_empty[slot], (use & 1) ^ 1, c.abort, a.wait_limit) ||
            !ptx::mbar_wait(&c.q_full[qb], (n >> 1) & 1, c.abort, a.wait_limit)) {
          fail(c, a.dev_status);
          break;
        }
        ptx::tc_fence_after();
        const int tiles = tiles_of<VAR>(a, it, TI);
        const uint32_t q_addr = ptx::smem_u32(base + Lay::OFF_Q + qb * Lay::Q_BYTES);
        bool ok = true;
        for (int t = 0; t < TI; ++t) {
          if (t < tiles) {
            const int stage = g % Lay::STAGES;
            const uint32_t round = g / Lay::STAGES;
            if (!ptx::mbar_wait(&c.full[stage], round & 1, c.abort, a.wait_limit)) {
              fail(c, a.dev_status);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t a_addr = ptx::smem_u32(base + Lay::OFF_K + stage * Lay::STAGE_BYTES);
            const uint32_t d_tmem = tmem_base + (uint32_t)(slot * TI * N + t * N);
#pragma unroll
            for (int kb = 0; kb < Lay::KB; ++kb) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ad = ptx::smem_desc_k_sw128(a_addr + kb * Lay::A_BYTES + ks * 32);
                const uint64_t bd = ptx::smem_desc_k_sw128(q_addr + kb * Lay::QB_BYTES + ks * 32);
                ptx::mma_bf16(d_tmem, ad, bd, Lay::IDESC, (kb | ks) != 0);
              }
            }
            ptx::mma_commit(&c.empty[stage]);
            ++g;
          }
          ptx::mma_commit(&c.tile_full[slot * TI + t]);
        }
        if (!ok) break;
        ptx::mma_commit(&c.q_empty[qb]);
      }
      ptx::mma_commit(c.final_bar);
      ptx::mbar_wait(c.final_bar, 0, &no_abort, kDrainLimit);
    }
    teardown();
    return;
  } else if (warp < kCtlWarps) {
    teardown();   // warps 2 and 3 only lend their registers
    return;
  } else {
    // ------------------------------------------------------------ epilogue (warps 4 .. 4 + 4G - 1)
    const int q4 = warp & 3;                         // TMEM lane quarter this warp may access
    const int gw = (warp - kCtlWarps) & 3;           // warp within its group
    const int grp = (warp - kCtlWarps) >> 2;         // group: items n = grp, grp + ng, ...
    const int gtid = (threadIdx.x - kCtlWarps * 32) & 127;   // thread within its group
    const int bar_id = 1 + grp;
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const int key_in_tile = q4 * 32 + lane;
    constexpr int R = N < 32 ? N : 32;               // rows per register chunk
    float* gred = red + grp * 4 * N;
    float* growc = rowc + grp * N;
    __shared__ int sh_stop[kMaxGroups];

    // Abort decision shared by the group's 128 threads (named barriers have no timeout, so every
    // thread of a group must take the same path between them).
    auto stop_uniform = [&]() -> bool {
      if (gtid == 0) sh_stop[grp] = *c.abort;
      ptx::named_barrier(bar_id, 128);
      const bool r = sh_stop[grp] != 0;
      ptx::named_barrier(bar_id, 128);
      return r;
    };
    auto load_rows = [&](uint32_t col, float* acc) {
      __syncwarp();
#pragma unroll
      for (int h = 0; h < R; h += 16) ptx::tmem_ld16(tmem_base + lane_addr + col + h, acc + h);
      ptx::tmem_wait_ld();
    };
    auto store_rows = [&](uint32_t col, const float* val) {
      __syncwarp();
#pragma unroll
      for (int h = 0; h < R; h += 16) ptx::tmem_st16(tmem_base + lane_addr + col + h, val + h);
    };
    // Per-warp row results after a butterfly: lane l holds row l (R == 32) or l/2 (R == 16).
    auto stash_rows = [&](float* v, int r0) {
      if constexpr (R == 32) {
        gred[gw * N + r0 + lane] = v[0];
      } else {
        if ((lane & 1) == 0) gred[gw * N + r0 + (lane >> 1)] = v[0];
      }
    };
    // Waits (bounded) for the item's tiles in its TMEM slot. A timed-out wait only raises the abort
    // flag: the thread carries on (reading stale TMEM is harmless) so that it meets its peers at
    // every barrier.
    auto wait_tiles = [&](int slot, int use) {
      for (int t = 0; t < TI; ++t)
        if (!ptx::mbar_wait(&c.tile_full[slot * TI + t], use & 1, c.abort, a.wait_limit)) fail(c, a.dev_status);
      ptx::tc_fence_after();
    };

    // A item: per 32-row chunk, the row maxima, then the row sums of 2^(s - max). In re-read mode
    // the slot is released after the last TMEM read.
    auto item_stats = [&](int n, const Item& it) {
      const int slot = n % kSlots;
      const int tiles = tiles_of<VAR>(a, it, TI);
      const int item_key0 = it.chunk * a.keys_per_item;
      const int l_prompt = (int)prompt_of<VAR>(a, it);
      const int l_prefix = VAR ? l_prompt - a.l_obs : (int)a.l_prefix;
      const int lim = a.scope == SNAPKV_SCOPE_PROMPT_CAUSAL ? l_prefix : l_prefix - 1;
      wait_tiles(slot, n / kSlots);
#pragma unroll 1
      for (int r0 = 0; r0 < N; r0 += R) {
        float v[R];
#pragma unroll
        for (int i = 0; i < R; ++i) v[i] = -INFINITY;
        for (int t = 0; t < tiles; ++t) {
          float acc[R];
          load_rows((uint32_t)(slot * TI * N + t * N + r0), acc);
          const int tkey0 = item_key0 + t * kTileKeys;
          if (tkey0 + kTileKeys <= l_prefix) {
#pragma unroll
            for (int i = 0; i < R; ++i) v[i] = fmaxf(v[i], acc[i]);
          } else {
            const int key = tkey0 + key_in_tile;
#pragma unroll
            for (int i = 0; i < R; ++i) {
              const int row = r0 + i;
              const bool vis = row < a.l_obs && key < l_prompt &&
                               (a.scope == SNAPKV_SCOPE_PROMPT_CAUSAL ? key <= lim + row : key <= lim);
              if (vis) v[i] = fmaxf(v[i], acc[i]);
            }
          }
        }
        tc::butterfly_max<R, 16>(v, lane);
        stash_rows(v, r0);
        ptx::named_barrier(bar_id, 128);
        if (gtid < R) {
          float mx = gred[r0 + gtid];
#pragma unroll
          for (int w = 1; w < 4; ++w) mx = fmaxf(mx, gred[w * N + r0 + gtid]);
          growc[r0 + gtid] = mx * a.scale_log2;       // log2-domain row maximum (or -inf)
          slot_max[slot * N + r0 + gtid] = mx * a.scale_log2;   // kept for the item's vote
        }
        ptx::named_barrier(bar_id, 128);
        // The row maxima are read from shared memory (a broadcast) rather than held in R registers,
        // which keeps the pass free of spills (ragged batch 0.530 -> 0.520 ms, long context -2 %).
        const float* mrow = growc + r0;
#pragma unroll
        for (int i = 0; i < R; ++i) v[i] = 0.f;
        for (int t = 0; t < tiles; ++t) {
          float acc[R];
          const uint32_t col = (uint32_t)(slot * TI * N + t * N + r0);
          load_rows(col, acc);
          const int tkey0 = item_key0 + t * kTileKeys;
          if (tkey0 + kTileKeys <= l_prefix) {
#pragma unroll
            for (int i = 0; i < R; ++i) {
              acc[i] = ex2(fmaf(acc[i], a.scale_log2, -mrow[i]));
              v[i] += acc[i];
            }
          } else {
            const int key = tkey0 + key_in_tile;
#pragma unroll
            for (int i = 0; i < R; ++i) {
              const int row = r0 + i;
              const bool vis = row < a.l_obs && key < l_prompt &&
                               (a.scope == SNAPKV_SCOPE_PROMPT_CAUSAL ? key <= lim + row : key <= lim);
              acc[i] = vis ? ex2(fmaf(acc[i], a.scale_log2, -mrow[i])) : 0.f;
              v[i] += acc[i];
            }
          }
          // A resident item's vote reads these exponentials back: 2^(s' - M_item) in place of s'.
          if (a.resident) store_rows(col, acc);
        }
        if (a.resident) ptx::tmem_wait_st();
        const bool last_read = !a.resident && r0 + R >= N;   // resident items keep the slot
        if (last_read) ptx::tc_fence_before();
        tc::butterfly_sum<R, 16>(v, lane);
        stash_rows(v, r0);
        ptx::named_barrier(bar_id, 128);
        if (last_read && gtid == 0) ptx::mbar_arrive(&c.tmem_empty[slot]);
        if (gtid < R && r0 + gtid < a.l_obs) {
          float zz = gred[r0 + gtid];
#pragma unroll
          for (int w = 1; w < 4; ++w) zz += gred[w * N + r0 + gtid];
          const float mx = growc[r0 + gtid];
          if (zz > 0.f) {   // the row saw at least one visible key in this item
            const float fl = floorf(mx);
            if (fabsf(fl) > 1000.f) report(a.dev_status, SNAPKV_ERR_UNSUPPORTED);
            // z * 2^M = (z * 2^(M - floor M)) * 2^floor M with z * 2^(M - floor M) in [1, 2^11):
            // the fp64 bits are assembled from the fp32 bits (no fp64 arithmetic).
            const uint32_t fb = __float_as_uint(zz * ex2(mx - fl));
            const long long e = (long long)fminf(fmaxf(fl, -1000.f), 1000.f) + (long long)((fb >> 23) & 0xFF) - 127;
            const long long db = ((e + 1023) << 52) | ((long long)(fb & 0x7FFFFF) << 29);
            if (in_bounds(it.head < a.bh_total && r0 + gtid < a.l_obs, a.dev_status))
              ptx::red_add_f64(a.zsum + (int64_t)it.head * a.l_obs + r0 + gtid, __longlong_as_double(db));
          }
        }
        ptx::named_barrier(bar_id, 128);
      }
      // The group's reductions are ordered before the counter update by the barrier above; the
      // release-ordered increment makes them visible to whoever acquires the counter.
      if (gtid == 0) ptx::red_add_release_u32(a.cnt + it.head, 1u);
    };

    // A item for windows of 64 or more rows: two 32-row chunks share each exchange, so the item
    // takes half the group barriers (the row maxima of pass 2 are read from shared memory).
    auto item_stats_pairs = [&](int n, const Item& it) {
      const int slot = n % kSlots;
      const int tiles = tiles_of<VAR>(a, it, TI);
      const int item_key0 = it.chunk * a.keys_per_item;
      const int l_prompt = (int)prompt_of<VAR>(a, it);
      const int l_prefix = VAR ? l_prompt - a.l_obs : (int)a.l_prefix;
      const int lim = a.scope == SNAPKV_SCOPE_PROMPT_CAUSAL ? l_prefix : l_prefix - 1;
      // Folds the visible logits of rows rb .. rb + R - 1 of tile t into v (max, or sum of 2^(s'-M));
      // the sum also writes each 2^(s'-M) (0 where not visible) back over its logit for the vote of
      // a resident item.
      auto fold = [&](int t, int rb, float* v, bool sum) {
        float acc[R];
        const uint32_t col = (uint32_t)(slot * TI * N + t * N + rb);
        load_rows(col, acc);
        const int tkey0 = item_key0 + t * kTileKeys;
        if (tkey0 + kTileKeys <= l_prefix) {
#pragma unroll
          for (int i = 0; i < R; ++i) {
            if (sum) {
              acc[i] = ex2(fmaf(acc[i], a.scale_log2, -growc[rb + i]));
              v[i] += acc[i];
            } else {
              v[i] = fmaxf(v[i], acc[i]);
            }
          }
        } else {
          const int key = tkey0 + key_in_tile;
#pragma unroll
          for (int i = 0; i < R; ++i) {
            const int row = rb + i;
            const bool vis = row < a.l_obs && key < l_prompt &&
                             (a.scope == SNAPKV_SCOPE_PROMPT_CAUSAL ? key <= lim + row : key <= lim);
            if (sum) {
              acc[i] = vis ? ex2(fmaf(acc[i], a.scale_log2, -growc[rb + i])) : 0.f;
              v[i] += acc[i];
            } else if (vis) {
              v[i] = fmaxf(v[i], acc[i]);
            }
          }
        }
        if (sum && a.resident) store_rows(col, acc);
      };
      wait_tiles(slot, n / kSlots);
#pragma unroll 1
      for (int r0 = 0; r0 < N; r0 += 2 * R) {
        {
          float va[R], vb[R];
#pragma unroll
          for (int i = 0; i < R; ++i) va[i] = vb[i] = -INFINITY;
          for (int t = 0; t < tiles; ++t) {
            fold(t, r0, va, false);
            fold(t, r0 + R, vb, false);
          }
          tc::butterfly_max<R, 16>(va, lane);
          stash_rows(va, r0);
          tc::butterfly_max<R, 16>(vb, lane);
          stash_rows(vb, r0 + R);
        }
        ptx::named_barrier(bar_id, 128);
        if (gtid < 2 * R) {
          float mx = gred[r0 + gtid];
#pragma unroll
          for (int w = 1; w < 4; ++w) mx = fmaxf(mx, gred[w * N + r0 + gtid]);
          growc[r0 + gtid] = mx * a.scale_log2;       // log2-domain row maximum (or -inf)
          slot_max[slot * N + r0 + gtid] = mx * a.scale_log2;   // kept for the item's vote
        }
        ptx::named_barrier(bar_id, 128);
        const bool last_read = !a.resident && r0 + 2 * R >= N;   // resident items keep the slot
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const int rb = r0 + h * R;
          float v[R];
#pragma unroll
          for (int i = 0; i < R; ++i) v[i] = 0.f;
          for (int t = 0; t < tiles; ++t) fold(t, rb, v, true);
          if (a.resident) ptx::tmem_wait_st();
          if (last_read && h == 1) ptx::tc_fence_before();
          tc::butterfly_sum<R, 16>(v, lane);
          stash_rows(v, rb);
        }
        ptx::named_barrier(bar_id, 128);
        if (last_read && gtid == 0) ptx::mbar_arrive(&c.tmem_empty[slot]);
        if (gtid < 2 * R && r0 + gtid < a.l_obs) {
          float zz = gred[r0 + gtid];
#pragma unroll
          for (int w = 1; w < 4; ++w) zz += gred[w * N + r0 + gtid];
          const float mx = growc[r0 + gtid];
          if (zz > 0.f) {   // the row saw at least one visible key in this item
            const float fl = floorf(mx);
            if (fabsf(fl) > 1000.f) report(a.dev_status, SNAPKV_ERR_UNSUPPORTED);
            const uint32_t fb = __float_as_uint(zz * ex2(mx - fl));
            const long long e = (long long)fminf(fmaxf(fl, -1000.f), 1000.f) + (long long)((fb >> 23) & 0xFF) - 127;
            const long long db = ((e + 1023) << 52) | ((long long)(fb & 0x7FFFFF) << 29);
            if (in_bounds(it.head < a.bh_total && r0 + gtid < a.l_obs, a.dev_status))
              ptx::red_add_f64(a.zsum + (int64_t)it.head * a.l_obs + r0 + gtid, __longlong_as_double(db));
          }
        }
        ptx::named_barrier(bar_id, 128);
      }
      if (gtid == 0) ptx::red_add_release_u32(a.cnt + it.head, 1u);
    };

    // B item (after its head's statistics are published): the vote of each prefix key,
    // C_j = sum_i 2^(s'_ij - c_i); the slot is released after the last TMEM read.
    auto item_vote = [&](int n, const Item& it) {
      const int slot = n % kSlots;
      const int tiles = tiles_of<VAR>(a, it, TI);
      const int item_key0 = it.chunk * a.keys_per_item;
      if (gtid == 0) {
        const uint32_t need =
            VAR ? (uint32_t)((it.l_prompt + a.keys_per_item - 1) / a.keys_per_item) : (uint32_t)a.n_chunk;
        if (ptx::ld_acquire_u32(a.cnt + it.head) < need) {
          const long long t0 = clock64();
          while (ptx::ld_acquire_u32(a.cnt + it.head) < need) {
            if (*c.abort || clock64() - t0 > a.wait_limit) {
              fail(c, a.dev_status);
              break;
            }
            __nanosleep(32);
          }
        }
      }
      ptx::named_barrier(bar_id, 128);
      if (gtid < N) {
        float cv = INFINITY;   // rows past L_obs: zero logits, zero weight
        if (gtid < a.l_obs) {
          // log2 Z_i = exponent + log2(mantissa in [1, 2)), read off the fp64 bits
          const long long zb = __double_as_longlong(__ldcg(a.zsum + (int64_t)it.head * a.l_obs + gtid));
          const int e = (int)((zb >> 52) & 0x7FF) - 1023;
          const float mant = __uint_as_float(0x3F800000u | (uint32_t)((zb >> 29) & 0x7FFFFF));
          cv = (zb & 0x7FF0000000000000LL) ? (float)e + log2f(mant) : -INFINITY;
        }
        // A resident item's slot holds 2^(s' - M_i) (M_i its row maximum): the weight is that times
        // f_i = 2^(M_i - log2 Z_i) <= 1, and 0 for rows past L_obs. Otherwise the slot holds the
        // logits and the row constant is log2 Z_i itself.
        growc[gtid] = a.resident ? (gtid < a.l_obs ? ex2(slot_max[slot * N + gtid] - cv) : 0.f) : cv;
      }
      wait_tiles(slot, n / kSlots);
      ptx::named_barrier(bar_id, 128);
      float cr[N];
#pragma unroll
      for (int i = 0; i < N; ++i) cr[i] = growc[i];
      const int vote_end = VAR ? (int)prompt_of<VAR>(a, it) - a.l_obs : (int)a.l_prefix;   // prefix keys only
      if (a.resident) {
        for (int t = 0; t < tiles; ++t) {
          const int key = item_key0 + t * kTileKeys + key_in_tile;
          float csum = 0.f;
#pragma unroll
          for (int r0 = 0; r0 < N; r0 += R) {
            float acc[R];
            load_rows((uint32_t)(slot * TI * N + t * N + r0), acc);
#pragma unroll
            for (int i = 0; i < R; ++i) csum = fmaf(acc[i], cr[r0 + i], csum);
          }
          if (key < vote_end && in_bounds(it.head < a.bh_total && key < a.c_stride, a.dev_status))
            a.c_out[(int64_t)it.head * a.c_stride + key] = csum;
        }
      } else {
        for (int t = 0; t < tiles; ++t) {
          const int key = item_key0 + t * kTileKeys + key_in_tile;
          float csum = 0.f;
#pragma unroll
          for (int r0 = 0; r0 < N; r0 += R) {
            float acc[R];
            load_rows((uint32_t)(slot * TI * N + t * N + r0), acc);
#pragma unroll
            for (int i = 0; i < R; ++i) csum += ex2(fmaf(acc[i], a.scale_log2, -cr[r0 + i]));
          }
          if (key < vote_end && in_bounds(it.head < a.bh_total && key < a.c_stride, a.dev_status))
            a.c_out[(int64_t)it.head * a.c_stride + key] = csum;
        }
      }
      ptx::tc_fence_before();
      ptx::named_barrier(bar_id, 128);
      if (gtid == 0) ptx::mbar_arrive(&c.tmem_empty[slot]);
    };

    // With at most grid items per head, the positions of a head's items are less than a grid apart,
    // so no CTA holds two of them. Otherwise each group holds two items at a time (one waiting for
    // its vote), and only two groups fit the four TMEM slots: the third one sits out.
    const bool lag0 = a.n_chunk <= (int)gridDim.x;
    const int ng = (a.resident && !lag0) ? 2 : G;   // groups taking items
    if (grp >= ng) {
      teardown();
      return;
    }
    int k = 0;
    for (;; ++k) {
      const int n = grp + ng * k;
      const int p = blockIdx.x + n * gridDim.x;
      if (p >= a.n_queue || stop_uniform()) break;
      const Item it = queue_item<VAR>(a, p);
      if (it.kind == 0) {
        if constexpr (N >= 2 * R)
          item_stats_pairs(n, it);
        else
          item_stats(n, it);
      } else {
        item_vote(n, it);
      }
      if (a.resident && lag0) {
        // A head has at most one item on this CTA: its vote may wait for the head right away.
        item_vote(n, it);
      } else if (a.resident && k > 0) {
        // Otherwise the vote of the group's previous item, whose logits are still in TMEM, comes
        // after the statistics of this one (so no item of the CTA waits without its pass A).
        const int m = n - ng;
        item_vote(m, queue_item<VAR>(a, blockIdx.x + m * gridDim.x));
      }
    }
    if (a.resident && !lag0 && k > 0 && !stop_uniform()) {
      const int m = grp + ng * (k - 1);
      item_vote(m, queue_item<VAR>(a, blockIdx.x + m * gridDim.x));
    }
    teardown();
    return;
  }
}

// Vote of each KV head = the sum of its G query heads' votes, added in query-head order.
__global__ void __launch_bounds__(256)
group_sum_kernel(const float* __restrict__ c_q, float* __restrict__ c, int64_t l_prefix, int64_t bh_kv, int group) {
  const int64_t total = bh_kv * l_prefix;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t h = u / l_prefix, j = u - h * l_prefix;
    const float* src = c_q + h * group * l_prefix + j;
    float sum = 0.f;
    for (int g = 0; g < group; ++g) sum += __ldcg(src + g * l_prefix);
    c[u] = sum;
  }
}

template <int D, int N>
cudaError_t launch_tc_typed(const CompressJob& job, int grid) {
  using Lay = TcLayout<D, N>;
  if (grid <= 0) return cudaErrorInvalidConfiguration;   // tc_grid() also set the smem attribute
  cudaError_t err;
  CUtensorMap mk, mq;
  const int group = job.q_rows / job.l_obs;                 // query heads per KV head
  const int64_t bh_kv = (int64_t)job.batch * job.heads;
  const int64_t bh = bh_kv * group;                           // query heads: the kernel's heads
  if (!tc::make_map(&mk, job.k, D, job.l_prompt, bh_kv, kTileKeys, job.kv_stride) ||
      !tc::make_map(&mq, job.q_obs, D, job.l_obs, bh, N))
    return cudaErrorInvalidValue;
  TcArgs a;
  a.l_prompt = job.l_prompt;
  a.l_prefix = job.l_prefix;
  a.c_stride = job.l_prefix;
  a.l_obs = job.l_obs;
  a.group = group;
  a.scope = job.scope;
  a.keys_per_item = Lay::TI * kTileKeys;
  a.n_chunk = (int)((job.l_prompt + a.keys_per_item - 1) / a.keys_per_item);
  a.bh_total = (int)bh;
  // Resident mode while a head has at most grid items (the vote follows its own statistics at once)
  // or, with two epilogue groups, at most four per CTA (the vote comes one item late and each group
  // holds two TMEM slots). With three groups the late vote would leave one of them idle, and
  // re-reading the keys from L2 with all three is faster: 384 against 475 us for 32 heads of 131072
  // keys and a 64-row window.
  const bool late_fits = a.n_chunk <= kSlots * grid;
  a.resident = (EpiCfg<N>::kGroups == 3 ? a.n_chunk <= grid : late_fits) ? 1 : 0;
  a.n_queue = (int)((a.resident ? 1 : 2) * bh * a.n_chunk);
  TcParams<true> pv;
  if (job.n_var > 0) {
    // Ragged batch: n_chunk holds the largest head's items (the queue's deadlock-freedom
    // conditions bound the items of a head), and the queue is resident only.
    if (job.n_var > kMaxVarSeq || group != 1 || !late_fits) return cudaErrorInvalidValue;
    a.resident = 1;
    pv.vs.n = job.n_var;
    pv.vs.heads = job.heads;
    int pos = 0;
    for (int b = 0; b < job.n_var; ++b) {
      pv.vs.item0[b] = pos;
      pv.vs.l_prompt[b] = job.var_l_prompt[b];
      pv.vs.n_chunk[b] = (int)((job.var_l_prompt[b] + a.keys_per_item - 1) / a.keys_per_item);
      pos += job.heads * pv.vs.n_chunk[b];
    }
    pv.vs.item0[job.n_var] = pos;
    a.n_queue = pos;
  }
  // B items of a head come about four grids of queue positions after its last A item (so they
  // seldom wait), unless the keys read in between would no longer fit comfortably in L2.
  const int64_t want = 1 + (4 * (int64_t)grid + 2 * (int64_t)a.n_chunk - 1) / (2 * (int64_t)a.n_chunk);
  const int64_t head_bytes = job.l_prompt * job.head_dim * 2;
  const int64_t l2_fit = (int64_t)(64 << 20) / (head_bytes > 0 ? head_bytes : 1);
  int64_t delta = want < l2_fit ? want : l2_fit;
  if (delta < 1) delta = 1;
  a.delta = (int)(delta < bh ? delta : bh);
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)job.head_dim));
  // Testing knob: SNAPKV_WAIT_LIMIT_CYCLES (a positive count of SM cycles) shortens every bounded
  // wait of this kernel, so that a test can make one run out and check the timeout report; unset, the
  // waits give up after ~2 s only.
  a.wait_limit = kWaitLimit;
  if (const char* env = getenv("SNAPKV_WAIT_LIMIT_CYCLES")) {
    const long long v = strtoll(env, nullptr, 10);
    if (v > 0) a.wait_limit = v;
  }
  a.zsum = job.tc_zsum;
  a.cnt = job.tc_cnt;
  a.c_out = group > 1 ? job.c_q : job.c;
  a.dev_status = job.dev_status;
  if (grid > a.n_queue) grid = a.n_queue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(EpiCfg<N>::kThreads);
  cfg.dynamicSmemBytes = Lay::BYTES;
  cfg.stream = job.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // The row sums and per-head counters start at zero on every call (the workspace is scratch).
  // The stage's start marker follows the memset, so that the stage times the kernel alone.
  err = cudaMemsetAsync(job.tc_zsum, 0, job.tc_zero_bytes, job.stream);
  if (err != cudaSuccess) return err;
  job.mark(2 * kStageScore);
  if (job.n_var > 0) {
    static_cast<TcArgs&>(pv) = a;
    err = cudaLaunchKernelEx(&cfg, vote_tc_kernel<D, N, true>, mk, mq, pv);
  } else {
    TcParams<false> pu;
    static_cast<TcArgs&>(pu) = a;
    err = cudaLaunchKernelEx(&cfg, vote_tc_kernel<D, N, false>, mk, mq, pu);
  }
  job.mark(2 * kStageScore + 1);
  job.mark(2 * kStageVote);
  if (err == cudaSuccess && group > 1) {
    const int64_t total = bh_kv * job.l_prefix;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    group_sum_kernel<<<(unsigned)blocks, 256, 0, job.stream>>>(job.c_q, job.c, job.l_prefix, bh_kv, group);
    err = cudaGetLastError();
  }
  job.mark(2 * kStageVote + 1);
  return err;
}

// Grid of the persistent kernel on the current device: one CTA per SM (each owns all 512 TMEM
// columns), or 0 if the kernel cannot be resident. The answer depends only on the device and the
// instantiation, so it is looked up once per (device, instantiation) and cached; the kernel's
// shared-memory attribute is set at the same time.
// The register split needs the launch to give every thread exactly kLaunchRegs registers (with
// fewer, the epilogue's request could not be met and its warps would wait for ever): a kernel
// built with another count is never launched (the grid is reported as not resident).
template <typename K>
bool launch_regs_ok(K kernel, int launch_regs) {
  cudaFuncAttributes fa{};
  return cudaFuncGetAttributes(&fa, kernel) == cudaSuccess && fa.numRegs == launch_regs;
}

template <int D, int N>
int tc_grid() {
  using Lay = TcLayout<D, N>;
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];   // 0: unknown, -1: not resident, > 0: grid
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  const int known = cache[dev].load(std::memory_order_acquire);
  if (known != 0) return known > 0 ? known : 0;
  int sms = 0, per_sm = 0;
  int grid = -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaFuncSetAttribute(vote_tc_kernel<D, N, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::BYTES) ==
          cudaSuccess &&
      cudaFuncSetAttribute(vote_tc_kernel<D, N, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::BYTES) ==
          cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vote_tc_kernel<D, N, false>, EpiCfg<N>::kThreads,
                                                    Lay::BYTES) == cudaSuccess &&
      per_sm > 0 && launch_regs_ok(vote_tc_kernel<D, N, false>, EpiCfg<N>::kLaunchRegs) &&
      launch_regs_ok(vote_tc_kernel<D, N, true>, EpiCfg<N>::kLaunchRegs))
    grid = sms;
  cache[dev].store(grid, std::memory_order_release);
  return grid > 0 ? grid : 0;
}

template <int D>
int tc_n_pad(int rows) {
  return rows <= 16 ? 16 : (rows <= 32 ? 32 : (rows <= 64 ? 64 : 128));
}

}  // namespace

int vote_tc_keys_per_item(int q_rows, int l_obs) {
  (void)q_rows;   // grouped query heads are separate heads of l_obs rows here
  return (128 / tc_n_pad<128>(l_obs)) * kTileKeys;
}

template <int D>
int tc_grid_n(int n) {
  return n == 16 ? tc_grid<D, 16>() : n == 32 ? tc_grid<D, 32>() : n == 64 ? tc_grid<D, 64>() : tc_grid<D, 128>();
}

template <int D>
cudaError_t launch_tc_n(const CompressJob& job, int n) {
  if (n == 16) return launch_tc_typed<D, 16>(job, tc_grid<D, 16>());
  if (n == 32) return launch_tc_typed<D, 32>(job, tc_grid<D, 32>());
  if (n == 64) return launch_tc_typed<D, 64>(job, tc_grid<D, 64>());
  return launch_tc_typed<D, 128>(job, tc_grid<D, 128>());
}

bool vote_tc_eligible(const CompressJob& job) {
  if (job.dtype != SNAPKV_BF16 || job.l_obs > 128) return false;
  if (job.head_dim != 64 && job.head_dim != 128) return false;
  const int n = tc_n_pad<128>(job.l_obs);
  const int grid = job.head_dim == 64 ? tc_grid_n<64>(n) : tc_grid_n<128>(n);
  if (grid <= 0) return false;
  const int64_t per_item = vote_tc_keys_per_item(job.q_rows, job.l_obs);
  const int64_t n_chunk = (job.l_prompt + per_item - 1) / per_item;
  const int64_t q_heads = (int64_t)job.batch * job.heads * (job.q_rows / job.l_obs);
  return 2 * n_chunk * q_heads < ((int64_t)1 << 31);
}

// A ragged batch in one launch: resident mode for the longest sequence, at most kMaxVarSeq
// sequences, no grouped query heads.
bool vote_tc_ragged_eligible(const CompressJob& job) {
  if (job.n_var < 1 || job.n_var > kMaxVarSeq || job.q_rows != job.l_obs || !vote_tc_eligible(job)) return false;
  const int n = tc_n_pad<128>(job.l_obs);
  const int grid = job.head_dim == 64 ? tc_grid_n<64>(n) : tc_grid_n<128>(n);
  const int64_t per_item = vote_tc_keys_per_item(job.q_rows, job.l_obs);
  const int64_t n_chunk = (job.l_prompt + per_item - 1) / per_item;
  return n_chunk <= (int64_t)kSlots * grid;
}

cudaError_t launch_vote_tc(const CompressJob& job) {
  const int n = tc_n_pad<128>(job.l_obs);
  return job.head_dim == 64 ? launch_tc_n<64>(job, n) : launch_tc_n<128>(job, n);
}

}  // namespace snapkv
