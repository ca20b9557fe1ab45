// Multi-head latent attention (MLA) decode over a paged latent cache, on the
// 5th-generation tensor cores.
//
// The operation: the MLA kernel of the vllm-metal architecture article
// (section 3: paged attention, MLA and GDN kernels as graph primitives), fed
// by the block table and sequence lengths of section 4.  Every query head
// attends over one shared latent cache whose rows are [c_kv (512) | k_pe (64)]:
// the key is the full 576-wide row, the value its first 512 columns; queries
// arrive already in latent space (the absorbed up-projection is upstream).
//
// Decomposition.  A (sequence, partition) is computed by a CLUSTER OF TWO CTAs
// (two SMs); nothing is computed twice and every latent byte is read once:
//   * scores: CTA r owns the key dimensions D_r = [256 r, 256 r + 256) of the
//     latent part plus [512 + 32 r, 512 + 32 r + 32) of the rope part and
//     computes the partial S_r = Q[:, D_r] K[:, D_r]^T for all 128 heads;
//   * softmax: CTA r owns heads [64 r, 64 r + 64).  It sends its partial scores
//     of the other 64 heads to the peer and receives the peer's partial of its
//     own heads (fp32, through distributed shared memory), runs the online
//     softmax of its heads, and sends P of its heads (bf16) plus their rescale
//     factors back, so both CTAs hold P of all heads;
//   * output: CTA r owns output columns [256 r, 256 r + 256) (O_r in TMEM), whose
//     values are exactly the latent columns it already loads for its keys.
//
// Granularity.  A UMMA costs at least ~46 cycles whatever its N, so the scores
// are computed for 64-token tiles (N = 64); the exchange, the softmax and P V run
// on 32-token units, two per tile.  Per CTA and unit that is 18 KB of latent
// (four 128-byte-swizzled 64-column blocks plus one 64-byte-swizzled 32-column
// rope half block), streamed through an 8-unit TMA ring laid out block-major so
// that the two units of a tile form one 64-row operand per block.
//
// TMEM (512 columns): O_r 256 | S 2 x 64 | the latent part of Q_r as bf16 pairs,
// 128 (the A operand of the score UMMA).  The rope part of Q_r and the P tiles
// (the A operand of P V) sit in shared memory, so a score buffer is free as soon
// as it has been read and the next scores never wait for P V.
//
// Head order.  TMEM lane L = 32 q + 16 g + i (quarter q, half g, i < 16) holds
// head 64 g + 16 q + i of the head tile, so every lane quarter -- and with it
// every SM sub-partition, since warp w may only touch quarter w % 4 -- holds 16
// heads of each CTA: the softmax work is spread over all four sub-partitions.
//
// Warps:
//   0-3   row warps (quarter = warp): stage the partial scores of the peer's 16
//         heads of the quarter one unit ahead; softmax of its own 16 heads with
//         two lanes per head (lane i and i ^ 16, 16 tokens each; row maxima and
//         sums combined by shuffles); write P and the rescale factors; epilogue
//   4-7   rescale warps (quarter = warp - 4): once P of a unit is complete in
//         both CTAs, apply its rescale factors (own and peer heads) to O in TMEM
//   8     TMA producer          9    TMEM allocation + UMMA issue
//   10    score exchange: bulk copy staged partials to the peer, credit the peer
//         once a receive buffer has been read
//   11    P exchange: bulk copy P rows of own heads (+ factors) to the peer,
//         credit the peer once P V has released a P slot; final row statistics
//
// A schedule kernel lists the (sequence, partition) work items heaviest first.
// A sequence with one partition writes its output directly; longer ones write
// fp32 partials that the log-sum-exp merge combines.
#include <math.h>

#include <algorithm>

#include "../../include/metis_attn.h"
#include "cluster.cuh"
#include "common.cuh"
#include "host.h"
#include "tcgen05.cuh"

namespace metis {

__device__ unsigned int g_status_mla = 0;

constexpr int kMlaDq = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaHalf = 256;       // output columns (and latent key columns) per CTA
constexpr int kMlaUnit = 32;        // tokens per exchange / softmax / P V unit and per ring stage
constexpr int kMlaTile = 64;        // tokens per score UMMA (two units)
constexpr int kMlaRows = 128;       // heads per head tile (the UMMA M)
constexpr int kMlaOwn = 64;         // heads whose softmax a CTA runs
constexpr int kMlaThreads = 512;    // 16 warps
constexpr int kMlaRegsRow = 160;    // warpgroups 0 and 3: the two row-warp sets
constexpr int kMlaRegsLow = 96;     // warpgroups 1 and 2: staging/rescale, TMA, UMMA, exchanges
static_assert(128 * (2 * kMlaRegsRow + 2 * kMlaRegsLow) <= 65536, "register split exceeds the register file");
constexpr int kMlaTmemCols = 512;
constexpr int kMlaSortMax = 2048;
#ifndef METIS_MLA_STAGES
#define METIS_MLA_STAGES 8
#define METIS_MLA_NX 2
#define METIS_MLA_NP 3
#endif
constexpr int kMlaStages = METIS_MLA_STAGES;  // ring stages of one unit (even: a tile is two adjacent stages)
constexpr int kMlaNX = METIS_MLA_NX;          // partial-score exchange slots (even: each row set uses every other)
constexpr int kMlaNP = METIS_MLA_NP;          // P tile slots
static_assert(kMlaStages % 2 == 0 && kMlaNX % 2 == 0, "stage and exchange-slot counts must be even");
constexpr uint32_t kTmO = 0;        // 256 fp32 columns: O_r
constexpr uint32_t kTmS = 256;      // 2 x 64 columns: partial scores of a tile
constexpr uint32_t kTmQ = 384;      // 128 columns: latent part of Q_r as bf16 pairs

struct MlaShape {
  static constexpr int kBlk = kMlaUnit * 128;             // one unit of one 64-column block (128-byte swizzle)
  static constexpr int kRopeU = kMlaUnit * 64;            // one unit of the rope half block (64-byte swizzle)
  static constexpr int kXBuf = kMlaOwn * kMlaUnit * 4;    // partial scores of 64 heads x one unit, fp32
  static constexpr int kPBuf = kMlaRows * kMlaUnit * 2;   // P of 128 lanes x one unit, bf16, 64-byte swizzle
  static constexpr int kKv = 0;                           // block b of stage s at kKv + (b * kMlaStages + s) * kBlk
  static constexpr int kRope = kKv + 4 * kMlaStages * kBlk;  // stage s at kRope + s * kRopeU
  static constexpr int kQr = kRope + kMlaStages * kRopeU;    // rope part of Q_r: 128 lanes x 64 B, 64-byte swizzle
  static constexpr int kStg = kQr + kMlaRows * 64;        // kMlaNX staging buffers (copied to the peer)
  static constexpr int kRx = kStg + kMlaNX * kXBuf;       // kMlaNX receive buffers (written by the peer)
  static constexpr int kP = kRx + kMlaNX * kXBuf;         // kMlaNP P tiles
  static constexpr int kAlpha = kP + kMlaNP * kPBuf;      // kMlaNP x 128 rescale factors (head order)
  static constexpr int kStat = kAlpha + kMlaNP * kMlaRows * 4;  // 128 x {m, l} (head order)
  static constexpr int kHand = kStat + kMlaRows * 8;       // 2 sets x 128 running maxima + 128 row-sum shares
  static constexpr int kBars = kHand + 3 * kMlaRows * 4;
  static constexpr int kSmem = kBars + 1024 + 1024;       // barriers + alignment slack
};
static_assert(MlaShape::kSmem <= 227 * 1024, "MLA shared memory exceeds the per-CTA limit");

// mbarrier layout (indices into the barrier area) and arrival counts
struct MlaBar {
  static constexpr int kKvFull = 0, kKvEmpty = kKvFull + kMlaStages, kSFull = kKvEmpty + kMlaStages,
                       kPvDone = kSFull + 2, kStaged = kPvDone + 4, kRxFull = kStaged + kMlaNX,
                       kRxRead = kRxFull + kMlaNX, kTxOk = kRxRead + kMlaNX, kPLocal = kTxOk + kMlaNX,
                       kPRemote = kPLocal + kMlaNP, kPRelay = kPRemote + kMlaNP, kPslotOk = kPRelay + kMlaNP,
                       kQFull = kPslotOk + kMlaNP, kStatLocal = kQFull + 1, kStatFull = kStatLocal + 1,
                       kDrain = kStatFull + 1, kSFree = kDrain + 1, kHand = kSFree + 2, kFin = kHand + 8,
                       kCount = kFin + 1;
  __host__ __device__ static constexpr int arrivals(int i) {
    return (i >= kSFree && i < kSFree + 2) ? 256
           : (i >= kHand && i < kHand + 8) ? 32
           : ((i >= kStaged && i < kStaged + kMlaNX) || (i >= kRxRead && i < kRxRead + kMlaNX) ||
              (i >= kPLocal && i < kPLocal + kMlaNP) || (i >= kPRelay && i < kPRelay + kMlaNP) || i == kQFull ||
              i == kStatLocal || i == kFin)
               ? 128
               : 1;
  }
};
static_assert((MlaBar::kCount + 2) * 8 <= 1024, "MLA barrier area");

struct MlaParams {
  const uint4* q;   // [S, H, 576] bf16, read as 16-byte chunks
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  float* lse_out;
  float* part_out;  // [S, H, max_parts, 512]
  float* part_lse;  // [S, H, max_parts]
  const int4* items;
  const int* item_count;
  int S, H, hrows, head_tiles, bs, max_blocks, num_blocks, cap, P, max_parts;
  float scale_log2;
};

// partitions of sequence s: the merge reads ceil(L / P) of them (at most max_parts)
__device__ __forceinline__ int mla_parts(const MlaParams& p, int L_raw) {
  if (p.P <= 0) return 1;
  return max(1, min(L_raw / p.P + (L_raw % p.P != 0), p.max_parts));   // ceil without overflow
}

__global__ void __launch_bounds__(1024) mla_schedule_kernel(const MlaParams p, int4* items, int* count,
                                                            int max_items) {
  __shared__ int scan[1024];
  __shared__ int4 buf[kMlaSortMax];
  pdl_launch_dependents();  // the attention kernel may start launching (it waits for the items)
  const int tid = threadIdx.x;
  const int per = (p.S + 1023) / 1024;
  const int s0 = min(p.S, tid * per), s1 = min(p.S, s0 + per);
  int local = 0;
  for (int s = s0; s < s1; ++s) local += mla_parts(p, p.seq_lens[s]);
  scan[tid] = local;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {
    const int v = tid >= off ? scan[tid - off] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  const int total = min(scan[1023], max_items);
  const bool sort = total <= kMlaSortMax;
  int pos = scan[tid] - local;
  for (int s = s0; s < s1; ++s) {
    const int L_raw = p.seq_lens[s];
    const int L = max(0, min(L_raw, p.cap));
    const int n = mla_parts(p, L_raw);
    for (int part = 0; part < n; ++part, ++pos) {
      if (pos >= total) break;
      const int t0 = p.P > 0 ? part * p.P : 0;
      const int t1 = p.P > 0 ? min(L, t0 + p.P) : L;
      const int4 it = make_int4(s, part, max(0, t1 - t0), 0);
      if (sort)
        buf[pos] = it;
      else
        items[pos] = it;
    }
  }
  if (sort) {
    __syncthreads();
    for (int i = tid; i < total; i += 1024) {
      const int4 me = buf[i];
      int rank = 0;
      for (int k = 0; k < total; ++k) {
        const int w = buf[k].z;
        rank += (w > me.z) || (w == me.z && k < i);
      }
      items[rank] = me;
    }
  }
  if (tid == 0) *count = total;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kMlaThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ CUtensorMap tmKVh,
                      const MlaParams p) {
  using Sh = MlaShape;
  pdl_wait();               // the schedule kernel's items are complete and visible
  pdl_launch_dependents();  // the merge may start launching; it waits for this grid to finish
  extern __shared__ uint8_t smem_raw[];
  const uint32_t slack = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + slack;
  uint8_t* sKV = smem + Sh::kKv;
  uint8_t* sRope = smem + Sh::kRope;
  uint8_t* sQr = smem + Sh::kQr;
  uint8_t* sStg = smem + Sh::kStg;
  uint8_t* sRx = smem + Sh::kRx;
  uint8_t* sP = smem + Sh::kP;
  float* sAlpha = reinterpret_cast<float*>(smem + Sh::kAlpha);
  float* sStat = reinterpret_cast<float*>(smem + Sh::kStat);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kBars);
  uint64_t* kv_full = bars + MlaBar::kKvFull;       // [kMlaStages]
  uint64_t* kv_empty = bars + MlaBar::kKvEmpty;     // [kMlaStages]
  uint64_t* s_full = bars + MlaBar::kSFull;         // [2] partial scores of tile j in S[j & 1]
  uint64_t* pv_done = bars + MlaBar::kPvDone;       // [4] P V of unit u completed, on u % 4
  uint64_t* staged = bars + MlaBar::kStaged;        // [kMlaNX] partial scores of the peer's heads staged (128 arrivals)
  uint64_t* rx_full = bars + MlaBar::kRxFull;       // [kMlaNX] the peer's partial of own heads landed (armed with expect_tx)
  uint64_t* rx_read = bars + MlaBar::kRxRead;       // [kMlaNX] a receive buffer has been read (128 arrivals)
  uint64_t* tx_ok = bars + MlaBar::kTxOk;           // [kMlaNX] credit from the peer: it has read what we sent (remote)
  uint64_t* p_local = bars + MlaBar::kPLocal;       // [kMlaNP] P of own heads + factors written (128 arrivals)
  uint64_t* p_remote = bars + MlaBar::kPRemote;     // [kMlaNP] P of the peer's heads + factors landed (armed with expect_tx)
  uint64_t* p_relay = bars + MlaBar::kPRelay;       // [kMlaNP] O rescaled for the unit, P complete (128 arrivals)
  uint64_t* pslot_ok = bars + MlaBar::kPslotOk;     // [kMlaNP] credit from the peer: its P slot is free (remote)
  uint64_t* q_full = bars + MlaBar::kQFull;         // Q_r in TMEM / shared memory (128 arrivals)
  uint64_t* stat_local = bars + MlaBar::kStatLocal; // final statistics of own heads written (128 arrivals)
  uint64_t* stat_full = bars + MlaBar::kStatFull;   // final statistics of the peer's heads landed (armed with expect_tx)
  uint64_t* drain = bars + MlaBar::kDrain;
  uint64_t* s_free = bars + MlaBar::kSFree;         // [2] both units of tile j have been read from S[j & 1] (256 arrivals)
  uint64_t* hand = bars + MlaBar::kHand;            // [2 sets][4 quarters] running max after a unit of that set (32 arrivals)
  uint64_t* fin = bars + MlaBar::kFin;              // set 1's share of the row sums handed to set 0 (128 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + MlaBar::kCount);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + MlaBar::kCount + 1);
  float* sHand = reinterpret_cast<float*>(smem + Sh::kHand);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // == blockIdx.x & 1
  const uint32_t peer = rank ^ 1u;
  const int rest = blockIdx.x >> 1;
  const int ht = rest % p.head_tiles;
  const int item_idx = rest / p.head_tiles;
  if (item_idx >= *p.item_count) return;  // both CTAs of the cluster take the same branch
  const int4 it = p.items[item_idx];
  const int s = it.x, part = it.y;
  const int L_raw = p.seq_lens[s];
  int L = L_raw;
  if (L > p.cap) {
    if (threadIdx.x == 0 && rank == 0 && ht == 0 && part == 0) atomicOr(&g_status_mla, METIS_STATUS_SEQ_TOO_LONG);
    L = p.cap;
  }
  if (L < 0) L = 0;
  const bool direct = mla_parts(p, L_raw) == 1;
  const int t0 = p.P > 0 ? part * p.P : 0;
  const int t1 = p.P > 0 ? min(L, t0 + p.P) : L;
  const int h0 = ht * kMlaRows;
  if (t1 <= t0) {
    // nothing readable: an empty sequence gets 0 / -inf, an empty partition lse = -inf
    for (int r = threadIdx.x; r < kMlaRows; r += kMlaThreads) {
      const int head = h0 + r;
      if (head >= p.H) continue;
      const size_t sh = (size_t)s * p.H + head;
      if (direct) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + sh * kMlaDv + rank * kMlaHalf;
        for (int c = 0; c < kMlaHalf; ++c) o[c] = __float2bfloat16(0.f);
        if (rank == 0 && p.lse_out) p.lse_out[sh] = -INFINITY;
      } else if (rank == 0) {
        p.part_lse[sh * p.max_parts + part] = -INFINITY;
      }
    }
    return;
  }
  const int n_units = (t1 - t0 + kMlaUnit - 1) / kMlaUnit;
  const int n_tiles = (n_units + 1) / 2;
  const int n_pages = (L + p.bs - 1) / p.bs;
  constexpr uint32_t kPHalfBytes = kMlaOwn * 64 + kMlaOwn * 4;  // P rows + factors of 64 heads

  if (threadIdx.x == 0) {
    for (int i = 0; i < MlaBar::kCount; ++i) mbar_init(&bars[i], MlaBar::arrivals(i));
    *abort_flag = 0;
    fence_barrier_init();
    // arm the receive slots for the first units and the final statistics
    for (int x = 0; x < kMlaNX; ++x) mbar_arrive_expect_tx(&rx_full[x], Sh::kXBuf);
    for (int x = 0; x < kMlaNP; ++x) mbar_arrive_expect_tx(&p_remote[x], kPHalfBytes);
    mbar_arrive_expect_tx(stat_full, kMlaOwn * 8);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, kMlaTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // A wait that also gives up when another role has aborted.  Cluster-scope
  // acquire, which also covers the peer's arrivals on this CTA's barriers.
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t ts = global_timer_ns();
    for (uint32_t i = 1; i < kMaxPolls; ++i) {
      if (mbar_try_wait_cluster(bar, parity)) return true;
      if ((i & 255u) == 0) {
        if (*abort_flag) return false;
        if (global_timer_ns() - ts > kMaxWaitNs) break;
      }
    }
    atomicOr(&g_status_mla, METIS_STATUS_WAIT_TIMEOUT);
    *abort_flag = 1;
    return false;
  };
  auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool { return __all_sync(0xffffffffu, wait(bar, parity)); };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    regs_dec<kMlaRegsLow>();
    // Per unit and page piece: lanes 5 pi + 0..3 load the latent blocks 4 r .. 4 r + 3,
    // lane 5 pi + 4 the rope half block 512 + 32 r .. + 31.
    const int32_t* bt_row = p.block_table + (size_t)s * p.max_blocks;
    if (lane == 0) {
      tma_prefetch_desc(&tmKV);
      tma_prefetch_desc(&tmKVh);
    }
    const int R = min(p.bs, kMlaUnit);  // rows per box
    const int pieces = kMlaUnit / R;
    const int pi = lane / 5, lb = lane - pi * 5;
    const uint64_t pol = l2_policy_evict_first();
    int issued = 0;
    for (int u = 0; u < n_units; ++u) {
      const int st = u % kMlaStages;
      const int tok = t0 + u * kMlaUnit + pi * R;
      const int pg = tok / p.bs;
      const bool live = pi < pieces && pg < n_pages;
      int rowc = 0;
      if (live) {
        const int b = checked_block(bt_row, pg, p.num_blocks, &g_status_mla);
        rowc = b < 0 ? -R : b * p.bs + (tok - pg * p.bs);
      }
      const uint32_t n_live = (uint32_t)__popc(__ballot_sync(0xffffffffu, live && lb == 0));
      if (u >= kMlaStages && !wait_all(&kv_empty[st], ((u / kMlaStages) - 1) & 1)) break;
      if (lane == 0) mbar_arrive_expect_tx(&kv_full[st], n_live * (uint32_t)(R * (4 * 128 + 64)));
      __syncwarp();
      if (live) {
        if (lb < 4)
          tma_load_3d(sKV + (lb * kMlaStages + st) * Sh::kBlk + pi * R * 128, &tmKV, &kv_full[st],
                      (4 * (int)rank + lb) * 64, 0, rowc, pol);
        else
          tma_load_3d(sRope + st * Sh::kRopeU + pi * R * 64, &tmKVh, &kv_full[st], kMlaDv + 32 * (int)rank, 0, rowc,
                      pol);
      }
      ++issued;
    }
    if (*abort_flag)
      for (int u = max(0, issued - kMlaStages); u < issued; ++u)
        mbar_wait(&kv_full[u % kMlaStages], (u / kMlaStages) & 1, &g_status_mla);
  } else if (warp == 9) {
    // ------------------------------------------------------------ UMMA issuer
    regs_dec<kMlaRegsLow>();
    constexpr uint32_t kIdQK = umma_idesc_bf16_f32(kMlaRows, kMlaTile, false, false);
    constexpr uint32_t kIdPV = umma_idesc_bf16_f32(kMlaRows, kMlaHalf, false, true);
    const uint32_t kv = smem_u32(sKV), rope = smem_u32(sRope), qr = smem_u32(sQr), pt = smem_u32(sP);
    bool issued = false;
    auto qk = [&](int j) {  // partial S_j = Q_r K_r^T over this CTA's 288 key dimensions, 64 tokens
      if (lane == 0) {
        const int s0 = (2 * j) % kMlaStages;
        const uint32_t d_tmem = tmem + kTmS + (j & 1) * kMlaTile;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          umma_bf16_tmem_a(d_tmem, tmem + kTmQ + kk * 8,
                           umma_desc_sw128(kv + ((kk >> 2) * kMlaStages + s0) * Sh::kBlk + (kk & 3) * 32, 16, 1024),
                           kIdQK, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          umma_bf16(d_tmem, umma_desc_sw64(qr + kk * 32, 512), umma_desc_sw64(rope + s0 * Sh::kRopeU + kk * 32, 512),
                    kIdQK, 1u);
        umma_commit(&s_full[j & 1]);
      }
    };
    auto wait_tile = [&](int j) -> bool {  // the latent units of tile j have landed
      const int u0 = 2 * j;
      if (!wait_all(&kv_full[u0 % kMlaStages], (u0 / kMlaStages) & 1)) return false;
      if (u0 + 1 < n_units && !wait_all(&kv_full[(u0 + 1) % kMlaStages], ((u0 + 1) / kMlaStages) & 1)) return false;
      tc_fence_after_sync();
      return true;
    };
    bool ok = wait_all(q_full, 0);
    if (ok) tc_fence_after_sync();
    for (int j = 0; ok && j < 2 && j < n_tiles; ++j) {
      if (!wait_tile(j)) {
        ok = false;
        break;
      }
      qk(j);
      issued = true;
      __syncwarp();
    }
    for (int j = 0; ok && j < n_tiles; ++j) {
      if (j + 2 < n_tiles) {  // QK_{j+2} into S[j & 1] once the row warps have read tile j
        if (!wait_all(&s_free[j & 1], (j >> 1) & 1) || !wait_tile(j + 2)) {
          ok = false;
          break;
        }
        qk(j + 2);
        __syncwarp();
      }
      for (int h = 0; ok && h < 2; ++h) {
        const int u = 2 * j + h;
        if (u >= n_units) break;
        const int x = u % kMlaNP;
        if (!wait_all(&p_relay[x], (u / kMlaNP) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int st = u % kMlaStages;
        const int tok0 = t0 + u * kMlaUnit;
        if (tok0 + kMlaUnit > t1) {
          // rows past the partition end (NaN tails, pieces not loaded): zero the value columns
          for (int row = (t1 - tok0) + lane; row < kMlaUnit; row += 32)
            for (int b = 0; b < 4; ++b) {
              uint4* d = reinterpret_cast<uint4*>(sKV + (b * kMlaStages + st) * Sh::kBlk + row * 128);
#pragma unroll
              for (int c = 0; c < 8; ++c) d[c] = make_uint4(0u, 0u, 0u, 0u);
            }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < kMlaUnit / 16; ++kk)
            umma_bf16(tmem + kTmO, umma_desc_sw64(pt + x * Sh::kPBuf + kk * 32, 512),
                      umma_desc_sw128(kv + st * Sh::kBlk + kk * 2048, kMlaStages * Sh::kBlk, 1024), kIdPV,
                      (u > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&pv_done[u % 4]);
          umma_commit(&kv_empty[st]);
        }
        __syncwarp();
      }
    }
    if (!ok && issued) {
      if (lane == 0) umma_commit(drain);
      __syncwarp();
      mbar_wait(drain, 0, &g_status_mla);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ score exchange
    regs_dec<kMlaRegsLow>();
    const uint32_t peer_rx = dsmem_map(smem_u32(sRx), peer);
    const uint32_t peer_rx_full = dsmem_map(smem_u32(rx_full), peer);
    const uint32_t peer_tx_ok = dsmem_map(smem_u32(tx_ok), peer);
    int armed[kMlaNX];
#pragma unroll
    for (int x = 0; x < kMlaNX; ++x) armed[x] = x < n_units ? x : -1;
    for (int t = 0; t <= n_units; ++t) {
      if (t < n_units) {  // staged unit t -> the peer's receive slot t % kMlaNX
        const int x = t % kMlaNX;
        if (!wait_all(&staged[x], (t / kMlaNX) & 1)) break;
        if (lane == 0)
          bulk_copy_to_peer(peer_rx + x * Sh::kXBuf, smem_u32(sStg) + x * Sh::kXBuf, Sh::kXBuf, peer_rx_full + x * 8);
        __syncwarp();
      }
      const int u = t - 1;  // credit: this CTA has read unit u, so the peer may send unit u + kMlaNX
      if (u >= 0 && u + kMlaNX < n_units) {
        const int x = u % kMlaNX;
        if (!wait_all(&rx_read[x], (u / kMlaNX) & 1)) break;
        // Relaxed: the credit orders nothing but the row warps' reads of the receive
        // slot, which returned before their rx_read arrival (release).
        if (lane == 0) {
          mbar_arrive_expect_tx(&rx_full[x], Sh::kXBuf);
          mbar_arrive_remote_relaxed(peer_tx_ok + x * 8);
        }
#pragma unroll
        for (int y = 0; y < kMlaNX; ++y)
          if (y == x) armed[y] = u + kMlaNX;
        __syncwarp();
      }
    }
    // after an abort, let the peer's copies already on their way land before this CTA exits
    if (lane == 0 && *abort_flag) {
#pragma unroll
      for (int x = 0; x < kMlaNX; ++x)
        if (armed[x] >= 0) mbar_wait(&rx_full[x], (armed[x] / kMlaNX) & 1, &g_status_mla);
    }
  } else if (warp == 11) {
    // ------------------------------------------------------------ P exchange
    regs_dec<kMlaRegsLow>();
    const uint32_t peer_p = dsmem_map(smem_u32(sP), peer);
    const uint32_t peer_alpha = dsmem_map(smem_u32(sAlpha), peer);
    const uint32_t peer_p_remote = dsmem_map(smem_u32(p_remote), peer);
    const uint32_t peer_pslot_ok = dsmem_map(smem_u32(pslot_ok), peer);
    const uint32_t own_a = (uint32_t)(rank * kMlaOwn * 4);
    int armed[kMlaNP];
#pragma unroll
    for (int x = 0; x < kMlaNP; ++x) armed[x] = x < n_units ? x : -1;
    bool ok = true;
    for (int t = 0; ok && t <= n_units; ++t) {
      if (t < n_units) {  // P rows + factors of own heads for unit t -> the peer's P slot t % kMlaNP
        const int x = t % kMlaNP;
        if (!wait_all(&p_local[x], (t / kMlaNP) & 1) ||
            (t >= kMlaNP && !wait_all(&pslot_ok[x], ((t / kMlaNP) - 1) & 1))) {
          ok = false;
          break;
        }
        if (lane < 4) {  // own heads occupy lanes 32 q + 16 r .. + 15 of each quarter q: 16 rows x 64 B
          const uint32_t off = x * Sh::kPBuf + (uint32_t)(32 * lane + 16 * rank) * 64;
          bulk_copy_to_peer(peer_p + off, smem_u32(sP) + off, 16 * 64, peer_p_remote + x * 8);
        } else if (lane == 4) {
          bulk_copy_to_peer(peer_alpha + x * kMlaRows * 4 + own_a, smem_u32(sAlpha) + x * kMlaRows * 4 + own_a,
                            kMlaOwn * 4, peer_p_remote + x * 8);
        }
        __syncwarp();
      }
      const int u = t - 1;  // credit: P V of unit u completed, so the peer may send unit u + kMlaNP
      if (u >= 0 && u + kMlaNP < n_units) {
        const int x = u % kMlaNP;
        if (!wait_all(&pv_done[u % 4], (u / 4) & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&p_remote[x], kPHalfBytes);
          mbar_arrive_remote_relaxed(peer_pslot_ok + x * 8);
        }
#pragma unroll
        for (int y = 0; y < kMlaNP; ++y)
          if (y == x) armed[y] = u + kMlaNP;
        __syncwarp();
      }
    }
    // final row statistics of own heads -> the peer
    if (ok && wait_all(stat_local, 0) && lane == 0)
      bulk_copy_to_peer(dsmem_map(smem_u32(sStat), peer) + rank * kMlaOwn * 8, smem_u32(sStat) + rank * kMlaOwn * 8,
                        kMlaOwn * 8, dsmem_map(smem_u32(stat_full), peer));
    __syncwarp();
    if (lane == 0 && *abort_flag) {
#pragma unroll
      for (int x = 0; x < kMlaNP; ++x)
        if (armed[x] >= 0) mbar_wait(&p_remote[x], (armed[x] / kMlaNP) & 1, &g_status_mla);
      mbar_wait(stat_full, 0, &g_status_mla);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ rescale warps
    regs_dec<kMlaRegsLow>();
    const int quarter = warp - 4;
    const int hh = 64 * (lane >> 4) + 16 * quarter + (lane & 15);  // head (in the tile) of this lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    bool ok = true;
    for (int t = 0; ok && t < n_units; ++t) {
      const int x = t % kMlaNP;
      if (!wait_all(&p_local[x], (t / kMlaNP) & 1) || !wait_all(&p_remote[x], (t / kMlaNP) & 1)) {
        ok = false;
        break;
      }
      const float a = sAlpha[x * kMlaRows + hh];
      if (t >= 1 && __any_sync(0xffffffffu, a != 1.0f)) {
        // O holds every earlier unit only once P V of unit t - 1 completed
        if (!wait_all(&pv_done[(t - 1) % 4], ((t - 1) / 4) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < kMlaHalf / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_base + kTmO + c * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * a);
          tmem_st32(lane_base + kTmO + c * 32, ov);
        }
        tmem_st_wait();
      }
      tc_fence_before_sync();
      mbar_arrive(&p_relay[x]);
    }
  } else {
    // ------------------------------------------------------------ row warps
    // Two sets over the same lanes: warps 0-3 take the even units, warps 12-15 the
    // odd ones; the running max passes from set to set after every unit.
    regs_inc<kMlaRegsRow>();
    const int set = warp >> 3;
    const int quarter = warp & 3;
    const int g = lane >> 4, li = lane & 15;
    const bool own = g == (int)rank;
    const int xi = 16 * quarter + li;               // row within a 64-head half
    const int hh = 64 * g + xi;                      // head (in the tile) of this lane
    const int head = h0 + hh;
    const bool row_valid = hh < p.hrows && head < p.H;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const int prow = 32 * quarter + 16 * (int)rank + li;  // P row / TMEM lane of the own head this lane works on
    const int tok_half = own ? 0 : 16;                // tokens of a unit this lane exponentiates
    if (set == 0) {
      // Q_r of this lane's head: latent dims 256 r .. 256 r + 255 into TMEM columns
      // kTmQ.. as bf16 pairs (the raw row words), rope dims 512 + 32 r .. + 31 into
      // row `lane` of the 64-byte-swizzled shared tile (chunk c at c ^ ((row >> 1) & 3)).
      const uint4* src = p.q + ((size_t)s * p.H + (row_valid ? head : 0)) * (kMlaDq / 8);
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 x4 = row_valid ? __ldg(src + 32 * rank + c0 / 4 + i) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * i] = x4.x, v[4 * i + 1] = x4.y, v[4 * i + 2] = x4.z, v[4 * i + 3] = x4.w;
        }
        tmem_st32(lane_base + kTmQ + c0, v);
      }
      const int row = 32 * quarter + lane;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 x4 = row_valid ? __ldg(src + kMlaDv / 8 + 4 * rank + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sQr + row * 64 + ((c ^ ((row >> 1) & 3)) << 4)) = x4;
      }
      fence_proxy_async_smem();  // the score UMMA reads the rope tile through the async proxy
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(q_full);
    }
    const float sl2 = p.scale_log2;
    const float sgn = sl2 < 0.f ? -1.f : 1.f;
    const float asl2 = fmaxf(fabsf(sl2), 1e-30f);
    auto load_s = [&](int u, uint32_t* v) -> bool {  // this CTA's partial scores of unit u, every lane
      const int j = u >> 1;
      if (!wait_all(&s_full[j & 1], (j >> 1) & 1)) return false;
      tc_fence_after_sync();
      tmem_ld32(lane_base + kTmS + (j & 1) * kMlaTile + (u & 1) * kMlaUnit, v);
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&s_free[j & 1]);  // each unit of a tile is read once, by the set that owns it
      return true;
    };
    auto stage = [&](int u, const uint32_t* v) -> bool {  // the peer's heads of unit u -> staging slot
      const int x = u % kMlaNX;
      if (u >= kMlaNX && !wait_all(&tx_ok[x], ((u / kMlaNX) - 1) & 1)) return false;
      if (!own) {
        uint8_t* dst = sStg + x * Sh::kXBuf + xi * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(dst + ((c ^ (xi & 7)) << 4)) = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        fence_proxy_async_smem();  // the bulk copy reads through the async proxy
      }
      mbar_arrive(&staged[x]);
      return true;
    };
    // The running max after unit v (processed by the other set): take it, and bring
    // this set's share of the row sum, kept relative to the max it last saw, up to date.
    auto catch_up = [&](int v, float& m_run, float& l_run) -> bool {
      const int other = set ^ 1;
      if (!wait_all(&hand[other * 4 + quarter], (v >> 1) & 1)) return false;
      const float m_o = sHand[other * kMlaRows + quarter * 32 + lane];
      if (m_o > m_run) {
        l_run *= exp2_approx(m_run - m_o);  // 0 when nothing was seen yet (m_run = -inf, l_run = 0)
        m_run = m_o;
      }
      return true;
    };
    uint32_t cur[kMlaUnit], nxt[kMlaUnit];
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = set < n_units ? load_s(set, cur) && stage(set, cur) : true;
    for (int u = set; ok && u < n_units; u += 2) {
      const int x = u % kMlaNX;
      if (!wait_all(&rx_full[x], (u / kMlaNX) & 1)) {
        ok = false;
        break;
      }
      float sc[kMlaUnit];
      if (own) {
        const uint8_t* rx = sRx + x * Sh::kXBuf + xi * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 r4 = *reinterpret_cast<const float4*>(rx + ((c ^ (xi & 7)) << 4));
          sc[4 * c] = __uint_as_float(cur[4 * c]) + r4.x;
          sc[4 * c + 1] = __uint_as_float(cur[4 * c + 1]) + r4.y;
          sc[4 * c + 2] = __uint_as_float(cur[4 * c + 2]) + r4.z;
          sc[4 * c + 3] = __uint_as_float(cur[4 * c + 3]) + r4.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < kMlaUnit; ++c) sc[c] = 0.f;
      }
      mbar_arrive(&rx_read[x]);
      // lane pair (i, i ^ 16) splits the own head's unit: the own lane keeps tokens 0..15,
      // the partner takes tokens 16..31
      float mine[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float hi = __shfl_xor_sync(0xffffffffu, sc[16 + k], 16);
        mine[k] = own ? sc[k] : hi;
      }
      const int vis = min(kMlaUnit, t1 - (t0 + u * kMlaUnit)) - tok_half;  // visible tokens among mine
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 16; ++c) mx[c & 3] = fmaxf(mx[c & 3], c < vis ? mine[c] * sgn : -INFINITY);
      float mxa = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 16));
      // the max after unit u - 1 comes from the other set
      if (u >= 1 && !catch_up(u - 1, m_run, l_run)) {
        ok = false;
        break;
      }
      const float m_new = fmaxf(m_run, mxa == -INFINITY ? -INFINITY : mxa * asl2);
      float alpha = 1.f;
      if (m_new > m_run + 8.0f) {
        alpha = exp2_approx(m_run - m_new);
        m_run = m_new;
      }
      l_run *= alpha;
      sHand[set * kMlaRows + quarter * 32 + lane] = m_run;
      mbar_arrive(&hand[set * 4 + quarter]);  // release: the other set may take unit u + 1
      // this set's next unit: scores from TMEM, the peer's heads staged (after this
      // unit's receive, so the two CTAs' credits never wait on each other)
      if (u + 2 < n_units && !(load_s(u + 2, nxt) && stage(u + 2, nxt))) {
        ok = false;
        break;
      }
      const float neg_m = -m_run;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[8];
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        const float e0 = c < vis ? exp2_approx(fmaf(mine[c] * sgn, asl2, neg_m)) : 0.f;
        const float e1 = c + 1 < vis ? exp2_approx(fmaf(mine[c + 1] * sgn, asl2, neg_m)) : 0.f;
        ls[c & 3] += e0;
        ls[(c + 1) & 3] += e1;
        pk[c >> 1] = pack_bf16x2(e0, e1);
      }
      l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      // P slot u % kMlaNP is free once P V of unit u - kMlaNP completed
      const int xp = u % kMlaNP;
      if (u >= kMlaNP && !wait_all(&pv_done[(u - kMlaNP) % 4], ((u - kMlaNP) / 4) & 1)) {
        ok = false;
        break;
      }
      uint8_t* pr = sP + xp * Sh::kPBuf + prow * 64;
      const int sw = (prow >> 1) & 3, c0 = own ? 0 : 2;
      *reinterpret_cast<uint4*>(pr + ((c0 ^ sw) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4*>(pr + (((c0 + 1) ^ sw) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      if (own) sAlpha[xp * kMlaRows + hh] = alpha;
      fence_proxy_async_smem();  // P V and the bulk copy read P through the async proxy
      mbar_arrive(&p_local[xp]);
#pragma unroll
      for (int c = 0; c < kMlaUnit; ++c) cur[c] = nxt[c];
    }
    // the max after the last unit, for the set that did not process it
    if (ok && ((n_units - 1) & 1) != set) ok = catch_up(n_units - 1, m_run, l_run);
    float* sL = sHand + 2 * kMlaRows;
    if (set == 1) {
      // hand this set's share of the row sums to set 0, which writes the rows
      sL[quarter * 32 + lane] = l_run;
      mbar_arrive(fin);
      ok = false;
    } else if (ok && wait_all(fin, 0)) {
      l_run += sL[quarter * 32 + lane];
    } else {
      ok = false;
    }
    if (ok && wait_all(&pv_done[(n_units - 1) % 4], ((n_units - 1) / 4) & 1)) {
      const float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);  // the own head's row sum
      if (own) {
        sStat[hh * 2] = m_run;
        sStat[hh * 2 + 1] = l_tot;
        fence_proxy_async_smem();  // copied to the peer by the bulk engine
      }
      mbar_arrive(stat_local);
      // this lane's row: an own head (local statistics) or a peer head (the peer's)
      bool have = true;
      float inv = 0.f;
      if (own) {
        inv = 1.0f / l_tot;
      } else {
        have = false;
      }
      if (!__all_sync(0xffffffffu, have)) {
        if (!wait_all(stat_full, 0)) ok = false;
        if (!own) inv = 1.0f / sStat[hh * 2 + 1];
      }
      if (ok) {
        tc_fence_after_sync();
        const size_t sh = (size_t)s * p.H + head;
#pragma unroll 1
        for (int c = 0; c < kMlaHalf / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_base + kTmO + c * 32, ov);
          tmem_ld_wait();
          if (!row_valid) continue;
          if (direct) {
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + sh * kMlaDv + rank * kMlaHalf + c * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(ov[i + 4]) * inv, __uint_as_float(ov[i + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(ov[i + 6]) * inv, __uint_as_float(ov[i + 7]) * inv);
              *reinterpret_cast<uint4*>(o + i) = v;
            }
          } else {
            float* o = p.part_out + (sh * p.max_parts + part) * kMlaDv + rank * kMlaHalf + c * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(o + i) =
                  make_float4(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv,
                              __uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
          }
        }
        if (row_valid && own) {
          const float lse = (m_run + log2f(l_tot)) * kLn2;
          if (direct) {
            if (p.lse_out) p.lse_out[sh] = lse;
          } else {
            p.part_lse[sh * p.max_parts + part] = lse;
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kMlaTmemCols);
  }
  cluster_sync_all();  // no DSMEM access may target a CTA that has exited
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int mla_status(uint32_t* bits, int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_status_mla, sizeof(v));
  if (e == cudaSuccess && clear) {
    unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_status_mla, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  *bits |= v;
  return METIS_OK;
}

struct MlaWorkspace {
  size_t items_off, part_off, lse_off, total;
  int max_parts;
  size_t max_items;
};

static MlaWorkspace mla_workspace_layout(int S, int H, int max_seq_len, int P) {
  MlaWorkspace w{};
  w.max_parts = P > 0 ? (int)std::max<long long>(1, ((long long)max_seq_len + P - 1) / P) : 1;
  w.max_items = (size_t)S * w.max_parts;
  w.items_off = 256;
  w.part_off = align_up(w.items_off + w.max_items * sizeof(int4), 256);
  const size_t units = P > 0 ? (size_t)S * H * w.max_parts : 0;
  w.lse_off = align_up(w.part_off + units * kMlaDv * sizeof(float), 256);
  w.total = align_up(w.lse_off + units * sizeof(float), 256);
  return w;
}

}  // namespace metis

using namespace metis;

extern "C" size_t metis_mla_workspace_bytes(int num_seqs, int num_heads, int max_seq_len, int partition_size) {
  if (num_seqs <= 0 || num_heads <= 0 || max_seq_len <= 0 || partition_size < 0) return 0;
  return mla_workspace_layout(num_seqs, num_heads, max_seq_len, partition_size).total;
}

extern "C" int metis_mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                                const int32_t* seq_lens, void* out, float* lse_out, int num_seqs, int num_heads,
                                int d_latent, int d_rope, int block_size, int max_blocks, int num_blocks, float scale,
                                int partition_size, int max_seq_len, void* workspace, size_t workspace_bytes,
                                void* stream) {
  clear_error();
  if (num_seqs < 0) return fail(METIS_E_SHAPE, "num_seqs < 0");
  if (num_seqs == 0) return METIS_OK;
  if (!q || !kv_cache || !block_table || !seq_lens || !out)
    return fail(METIS_E_NULL, "q, kv_cache, block_table, seq_lens and out are required");
  if (num_heads <= 0 || block_size <= 0 || max_blocks <= 0 || num_blocks <= 0 || max_seq_len <= 0)
    return fail(METIS_E_SHAPE, "sizes must be positive");
  if (d_latent != kMlaDv || d_rope != kMlaDq - kMlaDv)
    return fail(METIS_E_UNSUPPORTED, "MLA is built for a 512-wide latent plus a 64-wide rope key");
  if (!(num_heads % kMlaRows == 0 || (num_heads < kMlaRows && num_heads % 16 == 0)))
    return fail(METIS_E_UNSUPPORTED, "num_heads must be a multiple of 128, or a multiple of 16 below 128");
  if (block_size != 16 && block_size != 32 && block_size != 64)
    return fail(METIS_E_UNSUPPORTED, "block_size must be 16, 32 or 64");
  if (num_seqs > 65535) return fail(METIS_E_SHAPE, "num_seqs must be <= 65535");
  if ((long long)max_blocks * block_size > 0x7fffffffLL || (long long)num_blocks * block_size > 0x7fffffffLL)
    return fail(METIS_E_SHAPE, "max_blocks * block_size and num_blocks * block_size must fit in int32");
  if (partition_size < 0 || partition_size % kMlaUnit)
    return fail(METIS_E_SHAPE, "partition_size must be 0 or a positive multiple of 32");
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || !aligned(lse_out, 4))
    return fail(METIS_E_ALIGN, "tensors must be 16-byte aligned (index arrays and lse_out: 4-byte)");
  if (!(scale == scale)) return fail(METIS_E_SHAPE, "scale is NaN");
  const MlaWorkspace lay = mla_workspace_layout(num_seqs, num_heads, max_seq_len, partition_size);
  if (!workspace || workspace_bytes < lay.total || !aligned(workspace, 256))
    return fail(METIS_E_WORKSPACE, "workspace must hold %zu bytes (256-byte aligned)", lay.total);
  const int head_tiles = (num_heads + kMlaRows - 1) / kMlaRows;
  if (lay.max_items * head_tiles * 2 > 0x7fffffffull) return fail(METIS_E_SHAPE, "too many work items");

  MlaParams p{};
  p.q = reinterpret_cast<const uint4*>(q);
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.lse_out = lse_out;
  char* ws = reinterpret_cast<char*>(workspace);
  int* count = reinterpret_cast<int*>(ws);
  int4* items = reinterpret_cast<int4*>(ws + lay.items_off);
  p.part_out = reinterpret_cast<float*>(ws + lay.part_off);
  p.part_lse = reinterpret_cast<float*>(ws + lay.lse_off);
  p.items = items;
  p.item_count = count;
  p.S = num_seqs;
  p.H = num_heads;
  p.hrows = std::min(num_heads, kMlaRows);
  p.head_tiles = head_tiles;
  p.bs = block_size;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.cap = (int)std::min<long long>((long long)max_blocks * block_size, (long long)max_seq_len);
  p.P = partition_size;
  p.max_parts = lay.max_parts;
  p.scale_log2 = scale * kLog2e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  CUtensorMap tmKV, tmKVh;
  const uint64_t kdims[3] = {(uint64_t)kMlaDq, 1, (uint64_t)num_blocks * block_size};
  const uint64_t kstr[2] = {(uint64_t)kMlaDq * 2, (uint64_t)kMlaDq * 2};
  const uint32_t kbox[3] = {64, 1, (uint32_t)std::min(block_size, kMlaUnit)};
  int rc = encode_tiled(&tmKV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_cache, kdims, kstr, kbox,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint32_t khbox[3] = {32, 1, (uint32_t)std::min(block_size, kMlaUnit)};
  rc = encode_tiled(&tmKVh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_cache, kdims, kstr, khbox,
                    CU_TENSOR_MAP_SWIZZLE_64B);
  if (rc) return rc;

  mla_schedule_kernel<<<1, 1024, 0, st>>>(p, items, count, (int)lay.max_items);
  rc = check_launch("mla_schedule_kernel launch");
  if (rc) return rc;
  static int done = 0;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(mla_decode_kernel), MlaShape::kSmem, &done);
  if (rc) return rc;
  // the warpgroups' register targets draw on the launch allocation: refuse to launch
  // a build whose allocation is smaller (the raising warps would wait forever)
  static int regs_checked = 0;
  if (!regs_checked) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(mla_decode_kernel));
    if (e != cudaSuccess) return fail(METIS_E_CUDA, "cudaFuncGetAttributes: %s", cudaGetErrorString(e));
    if (fa.numRegs * kMlaThreads < 128 * (2 * kMlaRegsRow + 2 * kMlaRegsLow))
      return fail(METIS_E_CUDA, "MLA kernel built with %d registers per thread, %d needed", fa.numRegs,
                  (2 * kMlaRegsRow + 2 * kMlaRegsLow) / 4);
    regs_checked = 1;
  }
  rc = launch_dependent(mla_decode_kernel, dim3((unsigned)(lay.max_items * head_tiles * 2)), dim3(kMlaThreads),
                        MlaShape::kSmem, st, "mla_decode_kernel launch", tmKV, tmKVh, p);
  if (rc) return rc;
  if (partition_size > 0 && lay.max_parts > 1)
    rc = launch_merge_ex(p.part_out, p.part_lse, seq_lens, partition_size, out, lse_out, num_seqs, num_heads, kMlaDv,
                         lay.max_parts, METIS_BF16, 1, st);
  return rc;
}
