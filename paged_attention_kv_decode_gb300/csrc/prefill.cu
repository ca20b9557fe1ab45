// Chunked prefill over a paged KV cache (prefix cache + causal chunk), on the
// 5th-generation tensor cores.
//
// The operation: vllm-metis 0.1.0 page, introduction and "How the model maps
// onto vLLM -> Caches" (prefix caching and chunked prefill on vLLM's attention
// kernels), with the chunk sizes of the vllm-mblt 0.8.0 page ("Chunked Prefill
// Auto-Tuning").  Sequence s holds seq_lens[s] cached tokens, the last
// q_len = cu_q_lens[s+1] - cu_q_lens[s] of which are queried; query i sits at
// position L - q_len + i and sees every key t <= L - q_len + i (the cached
// prefix plus a causal mask inside the chunk).  Single-token decodes are the
// q_len = 1 case and run through the same tiles.
//
// Tiling.  A query tile is 128 rows of one KV head's group: the r = H/G query
// heads times 128/r consecutive query tokens (GQA packing).  One CTA per SM
// computes TWO consecutive query tiles of the same sequence and group against
// each 128-token K/V tile, so every K/V byte gathered (page by page, with TMA,
// 128-byte swizzle) feeds 256 query rows.
//
//   warps 0..3   softmax of query tile 0, one row (TMEM lane) per thread
//   warps 4..7   softmax of query tile 1
//   warps 8..11  TMA producers: both query tiles once, then K tiles (warps 8, 9)
//                and V tiles (warps 10, 11) into 2-stage rings, each tile's pages
//                split between two warps (16-token pages make many small boxes,
//                and one warp alone cannot issue them fast enough)
//   warps 13..15 idle (they complete the last warpgroup, which gives up
//                registers to the softmax groups)
//   warp 12      allocates TMEM (S0 | S1 | O0 | O1, 512 columns); one lane
//                issues the UMMAs in the order
//                  PV0_j, QK0_{j+1}, PV1_j, QK1_{j+1}
//                so that while one softmax group works the tensor pipe runs the
//                other group's products (ping-pong).
//                  S_w = Q_w K_j^T  (M 128, N 128, K = head_dim)
//                  O_w += P_w V_j   (M 128, N head_dim, K 128; P_w read from TMEM)
// Registers: the producer and UMMA warpgroups drop to kRegsLow so that each
// softmax thread holds its row's 128 scores at once (one TMEM read per tile).
// Softmax: running max in log2 units, P = exp2(S - m) written back as bf16
// pairs over its own S columns; O is rescaled in TMEM only when the max grows
// by more than 2^8.  Because QK_w_{j+1} is issued after PV_w_j, "S_w_j landed"
// already implies "PV_w_{j-1} finished", so the rescale never waits.
//
// A small schedule kernel first lists the (sequence, query-tile pair) items
// heaviest first, so the grid has no idle CTAs.
#include <math.h>

#include <algorithm>

#include "../../include/metis_attn.h"
#include "common.cuh"
#include "host.h"
#include "tcgen05.cuh"

namespace metis {

__device__ unsigned int g_status_prefill = 0;

constexpr int kPfThreads = 512;   // 2 softmax groups + 4 TMA warps + MMA warp + 3 idle warps
constexpr int kMmaWarp = 12;
constexpr int kRegsLaunch = 65536 / kPfThreads;  // 128: the block takes the whole register file
constexpr int kRegsSoftmax = 208;                 // warpgroups 0, 1
constexpr int kRegsLow = 48;                      // warpgroups 2, 3
static_assert(128 * (2 * kRegsSoftmax + 2 * kRegsLow) <= kPfThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
constexpr int kKStages = 3;       // K ring depth (V ring: 2)
constexpr int kKvTile = 128;      // tokens per K/V tile
constexpr int kRows = 128;        // query rows per tile
constexpr int kTmemCols = 512;    // S0 | S1 | O0 | O1
constexpr int kSortMax = 2048;    // schedule: heaviest-first sort up to this many items

struct PrefillParams {
  const int32_t* cu_q_lens;
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  float* lse_out;
  const int4* items;
  const int* item_count;
  int S, T, H, G, r, Tq, bs, max_blocks, num_blocks, cap;
  float scale_log2;
};

// Shared-memory layout (all tiles 128-byte swizzled, [64-column half][row][128 B]).
template <int D>
struct PfShape {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalf = kRows * 128;                   // 128 query rows x 64 bf16
  static constexpr int kQBytes = kHalves * kQHalf;             // one query tile
  static constexpr int kKvHalf = kKvTile * 128;                // 128 tokens x 64 bf16
  static constexpr int kKvBytes = kHalves * kKvHalf;
  static constexpr int kQ = 0;                                 // 2 query tiles
  static constexpr int kK = kQ + 2 * kQBytes;                  // kKStages stages
  static constexpr int kV = kK + kKStages * kKvBytes;          // 2 stages
  static constexpr int kTiles = kV + 2 * kKvBytes;             // 224 KB at head_dim 128
  // + 1 KB: the barriers live in the alignment slack (below the aligned base when it
  // is at least 256 B, else just past the tiles).  At least 120 KB so that one CTA
  // (all 512 TMEM columns) is resident per SM.
  static constexpr int kSmem = (kTiles + 1024) > 120 * 1024 ? (kTiles + 1024) : 120 * 1024;
};

// Effective (sequence length, query count) after clamping to what can be read.
__device__ __forceinline__ void pf_lengths(const PrefillParams& p, int s, int& L, int& q_len, bool flag) {
  L = p.seq_lens[s];
  q_len = p.cu_q_lens[s + 1] - p.cu_q_lens[s];
  if (L > p.cap) {
    if (flag) atomicOr(&g_status_prefill, METIS_STATUS_SEQ_TOO_LONG);
    L = p.cap;
  }
  if (L < 0) L = 0;
  if (q_len > L || q_len < 0) {
    if (flag) atomicOr(&g_status_prefill, METIS_STATUS_BAD_Q_LEN);
    q_len = q_len < 0 ? 0 : L;
  }
}

// K/V tiles a query tile needs: keys up to the position of its last valid query.
__device__ __forceinline__ int pf_kv_tiles(int L, int q_len, int tile, int Tq) {
  const int qi0 = tile * Tq;
  if (qi0 >= q_len) return 0;
  const int p_max = L - q_len + min(q_len - 1, qi0 + Tq - 1);
  return (p_max + kKvTile) / kKvTile;
}

// ---------------------------------------------------------------------------
// schedule: the (sequence, query-tile pair) work list, heaviest first
// ---------------------------------------------------------------------------
constexpr int kSchedThreads = 1024;

__global__ void __launch_bounds__(kSchedThreads) prefill_schedule_kernel(const PrefillParams p, int4* items,
                                                                          int* count, int max_items) {
  __shared__ int scan[kSchedThreads];
  __shared__ int4 buf[kSortMax];
  pdl_launch_dependents();  // the attention kernel may start launching (it waits for the items)
  const int tid = threadIdx.x;
  const int per = (p.S + kSchedThreads - 1) / kSchedThreads;
  const int s0 = min(p.S, tid * per), s1 = min(p.S, s0 + per);
  const int pair_tokens = 2 * p.Tq;
  int local = 0;
  for (int s = s0; s < s1; ++s) {
    int L, q_len;
    pf_lengths(p, s, L, q_len, false);
    local += (q_len + pair_tokens - 1) / pair_tokens;
  }
  scan[tid] = local;
  __syncthreads();
  for (int off = 1; off < kSchedThreads; off <<= 1) {
    const int v = tid >= off ? scan[tid - off] : 0;
    __syncthreads();
    scan[tid] += v;
    __syncthreads();
  }
  const int total = min(scan[kSchedThreads - 1], max_items);
  const bool sort = total <= kSortMax;
  int pos = scan[tid] - local;
  for (int s = s0; s < s1; ++s) {
    int L, q_len;
    pf_lengths(p, s, L, q_len, false);
    const int np = (q_len + pair_tokens - 1) / pair_tokens;
    for (int t = 0; t < np; ++t, ++pos) {
      if (pos >= total) break;
      const int work = pf_kv_tiles(L, q_len, 2 * t, p.Tq) + pf_kv_tiles(L, q_len, 2 * t + 1, p.Tq);
      const int4 it = make_int4(s, t, work, 0);
      if (sort)
        buf[pos] = it;
      else
        items[pos] = it;
    }
  }
  if (sort) {
    __syncthreads();
    for (int i = tid; i < total; i += kSchedThreads) {
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

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                       const __grid_constant__ CUtensorMap tmK,
                                                                       const __grid_constant__ CUtensorMap tmV,
                                                                       const PrefillParams p) {
  using Sh = PfShape<D>;
  constexpr int HALVES = Sh::kHalves;
  pdl_wait();  // the schedule kernel's items are complete and visible
  extern __shared__ uint8_t smem_raw[];
  const uint32_t slack = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + slack;
  uint8_t* sQ = smem + Sh::kQ;
  uint8_t* sK = smem + Sh::kK;
  uint8_t* sV = smem + Sh::kV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(slack >= 256 ? smem - 256 : smem + Sh::kTiles);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [kKStages]
  uint64_t* k_empty = bars + 4;   // [kKStages]
  uint64_t* v_full = bars + 7;    // [2 stages]
  uint64_t* v_empty = bars + 9;   // [2 stages]
  uint64_t* s_full = bars + 11;   // [2 groups] QK_w_j landed in S_w
  uint64_t* p_full = bars + 13;   // [2 groups] P_w_j written over S_w (128 arrivals)
  uint64_t* pv_done = bars + 15;  // [2 groups] PV_w_j completed
  uint64_t* drain = bars + 17;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 19);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item_idx = blockIdx.x / p.G, g = blockIdx.x - item_idx * p.G;
  if (item_idx >= *p.item_count) return;
  const int4 it = p.items[item_idx];
  const int s = it.x, pair = it.y;
  int L, q_len;
  pf_lengths(p, s, L, q_len, threadIdx.x == 0);
  const int n0 = pf_kv_tiles(L, q_len, 2 * pair, p.Tq);      // K/V tiles of query tile 0
  const int n1 = pf_kv_tiles(L, q_len, 2 * pair + 1, p.Tq);  // ... of query tile 1 (0: no second tile)
  if (n0 <= 0) return;
  const int n_kv = max(n0, n1);
  const int q0 = p.cu_q_lens[s];
  const int n_pages = (L + p.bs - 1) / p.bs;

  if (threadIdx.x == 0) {
    // full barriers: one arrival per producer warp of the ring; p_full: 128 softmax threads
    for (int i = 0; i < 18; ++i) mbar_init(&bars[i], (i == 13 || i == 14) ? 128 : ((i >= 1 && i <= 3) || (i >= 7 && i <= 8)) ? 2 : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // A wait that also gives up when another role has aborted.
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < kMaxPolls; ++i) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((i & 255u) == 0) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kMaxWaitNs) break;
      }
    }
    atomicOr(&g_status_prefill, METIS_STATUS_WAIT_TIMEOUT);
    *abort_flag = 1;
    return false;
  };
  // every role calls waits with all 32 lanes: agree on the outcome before any warp-collective op
  auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool { return __all_sync(0xffffffffu, wait(bar, parity)); };

  if (warp >= 8 && warp < kMmaWarp) {
    // ------------------------------------------------------------ TMA producers
    regs_dec<kRegsLow>();
    const int pw = warp - 8;
    const bool is_k = pw < 2;
    const int part = pw & 1;                   // which half of each tile's pages
    const int32_t* bt_row = p.block_table + (size_t)s * p.max_blocks;
    if (pw == 0 && lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int ntiles = n1 > 0 ? 2 : 1;
      mbar_arrive_expect_tx(q_full, (uint32_t)(ntiles * Sh::kQBytes));
      const uint64_t pol = l2_policy_evict_first();
      for (int w = 0; w < ntiles; ++w) {
        const int qi0 = (2 * pair + w) * p.Tq;
        for (int hh = 0; hh < p.r; ++hh)
          for (int h = 0; h < HALVES; ++h)
            tma_load_3d(sQ + w * Sh::kQBytes + h * Sh::kQHalf + hh * p.Tq * 128, &tmQ, q_full, h * 64, g * p.r + hh,
                        q0 + qi0, pol);
      }
    }
    const CUtensorMap* map = is_k ? &tmK : &tmV;
    uint8_t* ring = is_k ? sK : sV;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    const int npg = kKvTile / p.bs;            // pages per K/V tile (2, 4 or 8)
    const int half_pg = npg >> 1;              // pages of this warp
    const uint64_t pol = l2_policy_evict_last();
    const int depth = is_k ? kKStages : 2;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j % depth;
      const int lp = part * half_pg + lane;    // page index inside the tile
      const int pg = j * npg + lp;
      const bool live = lane < half_pg && pg < n_pages;
      int rowc = 0;
      if (live) {
        const int b = checked_block(bt_row, pg, p.num_blocks, &g_status_prefill);
        rowc = b < 0 ? -p.bs : b * p.bs;   // a bad id reads a box entirely out of bounds: zeros
      }
      const uint32_t bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, live)) * p.bs * 128 * HALVES;
      if (j >= depth && !wait_all(&empty[st], ((j / depth) - 1) & 1)) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
      __syncwarp();
      if (live)
        for (int h = 0; h < HALVES; ++h)
          tma_load_3d(ring + st * Sh::kKvBytes + h * Sh::kKvHalf + lp * p.bs * 128, map, &full[st], h * 64, g, rowc,
                      pol);
    }
    if (*abort_flag) {
      // let the loads still in flight land before the CTA's memory goes away
      for (int j = max(0, n_kv - depth); j < n_kv; ++j) mbar_wait(&full[j % depth], (j / depth) & 1, &g_status_prefill);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ UMMA issuer
    regs_dec<kRegsLow>();
    constexpr uint32_t kIdQK = umma_idesc_bf16_f32(kRows, kKvTile, false, false);
    constexpr uint32_t kIdPV = umma_idesc_bf16_f32(kRows, D, false, true);
    const int nw[2] = {n0, n1};
    bool issued = false;
    auto qk = [&](int w, int j) {  // S_w = Q_w K_j^T
      if (lane == 0) {
        const uint32_t qbase = smem_u32(sQ + w * Sh::kQBytes);
        const uint32_t kbase = smem_u32(sK + (j % kKStages) * Sh::kKvBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t within = (kk & 3) * 32;
          umma_bf16(tmem + w * kKvTile, umma_desc_sw128(qbase + (kk >> 2) * Sh::kQHalf + within, 16, 1024),
                    umma_desc_sw128(kbase + (kk >> 2) * Sh::kKvHalf + within, 16, 1024), kIdQK, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[w]);
      }
    };
    auto pv = [&](int w, int j) {  // O_w += P_w V_j, P_w from the first 64 columns of S_w
      if (lane == 0) {
        const uint32_t vbase = smem_u32(sV + (j & 1) * Sh::kKvBytes);
        const uint32_t o_tmem = tmem + 2 * kKvTile + w * D;
#pragma unroll
        for (int kk = 0; kk < kKvTile / 16; ++kk)
          umma_bf16_tmem_a(o_tmem, tmem + w * kKvTile + kk * 8,
                           umma_desc_sw128(vbase + kk * 2048, Sh::kKvHalf, 1024), kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&pv_done[w]);
      }
    };
    bool ok = wait_all(q_full, 0) && wait_all(&k_full[0], 0);
    if (ok) {
      tc_fence_after_sync();
      qk(0, 0);
      if (n1 > 0) qk(1, 0);
      if (lane == 0) umma_commit(&k_empty[0]);  // stage of tile 0
      issued = true;
      __syncwarp();
    }
    for (int j = 0; ok && j < n_kv; ++j) {
      const int vst = j & 1;
      if (!wait_all(&v_full[vst], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int tok0 = j * kKvTile;
      if (tok0 + kKvTile > L) {
        // rows past the sequence end may hold anything (NaN included): zero them so that P = 0 stays 0
        uint8_t* vb = sV + vst * Sh::kKvBytes;
        for (int row = (L - tok0) + lane; row < kKvTile; row += 32)
          for (int h = 0; h < HALVES; ++h) {
            uint4* d = reinterpret_cast<uint4*>(vb + h * Sh::kKvHalf + row * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) d[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const bool more = j + 1 < n_kv;
      bool k_ready = false;
      for (int w = 0; w < 2; ++w) {
        if (j < nw[w]) {
          if (!wait_all(&p_full[w], j & 1)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          pv(w, j);
          // the V stage is free once the last PV of this tile has run
          if (lane == 0 && (w == 1 || nw[1] <= j)) umma_commit(&v_empty[vst]);
        }
        if (more && j + 1 < nw[w]) {
          if (!k_ready) {  // K_{j+1} is waited for only after PV0_j is on its way
            if (!wait_all(&k_full[(j + 1) % kKStages], ((j + 1) / kKStages) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            k_ready = true;
          }
          qk(w, j + 1);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0 && more) umma_commit(&k_empty[(j + 1) % kKStages]);
      __syncwarp();
    }
    if (!ok && issued) {
      // wait (bounded) for every UMMA this warp issued before TMEM is freed
      if (lane == 0) umma_commit(drain);
      __syncwarp();
      mbar_wait(drain, 0, &g_status_prefill);
    }
  } else if (warp > kMmaWarp) {
    regs_dec<kRegsLow>();  // idle: give the registers to the softmax groups
  } else {
    // ------------------------------------------------------------ softmax groups
    regs_inc<kRegsSoftmax>();
    const int w = warp >> 2;                    // query tile of this group
    const int nkv = w ? n1 : n0;
    const int row = (warp & 3) * 32 + lane;
    const int hh = row / p.Tq;
    const int qi0 = (2 * pair + w) * p.Tq;
    const int qi = qi0 + (row - hh * p.Tq);
    const bool row_valid = nkv > 0 && qi < q_len;
    const int p_min = L - q_len + qi0;          // position of the tile's first query token
    const int p_max = L - q_len + min(q_len - 1, qi0 + p.Tq - 1);
    const int p_row = row_valid ? (L - q_len + qi) : p_max;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_tmem = lane_base + w * kKvTile;
    const uint32_t o_tmem = lane_base + 2 * kKvTile + w * D;
    const float sl2 = p.scale_log2;
    const float sgn = sl2 < 0.f ? -1.f : 1.f;   // max of sl2 * s = |sl2| * max(sgn * s)
    // |sl2| > 0 keeps -inf (hidden key) * |sl2| = -inf; a zero scale becomes 1e-30, which
    // leaves every exponent equal to the max to fp32 precision (uniform weights)
    const float asl2 = fmaxf(fabsf(sl2), 1e-30f);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!wait_all(&s_full[w], j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int tok0 = j * kKvTile;
      // Visible keys of this row in this tile form a prefix: t <= p_row.
      const int vis = tok0 + kKvTile - 1 > p_min ? min(max(p_row - tok0 + 1, 0), kKvTile) : kKvTile;
      const bool lean = vis == kKvTile && sgn > 0.f;   // the common case: no mask, positive scale
      // the row's 128 scores, read once
      uint32_t sv[kKvTile];
#pragma unroll
      for (int c = 0; c < kKvTile; c += 32) tmem_ld32(s_tmem + c, sv + c);
      tmem_ld_wait();
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
      if (lean) {
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2)
          mx[(c >> 1) & 7] = max3f(mx[(c >> 1) & 7], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
      } else {
#pragma unroll
        for (int c = 0; c < kKvTile; ++c)
          mx[c & 7] = fmaxf(mx[c & 7], c < vis ? __uint_as_float(sv[c]) * sgn : -INFINITY);
      }
      const float mxa = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m_run, mxa == -INFINITY ? -INFINITY : mxa * asl2);
      const bool grow = m_new > m_run + 8.0f;   // rescale only when the max grew past 2^8
      float alpha = 1.f;
      if (grow) {
        alpha = exp2_approx(m_run - m_new);
        m_run = m_new;
      }
      if (j >= 1 && __any_sync(0xffffffffu, grow)) {
        // PV_w_{j-1} has completed: it was issued before QK_w_j, whose result we hold
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(o_tmem + c * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st32(o_tmem + c * 32, ov);
        }
      }
      l_run *= alpha;
      // P = exp2(s * |sl2| - m) as bf16 pairs (even token in the low half), packed in
      // place into sv[0, 64) and stored over the first 64 columns of S_w
      const float neg_m = -m_run;
      uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};   // row sums, as packed pairs
      const uint64_t asl2_2 = f2_pack(asl2, asl2), neg_m2 = f2_pack(neg_m, neg_m);
      if (lean) {
        // per pair: one packed FMA, two exponentials, one packed add, one bf16x2 convert
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), asl2_2, neg_m2), x0, x1);
          const float e0 = exp2_approx(x0);
          const float e1 = exp2_approx(x1);
          ls2[(c >> 1) & 3] = f2_add(ls2[(c >> 1) & 3], f2_pack(e0, e1));
          sv[c >> 1] = pack_bf16x2(e0, e1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2) {
          const float e0 = c < vis ? exp2_approx(fmaf(__uint_as_float(sv[c]) * sgn, asl2, neg_m)) : 0.f;
          const float e1 = c + 1 < vis ? exp2_approx(fmaf(__uint_as_float(sv[c + 1]) * sgn, asl2, neg_m)) : 0.f;
          ls2[(c >> 1) & 3] = f2_add(ls2[(c >> 1) & 3], f2_pack(e0, e1));
          sv[c >> 1] = pack_bf16x2(e0, e1);
        }
      }
      tmem_st32(s_tmem, sv);
      tmem_st32(s_tmem + 32, sv + 32);
      float ls[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) f2_unpack(ls2[i], ls[2 * i], ls[2 * i + 1]);
      l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&p_full[w]);
    }
    if (nkv > 0 && ok && wait_all(&pv_done[w], (nkv - 1) & 1)) {
      tc_fence_after_sync();
      const float inv = 1.0f / l_run;
      const int head = g * p.r + hh;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)(q0 + qi) * p.H + head) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_tmem + c * 32, ov);
        tmem_ld_wait();
        if (row_valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(ov[i + 4]) * inv, __uint_as_float(ov[i + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(ov[i + 6]) * inv, __uint_as_float(ov[i + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + i) = v;
          }
        }
      }
      if (row_valid && p.lse_out) p.lse_out[(size_t)(q0 + qi) * p.H + head] = (m_run + log2f(l_run)) * kLn2;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int prefill_status(uint32_t* bits, int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_status_prefill, sizeof(v));
  if (e == cudaSuccess && clear) {
    unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_status_prefill, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  *bits |= v;
  return METIS_OK;
}

// (sequence, query-tile pair) items: at most ceil(T / (2 Tq)) + S
static size_t prefill_max_items(int num_seqs, int num_tokens, int Tq) {
  return (size_t)(num_tokens + 2 * Tq - 1) / (2 * Tq) + (size_t)num_seqs;
}

template <int D>
static int launch_prefill(const PrefillParams& p0, const void* q, const void* k_cache, const void* v_cache,
                          void* workspace, size_t max_items, cudaStream_t st) {
  PrefillParams p = p0;
  int* count = reinterpret_cast<int*>(workspace);
  int4* items = reinterpret_cast<int4*>(reinterpret_cast<char*>(workspace) + 256);
  p.items = items;
  p.item_count = count;
  CUtensorMap tmQ, tmK, tmV;
  const uint64_t qdims[3] = {(uint64_t)D, (uint64_t)p.H, (uint64_t)p.T};
  const uint64_t qstr[2] = {(uint64_t)D * 2, (uint64_t)p.H * D * 2};
  const uint32_t qbox[3] = {64, 1, (uint32_t)p.Tq};
  int rc = encode_tiled(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, qdims, qstr, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t kdims[3] = {(uint64_t)D, (uint64_t)p.G, (uint64_t)p.num_blocks * p.bs};
  const uint64_t kstr[2] = {(uint64_t)D * 2, (uint64_t)p.G * D * 2};
  const uint32_t kbox[3] = {64, 1, (uint32_t)p.bs};
  rc = encode_tiled(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_cache, kdims, kstr, kbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  rc = encode_tiled(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v_cache, kdims, kstr, kbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  prefill_schedule_kernel<<<1, kSchedThreads, 0, st>>>(p, items, count, (int)max_items);
  rc = check_launch("prefill_schedule_kernel launch");
  if (rc) return rc;
  constexpr int smem = PfShape<D>::kSmem;
  static int done = 0;
  auto kern = prefill_bf16_kernel<D>;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem, &done);
  if (rc) return rc;
  // the warpgroups' register targets draw on the launch allocation: refuse to launch
  // a build whose allocation is smaller (the raising warps would wait forever)
  static int regs_checked = 0;
  if (!regs_checked) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(kern));
    if (e != cudaSuccess) return fail(METIS_E_CUDA, "cudaFuncGetAttributes: %s", cudaGetErrorString(e));
    if (fa.numRegs < kRegsLaunch)
      return fail(METIS_E_CUDA, "prefill kernel built with %d registers per thread, %d needed", fa.numRegs,
                  kRegsLaunch);
    regs_checked = 1;
  }
  return launch_dependent(kern, dim3((unsigned)(max_items * p.G)), dim3(kPfThreads), smem, st,
                          "prefill_bf16_kernel launch", tmQ, tmK, tmV, p);
}

}  // namespace metis

using namespace metis;

extern "C" size_t metis_prefill_workspace_bytes(int num_seqs, int num_tokens, int num_heads, int num_kv_heads) {
  if (num_seqs <= 0 || num_tokens <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return 0;
  const int r = num_heads / num_kv_heads;
  if (r > kRows) return 0;
  return 256 + prefill_max_items(num_seqs, num_tokens, kRows / r) * sizeof(int4);
}

extern "C" int metis_paged_attn_prefill_chunk(const void* q, const int32_t* cu_q_lens, const void* k_cache,
                                              const void* v_cache, const int32_t* block_table,
                                              const int32_t* seq_lens, void* out, float* lse_out, int num_seqs,
                                              int num_tokens, int num_heads, int num_kv_heads, int head_dim,
                                              int block_size, int max_blocks, int num_blocks, int dtype, float scale,
                                              int max_seq_len, void* workspace, size_t workspace_bytes,
                                              void* stream) {
  clear_error();
  if (num_seqs < 0 || num_tokens < 0) return fail(METIS_E_SHAPE, "num_seqs and num_tokens must be >= 0");
  if (num_seqs == 0 || num_tokens == 0) return METIS_OK;
  if (!q || !cu_q_lens || !k_cache || !v_cache || !block_table || !seq_lens || !out)
    return fail(METIS_E_NULL, "q, cu_q_lens, k_cache, v_cache, block_table, seq_lens and out are required");
  if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_blocks <= 0 ||
      num_blocks <= 0 || max_seq_len <= 0)
    return fail(METIS_E_SHAPE, "sizes must be positive");
  if (num_heads % num_kv_heads) return fail(METIS_E_SHAPE, "num_heads %% num_kv_heads != 0");
  if ((long long)max_blocks * block_size > 0x7fffffffLL || (long long)num_blocks * block_size > 0x7fffffffLL)
    return fail(METIS_E_SHAPE, "max_blocks * block_size and num_blocks * block_size must fit in int32");
  if (dtype != METIS_BF16) return fail(METIS_E_UNSUPPORTED, "prefill is built for bf16");
  if (head_dim != 64 && head_dim != 128) return fail(METIS_E_UNSUPPORTED, "head_dim must be 64 or 128");
  if (block_size != 16 && block_size != 32 && block_size != 64)
    return fail(METIS_E_UNSUPPORTED, "block_size must be 16, 32 or 64");
  const int r = num_heads / num_kv_heads;
  if (r != 1 && r != 2 && r != 4 && r != 8 && r != 16)
    return fail(METIS_E_UNSUPPORTED, "num_heads / num_kv_heads must be 1, 2, 4, 8 or 16");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(cu_q_lens, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(lse_out, 4))
    return fail(METIS_E_ALIGN, "tensors must be 16-byte aligned (index arrays and lse_out: 4-byte)");
  if (!(scale == scale)) return fail(METIS_E_SHAPE, "scale is NaN");
  const size_t need = metis_prefill_workspace_bytes(num_seqs, num_tokens, num_heads, num_kv_heads);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
    return fail(METIS_E_WORKSPACE, "workspace must hold %zu bytes (256-byte aligned)", need);
  const size_t max_items = prefill_max_items(num_seqs, num_tokens, kRows / r);
  if (max_items * num_kv_heads > 0x7fffffffull) return fail(METIS_E_SHAPE, "too many query tiles");

  PrefillParams p{};
  p.cu_q_lens = cu_q_lens;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.lse_out = lse_out;
  p.S = num_seqs;
  p.T = num_tokens;
  p.H = num_heads;
  p.G = num_kv_heads;
  p.r = r;
  p.Tq = kRows / r;
  p.bs = block_size;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.cap = (int)std::min<long long>((long long)max_blocks * block_size, (long long)max_seq_len);
  p.scale_log2 = scale * kLog2e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return head_dim == 128 ? launch_prefill<128>(p, q, k_cache, v_cache, workspace, max_items, st)
                         : launch_prefill<64>(p, q, k_cache, v_cache, workspace, max_items, st);
}
