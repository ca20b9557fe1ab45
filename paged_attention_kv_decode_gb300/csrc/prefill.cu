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
// q_len = 1 case: with a head ratio up to 8 the entry point hands them to the
// decode kernel (memory-bound, 16-token page units per warp) and lists no tiles
// for them here; above 8 they run through the same tiles.
//
// Tiling.  A query tile is 128 rows of one KV head's group: the r = H/G query
// heads times 128/r consecutive query tokens (GQA packing).  One CTA per SM
// computes TWO consecutive query tiles of the same sequence and group against
// each 128-token K/V tile, so every K/V byte gathered (page by page, with TMA,
// 128-byte swizzle) feeds 256 query rows.
//
//   warps 0..3   softmax of query tile 0, one row (TMEM lane) per thread
//   warps 4..7   softmax of query tile 1
//   warps 8..11  TMA producers: K tiles (warps 8, 9) and V tiles (warps 10, 11)
//                into 3- and 2-stage rings, each tile's pages
//                split between two warps (16-token pages make many small boxes,
//                and one warp alone cannot issue them fast enough)
//   warp 13      query loader; warp 14 hands out the units; warp 15 idle (the
//                last warpgroup gives up registers to the softmax groups)
//   warp 12      allocates TMEM (S0 | S1 | O0 | O1, 512 columns); one lane
//                issues the UMMAs in the order
//                  PV0_j, QK0_{j+1}, PV1_j, QK1_{j+1}
//                so that while one softmax group works the tensor pipe runs the
//                other group's products (ping-pong).
//                  S_w = Q_w K_j^T  (M 128, N 128, K = head_dim)
//                  O_w += P_w V_j   (M 128, N head_dim, K 128; P_w read from TMEM)
// Registers: the producer and UMMA warpgroups drop to kRegsProd / kRegsMma so that each
// softmax thread holds its row's 128 scores at once (one TMEM read per tile).
// Softmax: running max in log2 units, P = exp2(S - m) written back as bf16
// pairs over its own S columns; O is rescaled in TMEM only when the max grows
// by more than 2^8.  Because QK_w_{j+1} is issued after PV_w_j, "S_w_j landed"
// already implies "PV_w_{j-1} finished", so the rescale never waits.
//
// Persistent mixed batch: a small schedule kernel lists the (sequence,
// query-tile pair) items heaviest first -- the chunks of every length in one
// list -- and one CTA per SM takes units (item, KV head) from that list as it
// goes (warp 14 claims the next one with an atomic once every warp has taken the
// current one, and publishes it with its derived fields to the other warps through
// a two-slot ring).  Every role keeps its ring and barrier counters
// running across units, so the next unit's queries (warp 13, once the current
// unit's last QK has completed) and K/V tiles stream in while the current unit's
// last softmax, PV and epilogue drain.
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
constexpr int kUnitReaders = 14;  // warps 0..13 read every unit from the unit ring
constexpr int kRegsLaunch = 65536 / kPfThreads;  // 128: the block takes the whole register file
#ifndef PF_REGS_SOFTMAX
#define PF_REGS_SOFTMAX 216
#define PF_REGS_PROD 40
#define PF_REGS_MMA 40
#endif
constexpr int kRegsSoftmax = PF_REGS_SOFTMAX;  // warpgroups 0, 1: softmax
constexpr int kRegsProd = PF_REGS_PROD;        // warpgroup 2: K/V producers
constexpr int kRegsMma = PF_REGS_MMA;          // warpgroup 3: UMMA issuer, query loader, idle warps
static_assert(128 * (2 * kRegsSoftmax + kRegsProd + kRegsMma) <= kPfThreads * kRegsLaunch,
              "register split exceeds the launch allocation");
#ifndef METIS_PF_K_STAGES
#define METIS_PF_K_STAGES 3
#define METIS_PF_V_STAGES 2
#endif
constexpr int kKStages = METIS_PF_K_STAGES;  // K ring depth
constexpr int kVStages = METIS_PF_V_STAGES;  // V ring depth
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
  int* unit_head;   // next unit to hand out (the schedule kernel zeroes it)
  int S, T, H, G, r, Tq, bs, max_blocks, num_blocks, cap;
  float scale_log2;
  int skip_decodes;  // single-token sequences are served by the decode kernel: list no tiles for them
  // Decodes beside the chunk kernel (dec_ctas != NULL): the schedule kernel writes the
  // number of SMs the decode kernel keeps (*dec_ctas) and zeroes its item counter
  // (*dec_next); this kernel then launches behind that decode kernel, which lets it
  // launch only once its CTAs have waited for the schedule, so the list is ready at
  // launch: no wait at the start, the wait for the decode grid just before exiting.
  int* dec_ctas;
  int* dec_next;
  int num_sms, D;
  int wait_at_exit;
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
  static constexpr int kV = kK + kKStages * kKvBytes;          // kVStages stages
  static constexpr int kTiles = kV + kVStages * kKvBytes;      // 224 KB at head_dim 128
  // + 1 KB: the barriers live in the alignment slack (below the aligned base when it
  // is at least 256 B, else just past the tiles).  At least 120 KB so that one CTA
  // (all 512 TMEM columns) is resident per SM.
  static constexpr int kSmem = (kTiles + 1024) > 120 * 1024 ? (kTiles + 1024) : 120 * 1024;
};

// mbarrier layout (indices into the barrier area) and arrival counts
struct PfBar {
  static constexpr int kQFull = 0, kKFull = 1, kKEmpty = kKFull + kKStages, kVFull = kKEmpty + kKStages,
                       kVEmpty = kVFull + kVStages, kSFull = kVEmpty + kVStages, kPFull = kSFull + 2,
                       kPvDone = kPFull + 2, kDrain = kPvDone + 2, kQFree = kDrain + 1, kUnitFull = kQFree + 1,
                       kUnitEmpty = kUnitFull + 2, kCount = kUnitEmpty + 2;
  // full barriers: one arrival per producer warp of the ring; p_full: 128 softmax threads
  __host__ __device__ static constexpr int arrivals(int i) {
    return (i >= kPFull && i < kPFull + 2) ? 128
           : ((i >= kKFull && i < kKFull + kKStages) || (i >= kVFull && i < kVFull + kVStages)) ? 2
           : (i >= kUnitEmpty && i < kUnitEmpty + 2) ? kUnitReaders
                                                      : 1;
  }
};
static_assert((PfBar::kCount + 4) * 8 <= 256, "prefill barrier area");

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
// One SM's rates, for sizing the decodes' share of SMs beside the chunks: decode
// K/V bytes per second while the chunks run (a CTA of two 4-warp groups, each warp
// a 3-stage ring: ~192 KB in flight; timestamps on a GB300 show 453 MB of decodes
// taking ~253 us on 24 SMs beside 16 chunks of 512, i.e. ~75 GB/s per SM.  Too few
// decode SMs, so that the decodes finish last, costs far more than a few too many),
// and the chunk kernel's FLOP/s (the chunks alone reach ~1.07-1.13 PFLOP/s on 152 SMs;
// with 7 TFLOP/s per SM the mixed batch above ends its decodes and chunks together).
constexpr float kDecSmBytesPerS = 75e9f;
constexpr float kChunkSmFlopsPerS = 7.0e12f;

__global__ void __launch_bounds__(kSchedThreads) prefill_schedule_kernel(const PrefillParams p, int4* items,
                                                                          int* count, int max_items) {
  __shared__ int warp_sums[32];
  __shared__ int4 buf[kSortMax];
  pdl_launch_dependents();  // the attention kernel may start launching (it waits for the items)
  pdl_wait();  // a programmatic dependent itself: inputs are read once the previous grid completed
  const int tid = threadIdx.x;
  const int per = (p.S + kSchedThreads - 1) / kSchedThreads;
  const int s0 = min(p.S, tid * per), s1 = min(p.S, s0 + per);
  const int pair_tokens = 2 * p.Tq;
  int local = 0;
  // decode tokens read; (query, key) pairs of the chunks.  Integers and a float ratio:
  // this GPU's fp64 rate is a small fraction of its fp32 rate.
  long long dec_tok = 0, chunk_qk = 0;
  int L_first = 0, q_first = 0;  // this thread's first sequence, kept for the listing pass
  bool routed_first = false;
  for (int s = s0; s < s1; ++s) {
    int L, q_len;
    const bool routed = p.skip_decodes && p.cu_q_lens[s + 1] - p.cu_q_lens[s] == 1;
    pf_lengths(p, s, L, q_len, routed);  // a routed decode's content errors are flagged here
    if (s == s0) {
      L_first = L;
      q_first = q_len;
      routed_first = routed;
    }
    if (!routed) {
      local += (q_len + pair_tokens - 1) / pair_tokens;
      chunk_qk += (long long)q_len * (L - q_len) + (long long)q_len * (q_len + 1) / 2;
    } else {
      dec_tok += L;
    }
  }
  // The decodes' share of SMs, from warp sums published before the scan's barriers
  // and combined by the last warp (no sequences there unless S > 992): off the path
  // of the listing and the sort.
  __shared__ long long red[2][kSchedThreads / 32];
  static_assert(kSchedThreads == 32 * 32, "one warp combines the warp sums");
  const int lane = tid & 31, warp = tid >> 5;
  if (p.dec_ctas) {
    for (int o = 16; o > 0; o >>= 1) {
      dec_tok += __shfl_xor_sync(0xffffffffu, dec_tok, o);
      chunk_qk += __shfl_xor_sync(0xffffffffu, chunk_qk, o);
    }
    if (lane == 0) {
      red[0][warp] = dec_tok;
      red[1][warp] = chunk_qk;
    }
  }
  int all;
  int pos = block_exclusive_scan<kSchedThreads>(local, warp_sums, &all);
  if (p.dec_ctas && warp == kSchedThreads / 32 - 1) {
    // SMs for the decodes beside the chunks: decodes on k SMs and chunks on the
    // other N - k finish together when k / N = d / (d + c), with d and c the SM time
    // each kind needs alone (rates of one SM: kDecSmBytesPerS, kChunkSmFlopsPerS)
    long long dt = red[0][lane], cq = red[1][lane];
    for (int o = 16; o > 0; o >>= 1) {
      dt += __shfl_xor_sync(0xffffffffu, dt, o);
      cq += __shfl_xor_sync(0xffffffffu, cq, o);
    }
    if (lane == 0) {
      const float d = (float)dt * ((float)p.G * p.D * 4.0f / kDecSmBytesPerS);   // K and V rows of every decode
      const float c = (float)cq * ((float)p.H * p.D * 4.0f / kChunkSmFlopsPerS);  // QK^T and PV of every chunk query
      int k = 0;
      if (dt > 0) k = cq > 0 ? (int)ceilf(p.num_sms * (d / (d + c))) : p.num_sms;
      *p.dec_ctas = min(max(k, dt > 0 ? 1 : 0), p.num_sms);
      *p.dec_next = 0;
    }
  }
  const int total = min(all, max_items);
  const bool sort = total <= kSortMax;
  for (int s = s0; s < s1; ++s) {
    int L = L_first, q_len = q_first;
    bool routed = routed_first;
    if (s != s0) {
      pf_lengths(p, s, L, q_len, false);
      routed = p.skip_decodes && p.cu_q_lens[s + 1] - p.cu_q_lens[s] == 1;
    }
    const int np = routed ? 0 : (q_len + pair_tokens - 1) / pair_tokens;
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
    // rank = number of items heavier than this one (ties: earlier in the list first);
    // `ways` threads (a power of two, within a warp) count a share of the list each
    __syncthreads();
    int ways = 1;
    while (ways < 32 && total * ways * 2 <= kSchedThreads) ways *= 2;
    const int sub = tid & (ways - 1);
    for (int base = 0; base < total; base += kSchedThreads / ways) {  // the same trip count in every thread
      const int i = base + tid / ways;
      const bool live = i < total;
      int4 me = make_int4(0, 0, 0, 0);
      int rank = 0;
      if (live) {
        me = buf[i];
        for (int k = sub; k < total; k += ways) {
          const int w = buf[k].z;
          rank += (w > me.z) || (w == me.z && k < i);
        }
      }
      for (int o = ways >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
      if (live && sub == 0) items[rank] = me;
    }
  }
  if (tid == 0) {
    *count = total;
    *p.unit_head = 0;
  }
}

// ---------------------------------------------------------------------------
// main kernel (persistent: one CTA per SM walks the work list)
// ---------------------------------------------------------------------------
// One unit of work as every role sees it: query-tile pair `pair` of sequence s,
// KV head g.  Each role derives it from the schedule's list on its own.
struct PfUnit {
  int s, pair, g, L, q_len, n0, n1, n_kv, q0, n_pages;
};

__device__ __forceinline__ bool pf_unit(const PrefillParams& p, int u, bool flag, PfUnit& it) {
  const int item_idx = u / p.G;
  it.g = u - item_idx * p.G;
  const int4 v = __ldcg(p.items + item_idx);  // written by this call's schedule kernel: read from L2
  it.s = v.x;
  it.pair = v.y;
  pf_lengths(p, it.s, it.L, it.q_len, flag && it.g == 0);
  it.n0 = pf_kv_tiles(it.L, it.q_len, 2 * it.pair, p.Tq);      // K/V tiles of query tile 0
  it.n1 = pf_kv_tiles(it.L, it.q_len, 2 * it.pair + 1, p.Tq);  // ... of query tile 1 (0: no second tile)
  it.n_kv = max(it.n0, it.n1);
  it.q0 = p.cu_q_lens[it.s];
  it.n_pages = (it.L + p.bs - 1) / p.bs;
  return it.n0 > 0;
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                       const __grid_constant__ CUtensorMap tmK,
                                                                       const __grid_constant__ CUtensorMap tmV,
                                                                       const PrefillParams p) {
  using Sh = PfShape<D>;
  constexpr int HALVES = Sh::kHalves;
  if (!p.wait_at_exit) pdl_wait();  // the schedule kernel's items are complete and visible
  extern __shared__ uint8_t smem_raw[];
  const uint32_t slack = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + slack;
  uint8_t* sQ = smem + Sh::kQ;
  uint8_t* sK = smem + Sh::kK;
  uint8_t* sV = smem + Sh::kV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(slack >= 256 ? smem - 256 : smem + Sh::kTiles);
  uint64_t* q_full = bars + PfBar::kQFull;
  uint64_t* k_full = bars + PfBar::kKFull;      // [kKStages]
  uint64_t* k_empty = bars + PfBar::kKEmpty;    // [kKStages]
  uint64_t* v_full = bars + PfBar::kVFull;      // [kVStages]
  uint64_t* v_empty = bars + PfBar::kVEmpty;    // [kVStages]
  uint64_t* s_full = bars + PfBar::kSFull;      // [2 groups] QK_w_j landed in S_w
  uint64_t* p_full = bars + PfBar::kPFull;      // [2 groups] P_w_j written over S_w (128 arrivals)
  uint64_t* pv_done = bars + PfBar::kPvDone;    // [2 groups] PV_w_j completed
  uint64_t* drain = bars + PfBar::kDrain;
  uint64_t* q_free = bars + PfBar::kQFree;      // every QK of a unit completed: its query tiles may be replaced
  uint64_t* unit_full = bars + PfBar::kUnitFull;    // [2] a unit index published
  uint64_t* unit_empty = bars + PfBar::kUnitEmpty;  // [2] every consuming warp has read it (kUnitReaders arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + PfBar::kCount);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + PfBar::kCount + 1);
  volatile int* unit_slot = reinterpret_cast<volatile int*>(bars + PfBar::kCount + 2);  // [2]
  __shared__ PfUnit unit_info[2];  // the published unit, derived once by the fetcher

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = __ldcg(p.item_count) * p.G;
  if ((int)blockIdx.x >= units) {
    if (p.wait_at_exit) pdl_wait();  // complete only after the decode grid in front of this one
    return;
  }

  if (threadIdx.x == 0) {
    // full barriers: one arrival per producer warp of the ring; p_full: 128 softmax threads
    for (int i = 0; i < PfBar::kCount; ++i) mbar_init(&bars[i], PfBar::arrivals(i));
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
  // The k-th unit of this CTA, from the unit ring: 1 = a unit, 0 = no more, -1 = aborted.
  // The fetcher publishes the unit's derived fields with it, so that no role waits on
  // global loads at a unit boundary.
  auto next_unit = [&](uint32_t& k, PfUnit& it) -> int {
    const int slot = k & 1;
    if (!wait_all(&unit_full[slot], (k >> 1) & 1)) return -1;
    const int u = unit_slot[slot];
    if (u >= 0) it = unit_info[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&unit_empty[slot]);  // release: the reads above are done
    ++k;
    return u < 0 ? 0 : 1;
  };

  // Ring positions run on across units: K/V tile t (counted over every unit this
  // CTA has processed) sits in K stage t % kKStages and V stage t % kVStages, and each
  // barrier's phase is the number of its earlier completions.
  if (warp >= 8 && warp < kMmaWarp) {
    // ------------------------------------------------------------ K/V producers
    regs_dec<kRegsProd>();
    const int pw = warp - 8;
    const bool is_k = pw < 2;
    const int part = pw & 1;                   // which half of each tile's pages
    const CUtensorMap* map = is_k ? &tmK : &tmV;
    uint8_t* ring = is_k ? sK : sV;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    const int npg = kKvTile / p.bs;            // pages per K/V tile (2, 4 or 8)
    const int half_pg = npg >> 1;              // pages of this warp
    const uint64_t pol = l2_policy_evict_last();
    const int depth = is_k ? kKStages : kVStages;
    if (lane == 0) tma_prefetch_desc(map);
    uint32_t t = 0, k = 0;                     // tiles issued so far, units read
    bool ok = true;
    PfUnit it;
    while (ok && next_unit(k, it) > 0) {
      const int32_t* bt_row = p.block_table + (size_t)it.s * p.max_blocks;
      for (int j = 0; j < it.n_kv; ++j, ++t) {
        const int st = t % depth;
        const int lp = part * half_pg + lane;  // page index inside the tile
        const int pg = j * npg + lp;
        const bool live = lane < half_pg && pg < it.n_pages;
        int rowc = 0;
        if (live) {
          const int b = checked_block(bt_row, pg, p.num_blocks, &g_status_prefill);
          rowc = b < 0 ? -p.bs : b * p.bs;   // a bad id reads a box entirely out of bounds: zeros
        }
        const uint32_t bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, live)) * p.bs * 128 * HALVES;
        if (t >= (uint32_t)depth && !wait_all(&empty[st], ((t / depth) - 1) & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
        __syncwarp();
        if (live)
          for (int h = 0; h < HALVES; ++h)
            tma_load_3d(ring + st * Sh::kKvBytes + h * Sh::kKvHalf + lp * p.bs * 128, map, &full[st], h * 64, it.g,
                        rowc, pol);
      }
    }
    if (*abort_flag) {
      // let the loads still in flight land before the CTA's memory goes away
      for (uint32_t k = t > (uint32_t)depth ? t - depth : 0; k < t; ++k)
        mbar_wait(&full[k % depth], (k / depth) & 1, &g_status_prefill);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ UMMA issuer
    regs_dec<kRegsMma>();
    constexpr uint32_t kIdQK = umma_idesc_bf16_f32(kRows, kKvTile, false, false);
    constexpr uint32_t kIdPV = umma_idesc_bf16_f32(kRows, D, false, true);
    bool issued = false;
    auto qk = [&](int w, uint32_t t) {  // S_w = Q_w K_t^T
      if (lane == 0) {
        const uint32_t qbase = smem_u32(sQ + w * Sh::kQBytes);
        const uint32_t kbase = smem_u32(sK + (t % kKStages) * Sh::kKvBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t within = (kk & 3) * 32;
          umma_bf16(tmem + w * kKvTile, umma_desc_sw128(qbase + (kk >> 2) * Sh::kQHalf + within, 16, 1024),
                    umma_desc_sw128(kbase + (kk >> 2) * Sh::kKvHalf + within, 16, 1024), kIdQK, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[w]);
      }
    };
    auto pv = [&](int w, uint32_t t, bool first) {  // O_w (+)= P_w V_t, P_w from the first 64 columns of S_w
      if (lane == 0) {
        const uint32_t vbase = smem_u32(sV + (t % kVStages) * Sh::kKvBytes);
        const uint32_t o_tmem = tmem + 2 * kKvTile + w * D;
#pragma unroll
        for (int kk = 0; kk < kKvTile / 16; ++kk)
          umma_bf16_tmem_a(o_tmem, tmem + w * kKvTile + kk * 8,
                           umma_desc_sw128(vbase + kk * 2048, Sh::kKvHalf, 1024), kIdPV, (!first || kk > 0) ? 1u : 0u);
        umma_commit(&pv_done[w]);
      }
    };
    uint32_t t_base = 0, n_units = 0, np[2] = {0u, 0u};  // tiles, units, p_full phases consumed
    uint32_t k = 0;
    bool ok = true;
    PfUnit it;
    while (ok) {
      const int r = next_unit(k, it);
      if (r <= 0) {
        ok = r == 0;
        break;
      }
      const int nw[2] = {it.n0, it.n1};
      if (!wait_all(q_full, n_units & 1) || !wait_all(&k_full[t_base % kKStages], (t_base / kKStages) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      qk(0, t_base);
      if (it.n1 > 0) qk(1, t_base);
      if (lane == 0) {
        umma_commit(&k_empty[t_base % kKStages]);
        if (it.n_kv == 1) umma_commit(q_free);  // the unit's last QK is issued
      }
      issued = true;
      __syncwarp();
      for (int j = 0; ok && j < it.n_kv; ++j) {
        const uint32_t t = t_base + j;
        const int vst = t % kVStages;
        if (!wait_all(&v_full[vst], (t / kVStages) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int tok0 = j * kKvTile;
        if (tok0 + kKvTile > it.L) {
          // rows past the sequence end may hold anything (NaN included): zero them so that P = 0 stays 0
          uint8_t* vb = sV + vst * Sh::kKvBytes;
          for (int row = (it.L - tok0) + lane; row < kKvTile; row += 32)
            for (int h = 0; h < HALVES; ++h) {
              uint4* d = reinterpret_cast<uint4*>(vb + h * Sh::kKvHalf + row * 128);
#pragma unroll
              for (int c = 0; c < 8; ++c) d[c] = make_uint4(0u, 0u, 0u, 0u);
            }
          fence_proxy_async_smem();
          __syncwarp();
        }
        const bool more = j + 1 < it.n_kv;
        bool k_ready = false;
        for (int w = 0; w < 2; ++w) {
          if (j < nw[w]) {
            if (!wait_all(&p_full[w], np[w] & 1)) {
              ok = false;
              break;
            }
            ++np[w];
            tc_fence_after_sync();
            pv(w, t, j == 0);
            // the V stage is free once the last PV of this tile has run
            if (lane == 0 && (w == 1 || nw[1] <= j)) umma_commit(&v_empty[vst]);
          }
          if (more && j + 1 < nw[w]) {
            if (!k_ready) {  // K_{t+1} is waited for only after PV0_t is on its way
              if (!wait_all(&k_full[(t + 1) % kKStages], ((t + 1) / kKStages) & 1)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              k_ready = true;
            }
            qk(w, t + 1);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0 && more) {
          umma_commit(&k_empty[(t + 1) % kKStages]);
          if (j + 2 == it.n_kv) umma_commit(q_free);  // the unit's last QK is issued
        }
        __syncwarp();
      }
      t_base += it.n_kv;
      ++n_units;
    }
    if (!ok && issued) {
      // wait (bounded) for every UMMA this warp issued before TMEM is freed
      if (lane == 0) umma_commit(drain);
      __syncwarp();
      mbar_wait(drain, 0, &g_status_prefill);
    }
  } else if (warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ query loader
    regs_dec<kRegsMma>();
    if (lane == 0) tma_prefetch_desc(&tmQ);
    uint32_t n_units = 0, k = 0;
    PfUnit it;
    while (next_unit(k, it) > 0) {
      // the previous unit's query tiles stay until its last QK has completed
      if (n_units > 0 && !wait_all(q_free, (n_units - 1) & 1)) break;
      if (lane == 0) {
        const int ntiles = it.n1 > 0 ? 2 : 1;
        mbar_arrive_expect_tx(q_full, (uint32_t)(ntiles * Sh::kQBytes));
        const uint64_t pol = l2_policy_evict_first();
        for (int w = 0; w < ntiles; ++w) {
          const int qi0 = (2 * it.pair + w) * p.Tq;
          for (int hh = 0; hh < p.r; ++hh)
            for (int h = 0; h < HALVES; ++h)
              tma_load_3d(sQ + w * Sh::kQBytes + h * Sh::kQHalf + hh * p.Tq * 128, &tmQ, q_full, h * 64,
                          it.g * p.r + hh, it.q0 + qi0, pol);
        }
      }
      __syncwarp();
      ++n_units;
    }
    if (*abort_flag && n_units > 0) mbar_wait(q_full, (n_units - 1) & 1, &g_status_prefill);
  } else if (warp == kMmaWarp + 2) {
    // ------------------------------------------------------------ unit fetcher
    // claims units from the global list, heaviest first, and publishes them to
    // the other warps through the two-slot unit ring; -1 ends the walk.  Unit k is
    // claimed only once every warp has taken unit k - 1: one unit of lookahead, so
    // that at the end of the list no CTA holds small units that an idle CTA could run.
    regs_dec<kRegsMma>();
    uint32_t k = 0;
    for (;;) {
      const int slot = k & 1;
      if (k >= 1 && !wait_all(&unit_empty[(k - 1) & 1], ((k - 1) >> 1) & 1)) break;
      int u = 0;
      if (lane == 0) u = atomicAdd(p.unit_head, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      PfUnit it;
      if (u < units) {
        if (!pf_unit(p, u, lane == 0, it)) continue;   // nothing to compute (length errors flagged here)
      } else {
        u = -1;
      }
      if (lane == 0) {
        if (u >= 0) unit_info[slot] = it;
        unit_slot[slot] = u;
        mbar_arrive(&unit_full[slot]);  // release: the unit's fields are visible to every waiter
      }
      __syncwarp();
      ++k;
      if (u < 0) break;
    }
  } else if (warp > kMmaWarp) {
    regs_dec<kRegsMma>();  // idle: give the registers to the softmax groups
  } else {
    // ------------------------------------------------------------ softmax groups
    regs_inc<kRegsSoftmax>();
    const int w = warp >> 2;                    // query tile of this group
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_tmem = lane_base + w * kKvTile;
    const uint32_t o_tmem = lane_base + 2 * kKvTile + w * D;
    const float sl2 = p.scale_log2;
    const float sgn = sl2 < 0.f ? -1.f : 1.f;   // max of sl2 * s = |sl2| * max(sgn * s)
    // |sl2| > 0 keeps -inf (hidden key) * |sl2| = -inf; a zero scale becomes 1e-30, which
    // leaves every exponent equal to the max to fp32 precision (uniform weights)
    const float asl2 = fmaxf(fabsf(sl2), 1e-30f);
    uint32_t ns = 0, npv = 0, k = 0;            // s_full phases consumed, PVs of this group, units read
    bool ok = true;
    PfUnit it;
    while (ok && next_unit(k, it) > 0) {
      const int nkv = w ? it.n1 : it.n0;
      if (nkv == 0) continue;                   // no second query tile in this unit
      const int L = it.L, q_len = it.q_len;
      const int hh = row / p.Tq;
      const int qi0 = (2 * it.pair + w) * p.Tq;
      const int qi = qi0 + (row - hh * p.Tq);
      const bool row_valid = qi < q_len;
      const int p_min = L - q_len + qi0;        // position of the tile's first query token
      const int p_max = L - q_len + min(q_len - 1, qi0 + p.Tq - 1);
      const int p_row = row_valid ? (L - q_len + qi) : p_max;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkv; ++j) {
        if (!wait_all(&s_full[w], ns & 1)) {
          ok = false;
          break;
        }
        ++ns;
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
        if (!lean) {
          // fold the mask (a select: NaN-safe) and a negative scale's sign into the
          // scores once, so that one code path serves every tile
#pragma unroll
          for (int c = 0; c < kKvTile; ++c)
            sv[c] = c < vis ? __float_as_uint(__uint_as_float(sv[c]) * sgn) : 0xff800000u;
        }
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2)
          mx[(c >> 1) & 7] = max3f(mx[(c >> 1) & 7], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
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
        // per pair: one packed FMA, two exponentials, one packed add, one bf16x2 convert
        // (a hidden key is -inf here and m_run is finite after tile 0, where every row sees
        // key 0: its exponential is exactly 0)
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), asl2_2, neg_m2), x0, x1);
          const float e0 = exp2_approx(x0);
          const float e1 = exp2_approx(x1);
          ls2[(c >> 1) & 3] = f2_add(ls2[(c >> 1) & 3], f2_pack(e0, e1));
          sv[c >> 1] = pack_bf16x2(e0, e1);
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
      if (!ok) break;
      npv += nkv;
      if (!wait_all(&pv_done[w], (npv - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float inv = 1.0f / l_run;
      const int head = it.g * p.r + hh;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)(it.q0 + qi) * p.H + head) * D;
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
      if (row_valid && p.lse_out) p.lse_out[(size_t)(it.q0 + qi) * p.H + head] = (m_run + log2f(l_run)) * kLn2;
      // the next unit's first PV_w overwrites O_w: every lane has read it
      tc_fence_before_sync();
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (p.wait_at_exit) pdl_wait();  // complete only after the decode grid in front of this one
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

// The schedule kernel, then `between(p)` (the decodes of a mixed batch, or
// nothing), then the chunk kernel.
template <int D, typename Between>
static int launch_prefill(const PrefillParams& p0, const void* q, const void* k_cache, const void* v_cache,
                          void* workspace, size_t max_items, int sms, cudaStream_t st, Between between) {
  PrefillParams p = p0;
  int* count = reinterpret_cast<int*>(workspace);
  int4* items = reinterpret_cast<int4*>(reinterpret_cast<char*>(workspace) + 256);
  p.items = items;
  p.item_count = count;
  p.unit_head = count + 1;
  if (p.skip_decodes) {
    p.dec_ctas = count + 2;
    p.dec_next = count + 3;
    p.wait_at_exit = 1;
  }
  p.num_sms = sms;
  p.D = D;
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
  // a programmatic dependent of the kernel before it (e.g. the paged K/V write): its
  // launch overlaps that kernel's tail
  rc = launch_dependent(prefill_schedule_kernel, dim3(1), dim3(kSchedThreads), 0, st, "prefill_schedule_kernel launch",
                        p, items, count, (int)max_items);
  if (rc) return rc;
  rc = between(p);
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
  // persistent: at most one CTA per SM, each taking units from the list as it goes
  // (beside the decodes: the CTAs past the SMs they keep start as their CTAs finish)
  const size_t grid = std::min<size_t>(max_items * p.G, (size_t)std::max(sms, 1));
  return launch_dependent(kern, dim3((unsigned)grid), dim3(kPfThreads), smem, st, "prefill_bf16_kernel launch", tmQ,
                          tmK, tmV, p);
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
  // Single-token sequences (the decodes of a mixed batch) go through the decode
  // kernel, which streams their K/V at the memory rate (a 128-row query tile would
  // hold r valid rows of them).  It runs beside the chunk kernel: the schedule
  // kernel gives it a share of the SMs in proportion to the decodes' bytes against
  // the chunks' FLOPs, its other CTAs exit at once, and the chunk kernel -- launched
  // behind it, which it allows only after its CTAs waited for the schedule -- takes
  // the remaining SMs at once and the decodes' SMs as they finish.  Head ratios
  // above 8 stay on the chunk path.
  p.skip_decodes = r <= 8 && num_seqs <= 65535;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "querying the SM count: %s", cudaGetErrorString(e));
  sms = std::max(sms, 1);
  auto between = [&](const PrefillParams& pp) -> int {
    if (!pp.skip_decodes) return METIS_OK;
    return launch_decode_rows_beside(q, k_cache, v_cache, block_table, seq_lens, cu_q_lens, out, lse_out, num_seqs,
                                     num_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks, scale,
                                     pp.cap, pp.dec_ctas, pp.dec_next, sms, st);
  };
  return head_dim == 128 ? launch_prefill<128>(p, q, k_cache, v_cache, workspace, max_items, sms, st, between)
                         : launch_prefill<64>(p, q, k_cache, v_cache, workspace, max_items, sms, st, between);
}
