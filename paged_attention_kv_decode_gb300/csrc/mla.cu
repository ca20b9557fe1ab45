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
// (two SMs), because one SM cannot hold the 128 x 512 fp32 output (all of TMEM)
// next to the scores and the queries:
//   * scores: CTA r owns the key dimensions D_r = [256 r, 256 r + 256) of the
//     latent part plus [512 + 32 r, 512 + 32 r + 32) of the rope part and
//     computes the partial S_r = Q[:, D_r] K[:, D_r]^T for all 128 heads;
//   * ONE exchange per 64-token unit: each CTA scales its partial scores of all
//     heads into the log2 domain, rounds them to fp16 and stores them straight
//     into the peer's shared memory (asynchronous distributed-shared-memory
//     stores that count their bytes on the peer's barrier, which the peer armed
//     with the 16 KB it awaits); both CTAs form S = f16(S_0) + f16(S_1) in fp32
//     (addition commutes: both get the same bits) and both run the softmax of
//     every head -- no probabilities travel back.  The rounding moves a score by
//     at most 2^-11 (|S_0| + |S_1|), below the bf16 rounding that the queries and
//     the latent carry (2^-9 each), and halves the slots, which buys the ring
//     its fifth stage;
//   * output: CTA r owns output columns [256 r, 256 r + 256) (O_r in TMEM), whose
//     values are exactly the latent columns it already loads for its keys.
//
// Online softmax with a lagged reference.  Two sets of row warps take the even
// and the odd units.  Unit u exponentiates against a reference c_u (log2
// domain): R_{u-2} = max(c_0 .. c_{u-2}), the reference O holds after unit
// u - 2, kept as long as the unit's own maximum stays within 2^8 of it, else the
// unit's maximum.  So P <= 2^8 always, every choice depends on the data alone
// (results are bitwise reproducible), and a set needs from the other set only
// R_{u-3}, which that set publishes as it starts unit u - 1, a unit ahead of
// use.  Each unit hands its
// P (bf16, shared memory), c and row sum to four rescale warps, which replay
// the units in order against O's reference C: c > C rescales O in TMEM by
// 2^(C - c) (after the previous P V completes); c < C scales the unit's P rows
// by 2^(c - C) instead (never O up, which could overflow); c = C costs nothing.
//
// Per 64-token unit and CTA: 36 KB of latent through a 5-stage TMA ring (four
// 128-byte-swizzled 64-column blocks and one 64-byte-swizzled 32-column rope
// block); the score UMMA is M 128 x N 64 x K 288 (Q_r's latent part from TMEM,
// its rope part from shared memory); P V is M 128 x N 256 x K 64.  The unit's
// 16 KB exchange slot first receives the peer's partial scores, then holds P
// (the peer writes the slot again only after P V of the unit completed, which
// the UMMA warp signals to it with a multicast commit).  The slot is laid out
// per row warp: warp w's 32 heads own bytes [4 KB w, 4 KB (w + 1)), the scores
// as [16-byte chunk][lane] (so one warp-wide store or load is 512 contiguous
// bytes, also across the cluster), and P's 128-byte-swizzled rows in dense 8-row
// groups (1 KB apart), so the P rows of warp w fall exactly on warp w's own scores:
// a warp overwrites what it has just read and needs no other warp.
//
// TMEM (512 columns): O_r 256 | S 2 x 64 | Q_r's latent part as bf16 pairs 128.
//
// Warps:
//   0-3, 4-7  row warps, set 0 (even units) and set 1 (odd units); thread =
//             head row = TMEM lane (warp w may only touch lanes 32 (w % 4) ..)
//   8-11      rescale warps: load Q_r, replay the units' references in order,
//             epilogue (O / l, lse)
//   12        TMA producer      13   TMEM allocation + score UMMAs      14   P V UMMAs      15 idle
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
constexpr int kMlaUnit = 64;        // tokens per unit: one score tile (UMMA N), exchange, softmax step and P V
constexpr int kMlaAlign = 32;       // partitions start on multiples of this many tokens (TMA boxes never cross pages)
constexpr int kMlaRows = 128;       // heads per head tile (the UMMA M)
constexpr int kMlaThreads = 512;    // 16 warps
constexpr int kMlaRegsRow = 144;    // warpgroups 0 and 1: the two row-warp sets
constexpr int kMlaRegsLow = 112;    // warpgroups 2 and 3: rescale, TMA, UMMA
static_assert(128 * (2 * kMlaRegsRow + 2 * kMlaRegsLow) <= 65536, "register split exceeds the register file");
constexpr int kMlaTmemCols = 512;
constexpr int kMlaSortMax = 2048;
constexpr int kMlaStages = 5;       // TMA ring stages (one unit each)
constexpr float kMlaSlack = 8.0f;   // a unit keeps a published reference while its maximum is within 2^8 of it
constexpr int kMlaWorkCache = 128;  // works per cluster kept in shared memory (beyond: read from the list)
constexpr int kMlaInlineSeqs = 512;  // batches up to this many sequences are ranked inside the kernel
constexpr uint32_t kTmO = 0;        // 256 fp32 columns: O_r
constexpr uint32_t kTmS = 256;      // 2 x 64 columns: partial scores of the units of set 0 / set 1
constexpr uint32_t kTmQ = 384;      // 128 columns: latent part of Q_r as bf16 pairs

struct MlaShape {
  static constexpr int kBlk = kMlaUnit * 128;             // one 64-column block of a unit (128-byte rows)
  static constexpr int kStage = 4 * kBlk;                 // the unit's latent columns of this CTA
  static constexpr int kRopeU = kMlaUnit * 64;            // the unit's rope half block (64-byte rows)
  static constexpr int kSlotB = kMlaRows * kMlaUnit * 2;  // exchange slot: fp16 partial scores, later bf16 P
  static constexpr int kWarpB = kSlotB / 4;               // a row warp's part of the slot
  static constexpr int kPGroup = 1024;                    // P: bytes between 8-row groups
  static constexpr int kKv = 0;                           // stage s at kKv + s * kStage, block b at + b * kBlk
  static constexpr int kRope = kKv + kMlaStages * kStage; // stage s at kRope + s * kRopeU
  static constexpr int kSlot = kRope + kMlaStages * kRopeU;  // slot k (units of set k) at kSlot + k * kSlotB
  static constexpr int kQr = kSlot + 2 * kSlotB;          // rope part of Q_r: 128 rows x 64 B, 64-byte swizzle
  static constexpr int kTag = kQr + kMlaRows * 64;        // per slot: 128 references c, 128 row sums l
  static constexpr int kRef = kTag + 2 * 2 * kMlaRows * 4;  // per set: R_w of its last unit w, 128 heads
  static constexpr int kWorks = kRef + 2 * kMlaRows * 4;   // the cluster's work list: int4 {s, part, ht, L_raw}
  static constexpr int kBars = kWorks + kMlaWorkCache * 16;
  static constexpr int kSmem = kBars + 512 + 1024;        // barriers + alignment slack
};
static_assert(MlaShape::kSmem <= 227 * 1024, "MLA shared memory exceeds the per-CTA limit");
static_assert(MlaShape::kSlot % 1024 == 0 && MlaShape::kSlotB % 1024 == 0, "P tiles must sit on 1024-byte atoms");

// mbarrier layout (indices into the barrier area) and arrival counts
struct MlaBar {
  static constexpr int kKvFull = 0, kKvEmpty = kKvFull + kMlaStages, kSFull = kKvEmpty + kMlaStages,
                       kSFree = kSFull + 2, kRxFull = kSFree + 2, kTxOk = kRxFull + 2,
                       kPFull = kTxOk + 2, kPGo = kPFull + 2, kPvDone = kPGo + 2, kRefFull = kPvDone + 2,
                       kQFull = kRefFull + 2, kOFree = kQFull + 1, kDrain = kOFree + 1, kCount = kDrain + 2;
  __host__ __device__ static constexpr int arrivals(int i) {
    return ((i >= kSFree && i < kSFree + 2) || (i >= kPFull && i < kPFull + 2) || (i >= kPGo && i < kPGo + 2) ||
            (i >= kRefFull && i < kRefFull + 2) || i == kQFull || i == kOFree)
               ? 128
               : 1;
  }
};
static_assert((MlaBar::kCount + 4) * 8 <= 512, "MLA barrier area");

struct MlaParams {
  const uint4* q;   // [S, H, 576] bf16, read as 16-byte chunks
  const void* kv;   // [num_blocks, bs, 576] bf16 (read through the tensor maps; its address for L2 prefetches)
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  float* lse_out;
  float* part_out;  // [S, H, max_parts, 512]
  float* part_lse;  // [S, H, max_parts]
  const int4* items;
  const int* item_count;
  int S, H, hrows, head_tiles, bs, max_blocks, num_blocks, cap, P, max_parts;
  int box_rows;     // rows per TMA box (a divisor of the unit that never crosses a page)
  float scale_log2;
  int q_v8;         // 1: q is 32-byte aligned (its rows are read in 32-byte pieces), else 16-byte pieces
  int inline_list;  // 1: each CTA ranks its own works (no schedule kernel, items / item_count unused)
};

// partitions of sequence s: the merge reads ceil(L / P) of them (at most max_parts)
__device__ __forceinline__ int mla_parts_of(int P, int max_parts, int L_raw) {
  if (P <= 0) return 1;
  return max(1, min(L_raw / P + (L_raw % P != 0), max_parts));   // ceil without overflow
}
__device__ __forceinline__ int mla_parts(const MlaParams& p, int L_raw) { return mla_parts_of(p.P, p.max_parts, L_raw); }

__global__ void __launch_bounds__(1024) mla_schedule_kernel(const MlaParams p, int4* items, int* count,
                                                            int max_items) {
  __shared__ int warp_sums[32];
  __shared__ int4 buf[kMlaSortMax];
  pdl_launch_dependents();  // the attention kernel may start launching (it waits for the items)
  pdl_wait();  // a programmatic dependent itself: inputs are read once the previous grid completed
  const int tid = threadIdx.x;
  const int per = (p.S + 1023) / 1024;
  const int s0 = min(p.S, tid * per), s1 = min(p.S, s0 + per);
  int local = 0;
  for (int s = s0; s < s1; ++s) local += mla_parts(p, p.seq_lens[s]);
  int all;
  int pos = block_exclusive_scan<1024>(local, warp_sums, &all);
  const int total = min(all, max_items);
  const bool sort = total <= kMlaSortMax;
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

// One (item, head tile) of a cluster's work: the tokens [t0, t1) of sequence s.
struct MlaWork {
  int s, part, ht, L_raw, t0, t1, n_units;
  bool direct;
};

// Position in the heaviest-first list of the r-th work of cluster c of G: the
// positions c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... (a snake over the list), which
// balances the lognormal lengths nearly as well as greedy longest-first
// assignment and needs no communication.
__device__ __forceinline__ long long mla_work_pos(int c, int G, int r) {
  return (long long)r * G + ((r & 1) ? G - 1 - c : c);
}

// {s, part, ht, L_raw} of list position pos (global reads)
__device__ __forceinline__ int4 mla_work_raw(const MlaParams& p, long long pos) {
  const int4 it = p.items[(int)(pos / p.head_tiles)];
  return make_int4(it.x, it.y, (int)(pos % p.head_tiles), p.seq_lens[it.x]);
}

__device__ __forceinline__ MlaWork mla_work_decode(const MlaParams& p, int4 raw) {
  MlaWork w;
  w.s = raw.x;
  w.part = raw.y;
  w.ht = raw.z;
  w.L_raw = raw.w;
  const int L = max(0, min(w.L_raw, p.cap));
  w.direct = mla_parts(p, w.L_raw) == 1;
  w.t0 = p.P > 0 ? w.part * p.P : 0;
  w.t1 = p.P > 0 ? min(L, w.t0 + p.P) : L;
  w.n_units = w.t1 > w.t0 ? (w.t1 - w.t0 + kMlaUnit - 1) / kMlaUnit : 0;
  return w;
}

// Warm L2 with the 16-byte aligned interior of [ptr, ptr + bytes): one bulk prefetch,
// no registers, no completion.
__device__ __forceinline__ void l2_prefetch_bytes(const void* ptr, size_t bytes) {
  const uintptr_t lo = (reinterpret_cast<uintptr_t>(ptr) + 15) & ~(uintptr_t)15;
  const uintptr_t hi = (reinterpret_cast<uintptr_t>(ptr) + bytes) & ~(uintptr_t)15;
  if (hi > lo)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"((uint32_t)(hi - lo)) : "memory");
}

// A work's cost, for dealing the list out: its units plus the fixed cost of a work
// boundary, ~5 units (per-cluster finish times on a GB300 fit 1.16 us per unit plus
// 5.7 us per work).
constexpr int kMlaWorkOverheadUnits = 5;
// Scratch (ints) that the in-kernel ranking uses, inside the exchange slots, which
// are free until the pipelines start.
constexpr int kMlaScratchInts = 2 * MlaShape::kSlotB / 4;
constexpr int kMlaDealFixed = 2 * kMlaInlineSeqs + 32 + 2 * kMlaThreads + kMlaWorkCache;
constexpr int kMlaDealMax = (kMlaScratchInts - kMlaDealFixed) / 2;  // works the dealt list can hold

// Small batches: the works of cluster cl of G, ranked by every CTA itself instead
// of by a schedule kernel.  The list is every (sequence, partition) ordered by
// tokens, heaviest first, ties in (sequence, partition) order -- the schedule
// kernel's order -- times the head tiles.  A sequence's partitions are `full` of P
// tokens, then at most one partial one (0 < rem < P tokens), then empty ones, so
// the list is: every full partition in sequence order (a prefix sum), the partial
// ones by rem (a count over the sequences), every empty one in sequence order (a
// prefix sum).  Without a split each sequence is one "partial" partition of all
// its tokens.  Thread t ranks sequence t (S <= the block size).
//
// The list is then dealt out in passes of G positions: pass 0 gives position c to
// cluster c; each later pass gives its positions, heaviest first, to the clusters
// in the order of their cost so far, lightest first (ties: lower cluster index),
// with the cost of a work its units plus kMlaWorkOverheadUnits -- longest-processing-
// time-first by passes.  (A snake over the list, positions c, 2G - 1 - c, 2G + c, ...,
// balances the units but hands the last partial pass's small works to clusters that
// already hold the heaviest ones.)  Lists longer than kMlaDealMax fall back to the
// snake.  sWorks[r] receives the cluster's r-th work, *n_mine the number of them
// (written by thread 0).  On the way, the thread that ranks the cluster's pass-0 work
// warms L2 with that work's queries and first pages (rank-0 CTA only).  Returns the
// number of works (items x head tiles); the list has fewer than 2^15 items.
// `scratch` holds kMlaScratchInts ints.
__device__ __forceinline__ int mla_rank_inline(const MlaParams& p, int* scratch, int4* sWorks, int cl, int G,
                                               int* n_mine) {
  const int S = p.S, P = p.P, cap = p.cap, max_parts = p.max_parts, head_tiles = p.head_tiles;
  int* sRem = scratch;                               // [S] tokens of the partial partition (0: none)
  int* sWarp = sRem + kMlaInlineSeqs;                // scan scratch
  int* sLen = sWarp + 32;                            // [S] raw lengths
  int* sLoad = sLen + kMlaInlineSeqs;                // [G] cost dealt to each cluster
  int* sOrder = sLoad + kMlaThreads;                 // [G] a cluster's place in a pass
  int* sMine = sOrder + kMlaThreads;                 // [passes] this cluster's list positions
  int* sCost = sMine + kMlaWorkCache;                // [n_work] cost of each list position
  int* sWork = sCost + kMlaDealMax;                  // [n_work] sq << 16 | q << 4 | ht of each position
  const int sq = threadIdx.x;
  int np = 0, full = 0, has = 0, rem = 0, Lr = 0;
  if (sq < S) {
    Lr = p.seq_lens[sq];
    const int Lc = max(0, min(Lr, cap));
    np = mla_parts_of(P, max_parts, Lr);
    if (P <= 0) {
      has = 1;
      rem = Lc;
    } else {
      full = min(np, Lc / P);
      rem = full < np ? Lc - full * P : 0;
      has = rem > 0;
    }
    sRem[sq] = rem;
    sLen[sq] = Lr;
  }
  const int empty = np - full - has;
  // full and empty counts packed in one scan (each list total is below 2^15)
  int tot;
  const int before = block_exclusive_scan<kMlaThreads>(full | (empty << 16), sWarp, &tot);
  const int n_partial = __syncthreads_count(has);
  const int F = tot & 0xffff, E = tot >> 16;
  const int n_work = (F + n_partial + E) * head_tiles;
  if (cl >= n_work) return n_work;
  const int passes = (n_work + G - 1) / G;
  const bool deal = n_work <= kMlaDealMax && G <= kMlaThreads && passes <= kMlaWorkCache && head_tiles < 16 &&
                    max_parts < 4096 && S <= 32767;
  // The rank of each sequence's partial partition: how many partial partitions are
  // heavier (ties: lower sequence first), counted by `ways` threads per sequence
  // (consecutive lanes), each over a share of the sequences.
  int* sPRank = sLoad;  // [S], free until the list is dealt
  {
    int ways = 1;
    while (ways < 8 && S * ways * 2 <= kMlaThreads) ways *= 2;
    const int s_of = threadIdx.x / ways, part = threadIdx.x & (ways - 1);
    int cnt = 0, rem_s = 0;
    const bool live = s_of < S;
    if (live) rem_s = sRem[s_of];
    // the sequence has a partial partition: any length when unsplit (P <= 0, the whole
    // sequence, possibly empty), else a remainder
    if (live && (P <= 0 || rem_s > 0)) {
      for (int t = part; t < S; t += ways) {
        const int r2 = sRem[t];
        cnt += (r2 > rem_s) || (r2 == rem_s && t < s_of);
      }
    }
    for (int o = ways >> 1; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (live && part == 0) sPRank[s_of] = cnt;
    __syncthreads();
  }
  const int partial_rank = F + (has ? sPRank[sq] : 0);
  for (int q = 0; q < np; ++q) {
    const int rank = q < full ? (before & 0xffff) + q
                     : (q == full && has) ? partial_rank
                                          : F + n_partial + (before >> 16) + (q - full - has);
    const int tokens = q < full ? P : (q == full && has) ? rem : 0;
    for (int ht = 0; ht < head_tiles; ++ht) {
      const int pos = rank * head_tiles + ht;
      if (pos == cl && (blockIdx.x & 1) == 0 && tokens > 0) {
        // The cluster's first work (pass 0): its queries and first pages are cold.
        // Warming L2 with them while the list is dealt lets the query load and the
        // ring's first TMA loads, which start after it, read L2.
        const int rows = min(kMlaRows, p.H - ht * kMlaRows);
        l2_prefetch_bytes(p.q + ((size_t)sq * p.H + ht * kMlaRows) * (kMlaDq / 8), (size_t)rows * kMlaDq * 2);
        // the pages of the ring's first units: their block ids are loaded together (a
        // load, then its prefetch, one page at a time holds every thread of the CTA at
        // the next barrier for a memory round trip per page)
        constexpr int kMaxPages = kMlaStages * kMlaUnit / 16;
        const int t0 = P > 0 ? q * P : 0, t1 = t0 + min(tokens, kMlaStages * kMlaUnit);
        const int pg0 = t0 / p.bs, n_pg = min(min((t1 - 1) / p.bs - pg0 + 1, kMaxPages), p.max_blocks - pg0);
        int bid[kMaxPages];
#pragma unroll
        for (int i = 0; i < kMaxPages; ++i)
          bid[i] = i < n_pg ? __ldg(p.block_table + (size_t)sq * p.max_blocks + pg0 + i) : -1;
#pragma unroll
        for (int i = 0; i < kMaxPages; ++i)
          if (bid[i] >= 0 && bid[i] < p.num_blocks)
            l2_prefetch_bytes(reinterpret_cast<const char*>(p.kv) + (size_t)bid[i] * p.bs * kMlaDq * 2,
                              (size_t)p.bs * kMlaDq * 2);
      }
      if (deal) {
        // clamped: a work that heavy is alone on its cluster anyway, and the sums stay in 32 bits
        sCost[pos] = min((tokens + kMlaUnit - 1) / kMlaUnit, 1 << 20) + kMlaWorkOverheadUnits;
        sWork[pos] = (sq << 16) | (q << 4) | ht;
      } else {
        const int row = pos / G, col = pos - row * G;
        if (((row & 1) ? G - 1 - col : col) == cl) sWorks[row] = make_int4(sq, q, ht, Lr);
      }
    }
  }
  if (!deal) {
    if (threadIdx.x == 0) {
      int n = 0;
      while (mla_work_pos(cl, G, n) < n_work) ++n;
      *n_mine = n;
    }
    return n_work;
  }
  __syncthreads();
  const int c = threadIdx.x;
  if (c < G) sLoad[c] = c < n_work ? sCost[c] : 0;
  if (c == 0) sMine[0] = cl;
  for (int r = 1; r < passes; ++r) {
    __syncthreads();
    if (c < G) {  // place of cluster c in this pass: lighter clusters first
      const int lc = sLoad[c];
      int order = 0, k = 0;
      for (; k + 8 <= G; k += 8) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int lk = sLoad[k + u];
          order += (lk < lc) || (lk == lc && k + u < c);
        }
      }
      for (; k < G; ++k) {
        const int lk = sLoad[k];
        order += (lk < lc) || (lk == lc && k < c);
      }
      sOrder[c] = order;
    }
    __syncthreads();
    if (c < G) {
      const int pos = r * G + sOrder[c];
      if (pos < n_work) sLoad[c] += sCost[pos];
      if (c == cl) sMine[r] = pos < n_work ? pos : -1;
    }
  }
  __syncthreads();
  if (c < passes) {
    const int pos = sMine[c];
    if (pos >= 0) {
      const int wv = sWork[pos], s = wv >> 16;
      sWorks[c] = make_int4(s, (wv >> 4) & 0xfff, wv & 15, sLen[s]);
    }
  }
  // only the last pass can leave a cluster without a position
  if (c == 0) *n_mine = sMine[passes - 1] >= 0 ? passes : passes - 1;
  return n_work;
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
  uint8_t* sSlot = smem + Sh::kSlot;
  uint8_t* sQr = smem + Sh::kQr;
  float* sTagC = reinterpret_cast<float*>(smem + Sh::kTag);          // [2][128]
  float* sTagL = sTagC + 2 * kMlaRows;                                // [2][128]
  float* sRef = reinterpret_cast<float*>(smem + Sh::kRef);           // [2][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::kBars);
  uint64_t* kv_full = bars + MlaBar::kKvFull;    // [stages] TMA landed
  uint64_t* kv_empty = bars + MlaBar::kKvEmpty;  // [stages] P V of the stage's unit completed
  uint64_t* s_full = bars + MlaBar::kSFull;      // [2] partial scores of unit g in S[g & 1]
  uint64_t* s_free = bars + MlaBar::kSFree;      // [2] S[k] has been read (128 arrivals)
  uint64_t* rx_full = bars + MlaBar::kRxFull;    // [2] the peer's partial scores landed in slot k (32 KB of tx)
  uint64_t* tx_ok = bars + MlaBar::kTxOk;        // [2] the peer's slot k is free again (peer's multicast commit)
  uint64_t* p_full = bars + MlaBar::kPFull;      // [2] P, references and row sums of a unit written (128)
  uint64_t* p_go = bars + MlaBar::kPGo;          // [2] the unit's references replayed: P V may run (128)
  uint64_t* pv_done = bars + MlaBar::kPvDone;    // [2] P V of unit g completed, on g & 1
  uint64_t* ref_full = bars + MlaBar::kRefFull;  // [2] set k published R of its unit in sRef[k] (128 arrivals)
  uint64_t* q_full = bars + MlaBar::kQFull;      // Q_r of the next work in TMEM and shared memory (128)
  uint64_t* o_free = bars + MlaBar::kOFree;      // O of a work read out: the next work may overwrite it (128)
  uint64_t* drain = bars + MlaBar::kDrain;        // [2] after an abort: the UMMAs each issuer warp issued completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + MlaBar::kCount);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + MlaBar::kCount + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // == blockIdx.x & 1
  const uint32_t peer = rank ^ 1u;
  const int cl = blockIdx.x >> 1, G = gridDim.x >> 1;
  // The cluster's works, cached in shared memory (every role walks the same list;
  // the units of all works are numbered g = 0, 1, ...).
  int4* sWorks = reinterpret_cast<int4*>(smem + Sh::kWorks);
  // [0] units of the cluster, [1] works, [2] works of the cluster (in-kernel list)
  int* sCount = reinterpret_cast<int*>(bars + MlaBar::kCount + 2);
  if (threadIdx.x == 0) sCount[0] = 0;
  int n_work, n_mine = 0;
  int my_units = 0;
  if (p.inline_list) {
    const int nw = mla_rank_inline(p, reinterpret_cast<int*>(sSlot), sWorks, cl, G, sCount + 2);
    // read back from shared memory: a value the compiler sees as uniform (a
    // per-thread copy would hold a register through every role below)
    if (threadIdx.x == 0) sCount[1] = nw;
    __syncthreads();
    n_work = sCount[1];
    if (cl >= n_work) return;  // both CTAs of the cluster take the same branch
    n_mine = sCount[2];
    for (int r = threadIdx.x; r < n_mine; r += kMlaThreads) my_units += mla_work_decode(p, sWorks[r]).n_units;
  } else {
    n_work = *p.item_count * p.head_tiles;
    if (cl >= n_work) return;  // both CTAs of the cluster take the same branch
    __syncthreads();
    for (int r = threadIdx.x; r < kMlaWorkCache; r += kMlaThreads) {
      const long long pos = mla_work_pos(cl, G, r);
      if (pos >= n_work) break;
      const int4 raw = mla_work_raw(p, pos);
      sWorks[r] = raw;
      my_units += mla_work_decode(p, raw).n_units;
    }
  }
  if (my_units) atomicAdd(sCount, my_units);
  __syncthreads();
  int g_total = sCount[0];
  if (!p.inline_list)
    for (int r = kMlaWorkCache;; ++r) {  // works past the cache (very long lists only)
      const long long pos = mla_work_pos(cl, G, r);
      if (pos >= n_work) break;
      g_total += mla_work_decode(p, mla_work_raw(p, pos)).n_units;
    }
  // the cluster's r-th work; false past the end
  auto mla_work = [&](const MlaParams&, int, int, int, int r, MlaWork& w) -> bool {
    if (p.inline_list) {
      if (r >= n_mine) return false;
      w = mla_work_decode(p, sWorks[r]);
      return true;
    }
    const long long pos = mla_work_pos(cl, G, r);
    if (pos >= n_work) return false;
    w = mla_work_decode(p, r < kMlaWorkCache ? sWorks[r] : mla_work_raw(p, pos));
    return true;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < MlaBar::kCount; ++i) mbar_init(&bars[i], MlaBar::arrivals(i));
    *abort_flag = 0;
    // the first unit of each set: expect the peer's 32 KB of partial scores
    for (int k = 0; k < 2; ++k)
      if (k < g_total) mbar_arrive_expect_tx(&rx_full[k], Sh::kSlotB);
    fence_barrier_init();
  }
  if (warp == 13) {
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

  // Q_r of head row hr (lane of quarter q) in work w: latent dims 256 r .. 256 r + 255
  // into TMEM columns kTmQ.. as bf16 pairs (the raw row words), rope dims
  // 512 + 32 r .. + 31 into row hr of the 64-byte-swizzled shared tile (chunk c at
  // c ^ ((row >> 1) & 3)).  Run by a warpgroup (all four lane quarters); arrives on q_full.
  auto q_row = [&](const MlaWork& w, int hr, bool& valid) -> const uint4* {
    const int head = w.ht * kMlaRows + hr;
    valid = hr < p.hrows && head < p.H;
    return p.q + ((size_t)w.s * p.H + (valid ? head : 0)) * (kMlaDq / 8);
  };
  auto load_q = [&](const MlaWork& w, int quarter) {
    const int hr = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    bool row_valid;
    const uint4* src = q_row(w, hr, row_valid);
    for (int c0 = 0; c0 < 128; c0 += 64) {  // two passes of 256 B of the row's latent half (rope last)
      uint32_t v[64];
      if (p.q_v8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (row_valid)
            ld_global_nc_v8(src + 32 * rank + c0 / 4 + 2 * i, v + 8 * i);
          else
#pragma unroll
            for (int k = 0; k < 8; ++k) v[8 * i + k] = 0u;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint4 x4 = row_valid ? __ldg(src + 32 * rank + c0 / 4 + i) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * i] = x4.x, v[4 * i + 1] = x4.y, v[4 * i + 2] = x4.z, v[4 * i + 3] = x4.w;
        }
      }
      tmem_st32(lane_base + kTmQ + c0, v);
      tmem_st32(lane_base + kTmQ + c0 + 32, v + 32);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 x4 = row_valid ? __ldg(src + kMlaDv / 8 + 4 * rank + c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sQr + hr * 64 + ((c ^ ((hr >> 1) & 3)) << 4)) = x4;
    }
    fence_proxy_async_smem();  // the score UMMA reads the rope tile through the async proxy
    tmem_st_wait();
    tc_fence_before_sync();
    mbar_arrive(q_full);
  };
  // warm L2 with a work's query row (its 576 B in this CTA's half: 256 latent + 32 rope dims)
  auto prefetch_q = [&](const MlaWork& w, int hr) {
    bool row_valid;
    const uint4* src = q_row(w, hr, row_valid);
    if (!row_valid) return;
#pragma unroll
    for (int c = 0; c < 4; ++c) prefetch_l2(src + 32 * rank + 8 * c);
    prefetch_l2(src + kMlaDv / 8 + 4 * rank);
  };
  // the next non-empty work at or after list position r (false: none)
  auto next_nonempty = [&](int r, MlaWork& w) -> bool {
    for (; mla_work(p, n_work, cl, G, r, w); ++r)
      if (w.n_units > 0) return true;
    return false;
  };

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    regs_dec<kMlaRegsLow>();
    // Per unit and page piece (R rows: the block size, at most 64, or at most 32
    // when partitions start on odd multiples of 32 tokens, so a piece never crosses
    // a page): lanes 5 pi + 0..3 load the latent blocks 4 r .. 4 r + 3, lane 5 pi + 4
    // the rope half block 512 + 32 r .. + 31.
    if (lane == 0) {
      tma_prefetch_desc(&tmKV);
      tma_prefetch_desc(&tmKVh);
    }
    const int R = p.box_rows;
    const int pieces = kMlaUnit / R;
    const int pi = lane / 5, lb = lane - pi * 5;
    const uint64_t pol = l2_policy_evict_first();
    int g = 0;
    bool ok = true;
    MlaWork w;
    for (int r = 0; ok && mla_work(p, n_work, cl, G, r, w); ++r) {
      const int32_t* bt_row = p.block_table + (size_t)w.s * p.max_blocks;
      for (int u = 0; u < w.n_units; ++u, ++g) {
        const int st = g % kMlaStages;
        const int tok = w.t0 + u * kMlaUnit + pi * R;
        const bool live = pi < pieces && tok < w.t1;
        int rowc = 0;
        if (live) {
          const int pg = tok / p.bs;
          const int b = checked_block(bt_row, pg, p.num_blocks, &g_status_mla);
          rowc = b < 0 ? -R : b * p.bs + (tok - pg * p.bs);
        }
        const uint32_t n_live = (uint32_t)__popc(__ballot_sync(0xffffffffu, live && lb == 0));
        if (g >= kMlaStages && !wait_all(&kv_empty[st], ((g / kMlaStages) - 1) & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&kv_full[st], n_live * (uint32_t)(R * (4 * 128 + 64)));
        __syncwarp();
        if (live) {
          if (lb < 4)
            tma_load_3d(sKV + st * Sh::kStage + lb * Sh::kBlk + pi * R * 128, &tmKV, &kv_full[st],
                        (4 * (int)rank + lb) * 64, 0, rowc, pol);
          else
            tma_load_3d(sRope + st * Sh::kRopeU + pi * R * 64, &tmKVh, &kv_full[st], kMlaDv + 32 * (int)rank, 0,
                        rowc, pol);
        }
      }
    }
    // after an abort, let the copies already on their way land before the CTA exits
    if (*abort_flag)
      for (int v = max(0, g - kMlaStages); v < g; ++v)
        mbar_wait(&kv_full[v % kMlaStages], (v / kMlaStages) & 1, &g_status_mla);
  } else if (warp == 13 || warp == 14) {
    // ------------------------------------------------------------ UMMA issuers
    // Warp 13 issues the score UMMAs, warp 14 the P V UMMAs, each blocking on its own
    // next barrier (the two streams touch disjoint TMEM: S buffers, O).
    regs_dec<kMlaRegsLow>();
    constexpr uint32_t kIdQK = umma_idesc_bf16_f32(kMlaRows, kMlaUnit, false, false);
    constexpr uint32_t kIdPV = umma_idesc_bf16_f32(kMlaRows, kMlaHalf, false, true);
    const uint32_t kv = smem_u32(sKV), rope = smem_u32(sRope), qr = smem_u32(sQr), slot = smem_u32(sSlot);
    const uint16_t peer_mask = (uint16_t)(1u << peer);
    const bool scores = warp == 13;
    bool issued = false, ok = true;
    int g = 0, qi = 0;  // global unit, non-empty works before the current one
    MlaWork w;
    for (int r = 0; ok && mla_work(p, n_work, cl, G, r, w); ++r) {
      if (w.n_units == 0) continue;
      for (int u = 0; u < w.n_units; ++u, ++g) {
        const int k = g & 1;
        const int st = g % kMlaStages;
        if (scores) {
          // partial S of unit g into S[k] over this CTA's 288 key dimensions, once the
          // work's Q is in place, the set owning S[k] has read its previous unit and
          // the latent has landed
          if ((g >= 2 && !wait_all(&s_free[k], ((g - 2) >> 1) & 1)) || (u == 0 && !wait_all(q_full, qi & 1)) ||
              !wait_all(&kv_full[st], (g / kMlaStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (lane == 0) {
            const uint32_t d_tmem = tmem + kTmS + k * kMlaUnit;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
              umma_bf16_tmem_a(d_tmem, tmem + kTmQ + kk * 8,
                               umma_desc_sw128(kv + st * Sh::kStage + (kk >> 2) * Sh::kBlk + (kk & 3) * 32, 16, 1024),
                               kIdQK, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk)
              umma_bf16(d_tmem, umma_desc_sw64(qr + kk * 32, 512),
                        umma_desc_sw64(rope + st * Sh::kRopeU + kk * 32, 512), kIdQK, 1u);
            umma_commit(&s_full[k]);
          }
          __syncwarp();
          issued = true;
        } else {
          // O_r (+)= P V of unit g, once its references are replayed (and, for a work's
          // first unit, once the previous work's O has been read out)
          if (!wait_all(&p_go[k], (g >> 1) & 1) || (u == 0 && qi > 0 && !wait_all(o_free, (qi - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const int tok0 = w.t0 + u * kMlaUnit;
          if (tok0 + kMlaUnit > w.t1) {
            // value rows past the work's end (cache tails, pieces not loaded): zero them,
            // since 0 * NaN would reach O (their scores are masked already)
            for (int row = (w.t1 - tok0) + lane; row < kMlaUnit; row += 32)
              for (int b = 0; b < 4; ++b) {
                uint4* d = reinterpret_cast<uint4*>(sKV + st * Sh::kStage + b * Sh::kBlk + row * 128);
#pragma unroll
                for (int q = 0; q < 8; ++q) d[q] = make_uint4(0u, 0u, 0u, 0u);
              }
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (lane == 0) {
            const uint32_t pt = slot + k * Sh::kSlotB;
#pragma unroll
            for (int kk = 0; kk < kMlaUnit / 16; ++kk)
              umma_bf16(tmem + kTmO, umma_desc_sw128(pt + kk * 32, 16, Sh::kPGroup),
                        umma_desc_sw128(kv + st * Sh::kStage + kk * 16 * 128, Sh::kBlk, 1024), kIdPV,
                        (u > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&kv_empty[st]);
            umma_commit(&pv_done[k]);
            // the slot of this unit is free again: the peer may send its partial of unit g + 2
            if (g + 2 < g_total) umma_commit_multicast(&tx_ok[k], peer_mask);
          }
          __syncwarp();
          issued = true;
        }
      }
      ++qi;
    }
    if (!ok && issued) {
      uint64_t* d = drain + (scores ? 0 : 1);
      if (lane == 0) umma_commit(d);
      __syncwarp();
      mbar_wait(d, 0, &g_status_mla);
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------ rescale warps
    regs_dec<kMlaRegsLow>();
    const int quarter = warp - 8;
    const int hr = quarter * 32 + lane;  // head row of this lane = its TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    // Q_r of this lane's head in work w: latent dims 256 r .. 256 r + 255 into TMEM
    // columns kTmQ.. as bf16 pairs (the raw row words), rope dims 512 + 32 r .. + 31
    // into row hr of the 64-byte-swizzled shared tile (chunk c at c ^ ((row >> 1) & 3)).
    bool ok = true;
    int g = 0;
    int qi = 0;  // non-empty works completed
    {
      MlaWork w0;
      if (next_nonempty(0, w0)) load_q(w0, quarter);  // later works: loaded by a row-warp set
    }
    MlaWork w;
    for (int r = 0; ok && mla_work(p, n_work, cl, G, r, w); ++r) {
      const int head = w.ht * kMlaRows + hr;
      const bool row_valid = hr < p.hrows && head < p.H;
      const size_t sh = (size_t)w.s * p.H + head;
      if (w.L_raw > p.cap && rank == 0 && w.ht == 0 && w.part == 0 && hr == 0)
        atomicOr(&g_status_mla, METIS_STATUS_SEQ_TOO_LONG);
      if (w.n_units == 0) {
        // nothing readable: an empty sequence gets 0 / -inf, an empty partition lse = -inf
        if (row_valid) {
          if (w.direct) {
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + sh * kMlaDv + rank * kMlaHalf;
            for (int c = 0; c < kMlaHalf; c += 8) *reinterpret_cast<uint4*>(o + c) = make_uint4(0u, 0u, 0u, 0u);
            if (rank == 0 && p.lse_out) p.lse_out[sh] = -INFINITY;
          } else if (rank == 0) {
            p.part_lse[sh * p.max_parts + w.part] = -INFINITY;
          }
        }
        continue;
      }
      MlaWork w2;
      if (next_nonempty(r + 1, w2)) prefetch_q(w2, hr);
      float C = -INFINITY, Lsum = 0.f;
      for (int u = 0; ok && u < w.n_units; ++u, ++g) {
        const int k = g & 1;
        if (!wait_all(&p_full[k], (g >> 1) & 1)) {
          ok = false;
          break;
        }
        const float c = sTagC[k * kMlaRows + hr];
        const float l = sTagL[k * kMlaRows + hr];
        float fo = 1.f;
        if (u == 0) {
          C = c;
          Lsum = l;
        } else if (c > C) {
          fo = exp2_approx(C - c);
          Lsum = fmaf(Lsum, fo, l);
          C = c;
        } else if (c < C) {
          // this unit exponentiated against a smaller reference: bring its P down to C
          const float gsc = exp2_approx(c - C);
          uint8_t* prow = sSlot + k * Sh::kSlotB + (hr >> 3) * Sh::kPGroup + (hr & 7) * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4* q4 = reinterpret_cast<uint4*>(prow + (j << 4));
            uint4 v = *q4;
            uint32_t* wv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&wv[i]));
              wv[i] = pack_bf16x2(f.x * gsc, f.y * gsc);
            }
            *q4 = v;
          }
          fence_proxy_async_smem();  // P V reads P through the async proxy
          Lsum = fmaf(l, gsc, Lsum);
        } else {
          Lsum += l;
        }
        if (__any_sync(0xffffffffu, fo != 1.f)) {
          // O holds every earlier unit of the work once P V of unit g - 1 completed
          if (!wait_all(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll 1
          for (int c32 = 0; c32 < kMlaHalf / 32; ++c32) {
            uint32_t ov[32];
            tmem_ld32(lane_base + kTmO + c32 * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * fo);
            tmem_st32(lane_base + kTmO + c32 * 32, ov);
          }
          tmem_st_wait();
        }
        tc_fence_before_sync();
        mbar_arrive(&p_go[k]);
      }
      if (!ok) break;
      // epilogue: O_r / l and the lse, once the work's last P V completed
      if (!wait_all(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float inv = 1.0f / Lsum;
      // Each thread holds its own row; a 4 x 4 transpose of 32-byte chunks inside each
      // group of four lanes lets a warp store write 8 rows x 128 contiguous bytes
      // (instead of 32 rows x 32 bytes).  Lane 4 q + i then holds chunk i of rows
      // 4 q .. 4 q + 3 of its warp's 32.
      const int gq = lane >> 2, gi = lane & 3;
      auto transpose4 = [&](uint32_t* wv, const int cw) {  // chunks of cw words (8 or 4)
        const int b0 = lane & 1, b1 = (lane >> 1) & 1;
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (k >= cw) break;
            const uint32_t x = b0 ? wv[cw * (2 * sl) + k] : wv[cw * (2 * sl + 1) + k];
            const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 1);
            if (b0)
              wv[cw * (2 * sl) + k] = y;
            else
              wv[cw * (2 * sl + 1) + k] = y;
          }
#pragma unroll
        for (int sl = 0; sl < 2; ++sl)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (k >= cw) break;
            const uint32_t x = b1 ? wv[cw * sl + k] : wv[cw * (2 + sl) + k];
            const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 2);
            if (b1)
              wv[cw * sl + k] = y;
            else
              wv[cw * (2 + sl) + k] = y;
          }
      };
      // O leaves TMEM a block at a time: once a block is converted into wv, the next
      // block's TMEM load is issued into the freed registers and stays in flight
      // while wv is transposed and stored
      if (w.direct) {
        // 32 bf16 columns (64 B) per row and block: 16-byte chunks, so a warp store
        // writes 8 rows x 64 contiguous bytes
        uint32_t ov[32], wv[16];
        tmem_ld32(lane_base + kTmO, ov);
#pragma unroll 1
        for (int c32 = 0; c32 < kMlaHalf / 32; ++c32) {
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            wv[j] = pack_bf16x2(__uint_as_float(ov[2 * j]) * inv, __uint_as_float(ov[2 * j + 1]) * inv);
          if (c32 + 1 < kMlaHalf / 32) tmem_ld32(lane_base + kTmO + (c32 + 1) * 32, ov);
          transpose4(wv, 4);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int rr = quarter * 32 + 4 * gq + c;  // the row this lane writes a chunk of
            const int hd = w.ht * kMlaRows + rr;
            if (rr < p.hrows && hd < p.H)
              *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)w.s * p.H + hd) * kMlaDv +
                                        rank * kMlaHalf + c32 * 32 + gi * 8) =
                  make_uint4(wv[4 * c], wv[4 * c + 1], wv[4 * c + 2], wv[4 * c + 3]);
          }
        }
      } else {
        // 32 fp32 columns (128 B) per row and block
        uint32_t ov[32], wv[32];
        tmem_ld32(lane_base + kTmO, ov);
#pragma unroll 1
        for (int c32 = 0; c32 < kMlaHalf / 32; ++c32) {
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) wv[j] = __float_as_uint(__uint_as_float(ov[j]) * inv);
          if (c32 + 1 < kMlaHalf / 32) tmem_ld32(lane_base + kTmO + (c32 + 1) * 32, ov);
          transpose4(wv, 8);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int rr = quarter * 32 + 4 * gq + c;
            const int hd = w.ht * kMlaRows + rr;
            if (rr < p.hrows && hd < p.H)
              st_global_v8(p.part_out + (((size_t)w.s * p.H + hd) * p.max_parts + w.part) * kMlaDv + rank * kMlaHalf +
                               c32 * 32 + gi * 8,
                           wv + 8 * c);
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(o_free);  // the next work's first P V may overwrite O
      ++qi;
      if (row_valid && rank == 0) {
        const float lse = (C + log2f(Lsum)) * kLn2;
        if (w.direct) {
          if (p.lse_out) p.lse_out[sh] = lse;
        } else {
          p.part_lse[sh * p.max_parts + w.part] = lse;
        }
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ row warps
    regs_inc<kMlaRegsRow>();
    const int set = warp >> 2;
    const int quarter = warp & 3;
    const int hr = quarter * 32 + lane;  // head row of this lane = its TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* my_slot = sSlot + set * Sh::kSlotB;
    // scores of this lane: chunk j at j * 512 + lane * 16 within the warp's part
    const uint32_t peer_part = dsmem_map(smem_u32(my_slot), peer) + quarter * Sh::kWarpB + lane * 16;
    const uint8_t* rx_part = my_slot + quarter * Sh::kWarpB + lane * 16;
    const uint32_t peer_rx_full = dsmem_map(smem_u32(&rx_full[set]), peer);
    uint8_t* prow = my_slot + (hr >> 3) * Sh::kPGroup + (hr & 7) * 128;   // inside this warp's part
    const int sw8 = hr & 7;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g0 = 0;  // first unit of the current work
    MlaWork w;
    for (int r = 0; ok && mla_work(p, n_work, cl, G, r, w); g0 += w.n_units, ++r) {
      float c_prev = -INFINITY;  // c_{u-2}: this set's reference of its previous unit of the work
      const int u_first = (set - g0) & 1;  // this set takes the units with g = g0 + u of its parity
      for (int u = u_first; u < w.n_units; u += 2) {
        const int g = g0 + u;
        const uint32_t ph = (g >> 1) & 1;
        // R_{u-2} = max(R_{u-3}, c_{u-2}) within the work; R_{u-3} comes from the other
        // set, which published a value as it started unit g - 1 (every unit publishes,
        // so the hand-over is the same at work boundaries).  Publish R_{u-2}.
        float r3 = -INFINITY;
        if (g >= 1) {
          if (!wait_all(&ref_full[(g - 1) & 1], ((g - 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          r3 = sRef[((g - 1) & 1) * kMlaRows + hr];
        }
        const float base = u >= 2 ? fmaxf(u >= 3 ? r3 : -INFINITY, c_prev) : -INFINITY;
        sRef[set * kMlaRows + hr] = base;
        mbar_arrive(&ref_full[set]);
        // this CTA's partial scores of the unit
        if (!wait_all(&s_full[set], ph)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t sv[kMlaUnit];
        tmem_ld32(lane_base + kTmS + set * kMlaUnit, sv);
        tmem_ld32(lane_base + kTmS + set * kMlaUnit + 32, sv + 32);
        tmem_ld_wait();
        tc_fence_before_sync();
        mbar_arrive(&s_free[set]);
        // ... into the peer's slot (free again once the peer's P V of unit g - 2 completed)
        if (g >= 2 && !wait_all(&tx_ok[set], ((g >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        // this CTA's partial in the log2 domain, rounded to fp16 (saturating): what
        // travels, and what this CTA adds, so that both CTAs hold the same sums
        uint32_t hv[kMlaUnit / 2];
#pragma unroll
        for (int j = 0; j < kMlaUnit / 2; ++j)
          hv[j] = pack_f16x2_sat(__uint_as_float(sv[2 * j]) * sl2, __uint_as_float(sv[2 * j + 1]) * sl2);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          st_async_v4(peer_part + j * 512, hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3], peer_rx_full);
        // the peer's partial of the same unit, in this CTA's slot
        if (!wait_all(&rx_full[set], ph)) {
          ok = false;
          break;
        }
        // expect the peer's partial of this set's next unit (it can only come after
        // this unit's P V, which follows everything below)
        if (quarter == 0 && lane == 0 && g + 2 < g_total) mbar_arrive_expect_tx(&rx_full[set], Sh::kSlotB);
        // full scores in the log2 domain: x = own + peer (fp32 sum of the fp16 partials)
        float x[kMlaUnit];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 r4 = *reinterpret_cast<const uint4*>(rx_part + j * 512);
          const uint32_t rw[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 a = unpack_f16x2(hv[4 * j + i]);
            const float2 b = unpack_f16x2(rw[i]);
            f2_unpack(f2_add(f2_pack(a.x, a.y), f2_pack(b.x, b.y)), x[8 * j + 2 * i], x[8 * j + 2 * i + 1]);
          }
        }
        __syncwarp();  // the warp's scores are read before its P overwrites them
        const int vis = min(kMlaUnit, w.t1 - (w.t0 + u * kMlaUnit));
        if (vis < kMlaUnit) {
#pragma unroll
          for (int i = 0; i < kMlaUnit; ++i) x[i] = i < vis ? x[i] : -INFINITY;
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < kMlaUnit; i += 8) {
          m4[0] = max3f(m4[0], x[i], x[i + 1]);
          m4[1] = max3f(m4[1], x[i + 2], x[i + 3]);
          m4[2] = max3f(m4[2], x[i + 4], x[i + 5]);
          m4[3] = max3f(m4[3], x[i + 6], x[i + 7]);
        }
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float c = mx <= base + kMlaSlack ? base : mx;  // the unit's maximum also when base = -inf
        c_prev = c;
        const uint64_t negc = f2_pack(-c, -c);
        uint64_t l2[2] = {0ull, 0ull};
        uint32_t pk[kMlaUnit / 2];
#pragma unroll
        for (int i = 0; i < kMlaUnit; i += 2) {
          float d0, d1;
          f2_unpack(f2_add(f2_pack(x[i], x[i + 1]), negc), d0, d1);
          const float e0 = exp2_approx(d0);
          const float e1 = exp2_approx(d1);
          l2[(i >> 1) & 1] = f2_add(l2[(i >> 1) & 1], f2_pack(e0, e1));
          pk[i >> 1] = pack_bf16x2(e0, e1);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(prow + ((j ^ sw8) << 4)) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                                                                          pk[4 * j + 3]);
        float la, lb, lc, ld;
        f2_unpack(l2[0], la, lb);
        f2_unpack(l2[1], lc, ld);
        sTagC[set * kMlaRows + hr] = c;
        sTagL[set * kMlaRows + hr] = (la + lb) + (lc + ld);
        fence_proxy_async_smem();  // P V reads P through the async proxy
        mbar_arrive(&p_full[set]);
      }
      if (!ok) break;
      // The set that does not take the work's last unit would next wait for scores that
      // need the next work's Q: it loads that Q, as soon as the work's last score UMMA
      // (the last reader of the current Q) has completed.
      const int g_last = g0 + w.n_units - 1;
      MlaWork w2;
      if (w.n_units > 0 && ((g_last & 1) ^ 1) == set && next_nonempty(r + 1, w2)) {
        if (!wait_all(&s_full[g_last & 1], (g_last >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        load_q(w2, quarter);
      }
    }
  } else {
    regs_dec<kMlaRegsLow>();  // warp 15: no role
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 13) {
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
  if (partition_size < 0 || partition_size % kMlaAlign)
    return fail(METIS_E_SHAPE, "partition_size must be 0 or a positive multiple of 32");
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 32) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4) || !aligned(lse_out, 4))
    return fail(METIS_E_ALIGN, "q and kv_cache must be 16-byte aligned, out 32-byte, index arrays and lse_out 4-byte");
  if (!(scale == scale)) return fail(METIS_E_SHAPE, "scale is NaN");
  const MlaWorkspace lay = mla_workspace_layout(num_seqs, num_heads, max_seq_len, partition_size);
  if (!workspace || workspace_bytes < lay.total || !aligned(workspace, 256))
    return fail(METIS_E_WORKSPACE, "workspace must hold %zu bytes (256-byte aligned)", lay.total);
  const int head_tiles = (num_heads + kMlaRows - 1) / kMlaRows;
  if (lay.max_items * head_tiles * 2 > 0x7fffffffull) return fail(METIS_E_SHAPE, "too many work items");

  MlaParams p{};
  p.q = reinterpret_cast<const uint4*>(q);
  p.kv = kv_cache;
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

  // 64-row boxes (fewer, larger TMA copies) when every unit starts on a multiple of 64 tokens
  p.box_rows = std::min(block_size, (partition_size % kMlaUnit == 0) ? kMlaUnit : kMlaAlign);
  p.q_v8 = aligned(q, 32);
  CUtensorMap tmKV, tmKVh;
  const uint64_t kdims[3] = {(uint64_t)kMlaDq, 1, (uint64_t)num_blocks * block_size};
  const uint64_t kstr[2] = {(uint64_t)kMlaDq * 2, (uint64_t)kMlaDq * 2};
  const uint32_t kbox[3] = {64, 1, (uint32_t)p.box_rows};
  int rc = encode_tiled(&tmKV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_cache, kdims, kstr, kbox,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint32_t khbox[3] = {32, 1, (uint32_t)p.box_rows};
  rc = encode_tiled(&tmKVh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_cache, kdims, kstr, khbox,
                    CU_TENSOR_MAP_SWIZZLE_64B);
  if (rc) return rc;

  // persistent: one cluster (two SMs) per SM pair, each walking its share of the work list
  int dev = 0, sms = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return fail(METIS_E_CUDA, "SM count: %s", cudaGetErrorString(ce));
  const size_t clusters = std::max<size_t>(1, std::min<size_t>((size_t)(sms / 2), lay.max_items * head_tiles));
  // Small batches: every CTA ranks its own works (no schedule kernel on the critical
  // path); otherwise a schedule kernel lists them, heaviest first.
  p.inline_list = num_seqs <= kMlaInlineSeqs && lay.max_items < 32768 &&
                  lay.max_items * head_tiles <= (size_t)kMlaWorkCache * clusters;
  if (!p.inline_list) {
    // a programmatic dependent of the kernel before it (e.g. the latent-cache write)
    rc = launch_dependent(mla_schedule_kernel, dim3(1), dim3(1024), 0, st, "mla_schedule_kernel launch", p, items,
                          count, (int)lay.max_items);
    if (rc) return rc;
  }
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
  rc = launch_dependent(mla_decode_kernel, dim3((unsigned)(clusters * 2)), dim3(kMlaThreads), MlaShape::kSmem, st,
                        "mla_decode_kernel launch", tmKV, tmKVh, p);
  if (rc) return rc;
  if (partition_size > 0 && lay.max_parts > 1)
    rc = launch_merge_split_rows(p.part_out, p.part_lse, seq_lens, partition_size, out, lse_out, num_seqs, num_heads,
                                 kMlaDv, lay.max_parts, METIS_BF16, sms, st);
  return rc;
}
