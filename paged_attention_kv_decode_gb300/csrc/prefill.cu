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
// Tiling.  One CTA computes a 128-row query tile of one KV head's group: the
// r = H/G query heads of the group times 128/r consecutive query tokens
// (GQA packing, so every K/V tile is read once for the whole group), against
// 128-token K/V tiles gathered page by page with TMA (128-byte swizzle).
//
//   warp 4       TMA producer: Q tile once, then K and V tiles into 2-stage rings
//   warp 5       allocates TMEM; one lane issues the UMMAs:
//                  S_j = Q K_j^T   (M 128, N 128, K = head_dim)  -> TMEM, double-buffered
//                  O  += P_j V_j   (M 128, N head_dim, K 128)     -> TMEM
//   warps 0..3   softmax, one TMEM lane (= one query row) per thread: mask,
//                running max in log2 units, rescale O in TMEM only when the
//                max grows by more than 2^8, P = exp2(S - m) as bf16 into a
//                swizzled shared-memory tile for the PV UMMA; epilogue O / l.
//
// A small schedule kernel first lists the (sequence, query tile) pairs with
// work, heaviest first, so the main grid has no idle CTAs.
#include <math.h>

#include <algorithm>

#include "../../include/metis_attn.h"
#include "common.cuh"
#include "host.h"
#include "tcgen05.cuh"

namespace metis {

__device__ unsigned int g_status_prefill = 0;

constexpr int kPfThreads = 192;   // 4 softmax warps + TMA warp + MMA warp
constexpr int kKvTile = 64;       // tokens per K/V tile
constexpr int kRows = 128;        // query rows per tile
constexpr int kTmemCols = 256;    // S0 | S1 | O: two CTAs share an SM's 512 columns
constexpr int kSortMax = 2048;    // schedule: heaviest-first sort up to this many tiles

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
  static constexpr int kQBytes = kHalves * kQHalf;
  static constexpr int kKvHalf = kKvTile * 128;                // 64 tokens x 64 bf16
  static constexpr int kKvBytes = kHalves * kKvHalf;
  static constexpr int kPBytes = kRows * kKvTile * 2;          // P: 128 rows x 64 tokens (one half)
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;                      // 2 stages
  static constexpr int kV = kK + 2 * kKvBytes;                 // 2 stages
  static constexpr int kP = kV + 2 * kKvBytes;
  static constexpr int kTiles = kP + kPBytes;                  // 112 KB at head_dim 128
  // + 1 KB: the barriers live in the alignment slack (below the aligned base when
  // it is at least 256 B, else just past the tiles).  At least 80 KB, so that at
  // most two CTAs -- 2 x 256 TMEM columns -- are resident per SM.
  static constexpr int kSmem = (kTiles + 1024) > 80 * 1024 ? (kTiles + 1024) : 80 * 1024;
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

// ---------------------------------------------------------------------------
// schedule: the (sequence, query tile) work list, heaviest first
// ---------------------------------------------------------------------------
constexpr int kSchedThreads = 1024;

__global__ void __launch_bounds__(kSchedThreads) prefill_schedule_kernel(const PrefillParams p, int4* items,
                                                                          int* count, int max_items) {
  __shared__ int scan[kSchedThreads];
  __shared__ int4 buf[kSortMax];
  const int tid = threadIdx.x;
  const int per = (p.S + kSchedThreads - 1) / kSchedThreads;
  const int s0 = min(p.S, tid * per), s1 = min(p.S, s0 + per);
  int local = 0;
  for (int s = s0; s < s1; ++s) {
    int L, q_len;
    pf_lengths(p, s, L, q_len, false);
    local += (q_len + p.Tq - 1) / p.Tq;
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
    const int nt = (q_len + p.Tq - 1) / p.Tq;
    for (int t = 0; t < nt; ++t, ++pos) {
      if (pos >= total) break;
      const int p_max = L - q_len + min(q_len - 1, t * p.Tq + p.Tq - 1);
      const int4 it = make_int4(s, t, (p_max + kKvTile) / kKvTile, 0);
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
__global__ void __launch_bounds__(kPfThreads, 2) prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                       const __grid_constant__ CUtensorMap tmK,
                                                                       const __grid_constant__ CUtensorMap tmV,
                                                                       const PrefillParams p) {
  using Sh = PfShape<D>;
  constexpr int HALVES = Sh::kHalves;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t slack = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + slack;
  uint8_t* sQ = smem + Sh::kQ;
  uint8_t* sK = smem + Sh::kK;
  uint8_t* sV = smem + Sh::kV;
  uint8_t* sP = smem + Sh::kP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(slack >= 256 ? smem - 256 : smem + Sh::kTiles);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;   // [2]
  uint64_t* v_empty = bars + 7;  // [2]
  uint64_t* s_full = bars + 9;   // [2]
  uint64_t* p_full = bars + 11;
  uint64_t* pv_done = bars + 12;
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 15);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item_idx = blockIdx.x / p.G, g = blockIdx.x - item_idx * p.G;
  if (item_idx >= *p.item_count) return;
  const int4 it = p.items[item_idx];
  const int s = it.x, tile = it.y;
  int L, q_len;
  pf_lengths(p, s, L, q_len, threadIdx.x == 0);
  const int qi0 = tile * p.Tq;
  if (q_len <= 0 || qi0 >= q_len) return;
  const int q0 = p.cu_q_lens[s];
  const int valid_tokens = min(p.Tq, q_len - qi0);
  const int p_min = L - q_len + qi0;             // position of the tile's first query token
  const int p_max = p_min + valid_tokens - 1;    // ... and of its last valid one
  const int n_kv = (p_max + kKvTile) / kKvTile;
  const int n_pages = (L + p.bs - 1) / p.bs;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 14; ++i) mbar_init(&bars[i], i == 11 ? 128 : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
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

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    const int32_t* bt_row = p.block_table + (size_t)s * p.max_blocks;
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, Sh::kQBytes);
      const uint64_t pol = l2_policy_evict_first();
      for (int hh = 0; hh < p.r; ++hh)
        for (int h = 0; h < HALVES; ++h)
          tma_load_3d(sQ + h * Sh::kQHalf + hh * p.Tq * 128, &tmQ, q_full, h * 64, g * p.r + hh, q0 + qi0, pol);
    }
    const int npg = kKvTile / p.bs;  // pages per K/V tile
    const uint64_t pol = l2_policy_evict_last();
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      const int pg = j * npg + lane;
      const bool live = lane < npg && pg < n_pages;
      int rowc = 0;
      if (live) {
        const int b = checked_block(bt_row, pg, p.num_blocks, &g_status_prefill);
        rowc = b < 0 ? -p.bs : b * p.bs;   // a bad id reads a box entirely out of bounds: zeros
      }
      const uint32_t bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, live)) * p.bs * 128 * HALVES;
      if (j >= 2 && !wait_all(&k_empty[st], ((j >> 1) - 1) & 1)) break;
      if (lane == 0) mbar_arrive_expect_tx(&k_full[st], bytes);
      __syncwarp();
      if (live)
        for (int h = 0; h < HALVES; ++h)
          tma_load_3d(sK + st * Sh::kKvBytes + h * Sh::kKvHalf + lane * p.bs * 128, &tmK, &k_full[st], h * 64, g,
                      rowc, pol);
      if (j >= 2 && !wait_all(&v_empty[st], ((j >> 1) - 1) & 1)) break;
      if (lane == 0) mbar_arrive_expect_tx(&v_full[st], bytes);
      __syncwarp();
      if (live)
        for (int h = 0; h < HALVES; ++h)
          tma_load_3d(sV + st * Sh::kKvBytes + h * Sh::kKvHalf + lane * p.bs * 128, &tmV, &v_full[st], h * 64, g,
                      rowc, pol);
    }
    if (*abort_flag) {
      // let the loads of the last two tiles land before the CTA's memory goes away
      for (int j = max(0, n_kv - 2); j < n_kv; ++j) {
        mbar_wait(&k_full[j & 1], (j >> 1) & 1, &g_status_prefill);
        mbar_wait(&v_full[j & 1], (j >> 1) & 1, &g_status_prefill);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ UMMA issuer
    constexpr uint32_t kIdQK = umma_idesc_bf16_f32(kRows, kKvTile, false, false);
    constexpr uint32_t kIdPV = umma_idesc_bf16_f32(kRows, D, false, true);
    const uint32_t o_tmem = tmem + 2 * kKvTile;
    bool issued = false;
    auto do_pv = [&](int i) -> bool {
      const int st = i & 1;
      if (!wait_all(p_full, i & 1)) return false;
      if (!wait_all(&v_full[st], (i >> 1) & 1)) return false;
      tc_fence_after_sync();
      const int tok0 = i * kKvTile;
      if (tok0 + kKvTile > L) {
        // rows past the sequence end may hold anything (NaN included): zero them so that P = 0 stays 0
        const int first = L - tok0;
        uint8_t* vb = sV + st * Sh::kKvBytes;
        for (int row = first + lane; row < kKvTile; row += 32)
          for (int h = 0; h < HALVES; ++h) {
            uint4* d = reinterpret_cast<uint4*>(vb + h * Sh::kKvHalf + row * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) d[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t pbase = smem_u32(sP);
        const uint32_t vbase = smem_u32(sV + st * Sh::kKvBytes);
#pragma unroll
        for (int kk = 0; kk < kKvTile / 16; ++kk) {
          const uint64_t a = umma_desc_sw128(pbase + kk * 32, 16, 1024);             // P: one 64-token half
          const uint64_t b = umma_desc_sw128(vbase + kk * 2048, Sh::kKvHalf, 1024);  // V: MN-major
          umma_bf16(o_tmem, a, b, kIdPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(pv_done);
        umma_commit(&v_empty[st]);
      }
      __syncwarp();
      return true;
    };
    bool ok = wait_all(q_full, 0);
    for (int j = 0; ok && j < n_kv; ++j) {
      const int st = j & 1;
      if (!wait_all(&k_full[st], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (lane == 0) {
        const uint32_t qbase = smem_u32(sQ);
        const uint32_t kbase = smem_u32(sK + st * Sh::kKvBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t within = (kk & 3) * 32;
          umma_bf16(tmem + (j & 1) * kKvTile, umma_desc_sw128(qbase + (kk >> 2) * Sh::kQHalf + within, 16, 1024),
                    umma_desc_sw128(kbase + (kk >> 2) * Sh::kKvHalf + within, 16, 1024), kIdQK, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
        umma_commit(&k_empty[st]);
      }
      issued = true;
      __syncwarp();
      if (j >= 1 && !do_pv(j - 1)) ok = false;
    }
    if (ok) ok = do_pv(n_kv - 1);
    if (!ok && issued) {
      // wait (bounded) for every UMMA this warp issued before TMEM is freed
      if (lane == 0) umma_commit(drain);
      __syncwarp();
      mbar_wait(drain, 0, &g_status_prefill);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int row = warp * 32 + lane;
    const int hh = row / p.Tq;
    const int qi = qi0 + (row - hh * p.Tq);
    const bool row_valid = qi < q_len;
    const int p_row = row_valid ? (L - q_len + qi) : p_max;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t o_tmem = lane_base + 2 * kKvTile;
    const float sl2 = p.scale_log2;
    const float sgn = sl2 < 0.f ? -1.f : 1.f;   // max of sl2 * s = |sl2| * max(sgn * s)
    const float asl2 = fabsf(sl2);
    uint8_t* prow = sP + row * 128;
    const int sw = row & 7;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!wait_all(&s_full[j & 1], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t sv[kKvTile];
#pragma unroll
      for (int c = 0; c < kKvTile / 32; ++c) tmem_ld32(lane_base + (j & 1) * kKvTile + c * 32, sv + c * 32);
      tmem_ld_wait();
      float* sc = reinterpret_cast<float*>(sv);
      const int tok0 = j * kKvTile;
      // Visible keys of this row in this tile form a prefix: t <= p_row.  Scores stay raw
      // (times the sign of the scale); |scale| * log2(e) is folded into the max and into
      // one FMA per exponent.
      const int vis = tok0 + kKvTile - 1 > p_min ? min(max(p_row - tok0 + 1, 0), kKvTile) : kKvTile;
      const bool lean = vis == kKvTile && sgn > 0.f;   // the common case: no mask, positive scale
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (lean) {
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2) {
          mx0 = fmaxf(mx0, sc[c]);
          mx1 = fmaxf(mx1, sc[c + 1]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kKvTile; c += 2) {
          mx0 = fmaxf(mx0, c < vis ? sc[c] * sgn : -INFINITY);
          mx1 = fmaxf(mx1, c + 1 < vis ? sc[c + 1] * sgn : -INFINITY);
        }
      }
      const float m_new = fmaxf(m_run, fmaxf(mx0, mx1) * asl2);
      const bool grow = m_new > m_run + 8.0f;   // rescale only when the max grew past 2^8
      float alpha = 1.f;
      if (grow) {
        alpha = exp2_approx(m_run - m_new);
        m_run = m_new;
      }
      if (j >= 1) {
        // PV of the previous tile must be done: it reads P and accumulates into O
        if (!wait_all(pv_done, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(o_tmem + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(o_tmem + c * 32, ov);
          }
          tmem_st_wait();
        }
      }
      l_run *= alpha;
      float lsum0 = 0.f, lsum1 = 0.f;
      const float neg_m = -m_run;
#pragma unroll
      for (int c8 = 0; c8 < kKvTile / 8; ++c8) {
        float e[8];
        if (lean) {
#pragma unroll
          for (int i = 0; i < 8; ++i) e[i] = exp2_approx(fmaf(sc[c8 * 8 + i], asl2, neg_m));
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            e[i] = c8 * 8 + i < vis ? exp2_approx(fmaf(sc[c8 * 8 + i] * sgn, asl2, neg_m)) : 0.f;
        }
        lsum0 += (e[0] + e[1]) + (e[2] + e[3]);
        lsum1 += (e[4] + e[5]) + (e[6] + e[7]);
        uint4 v;
        v.x = pack_bf16x2(e[0], e[1]);
        v.y = pack_bf16x2(e[2], e[3]);
        v.z = pack_bf16x2(e[4], e[5]);
        v.w = pack_bf16x2(e[6], e[7]);
        *reinterpret_cast<uint4*>(prow + (((c8 & 7) ^ sw) << 4)) = v;
      }
      l_run += lsum0 + lsum1;
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(p_full);
    }
    if (ok && wait_all(pv_done, (n_kv - 1) & 1)) {
      tc_fence_after_sync();
      const float inv = 1.0f / l_run;
      const int head = g * p.r + hh;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)(q0 + qi) * p.H + head) * D;
#pragma unroll
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
  if (warp == 5) {
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

static size_t prefill_max_items(int num_seqs, int num_tokens, int Tq) {
  return (size_t)(num_tokens + Tq - 1) / Tq + (size_t)num_seqs;
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
  kern<<<(unsigned)(max_items * p.G), kPfThreads, smem, st>>>(tmQ, tmK, tmV, p);
  return check_launch("prefill_bf16_kernel launch");
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
