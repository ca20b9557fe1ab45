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
// Tiling.  The 128 x 512 fp32 output accumulator alone would fill all 512
// TMEM columns, so a (sequence, partition) is computed by two CTAs, each
// owning one 256-column half of the output: O_half (256 columns) plus a
// double-buffered score tile S (2 x 32 columns) fit in TMEM.  Both CTAs compute
// the same S = Q K^T (M 128 heads, N 32 tokens, K 576); the query (128 x 576
// bf16, 144 KB) stays in shared memory, 32-token latent tiles stream through
// a 2-stage TMA ring (128-byte swizzle), and P goes through a 64-byte-swizzled
// tile into O_half += P V_half (N 256, K 32, V MN-major from the same tile).
//
//   warp 4       TMA producer (Q once, then latent tiles)
//   warp 5       TMEM allocation; one lane issues the UMMAs
//   warps 0..3   softmax: one head (TMEM lane) per thread, running max in
//                log2 units, O rescaled in TMEM only when the max grows past
//                2^8; epilogue O / l
//
// A schedule kernel lists the (sequence, partition) work items heaviest first.
// A sequence with one partition writes its output directly; longer ones write
// fp32 partials that the log-sum-exp merge combines.
#include <math.h>

#include <algorithm>

#include "../../include/metis_attn.h"
#include "common.cuh"
#include "host.h"
#include "tcgen05.cuh"

namespace metis {

__device__ unsigned int g_status_mla = 0;

constexpr int kMlaDq = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaHalf = 256;              // output columns per CTA
constexpr int kMlaBlocks = kMlaDq / 64;    // 64-column blocks of a latent row
constexpr int kMlaTile = 32;               // tokens per latent tile
constexpr int kMlaRows = 128;              // heads per CTA (the UMMA M)
constexpr int kMlaThreads = 192;
constexpr int kMlaTmemCols = 512;          // S0 | S1 | O_half
constexpr int kMlaSortMax = 2048;

struct MlaShape {
  static constexpr int kQBlock = kMlaRows * 128;              // 128 heads x 64 bf16
  static constexpr int kQBytes = kMlaBlocks * kQBlock;        // 144 KB
  static constexpr int kKvBlock = kMlaTile * 128;             // 32 tokens x 64 bf16
  static constexpr int kKvBytes = kMlaBlocks * kKvBlock;      // 36 KB
  static constexpr int kQ = 0;
  static constexpr int kKv = kQ + kQBytes;                    // 2 stages
  static constexpr int kP = kKv + 2 * kKvBytes;               // 128 heads x 32 tokens, 64-byte rows
  static constexpr int kPBytes = kMlaRows * 64;
  static constexpr int kTiles = kP + kPBytes;                 // 224 KB
  static constexpr int kSmem = kTiles + 1024;                 // barriers live in the alignment slack
};

struct MlaParams {
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
  return max(1, min((L_raw + p.P - 1) / p.P, p.max_parts));
}

__global__ void __launch_bounds__(1024) mla_schedule_kernel(const MlaParams p, int4* items, int* count,
                                                            int max_items) {
  __shared__ int scan[1024];
  __shared__ int4 buf[kMlaSortMax];
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

__global__ void __launch_bounds__(kMlaThreads, 1) mla_decode_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                     const __grid_constant__ CUtensorMap tmKV,
                                                                     const MlaParams p) {
  using Sh = MlaShape;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t slack = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + slack;
  uint8_t* sQ = smem + Sh::kQ;
  uint8_t* sKV = smem + Sh::kKv;
  uint8_t* sP = smem + Sh::kP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(slack >= 256 ? smem - 256 : smem + Sh::kTiles);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;
  uint64_t* pv_done = bars + 8;
  uint64_t* drain = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 11);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = blockIdx.x & 1;
  const int rest = blockIdx.x >> 1;
  const int ht = rest % p.head_tiles;
  const int item_idx = rest / p.head_tiles;
  if (item_idx >= *p.item_count) return;
  const int4 it = p.items[item_idx];
  const int s = it.x, part = it.y;
  const int L_raw = p.seq_lens[s];
  int L = L_raw;
  if (L > p.cap) {
    if (threadIdx.x == 0 && half == 0 && ht == 0 && part == 0) atomicOr(&g_status_mla, METIS_STATUS_SEQ_TOO_LONG);
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
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + sh * kMlaDv + half * kMlaHalf;
        for (int c = 0; c < kMlaHalf; ++c) o[c] = __float2bfloat16(0.f);
        if (half == 0 && p.lse_out) p.lse_out[sh] = -INFINITY;
      } else if (half == 0) {
        p.part_lse[sh * p.max_parts + part] = -INFINITY;
      }
    }
    return;
  }
  const int n_tiles = (t1 - t0 + kMlaTile - 1) / kMlaTile;
  const int n_pages = (L + p.bs - 1) / p.bs;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 10; ++i) mbar_init(&bars[i], i == 7 ? 128 : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kMlaTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t tstart = global_timer_ns();
    for (uint32_t i = 1; i < kMaxPolls; ++i) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((i & 255u) == 0) {
        if (*abort_flag) return false;
        if (global_timer_ns() - tstart > kMaxWaitNs) break;
      }
    }
    atomicOr(&g_status_mla, METIS_STATUS_WAIT_TIMEOUT);
    *abort_flag = 1;
    return false;
  };
  auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool { return __all_sync(0xffffffffu, wait(bar, parity)); };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    const int32_t* bt_row = p.block_table + (size_t)s * p.max_blocks;
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmKV);
      mbar_arrive_expect_tx(q_full, (uint32_t)(kMlaBlocks * p.hrows * 128));
      const uint64_t pol = l2_policy_evict_first();
      for (int b = 0; b < kMlaBlocks; ++b) tma_load_3d(sQ + b * Sh::kQBlock, &tmQ, q_full, b * 64, h0, s, pol);
    }
    const int R = min(p.bs, kMlaTile);    // rows per box
    const int boxes = kMlaTile / R;       // boxes per tile
    const uint64_t pol = l2_policy_evict_first();
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j & 1;
      const int tok = t0 + j * kMlaTile + lane * R;
      const int pg = tok / p.bs;
      const bool live = lane < boxes && pg < n_pages;
      int rowc = 0;
      if (live) {
        const int b = checked_block(bt_row, pg, p.num_blocks, &g_status_mla);
        rowc = b < 0 ? -R : b * p.bs + (tok - pg * p.bs);
      }
      const uint32_t bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, live)) * R * 128 * kMlaBlocks;
      if (j >= 2 && !wait_all(&kv_empty[st], ((j >> 1) - 1) & 1)) break;
      if (lane == 0) mbar_arrive_expect_tx(&kv_full[st], bytes);
      __syncwarp();
      if (live)
        for (int b = 0; b < kMlaBlocks; ++b)
          tma_load_3d(sKV + st * Sh::kKvBytes + b * Sh::kKvBlock + lane * R * 128, &tmKV, &kv_full[st], b * 64, 0,
                      rowc, pol);
    }
    if (*abort_flag)
      for (int j = max(0, n_tiles - 2); j < n_tiles; ++j) mbar_wait(&kv_full[j & 1], (j >> 1) & 1, &g_status_mla);
  } else if (warp == 5) {
    // ------------------------------------------------------------ UMMA issuer
    constexpr uint32_t kIdQK = umma_idesc_bf16_f32(kMlaRows, kMlaTile, false, false);
    constexpr uint32_t kIdPV = umma_idesc_bf16_f32(kMlaRows, kMlaHalf, false, true);
    const uint32_t o_tmem = tmem + 2 * kMlaTile;
    bool issued = false;
    auto do_pv = [&](int i) -> bool {
      const int st = i & 1;
      if (!wait_all(p_full, i & 1)) return false;
      tc_fence_after_sync();
      const int tok0 = t0 + i * kMlaTile;
      uint8_t* vb = sKV + st * Sh::kKvBytes + half * 4 * Sh::kKvBlock;
      if (tok0 + kMlaTile > t1) {
        // rows past the partition end (NaN tails, pages not loaded): zero this half's value columns
        for (int row = (t1 - tok0) + lane; row < kMlaTile; row += 32)
          for (int b = 0; b < 4; ++b) {
            uint4* d = reinterpret_cast<uint4*>(vb + b * Sh::kKvBlock + row * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) d[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        const uint32_t pbase = smem_u32(sP);
        const uint32_t vbase = smem_u32(vb);
#pragma unroll
        for (int kk = 0; kk < kMlaTile / 16; ++kk)
          umma_bf16(o_tmem, umma_desc_sw64(pbase + kk * 32, 512), umma_desc_sw128(vbase + kk * 2048, Sh::kKvBlock, 1024),
                    kIdPV, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(pv_done);
        umma_commit(&kv_empty[st]);
      }
      __syncwarp();
      return true;
    };
    bool ok = wait_all(q_full, 0);
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int st = j & 1;
      if (!wait_all(&kv_full[st], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (lane == 0) {
        const uint32_t qbase = smem_u32(sQ);
        const uint32_t kbase = smem_u32(sKV + st * Sh::kKvBytes);
#pragma unroll 4
        for (int kk = 0; kk < kMlaDq / 16; ++kk) {
          const uint32_t within = (kk & 3) * 32;
          umma_bf16(tmem + (j & 1) * kMlaTile,
                    umma_desc_sw128(qbase + (kk >> 2) * Sh::kQBlock + within, 16, 1024),
                    umma_desc_sw128(kbase + (kk >> 2) * Sh::kKvBlock + within, 16, 1024), kIdQK, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
      }
      issued = true;
      __syncwarp();
      if (j >= 1 && !do_pv(j - 1)) ok = false;
    }
    if (ok) ok = do_pv(n_tiles - 1);
    if (!ok && issued) {
      if (lane == 0) umma_commit(drain);
      __syncwarp();
      mbar_wait(drain, 0, &g_status_mla);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int row = warp * 32 + lane;
    const int head = h0 + row;
    const bool row_valid = row < p.hrows && head < p.H;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t o_tmem = lane_base + 2 * kMlaTile;
    const float sl2 = p.scale_log2;
    const float sgn = sl2 < 0.f ? -1.f : 1.f;
    const float asl2 = fabsf(sl2);
    uint8_t* prow = sP + row * 64;
    const int sw = (row >> 1) & 3;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!wait_all(&s_full[j & 1], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t sv[kMlaTile];
      tmem_ld32(lane_base + (j & 1) * kMlaTile, sv);
      tmem_ld_wait();
      const float* sc = reinterpret_cast<const float*>(sv);
      const int vis = min(kMlaTile, t1 - (t0 + j * kMlaTile));
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int c = 0; c < kMlaTile; c += 2) {
        mx0 = fmaxf(mx0, c < vis ? sc[c] * sgn : -INFINITY);
        mx1 = fmaxf(mx1, c + 1 < vis ? sc[c + 1] * sgn : -INFINITY);
      }
      const float m_new = fmaxf(m_run, fmaxf(mx0, mx1) * asl2);
      const bool grow = m_new > m_run + 8.0f;
      float alpha = 1.f;
      if (grow) {
        alpha = exp2_approx(m_run - m_new);
        m_run = m_new;
      }
      if (j >= 1) {
        if (!wait_all(pv_done, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int c = 0; c < kMlaHalf / 32; ++c) {
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
      float lsum = 0.f;
      const float neg_m = -m_run;
#pragma unroll
      for (int c8 = 0; c8 < kMlaTile / 8; ++c8) {
        float e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          e[i] = c8 * 8 + i < vis ? exp2_approx(fmaf(sc[c8 * 8 + i] * sgn, asl2, neg_m)) : 0.f;
        lsum += ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
        uint4 v;
        v.x = pack_bf16x2(e[0], e[1]);
        v.y = pack_bf16x2(e[2], e[3]);
        v.z = pack_bf16x2(e[4], e[5]);
        v.w = pack_bf16x2(e[6], e[7]);
        *reinterpret_cast<uint4*>(prow + ((c8 ^ sw) << 4)) = v;
      }
      l_run += lsum;
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(p_full);
    }
    if (ok && wait_all(pv_done, (n_tiles - 1) & 1)) {
      tc_fence_after_sync();
      const float inv = 1.0f / l_run;
      const size_t sh = (size_t)s * p.H + head;
#pragma unroll 1
      for (int c = 0; c < kMlaHalf / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_tmem + c * 32, ov);
        tmem_ld_wait();
        if (!row_valid) continue;
        if (direct) {
          __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + sh * kMlaDv + half * kMlaHalf + c * 32;
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
          float* o = p.part_out + (sh * p.max_parts + part) * kMlaDv + half * kMlaHalf + c * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(o + i) =
                make_float4(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv,
                            __uint_as_float(ov[i + 2]) * inv, __uint_as_float(ov[i + 3]) * inv);
        }
      }
      if (row_valid && half == 0) {
        const float lse = (m_run + log2f(l_run)) * kLn2;
        if (direct) {
          if (p.lse_out) p.lse_out[sh] = lse;
        } else {
          p.part_lse[sh * p.max_parts + part] = lse;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kMlaTmemCols);
  }
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
  w.max_parts = P > 0 ? std::max(1, (max_seq_len + P - 1) / P) : 1;
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
  if (partition_size < 0 || partition_size % kMlaTile)
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

  CUtensorMap tmQ, tmKV;
  const uint64_t qdims[3] = {(uint64_t)kMlaDq, (uint64_t)num_heads, (uint64_t)num_seqs};
  const uint64_t qstr[2] = {(uint64_t)kMlaDq * 2, (uint64_t)num_heads * kMlaDq * 2};
  const uint32_t qbox[3] = {64, (uint32_t)p.hrows, 1};
  int rc = encode_tiled(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, qdims, qstr, qbox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  const uint64_t kdims[3] = {(uint64_t)kMlaDq, 1, (uint64_t)num_blocks * block_size};
  const uint64_t kstr[2] = {(uint64_t)kMlaDq * 2, (uint64_t)kMlaDq * 2};
  const uint32_t kbox[3] = {64, 1, (uint32_t)std::min(block_size, kMlaTile)};
  rc = encode_tiled(&tmKV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_cache, kdims, kstr, kbox,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;

  mla_schedule_kernel<<<1, 1024, 0, st>>>(p, items, count, (int)lay.max_items);
  rc = check_launch("mla_schedule_kernel launch");
  if (rc) return rc;
  static int done = 0;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(mla_decode_kernel), MlaShape::kSmem, &done);
  if (rc) return rc;
  mla_decode_kernel<<<(unsigned)(lay.max_items * head_tiles * 2), kMlaThreads, MlaShape::kSmem, st>>>(tmQ, tmKV, p);
  rc = check_launch("mla_decode_kernel launch");
  if (rc) return rc;
  if (partition_size > 0 && lay.max_parts > 1)
    rc = launch_merge_ex(p.part_out, p.part_lse, seq_lens, partition_size, out, lse_out, num_seqs, num_heads, kMlaDv,
                         lay.max_parts, METIS_BF16, 1, st);
  return rc;
}
