// Paged-attention decode (one query token per sequence) and the split-KV
// log-sum-exp merge.
//
// The operation is the paged-attention kernel of the vllm-metal architecture
// article (section 3: paged attention and MLA kernels as graph primitives;
// section 4: fed by the scheduler's block table and sequence lengths).  The
// pages print no formula; this is textbook softmax attention of the query
// over its sequence's cached tokens, accumulated online (running max and
// running sum, rescaling the accumulator when the max grows), optionally in
// independent token partitions whose normalised partials are merged by
// log-sum-exp.
//
// Kernels
//   decode_bf16_kernel  bf16 K/V.  One CTA per (partition, kv head, sequence);
//                       the group's r = H/G query heads share every K/V page
//                       read.  Each warp owns a private ring of 16-token K/V
//                       units that it fills with TMA tile loads (one 64-dim
//                       half per load, 128-byte swizzle) and consumes with
//                       bf16 mma.sync: S^T = K q^T (tokens x heads), online
//                       softmax with warp shuffles, then O^T += V^T P^T.
//                       Warps merge their (m, l, O) states in shared memory.
//   decode_f32_kernel   fp32 K/V on FMA units (the 1e-5 path): each warp
//                       walks tokens, lanes split head_dim.
//   merge_kernel        one CTA per (sequence, head): the log-sum-exp merge of
//                       many partitions.
//   merge_warp_kernel   one warp per (sequence, head): the merge of at most 16.
//   merge_split_rows_kernel  the rows of the sequences with two or more
//                       partitions only, one CTA per SM (MLA's merge).
//   decode_rows_beside_kernel  the single-token sequences of a chunked-prefill
//                       batch, persistent, on the SMs the chunk kernel leaves
//                       them.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "../../include/metis_attn.h"
#include "common.cuh"
#include "host.h"

namespace metis {

__device__ unsigned int g_status_decode = 0;

struct DecodeParams {
  const void* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  float* lse_out;
  float* part_out;  // split-KV partials [S, H, max_parts, D] (NULL: no split)
  float* part_lse;  // [S, H, max_parts]
  int S, H, G, D, bs, max_blocks, num_blocks, r;
  float scale_log2;  // softmax scale * log2(e)
  int partition_size;
  int max_parts;
  int cap;  // tokens readable per sequence: min(max_blocks * bs, max_seq_len)
  // Decodes of a chunked-prefill batch (NULL otherwise): the batch's cu_q_lens.
  // Sequence s is handled only if rows[s + 1] - rows[s] == 1; its query, output
  // and lse row is rows[s] of the packed [T, H, D] tensors.
  const int32_t* rows;
};

// Output (and query) row of sequence s; -1 when the call skips it (a sequence
// with more than one query token in a mixed batch).
__device__ __forceinline__ int decode_row(const DecodeParams& p, int s) {
  if (!p.rows) return s;
  const int r0 = p.rows[s];
  return p.rows[s + 1] - r0 == 1 ? r0 : -1;
}

// Token range of this CTA, after clamping the sequence length.  Returns
// false when the CTA has nothing to do (after writing what an empty
// partition or sequence must leave behind).
// tid / nthr: this thread's index among the threads that share the item.
template <typename OutT>
__device__ __forceinline__ bool decode_range(const DecodeParams& p, int part, int g, int s, int orow, int& t0,
                                             int& t1, int tid, int nthr) {
  int L_raw = p.seq_lens[s];
  int L = L_raw;
  if (L > p.cap) {
    if (tid == 0) atomicOr(&g_status_decode, METIS_STATUS_SEQ_TOO_LONG);
    L = p.cap;
  }
  if (L < 0) L = 0;
  if (p.partition_size > 0) {
    t0 = part * p.partition_size;
    t1 = min(L, t0 + p.partition_size);
  } else {
    t0 = 0;
    t1 = L;
  }
  if (t1 > t0) return true;
  if (p.partition_size > 0) {
    // A partition the merge will look at but that holds no readable token.
    if (L_raw > 0 && t0 < L_raw && tid < p.r)
      p.part_lse[((size_t)s * p.H + g * p.r + tid) * p.max_parts + part] = -INFINITY;
  } else {
    OutT* o = reinterpret_cast<OutT*>(p.out) + ((size_t)orow * p.H + (size_t)g * p.r) * p.D;
    for (int i = tid; i < p.r * p.D; i += nthr) o[i] = OutT(0.0f);
    if (p.lse_out && tid < p.r) p.lse_out[(size_t)orow * p.H + g * p.r + tid] = -INFINITY;
  }
  return false;
}

template <typename OutT>
__device__ __forceinline__ void store4(OutT* dst, float a, float b, float c, float d);

template <>
__device__ __forceinline__ void store4<float>(float* dst, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
}

template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b, float c, float d) {
  uint2 v;
  v.x = pack_bf16x2(a, b);
  v.y = pack_bf16x2(c, d);
  *reinterpret_cast<uint2*>(dst) = v;
}

// Merge the per-warp online-softmax states held in shared memory (cm, cl:
// [NW][8] running max in log2 units and running sum; co: [NW][D][8] unnormalised
// accumulators) and write the CTA's result: the final output row or a
// split-KV partial.
template <typename OutT, int NW>
__device__ __forceinline__ void combine_and_store(const DecodeParams& p, const float* cm, const float* cl,
                                                  const float* co, int part, int g, int s, int orow, int tid) {
  const int D = p.D;
  const int nq = D / 4;
  for (int idx = tid; idx < p.r * nq; idx += NW * 32) {
    const int h = idx / nq;
    const int d = (idx - h * nq) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, cm[w * 8 + h]);
    float Lsum = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = cm[w * 8 + h];
      if (mw == -INFINITY) continue;
      const float f = exp2_approx(mw - M);
      Lsum += cl[w * 8 + h] * f;
      const float* c = co + ((size_t)w * D + d) * 8 + h;
      a0 += c[0] * f;
      a1 += c[8] * f;
      a2 += c[16] * f;
      a3 += c[24] * f;
    }
    const float inv = 1.0f / Lsum;
    const int head = g * p.r + h;
    const float lse = (M + log2f(Lsum)) * kLn2;
    if (p.partition_size > 0) {
      float* dst = p.part_out + (((size_t)s * p.H + head) * p.max_parts + part) * D + d;
      *reinterpret_cast<float4*>(dst) = make_float4(a0 * inv, a1 * inv, a2 * inv, a3 * inv);
      if (d == 0) p.part_lse[((size_t)s * p.H + head) * p.max_parts + part] = lse;
    } else {
      OutT* dst = reinterpret_cast<OutT*>(p.out) + ((size_t)orow * p.H + head) * D + d;
      store4<OutT>(dst, a0 * inv, a1 * inv, a2 * inv, a3 * inv);
      if (d == 0 && p.lse_out) p.lse_out[(size_t)orow * p.H + head] = lse;
    }
  }
}

// ---------------------------------------------------------------------------
// bf16 decode: TMA page units + mma.sync
// ---------------------------------------------------------------------------
constexpr int kUnit = 16;              // tokens per pipeline unit (one m16 tile)
constexpr int kBoxBytes = kUnit * 128; // one 16-token x 64-dim bf16 box, 128-byte rows

template <int D>
struct Bf16DecodeShape {
  static constexpr int kHalves = D / 64;
  static constexpr int kStageBytes = 2 * kHalves * kBoxBytes;  // K halves, then V halves
  static constexpr int kSteps = D / 16;                        // QK k-steps == PV m-tiles
};

template <int D, int NW, int STAGES>
constexpr int bf16_decode_smem_bytes() {
  return 1024 + NW * STAGES * Bf16DecodeShape<D>::kStageBytes + NW * STAGES * 8;
}

// Longest-first order for the unsplit path: CTAs launch in grid order, so the
// CTA with z-index k takes the sequence of rank k by length (ties: lower index
// first).  Every CTA ranks the whole batch itself -- S^2 / blockDim comparisons in
// shared memory, small for the batches it is used on (kMaxRankSeqs) -- which
// needs no schedule kernel and no workspace.  The heaviest sequences start first
// and the short ones fill the SMs that free up, instead of a ragged last wave.
constexpr int kMaxRankSeqs = 128;

__device__ __forceinline__ int seq_of_rank(const DecodeParams& p, int rank, int* lens, int* found) {
  // sequences the call skips rank last
  for (int i = threadIdx.x; i < p.S; i += blockDim.x)
    lens[i] = decode_row(p, i) < 0 ? -1 : min(max(p.seq_lens[i], 0), p.cap);
  if (threadIdx.x == 0) *found = rank;
  __syncthreads();
  for (int c = threadIdx.x; c < p.S; c += blockDim.x) {
    const int Lc = lens[c];
    int r = 0;
    for (int k = 0; k < p.S; ++k) r += (lens[k] > Lc) || (lens[k] == Lc && k < c);
    if (r == rank) *found = c;
  }
  __syncthreads();
  return *found;
}

// One work item of the bf16 decode: the tokens [t0, t1) of KV head g of sequence s
// (query / output row orow), run by NW warps (warp 0 .. NW - 1 of the caller's
// group; tid = the thread's index in the group) over their NW x STAGES TMA ring at
// smem with its barriers at bars.  kb: this warp's ring position before the item
// (ring stages and barrier phases run on across the items of a persistent group),
// advanced past the item's units.  sync(): a barrier over the group's threads.
// The combine step reuses the ring: the caller syncs the group before the next
// item's loads.  Returns false when a wait gave up.
template <int D, int NW, int STAGES, typename Sync>
__device__ __forceinline__ bool decode_bf16_item(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeParams& p,
                                                 uint8_t* smem, uint64_t* bars, int part, int g, int s, int orow,
                                                 int t0, int t1, int warp, int lane, int tid, int& kb, Sync sync) {
  using Shape = Bf16DecodeShape<D>;
  constexpr int HALVES = Shape::kHalves;
  constexpr int STAGE_BYTES = Shape::kStageBytes;
  constexpr int KS = Shape::kSteps;

  // this warp's units: u0 + warp + k * NW, k < n_my
  const int u0 = t0 / kUnit;
  const int n_units = (t1 - u0 * kUnit + kUnit - 1) / kUnit;
  const int n_my = warp < n_units ? (n_units - warp + NW - 1) / NW : 0;
  const int32_t* bt_row = p.block_table + (size_t)s * p.max_blocks;

  // Lane l holds the TMA row coordinate (block * bs + slot) of unit k = 32 * batch + l;
  // -kUnit (a box entirely outside the tensor, read as zeros) marks a bad block id.
  auto row_coord = [&](int k) -> int {
    if (k >= n_my) return -kUnit;
    const int tok = (u0 + warp + k * NW) * kUnit;
    const int page = tok / p.bs;
    const int b = checked_block(bt_row, page, p.num_blocks, &g_status_decode);
    return b < 0 ? -kUnit : b * p.bs + (tok - page * p.bs);
  };
  int win_cur = row_coord(lane);
  int win_next = row_coord(32 + lane);
  const uint64_t policy = l2_policy_evict_first();

  auto issue = [&](int k) {  // called by all lanes, in order k = 0, 1, 2, ...
    if (k > 0 && (k & 31) == 0) {
      win_cur = win_next;
      win_next = row_coord(k + 32 + lane);
    }
    const int row = __shfl_sync(0xffffffffu, win_cur, k & 31);
    const int st = (kb + k) % STAGES;
    uint8_t* base = smem + (warp * STAGES + st) * STAGE_BYTES;
    uint64_t* bar = &bars[warp * STAGES + st];
    if (lane == 0) mbar_arrive_expect_tx(bar, STAGE_BYTES);
    __syncwarp();
    // one box per lane: a single thread issues TMA instructions far slower than several
    if (lane < 2 * HALVES) {
      const int h = lane % HALVES;
      tma_load_3d(base + lane * kBoxBytes, lane < HALVES ? &tmK : &tmV, bar, h * 64, g, row, policy);
    }
  };

  // q^T as the B operand of S^T = K q^T: lane holds head n = lane / 4, dims 2*(lane%4) (+1, +8, +9)
  const int q4 = lane & 3, rA = lane >> 2;
  uint32_t qf[KS][2];
  {
    const bool live = rA < p.r;
    const __nv_bfloat16* qrow =
        reinterpret_cast<const __nv_bfloat16*>(p.q) + ((size_t)orow * p.H + g * p.r + (live ? rA : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      qf[kk][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * q4) : 0u;
      qf[kk][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * q4) : 0u;
    }
  }

  float o[KS][4];
#pragma unroll
  for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2*q4 and 2*q4+1
  const float sl2 = p.scale_log2;

  const int prologue = n_my < STAGES ? n_my : STAGES;
  for (int k = 0; k < prologue; ++k) issue(k);

  int k = 0;
  bool ok = true;
  for (; k < n_my; ++k) {
    const int st = (kb + k) % STAGES;
    const bool landed = mbar_wait(&bars[warp * STAGES + st], ((kb + k) / STAGES) & 1, &g_status_decode);
    if (!__all_sync(0xffffffffu, landed)) {  // leave the loop together
      ok = false;
      break;
    }
    const int tok0 = (u0 + warp + k * NW) * kUnit;
    const int nv = min(kUnit, t1 - tok0);  // valid tokens in this unit, >= 1
    const uint32_t kbase = smem_u32(smem + (warp * STAGES + st) * STAGE_BYTES);
    const uint32_t vbase = kbase + HALVES * kBoxBytes;

    // S^T (16 tokens x 8 heads) = K (16 x D) . q^T (D x 8), in two independent
    // accumulation chains (even / odd k-steps) to halve the dependent-MMA latency
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      float sacc2[4] = {0.f, 0.f, 0.f, 0.f};
      const int j = lane >> 3;
      const int row = ((j & 1) << 3) + (lane & 7);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const int c = kk * 2 + (j >> 1);
        const uint32_t addr = kbase + (c >> 3) * kBoxBytes + row * 128 + ((((c & 7) ^ (row & 7))) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
        mma_bf16_16816((kk & 1) ? sacc2 : sacc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[i] += sacc2[i];
    }

    // online softmax over this unit; the thread holds tokens rA, rA+8 of heads 2*q4, 2*q4+1
    float s0 = sacc[0] * sl2, s1 = sacc[1] * sl2, s2 = sacc[2] * sl2, s3 = sacc[3] * sl2;
    if (rA >= nv) s0 = s1 = -INFINITY;
    if (rA + 8 >= nv) s2 = s3 = -INFINITY;
    const float mn0 = fmaxf(m0, warp_max_xor(fmaxf(s0, s2), 4));
    const float mn1 = fmaxf(m1, warp_max_xor(fmaxf(s1, s3), 4));
    const float al0 = exp2_approx(m0 - mn0), al1 = exp2_approx(m1 - mn1);
    const float p0 = exp2_approx(s0 - mn0), p1 = exp2_approx(s1 - mn1);
    const float p2 = exp2_approx(s2 - mn0), p3 = exp2_approx(s3 - mn1);
    l0 = l0 * al0 + (p0 + p2);
    l1 = l1 * al1 + (p1 + p3);
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al1;
      o[i][2] *= al0;
      o[i][3] *= al1;
    }
    // P^T (tokens x heads) -> B operand (k = token, n = head) by 8x8 transposes
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));

    // Rows past the last valid token may hold anything (NaN included): zero
    // them in the V^T fragments so that 0 * garbage cannot poison O.
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (nv < kUnit) {
      const int t = 2 * q4;
      mlo = (t < nv ? 0x0000ffffu : 0u) | (t + 1 < nv ? 0xffff0000u : 0u);
      mhi = (t + 8 < nv ? 0x0000ffffu : 0u) | (t + 9 < nv ? 0xffff0000u : 0u);
    }
    // O^T (D x 8 heads) += V^T (D x 16 tokens) . P^T (16 tokens x 8 heads)
    {
      const int j = lane >> 3;
      const int row = ((j >> 1) << 3) + (lane & 7);
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int c = mt * 2 + (j & 1);
        const uint32_t addr = vbase + (c >> 3) * kBoxBytes + row * 128 + ((((c & 7) ^ (row & 7))) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(addr, a0, a1, a2, a3);
        mma_bf16_16816(o[mt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, pb0, pb1);
      }
    }
    __syncwarp();
    if (k + STAGES < n_my) issue(k + STAGES);
  }
  if (!ok) {
    // drain this warp's loads still in flight (bounded) before the ring is reused
    for (int kk = k + 1; kk < n_my && kk < k + STAGES; ++kk) {
      const int st = (kb + kk) % STAGES;
      mbar_wait(&bars[warp * STAGES + st], ((kb + kk) / STAGES) & 1, &g_status_decode);
    }
  }

  l0 = warp_sum_xor(l0, 4);
  l1 = warp_sum_xor(l1, 4);
  sync();  // every warp is done with its ring

  float* cm = reinterpret_cast<float*>(smem);
  float* cl = cm + NW * 8;
  float* co = cl + NW * 8;
  if (lane < 4) {
    cm[warp * 8 + 2 * lane] = m0;
    cm[warp * 8 + 2 * lane + 1] = m1;
    cl[warp * 8 + 2 * lane] = l0;
    cl[warp * 8 + 2 * lane + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    const int d0 = mt * 16 + rA;
    float* c0 = co + ((size_t)warp * D + d0) * 8 + 2 * q4;
    float* c1 = c0 + 8 * 8;
    c0[0] = o[mt][0];
    c0[1] = o[mt][1];
    c1[0] = o[mt][2];
    c1[1] = o[mt][3];
  }
  sync();
  combine_and_store<__nv_bfloat16, NW>(p, cm, cl, co, part, g, s, orow, tid);
  kb += n_my;
  return ok;
}

template <int D, int NW, int STAGES>
__global__ void __launch_bounds__(NW * 32) decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                                                               const __grid_constant__ CUtensorMap tmV,
                                                               const DecodeParams p) {
  using Shape = Bf16DecodeShape<D>;
  constexpr int STAGE_BYTES = Shape::kStageBytes;
  static_assert(NW * (64 + D * 32) <= NW * STAGES * STAGE_BYTES, "combine area must fit in the ring");
  // Launched as a programmatic dependent (e.g. of the paged K/V write): every input
  // is read after the previous grid in the stream has completed.  Only then may the
  // next grid launch (the merge, which waits for this grid to finish anyway).
  pdl_wait();
  pdl_launch_dependents();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-aligned for the swizzle
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * STAGES * STAGE_BYTES);

  __shared__ int rank_lens[kMaxRankSeqs];
  __shared__ int rank_found;
  const int part = blockIdx.x, g = blockIdx.y;
  const int s = (p.partition_size == 0 && p.S <= kMaxRankSeqs) ? seq_of_rank(p, blockIdx.z, rank_lens, &rank_found)
                                                                : (int)blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int orow = decode_row(p, s);
  if (orow < 0) return;  // not a decode of this mixed batch
  int t0, t1;
  if (!decode_range<__nv_bfloat16>(p, part, g, s, orow, t0, t1, threadIdx.x, blockDim.x)) return;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < NW * STAGES; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  int kb = 0;
  decode_bf16_item<D, NW, STAGES>(tmK, tmV, p, smem, bars, part, g, s, orow, t0, t1, warp, lane, threadIdx.x, kb,
                                  [] { __syncthreads(); });
}

// bf16 decode configuration: warps per CTA and ring depth per warp.
#ifndef METIS_DECODE_WARPS
#define METIS_DECODE_WARPS 4
#endif
#ifndef METIS_DECODE_STAGES
#define METIS_DECODE_STAGES 3
#endif
constexpr int kBf16Warps = METIS_DECODE_WARPS;
constexpr int kBf16Stages = METIS_DECODE_STAGES;

// ---------------------------------------------------------------------------
// the decodes of a mixed chunked-prefill batch, beside the chunk kernel
// ---------------------------------------------------------------------------
// The chunk kernel takes whole SMs.  Beside it, the batch's decodes run on the
// first n_ctas SMs only (the prefill schedule kernel sizes n_ctas from the batch's
// decode bytes and chunk FLOPs) rather than on every SM for a shorter time.  One
// CTA per SM (its shared memory request sees to that), kDecGroups groups of
// kBf16Warps warps each; a group takes (sequence, KV head) items -- sequences
// longest first -- from a counter that the schedule kernel zeroed.
constexpr int kDecGroups = 2;

template <int D>
constexpr int dec_beside_smem_bytes() {
  constexpr int need = 1024 + kDecGroups * kBf16Warps * kBf16Stages * (Bf16DecodeShape<D>::kStageBytes + 8);
  return need > 116 * 1024 ? need : 116 * 1024;  // never two CTAs on one SM
}

template <int D>
__global__ void __launch_bounds__(kDecGroups * kBf16Warps * 32, 1)
    decode_rows_beside_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                              const DecodeParams p, const int* n_ctas, int* next_item) {
  constexpr int NW = kBf16Warps, STAGES = kBf16Stages, GT = NW * 32;
  constexpr int STAGE_BYTES = Bf16DecodeShape<D>::kStageBytes;
  static_assert(NW * (64 + D * 32) <= NW * STAGES * STAGE_BYTES, "combine area must fit in the ring");
  pdl_wait();  // the schedule kernel (n_ctas, the zeroed counter) and every kernel before it completed
  if ((int)blockIdx.x >= __ldcg(n_ctas)) return;
  pdl_launch_dependents();  // every CTA of the grid has waited by now: the chunk kernel may launch

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-aligned for the swizzle
  __shared__ int rank_seq[kMaxRankSeqs];
  __shared__ int lens[kMaxRankSeqs];
  __shared__ int n_dec;
  __shared__ int item_slot[kDecGroups];
  __shared__ int gave_up[kDecGroups];  // a warp of the group gave up a wait: the group stops
  // the batch's decodes, longest first (larger batches: in sequence order)
  const bool ranked = p.S <= kMaxRankSeqs;
  if (ranked) {
    if (threadIdx.x == 0) n_dec = 0;
    for (int i = threadIdx.x; i < p.S; i += blockDim.x)
      lens[i] = decode_row(p, i) < 0 ? -1 : min(max(p.seq_lens[i], 0), p.cap);
    __syncthreads();
    for (int c = threadIdx.x; c < p.S; c += blockDim.x) {
      const int Lc = lens[c];
      if (Lc < 0) continue;
      int r = 0;
      for (int k = 0; k < p.S; ++k) r += (lens[k] > Lc) || (lens[k] == Lc && k < c);
      rank_seq[r] = c;
      atomicAdd(&n_dec, 1);
    }
  }
  const int grp = threadIdx.x / GT, tid = threadIdx.x - grp * GT;
  const int warp = tid >> 5, lane = tid & 31;
  uint8_t* gsmem = smem + grp * NW * STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kDecGroups * NW * STAGES * STAGE_BYTES) + grp * NW * STAGES;
  if (tid == 0) {
    if (grp == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    for (int i = 0; i < NW * STAGES; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    gave_up[grp] = 0;
  }
  __syncthreads();
  const int n_items = (ranked ? n_dec : p.S) * p.G;
  auto gsync = [grp] { named_barrier_sync(1 + grp, GT); };
  int kb = 0;  // this warp's ring position, across the group's items
  for (;;) {
    gsync();  // the previous item's combine is done with the ring, and the slot was read
    if (gave_up[grp]) break;  // read after the barrier: the whole group leaves together
    if (tid == 0) item_slot[grp] = atomicAdd(next_item, 1);
    gsync();
    const int it = item_slot[grp];
    if (it >= n_items) break;
    const int rank = it / p.G, g = it - rank * p.G;
    const int s = ranked ? rank_seq[rank] : rank;
    const int orow = decode_row(p, s);
    if (orow < 0) continue;  // not a decode (unranked order only)
    int t0, t1;
    if (!decode_range<__nv_bfloat16>(p, 0, g, s, orow, t0, t1, tid, GT)) continue;
    // A wait that gave up (flagged) is seen by its warp only: every warp of the group
    // still reaches the item's barriers and the next one above, where they all stop.
    if (!decode_bf16_item<D, NW, STAGES>(tmK, tmV, p, gsmem, bars, 0, g, s, orow, t0, t1, warp, lane, tid, kb, gsync) &&
        lane == 0)
      gave_up[grp] = 1;
  }
}

// ---------------------------------------------------------------------------
// fp32 decode on FMA units
// ---------------------------------------------------------------------------
constexpr int kF32Warps = 8;

template <int D>
__global__ void __launch_bounds__(kF32Warps * 32) decode_f32_kernel(const float* __restrict__ k_cache,
                                                                     const float* __restrict__ v_cache,
                                                                     const DecodeParams p) {
  constexpr int DPL = D / 32;  // dims per lane
  pdl_launch_dependents();
  pdl_wait();  // inputs are read after the previous grid in the stream has completed
  __shared__ float cm[kF32Warps * 8], cl[kF32Warps * 8];
  __shared__ float co[kF32Warps * D * 8];

  const int part = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int t0, t1;
  if (!decode_range<float>(p, part, g, s, s, t0, t1, threadIdx.x, blockDim.x)) return;

  const float* q = reinterpret_cast<const float*>(p.q) + ((size_t)s * p.H + (size_t)g * p.r) * D;
  float qv[8][DPL];
#pragma unroll
  for (int h = 0; h < 8; ++h)
#pragma unroll
    for (int i = 0; i < DPL; ++i) qv[h][i] = h < p.r ? q[h * D + lane * DPL + i] * p.scale_log2 : 0.f;

  float m[8], l[8], o[8][DPL];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[h][i] = 0.f;
  }
  const int32_t* bt_row = p.block_table + (size_t)s * p.max_blocks;
  const size_t row_stride = (size_t)p.G * D;
  // The warp's tokens t0 + warp, + kF32Warps, ... in groups of kF32Batch: the block ids
  // and K/V rows of a group are loaded together, then folded in one at a time in token
  // order (the same order as without grouping).
  constexpr int kF32Batch = D == 64 ? 8 : 4;
  for (int tb = t0 + warp; tb < t1; tb += kF32Batch * kF32Warps) {
    float kv[kF32Batch][DPL], vv[kF32Batch][DPL];
#pragma unroll
    for (int u = 0; u < kF32Batch; ++u) {
      const int t = tb + u * kF32Warps;
      int b = -1, page = 0;
      if (t < t1) {
        page = t / p.bs;
        b = checked_block(bt_row, page, p.num_blocks, &g_status_decode);
      }
      if (b >= 0) {
        const size_t off = ((size_t)b * p.bs + (t - page * p.bs)) * row_stride + (size_t)g * D + lane * DPL;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          kv[u][i] = __ldg(k_cache + off + i);
          vv[u][i] = __ldg(v_cache + off + i);
        }
      } else {
#pragma unroll
        for (int i = 0; i < DPL; ++i) kv[u][i] = vv[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kF32Batch; ++u) {
      if (tb + u * kF32Warps >= t1) break;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h < p.r) {
          float dot = 0.f;
#pragma unroll
          for (int i = 0; i < DPL; ++i) dot = fmaf(qv[h][i], kv[u][i], dot);
          dot = warp_sum_xor(dot, 1);
          const float mn = fmaxf(m[h], dot);
          const float al = exp2_approx(m[h] - mn);
          const float pr = exp2_approx(dot - mn);
          l[h] = l[h] * al + pr;
#pragma unroll
          for (int i = 0; i < DPL; ++i) o[h][i] = fmaf(pr, vv[u][i], o[h][i] * al);
          m[h] = mn;
        }
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      cm[warp * 8 + h] = m[h];
      cl[warp * 8 + h] = l[h];
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h)
#pragma unroll
    for (int i = 0; i < DPL; ++i) co[((size_t)warp * D + lane * DPL + i) * 8 + h] = o[h][i];
  __syncthreads();
  combine_and_store<float, kF32Warps>(p, cm, cl, co, part, g, s, s, threadIdx.x);
}

// ---------------------------------------------------------------------------
// log-sum-exp merge of split-KV partials
// ---------------------------------------------------------------------------
constexpr int kMergeThreads = 128;
constexpr int kMergeMaxD = 512;

// One CTA per (sequence, head) when there are many partitions.  The partition
// weights exp(lse_i - max) are computed once into shared memory; then each warp
// sums every kMergeWarps-th partition, kMergeUnroll partitions per step so that
// that many row loads per lane are in flight at once (the sum is bound by memory
// latency, not by bandwidth, at one row per warp).
constexpr int kMergeWarps = 8;
constexpr int kMergeUnroll = 4;
constexpr int kMergeCache = 2048;   // partitions whose weights are cached (beyond: recomputed per row)

template <typename OutT>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const float* __restrict__ part_out,
                                                                 const float* __restrict__ part_lse,
                                                                 const int32_t* __restrict__ seq_lens, int P,
                                                                 OutT* __restrict__ out, float* __restrict__ lse_out,
                                                                 int H, int D, int max_parts, int skip_single) {
  constexpr int NT = kMergeWarps * 32;
  constexpr int NJ = kMergeMaxD / 128;   // float4 columns per lane
  __shared__ float red[kMergeWarps];
  __shared__ float wts[kMergeCache];
  __shared__ float4 acc_s[kMergeWarps][kMergeMaxD / 4];
  pdl_wait();  // the partials of the kernel before this one are complete and visible
  const size_t sh = blockIdx.x;
  const int s = (int)(sh / H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = seq_lens[s];
  const int n = L > 0 ? min(L / P + (L % P != 0), max_parts) : 0;   // ceil(L / P) without overflow
  if (skip_single && n <= 1) return;  // written directly by the producing kernel
  const float* lrow = part_lse + sh * max_parts;

  // max of the partition lse values (natural log)
  float M = -INFINITY;
  for (int i = threadIdx.x; i < n; i += NT) M = fmaxf(M, lrow[i]);
  M = warp_max_xor(M, 1);
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kMergeWarps; ++w) M = fmaxf(M, red[w]);
  const bool empty = !(M > -INFINITY);
  const float M2 = M * kLog2e;
  __syncthreads();

  // weights (0 for an empty partition, whose row is never read) and their sum
  float W = 0.f;
  if (!empty)
    for (int i = threadIdx.x; i < n; i += NT) {
      const float x = lrow[i];
      const float w = x > -INFINITY ? exp2_approx(fmaf(x, kLog2e, -M2)) : 0.f;
      if (i < kMergeCache) wts[i] = w;
      W += w;
    }
  W = warp_sum_xor(W, 1);
  if (lane == 0) red[warp] = W;
  __syncthreads();
  W = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) W += red[w];

  // warp w sums partitions w, w + kMergeWarps, ...; lane owns float4 columns lane, lane + 32, ...
  const int nq = D / 4;
  float4 acc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!empty) {
    const float4* prow = reinterpret_cast<const float4*>(part_out + sh * max_parts * D);
    for (int i0 = warp; i0 < n; i0 += kMergeWarps * kMergeUnroll) {
      float w[kMergeUnroll];
      float4 v[kMergeUnroll][NJ];
#pragma unroll
      for (int k = 0; k < kMergeUnroll; ++k) {
        const int i = i0 + k * kMergeWarps;
        w[k] = 0.f;
        if (i < n) {
          if (i < kMergeCache) {
            w[k] = wts[i];
          } else {
            const float x = lrow[i];
            w[k] = x > -INFINITY ? exp2_approx(fmaf(x, kLog2e, -M2)) : 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int c = lane + 32 * j;
          v[k][j] = (w[k] != 0.f && c < nq) ? __ldg(prow + (size_t)i * nq + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int k = 0; k < kMergeUnroll; ++k)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          acc[j].x = fmaf(w[k], v[k][j].x, acc[j].x);
          acc[j].y = fmaf(w[k], v[k][j].y, acc[j].y);
          acc[j].z = fmaf(w[k], v[k][j].z, acc[j].z);
          acc[j].w = fmaf(w[k], v[k][j].w, acc[j].w);
        }
    }
  }
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = lane + 32 * j;
    if (c < nq) acc_s[warp][c] = acc[j];
  }
  __syncthreads();
  const float inv = empty ? 0.f : 1.0f / W;
  for (int c = threadIdx.x; c < nq; c += NT) {
    float4 t = acc_s[0][c];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) {
      t.x += acc_s[w][c].x;
      t.y += acc_s[w][c].y;
      t.z += acc_s[w][c].z;
      t.w += acc_s[w][c].w;
    }
    store4<OutT>(out + sh * D + (size_t)c * 4, t.x * inv, t.y * inv, t.z * inv, t.w * inv);
  }
  if (threadIdx.x == 0 && lse_out) lse_out[sh] = empty ? -INFINITY : M + log2f(W) * kLn2;
}

// The merge of row sh = (sequence, head) over its n partitions by one warp: lanes
// share the lse reductions and own float4 columns lane, lane + 32, ...
template <typename OutT>
__device__ __forceinline__ void merge_row(const float* __restrict__ part_out, const float* __restrict__ part_lse,
                                          OutT* __restrict__ out, float* __restrict__ lse_out, size_t sh, int n,
                                          int D, int max_parts, int lane) {
  const float* lrow = part_lse + sh * max_parts;
  float M = -INFINITY;
  for (int i = lane; i < n; i += 32) M = fmaxf(M, lrow[i]);
  M = warp_max_xor(M, 1);
  const bool empty = !(M > -INFINITY);
  const float M2 = M * kLog2e;
  float W = 0.f;
  if (!empty)
    for (int i = lane; i < n; i += 32) {
      const float x = lrow[i];
      if (x > -INFINITY) W += exp2_approx(fmaf(x, kLog2e, -M2));
    }
  W = warp_sum_xor(W, 1);
  const int nq = D / 4;
  float4 acc[kMergeMaxD / 128];
#pragma unroll
  for (int j = 0; j < kMergeMaxD / 128; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!empty) {
    // kMergeUnroll partitions per step, so that many row loads per lane are in
    // flight at once (one at a time, the sum waits on memory latency)
    const float4* prow = reinterpret_cast<const float4*>(part_out + sh * max_parts * D);
    for (int i0 = 0; i0 < n; i0 += kMergeUnroll) {
      float w[kMergeUnroll];
      float4 v[kMergeUnroll][kMergeMaxD / 128];
#pragma unroll
      for (int k = 0; k < kMergeUnroll; ++k) {
        const int i = i0 + k;
        const float x = i < n ? lrow[i] : -INFINITY;
        w[k] = x > -INFINITY ? exp2_approx(fmaf(x, kLog2e, -M2)) : 0.f;
#pragma unroll
        for (int j = 0; j < kMergeMaxD / 128; ++j) {
          const int c = lane + 32 * j;
          v[k][j] = (w[k] != 0.f && c < nq) ? __ldg(prow + (size_t)i * nq + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int k = 0; k < kMergeUnroll; ++k)
#pragma unroll
        for (int j = 0; j < kMergeMaxD / 128; ++j) {
          acc[j].x = fmaf(w[k], v[k][j].x, acc[j].x);
          acc[j].y = fmaf(w[k], v[k][j].y, acc[j].y);
          acc[j].z = fmaf(w[k], v[k][j].z, acc[j].z);
          acc[j].w = fmaf(w[k], v[k][j].w, acc[j].w);
        }
    }
  }
  const float inv = empty ? 0.f : 1.0f / W;
#pragma unroll
  for (int j = 0; j < kMergeMaxD / 128; ++j) {
    const int c = lane + 32 * j;
    if (c < nq) store4<OutT>(out + sh * D + (size_t)c * 4, acc[j].x * inv, acc[j].y * inv, acc[j].z * inv,
                             acc[j].w * inv);
  }
  if (lane == 0 && lse_out) lse_out[sh] = empty ? -INFINITY : M + log2f(W) * kLn2;
}

// One warp per (sequence, head) when there are few partitions.
template <typename OutT>
__global__ void __launch_bounds__(kMergeThreads) merge_warp_kernel(const float* __restrict__ part_out,
                                                                   const float* __restrict__ part_lse,
                                                                   const int32_t* __restrict__ seq_lens, int P,
                                                                   OutT* __restrict__ out,
                                                                   float* __restrict__ lse_out, int S, int H, int D,
                                                                   int max_parts, int skip_single) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();  // the partials of the kernel before this one are complete and visible
  const size_t sh = (size_t)blockIdx.x * (kMergeThreads / 32) + warp;
  if (sh >= (size_t)S * H) return;
  const int s = (int)(sh / H);
  const int L = seq_lens[s];
  const int n = L > 0 ? min(L / P + (L % P != 0), max_parts) : 0;   // ceil(L / P) without overflow
  if (skip_single && n <= 1) return;
  merge_row<OutT>(part_out, part_lse, out, lse_out, sh, n, D, max_parts, lane);
}

// Only the sequences with two or more partitions (the others were written
// directly), for batches of up to kMergeListThreads sequences: every CTA lists
// those sequences itself (a scan over seq_lens), and the grid's warps -- one CTA
// per SM, a single wave -- take their (sequence, head) rows in turn.  Few CTAs
// instead of one per four rows of every sequence: when most sequences have one
// partition, most of those CTAs would only check a length and exit.
constexpr int kMergeListThreads = 512;  // 128 registers a thread: the row merge needs ~94
template <typename OutT>
__global__ void __launch_bounds__(kMergeListThreads, 1) merge_split_rows_kernel(
    const float* __restrict__ part_out, const float* __restrict__ part_lse, const int32_t* __restrict__ seq_lens,
    int P, OutT* __restrict__ out, float* __restrict__ lse_out, int S, int H, int D, int max_parts) {
  __shared__ int warp_sums[32];
  __shared__ int list_s[kMergeListThreads];
  __shared__ int list_n[kMergeListThreads];
  pdl_wait();  // the partials of the kernel before this one are complete and visible
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int n = 0;
  if (tid < S) {
    const int L = seq_lens[tid];
    n = L > 0 ? min(L / P + (L % P != 0), max_parts) : 0;
  }
  const int split = n >= 2;
  int total;
  const int pos = block_exclusive_scan<kMergeListThreads>(split, warp_sums, &total);
  if (split) {
    list_s[pos] = tid;
    list_n[pos] = n;
  }
  __syncthreads();
  const long long rows = (long long)total * H;
  const long long stride = (long long)gridDim.x * (kMergeListThreads / 32);
  for (long long r = (long long)blockIdx.x * (kMergeListThreads / 32) + warp; r < rows; r += stride) {
    const int k = (int)(r / H), h = (int)(r - (long long)k * H);
    merge_row<OutT>(part_out, part_lse, out, lse_out, (size_t)list_s[k] * H + h, list_n[k], D, max_parts, lane);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int decode_status(uint32_t* bits, int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_status_decode, sizeof(v));
  if (e == cudaSuccess && clear) {
    unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_status_decode, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  *bits |= v;
  return METIS_OK;
}

// Few partitions: a warp per (sequence, head); many: a CTA per (sequence, head)
// whose warps split the partitions.
int launch_merge_ex(const float* part_out, const float* part_lse, const int32_t* seq_lens, int P, void* out,
                    float* lse_out, int S, int H, int D, int max_parts, int out_dtype, int skip_single,
                    cudaStream_t st) {
  const size_t pairs = (size_t)S * H;
  // launched as a programmatic dependent: its launch overlaps the tail of the kernel
  // that wrote the partials, and it waits (pdl_wait) for that kernel to finish
  if (max_parts <= 16) {
    const dim3 grid((unsigned)((pairs + kMergeThreads / 32 - 1) / (kMergeThreads / 32)));
    if (out_dtype == METIS_BF16)
      return launch_dependent(merge_warp_kernel<__nv_bfloat16>, grid, dim3(kMergeThreads), 0, st, "merge kernel launch",
                              part_out, part_lse, seq_lens, P, reinterpret_cast<__nv_bfloat16*>(out), lse_out, S, H, D,
                              max_parts, skip_single);
    return launch_dependent(merge_warp_kernel<float>, grid, dim3(kMergeThreads), 0, st, "merge kernel launch", part_out,
                            part_lse, seq_lens, P, reinterpret_cast<float*>(out), lse_out, S, H, D, max_parts,
                            skip_single);
  }
  const dim3 grid((unsigned)pairs);
  if (out_dtype == METIS_BF16)
    return launch_dependent(merge_kernel<__nv_bfloat16>, grid, dim3(kMergeWarps * 32), 0, st, "merge kernel launch",
                            part_out, part_lse, seq_lens, P, reinterpret_cast<__nv_bfloat16*>(out), lse_out, H, D,
                            max_parts, skip_single);
  return launch_dependent(merge_kernel<float>, grid, dim3(kMergeWarps * 32), 0, st, "merge kernel launch", part_out,
                          part_lse, seq_lens, P, reinterpret_cast<float*>(out), lse_out, H, D, max_parts, skip_single);
}

int launch_merge_split_rows(const float* part_out, const float* part_lse, const int32_t* seq_lens, int P, void* out,
                            float* lse_out, int S, int H, int D, int max_parts, int out_dtype, int sms,
                            cudaStream_t st) {
  if (S > kMergeListThreads || max_parts > 16 || D > kMergeMaxD)  // outside this kernel's reach
    return launch_merge_ex(part_out, part_lse, seq_lens, P, out, lse_out, S, H, D, max_parts, out_dtype, 1, st);
  const dim3 grid((unsigned)std::max(sms, 1));
  if (out_dtype == METIS_BF16)
    return launch_dependent(merge_split_rows_kernel<__nv_bfloat16>, grid, dim3(kMergeListThreads), 0, st,
                            "merge kernel launch", part_out, part_lse, seq_lens, P,
                            reinterpret_cast<__nv_bfloat16*>(out), lse_out, S, H, D, max_parts);
  return launch_dependent(merge_split_rows_kernel<float>, grid, dim3(kMergeListThreads), 0, st, "merge kernel launch",
                          part_out, part_lse, seq_lens, P, reinterpret_cast<float*>(out), lse_out, S, H, D, max_parts);
}

static int launch_merge(const float* part_out, const float* part_lse, const int32_t* seq_lens, int P, void* out,
                        float* lse_out, int S, int H, int D, int max_parts, int out_dtype, cudaStream_t st) {
  return launch_merge_ex(part_out, part_lse, seq_lens, P, out, lse_out, S, H, D, max_parts, out_dtype, 0, st);
}

// Partitions a split call launches: ceil(max_seq_len / partition_size), in 64
// bits (max_seq_len near INT_MAX must not overflow); 0 when unsplit.
static size_t split_parts(int max_seq_len, int partition_size) {
  if (partition_size <= 0 || max_seq_len <= 0) return 0;
  return (size_t)(((long long)max_seq_len + partition_size - 1) / partition_size);
}

// The longest sequence a call can read: max_seq_len, clamped to what a
// block-table row addresses (max_blocks * block_size).  Partitions past it
// would only ever be empty, so they are neither launched nor given scratch.
static int effective_max_len(int max_seq_len, int max_blocks, int block_size) {
  return (int)std::min<long long>((long long)max_blocks * block_size, (long long)max_seq_len);
}

// TMA maps of the K and V caches: 16-token x 64-dim boxes of one KV head.
template <int D>
static int encode_kv_maps(const DecodeParams& p, const void* k_cache, const void* v_cache, CUtensorMap* tmK,
                          CUtensorMap* tmV) {
  const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.G, (uint64_t)p.num_blocks * p.bs};
  const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.G * D * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)kUnit};
  int rc = encode_tiled(tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, k_cache, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  return encode_tiled(tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, v_cache, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D>
static int launch_bf16(const DecodeParams& p, const void* k_cache, const void* v_cache, dim3 grid, cudaStream_t st) {
  CUtensorMap tmK, tmV;
  int rc = encode_kv_maps<D>(p, k_cache, v_cache, &tmK, &tmV);
  if (rc) return rc;
  constexpr int smem = bf16_decode_smem_bytes<D, kBf16Warps, kBf16Stages>();
  static int done = 0;
  auto kern = decode_bf16_kernel<D, kBf16Warps, kBf16Stages>;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem, &done);
  if (rc) return rc;
  return launch_dependent(kern, grid, dim3(kBf16Warps * 32), (size_t)smem, st, "decode_bf16_kernel launch", tmK, tmV,
                          p);
}

static DecodeParams rows_params(const void* q, const int32_t* block_table, const int32_t* seq_lens,
                                const int32_t* rows, void* out, float* lse_out, int S, int H, int G, int D, int bs,
                                int max_blocks, int num_blocks, float scale, int cap) {
  DecodeParams p;
  p.q = q;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.lse_out = lse_out;
  p.part_out = nullptr;
  p.part_lse = nullptr;
  p.S = S;
  p.H = H;
  p.G = G;
  p.D = D;
  p.bs = bs;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.r = H / G;
  p.scale_log2 = scale * kLog2e;
  p.partition_size = 0;
  p.max_parts = 1;
  p.cap = cap;
  p.rows = rows;
  return p;
}

// The single-token sequences of a chunked-prefill batch, through the decode
// kernel (unsplit, longest first): rows = the batch's cu_q_lens.  The caller has
// validated the shapes (bf16, head_dim 64 or 128, head ratio 1, 2, 4 or 8).
int launch_decode_rows(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* seq_lens, const int32_t* rows, void* out, float* lse_out, int S, int H, int G,
                       int D, int bs, int max_blocks, int num_blocks, float scale, int cap, cudaStream_t st) {
  const DecodeParams p =
      rows_params(q, block_table, seq_lens, rows, out, lse_out, S, H, G, D, bs, max_blocks, num_blocks, scale, cap);
  const dim3 grid(1u, (unsigned)G, (unsigned)S);
  return D == 64 ? launch_bf16<64>(p, k_cache, v_cache, grid, st) : launch_bf16<128>(p, k_cache, v_cache, grid, st);
}

template <int D>
static int launch_beside(const DecodeParams& p, const void* k_cache, const void* v_cache, const int* n_ctas,
                         int* next_item, int grid, cudaStream_t st) {
  CUtensorMap tmK, tmV;
  int rc = encode_kv_maps<D>(p, k_cache, v_cache, &tmK, &tmV);
  if (rc) return rc;
  constexpr int smem = dec_beside_smem_bytes<D>();
  static int done = 0;
  auto kern = decode_rows_beside_kernel<D>;
  rc = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem, &done);
  if (rc) return rc;
  return launch_dependent(kern, dim3((unsigned)grid), dim3(kDecGroups * kBf16Warps * 32), (size_t)smem, st,
                          "decode_rows_beside_kernel launch", tmK, tmV, p, n_ctas, next_item);
}

int launch_decode_rows_beside(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                              const int32_t* seq_lens, const int32_t* rows, void* out, float* lse_out, int S, int H,
                              int G, int D, int bs, int max_blocks, int num_blocks, float scale, int cap,
                              const int* n_ctas, int* next_item, int grid, cudaStream_t st) {
  const DecodeParams p =
      rows_params(q, block_table, seq_lens, rows, out, lse_out, S, H, G, D, bs, max_blocks, num_blocks, scale, cap);
  return D == 64 ? launch_beside<64>(p, k_cache, v_cache, n_ctas, next_item, grid, st)
                 : launch_beside<128>(p, k_cache, v_cache, n_ctas, next_item, grid, st);
}

}  // namespace metis

using namespace metis;

extern "C" size_t metis_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_seq_len,
                                               int partition_size) {
  if (partition_size <= 0 || num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_seq_len <= 0) return 0;
  const size_t parts = split_parts(max_seq_len, partition_size);
  const size_t units = (size_t)num_seqs * num_heads * parts;
  return align_up(units * head_dim * sizeof(float), 256) + align_up(units * sizeof(float), 256);
}

namespace metis {

static int paged_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        const int32_t* seq_lens, void* out, float* lse_out, int num_seqs, int num_heads,
                        int num_kv_heads, int head_dim, int block_size, int max_blocks, int num_blocks, int dtype,
                        float scale, int partition_size, int max_seq_len, void* workspace, size_t workspace_bytes,
                        void* stream, bool merge) {
  clear_error();
  if (num_seqs < 0) return fail(METIS_E_SHAPE, "num_seqs < 0");
  if (num_seqs == 0) return METIS_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || (merge && !out))
    return fail(METIS_E_NULL, "q, k_cache, v_cache, block_table, seq_lens and out are required");
  if (!merge && partition_size <= 0) return fail(METIS_E_SHAPE, "partials need partition_size > 0");
  if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_blocks <= 0 ||
      num_blocks <= 0 || max_seq_len <= 0)
    return fail(METIS_E_SHAPE, "sizes must be positive");
  if (num_heads % num_kv_heads) return fail(METIS_E_SHAPE, "num_heads %% num_kv_heads != 0");
  if (num_seqs > 65535 || num_kv_heads > 65535) return fail(METIS_E_SHAPE, "num_seqs and num_kv_heads must be <= 65535");
  if ((long long)max_blocks * block_size > 0x7fffffffLL || (long long)num_blocks * block_size > 0x7fffffffLL)
    return fail(METIS_E_SHAPE, "max_blocks * block_size and num_blocks * block_size must fit in int32");
  if (head_dim != 64 && head_dim != 128) return fail(METIS_E_UNSUPPORTED, "head_dim must be 64 or 128");
  if (block_size != 16 && block_size != 32 && block_size != 64)
    return fail(METIS_E_UNSUPPORTED, "block_size must be 16, 32 or 64");
  const int r = num_heads / num_kv_heads;
  if (dtype != METIS_F32 && dtype != METIS_BF16) return fail(METIS_E_UNSUPPORTED, "dtype must be METIS_F32 or METIS_BF16");
  if (r > 8) return fail(METIS_E_UNSUPPORTED, "num_heads / num_kv_heads must be <= 8");
  if (dtype == METIS_BF16 && (r & (r - 1))) return fail(METIS_E_UNSUPPORTED, "bf16 needs a head ratio of 1, 2, 4 or 8");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(lse_out, 4))
    return fail(METIS_E_ALIGN, "tensors must be 16-byte aligned (block_table, seq_lens, lse_out: 4-byte)");
  if (partition_size < 0 || (partition_size % kUnit))
    return fail(METIS_E_SHAPE, "partition_size must be 0 or a positive multiple of 16");
  if (!(scale == scale)) return fail(METIS_E_SHAPE, "scale is NaN");

  const int eff_len = effective_max_len(max_seq_len, max_blocks, block_size);
  const size_t parts = split_parts(eff_len, partition_size);
  if (parts > 0x7fffffff) return fail(METIS_E_SHAPE, "too many partitions");
  const size_t need = metis_decode_workspace_bytes(num_seqs, num_heads, head_dim, eff_len, partition_size);
  if (need && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
    return fail(METIS_E_WORKSPACE, "workspace must hold %zu bytes (256-byte aligned)", need);

  DecodeParams p;
  p.q = q;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.lse_out = lse_out;
  p.S = num_seqs;
  p.H = num_heads;
  p.G = num_kv_heads;
  p.D = head_dim;
  p.bs = block_size;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.r = r;
  p.scale_log2 = scale * kLog2e;
  p.partition_size = partition_size;
  p.max_parts = parts ? (int)parts : 1;
  p.cap = eff_len;
  p.rows = nullptr;
  if (parts) {
    const size_t units = (size_t)num_seqs * num_heads * parts;
    p.part_out = reinterpret_cast<float*>(workspace);
    p.part_lse = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) +
                                          align_up(units * head_dim * sizeof(float), 256));
  } else {
    p.part_out = nullptr;
    p.part_lse = nullptr;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid((unsigned)p.max_parts, (unsigned)num_kv_heads, (unsigned)num_seqs);

  int rc;
  if (dtype == METIS_F32) {
    const float* kc = reinterpret_cast<const float*>(k_cache);
    const float* vc = reinterpret_cast<const float*>(v_cache);
    rc = head_dim == 64 ? launch_dependent(decode_f32_kernel<64>, grid, dim3(kF32Warps * 32), 0, st,
                                           "decode_f32_kernel launch", kc, vc, p)
                        : launch_dependent(decode_f32_kernel<128>, grid, dim3(kF32Warps * 32), 0, st,
                                           "decode_f32_kernel launch", kc, vc, p);
  } else {
    rc = head_dim == 64 ? launch_bf16<64>(p, k_cache, v_cache, grid, st) : launch_bf16<128>(p, k_cache, v_cache, grid, st);
  }
  if (rc) return rc;
  if (parts && merge)
    rc = launch_merge(p.part_out, p.part_lse, seq_lens, partition_size, out, lse_out, num_seqs, num_heads, head_dim,
                      p.max_parts, dtype, st);
  return rc;
}

}  // namespace metis

extern "C" int metis_paged_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* seq_lens, void* out,
                                       float* lse_out, int num_seqs, int num_heads, int num_kv_heads,
                                       int head_dim, int block_size, int max_blocks, int num_blocks, int dtype,
                                       float scale, int partition_size, int max_seq_len, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  return metis::paged_decode(q, k_cache, v_cache, block_table, seq_lens, out, lse_out, num_seqs, num_heads,
                             num_kv_heads, head_dim, block_size, max_blocks, num_blocks, dtype, scale, partition_size,
                             max_seq_len, workspace, workspace_bytes, stream, true);
}

extern "C" int metis_paged_attn_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                                                const int32_t* block_table, const int32_t* seq_lens,
                                                int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                int block_size, int max_blocks, int num_blocks, int dtype,
                                                float scale, int partition_size, int max_seq_len, void* workspace,
                                                size_t workspace_bytes, void* stream) {
  return metis::paged_decode(q, k_cache, v_cache, block_table, seq_lens, nullptr, nullptr, num_seqs, num_heads,
                             num_kv_heads, head_dim, block_size, max_blocks, num_blocks, dtype, scale, partition_size,
                             max_seq_len, workspace, workspace_bytes, stream, false);
}

extern "C" int metis_merge_attn_states(const float* part_out, const float* part_lse, const int32_t* seq_lens,
                                       int partition_size, void* out, float* lse_out, int num_seqs, int num_heads,
                                       int head_dim, int max_parts, int out_dtype, void* stream) {
  clear_error();
  if (num_seqs < 0) return fail(METIS_E_SHAPE, "num_seqs < 0");
  if (num_seqs == 0) return METIS_OK;
  if (!part_out || !part_lse || !seq_lens || !out)
    return fail(METIS_E_NULL, "part_out, part_lse, seq_lens and out are required");
  if (num_heads <= 0 || head_dim <= 0 || max_parts <= 0 || partition_size <= 0)
    return fail(METIS_E_SHAPE, "sizes must be positive");
  if (head_dim % 4 || head_dim > kMergeMaxD) return fail(METIS_E_UNSUPPORTED, "head_dim must be a multiple of 4 up to 512");
  if (out_dtype != METIS_F32 && out_dtype != METIS_BF16) return fail(METIS_E_UNSUPPORTED, "bad out_dtype");
  if ((size_t)num_seqs * num_heads > 0x7fffffffull) return fail(METIS_E_SHAPE, "num_seqs * num_heads too large");
  if (!aligned(part_out, 16) || !aligned(out, out_dtype == METIS_F32 ? 16 : 8) || !aligned(part_lse, 4) ||
      !aligned(seq_lens, 4) || !aligned(lse_out, 4))
    return fail(METIS_E_ALIGN, "misaligned pointer");
  return launch_merge(part_out, part_lse, seq_lens, partition_size, out, lse_out, num_seqs, num_heads, head_dim,
                      max_parts, out_dtype, reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Decode with the library's own static scratch, for callers that cannot
// allocate device memory.
// ---------------------------------------------------------------------------
namespace metis {

// Split-KV partials (part_out + part_lse) of one call.  Module-scope device
// memory: every GPU that loads the library holds these bytes until the process
// exits.  All calls share it, and it keeps whatever the last call left; the
// decode writes every partial the merge reads, so nothing needs clearing.
constexpr size_t kNoAllocScratchBytes = METIS_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's name is only a host-side stand-in in host code: its device
// address is looked up with cudaGetSymbolAddress (with the device current) and
// cached per device together with the context it was looked up in.  A new
// primary context on that device (after cudaDeviceReset, say) loads the module
// afresh, so a context that differs from the cached one triggers a new lookup.
constexpr int kNoAllocMaxDevices = 64;
struct NoAllocAddr {
  CUcontext ctx;
  void* ptr;
};
static NoAllocAddr g_noalloc[kNoAllocMaxDevices];
static std::mutex g_noalloc_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
static CtxGetCurrentFn g_ctx_get_current = nullptr;
static std::once_flag g_ctx_once;

static void load_ctx_get_current() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
}

static int noalloc_scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(METIS_E_UNSUPPORTED, "device ordinal %d: the static scratch serves devices 0..%d", dev,
                kNoAllocMaxDevices - 1);
  std::call_once(g_ctx_once, load_ctx_get_current);
  if (!g_ctx_get_current) return fail(METIS_E_CUDA, "cuCtxGetCurrent unavailable from the driver");
  // null before the runtime has set up this device's context on this thread
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocAddr& slot = g_noalloc[dev];
  if (!slot.ptr || !ctx || slot.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // sets up the context if needed
    if (e != cudaSuccess) return fail(METIS_E_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return fail(METIS_E_CUDA, "no current CUDA context");
    slot.ctx = ctx;
    slot.ptr = p;
  }
  *out = slot.ptr;
  return METIS_OK;
}

}  // namespace metis

extern "C" int metis_paged_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                               const int32_t* block_table, const int32_t* seq_lens, void* out,
                                               float* lse_out, int num_seqs, int num_heads, int num_kv_heads,
                                               int head_dim, int block_size, int max_blocks, int num_blocks,
                                               int dtype, float scale, int partition_size, int max_seq_len,
                                               void* stream) {
  clear_error();
  // scratch for the partitions the call will launch (max_seq_len clamped to
  // what a block-table row addresses, as the decode itself does)
  const int eff_len = max_blocks > 0 && block_size > 0 ? effective_max_len(max_seq_len, max_blocks, block_size) : 0;
  const size_t need = metis_decode_workspace_bytes(num_seqs, num_heads, head_dim, eff_len, partition_size);
  if (need > kNoAllocScratchBytes)
    return fail(METIS_E_WORKSPACE,
                "split-KV scratch of %zu bytes needed; the static scratch holds %zu bytes (use a larger "
                "partition_size, a smaller batch, or metis_paged_attn_decode with your own workspace)",
                need, kNoAllocScratchBytes);
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (need > 0) {
    const int rc = noalloc_scratch_address(&ws);
    if (rc) return rc;
    ws_bytes = kNoAllocScratchBytes;
  }
  return metis::paged_decode(q, k_cache, v_cache, block_table, seq_lens, out, lse_out, num_seqs, num_heads,
                             num_kv_heads, head_dim, block_size, max_blocks, num_blocks, dtype, scale, partition_size,
                             max_seq_len, ws, ws_bytes, stream, true);
}
