// Prefix-cache page lookup on the device: chained page keys, then
// lookup-or-allocate against an open-addressing table and a free-page stack.
//
// Prefix caching reuses the KV pages of an earlier prompt with the same leading
// tokens (vllm-metis 0.1.0 page, "How the model maps onto vLLM", "Caches", and
// "Status": prefix-cache hits).  Page b of a sequence is found by
//   local_b = fold over its tokens of  x = mix64(x XOR token),  x0 = 0x9E3779B97F4A7C15
//   key_b   = mix64(key_{b-1} XOR local_b),  key_{-1} = 0,  a key of 0 becomes 1
// (mix64: splitmix64's output function, Steele, Lea and Flood 2014), and the
// keys of a batch are looked up in page order: a key in the table is a hit
// (page reused, reference count + 1); a new key takes the page on top of the
// free stack (reference count 1); a key repeated in the batch is new only at its
// first occurrence; with the stack empty a new key gets page -1.
//
// The order rule is kept exactly without any thread waiting on another: a
// claim kernel inserts each new key with atomicCAS and records the lowest batch
// index per new slot with atomicMin (that index owns the slot); the owners are
// ranked in batch order by a reduce-then-scan over CTAs and take stack pages
// top down; a resolve kernel reads every key's page.  Kernel boundaries are the
// only synchronisation (each later kernel is a programmatic dependent launch
// that waits for its predecessor before touching memory).
#include <limits.h>

#include "../../include/metis_attn.h"
#include "common.cuh"
#include "host.h"

namespace metis {

__device__ unsigned int g_status_prefix = 0;

constexpr uint64_t kSeed = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// The sequence holding page i: the last s with cu_pages[s] <= i (-1 if none),
// found from the guess i * S / total by galloping, then bisection -- a few
// loads for any length mix instead of log2(S) dependent ones.
__device__ __forceinline__ int seq_of_page(const int32_t* __restrict__ cu, int S, int total, int i) {
  int g = (int)(((long long)i * S) / (total > 0 ? total : 1));
  g = min(max(g, 0), S - 1);
  int lo, hi;  // cu[lo] <= i (or lo == -1) and cu[hi] > i (or hi == S)
  if (cu[g] <= i) {
    lo = g;
    for (int step = 1;; step <<= 1) {
      hi = lo + step;
      if (hi >= S) {
        hi = S;
        break;
      }
      if (cu[hi] > i) break;
      lo = hi;
    }
  } else {
    hi = g;
    for (int step = 1;; step <<= 1) {
      lo = hi - step;
      if (lo < 0) {
        lo = -1;
        break;
      }
      if (cu[lo] <= i) break;
      hi = lo;
    }
  }
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= i) lo = mid;
    else hi = mid;
  }
  return lo;
}

// one thread per full page: fold its tokens into keys[i] (the local hash).
// A warp's 32 consecutive pages lie in a short stretch of the token array; the
// warp copies that stretch into shared memory with coalesced loads (one padding
// word per 16 so that 16-token pages read without bank conflicts) and folds from
// there; a stretch too long for the buffer is folded from global memory.
constexpr int kLocalWarps = 8;
constexpr int kStageSpan = 1024;                             // tokens per warp
constexpr int kStageWords = kStageSpan + kStageSpan / 16;    // with padding
__global__ void __launch_bounds__(kLocalWarps * 32)
    prefix_local_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ cu_tokens,
                        const int32_t* __restrict__ cu_pages, int S, int bs, int total, uint64_t* __restrict__ keys) {
  __shared__ int32_t stage[kLocalWarps][kStageWords];
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i = (blockIdx.x * kLocalWarps + warp) * 32 + lane;
  if ((blockIdx.x * kLocalWarps + warp) * 32 >= total) return;  // whole warp idle
  bool ok = false;
  int start = 0;
  if (i < total) {
    const int s = seq_of_page(cu_pages, S, total, i);
    if (s >= 0) {
      const long long b = (long long)i - cu_pages[s];
      const long long t0 = cu_tokens[s];
      ok = t0 >= 0 && (b + 1) * bs <= (long long)cu_tokens[s + 1] - t0;
      start = ok ? (int)(t0 + b * bs) : 0;
    }
    if (!ok) {
      atomicOr(&g_status_prefix, METIS_STATUS_BAD_OFFSETS);  // cu_pages disagrees with cu_tokens
      keys[i] = 0;
    }
  }
  int lo = ok ? start : INT_MAX, hi = ok ? start + bs : INT_MIN;
  for (int off = 16; off; off >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
  }
  if (lo > hi) return;  // no page of this warp is readable
  uint64_t x = kSeed;
  if ((long long)hi - lo <= kStageSpan) {
    int32_t* st = stage[warp];
    for (int w = lane; w < hi - lo; w += 32) st[w + (w >> 4)] = __ldg(tokens + lo + w);
    __syncwarp();
    if (!ok) return;
    const int base = start - lo;
#pragma unroll 4
    for (int k = 0; k < bs; ++k) {
      const int w = base + k;
      x = mix64(x ^ (uint64_t)(uint32_t)st[w + (w >> 4)]);
    }
  } else {
    if (!ok) return;
    const int32_t* t = tokens + start;
#pragma unroll 4
    for (int k = 0; k < bs; ++k) x = mix64(x ^ (uint64_t)(uint32_t)__ldg(t + k));
  }
  keys[i] = x;
}

// one thread per sequence: chain the local hashes of its pages in place, in
// register batches of 8 with the next batch's loads in flight
constexpr int kChainThreads = 64;
constexpr int kChainBatch = 8;
__global__ void __launch_bounds__(kChainThreads)
    prefix_chain_kernel(const int32_t* __restrict__ cu_pages, int S, int total, uint64_t* keys) {
  pdl_wait();
  const int s = blockIdx.x * kChainThreads + threadIdx.x;
  if (s >= S) return;
  const int p0 = max(cu_pages[s], 0), p1 = min(cu_pages[s + 1], total);
  uint64_t cur[kChainBatch], nxt[kChainBatch];
#pragma unroll
  for (int u = 0; u < kChainBatch; ++u) cur[u] = p0 + u < p1 ? keys[p0 + u] : 0;
  uint64_t key = 0;
  for (int base = p0; base < p1; base += kChainBatch) {
#pragma unroll
    for (int u = 0; u < kChainBatch; ++u) {
      const int j = base + kChainBatch + u;
      nxt[u] = j < p1 ? keys[j] : 0;
    }
#pragma unroll
    for (int u = 0; u < kChainBatch; ++u) {
      if (base + u < p1) {
        key = mix64(key ^ cur[u]);
        if (key == 0) key = 1;
        keys[base + u] = key;
      }
    }
#pragma unroll
    for (int u = 0; u < kChainBatch; ++u) cur[u] = nxt[u];
  }
}

__global__ void prefix_table_init_kernel(uint64_t* keys, int32_t* pages, int32_t* claim, int cap) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= cap) return;
  keys[i] = 0;
  pages[i] = -1;
  claim[i] = INT_MAX;
}

// one thread per batch key: find or insert its slot; new slots keep the lowest batch index
__global__ void prefix_claim_kernel(const uint64_t* __restrict__ batch, int n, uint64_t* table_keys,
                                    const int32_t* table_pages, int32_t* claim, int cap, int32_t* slot_of,
                                    int32_t* done) {
  pdl_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) *done = 0;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint64_t k = batch[i] ? batch[i] : 1ull;  // 0 marks an empty slot; hashing never yields it
  const unsigned mask = (unsigned)cap - 1u;
  unsigned slot = (unsigned)(k ^ (k >> 32)) & mask;
  int found = -1;
  for (int p = 0; p < cap; ++p, slot = (slot + 1u) & mask) {
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(&table_keys[slot]);
    if (cur == 0ull) cur = atomicCAS(reinterpret_cast<unsigned long long*>(&table_keys[slot]), 0ull, (unsigned long long)k);
    if (cur == 0ull || cur == (unsigned long long)k) {
      found = (int)slot;
      break;
    }
  }
  slot_of[i] = found;
  if (found < 0) {
    atomicOr(&g_status_prefix, METIS_STATUS_TABLE_FULL);
    return;
  }
  if (table_pages[found] < 0) atomicMin(&claim[found], i);  // new in this batch
}

// The owner of a new slot is its lowest batch index.  Owners are ranked in batch
// order by reduce-then-scan: every CTA counts its owners, the last CTA to finish
// scans the counts (a CTA learns it is last from a completion counter that the
// claim kernel zeroes), then each CTA ranks its own owners on top of its offset.
constexpr int kLookupThreads = 256;

// grid, one thread per key: owner flag and the CTA's owner count; the last CTA
// turns the counts into exclusive offsets, saves the clamped stack depth for the
// allocation pass and pops the pages taken
__global__ void __launch_bounds__(kLookupThreads)
    prefix_mark_kernel(int n, const int32_t* __restrict__ slot_of, const int32_t* table_pages,
                       const int32_t* claim, uint8_t* __restrict__ owner, int32_t* cta_count, int32_t* done,
                       int32_t* free_count, int free_capacity, int32_t* fc_saved) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int warp_sum[kLookupThreads / 32];
  __shared__ int carry;
  __shared__ bool last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i = blockIdx.x * kLookupThreads + tid;
  bool own = false;
  if (i < n) {
    const int slot = slot_of[i];
    own = slot >= 0 && table_pages[slot] < 0 && claim[slot] == i;
    owner[i] = own ? 1 : 0;
  }
  const int cnt = __syncthreads_count(own);
  if (tid == 0) {
    cta_count[blockIdx.x] = cnt;
    __threadfence();
    last = atomicAdd(done, 1) == (int)gridDim.x - 1;
    carry = 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int ctas = gridDim.x;
  for (int base = 0; base < ctas; base += kLookupThreads) {
    const int c = base + tid;
    const int v = c < ctas ? __ldcg(cta_count + c) : 0;
    int x = v;  // inclusive warp scan
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    int before = carry;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    if (c < ctas) cta_count[c] = before + x - v;
    __syncthreads();
    if (tid == kLookupThreads - 1) carry = before + x;
    __syncthreads();
  }
  if (tid == 0) {
    const int fc = min(max(*free_count, 0), free_capacity);
    *fc_saved = fc;
    *free_count = fc - min(carry, fc);
  }
}

// grid, one thread per key: an owner takes stack page (depth - 1 - rank)
__global__ void __launch_bounds__(kLookupThreads)
    prefix_alloc_kernel(int n, const int32_t* __restrict__ slot_of, const uint8_t* __restrict__ owner,
                        const int32_t* __restrict__ cta_offset, const int32_t* __restrict__ fc_saved,
                        int32_t* table_pages, int32_t* claim, const int32_t* __restrict__ free_stack,
                        int32_t* refcount, int num_pages) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int warp_cnt[kLookupThreads / 32];
  const int i = blockIdx.x * kLookupThreads + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool own = i < n && owner[i];
  const unsigned ball = __ballot_sync(0xffffffffu, own);
  if (lane == 0) warp_cnt[warp] = __popc(ball);
  __syncthreads();
  if (!own) return;
  int rank = cta_offset[blockIdx.x] + __popc(ball & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) rank += warp_cnt[w];
  const int slot = slot_of[i];
  const int pos = *fc_saved - 1 - rank;
  if (pos >= 0) {
    const int page = free_stack[pos];
    if (page >= 0 && page < num_pages) {
      table_pages[slot] = page;
      refcount[page] = 1;
    } else {
      atomicOr(&g_status_prefix, METIS_STATUS_BAD_BLOCK_ID);
    }
  } else {
    atomicOr(&g_status_prefix, METIS_STATUS_OUT_OF_PAGES);
  }
  claim[slot] = INT_MAX;  // ready for the next batch
}

// grid, one thread per key: its page and whether it was a hit
__global__ void __launch_bounds__(kLookupThreads)
    prefix_resolve_kernel(int n, const int32_t* __restrict__ slot_of, const int32_t* table_pages,
                          const uint8_t* __restrict__ owner, int32_t* refcount, int num_pages,
                          int32_t* __restrict__ pages_out, uint8_t* __restrict__ hits_out) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * kLookupThreads + threadIdx.x;
  if (i >= n) return;
  const int slot = slot_of[i];
  const int page = slot >= 0 ? table_pages[slot] : -1;
  const bool hit = page >= 0 && !owner[i];
  if (hit && page < num_pages) atomicAdd(&refcount[page], 1);
  pages_out[i] = page;
  hits_out[i] = hit ? 1 : 0;
}

int prefix_status(uint32_t* bits, int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_status_prefix, sizeof(v));
  if (e == cudaSuccess && clear) {
    unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_status_prefix, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  *bits |= v;
  return METIS_OK;
}

static int lookup_ctas(int n) { return (n + kLookupThreads - 1) / kLookupThreads; }

// workspace: slot_of int32[n] | owner uint8[n] | CTA counts int32[ctas] | saved stack depth, completion counter
static size_t lookup_ws(int n) {
  return align_up((size_t)n * 4, 256) + align_up((size_t)n, 256) + align_up((size_t)lookup_ctas(n) * 4, 256) + 256;
}

}  // namespace metis

using namespace metis;

extern "C" int metis_prefix_block_hashes(const int32_t* token_ids, const int32_t* cu_tokens, const int32_t* cu_pages,
                                         int num_seqs, int block_size, int total_pages, uint64_t* keys_out,
                                         void* stream) {
  clear_error();
  if (num_seqs < 0 || total_pages < 0) return fail(METIS_E_SHAPE, "num_seqs and total_pages must be >= 0");
  if (num_seqs == 0 || total_pages == 0) return METIS_OK;
  if (!token_ids || !cu_tokens || !cu_pages || !keys_out) return fail(METIS_E_NULL, "all pointers are required");
  if (block_size <= 0) return fail(METIS_E_SHAPE, "block_size must be positive");
  if (!aligned(token_ids, 4) || !aligned(cu_tokens, 4) || !aligned(cu_pages, 4) || !aligned(keys_out, 8))
    return fail(METIS_E_ALIGN, "index arrays must be 4-byte aligned, keys_out 8-byte");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int local_ctas = (total_pages + kLocalWarps * 32 - 1) / (kLocalWarps * 32);
  prefix_local_kernel<<<local_ctas, kLocalWarps * 32, 0, st>>>(token_ids, cu_tokens, cu_pages, num_seqs, block_size,
                                                               total_pages, keys_out);
  int rc = check_launch("prefix_local_kernel launch");
  if (rc) return rc;
  return launch_dependent(prefix_chain_kernel, dim3((unsigned)((num_seqs + kChainThreads - 1) / kChainThreads)),
                          dim3(kChainThreads), 0, st,
                          "prefix_chain_kernel launch", cu_pages, num_seqs, total_pages, keys_out);
}

extern "C" int metis_prefix_table_init(uint64_t* table_keys, int32_t* table_pages, int32_t* table_claim, int capacity,
                                       void* stream) {
  clear_error();
  if (!table_keys || !table_pages || !table_claim) return fail(METIS_E_NULL, "table arrays are required");
  if (capacity <= 0 || (capacity & (capacity - 1))) return fail(METIS_E_SHAPE, "capacity must be a power of two");
  if (!aligned(table_keys, 8) || !aligned(table_pages, 4) || !aligned(table_claim, 4))
    return fail(METIS_E_ALIGN, "table_keys must be 8-byte aligned, the others 4-byte");
  prefix_table_init_kernel<<<(capacity + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      table_keys, table_pages, table_claim, capacity);
  return check_launch("prefix_table_init_kernel launch");
}

extern "C" size_t metis_prefix_lookup_workspace_bytes(int n) { return n > 0 ? lookup_ws(n) : 0; }

extern "C" int metis_prefix_lookup(const uint64_t* keys, int n, uint64_t* table_keys, int32_t* table_pages,
                                   int32_t* table_claim, int capacity, const int32_t* free_stack, int free_capacity,
                                   int32_t* free_count, int32_t* refcount, int num_pages, int32_t* pages_out,
                                   uint8_t* hits_out, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  if (n < 0) return fail(METIS_E_SHAPE, "n < 0");
  if (n == 0) return METIS_OK;
  if (!keys || !table_keys || !table_pages || !table_claim || !free_stack || !free_count || !refcount || !pages_out ||
      !hits_out)
    return fail(METIS_E_NULL, "all arrays are required");
  if (capacity <= 0 || (capacity & (capacity - 1))) return fail(METIS_E_SHAPE, "capacity must be a power of two");
  if (free_capacity < 0 || num_pages <= 0) return fail(METIS_E_SHAPE, "free_capacity >= 0 and num_pages > 0 required");
  if (!aligned(keys, 8) || !aligned(table_keys, 8) || !aligned(table_pages, 4) || !aligned(table_claim, 4) ||
      !aligned(free_stack, 4) || !aligned(free_count, 4) || !aligned(refcount, 4) || !aligned(pages_out, 4))
    return fail(METIS_E_ALIGN, "keys 8-byte, int32 arrays 4-byte aligned");
  if (!workspace || workspace_bytes < lookup_ws(n) || !aligned(workspace, 256))
    return fail(METIS_E_WORKSPACE, "workspace must hold %zu bytes (256-byte aligned)", lookup_ws(n));
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  int32_t* slot_of = reinterpret_cast<int32_t*>(ws);
  ws += align_up((size_t)n * 4, 256);
  uint8_t* owner = ws;
  ws += align_up((size_t)n, 256);
  int32_t* cta_count = reinterpret_cast<int32_t*>(ws);
  ws += align_up((size_t)lookup_ctas(n) * 4, 256);
  int32_t* fc_saved = reinterpret_cast<int32_t*>(ws);
  int32_t* done = fc_saved + 1;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int ctas = lookup_ctas(n);
  const dim3 grid((unsigned)ctas), block(kLookupThreads);
  prefix_claim_kernel<<<grid, block, 0, st>>>(keys, n, table_keys, table_pages, table_claim, capacity, slot_of, done);
  int rc = check_launch("prefix_claim_kernel launch");
  if (rc) return rc;
  rc = launch_dependent(prefix_mark_kernel, grid, block, 0, st, "prefix_mark_kernel launch", n,
                        (const int32_t*)slot_of, (const int32_t*)table_pages, (const int32_t*)table_claim, owner,
                        cta_count, done, free_count, free_capacity, fc_saved);
  if (rc) return rc;
  rc = launch_dependent(prefix_alloc_kernel, grid, block, 0, st, "prefix_alloc_kernel launch", n,
                        (const int32_t*)slot_of, (const uint8_t*)owner, (const int32_t*)cta_count,
                        (const int32_t*)fc_saved, table_pages, table_claim, free_stack, refcount, num_pages);
  if (rc) return rc;
  return launch_dependent(prefix_resolve_kernel, grid, block, 0, st, "prefix_resolve_kernel launch", n,
                          (const int32_t*)slot_of, (const int32_t*)table_pages, (const uint8_t*)owner, refcount,
                          num_pages, pages_out, hits_out);
}
