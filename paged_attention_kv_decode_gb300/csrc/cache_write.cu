// The paged KV-cache write: one step's new key/value rows into their pages.
//
// In front of every attention call the new tokens' keys and values go into the
// pages that the attention kernels then read through the block table (vLLM's
// cache manager owns one paged KV layer per attention layer: vllm-metis 0.1.0
// page, "How the model maps onto vLLM", "Caches"; the scheduler's block table
// addresses the pages: vllm-metal article, section 4).  Token n goes to slot
// s = slot_mapping[n] = block * block_size + offset; s < 0 is a padding token.
//
// For one (block, offset) the [num_kv_heads, head_dim] part of a
// [num_blocks, block_size, num_kv_heads, head_dim] cache is contiguous, and so
// is a token's row of the [num_tokens, num_kv_heads, head_dim] input: each token
// is two contiguous copies (K and V) of the same length, done with 16-byte
// vector loads and stores by one CTA per token.  HBM-bound: 2 reads + 2 writes
// of the row per token.  The MLA cache row [c_kv | k_pe] is assembled from the
// two inputs the same way.
#include "../../include/metis_attn.h"
#include "common.cuh"
#include "host.h"

namespace metis {

__device__ unsigned int g_status_cache = 0;

// row_vecs: 16-byte vectors per token row; total_slots = num_blocks * block_size
__global__ void __launch_bounds__(128) reshape_and_cache_kernel(const uint4* __restrict__ key,
                                                                const uint4* __restrict__ value,
                                                                uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                                const int64_t* __restrict__ slot_mapping,
                                                                int row_vecs, long long total_slots) {
  // The attention call that follows may start launching now: it waits for this
  // grid (pdl_wait) before it reads the cache.
  pdl_launch_dependents();
  const int n = blockIdx.x;
  const long long slot = slot_mapping[n];
  if (slot < 0) return;  // padding token
  if (slot >= total_slots) {
    if (threadIdx.x == 0) atomicOr(&g_status_cache, METIS_STATUS_BAD_BLOCK_ID);
    return;
  }
  const uint4* ks = key + (size_t)n * row_vecs;
  const uint4* vs = value + (size_t)n * row_vecs;
  uint4* kd = k_cache + (size_t)slot * row_vecs;
  uint4* vd = v_cache + (size_t)slot * row_vecs;
  for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) {
    const uint4 k = __ldg(ks + i);
    const uint4 v = __ldg(vs + i);
    kd[i] = k;
    vd[i] = v;
  }
}

// kv_cache row = [kv_c (lat_vecs vectors) | k_pe (rope_vecs vectors)]
__global__ void __launch_bounds__(128) mla_reshape_and_cache_kernel(const uint4* __restrict__ kv_c,
                                                                    const uint4* __restrict__ k_pe,
                                                                    uint4* __restrict__ kv_cache,
                                                                    const int64_t* __restrict__ slot_mapping,
                                                                    int lat_vecs, int rope_vecs,
                                                                    long long total_slots) {
  pdl_launch_dependents();  // as in reshape_and_cache_kernel
  const int n = blockIdx.x;
  const long long slot = slot_mapping[n];
  if (slot < 0) return;
  if (slot >= total_slots) {
    if (threadIdx.x == 0) atomicOr(&g_status_cache, METIS_STATUS_BAD_BLOCK_ID);
    return;
  }
  const int row_vecs = lat_vecs + rope_vecs;
  uint4* d = kv_cache + (size_t)slot * row_vecs;
  for (int i = threadIdx.x; i < row_vecs; i += blockDim.x)
    d[i] = i < lat_vecs ? __ldg(kv_c + (size_t)n * lat_vecs + i) : __ldg(k_pe + (size_t)n * rope_vecs + (i - lat_vecs));
}

// Test support: an mbarrier wait that nothing can complete (the barrier expects
// one arrival that never comes), bounded by limit_ns: the wait gives up, sets
// METIS_STATUS_WAIT_TIMEOUT and the kernel returns.  This is the give-up path of
// every pipeline wait in the library, run on purpose.
__global__ void __launch_bounds__(32) wait_probe_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait_for(&bar, 0, &g_status_cache, limit_ns);
}

int cache_status(uint32_t* bits, int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_status_cache, sizeof(v));
  if (e == cudaSuccess && clear) {
    unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_status_cache, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  *bits |= v;
  return METIS_OK;
}

static int threads_for(int row_vecs) { return row_vecs >= 128 ? 128 : ((row_vecs + 31) / 32) * 32; }

}  // namespace metis

using namespace metis;

extern "C" int metis_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                       const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                                       int block_size, int num_blocks, int dtype, void* stream) {
  clear_error();
  if (num_tokens < 0) return fail(METIS_E_SHAPE, "num_tokens < 0");
  if (num_tokens == 0) return METIS_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping)
    return fail(METIS_E_NULL, "key, value, k_cache, v_cache and slot_mapping are required");
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return fail(METIS_E_SHAPE, "sizes must be positive");
  if (dtype != METIS_F32 && dtype != METIS_BF16) return fail(METIS_E_UNSUPPORTED, "dtype must be METIS_F32 or METIS_BF16");
  const long long row_bytes = (long long)num_kv_heads * head_dim * (dtype == METIS_F32 ? 4 : 2);
  if (row_bytes % 16) return fail(METIS_E_UNSUPPORTED, "num_kv_heads * head_dim * element size must be a multiple of 16 bytes");
  if (row_bytes / 16 > 0x7fffffffLL) return fail(METIS_E_SHAPE, "token row too large");
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(METIS_E_ALIGN, "tensors must be 16-byte aligned (slot_mapping: 8-byte)");
  const int row_vecs = (int)(row_bytes / 16);
  reshape_and_cache_kernel<<<(unsigned)num_tokens, threads_for(row_vecs), 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(key), reinterpret_cast<const uint4*>(value), reinterpret_cast<uint4*>(k_cache),
      reinterpret_cast<uint4*>(v_cache), slot_mapping, row_vecs, (long long)num_blocks * block_size);
  return check_launch("reshape_and_cache_kernel launch");
}

extern "C" int metis_mla_reshape_and_cache(const void* kv_c, const void* k_pe, void* kv_cache,
                                           const int64_t* slot_mapping, int num_tokens, int d_latent, int d_rope,
                                           int block_size, int num_blocks, void* stream) {
  clear_error();
  if (num_tokens < 0) return fail(METIS_E_SHAPE, "num_tokens < 0");
  if (num_tokens == 0) return METIS_OK;
  if (!kv_c || !k_pe || !kv_cache || !slot_mapping)
    return fail(METIS_E_NULL, "kv_c, k_pe, kv_cache and slot_mapping are required");
  if (d_latent <= 0 || d_rope <= 0 || block_size <= 0 || num_blocks <= 0)
    return fail(METIS_E_SHAPE, "sizes must be positive");
  if ((d_latent * 2) % 16 || (d_rope * 2) % 16)
    return fail(METIS_E_UNSUPPORTED, "d_latent and d_rope must be multiples of 8 (16-byte bf16 rows)");
  if (!aligned(kv_c, 16) || !aligned(k_pe, 16) || !aligned(kv_cache, 16) || !aligned(slot_mapping, 8))
    return fail(METIS_E_ALIGN, "tensors must be 16-byte aligned (slot_mapping: 8-byte)");
  const int lat_vecs = d_latent * 2 / 16, rope_vecs = d_rope * 2 / 16;
  mla_reshape_and_cache_kernel<<<(unsigned)num_tokens, threads_for(lat_vecs + rope_vecs), 0,
                                 reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(kv_c), reinterpret_cast<const uint4*>(k_pe), reinterpret_cast<uint4*>(kv_cache),
      slot_mapping, lat_vecs, rope_vecs, (long long)num_blocks * block_size);
  return check_launch("mla_reshape_and_cache_kernel launch");
}

extern "C" int metis_debug_wait_probe(uint64_t limit_ns, void* stream) {
  clear_error();
  if (limit_ns == 0 || limit_ns > 1000000000ull)
    return fail(METIS_E_SHAPE, "limit_ns must be in (0, 1e9]");
  wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
  return check_launch("wait_probe_kernel launch");
}
