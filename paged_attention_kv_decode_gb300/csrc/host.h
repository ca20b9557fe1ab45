// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/metis_attn.h"

namespace metis {

// Record a message for metis_last_error() and return `code`.
int fail(int code, const char* fmt, ...);
void clear_error();

// cudaGetLastError() after a launch: METIS_OK, or METIS_E_CUDA with a message.
int check_launch(const char* what);

// Encode a tiled TMA descriptor (cuTensorMapEncodeTiled, fetched from the
// driver at run time).  dims / box are innermost first; strides are the byte
// strides of dims 1..rank-1.  Returns METIS_OK or an error code.
int encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle);

// Launch `kernel` as a programmatic dependent of the previous kernel in the
// stream: it may start launching while that kernel still runs, so it must
// execute pdl_wait() (common.cuh) before touching anything the previous kernel
// writes.  Returns METIS_OK or METIS_E_CUDA.
template <typename... KArgs, typename... Args>
int launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, const char* what,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) return fail(METIS_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return METIS_OK;
}

// Raise a kernel's dynamic shared memory limit once per device.
int set_max_dynamic_smem(const void* func, int bytes, int* done_mask);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Log-sum-exp merge of split partials [S, H, max_parts, D] (decode.cu); with
// skip_single, sequences with at most one partition are left untouched.
int launch_merge_ex(const float* part_out, const float* part_lse, const int32_t* seq_lens, int P, void* out,
                    float* lse_out, int S, int H, int D, int max_parts, int out_dtype, int skip_single,
                    cudaStream_t st);
// The merge of the sequences with two or more partitions only (the others were
// written directly): one CTA per SM lists them and takes their rows in turn.
// Falls back to launch_merge_ex(..., skip_single = 1) outside its reach.
int launch_merge_split_rows(const float* part_out, const float* part_lse, const int32_t* seq_lens, int P, void* out,
                            float* lse_out, int S, int H, int D, int max_parts, int out_dtype, int sms,
                            cudaStream_t st);

// The single-token sequences of a chunked-prefill batch through the bf16 decode
// kernel (decode.cu); rows = the batch's cu_q_lens.  Other sequences are skipped.
int launch_decode_rows(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* seq_lens, const int32_t* rows, void* out, float* lse_out, int S, int H, int G,
                       int D, int bs, int max_blocks, int num_blocks, float scale, int cap, cudaStream_t st);

// The same, persistent, beside the chunk kernel: one CTA per SM in a grid of `grid`
// CTAs, of which the first *n_ctas (device value, written by the prefill schedule
// kernel before this grid reads it) take (sequence, KV head) items from the
// counter *next_item (zeroed by that kernel); the others exit at once.  Every CTA
// lets the next grid launch only after waiting for the previous one.
int launch_decode_rows_beside(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                              const int32_t* seq_lens, const int32_t* rows, void* out, float* lse_out, int S, int H,
                              int G, int D, int bs, int max_blocks, int num_blocks, float scale, int cap,
                              const int* n_ctas, int* next_item, int grid, cudaStream_t st);

// Per-translation-unit device status words.
int decode_status(uint32_t* bits, int clear);
int prefill_status(uint32_t* bits, int clear);
int mla_status(uint32_t* bits, int clear);
int cache_status(uint32_t* bits, int clear);
int prefix_status(uint32_t* bits, int clear);

}  // namespace metis
