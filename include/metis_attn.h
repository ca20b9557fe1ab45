/*
 * metis_attn -- attention over a paged KV cache on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the one the vLLM plugin pages build on: paged attention
 * and MLA kernels fed by the scheduler's block tables and sequence lengths
 * (vllm-metal architecture article, sections 3 and 4), with prefix caching and
 * chunked prefill on the engine side (vllm-metis 0.1.0 page, introduction and
 * "How the model maps onto vLLM", "Caches").  The pages name the operation but
 * print no formula; every entry point computes textbook scaled-dot-product
 * softmax attention of each query row over the tokens its sequence has cached:
 *
 *     z_t = scale * q . k_t,   out = sum_t softmax(z)_t v_t,   lse = ln sum_t exp(z_t)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every tensor pointer is a DEVICE pointer owned by the caller; the
 *   library never allocates, frees, copies to or from the host, or
 *   synchronises inside a compute call, so calls can be captured in a CUDA
 *   graph.  Tensors are dense, row-major (C order), 16-byte aligned.
 * Stream.  `stream` is a cudaStream_t passed as void*; NULL is the legacy
 *   default stream.  Work is enqueued asynchronously on it.
 * KV pages.  k_cache / v_cache are [num_blocks, block_size, num_kv_heads,
 *   head_dim].  Logical token t of sequence s is in physical block
 *   block_table[s * max_blocks + t / block_size], slot t % block_size.
 *   block_table is int32 [num_seqs, max_blocks]; only its first
 *   ceil(seq_lens[s] / block_size) entries of row s are read.  seq_lens is
 *   int32 [num_seqs]: the number of cached tokens, INCLUDING the queried ones
 *   (their K/V must already be in the pages).  Page slots at or beyond
 *   seq_lens[s] are never used, so they may hold anything (NaN included).
 * GQA.  q head h reads kv head h / (num_heads / num_kv_heads).
 * dtype.  METIS_F32 or METIS_BF16; q, the caches and out share it.  All
 *   accumulation, the softmax statistics, lse and split partials are fp32.
 * lse.  Natural-log log-sum-exp of the scaled scores, fp32; -inf for an
 *   empty sequence (whose output row is 0).
 * Errors.  Return 0 on success.  A negative METIS_E_* code means the
 *   arguments were rejected on the host and NOTHING was launched;
 *   metis_last_error() then holds a message.  METIS_E_CUDA means a launch
 *   failed.  Content errors that only the device can see (a block id outside
 *   [0, num_blocks), a sequence longer than its table row or than
 *   max_seq_len) never fault: the offending page reads as zeros, and a bit
 *   is set in the device status word read by metis_read_status().
 */
#ifndef METIS_ATTN_H
#define METIS_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtypes */
#define METIS_F32  0
#define METIS_BF16 1

/* status codes */
#define METIS_OK              0
#define METIS_E_NULL         -1  /* a required pointer is NULL */
#define METIS_E_SHAPE        -2  /* inconsistent or non-positive sizes */
#define METIS_E_UNSUPPORTED  -3  /* head_dim / block_size / head ratio / dtype not built */
#define METIS_E_ALIGN        -4  /* a pointer is not 16-byte aligned */
#define METIS_E_WORKSPACE    -5  /* workspace NULL or smaller than required */
#define METIS_E_CUDA         -6  /* a CUDA call failed (message in metis_last_error) */

/* device status word bits (metis_read_status) */
#define METIS_STATUS_BAD_BLOCK_ID  1u  /* a block id outside [0, num_blocks) */
#define METIS_STATUS_SEQ_TOO_LONG  2u  /* seq_lens[s] > max_blocks * block_size or > max_seq_len */
#define METIS_STATUS_WAIT_TIMEOUT  4u  /* a pipeline wait gave up (a library bug) */
#define METIS_STATUS_BAD_Q_LEN     8u  /* prefill: q_len > seq_len or a negative q_len */
#define METIS_STATUS_TABLE_FULL   16u  /* prefix lookup: a key found no free table slot */
#define METIS_STATUS_OUT_OF_PAGES 32u  /* prefix lookup: a new key found the free stack empty */
#define METIS_STATUS_BAD_OFFSETS  64u  /* page keys: cu_pages asks for a page past its sequence's tokens */

/*
 * metis_paged_attn_decode -- one query token per sequence over its pages
 * (the paged-attention kernel of the vllm-metal article, section 3, fed by
 * the block table and sequence lengths of section 4).
 *
 *   q            [num_seqs, num_heads, head_dim]      dtype
 *   k_cache      [num_blocks, block_size, num_kv_heads, head_dim]
 *   v_cache      same shape as k_cache
 *   block_table  int32 [num_seqs, max_blocks]
 *   seq_lens     int32 [num_seqs]; the query is the last cached token
 *   out          [num_seqs, num_heads, head_dim]      dtype (written)
 *   lse_out      fp32 [num_seqs, num_heads] or NULL   (written when non-NULL)
 *   scale        softmax scale (e.g. 1/sqrt(head_dim))
 *   partition_size
 *                0: one pass over each sequence.  > 0: split-KV -- tokens
 *                [p*P, (p+1)*P) form partition p; each partition's normalised
 *                partial output and lse go to the workspace, then
 *                metis_merge_attn_states' kernel combines them on the same
 *                stream.  Must be a positive multiple of 16.
 *   max_seq_len  host-side upper bound on seq_lens (sizes the grid); tokens
 *                beyond it are not read (status bit SEQ_TOO_LONG).
 *   workspace    device scratch of at least metis_decode_workspace_bytes(...)
 *                bytes (may be NULL when that is 0); contents need no
 *                initialisation and are clobbered.
 *
 * Supported: head_dim in {64, 128}; block_size in {16, 32, 64}; bf16 needs
 * num_heads / num_kv_heads in {1, 2, 4, 8}; fp32 any ratio up to 8.
 * num_seqs == 0 is a successful no-op.
 */
int metis_paged_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_table, const int32_t* seq_lens,
                            void* out, float* lse_out,
                            int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks, int num_blocks, int dtype,
                            float scale, int partition_size, int max_seq_len,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * metis_paged_attn_decode_partials -- the first half of a split-KV decode:
 * the same arguments as metis_paged_attn_decode without out / lse_out, and
 * partition_size must be > 0.  Writes each partition's normalised partial
 * output and lse into the workspace and launches nothing else; the second
 * half is metis_merge_attn_states over
 *
 *   part_out = (float*)workspace                       [num_seqs, num_heads, max_parts, head_dim]
 *   part_lse = (float*)((char*)workspace + align256(4 * num_seqs * num_heads * max_parts * head_dim))
 *                                                       [num_seqs, num_heads, max_parts]
 *
 * with max_parts = ceil(max_seq_len / partition_size).  Partitions past a
 * sequence's end are not written (the merge does not read them).
 */
int metis_paged_attn_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* seq_lens,
                                     int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                     int block_size, int max_blocks, int num_blocks, int dtype,
                                     float scale, int partition_size, int max_seq_len,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * metis_paged_attn_decode_noalloc -- metis_paged_attn_decode for callers that
 * cannot allocate device memory.
 *
 * The pages have no counterpart of this call: it exists for callers that
 * cannot call cudaMalloc -- a host framework that owns all device memory and
 * hands its plugins no allocator, or a latency-critical path that cannot take
 * the implicit device synchronisation of an allocation.  Arguments and
 * results are those of metis_paged_attn_decode, without the workspace: the
 * split-KV partials go to a scratch array of METIS_NOALLOC_SCRATCH_BYTES
 * (64 MiB) that the library itself declares in device memory.
 *
 *  - Nothing is allocated or freed: no cudaMalloc / cudaFree, no allocating
 *    library routine.  The caller still passes q, the caches, the tables and
 *    out / lse_out.
 *  - Every GPU that loads the library holds the 64 MiB until the process
 *    exits.
 *  - A split that needs more than METIS_NOALLOC_SCRATCH_BYTES
 *    (metis_decode_workspace_bytes(...) > the limit, with max_seq_len clamped
 *    to max_blocks * block_size) is rejected with METIS_E_WORKSPACE and
 *    nothing is launched.  partition_size 0 needs no scratch.
 *  - The first split call on a device looks up the array's device address
 *    for that device (cudaGetSymbolAddress) and caches it with the current
 *    CUDA context; a call under a different context (after cudaDeviceReset,
 *    say) looks it up again.  Make the first call on a device, and the first
 *    after a context change, before any stream capture.
 *  - Every call shares the one array.  Calls whose work overlaps on the GPU
 *    (other streams, other threads, without ordering between them) race on
 *    it and give wrong results; calls in one stream are ordered and safe.
 *    The array keeps the last call's contents; nothing in it needs clearing,
 *    because each call writes every partial it reads.
 */
#define METIS_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int metis_paged_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_table, const int32_t* seq_lens,
                                    void* out, float* lse_out,
                                    int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                    int block_size, int max_blocks, int num_blocks, int dtype,
                                    float scale, int partition_size, int max_seq_len, void* stream);

/* Bytes of workspace metis_paged_attn_decode needs (0 when partition_size == 0). */
size_t metis_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                    int max_seq_len, int partition_size);

/*
 * metis_paged_attn_prefill_chunk -- chunked prefill over a paged KV cache with
 * a cached prefix (vllm-metis 0.1.0 page, introduction and "How the model maps
 * onto vLLM -> Caches": prefix caching and chunked prefill; chunk sizes of the
 * vllm-mblt 0.8.0 page, "Chunked Prefill Auto-Tuning"), mixed freely with
 * single-token decodes (q_len = 1).
 *
 * Sequence s holds L = seq_lens[s] cached tokens whose K/V are already in the
 * pages; its last q_len = cu_q_lens[s+1] - cu_q_lens[s] tokens are queried.
 * Query row i of the sequence sits at position L - q_len + i and attends to
 * every key t <= L - q_len + i: the whole cached prefix plus a causal mask
 * inside the chunk (bottom-right aligned; with no prefix this is plain causal
 * attention, and splitting a prompt into chunks does not change the result).
 *
 *   q          [num_tokens, num_heads, head_dim] bf16; the sequences' query
 *              rows back to back, sequence s at rows cu_q_lens[s] ..
 *   cu_q_lens  int32 [num_seqs + 1], cu_q_lens[0] = 0, non-decreasing,
 *              cu_q_lens[num_seqs] = num_tokens
 *   k_cache, v_cache, block_table, seq_lens   as for metis_paged_attn_decode
 *   out        [num_tokens, num_heads, head_dim] bf16 (written)
 *   lse_out    fp32 [num_tokens, num_heads] or NULL
 *   max_seq_len  host-side upper bound on seq_lens
 *   workspace  >= metis_prefill_workspace_bytes(...) bytes, 256-byte aligned,
 *              no initialisation needed (holds the tile schedule)
 *
 * Supported: dtype METIS_BF16 (tensor cores: bf16 operands, fp32 accumulation);
 * head_dim 64 or 128; block_size 16, 32 or 64; num_heads / num_kv_heads in
 * {1, 2, 4, 8, 16}.  A q_len larger than the sequence length is clamped to it
 * (status bit METIS_STATUS_BAD_Q_LEN).  num_seqs == 0 or num_tokens == 0 is a
 * successful no-op.
 */
int metis_paged_attn_prefill_chunk(const void* q, const int32_t* cu_q_lens,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   void* out, float* lse_out,
                                   int num_seqs, int num_tokens, int num_heads, int num_kv_heads,
                                   int head_dim, int block_size, int max_blocks, int num_blocks,
                                   int dtype, float scale, int max_seq_len,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace metis_paged_attn_prefill_chunk needs (0 for invalid sizes). */
size_t metis_prefill_workspace_bytes(int num_seqs, int num_tokens, int num_heads, int num_kv_heads);

/*
 * metis_mla_decode -- multi-head latent attention decode over a paged latent
 * cache (the MLA kernel of the vllm-metal article, section 3, fed by the block
 * table and sequence lengths of section 4).
 *
 * All heads share one latent cache whose rows are [c_kv (d_latent) | k_pe
 * (d_rope)]; queries arrive already in latent space.  For head h of sequence s:
 *   z_t = scale * q[s,h,:] . kv[t, 0:d_latent+d_rope]
 *   out[s,h,:] = sum_t softmax(z)_t kv[t, 0:d_latent]
 *
 *   q          [num_seqs, num_heads, d_latent + d_rope] bf16
 *   kv_cache   [num_blocks, block_size, d_latent + d_rope] bf16
 *   block_table, seq_lens   as for metis_paged_attn_decode
 *   out        [num_seqs, num_heads, d_latent] bf16 (written), 32-byte aligned
 *   lse_out    fp32 [num_seqs, num_heads] or NULL
 *   partition_size  0: one pass per sequence; > 0 (a multiple of 32): tokens
 *              are split into partitions of that size, computed in parallel and
 *              merged by log-sum-exp (a sequence with one partition is written
 *              directly)
 *   workspace  >= metis_mla_workspace_bytes(...) bytes, 256-byte aligned, no
 *              initialisation needed
 *
 * Supported: d_latent 512, d_rope 64; num_heads a multiple of 128, or a
 * multiple of 16 below 128; block_size 16, 32 or 64.  Tensor cores: bf16
 * operands, fp32 accumulation.  Persistent clusters of two CTAs (two SMs), one
 * per SM pair, split the key dimensions and the output columns of each work
 * item (a sequence, or a partition of one) and walk their share of the items.
 * The two halves of each score (288 key dimensions each, accumulated in fp32)
 * are scaled by scale * log2(e) and rounded to fp16 before they are added, so a
 * score carries an extra error of at most 2^-11 (|S_0| + |S_1|) in log2 units.
 */
int metis_mla_decode(const void* q, const void* kv_cache,
                     const int32_t* block_table, const int32_t* seq_lens,
                     void* out, float* lse_out,
                     int num_seqs, int num_heads, int d_latent, int d_rope,
                     int block_size, int max_blocks, int num_blocks, float scale,
                     int partition_size, int max_seq_len,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace metis_mla_decode needs. */
size_t metis_mla_workspace_bytes(int num_seqs, int num_heads, int max_seq_len, int partition_size);

/*
 * metis_merge_attn_states -- the log-sum-exp merge of split-KV partials:
 *
 *   lse = m + ln sum_p exp(lse_p - m),  m = max_p lse_p
 *   out = sum_p exp(lse_p - lse) * o_p
 *
 * over partitions p < min(ceil(seq_lens[s] / partition_size), max_parts);
 * partitions with lse_p = -inf weigh nothing, and a sequence with no
 * partition gets out = 0, lse = -inf.
 *
 *   part_out   fp32 [num_seqs, num_heads, max_parts, head_dim] (normalised o_p)
 *   part_lse   fp32 [num_seqs, num_heads, max_parts]            (natural log)
 *   seq_lens   int32 [num_seqs]
 *   out        [num_seqs, num_heads, head_dim] in out_dtype (written)
 *   lse_out    fp32 [num_seqs, num_heads] or NULL
 *
 * Supported: head_dim a multiple of 4 up to 512.
 */
int metis_merge_attn_states(const float* part_out, const float* part_lse, const int32_t* seq_lens,
                            int partition_size, void* out, float* lse_out,
                            int num_seqs, int num_heads, int head_dim, int max_parts,
                            int out_dtype, void* stream);

/*
 * metis_reshape_and_cache -- write one step's new key/value rows into their
 * pages, the step in front of every attention call (vLLM's cache manager owns
 * one paged KV layer per attention layer: vllm-metis 0.1.0 page, "How the
 * model maps onto vLLM", "Caches"; the scheduler's block table addresses the
 * same pages: vllm-metal article, section 4).  For n < num_tokens with
 * slot = slot_mapping[n] >= 0:
 *   k_cache[slot / block_size, slot % block_size, :, :] = key[n, :, :]
 *   v_cache[slot / block_size, slot % block_size, :, :] = value[n, :, :]
 *
 *   key, value     [num_tokens, num_kv_heads, head_dim], dtype, contiguous
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim], dtype
 *   slot_mapping   int64 [num_tokens]: block id * block_size + offset; < 0 is a
 *                  padding token (not written)
 *   dtype          METIS_F32 or METIS_BF16 (a byte copy)
 * All pointers are caller-owned device memory, 16-byte aligned (slot_mapping
 * 8-byte); num_kv_heads * head_dim * element size must be a multiple of 16.
 * Two tokens with the same slot: one of the two rows is written (which one is
 * unspecified).  A slot >= num_blocks * block_size is not written and sets
 * METIS_STATUS_BAD_BLOCK_ID.  Returns METIS_OK or METIS_E_* (nothing launched);
 * num_tokens == 0 is a successful no-op.  Asynchronous on `stream`.
 */
int metis_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                            const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, int dtype, void* stream);

/*
 * metis_mla_reshape_and_cache -- the same write for the MLA latent cache
 * (vllm-metal article, section 3): row [c_kv | k_pe] of token n goes to
 *   kv_cache[slot / block_size, slot % block_size, 0 : d_latent] = kv_c[n, :]
 *   kv_cache[slot / block_size, slot % block_size, d_latent :]   = k_pe[n, :]
 *
 *   kv_c   bf16 [num_tokens, d_latent];  k_pe  bf16 [num_tokens, d_rope]
 *   kv_cache  bf16 [num_blocks, block_size, d_latent + d_rope]
 *   slot_mapping  int64 [num_tokens], as above
 * d_latent and d_rope multiples of 8; alignment, errors and status as above.
 */
int metis_mla_reshape_and_cache(const void* kv_c, const void* k_pe, void* kv_cache,
                                const int64_t* slot_mapping, int num_tokens, int d_latent, int d_rope,
                                int block_size, int num_blocks, void* stream);

/*
 * Prefix cache: page keys and lookup-or-allocate.  A new prompt reuses the KV
 * pages of an earlier prompt with the same leading tokens (vllm-metis 0.1.0
 * page, "How the model maps onto vLLM", "Caches": vLLM's cache manager runs
 * prefix caching; "Status": most of a repeated prompt's tokens come from the
 * cache).  The pages are those of the block table (vllm-metal article,
 * section 4).
 *
 * metis_prefix_block_hashes -- one chained 64-bit key per FULL page:
 *   local_b = fold over the page's tokens t of  x = mix64(x ^ (uint32)t),
 *             starting from x = 0x9E3779B97F4A7C15
 *   key_b   = mix64(key_{b-1} ^ local_b), key_{-1} = 0; a key of 0 becomes 1
 * with mix64 splitmix64's output function (Steele, Lea and Flood 2014), so a
 * key names a page's tokens and every token before them.
 *
 *   token_ids  int32 [cu_tokens[num_seqs]]: the sequences' tokens, concatenated
 *   cu_tokens  int32 [num_seqs + 1]: token offsets (cu_tokens[0] = 0)
 *   cu_pages   int32 [num_seqs + 1]: key offsets; cu_pages[s + 1] - cu_pages[s]
 *              must equal (cu_tokens[s + 1] - cu_tokens[s]) / block_size (the
 *              partial last page has no key) -- the caller computes it on the
 *              host, where it sizes keys_out
 *   total_pages  cu_pages[num_seqs]
 *   keys_out   uint64 [total_pages], sequence-major
 * A page that cu_pages places past its sequence's tokens is not read: its key
 * is 0 and METIS_STATUS_BAD_OFFSETS is set.
 * Device pointers, caller-owned; index arrays 4-byte aligned, keys_out
 * 8-byte.  num_seqs == 0 or total_pages == 0 is a successful no-op.
 *
 * metis_prefix_table_init -- empty an open-addressing table of `capacity`
 * slots (a power of two): table_keys[i] = 0 (0 is never a key),
 * table_pages[i] = -1, table_claim[i] = INT_MAX.  The three arrays are
 * caller-owned device memory that persists across lookups; table_claim is
 * scratch the lookup leaves at INT_MAX.
 *
 * metis_prefix_lookup -- look the n keys up in order (sequence-major, as
 * metis_prefix_block_hashes writes them), with the result of one-at-a-time
 * processing:
 *   a key whose slot holds a page p >= 0 is a hit: pages_out = p,
 *     hits_out = 1, refcount[p] += 1;
 *   otherwise the key is new; the FIRST new occurrence of a key in the batch
 *     takes the page on top of the free stack (free_stack[*free_count - 1],
 *     then the one below ...): pages_out = that page, hits_out = 0,
 *     refcount[page] = 1, and the slot keeps the page; later occurrences in
 *     the same batch are hits on it;
 *   a new key with the stack empty gets pages_out = -1, hits_out = 0 and
 *     sets METIS_STATUS_OUT_OF_PAGES; its slot keeps page -1, which later
 *     lookups treat as absent.
 *   keys         uint64 [n], none 0
 *   table_*      as metis_prefix_table_init left them (or earlier lookups)
 *   free_stack   int32 [free_capacity]: free page ids, the top at the end
 *   free_count   int32 (one device value): pages on the stack; decremented by
 *                the pages taken (read clamped to [0, free_capacity])
 *   refcount     int32 [num_pages]
 *   pages_out    int32 [n];  hits_out  uint8 [n]
 *   workspace    metis_prefix_lookup_workspace_bytes(n) bytes, 256-byte aligned
 * A key that finds no free table slot (probing wraps around) gets page -1 and
 * sets METIS_STATUS_TABLE_FULL; a stack entry outside [0, num_pages) is not
 * used and sets METIS_STATUS_BAD_BLOCK_ID.  Keeping the table at most half full
 * is the caller's job.  Device pointers, caller-owned; uint64 arrays 8-byte and
 * int32 arrays 4-byte aligned.  Returns METIS_OK or METIS_E_* (nothing
 * launched); n == 0 is a successful no-op.  All three calls are asynchronous on
 * `stream`, allocate nothing, and can be captured in a CUDA graph.
 */
int metis_prefix_block_hashes(const int32_t* token_ids, const int32_t* cu_tokens, const int32_t* cu_pages,
                              int num_seqs, int block_size, int total_pages, uint64_t* keys_out, void* stream);

int metis_prefix_table_init(uint64_t* table_keys, int32_t* table_pages, int32_t* table_claim, int capacity,
                            void* stream);

size_t metis_prefix_lookup_workspace_bytes(int n);

int metis_prefix_lookup(const uint64_t* keys, int n, uint64_t* table_keys, int32_t* table_pages,
                        int32_t* table_claim, int capacity, const int32_t* free_stack, int free_capacity,
                        int32_t* free_count, int32_t* refcount, int num_pages, int32_t* pages_out,
                        uint8_t* hits_out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * metis_debug_wait_probe -- test support for the bounded waits.
 *
 * Every pipeline wait in the library (an mbarrier phase a producer or the
 * tensor cores complete) gives up after a time limit instead of spinning
 * forever: it sets METIS_STATUS_WAIT_TIMEOUT in the device status word and the
 * kernel returns, so a library bug surfaces as a status bit and the CUDA
 * context stays usable.  This call runs that give-up path on purpose: it
 * launches one warp whose wait on an mbarrier can never complete (the barrier
 * expects an arrival that never comes), bounded by limit_ns nanoseconds.
 *
 *   limit_ns   (0, 1e9]: the wait's wall-time limit; otherwise METIS_E_SHAPE
 *              and nothing is launched
 *
 * Asynchronous on `stream`; afterwards metis_read_status() reports
 * METIS_STATUS_WAIT_TIMEOUT.  Not part of any attention path.
 */
int metis_debug_wait_probe(uint64_t limit_ns, void* stream);

/*
 * metis_read_status -- the device status word (METIS_STATUS_* bits, OR-ed
 * over every launch since it was last cleared) of the current device.
 * Synchronises the device: for tests and debugging, not for the hot path.
 * clear != 0 resets it to 0.  Returns METIS_OK or METIS_E_CUDA.
 */
int metis_read_status(uint32_t* status_out, int clear);

/* Message for the last non-zero return on the calling thread ("" if none). */
const char* metis_last_error(void);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int metis_version(void);

#ifdef __cplusplus
}
#endif

#endif /* METIS_ATTN_H */
