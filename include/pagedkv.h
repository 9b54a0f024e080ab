/*
 * pagedkv.h -- C ABI of a GB300 (sm_103a) library for PagedAttention decode.
 *
 * The problem, as the pages state it ("Lesson 4: Model deployment and inference
 * acceleration", section 4.2 "PagedAttention: virtual-memory-style KV management";
 * "Efficient AI Lecture 13: LLM Deployment Techniques", section "PagedAttention"):
 * the KV cache is cut into fixed blocks of 16 tokens taken from one pre-allocated
 * pool; every request keeps a page table (block table) from its logical blocks to
 * physical blocks; attention fetches the blocks wherever they sit, and the result is
 * plain attention softmax(q K^T / sqrt(d)) V over the request's tokens.
 *
 * Conventions for every call:
 *  - Pointers named "device" point to GPU memory that the caller allocated and owns;
 *    the library never frees caller memory.  Pointers named "host" point to host memory.
 *  - Work is enqueued on the caller's stream (a cudaStream_t passed as void*; NULL is
 *    the legacy default stream) and runs asynchronously.  Calls do not synchronise,
 *    except pkv_get_device_error, which waits for its own stream.
 *  - Every call validates its host-side arguments before launching anything and
 *    returns a status; no exception crosses the ABI.  A launch failure maps to
 *    PKV_ERR_CUDA (the CUDA error text is available from pkv_last_cuda_error).
 *  - Device-side checks never trap: an out-of-range block id, slot or context length
 *    found by a kernel sets a bit in the pool's device error word (see
 *    pkv_get_device_error), and the offending access is skipped.
 *  - Layouts are row-major ("C order"); element sizes are those of the named types.
 *  - Calls on one pool must be ordered on one stream (or otherwise serialised): the
 *    pool's device error word and its scheduler counters are shared by its calls.
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

/* Exported symbols (the library is built with hidden visibility by default). */
#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Tokens per physical block; fixed ("Lesson 4", 4.2: 16 tokens per block by default). */
#define PKV_BLOCK_SIZE 16

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* a pointer, size or layout argument is invalid         */
  PKV_ERR_UNSUPPORTED = 2, /* valid but not built (head_dim, forced kernel, ...)      */
  PKV_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed            */
  PKV_ERR_WORKSPACE = 4,   /* the workspace passed is smaller than the call needs    */
  PKV_ERR_CAPACITY = 5     /* out of free blocks, sequence slots or table capacity   */
} pkv_status;

typedef enum pkv_kv_dtype {
  /* K/V stored as bf16. */
  PKV_KV_BF16 = 0,
  /* K/V stored as int8 codes with one fp32 scale per (token, kv head) row, symmetric:
   * s = max|x| / 127, code = round(x / s) ("Lesson 4", 5.3 "KV Cache Quantization"). */
  PKV_KV_INT8 = 1,
  /* K/V stored as FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
   * infinities, largest finite 448) with one fp32 scale per (token, kv head) row:
   * s = max|x| / 448, code = nearest E4M3 of x / s, ties to even, saturating at +-448.
   * The same section names FP8 KV caches and their larger dynamic range; it gives no
   * scaling rule, and this is the INT8 scheme with E4M3 codes. */
  PKV_KV_FP8_E4M3 = 2
} pkv_kv_dtype;

/* Bits of the device error word. */
#define PKV_DEVERR_BLOCK_ID 0x1u    /* a block-table entry read by decode was < 0 or >= num_blocks */
#define PKV_DEVERR_CONTEXT_LEN 0x2u /* a context length was < k (1 for one query token) or > max_context_len */
#define PKV_DEVERR_SLOT 0x4u        /* a slot_mapping entry was >= num_blocks * 16               */
#define PKV_DEVERR_TIMEOUT 0x8u     /* an asynchronous copy did not arrive within the time limit */

/* Opaque, host-owned pool descriptor. */
typedef struct pkv_pool pkv_pool;

/* Text for a status code (static storage). */
PKV_API const char* pkv_status_string(pkv_status status);

/* Text of the last CUDA error seen by this thread inside the library (static per thread). */
PKV_API const char* pkv_last_cuda_error(void);

/* Library version string, e.g. "0.1.0". */
PKV_API const char* pkv_version(void);

/*
 * Bytes the caller must allocate for a pool ("Lesson 4", 4.2: one global, pre-allocated
 * block pool).  *kv_bytes_each receives the size of the K array (the V array has the
 * same size): num_blocks * kv_heads * 16 * head_dim * element size.  *scale_bytes_each
 * receives the size of each fp32 scale array, num_blocks * kv_heads * 16 * 4, or 0 for
 * bf16.  Either output pointer may be NULL.
 * Errors: PKV_ERR_INVALID_ARG for num_blocks < 1, kv_heads < 1, head_dim < 1 or an
 * unknown dtype.
 */
PKV_API pkv_status pkv_pool_bytes(int64_t num_blocks, int kv_heads, int head_dim, pkv_kv_dtype dtype,
                          size_t* kv_bytes_each, size_t* scale_bytes_each);

/*
 * Describe a pool of physical KV blocks that the caller has allocated on the current
 * device ("Lesson 4", 4.2, global block pool).
 *   k_cache, v_cache (device): [num_blocks, kv_heads, 16, head_dim] of bf16, int8 or E4M3
 *                              bytes, each 16-byte aligned.
 *   k_scale, v_scale (device): [num_blocks, kv_heads, 16] fp32 for PKV_KV_INT8 and
 *                              PKV_KV_FP8_E4M3, 16-byte aligned; must be NULL for
 *                              PKV_KV_BF16.
 *   block_size must be PKV_BLOCK_SIZE.
 * The library records the pointers and allocates a small device error word for the
 * pool on the current device (freed by pkv_pool_destroy).  The pool contents are not
 * touched.  *out receives the descriptor.
 * Errors: PKV_ERR_INVALID_ARG (NULL or misaligned pointers, bad sizes, scales given for
 * bf16 or missing for int8); PKV_ERR_UNSUPPORTED (head_dim not 64 or 128, block_size
 * not 16); PKV_ERR_CUDA (no device, allocation failure).
 */
PKV_API pkv_status pkv_pool_create(int64_t num_blocks, int kv_heads, int head_dim, int block_size,
                           pkv_kv_dtype dtype, void* k_cache, void* v_cache, float* k_scale,
                           float* v_scale, pkv_pool** out);

/* Free the descriptor and its device error word (not the caller's arrays).  NULL is a no-op. */
PKV_API pkv_status pkv_pool_destroy(pkv_pool* pool);

/*
 * Append new tokens' K and V to the cache: for token t and kv head h,
 *   slot = slot_mapping[t], block = slot / 16, offset = slot % 16,
 *   k_cache[block][h][offset][:] = key[t][h][:]   (and the same for V).
 * Only the new tokens' K/V are written ("Lesson 4", 4.2; "LLM Engineer's Handbook --
 * inference optimisation", section "KV cache").  For an INT8 pool each (t, h) row of
 * key and of value is quantised on the way in ("Lesson 4", 5.3):
 *   s = max_c |x_c| / 127 (fp32, IEEE division), code_c = round_half_even(x_c / s),
 *   clamped to [-127, 127]; a row of zeros stores s = 0 and zero codes;
 *   k_scale[block][h][offset] = s.
 * An FP8 pool does the same with s = max_c |x_c| / 448 and code_c = nearest E4M3 of
 * x_c / s (ties to even, saturating).
 *   key, value   (device): bf16 [num_tokens, kv_heads, head_dim], 16-byte aligned.
 *   slot_mapping (device): int32 [num_tokens]; a negative slot skips that token.
 * Slots must be distinct among the tokens of one call (two writes to one slot race).
 * A slot >= num_blocks * 16 is skipped and sets PKV_DEVERR_SLOT.
 * num_tokens == 0 is a no-op.  Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA.
 */
PKV_API pkv_status pkv_reshape_and_cache(const pkv_pool* pool, const void* key, const void* value,
                                 const int32_t* slot_mapping, int64_t num_tokens, void* stream);

/*
 * Copy whole blocks inside the pool: for each pair (src, dst), every kv head's 16 K and V
 * rows of block src (and their scales, for INT8/FP8) are copied to block dst.  This is the
 * copy-on-write step of block sharing: when a sequence that shares a partly filled block
 * with others appends a token, it first gets its own copy of that block
 * ("Efficient AI Lecture 13: LLM Deployment Techniques", section "PagedAttention": shared
 * prompt prefixes reuse physical blocks for parallel sampling and beam search).
 *   pairs (device): int32 [num_pairs][2]; a dst must not appear twice or also as a src in
 *                   the same call.  Out-of-range ids are skipped and set PKV_DEVERR_BLOCK_ID.
 * num_pairs == 0 is a no-op.  Errors: PKV_ERR_INVALID_ARG (num_pairs > 65535), PKV_ERR_CUDA.
 */
PKV_API pkv_status pkv_copy_blocks(const pkv_pool* pool, const int32_t* pairs, int num_pairs,
                                   void* stream);

/*
 * Host-side block manager (no device memory, no CUDA calls): the free list of a pool's
 * num_blocks physical blocks, a reference count per block, and a page table per sequence
 * ("Efficient AI Lecture 13", section "PagedAttention / How it works": allocate physical
 * blocks on demand, translate logical blocks through a block table; "Lesson 4", 4.2: a
 * pre-allocated pool with dynamic allocation and release).  Sequences are small integer
 * handles in [0, max_seqs).  A manager serialises its own calls (one mutex).
 */
typedef struct pkv_block_manager pkv_block_manager;

/* Errors: PKV_ERR_INVALID_ARG (sizes < 1, num_blocks > 2^31 - 1), PKV_ERR_CAPACITY (memory). */
PKV_API pkv_status pkv_block_manager_create(int64_t num_blocks, int max_seqs,
                                            int max_blocks_per_seq, pkv_block_manager** out);
PKV_API pkv_status pkv_block_manager_destroy(pkv_block_manager* manager);

/* A new empty sequence; *seq receives its handle.  PKV_ERR_CAPACITY when all handles are in use. */
PKV_API pkv_status pkv_block_manager_add_sequence(pkv_block_manager* manager, int* seq);

/*
 * A new sequence that shares every block of `parent` (each block's count + 1) and has its
 * length: prefix sharing for parallel sampling and beam search.
 */
PKV_API pkv_status pkv_block_manager_fork(pkv_block_manager* manager, int parent, int* child);

/* Release a sequence: each of its blocks' count - 1; blocks reaching 0 return to the pool. */
PKV_API pkv_status pkv_block_manager_free_sequence(pkv_block_manager* manager, int seq);

/*
 * Reserve cache slots for new tokens: sequence seqs[i] grows by num_new_tokens[i] tokens.
 * slot_mapping (host, int32, sum of num_new_tokens) receives the slot of each new token in
 * order (for pkv_reshape_and_cache).  A new block is taken whenever a token starts one.  If
 * a sequence's last block is shared and partly filled, it is first replaced by a fresh
 * block and the pair (old, new) is written to copy_pairs (host, int32 [max_copies][2]) for
 * pkv_copy_blocks, which must run before the new tokens are written; *num_copies receives
 * the number of pairs.  All or nothing: on error nothing changes.
 * Errors: PKV_ERR_INVALID_ARG (unknown or repeated sequence, negative count, copy_pairs
 * too small), PKV_ERR_CAPACITY (not enough free blocks, or a table would exceed
 * max_blocks_per_seq).
 */
PKV_API pkv_status pkv_block_manager_append(pkv_block_manager* manager, const int* seqs,
                                            const int* num_new_tokens, int n,
                                            int32_t* slot_mapping, int32_t* copy_pairs,
                                            int max_copies, int* num_copies);

/*
 * Shorten a sequence to its first num_tokens tokens (0 <= num_tokens <= its length, and not
 * below its released blocks, see pkv_block_manager_release_before): the
 * blocks past ceil(num_tokens / 16) are released (count - 1).  Speculative decoding uses it
 * to drop the draft tokens the target model rejected ("Lesson 4", 5.2: only the accepted
 * prefix is kept).  The slots past num_tokens in the last kept block are reused by the
 * next append, with a copy first if that block is shared.
 * Errors: PKV_ERR_INVALID_ARG (unknown sequence, num_tokens out of range).
 */
PKV_API pkv_status pkv_block_manager_truncate(pkv_block_manager* manager, int seq, int num_tokens);

/*
 * Sliding window ("LLM/MLLM inference optimisation", 2.3: keep only the most recent window
 * of the cache, for a fixed memory footprint): release the sequence's blocks that hold only
 * tokens before position `token` (block j when 16 (j + 1) <= token).  Their table entries
 * become -1 and each block's count drops by one; the sequence's length and the positions of
 * its later tokens do not change.  A decode with window W and k query tokens reads from
 * token T - (k - 1) - W on, so token = T + n - (k - 1) - W keeps every block a decode after
 * n more appended tokens needs.  Releasing already released blocks is a no-op; truncate
 * below a released block is refused.
 * Errors: PKV_ERR_INVALID_ARG (unknown sequence, token < 0 or past the length).
 */
PKV_API pkv_status pkv_block_manager_release_before(pkv_block_manager* manager, int seq, int token);

/*
 * Page tables and lengths of sequences seqs[0..n): block_tables (host, int32
 * [n][max_blocks_per_seq], -1 past each table) and context_lens (host, int32 [n]), the
 * inputs of pkv_paged_attention_decode once copied to the device.
 */
PKV_API pkv_status pkv_block_manager_tables(const pkv_block_manager* manager, const int* seqs,
                                            int n, int32_t* block_tables, int32_t* context_lens);

/* Free blocks and live sequences (either pointer may be NULL). */
PKV_API pkv_status pkv_block_manager_stats(const pkv_block_manager* manager, int64_t* free_blocks,
                                           int* live_seqs);

/* Reference count of a block (0 = free), or -1 for an id out of range. */
PKV_API int32_t pkv_block_manager_refcount(const pkv_block_manager* manager, int32_t block);

/*
 * Decode-plan knobs.  Zero-initialise and set what you need; zero means automatic.
 *   partition_blocks: context partition (split-K) size P in 16-token blocks; each
 *     (sequence, kv head, partition) becomes one work item, and sequences longer than
 *     one partition are combined by a log-sum-exp reduce.  Partitions start at multiples
 *     of P; a sequence's last partition also takes a remainder of at most P / 4 blocks
 *     (so a partition holds up to P + P / 4 blocks).  0 = chosen from the batch shape and
 *     the device's SM count.
 *   kernel: which decode kernel family runs.  Both serve, per (sequence, kv head), a tile
 *     of group * num_queries query columns, in chunks of up to 16 (tensor cores) or 8
 *     (CUDA cores) columns, each chunk one work unit that reads the kv head's blocks.
 *     PKV_KERNEL_AUTO (0) picks the tensor-core kernel, which is built for every pool type
 *     at head_dim 64 and 128 and measured faster than the CUDA-core kernel on every such
 *     shape, MHA included; PKV_KERNEL_CUDA_CORE (1) and PKV_KERNEL_TENSOR_CORE (2) force
 *     one (PKV_ERR_UNSUPPORTED if it is not built for the shape).  Both compute the same
 *     function.
 *   schedule: how CTAs map to work items.  PKV_SCHEDULE_AUTO (0) picks;
 *     PKV_SCHEDULE_GRID (1) launches one CTA per (partition slot, sequence, kv head), slots
 *     past a sequence's partition count exiting at once; PKV_SCHEDULE_PERSISTENT (2)
 *     launches about one wave of CTAs that take items from a counter in the pool's device
 *     memory (batches of up to 4096 sequences; larger batches use the grid).
 *   stages, blocks_per_stage: shape of each warp's shared-memory ring in the tensor-core
 *     kernel (0 = automatic; otherwise a built shape, PKV_ERR_UNSUPPORTED for others).
 *     Shallower rings fit more CTAs on an SM; two blocks per stage run the softmax once
 *     per 32 tokens.
 *   num_queries: query tokens per sequence, k (0 = 1).  With k > 1 the call verifies k
 *     draft tokens in one pass ("Lesson 4", 5.2 "Speculative Decoding"; the target model
 *     scores all drafts at once): the k queries are the sequence's last k cached
 *     positions, appended beforehand by pkv_reshape_and_cache, and query i attends
 *     causally, to tokens t < T_b - (k - 1 - i).  q and out are then
 *     [num_seqs, k, num_q_heads, head_dim]; each K/V block is read once per kv head and
 *     column chunk (one chunk while group * k <= 16 on the tensor cores).  1 <= k <= 16,
 *     max_context_len >= k, and a sequence with T_b < k counts as out of range.
 *   window: sliding-window attention ("LLM/MLLM inference optimisation", 2.3: keep only the
 *     most recent window of the KV cache), 0 = none.  With window W > 0 a query at
 *     position p attends to tokens p - W + 1 .. p only.  The blocks before the first one
 *     any query sees are never read, so their block_tables entries may be -1 (see
 *     pkv_block_manager_release_before); slots before the window in that first block may
 *     hold anything.  Fewer blocks are read, and the plan sizes partitions and the
 *     workspace for the window.
 */
#define PKV_KERNEL_AUTO 0
#define PKV_KERNEL_CUDA_CORE 1
#define PKV_KERNEL_TENSOR_CORE 2
#define PKV_SCHEDULE_AUTO 0
#define PKV_SCHEDULE_GRID 1
#define PKV_SCHEDULE_PERSISTENT 2
typedef struct pkv_decode_options {
  int partition_blocks;
  int kernel;
  int schedule;
  int stages;
  int blocks_per_stage;
  int num_queries;
  int window;
  int reserved[1];
} pkv_decode_options;

/*
 * Bytes of device workspace that pkv_paged_attention_decode needs for this batch shape
 * (0 when no sequence is split).  max_context_len is the largest context length the
 * call will see.  options may be NULL.
 */
PKV_API pkv_status pkv_decode_workspace_bytes(const pkv_pool* pool, int num_seqs, int num_q_heads,
                                      int max_context_len, const pkv_decode_options* options,
                                      size_t* bytes);

/*
 * The plan the decode call would use for this shape: partition size in blocks, the
 * largest number of partitions of one sequence, kernels launched per call (1 or 2) and
 * the kernel family (PKV_KERNEL_CUDA_CORE or PKV_KERNEL_TENSOR_CORE).  Any output pointer
 * may be NULL.  Errors: as pkv_decode_workspace_bytes, and PKV_ERR_UNSUPPORTED when the
 * options force a kernel family that is not built for the shape.
 */
PKV_API pkv_status pkv_decode_plan(const pkv_pool* pool, int num_seqs, int num_q_heads,
                           int max_context_len, const pkv_decode_options* options,
                           int* partition_blocks, int* max_partitions, int* kernels_per_call,
                           int* kernel);

/*
 * PagedAttention decode: one new query token per sequence attends over the sequence's
 * cached tokens ("Lesson 4", 4.2, attention-invariance equation):
 *   out[b][h][:] = sum_{t < T_b} softmax_t(scale * q[b][h] . K_b[t]) V_b[t]
 * where token t of sequence b lives in physical block block_tables[b][t / 16] at offset
 * t % 16, T_b = context_lens[b], and query head h reads kv head h / (num_q_heads /
 * kv_heads) (contiguous GQA groups; "LLM/MLLM inference optimisation", 2.3).  For INT8
 * and FP8 pools K and V are the dequantised values s * value(code).  Accumulation is fp32; out is
 * rounded to bf16 (round to nearest even).
 *   q            (device): bf16 [num_seqs, num_q_heads, head_dim], 16-byte aligned.
 *   block_tables (device): int32 [num_seqs, max_blocks_per_seq]; entries past
 *                          ceil(T_b / 16) are never used and may hold anything (a
 *                          kernel may load them along with the used ones, so every row
 *                          must be max_blocks_per_seq entries long).
 *   context_lens (device): int32 [num_seqs], 1 <= T_b <= max_context_len (k <= T_b with
 *                          k query tokens per sequence).
 *   max_context_len (host int): an upper bound on every T_b; it sizes the plan and the
 *                          workspace and must be <= max_blocks_per_seq * 16.
 *   scale: softmax scale, usually 1 / sqrt(head_dim).
 *   out          (device): bf16 [num_seqs, num_q_heads, head_dim], 16-byte aligned.
 *   workspace    (device): at least pkv_decode_workspace_bytes(...) bytes, 16-byte
 *                          aligned; may be NULL when that size is 0.  Its contents need no
 *                          initialisation and are overwritten.
 * A sequence whose T_b is out of range gets a zero output and sets
 * PKV_DEVERR_CONTEXT_LEN; a block id out of range is skipped and sets
 * PKV_DEVERR_BLOCK_ID.  num_seqs == 0 is a no-op.
 * num_q_heads must be a multiple of kv_heads (else PKV_ERR_INVALID_ARG); any group size
 * G = num_q_heads / kv_heads is served: MHA (G = 1), GQA (1 < G < num_q_heads, powers of
 * two or not) and MQA (kv_heads = 1, G = num_q_heads) ("LLM/MLLM inference
 * optimisation", 2.2 and the 2.3 table).  A group that is not a power of two fills the
 * next power-of-two column tile with its unused slots idle; groups wider than a tile (16
 * columns on the tensor cores, 8 on the CUDA cores) are served in column chunks.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA.
 */
PKV_API pkv_status pkv_paged_attention_decode(const pkv_pool* pool, const void* q,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int num_seqs, int num_q_heads,
                                      int max_context_len, float scale, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * pkv_paged_attention_decode with explicit plan options (NULL = automatic), including
 * options->num_queries for multi-query (draft verification) calls and options->window for
 * sliding-window attention.
 */
PKV_API pkv_status pkv_paged_attention_decode_ex(const pkv_pool* pool, const void* q,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* context_lens, int num_seqs,
                                         int num_q_heads, int max_context_len, float scale,
                                         void* out, void* workspace, size_t workspace_bytes,
                                         const pkv_decode_options* options, void* stream);

/*
 * Size of the fixed device scratch array used by
 * pkv_paged_attention_decode_static_scratch (16 MiB).
 */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * pkv_paged_attention_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart to this call; it exists for users of this library, not for the
 * method.  Some callers cannot allocate where they decode -- for example a plugin hosted
 * by another runtime that owns the whole device-memory budget and gives its plugins no
 * allocator, or a latency-critical serving loop that must not call cudaMalloc.  This call
 * takes the same arguments as pkv_paged_attention_decode minus the workspace, and keeps
 * the split-K scratch in a fixed array of PKV_STATIC_SCRATCH_BYTES inside the library's
 * device image instead; it calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Every GPU that loads the library holds that array until the process exits.
 *  - The first call on a device looks up the array's device address (with that device
 *    current) and caches it; make that first call before any stream capture.
 *  - Call it with the pool's device current (else PKV_ERR_INVALID_ARG, nothing launched).
 *  - All calls on a device share the array, which keeps the last call's contents.
 *    Nothing in it needs to start at zero: each call writes every partial it reads.
 *    Calls whose work overlaps on the GPU (other streams, other host threads) race on
 *    the array; serialise them.
 * Errors: as pkv_paged_attention_decode, and PKV_ERR_WORKSPACE when the batch shape
 * needs more scratch than PKV_STATIC_SCRATCH_BYTES (pkv_static_scratch_error() then
 * gives the sizes); nothing is launched in that case.
 */
PKV_API pkv_status pkv_paged_attention_decode_static_scratch(
    const pkv_pool* pool, const void* q, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int max_context_len, float scale,
    void* out, void* stream);

/*
 * Text of the last pkv_paged_attention_decode_static_scratch outcome in this thread
 * ("no error" after a call that succeeded; static storage per thread).  For
 * PKV_ERR_CUDA it names the status only; pkv_last_cuda_error() has the CUDA text.
 */
PKV_API const char* pkv_static_scratch_error(void);

/*
 * Read and clear the pool's device error word (PKV_DEVERR_* bits).  Waits for the work
 * already enqueued on `stream`, then copies the word to *flags (host) and zeroes it.
 */
PKV_API pkv_status pkv_get_device_error(const pkv_pool* pool, uint32_t* flags, void* stream);

/* Number of kernels this library has launched in this process (all threads). */
PKV_API uint64_t pkv_launch_count(void);

/*
 * Failure-detection self-test (no counterpart on the pages; for tests of this library).
 * Runs the decode kernels' bounded mbarrier wait, in a one-warp kernel on `stream`, on a
 * barrier that nothing completes, with a limit of limit_ns (1e5 .. 2e9 ns; the decode
 * kernels use 2e9).  The wait must give up: *flags receives PKV_DEVERR_TIMEOUT and
 * *waited_ns the wall time the kernel waited (at least limit_ns, plus at most 64 polls of
 * up to 1 ms).  The CUDA context stays usable.  Synchronises `stream`.
 * Errors: PKV_ERR_INVALID_ARG, PKV_ERR_CUDA.
 */
PKV_API pkv_status pkv_selftest_bounded_wait(uint64_t limit_ns, uint32_t* flags, uint64_t* waited_ns,
                                             void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
