/*
 * pa.h — C ABI of libpa: PagedAttention decode on GB300 (sm_103a).
 *
 * Three device operations make up the hot path, plus a host block allocator
 * that builds their index inputs. Sources are the PagedAttention pages, cited
 * by title and section:
 *   [book]    "第4章 PagedAttention：虚拟内存的启示" (vLLM source-reading book)
 *   [digest]  "PagedAttention: virtual memory for the KV cache" (digest of
 *             thegustafson.com)
 *   [codex]   "01 · PagedAttention 与 KV cache 块管理"
 *   [lecture] "4. PagedAttention原理（下）"
 *
 * Conventions shared by every call
 * --------------------------------
 * - KV pool: one per layer, a dense row-major array shaped
 *   (2, num_blocks, block_size, num_kv_heads, head_size); index 0 of the
 *   first dimension holds K, index 1 holds V; head_size is innermost
 *   ([book] §4.3.1, §4.3.2). Element type: PA_F16 or PA_BF16.
 * - Pointers named "device" must point to GPU memory of the current device
 *   and be 16-byte aligned; the caller owns every buffer. The library never
 *   allocates device memory.
 * - Index arrays are int32 ([book] §4.4.1, §4.4.3).
 * - Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream). A return value of PA_OK means the work was
 *   validated and enqueued. Argument errors are detected on the host before
 *   any CUDA call and return a negative PA_ERR_* code; pa_last_error()
 *   returns a message for the calling thread's most recent failure.
 * - Data-dependent errors (a block id, slot or sequence length outside the
 *   pool or table) cannot be seen on the host. Kernels never read or write
 *   outside the buffers because of them: the offending item is skipped (or
 *   read as zeros) and a bit is set in a per-device error word, which
 *   pa_get_device_error() returns and clears.
 * - block_size must be a positive multiple of 16 ([book] §4.3.4: the CUDA
 *   backends require block_size % 16 == 0).
 * - FP8 cache (the *_fp8 calls): the same pool shape with 1-byte elements,
 *   each an OCP E4M3 code (1 sign, 4 exponent bits with bias 7, 3 fraction
 *   bits; no infinities; 0x7F / 0xFF are NaN; largest finite 448). A K code
 *   c stands for e4m3(c) * k_scale and a V code for e4m3(c) * v_scale, one
 *   scale per tensor. The pages name a lower-precision KV cache only as a
 *   capacity lever ([book] §4.8); the format, the per-tensor scales and the
 *   rounding below are the reading this library takes.
 */
#ifndef PAGED_KV_CACHE_PA_H
#define PAGED_KV_CACHE_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including CUDA headers (same type). */
typedef struct CUstream_st *pa_stream_t;

/* Status codes. */
#define PA_OK                  0
#define PA_ERR_INVALID_ARG    -1  /* null pointer, bad size, misalignment */
#define PA_ERR_UNSUPPORTED    -2  /* dtype / head_size / group shape not built */
#define PA_ERR_CUDA           -3  /* a CUDA runtime or driver call failed */
#define PA_ERR_WORKSPACE      -4  /* workspace missing or too small */
#define PA_ERR_OUT_OF_BLOCKS  -5  /* allocator: free list exhausted */
#define PA_ERR_NOT_FOUND      -6  /* allocator: unknown sequence id */

/* Element types of Q, K, V and the output. */
#define PA_F16   0
#define PA_BF16  1
/* Element type of an FP8 pool (pa_copy_blocks only; the FP8 calls below take
 * the 16-bit type of their activations as `dtype`). */
#define PA_FP8_E4M3  2

/* pa_decode flags. */
#define PA_DECODE_SHARED_BLOCKS 1u  /* some physical block appears in more than one
                                       sequence's table (prefix sharing, parallel
                                       sampling): keep K/V at normal L2 priority */
#define PA_DECODE_LENS_READY    2u  /* the caller guarantees that seq_lens already
                                       holds its final values when the kernel
                                       enqueued just before this call starts (it was
                                       copied from the host, or written by an
                                       earlier kernel): the decode may then read it
                                       while that kernel finishes */

/* Bits of the device error word. */
#define PA_DEVERR_BLOCK_ID  1   /* a block table entry outside [0, num_blocks) */
#define PA_DEVERR_SLOT      2   /* a slot >= num_blocks * block_size */
#define PA_DEVERR_SEQ_LEN   4   /* a seq_len < 0 or > max_blocks_per_seq * block_size */
#define PA_DEVERR_PAIR      8   /* a copy pair out of range, or a dst repeated / also a src */
#define PA_DEVERR_TIMEOUT  16   /* a bounded wait inside a kernel gave up */

/* Library version (major * 10000 + minor * 100 + patch). */
int pa_version(void);

/* Message for the calling thread's most recent failed call ("" if none).
 * The string stays valid until that thread's next failing call. */
const char *pa_last_error(void);

/*
 * pa_reshape_and_cache — write this step's new K/V rows into their slots.
 * [book] §4.4.3 (slot_mapping: one physical slot per new token, slot =
 * block_table[pos / B] * B + pos % B) and §4.5 step 1 (the step's K/V are
 * written into the cache by slot before attention reads it).
 *
 *   key, value    device, [num_tokens][num_kv_heads][head_size], contiguous
 *   kv_cache      device, the layer's pool (see conventions)
 *   slot_mapping  device, [num_tokens] int32. Token t goes to
 *                 kv_cache[0 or 1][slot / block_size][slot % block_size].
 *                 A negative slot means "skip this token" (padding).
 *                 A slot >= num_blocks * block_size is skipped and sets
 *                 PA_DEVERR_SLOT.
 *   num_tokens    >= 0 (0 is a no-op)
 *   head_size     num_kv_heads * head_size must be a multiple of 8
 * Writes are bit copies. Two tokens with the same slot race (last writer
 * unspecified). Returns PA_OK or a PA_ERR_* code.
 */
int pa_reshape_and_cache(const void *key, const void *value, void *kv_cache,
                         const int32_t *slot_mapping, int num_tokens,
                         int num_blocks, int block_size, int num_kv_heads,
                         int head_size, int dtype, pa_stream_t stream);

/*
 * pa_decode_workspace_size — bytes of device workspace pa_decode needs for
 * this batch shape on the current device (it depends on the device's SM
 * count). The same arguments must be passed to pa_decode. Writes *bytes.
 */
int pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                             int head_size, int block_size, int dtype,
                             size_t *bytes);

/*
 * pa_decode — one query token per sequence attends over all its cached
 * tokens through the block table ([book] §4.5 step 2: each logical block's
 * physical id is looked up in the sequence's table row before its K/V are
 * read; §4.4.1 block table; [digest] "注意力内核为何能正常工作").
 *
 *   out            device, [num_seqs][num_q_heads][head_size], dtype
 *   query          device, [num_seqs][num_q_heads][head_size], dtype
 *   kv_cache       device, the layer's pool (see conventions)
 *   block_tables   device, [num_seqs][max_blocks_per_seq] int32; row s,
 *                  column j = physical block of logical block j of sequence
 *                  s. Only the first ceil(seq_lens[s] / block_size) entries
 *                  of a row are read; the rest may hold anything.
 *   seq_lens       device, [num_seqs] int32: tokens cached for each
 *                  sequence, this step's token included. 0 gives a zero
 *                  output row.
 *   scale          multiplies q.k before the softmax (1/sqrt(head_size) in
 *                  the pages' pseudo-code)
 *   num_q_heads, num_kv_heads: num_q_heads % num_kv_heads == 0. Query head
 *                  hq reads kv head hq / (num_q_heads / num_kv_heads)
 *                  (contiguous groups: MHA, GQA, MQA). The group size G must
 *                  be <= 16 or a multiple of 16.
 *   head_size      64 or 128
 *   workspace      device, >= pa_decode_workspace_size(...) bytes, 256-byte
 *                  aligned: split-K partial results. Its contents need no
 *                  initialisation and are not preserved. Calls that share a
 *                  workspace must not overlap on the GPU.
 *
 *   flags          a bitwise OR of:
 *                  PA_DECODE_SHARED_BLOCKS: without it the K/V tiles are
 *                  streamed with an L2 evict-first hint (each byte is read
 *                  once per call, and the split-K records and tables stay
 *                  in L2); with it they keep normal priority so that
 *                  sequences sharing blocks hit L2.
 *                  PA_DECODE_LENS_READY: seq_lens is final before the kernel
 *                  enqueued just before this call starts (see Launch).
 *                  Results are identical under every combination; only the
 *                  speed differs.
 *
 * Launch: two kernels (the stream and the split-K merge), both with
 * programmatic dependent launch. The first may start while the preceding
 * kernel in the stream is finishing (typically this step's
 * pa_reshape_and_cache). By default it waits for that kernel before it
 * reads anything, so seq_lens may be written by the kernel just before
 * this call (a scheduler or length-update kernel). With PA_DECODE_LENS_READY
 * it reads seq_lens and plans its split while that kernel finishes, and
 * waits only before it reads the pool or writes anything; seq_lens must then
 * not be written by that kernel (host copies and earlier kernels are fine:
 * they complete before it starts).
 *
 * Result: out[s][hq] = sum_i softmax_i(scale * q.k_i) v_i over the
 * seq_lens[s] logical tokens, computed with fp32 dot products, an fp32
 * online softmax ([book] §4.6), split-K partial states merged with the same
 * (m, s, O) rule, and one rounding to dtype at the end. For a given device
 * and batch shape the result does not depend on where the blocks sit in
 * the pool (bit-identical under any permutation of physical placement).
 * num_seqs must be <= 4096. Returns PA_OK or a PA_ERR_* code.
 */
int pa_decode(void *out, const void *query, const void *kv_cache,
              const int32_t *block_tables, int max_blocks_per_seq,
              const int32_t *seq_lens, int num_seqs, float scale,
              int num_q_heads, int num_kv_heads, int head_size,
              int num_blocks, int block_size, int dtype,
              void *workspace, size_t workspace_bytes, unsigned flags,
              pa_stream_t stream);

/*
 * pa_decode_static_scratch — pa_decode for callers that cannot allocate
 * device memory. It has no counterpart on the PagedAttention pages; it
 * exists because some callers cannot call cudaMalloc: a host framework whose
 * allocator owns all of the GPU's memory, a plugin held to a fixed memory
 * budget, or a latency-critical loop where an allocation (which can
 * synchronise the device) is not allowed.
 *
 * Same arguments, result and launch behaviour as pa_decode, without the
 * workspace: the split-K scratch lives in a 16 MiB static device array
 * inside the library, which every GPU that loads the library holds until the
 * process exits. The call allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine).
 *   - Shapes whose scratch need (pa_decode_workspace_size) exceeds 16 MiB are
 *     rejected with PA_ERR_WORKSPACE and a message saying so. On a 152-SM
 *     GB300 that admits every query group of up to 8 heads (and every shape
 *     with head_size 64); groups of 9 or more at head_size 128 need pa_decode.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call on a device shares the one array. Nothing in it has to start
 *     at zero (each call writes what it reads), but calls that overlap on the
 *     GPU race on it: serialise them (one stream, or events).
 */
int pa_decode_static_scratch(void *out, const void *query, const void *kv_cache,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *seq_lens, int num_seqs, float scale,
                             int num_q_heads, int num_kv_heads, int head_size,
                             int num_blocks, int block_size, int dtype,
                             unsigned flags, pa_stream_t stream);

/*
 * pa_reshape_and_cache_fp8 — pa_reshape_and_cache into an FP8 pool: the same
 * slots and skipping rules, with every element quantised on the way in.
 *
 *   key, value    device, [num_tokens][num_kv_heads][head_size], dtype
 *                 (PA_F16 or PA_BF16)
 *   kv_cache      device, the layer's FP8 pool (1-byte elements)
 *   k_scale, v_scale  finite and > 0
 * The code stored for a K element x is the E4M3 value nearest to the IEEE
 * fp32 quotient x / k_scale (ties to the even code); quotients beyond +-448
 * store +-448 (saturation); NaN stores a NaN code. V likewise with v_scale.
 * Returns PA_OK or a PA_ERR_* code.
 */
int pa_reshape_and_cache_fp8(const void *key, const void *value, void *kv_cache,
                             const int32_t *slot_mapping, int num_tokens,
                             int num_blocks, int block_size, int num_kv_heads,
                             int head_size, int dtype, float k_scale, float v_scale,
                             pa_stream_t stream);

/* Workspace bytes pa_decode_fp8 needs (same rules as pa_decode_workspace_size). */
int pa_decode_fp8_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                 int head_size, int block_size, int dtype,
                                 size_t *bytes);

/*
 * pa_decode_fp8 — pa_decode over an FP8 pool. Arguments, launch behaviour
 * and guarantees are those of pa_decode (dtype is the type of query and
 * out), plus k_scale and v_scale (finite, > 0) as in the conventions. The
 * workspace is sized by pa_decode_fp8_workspace_size.
 *
 * Result: the attention of pa_decode with every cached element replaced by
 * its value e4m3(c) * scale. Codes are widened to dtype exactly (every E4M3
 * value is an fp16 and a bf16 value); k_scale is applied to the fp32 score
 * scale and v_scale at the final normalisation. A NaN code in a token that
 * is attended to makes that output row NaN.
 */
int pa_decode_fp8(void *out, const void *query, const void *kv_cache,
                  const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *seq_lens, int num_seqs, float scale,
                  int num_q_heads, int num_kv_heads, int head_size,
                  int num_blocks, int block_size, int dtype,
                  float k_scale, float v_scale,
                  void *workspace, size_t workspace_bytes, unsigned flags,
                  pa_stream_t stream);

/*
 * pa_prefill — causal attention of a chunk of new query tokens per sequence
 * over the paged cache (chunked prefill). [book] §4.5 step 2: the backend
 * hands the cache, the block table, the query offsets cu_seqlens_q and the
 * used lengths seqused_k to one varlen attention call; §4.6 for the online
 * softmax. Reading taken: the chunk of sequence s is the last
 * q_len = cu_seqlens_q[s+1] - cu_seqlens_q[s] of its seq_lens[s] cached
 * tokens (written first by pa_reshape_and_cache), and query i of the chunk,
 * at position p = seq_lens[s] - q_len + i, attends to tokens 0..p. With
 * q_len = 1 this is pa_decode's result (computed by a different kernel).
 *
 *   out, query     device, [total_q][num_q_heads][head_size], dtype; row
 *                  cu_seqlens_q[s] + i belongs to query i of sequence s
 *   kv_cache, block_tables, max_blocks_per_seq: as for pa_decode
 *   cu_seqlens_q   device, [num_seqs + 1] int32, non-decreasing, from 0 to
 *                  total_q
 *   seq_lens       device, [num_seqs] int32, >= the sequence's q_len
 *   total_q        rows of query / out (host int)
 *   max_seqlen_q   host int >= every q_len (sizes the list of work units; larger
 *                  is only slower; a chunk longer than it is an inconsistent
 *                  length, below)
 *   head_size      64 or 128; the group num_q_heads / num_kv_heads must be <= 16
 *                  or a multiple of 16
 *   workspace      device, NULL or >= pa_prefill_workspace_size(...) bytes,
 *                  256-byte aligned; workspace_bytes its size. With few work
 *                  units (a unit: up to 256 query rows of one sequence and kv
 *                  head; at most 4 per SM, e.g. a few long sequences with
 *                  short chunks) and a workspace, the units' K/V ranges are
 *                  split into equal shares across all SMs and the pieces
 *                  merged with the rule of [book] §4.6 (partial max, sum and
 *                  output over disjoint token ranges). NULL: each unit's range
 *                  stays whole (same result up to fp32 rounding). Its contents
 *                  need no initialisation and are not preserved; calls that
 *                  share it must not overlap on the GPU. A non-NULL workspace
 *                  that is too small or misaligned when a split is planned
 *                  gives PA_ERR_WORKSPACE.
 * Rows of sequences whose offsets or lengths are inconsistent are not
 * written and set PA_DEVERR_SEQ_LEN; block ids outside the pool read as
 * zeros and set PA_DEVERR_BLOCK_ID. Computed on the tcgen05 tensor cores:
 * S = Q K^T and O = P V in fp32 (tensor memory), an fp32 online softmax in
 * base 2 with P rounded once to dtype, split pieces combined in fp32 in a
 * fixed order, one rounding of O / l at the end. For a given device, shape
 * and workspace choice the result is deterministic. Launch: one persistent
 * kernel; with a split, a second (the merge) follows with programmatic
 * dependent launch. Allocates nothing. Returns PA_OK or a PA_ERR_* code.
 */
int pa_prefill(void *out, const void *query, const void *kv_cache,
               const int32_t *block_tables, int max_blocks_per_seq,
               const int32_t *cu_seqlens_q, const int32_t *seq_lens, int num_seqs,
               int total_q, int max_seqlen_q, float scale,
               int num_q_heads, int num_kv_heads, int head_size,
               int num_blocks, int block_size, int dtype,
               void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_prefill_workspace_size — bytes of workspace with which pa_prefill and
 * pa_prefill_fp8 split the K/V ranges of this shape on the current device
 * (it depends on the SM count); 0 when they would not split (many work
 * units). Same shape arguments as the calls. Writes *bytes.
 */
int pa_prefill_workspace_size(int num_seqs, int max_seqlen_q, int num_q_heads,
                              int num_kv_heads, int head_size, size_t *bytes);

/*
 * pa_prefill_fp8 — pa_prefill over an FP8 (E4M3) pool written by
 * pa_reshape_and_cache_fp8 ([book] §4.8's lower-precision cache, with the
 * FP8 conventions above): a cached K element stands for e4m3(code) * k_scale
 * and a V element for e4m3(code) * v_scale. kv_cache is the byte pool
 * (2, num_blocks, block_size, num_kv_heads, head_size); dtype is the type of
 * query and out (PA_F16 or PA_BF16). The codes are widened exactly to that
 * type on the way to the tensor cores; k_scale joins the score scale and
 * v_scale the final normalisation. Same shapes, limits and error behaviour
 * as pa_prefill (head_size 64 or 128, the same workspace rules and size);
 * k_scale and v_scale must be finite and > 0.
 */
int pa_prefill_fp8(void *out, const void *query, const void *kv_cache,
                   const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *cu_seqlens_q, const int32_t *seq_lens, int num_seqs,
                   int total_q, int max_seqlen_q, float scale,
                   int num_q_heads, int num_kv_heads, int head_size,
                   int num_blocks, int block_size, int dtype, float k_scale, float v_scale,
                   void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_copy_blocks — copy-on-write clones of whole physical blocks
 * ([digest] "写时复制": a shared block is cloned before a write and the
 * writer's table retargeted; [lecture] §4.3 steps: allocate Q, copy P into
 * Q). A block spans every layer ([book] §4.3.1: a "complete block" covers
 * all layers), so each pair is copied in every given pool.
 *
 *   kv_caches      HOST array of num_layers device pointers, one pool each;
 *                  1 <= num_layers <= 512
 *   src_dst_pairs  device, [num_pairs][2] int32 (src, dst)
 *   dtype          PA_F16, PA_BF16 or PA_FP8_E4M3 (the pools' element type;
 *                  a token's row, num_kv_heads * head_size elements, must be
 *                  a multiple of 16 bytes)
 * For every pair and layer, kv_cache[c][dst] = kv_cache[c][src] for c in
 * {0, 1}: all block_size slots, all heads, bit for bit. Preconditions: ids in
 * [0, num_blocks); no dst appears twice; no dst is also a src. A pair that
 * breaks them is not copied and sets PA_DEVERR_PAIR; the other pairs are
 * copied from the pre-call contents. Returns PA_OK or a PA_ERR_* code.
 */
int pa_copy_blocks(void *const *kv_caches, int num_layers,
                   const int32_t *src_dst_pairs, int num_pairs,
                   int num_blocks, int block_size, int num_kv_heads,
                   int head_size, int dtype, pa_stream_t stream);

/*
 * pa_get_device_error — read and clear the current device's error word
 * (PA_DEVERR_* bits, 0 if none). Synchronises the device first, so every
 * earlier launch has finished. Returns PA_OK or PA_ERR_CUDA.
 */
int pa_get_device_error(int *bits);

/* ------------------------------------------------------------------ */
/* Host block allocator: builds block tables, slot mappings and COW    */
/* pairs ([digest] "调度器机制简述" and "写时复制"; [codex] §3, §4.3;   */
/* [lecture] §4.3). Host memory only; not thread-safe per handle.      */
/* ------------------------------------------------------------------ */

typedef struct pa_allocator pa_allocator;

/*
 * Create a pool of num_blocks blocks of block_size tokens. `order` (may be
 * NULL = 0, 1, ..., num_blocks-1) is the initial free list, head first:
 * allocation pops the head, so an explicit order reproduces a given
 * placement and a random permutation gives random non-repeating ids.
 * Blocks whose count drops to 0 return to the head (LIFO reuse of freed
 * blocks, [codex] §4.3). Returns NULL on bad arguments (order must list
 * every block exactly once).
 */
pa_allocator *pa_alloc_create(int num_blocks, int block_size, const int32_t *order);
void pa_alloc_destroy(pa_allocator *a);

int pa_alloc_num_free(const pa_allocator *a);
/* Reference count of a block (0 = on the free list), or PA_ERR_INVALID_ARG. */
int pa_alloc_ref_count(const pa_allocator *a, int block);

/* New sequence holding num_tokens tokens: ceil(num_tokens / block_size)
 * blocks. All-or-nothing: PA_ERR_OUT_OF_BLOCKS leaves the pool unchanged. */
int pa_alloc_add_seq(pa_allocator *a, int num_tokens, int *seq_id);

/* New sequence sharing every block of `parent` (each block's count + 1),
 * as parallel sampling or a shared prompt does ([book] §4.7.1). */
int pa_alloc_fork(pa_allocator *a, int parent, int *child);

/*
 * Reserve the slot of the sequence's next token (position = its length).
 * If the last block is full (or there is none), a new block is taken. If the
 * last block has room but is shared (count > 1), it is copied on write: a
 * new block Q is taken, *cow_src = old block, *cow_dst = Q, the sequence's
 * table points at Q, and the old block's count drops by 1 ([lecture] §4.3).
 * Otherwise *cow_src = *cow_dst = -1. *slot = table[pos / B] * B + pos % B
 * ([book] §4.4.3). The caller must run pa_copy_blocks on the pair before
 * writing the token. PA_ERR_OUT_OF_BLOCKS leaves everything unchanged.
 */
int pa_alloc_append_token(pa_allocator *a, int seq_id, int32_t *slot,
                          int32_t *cow_src, int32_t *cow_dst);

/* Release a sequence: its blocks in reverse table order, each count - 1. */
int pa_alloc_free_seq(pa_allocator *a, int seq_id);

/* Tokens held by a sequence (>= 0), or a PA_ERR_* code. */
int pa_alloc_seq_len(const pa_allocator *a, int seq_id);

/* Number of blocks in a sequence's table (>= 0), or a PA_ERR_* code. */
int pa_alloc_seq_num_blocks(const pa_allocator *a, int seq_id);

/* Fill out[n][max_blocks_per_seq] (host, int32) with the tables of the
 * given sequences, padding each row with -1. PA_ERR_INVALID_ARG if a table
 * is longer than max_blocks_per_seq. */
int pa_alloc_block_tables(const pa_allocator *a, const int *seq_ids, int n,
                          int max_blocks_per_seq, int32_t *out);

/* Fill out[n] (host, int32) with the sequences' lengths. */
int pa_alloc_seq_lens(const pa_allocator *a, const int *seq_ids, int n, int32_t *out);

/* ------------------------------------------------------------------ */
/* Host prefix-cache block pool ([codex] §4.2-§4.5, §5): full blocks carry */
/* a chained hash, a new prompt reuses the longest cached prefix, freed  */
/* blocks stay cached until reused. Host memory only; not thread-safe.   */
/* ------------------------------------------------------------------ */

typedef struct pa_prefix_cache pa_prefix_cache;

/*
 * Create a pool of num_blocks blocks of block_size tokens. Block 0 is the
 * null block and is never handed out; the free queue starts as 1, 2, ...,
 * num_blocks - 1 (head first = evicted first). Returns NULL on bad
 * arguments (num_blocks >= 2, block_size > 0).
 *
 * Hashes: a full block's hash is SHA-256(parent hash || its token ids as
 * little-endian int32), the first block's parent being 32 zero bytes
 * ([codex] §4.4; the serialisation and the root are the reading taken).
 */
pa_prefix_cache *pa_pcache_create(int num_blocks, int block_size);
void pa_pcache_destroy(pa_prefix_cache *c);

/* Blocks on the free queue (cached ones included). */
int pa_pcache_num_free(const pa_prefix_cache *c);

/*
 * New sequence with the prompt tokens[num_tokens] (num_tokens > 0). Its full
 * blocks' hash chain is matched against the cache from the first block; the
 * match ends at the first miss and covers at most num_tokens - 1 tokens (the
 * last prompt token is always recomputed). Matched blocks are touched
 * (count + 1, taken off the free queue if they were on it); the rest come
 * from the free queue's head, each losing any hash it still carried (lazy
 * eviction), and the prompt's full new blocks are recorded as cached.
 * *num_cached_tokens = the matched tokens (a multiple of block_size): the
 * caller writes K/V only for positions >= that. All-or-nothing:
 * PA_ERR_OUT_OF_BLOCKS leaves the pool unchanged.
 */
int pa_pcache_add_seq(pa_prefix_cache *c, const int32_t *tokens, int num_tokens,
                      int *seq_id, int *num_cached_tokens);

/* pa_pcache_admit flag: the requests neither match nor record (every block
 * fresh and unhashed, freed to the queue's head) - prefix caching off. */
#define PA_PCACHE_NO_CACHE 1

/*
 * Admit a wave of n prompts, in order, each as pa_pcache_add_seq does (or,
 * with PA_PCACHE_NO_CACHE, without matching or recording), and build the
 * prefill inputs for them in one call. Request r's tokens are
 * tokens[cu_tokens[r] .. cu_tokens[r+1]) (host; cu_tokens[0] = 0, every
 * request non-empty, at most max_blocks_per_seq blocks).
 *
 * Outputs (host int32, caller-owned; may be pinned memory that is then
 * copied to the device), for the admitted requests r < return value:
 *   seq_ids[r], num_cached[r]      the sequence and its matched tokens;
 *   seq_lens[r]                    the prompt length;
 *   cu_seqlens_q[0 .. r+1]         offsets of the uncached tokens, whose
 *                                  queries the caller packs in this order;
 *   slot_mapping[cu_seqlens_q[r] + i]  slot of position num_cached[r] + i
 *                                  (slot_capacity >= cu_tokens[n] entries);
 *   block_tables[r][max_blocks_per_seq] the table, padded with -1.
 * Admission stops at the first request the free queue cannot supply (that
 * request and the rest are untouched). Returns the number admitted (0..n),
 * or a negative PA_ERR_* on bad arguments (nothing admitted).
 * The requests' block hashes are computed first, on up to
 * PA_PCACHE_THREADS helper threads (environment, read once per pool;
 * default min(16, hardware threads - 1); 0 = none), sharing the hashes of the
 * leading blocks that equal request 0's token for token; matching and
 * allocation then run in request order. Results do not depend on the
 * thread count.
 */
int pa_pcache_admit(pa_prefix_cache *c, const int32_t *tokens, const int64_t *cu_tokens, int n,
                    int flags, int max_blocks_per_seq, int32_t *seq_ids, int32_t *num_cached,
                    int32_t *cu_seqlens_q, int32_t *seq_lens, int32_t *slot_mapping,
                    int64_t slot_capacity, int32_t *block_tables);

/* Reserve the next token's slot (*slot = table[pos / B] * B + pos % B); a
 * block that becomes full is hashed and recorded as cached. */
int pa_pcache_append_token(pa_prefix_cache *c, int seq_id, int32_t token, int32_t *slot);

/* Release a sequence: its blocks in reverse table order, count - 1; a block
 * reaching 0 goes to the free queue's head if it has no hash and to its tail
 * if it has one ([codex] §4.3). */
int pa_pcache_free_seq(pa_prefix_cache *c, int seq_id);

/* pa_pcache_free_seq for seq_ids[n] in order; every id must be live and
 * listed once, else nothing is freed. */
int pa_pcache_free_seqs(pa_prefix_cache *c, const int32_t *seq_ids, int n);

/* Tokens of a sequence, or a PA_ERR_* code. */
int pa_pcache_seq_len(const pa_prefix_cache *c, int seq_id);

/* Block tables of the given sequences into out[n][max_blocks_per_seq]
 * (host, int32, padded with -1). */
int pa_pcache_block_tables(const pa_prefix_cache *c, const int *seq_ids, int n,
                           int max_blocks_per_seq, int32_t *out);

/* Slots of positions first_pos .. first_pos + n - 1 of a sequence (host). */
int pa_pcache_slots(const pa_prefix_cache *c, int seq_id, int first_pos, int n, int32_t *out);

/* The free queue, head first, into out[capacity]; returns its length. */
int pa_pcache_free_queue(const pa_prefix_cache *c, int32_t *out, int capacity);

/* Reference count of a block, or PA_ERR_INVALID_ARG. */
int pa_pcache_ref_count(const pa_prefix_cache *c, int block);

/* 1 and the block's 32-byte hash in out if it carries one, else 0. */
int pa_pcache_block_hash(const pa_prefix_cache *c, int block, uint8_t *out);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_CACHE_PA_H */
