/*
 * pa.h -- C ABI of the paged-KV-cache decode path for one GB300 (sm_103a).
 *
 * The KV cache of every layer is a pool of fixed-size blocks of 16 tokens
 * (other block sizes through the *_ex entry points);
 * each sequence reaches its tokens through a block table of physical block
 * ids, and the kernels see nothing but those ids and the sequence lengths
 * [Efficient Memory Management for Large Language Model Serving with
 * PagedAttention, "KV Cache Manager: Block Table Mapping" (logical-to-physical
 * separation) and "Kernel-Level Optimizations"].
 *
 * Three operations, one per kernel family the pages name:
 *   pa_cache_write       fused reshape and block write of the new tokens' K/V
 *   pa_decode_attention  fused block read and attention (with context-split
 *                        partitions and a merge for long sequences)
 *   pa_copy_blocks       fused copy-on-write block copy, all pairs and layers
 * and the pages' other block move:
 *   pa_swap_blocks       swap-out / swap-in between the GPU pool and a CPU
 *                        swap space, all pairs and layers
 *
 * Conventions for every entry point:
 *   - Every pointer named "device" is device memory owned by the caller; the
 *     library allocates nothing, keeps no state between calls and never
 *     synchronises the stream.  Work is enqueued on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream) and runs
 *     asynchronously.
 *   - Tensors are dense and row-major in the layouts stated below, with base
 *     addresses aligned to 16 bytes.
 *   - Problems visible on the host (null pointers, unsupported sizes, dtype
 *     mismatch, small workspace) return a status before anything is enqueued.
 *   - Problems only visible on the device (a block id or slot out of range, a
 *     context length above the stated bound) skip the offending unit and OR a
 *     PA_ERRBIT_* bit into *dev_error_word (a device unsigned int the caller
 *     zeroes and reads after synchronising; may be NULL).  No kernel traps,
 *     asserts or spins without a bound.
 *   - Launch failures return PA_ERR_CUDA (the CUDA error is left for
 *     cudaGetLastError).
 *
 * Block layout (both pools of a layer):
 *   k_cache, v_cache: [num_blocks][num_kv_heads][PA_BLOCK_SIZE][head_dim]
 *   element type pa_dtype_t (PA_F16 or PA_BF16).  Token t of a sequence lives
 *   at block block_tables[s][t / 16], offset t % 16, for every KV head
 *   [Paged Attention: Managing the KV Cache Like Virtual Memory, "A paged KV
 *   cache, in code": pools of [blocks, key-value heads, 16 tokens, head
 *   dimension]; "Attention over scattered blocks": row() addressing].
 */
#ifndef PA_GB300_H
#define PA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st *), declared without CUDA headers. */
typedef struct CUstream_st *pa_stream_t;

typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2 } pa_dtype_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned base, bad enum */
    PA_ERR_UNSUPPORTED = 2,   /* a size no kernel of the library handles */
    PA_ERR_CUDA = 3,          /* a CUDA launch or attribute call failed */
    PA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required */
    PA_ERR_TIMEOUT = 5,       /* reserved: reported through PA_ERRBIT_TIMEOUT */
    PA_ERR_NO_BLOCKS = 6      /* block manager (pa_bm.h): not enough free blocks */
} pa_status_t;

#define PA_BLOCK_SIZE 16

/* Block sizes the *_ex entry points accept: powers of two in this range.  A
 * pool of block size B is [num_blocks][num_kv_heads][B][head_dim] and token t
 * of a sequence lives at block block_tables[s][t / B], offset t % B
 * [Efficient Memory Management ..., "PagedAttention Algorithm": the KV cache
 * is split into blocks of B tokens; Paged Attention: Managing the KV Cache
 * ..., benchmark section: the same kernel over a range of block sizes]. */
#define PA_MIN_BLOCK_SIZE 8
#define PA_MAX_BLOCK_SIZE 256

/* Bits OR-ed into *dev_error_word by the kernels. */
#define PA_ERRBIT_BLOCK_OOB   1u  /* a block id (table entry or copy pair) outside [0, num_blocks) */
#define PA_ERRBIT_SLOT_OOB    2u  /* a slot >= num_blocks * block size */
#define PA_ERRBIT_CONTEXT_LEN 4u  /* context_lens[s] < 0 or > max_context_len */
#define PA_ERRBIT_TIMEOUT     8u  /* a bounded wait inside a kernel gave up */
/* Only in a library built with -DPA_DEBUG: a work item or partition index
 * that the decode plan produced failed the kernels' consistency checks (a
 * sequence, token range or partition slot out of range); the item is skipped.
 * A production build never sets it. */
#define PA_ERRBIT_INTERNAL   16u

/*
 * pa_cache_write -- write each new token's key and value rows into the pool
 * slot named by slot_mapping.
 *
 * Defines: for every token t with slot = slot_mapping[t] >= 0 and every KV head
 * h, k_cache[slot / 16][h][slot % 16][:] = key[t][h][:], and the same for
 * value / v_cache; the bytes are copied unchanged.  slot_mapping[t] < 0 skips
 * token t (padding).
 * [Efficient Memory Management ..., "Kernel-Level Optimizations", 1. fused
 * reshape and block write; Paged Attention: Managing the KV Cache ...,
 * PagedLayer.update (writes through block and offset) and the slot-mapping
 * note after the interleaving test]
 *
 * key, value    device, [num_tokens][num_kv_heads][head_dim], dtype
 * k_cache, v_cache  device pools, layout above, written in place
 * slot_mapping  device int64 [num_tokens]
 * head_dim      64, 128 or 256
 * dev_error_word  device, may be NULL: PA_ERRBIT_SLOT_OOB for a slot past the
 *               pool (that token is skipped)
 * Distinct tokens must name distinct slots (two writes to one slot race).
 */
pa_status_t pa_cache_write(const void *key, const void *value, void *k_cache, void *v_cache,
                           const int64_t *slot_mapping, int num_tokens, int num_blocks,
                           int num_kv_heads, int head_dim, pa_dtype_t dtype,
                           unsigned int *dev_error_word, pa_stream_t stream);

/*
 * pa_cache_write_ex -- pa_cache_write for pools of block_size tokens per
 * block: k_cache[slot / block_size][h][slot % block_size][:] = key[t][h][:].
 * block_size: a power of two in [PA_MIN_BLOCK_SIZE, PA_MAX_BLOCK_SIZE]
 * (others: PA_ERR_UNSUPPORTED).  pa_cache_write(...) is
 * pa_cache_write_ex(..., num_blocks, PA_BLOCK_SIZE, ...).
 */
pa_status_t pa_cache_write_ex(const void *key, const void *value, void *k_cache,
                              void *v_cache, const int64_t *slot_mapping, int num_tokens,
                              int num_blocks, int block_size, int num_kv_heads, int head_dim,
                              pa_dtype_t dtype, unsigned int *dev_error_word,
                              pa_stream_t stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode_attention
 * needs for these sizes (0 never; always at least the scheduling header).
 * The result depends only on its arguments.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int max_context_len);

/*
 * pa_decode_partition_tokens -- context-partition size (tokens: 256 or 512)
 * that pa_decode_attention uses for these sizes.  A
 * sequence longer than this is split into partitions whose partial results
 * a merge kernel combines; the merge kernel is enqueued only when
 * max_context_len exceeds it.  Returns 0 for invalid sizes.
 */
int pa_decode_partition_tokens(int num_seqs, int num_kv_heads, int max_context_len);

/*
 * pa_decode_kernel_launches -- how many kernels pa_decode_attention (and its
 * _ex and _noalloc forms) enqueues for these sizes: the plan, one attention
 * kernel or, when shared-prefix items may form with one query head per KV
 * head, two (the tensor-core kernel for the shared prefixes, the CUDA-core
 * kernel for the rest), and the merge when a sequence may have more than one
 * partition.  1 (the attention kernel alone) for a batch of at most 256
 * (sequence, KV head) pairs whose contexts fit one partition and that forms
 * no shared-prefix items.  0 for invalid sizes.  Host only, no CUDA calls.
 */
int pa_decode_kernel_launches(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int max_context_len);

/*
 * pa_decode_attention -- one decode step of attention over a paged KV cache.
 *
 * Defines: for sequence s and query head h, with KV head hk = h / G,
 * G = num_heads / num_kv_heads (query heads hk*G .. hk*G+G-1 share KV head
 * hk), L = context_lens[s], and token t read at block block_tables[s][t/16],
 * offset t%16:
 *     x_t = scale * <query[s][h], k_t>,
 *     out[s][h] = sum_t exp(x_t - max x) v_t / sum_t exp(x_t - max x),
 * the standard attention equation evaluated block by block, blocks visited
 * in any order and combined exactly.  Scores, softmax and sums are computed
 * in fp32 from the 16-bit inputs.  L = 0 gives a zero row.
 * [Efficient Memory Management ..., "PagedAttention Algorithm": attention
 * equation and its block-wise reformulation; "Kernel-Level Optimizations",
 * 2. fused block read and attention; Paged Attention: Managing the KV Cache
 * ..., "Attention over scattered blocks" (running softmax for the query heads
 * that share a KV head); vLLM Internals ..., "The kernel pays for the
 * indirection" (a partition axis in the grid)]
 *
 * out           device [num_seqs][num_heads][head_dim], out_dtype = PA_F32 or
 *               the input dtype (round to nearest even from the fp32 result)
 * query         device [num_seqs][num_heads][head_dim], dtype
 * k_cache, v_cache  device pools, layout above
 * block_tables  device int32 [num_seqs][max_blocks_per_seq]; entries past a
 *               sequence's ceil(L/16) blocks are never read
 * context_lens  device int32 [num_seqs], each in [0, max_context_len]
 *               context_lens and block_tables are read as soon as the
 *               call's first kernel starts, which may be before the kernel
 *               enqueued ahead of it has finished (the call's kernels use
 *               programmatic dependent launch), so they must not be written
 *               by a kernel that lets dependents launch before writing them
 *               (ordinary kernels and copies are fine)
 * max_context_len  host-known upper bound on context_lens,
 *               <= 16 * max_blocks_per_seq
 * num_heads % num_kv_heads == 0, num_heads / num_kv_heads <= 8,
 * head_dim in {64, 128, 256}, dtype PA_F16 or PA_BF16
 * workspace     device, >= pa_decode_workspace_size(...) bytes, 256-byte
 *               aligned; holds the work plan and the per-partition partial
 *               results; its contents need no initialisation, and two calls
 *               in flight at once must not share one workspace
 * dev_error_word  device, may be NULL: PA_ERRBIT_BLOCK_OOB (the block is
 *               skipped), PA_ERRBIT_CONTEXT_LEN (the sequence gets a zero
 *               row), PA_ERRBIT_TIMEOUT
 * Shared prefixes: when consecutive sequences' tables start with the same
 * block ids (beam search, parallel sampling, a common prompt), the blocks
 * that are full in all of them are read once for the run, with every
 * member's query, and merged with each member's own remainder; the result
 * is each sequence's own attention either way.  Detection looks only at the
 * ids, for head_dim <= 128, num_heads / num_kv_heads <= 4,
 * 2 <= num_seqs <= 4096 and max_context_len >= 256.
 * [Efficient Memory Management ..., "Shared prefix" and "Beam search": one
 * physical copy of shared blocks serves every sequence that maps them]
 *
 * Enqueues, chained with programmatic dependent launch: a plan kernel (the
 * work lists), one attention kernel (or two: shared prefixes on the
 * tensor-core kernel and the rest on the CUDA-core kernel when
 * num_heads == num_kv_heads), and a merge kernel when a sequence may have
 * more than one partition.  A small batch (at most 256 (sequence, KV head)
 * pairs, every context within one partition, no shared prefixes) skips the
 * plan: the attention kernel takes the pairs directly.
 * pa_decode_kernel_launches gives the count.
 */
pa_status_t pa_decode_attention(void *out, pa_dtype_t out_dtype, const void *query,
                                const void *k_cache, const void *v_cache,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, int max_context_len,
                                int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int num_blocks, float scale, pa_dtype_t dtype,
                                void *workspace, size_t workspace_bytes,
                                unsigned int *dev_error_word, pa_stream_t stream);

/*
 * pa_decode_attention_ex -- pa_decode_attention over pools of block_size
 * tokens per block: token t of sequence s is read at block
 * block_tables[s][t / block_size], offset t % block_size; max_context_len
 * <= block_size * max_blocks_per_seq.  block_size: a power of two in
 * [PA_MIN_BLOCK_SIZE, PA_MAX_BLOCK_SIZE] (others: PA_ERR_UNSUPPORTED).
 * Results do not depend on the block size.  Workspace, errors and kernels
 * are those of pa_decode_attention, which is
 * pa_decode_attention_ex(..., num_blocks, PA_BLOCK_SIZE, ...).
 */
pa_status_t pa_decode_attention_ex(void *out, pa_dtype_t out_dtype, const void *query,
                                   const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, int max_context_len,
                                   int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                   int num_blocks, int block_size, float scale,
                                   pa_dtype_t dtype, void *workspace, size_t workspace_bytes,
                                   unsigned int *dev_error_word, pa_stream_t stream);

/*
 * pa_prefill_workspace_size -- bytes of device workspace pa_prefill_attention
 * needs for these sizes: the work list (8-16 bytes per work item) and room
 * for the partial results of up to 160 split items (4 x 128 x (head_dim + 2)
 * floats each); 0 if the sizes are invalid (head_dim not 64 or 128, heads not
 * a multiple of KV heads).  Host only, no CUDA calls.
 */
size_t pa_prefill_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                 int max_query_len);

/*
 * pa_prefill_attention -- chunked-prefill attention over the paged KV cache:
 * every new token of a batch of sequences attends causally over its
 * sequence's cached tokens up to its own position.
 *
 * Defines: sequence s has n_s = query_start_loc[s+1] - query_start_loc[s] new
 * tokens, query rows query_start_loc[s] .. query_start_loc[s+1]-1, whose K/V
 * are already in the cache (pa_cache_write) as the sequence's last n_s of
 * context_lens[s] positions.  New token i (0-based) is at position
 * p = context_lens[s] - n_s + i, and for query head h (KV head h / G):
 *     out[t][h] = sum_{j <= p} exp(x_j - max x) v_j / sum_{j <= p} exp(x_j - max x),
 *     x_j = scale * <query[t][h], k_j>,
 * with token j of the sequence read at block block_tables[s][j / block_size],
 * offset j % block_size.  A sequence with n_s = 1 is a decode step; one with
 * context_lens[s] = n_s is a whole prompt.  fp32 accumulation; P V uses the
 * probabilities rounded to the operand type (in two parts for bf16).
 * [Efficient Memory Management ..., "End-to-End Decoding": the prompt phase
 * computes and stores the KV cache of all prompt tokens and attends over them
 * in one pass; "PagedAttention Algorithm"; vLLM Internals ..., the
 * scheduler's chunked prefill, a prompt processed a token budget at a time]
 *
 * out           device [num_tokens][num_heads][head_dim], out_dtype = PA_F32
 *               or the input dtype (round to nearest even)
 * query         device [num_tokens][num_heads][head_dim], dtype
 * k_cache, v_cache  device pools [num_blocks][num_kv_heads][block_size][head_dim]
 * block_tables  device int32 [num_seqs][max_blocks_per_seq]
 * query_start_loc  device int32 [num_seqs + 1], non-decreasing from 0 to
 *               num_tokens
 * context_lens  device int32 [num_seqs], n_s <= context_lens[s] <= max_context_len
 * max_query_len host-known bound on n_s; max_context_len host-known bound on
 *               context_lens, <= block_size * max_blocks_per_seq
 * head_dim 64 or 128 (PA_ERR_UNSUPPORTED otherwise); block_size a power of
 * two in [PA_MIN_BLOCK_SIZE, PA_MAX_BLOCK_SIZE]; num_heads % num_kv_heads == 0
 * workspace     device, >= pa_prefill_workspace_size(...) bytes, 256-byte
 *               aligned (PA_ERR_WORKSPACE otherwise); holds the work list and
 *               the partial results of split items.  Calls in flight at once
 *               must not share one workspace.
 * dev_error_word  device, may be NULL: PA_ERRBIT_CONTEXT_LEN for a sequence
 *               whose lengths break the rules above (its rows are zeroed),
 *               PA_ERRBIT_BLOCK_OOB (the block's keys are skipped),
 *               PA_ERRBIT_TIMEOUT.
 * Enqueues two kernels: a plan (one CTA: the work items -- two 128-token
 * query tiles that read the same keys -- that have work, heaviest first; an
 * item with more than twice an SM's even share of the K/V tiles is split in
 * two parts over its keys, merged exactly by the part that finishes second)
 * and the
 * attention kernel (persistent, one CTA per SM, taking entries from the list
 * in order).
 */
pa_status_t pa_prefill_attention(void *out, pa_dtype_t out_dtype, const void *query,
                                 const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *query_start_loc, const int32_t *context_lens,
                                 int max_query_len, int max_context_len, int num_seqs,
                                 int num_tokens, int num_heads, int num_kv_heads, int head_dim,
                                 int num_blocks, int block_size, float scale, pa_dtype_t dtype,
                                 void *workspace, size_t workspace_bytes,
                                 unsigned int *dev_error_word, pa_stream_t stream);

/*
 * pa_decode_attention_contiguous -- the same decode attention over a
 * contiguous (unpaged) KV cache: sequence s's tokens for KV head hk are rows
 * 0 .. context_lens[s]-1 of k_cache[s][hk] and v_cache[s][hk]; no block
 * table.  This is the layout a paged cache replaces; the entry point exists
 * to measure what the table indirection costs on this GPU
 * [Efficient Memory Management ..., "Kernel-Level Optimizations" (the paged
 * kernel against FasterTransformer's contiguous one); Paged Attention:
 * Managing the KV Cache ..., "Attention over scattered blocks" (the same
 * kernel with and without the table)].
 *
 * k_cache, v_cache  device [num_seqs][num_kv_heads][max_rows][head_dim], dtype
 * max_rows      rows per (sequence, KV head): a multiple of 16, >= max_context_len
 * Every other argument, the workspace (pa_decode_workspace_size) and the
 * error behaviour are those of pa_decode_attention.
 */
pa_status_t pa_decode_attention_contiguous(void *out, pa_dtype_t out_dtype, const void *query,
                                           const void *k_cache, const void *v_cache,
                                           int max_rows, const int32_t *context_lens,
                                           int max_context_len, int num_seqs, int num_heads,
                                           int num_kv_heads, int head_dim, float scale,
                                           pa_dtype_t dtype, void *workspace,
                                           size_t workspace_bytes,
                                           unsigned int *dev_error_word, pa_stream_t stream);

/* Size of the workspace array built into the library for
 * pa_decode_attention_noalloc (32 MiB on every GPU that loads the library). */
#define PA_NOALLOC_WORKSPACE_BYTES (32u << 20)

/*
 * pa_decode_attention_noalloc -- pa_decode_attention for callers that cannot
 * allocate device memory.  The paper has no counterpart: this entry point
 * exists for callers of this library, not for the method.
 *
 * Who needs it: code that runs attention where allocation is not allowed or
 * not reachable -- inside another engine's execution phase (plugins whose
 * enqueue step must not allocate, because all memory is planned up front),
 * or from C code whose device allocator belongs to a framework it cannot
 * call.  Such callers still own query, pools, tables, lengths and out, but
 * cannot provide a workspace.
 *
 * Arguments, results and errors are those of pa_decode_attention, without
 * the workspace: the workspace is an array of PA_NOALLOC_WORKSPACE_BYTES
 * built into the library, which every GPU that loads the library keeps until
 * the process exits.  It calls no allocator (no cudaMalloc, cudaFree or
 * allocating library routine).
 *   - Arguments are checked exactly as pa_decode_attention checks them, in
 *     the same order; otherwise valid sizes whose pa_decode_workspace_size
 *     exceeds PA_NOALLOC_WORKSPACE_BYTES are then rejected with
 *     PA_ERR_WORKSPACE.  Nothing is enqueued on any error.
 *   - Every call looks up the array's device address (cudaGetSymbolAddress)
 *     in the context current at the call, so a device reset or another
 *     context on the same device is followed.  The first call in a context
 *     loads the library's device code there; make that first call before any
 *     stream capture.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents; nothing in it needs to start at zero.  Calls that overlap on
 *     the GPU (e.g. on unordered streams) race on it: order them.
 */
pa_status_t pa_decode_attention_noalloc(void *out, pa_dtype_t out_dtype, const void *query,
                                        const void *k_cache, const void *v_cache,
                                        const int32_t *block_tables, int max_blocks_per_seq,
                                        const int32_t *context_lens, int max_context_len,
                                        int num_seqs, int num_heads, int num_kv_heads,
                                        int head_dim, int num_blocks, float scale,
                                        pa_dtype_t dtype, unsigned int *dev_error_word,
                                        pa_stream_t stream);

/* Upper bound on num_layers accepted by pa_copy_blocks. */
#define PA_MAX_LAYERS 128

/*
 * pa_copy_blocks -- copy-on-write block copies, every pair and every layer in
 * one launch.
 *
 * Defines: for every layer l < num_layers and pair i < num_pairs with
 * (src, dst) = (block_pairs[2i], block_pairs[2i+1]):
 *     k_caches[l][dst] = k_caches[l][src] and v_caches[l][dst] = v_caches[l][src],
 * whole blocks (num_kv_heads * 16 * head_dim elements), bytes unchanged;
 * the source blocks are left as they were.
 * [Efficient Memory Management ..., "Kernel-Level Optimizations", 3. fused
 * block copy; "Copy-on-write mechanism" (copy the entire old block into the
 * new one)]
 *
 * k_caches, v_caches  HOST arrays of num_layers device pool pointers, each
 *               pool [num_blocks][num_kv_heads][16][head_dim]
 * block_pairs   device int64 [num_pairs][2] (src, dst)
 * num_layers    1 .. PA_MAX_LAYERS
 * Each dst must be distinct and must not be another pair's src (true of
 * copy-on-write, whose destinations are fresh blocks); a pair with
 * src == dst is a no-op.
 * dev_error_word  device, may be NULL: PA_ERRBIT_BLOCK_OOB (pair skipped)
 */
pa_status_t pa_copy_blocks(void *const *k_caches, void *const *v_caches, int num_layers,
                           const int64_t *block_pairs, int num_pairs, int num_blocks,
                           int num_kv_heads, int head_dim, pa_dtype_t dtype,
                           unsigned int *dev_error_word, pa_stream_t stream);

/*
 * pa_copy_blocks_ex -- pa_copy_blocks for pools of block_size tokens per
 * block (whole blocks of num_kv_heads * block_size * head_dim elements).
 * block_size: a power of two in [PA_MIN_BLOCK_SIZE, PA_MAX_BLOCK_SIZE]
 * (others: PA_ERR_UNSUPPORTED).  pa_copy_blocks(...) is
 * pa_copy_blocks_ex(..., num_blocks, PA_BLOCK_SIZE, ...).
 */
pa_status_t pa_copy_blocks_ex(void *const *k_caches, void *const *v_caches, int num_layers,
                              const int64_t *block_pairs, int num_pairs, int num_blocks,
                              int block_size, int num_kv_heads, int head_dim, pa_dtype_t dtype,
                              unsigned int *dev_error_word, pa_stream_t stream);

/*
 * pa_swap_blocks -- move whole blocks between two pools, every pair and
 * every layer in one launch: the swap-out of a preempted sequence's blocks
 * from the GPU pool to a CPU swap space, and the swap-in that brings them
 * back when it resumes.
 *
 * Defines: for every layer l < num_layers and pair i < num_pairs with
 * (src, dst) = (block_pairs[2i], block_pairs[2i+1]):
 *     dst_k_caches[l][dst] = src_k_caches[l][src] and the same for V,
 * whole blocks (num_kv_heads * block_size * head_dim elements), bytes
 * unchanged; the source pools are left as they were.
 * [Efficient Memory Management ..., "Scheduling and Preemption": swapping
 * copies the evicted blocks to CPU RAM and back to GPU DRAM when the
 * sequence is rescheduled, with a CPU block allocator beside the GPU one;
 * the swap-space bound (never more blocks than the GPU pool holds) is the
 * caller's allocator's to keep]
 *
 * dst_k_caches, dst_v_caches, src_k_caches, src_v_caches
 *               HOST arrays of num_layers pool pointers.  Each pool is
 *               [num_blocks][num_kv_heads][block_size][head_dim] with
 *               num_dst_blocks / num_src_blocks blocks, and is either device
 *               memory of the current device, managed memory, or pinned
 *               (page-locked, mapped) host memory such as cudaHostAlloc or
 *               cudaHostRegister gives; the kernel reads and writes host pools
 *               directly through their device mapping.  Pageable host memory
 *               is refused (PA_ERR_INVALID_ARG) before anything is enqueued.
 * block_pairs   int64 [num_pairs][2] (src, dst), device or pinned host memory
 * block_size    a power of two in [PA_MIN_BLOCK_SIZE, PA_MAX_BLOCK_SIZE]
 * num_layers    1 .. PA_MAX_LAYERS
 * Each dst must be distinct; src == dst is a real copy (two pools).  The
 * host memory must stay pinned until the work on `stream` has finished.
 * dev_error_word  device, may be NULL: PA_ERRBIT_BLOCK_OOB (pair skipped)
 */
pa_status_t pa_swap_blocks(void *const *dst_k_caches, void *const *dst_v_caches,
                           const void *const *src_k_caches, const void *const *src_v_caches,
                           int num_layers, const int64_t *block_pairs, int num_pairs,
                           int num_dst_blocks, int num_src_blocks, int block_size,
                           int num_kv_heads, int head_dim, pa_dtype_t dtype,
                           unsigned int *dev_error_word, pa_stream_t stream);

/* Static, human-readable name of a status. */
const char *pa_status_string(pa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* PA_GB300_H */
