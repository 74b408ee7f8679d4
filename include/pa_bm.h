/*
 * pa_bm.h -- C ABI of the host-side KV block manager (CPU code, no GPU work).
 *
 * The bookkeeping above the kernels: it hands out physical blocks of the GPU
 * pool and of a CPU swap space, counts references, forks sequences (sharing
 * every block), appends tokens with copy-on-write of a shared, partially
 * filled last block, frees, and swaps whole sequence groups out to the CPU
 * space and back.  It produces exactly the kernels' inputs: block tables and
 * context lengths (pa_decode_attention), the slot of every new token
 * (pa_cache_write), copy-on-write pairs (pa_copy_blocks) and swap pairs
 * (pa_swap_blocks).  No data moves here.
 * [Efficient Memory Management for Large Language Model Serving with
 * PagedAttention, "KV Cache Manager: Block Table Mapping", "The three
 * primitive operations", "Copy-on-write mechanism", "Scheduling and
 * Preemption" (all-or-nothing eviction of a sequence group; swapping to a CPU
 * block allocator that mirrors the GPU one); vLLM Internals ..., "PagedAttention:
 * page tables, for KV" (block allocator with reference counts); Paged
 * Attention: Managing the KV Cache Like Virtual Memory, "A paged KV cache, in
 * code" (Sequence.reserve / fork / free; slot = block * B + offset)]
 *
 * Allocation order: the lowest free block id first, after any ids given to
 * pa_bm_set_free_order (the order the pages' worked examples print).
 *
 * Conventions: sequences are named by the int64 ids the manager returns;
 * every call is all-or-nothing (on an error nothing changes); a manager may
 * be used from several threads (calls are serialised inside).  Errors:
 * PA_ERR_INVALID_ARG (bad size, unknown sequence, a sequence in the wrong
 * place), PA_ERR_NO_BLOCKS (not enough free blocks).
 */
#ifndef PA_GB300_BM_H
#define PA_GB300_BM_H

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager_t;

/* New manager: GPU block ids 0 .. num_gpu_blocks-1, CPU swap-space ids
 * 0 .. num_cpu_blocks-1 (0: no swap space), block_size tokens per block
 * (any positive size; the kernels take 8..256).  *out gets the handle. */
pa_status_t pa_bm_create(int num_gpu_blocks, int num_cpu_blocks, int block_size,
                         pa_block_manager_t **out);
void pa_bm_destroy(pa_block_manager_t *bm);

/* Hand out these free GPU block ids first, in this order (then the rest,
 * lowest first).  Only on a manager with no block in use. */
pa_status_t pa_bm_set_free_order(pa_block_manager_t *bm, const int32_t *order, int n);

int pa_bm_num_free_gpu(const pa_block_manager_t *bm);
int pa_bm_num_free_cpu(const pa_block_manager_t *bm);
int pa_bm_block_size(const pa_block_manager_t *bm);
/* Reference count of a GPU (on_cpu = 0) or CPU block; -1 for a bad id. */
int pa_bm_refcount(const pa_block_manager_t *bm, int on_cpu, int block);

/* A new, empty sequence. */
pa_status_t pa_bm_seq_create(pa_block_manager_t *bm, int64_t *seq_out);
/* A child sharing every block of `parent` (references + 1 each), same length. */
pa_status_t pa_bm_seq_fork(pa_block_manager_t *bm, int64_t parent, int64_t *child_out);
/* Release every block of the sequence (GPU or CPU) and forget it. */
pa_status_t pa_bm_seq_free(pa_block_manager_t *bm, int64_t seq);
/* Make room for num_tokens more tokens of a sequence in the GPU pool: if its
 * last block is partially filled and shared, copy it first (a fresh block;
 * the (old, new) pair is queued for pa_bm_take_copies), then append blocks
 * until the tokens fit.  slots_out (may be NULL) gets the num_tokens slots,
 * slot = block * block_size + offset.  PA_ERR_NO_BLOCKS if the pool cannot
 * hold them (nothing changes). */
pa_status_t pa_bm_seq_append(pa_block_manager_t *bm, int64_t seq, int num_tokens,
                             int64_t *slots_out);
/* GPU blocks that appending num_tokens would allocate (copy included); -1 for
 * an unknown sequence or one in the swap space. */
int pa_bm_blocks_needed(const pa_block_manager_t *bm, int64_t seq, int num_tokens);
/* Stored tokens of a sequence; -1 if unknown. */
int pa_bm_seq_len(const pa_block_manager_t *bm, int64_t seq);
/* 1 if the sequence's blocks are in the CPU swap space, 0 on the GPU, -1 unknown. */
int pa_bm_seq_on_cpu(const pa_block_manager_t *bm, int64_t seq);
/* The sequence's block table: copies min(cap, blocks) ids to out (may be
 * NULL with cap 0) and returns the number of blocks; -1 if unknown. */
int pa_bm_seq_table(const pa_block_manager_t *bm, int64_t seq, int32_t *out, int cap);

/* Kernel inputs for a batch of GPU-resident sequences: block_tables
 * [n][max_blocks_per_seq] (entries past a sequence's blocks are -1) and
 * context_lens [n], host memory.  PA_ERR_INVALID_ARG if a sequence is
 * unknown, swapped out, or has more blocks than max_blocks_per_seq. */
pa_status_t pa_bm_build_batch(const pa_block_manager_t *bm, const int64_t *seqs, int n,
                              int32_t *block_tables, int max_blocks_per_seq,
                              int32_t *context_lens);

/* Copy-on-write pairs queued so far, oldest first: moves up to cap pairs to
 * pairs_out ([cap][2] int64, (src, dst)) and returns how many it moved;
 * pa_bm_num_copies tells how many are queued. */
int pa_bm_take_copies(pa_block_manager_t *bm, int64_t *pairs_out, int cap);
int pa_bm_num_copies(const pa_block_manager_t *bm);

/* Swap a sequence group out of the GPU pool (all or nothing): every distinct
 * GPU block of the n sequences gets a CPU block with the same reference
 * count, and is freed on the GPU; the sequences' tables now name CPU ids.
 * pairs_out ([cap][2] int64) gets the (gpu, cpu) pairs for pa_swap_blocks,
 * *num_pairs their number.  The group must hold every reference to its
 * blocks (PA_ERR_INVALID_ARG otherwise), the sequences must be on the GPU,
 * cap must be >= the distinct block count; PA_ERR_NO_BLOCKS if the swap
 * space is short. */
pa_status_t pa_bm_swap_out(pa_block_manager_t *bm, const int64_t *seqs, int n,
                           int64_t *pairs_out, int cap, int *num_pairs);
/* The reverse: (cpu, gpu) pairs; the sequences must be in the swap space. */
pa_status_t pa_bm_swap_in(pa_block_manager_t *bm, const int64_t *seqs, int n,
                          int64_t *pairs_out, int cap, int *num_pairs);

#ifdef __cplusplus
}
#endif

#endif /* PA_GB300_BM_H */
