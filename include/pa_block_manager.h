/*
 * pa_block_manager.h - host-side KV block manager of the paged decode path (libpa.so).
 *
 * It produces the metadata the kernels consume: per-sequence block tables,
 * context lengths, slot_mapping entries for new tokens, and (src, dst) pairs
 * for copy-on-write block copies.  Host memory only; not thread-safe (one
 * manager per scheduler thread).
 *
 * Sources (page title, section):
 *  [P1] "PagedAttention 详解：缓存的存储结构" - "Block Table" (block IDs appended in
 *       token order), "写入新 K/V" (slot = block_id * B + offset), "使用流程"
 *       (full blocks get a chained content hash h_i = hash(tokens_i, h_{i-1});
 *       hits reuse the block and raise its ref_cnt, misses take a free block).
 *  [P2] "PagedAttention 笔记" - "写时复制是正确性的边界" (a write into a block with
 *       ref_count > 1: allocate, copy, remap, ref_count--, then write).
 *  [P3] "vLLM 核心工程深度剖析" - "2.2 显存分配器实现" (allocate / append_slot / free
 *       with a free list and reference counts), "4.1 Beam Search 中的 CoW" (fork:
 *       the child shares the parent's blocks, ref += 1).
 *  [P4] "PagedAttention是什麼？" - "vLLM v1的Block Pool", "Eviction與Free Queue"
 *       (new blocks come from the head of the free queue, freed blocks go to its
 *       tail; a freed block keeps its content hash and can still be hit until the
 *       queue hands it out again, at which point its cache entry is dropped).
 *
 * Return codes: PA_BM_OK (0) or a negative PA_BM_ERR_* code; on error nothing
 * changes.
 */
#ifndef PA_BLOCK_MANAGER_H_
#define PA_BLOCK_MANAGER_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  PA_BM_OK = 0,
  PA_BM_ERR_INVALID_ARG = -1, /* NULL pointer, negative size, capacity too small */
  PA_BM_ERR_UNKNOWN_SEQ = -2, /* no sequence with that id */
  PA_BM_ERR_NO_BLOCKS = -3,   /* the free queue cannot supply the blocks needed */
  PA_BM_ERR_SEQ_EXISTS = -4   /* a sequence with that id already exists */
};

typedef struct pa_block_manager pa_block_manager; /* opaque */

/* A pool of num_blocks blocks of block_size tokens.  The free queue starts as
 * 0..num_blocks-1, or as a permutation of it drawn from `shuffle_seed` when that
 * is non-zero (splitmix64 + Fisher-Yates).  Returns NULL on invalid sizes. */
pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, uint64_t shuffle_seed);
void pa_bm_destroy(pa_block_manager* bm);

int32_t pa_bm_num_free(const pa_block_manager* bm);        /* blocks in the free queue */
int32_t pa_bm_ref_count(const pa_block_manager* bm, int32_t block); /* -1 for an invalid id */

/* New sequence `seq` holding `num_tokens` tokens in ceil(num_tokens / B) fresh blocks. */
int pa_bm_allocate(pa_block_manager* bm, int64_t seq, int32_t num_tokens);

/* New sequence `seq` whose first `num_tokens` tokens are `tokens`.  Each full
 * block's chained hash is looked up in the prefix cache: a hit reuses the
 * cached block (ref += 1), a miss takes a free block and enters it in the cache.
 * The trailing partial block is always fresh.  *num_hit_blocks (nullable) gets
 * the number of leading blocks served from the cache, whose K/V need no
 * recomputation. */
int pa_bm_allocate_with_prefix(pa_block_manager* bm, int64_t seq, const int32_t* tokens, int32_t num_tokens,
                               int32_t* num_hit_blocks);

/* Room for one more token of `seq`: returns its slot (block * B + offset) in
 * *slot.  When the last block is full a fresh block is appended.  When the
 * last block is partly filled but shared (ref_count > 1), copy-on-write: a
 * fresh block replaces it in this sequence's table, the shared block's
 * ref_count drops by one and (*cow_src, *cow_dst) is the block copy the caller
 * must run (pa_copy_blocks) before writing the token; otherwise both are -1. */
int pa_bm_append_slot(pa_block_manager* bm, int64_t seq, int64_t* slot, int32_t* cow_src, int32_t* cow_dst);

/* append_slot for n sequences at once (one decode step).  slots[n]; the copy
 * pairs go to pairs[2 * k] (src, dst) and their count to *num_pairs (pairs must
 * hold 2 * n entries).  Stops at the first error; the sequences before it keep
 * their new slots. */
int pa_bm_append_slots(pa_block_manager* bm, const int64_t* seqs, int32_t n, int64_t* slots, int32_t* pairs,
                       int32_t* num_pairs);

/* The child shares every block of the parent (ref += 1) and its length. */
int pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child);

/* Drops the sequence: ref -= 1 on each of its blocks; blocks reaching 0 go to
 * the tail of the free queue (keeping their cache entry, if any). */
int pa_bm_free(pa_block_manager* bm, int64_t seq);

/* Length (tokens) and number of blocks of `seq`; -2 if unknown. */
int32_t pa_bm_seq_len(const pa_block_manager* bm, int64_t seq);
int32_t pa_bm_num_seq_blocks(const pa_block_manager* bm, int64_t seq);

/* Largest number of blocks among seqs[0..n) (the table width a decode step
 * needs); PA_BM_ERR_UNKNOWN_SEQ / PA_BM_ERR_INVALID_ARG on errors. */
int32_t pa_bm_max_seq_blocks(const pa_block_manager* bm, const int64_t* seqs, int32_t n);

/* Decode-step metadata: row i of tables_out (width entries, zero-padded) is the
 * block table of seqs[i], lens_out[i] its length.  PA_BM_ERR_INVALID_ARG if a
 * table is wider than `width`. */
int pa_bm_build_tables(const pa_block_manager* bm, const int64_t* seqs, int32_t n, int32_t width,
                       int32_t* tables_out, int32_t* lens_out);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H_ */
