/*
 * Host block manager of the paged KV cache: which physical blocks each
 * sequence owns, prefix-cache reuse of full blocks, and the progress of a
 * chunked prefill.  Its block tables feed pa_prepare_prefill /
 * pa_prepare_decode (slot_mapping, block_tables) of pa.h.
 *
 * "nano-vllm notes - Llama", scheduler.py and model_runner.py: the
 * BlockManager decides whether a request's blocks can be allocated and how
 * many of its blocks a prefix-cache hit lets it reuse (those tokens are not
 * prefilled again, only the rest); before a decode step it checks that a
 * sequence has room for one more token; a preempted or finished request
 * gives its blocks back; block_tables tell attention where the old tokens
 * of a prefix-cache hit or of an earlier prefill chunk are.  The page does
 * not say how blocks are matched, so (a reading, stated here):
 *   - only full blocks (block_size tokens) are shared;
 *   - block i of a sequence is identified by a 64-bit chained hash
 *     h_i = H(h_{i-1}, tokens of block i), h_{-1} = 0 (FNV-1a over the
 *     previous hash's and the tokens' bytes), so a block matches only when
 *     its whole prefix matches; a hash hit is confirmed by comparing the
 *     stored tokens;
 *   - matching stops at the first block that misses;
 *   - a fully matched prompt still recomputes its last token (the caller
 *     needs that token's attention output), so num_cached <= tokens - 1;
 *   - a freed block keeps its hash and can be matched again until it is
 *     handed out anew (free blocks are reused oldest-freed first; a
 *     sequence's blocks are freed last block first).
 * A block's hash is registered when the block is allocated full (prompt) or
 * becomes full (decode).  Its K/V are written by the pa_rope_kv_write of
 * the step that computes those tokens, which precedes in stream order the
 * attention of any later sequence that matches it, including one in the
 * same batch.
 *
 * Single-threaded host object: callers serialise calls on one manager.
 * Sequence ids are caller-chosen 64-bit integers.  Errors: PA_ERR_INVALID
 * (unknown or duplicate sequence, bad argument), PA_ERR_WORKSPACE (not
 * enough free blocks: nothing changed).
 */
#ifndef PA_BLOCK_MANAGER_H
#define PA_BLOCK_MANAGER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager *pa_bm_t;

/* A manager of num_blocks blocks of block_size tokens; NULL on bad sizes
 * (either not positive, or num_blocks * block_size past INT32_MAX: slot ids
 * are int32). */
pa_bm_t pa_bm_create(int num_blocks, int block_size);
void pa_bm_destroy(pa_bm_t bm);

/* Free blocks (including freed blocks still matchable by their hash). */
int pa_bm_num_free(pa_bm_t bm);

/* Blocks a new prompt of num_tokens tokens needs if nothing matches. */
int pa_bm_blocks_needed(pa_bm_t bm, int num_tokens);

/*
 * Admit sequence seq_id with its prompt tokens[0 .. num_tokens): reuse the
 * matching full blocks, take free blocks for the rest.  *num_cached receives
 * the tokens whose K/V are already in the cache (a multiple of block_size,
 * at most num_tokens - 1); the sequence's prefill starts there.
 */
int pa_bm_allocate(pa_bm_t bm, int64_t seq_id, const int32_t *tokens, int num_tokens,
                   int *num_cached);

/*
 * Chunked prefill: the next chunk of at most max_tokens (> 0) prompt tokens
 * of seq_id to compute: *num_cached = tokens already computed (or cached),
 * *num_new = min(max_tokens, prompt tokens left), 0 once the prompt is done.
 * pa_bm_mark_computed(bm, seq_id, n) records n more computed tokens.
 */
int pa_bm_next_chunk(pa_bm_t bm, int64_t seq_id, int max_tokens, int *num_cached, int *num_new);
int pa_bm_mark_computed(pa_bm_t bm, int64_t seq_id, int num_tokens);

/*
 * Decode: can seq_id take one more token (a new block is needed only when
 * its last block is full)?  1 yes, 0 no, negative on error.
 */
int pa_bm_can_append(pa_bm_t bm, int64_t seq_id);

/*
 * Decode: append `token` to seq_id, taking a new block when the last one is
 * full; the token counts as computed.  *slot receives its cache slot
 * (block * block_size + offset).  Registers a block's hash when it fills.
 */
int pa_bm_append(pa_bm_t bm, int64_t seq_id, int32_t token, int32_t *slot);

/* Tokens of seq_id (prompt + appended) and its blocks: table[0 .. n). */
int pa_bm_num_tokens(pa_bm_t bm, int64_t seq_id);
int pa_bm_block_table(pa_bm_t bm, int64_t seq_id, int32_t *table, int max_blocks,
                      int *num_blocks);

/* Give back seq_id's blocks (finished or preempted); the id may be reused. */
int pa_bm_free(pa_bm_t bm, int64_t seq_id);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H */
