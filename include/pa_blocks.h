/*
 * pa_blocks.h -- host-side manager of the paged KV cache's physical blocks.
 *
 * It produces what the attention entry points of pa.h consume: per-sequence
 * block tables, context lengths and the slot mapping of new tokens.  It follows
 * "PyTorch LLM Serving Engine", "What is implemented" (fixed-size physical
 * blocks, per-sequence block tables, an O(1) free-list allocator, memory
 * accounting, explicit recomputation counters after preemption) and "MicroGen",
 * "Key Features" (logical-to-physical block mapping; sliding window eviction;
 * KV cache state rollback when speculative tokens are rejected; "Prompt Prefix
 * Caching": token sequence hashing with sub-sequence prefix lookup).
 *
 * Layout conventions are those of pa.h: position p of a sequence lives in the
 * physical block block_tables[seq][p / block_size] at offset p % block_size,
 * slot = block * block_size + offset; table entries without a block are -1.
 *
 * Host memory only: nothing here touches a GPU.  A manager is not safe for
 * concurrent use: callers serialise calls on one manager.  Every call that can
 * fail returns a pa_status and changes nothing when it fails.
 */
#ifndef PA_BLOCKS_H
#define PA_BLOCKS_H

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_blocks pa_blocks; /* opaque */

typedef struct {
    int num_blocks;              /* physical blocks in the pool */
    int free_blocks;             /* on the free list */
    int live_seqs;               /* sequences holding at least one token */
    long long tokens_held;       /* sum of the context lengths */
    long long preemptions;       /* pa_blocks_preempt calls that freed something */
    long long recompute_tokens;  /* tokens dropped by preemption, to be computed again */
    long long evicted_blocks;    /* blocks freed by sliding-window eviction */
    long long rolled_back_tokens;/* tokens dropped by pa_blocks_rollback */
    long long published_blocks;  /* blocks registered under a prefix key */
    long long prefix_hit_blocks; /* blocks attached from the prefix cache (not recomputed) */
    int shared_blocks;           /* blocks currently held by more than one sequence */
    int cached_blocks;           /* registered blocks no sequence holds, kept for reuse */
    long long revived_blocks;    /* prefix hits on cached blocks (no holder at the time) */
    long long reclaimed_blocks;  /* cached blocks taken back for new positions (LRU) */
} pa_blocks_stats;

/*
 * pa_blocks_create -- a pool of num_blocks physical blocks of block_size tokens
 * for sequences 0 .. max_seqs-1, each holding at most max_blocks_per_seq
 * logical blocks.  window > 0 is the sliding-window length used by
 * pa_blocks_evict_window (0: no window).  Returns NULL on bad sizes or when
 * memory runs out.  The caller frees it with pa_blocks_destroy.
 */
pa_blocks *pa_blocks_create(int num_blocks, int block_size, int max_seqs,
                            int max_blocks_per_seq, int window);
void pa_blocks_destroy(pa_blocks *bm);

/*
 * pa_blocks_append -- reserve num_tokens new positions at the end of sequence
 * seq, taking blocks from the free list (O(1) each), and when it is empty from
 * the prefix cache (least recently used first, O(1) each), as the context
 * crosses block boundaries, and write the new positions' slots to
 * slots_out[num_tokens].  All or nothing: PA_ERR_OUT_OF_BLOCKS when the pool
 * lacks free and cached blocks,
 * PA_ERR_UNSUPPORTED when the sequence would exceed max_blocks_per_seq blocks,
 * PA_ERR_INVALID_ARG for a bad seq, negative num_tokens or NULL slots_out (when
 * num_tokens > 0).  The context length afterwards counts the new tokens (the
 * convention of pa.h: write, then attend).
 */
pa_status pa_blocks_append(pa_blocks *bm, int seq, int num_tokens, int32_t *slots_out);

/*
 * pa_blocks_rollback -- drop the last num_tokens positions of seq (rejected
 * speculative tokens).  Blocks left without any position are released (see
 * reference counts below); the dropped slots keep their stale contents, which no
 * attention call reads once the context is shorter, and the next append
 * overwrites.  PA_ERR_INVALID_ARG when num_tokens exceeds the context, when
 * blocks were evicted and the window of the next query (at the shortened context
 * length L2: keys L2-W+1 .. L2) would reach into them, or when L2 would end
 * inside a block another sequence shares (the next append would write into it).
 */
pa_status pa_blocks_rollback(pa_blocks *bm, int seq, int num_tokens);

/* pa_blocks_release -- the sequence is finished: it lets all its blocks go (see
 * prefix caching below: registered blocks stay in the prefix cache, the others
 * return to the free list) and its context length becomes 0. */
pa_status pa_blocks_release(pa_blocks *bm, int seq);

/*
 * pa_blocks_preempt -- free all blocks of seq to make room for others; its
 * tokens are counted in recompute_tokens (they must be prefilled again) and its
 * context length becomes 0.
 */
pa_status pa_blocks_preempt(pa_blocks *bm, int seq);

/*
 * pa_blocks_evict_window -- with a window W > 0, free the blocks of seq that no
 * query at position oldest_query or later can see: every block whose positions
 * all lie before oldest_query - W + 1 (a query at position i sees keys j with
 * i - W < j <= i).  Their table entries become -1; the attention kernels never
 * visit blocks before the window, so the freed blocks may be reused at once.
 * Writes the freed block ids to freed_out (up to cap of them; NULL allowed) and
 * returns how many blocks were freed, or -1 on a bad argument.
 */
int pa_blocks_evict_window(pa_blocks *bm, int seq, int oldest_query, int32_t *freed_out, int cap);

/*
 * pa_blocks_tables -- block tables and context lengths of sequences seqs[0..n-1]
 * in the layout of pa.h: tables_out[n][max_blocks_per_seq] (-1 where there is no
 * block), context_lens_out[n].  Either output may be NULL.
 */
pa_status pa_blocks_tables(const pa_blocks *bm, const int32_t *seqs, int n, int32_t *tables_out,
                           int32_t *context_lens_out);

/*
 * Prefix caching ("MicroGen", Key Features, "Prompt Prefix Caching"; "llminfer",
 * Architecture: a prefix cache (LRU), and its prefix-reuse example, where a
 * finished request's prompt serves the next one).  Physical blocks are reference
 * counted.  When the last sequence holding a block lets it go (release,
 * preempt, eviction, rollback), an unregistered block returns to the free list;
 * a block registered under a prefix key stays in the prefix cache with its K/V
 * and its key, so a later request with the same prefix finds it.  Allocations
 * (pa_blocks_append) take free blocks first and then reclaim cached blocks,
 * least recently let go first, dropping their keys; the blocks of one sequence
 * enter the cache last block first, so a prefix loses its later blocks before
 * its earlier ones.  free_blocks counts the free list only; append can use
 * free_blocks + cached_blocks.  Only full blocks are shared, so appends never
 * write into a shared block and no copy is ever needed.
 *
 * pa_blocks_publish -- register the first n_blocks blocks of seq, which must be
 * full (n_blocks * block_size <= its context) and not evicted, under the
 * caller's content keys keys[0..n_blocks-1] (for block i, a hash of every token
 * of the sequence up to the block's end, so that equal keys mean equal K/V).  A
 * key already registered keeps its block.  A block leaves the registry only when
 * it is reclaimed.
 *
 * pa_blocks_attach_prefix -- for an empty sequence seq, attach the longest run
 * of registered blocks matching keys[0], keys[1], ... (stopping at the first key
 * not registered, or at max_blocks_per_seq), whether other sequences hold them
 * or they wait in the prefix cache: the sequence's table starts with those
 * blocks, each gaining a reference, and its context length becomes (blocks
 * attached) * block_size.  Returns the number of blocks attached (0 when the
 * first key misses), or -1 on a bad argument or a non-empty sequence.
 */
pa_status pa_blocks_publish(pa_blocks *bm, int seq, const uint64_t *keys, int n_blocks);
int pa_blocks_attach_prefix(pa_blocks *bm, int seq, const uint64_t *keys, int n_blocks);

/* Context length of seq, or -1 for a bad seq. */
int pa_blocks_context_len(const pa_blocks *bm, int seq);

/* Memory accounting; out must not be NULL. */
pa_status pa_blocks_get_stats(const pa_blocks *bm, pa_blocks_stats *out);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCKS_H */
