/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * The operations are the hot path that the three inference-engine pages share:
 *   - "PyTorch LLM Serving Engine", section "Loading": each layer writes K/V to a
 *     physical cache slot, then runs a numerically stable online softmax while
 *     walking the sequence's block table; section "What is implemented":
 *     fixed-size physical blocks, per-sequence block tables, chunked prefill.
 *   - "MicroGen: Modular, Hardware-Aware LLM Inference Engine", Key Features,
 *     "Paged & Quantized INT8 KV Cache": logical-to-physical block mapping,
 *     sliding-window length, GQA (repeat_kv), dynamic INT8 KV quantisation with
 *     a vector scale.
 *   - "llminfer: A GPU-efficient LLM inference engine", "Paged KV Cache And
 *     Continuous Batching": 16-token pages.
 *
 * Conventions shared by every entry point
 *   - All pointers named *_cache, k, v, q, out, slot_mapping, block_tables,
 *     context_lens, cu_q_lens, workspace and err_flag are DEVICE pointers owned
 *     by the caller; the library allocates nothing and, apart from the fixed
 *     scratch array behind pa_decode_noalloc, keeps no state between calls.
 *     `pa_cache` itself is a host struct read during the call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream) of the current
 *     device; all work is enqueued on it asynchronously and nothing is
 *     synchronised.  The caller makes the device current.
 *   - Layouts are dense row-major:
 *       k_cache, v_cache  [num_blocks][num_kv_heads][block_size][head_dim]
 *       k_scale, v_scale  [num_blocks][num_kv_heads][block_size]    (fp32, int8 only)
 *       slot              physical_block * block_size + offset; < 0 = padding
 *       block_tables      [num_seqs][max_blocks_per_seq] int32, logical -> physical
 *       context_lens      [num_seqs] int32, tokens of the sequence AFTER this
 *                         step's write (the new token attends to itself)
 *       q, out            [tokens][num_q_heads][head_dim]
 *   - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - A query at position i sees keys j in [lo, i], lo = max(0, i - window + 1)
 *     when window > 0, else 0.  A query that sees no key returns zeros.
 *   - INT8 cache rows hold code[d] with value code[d] * scale; the write computes
 *     scale = amax / 127 (fp32 IEEE division) and code = x / scale (fp32 IEEE
 *     division) rounded half to even and clamped to [-127, 127]; amax = 0 gives
 *     scale 0 and zero codes.  K and V have separate scales per (token, kv head).
 *     Each code is stored as one offset-binary byte, code + 128 (the code's
 *     two's-complement byte with its top bit flipped): the readers turn bytes
 *     into exact f16 operands (1024 + byte) without a sign fix-up.
 *   - Supported: block_size 16, head_dim 64 or 128, 16-bit caches (fp16, bf16)
 *     with q of the same type, int8 caches with fp16 or bf16 q.  `out` has q's
 *     type.  Every device pointer must be 16-byte aligned.
 *   - int8 caches: any finite magnitudes.  The kernels' tensor-core operands are
 *     f16; a bf16 query row beyond the f16 range is scaled by a power of two
 *     into it (and its scores back), and each token's V scale enters the P V
 *     product relative to a running reference, so rows of any scale (1e-30 or
 *     1e30 with bf16 q and output), mixed in one sequence, keep errors relative
 *     to the output.
 *
 * Errors
 *   - Problems visible on the host (NULL pointers, unsupported shapes or types,
 *     misalignment, workspace too small) return a status other than PA_OK and
 *     launch nothing.  A failed launch returns PA_ERR_CUDA.
 *   - Bad DEVICE data never traps: the offending row is skipped (slot or block id
 *     out of range) or clamped (context length) and a PA_FLAG_* bit is OR-ed into
 *     *err_flag, which the caller zeroes before and reads after the work.
 *     pa_check_flags() turns a flag word into PA_ERR_DEVICE_DATA.
 *   - Every wait inside a kernel is bounded; a wait that runs out sets
 *     PA_FLAG_TIMEOUT and the kernel returns without writing its outputs.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,
    PA_ERR_UNSUPPORTED = 2,
    PA_ERR_CUDA = 3,
    PA_ERR_DEVICE_DATA = 4,
    PA_ERR_OUT_OF_BLOCKS = 5 /* pa_blocks.h: the pool has too few free blocks */
} pa_status;

typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_I8 = 2 } pa_dtype;

/* Bits OR-ed into *err_flag by the kernels. */
enum {
    PA_FLAG_SLOT_RANGE = 1,   /* slot >= num_blocks * block_size: token skipped */
    PA_FLAG_BLOCK_ID = 2,     /* block-table entry outside [0, num_blocks): block's keys left out */
    PA_FLAG_CONTEXT_LEN = 4,  /* context length < 0 or > max_blocks_per_seq * block_size: clamped */
    PA_FLAG_Q_LEN = 8,        /* bad cu_q_lens entry (negative, decreasing, > max_q_len, > context,
                                 past num_q_tokens): the chunk is clamped or skipped */
    PA_FLAG_TIMEOUT = 16      /* a bounded in-kernel wait ran out; outputs not written */
};

/* The paged cache.  Host struct; its pointers are device pointers. */
typedef struct {
    int num_blocks;    /* physical blocks in the pool (>= 1) */
    int block_size;    /* tokens per block: 16 */
    int num_kv_heads;  /* >= 1 */
    int head_dim;      /* 64 or 128 */
    pa_dtype dtype;    /* PA_F16, PA_BF16 or PA_I8 */
    void *k_cache;     /* [num_blocks][num_kv_heads][block_size][head_dim] */
    void *v_cache;
    float *k_scale;    /* [num_blocks][num_kv_heads][block_size]; PA_I8 only, else NULL */
    float *v_scale;
} pa_cache;

/*
 * pa_write_kv -- scatter the new tokens' K and V rows into their cache slots
 * ("PyTorch LLM Serving Engine", "Loading": K/V written to a physical cache
 * slot; "MicroGen", Key Features: dynamic INT8 KV quantisation, vector scale).
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim] of in_dtype (PA_F16/PA_BF16)
 *   slot_mapping  [num_tokens] int32; token t goes to block slot/16, offset slot%16;
 *                 slot < 0 skips the token; slot >= num_blocks*16 skips it and sets
 *                 PA_FLAG_SLOT_RANGE.  Two tokens must not name the same slot.
 *   16-bit caches: in_dtype must equal cache->dtype; the bits are copied.
 *   int8 caches: each (token, kv head) row of K and of V is quantised with its
 *                own scale (rule above); codes and scale are stored.
 *   Slots not named are left untouched.  num_tokens == 0 is a no-op.
 */
pa_status pa_write_kv(const pa_cache *cache, const void *k, const void *v, pa_dtype in_dtype,
                      const int32_t *slot_mapping, int num_tokens, int32_t *err_flag,
                      void *stream);

/*
 * pa_decode -- one query per sequence attends to its whole paged context
 * ("PyTorch LLM Serving Engine", "Loading": online softmax while traversing the
 * block table; "MicroGen", Key Features: GQA, sliding window).  The query of
 * sequence b sits at position context_lens[b] - 1.
 *
 *   q, out        [num_seqs][num_q_heads][head_dim]
 *   sm_scale      multiplies q.k (1/sqrt(head_dim) is the usual choice)
 *   window        0 = no window; W > 0 keeps the last W keys (self included)
 *   workspace     device scratch for split-K partials, at least
 *                 pa_decode_workspace_bytes(...) bytes (may be NULL if that is 0)
 *
 * Long contexts are cut into partitions of whole blocks, each with its own
 * online-softmax state (max, normaliser, unnormalised output); the states go to
 * the workspace and a second kernel merges them.  The partition size (64 blocks,
 * halved while the batch leaves SMs without two CTAs each) is chosen from the
 * batch shape and the device's SM count; the result does not depend on it
 * beyond rounding.  A small batch whose block tables span at most 256 blocks and
 * whose (sequence, kv head) pairs fill the SMs at 16 CTAs each is instead split
 * into 16 partitions per sequence that merge inside the launch (a thread-block
 * cluster; no workspace needed: pa_decode_workspace_bytes returns 0).
 * pa_decode_partitioned chooses the partitioning explicitly.
 */
pa_status pa_decode(const pa_cache *cache, void *out, const void *q, pa_dtype q_dtype,
                    int num_seqs, int num_q_heads, const int32_t *block_tables,
                    int max_blocks_per_seq, const int32_t *context_lens, float sm_scale,
                    int window, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                    void *stream);

/*
 * pa_decode_partitioned -- pa_decode with an explicit partitioning:
 *   partition_blocks >= 1   partitions of that many blocks, merged through the
 *                           workspace (a size at least as large as the longest
 *                           context gives a single pass with no merge);
 *   partition_blocks <= -1  each sequence's visible blocks split evenly into
 *                           -partition_blocks partitions (at most 16, fewer when
 *                           the sequence has fewer blocks), merged in the launch
 *                           by a thread-block cluster (falls back to the
 *                           workspace merge if the device cannot hold it);
 *   0                       the automatic choice of pa_decode.
 */
pa_status pa_decode_partitioned(const pa_cache *cache, void *out, const void *q,
                                pa_dtype q_dtype, int num_seqs, int num_q_heads,
                                const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, float sm_scale, int window,
                                int partition_blocks, void *workspace,
                                size_t workspace_bytes, int32_t *err_flag, void *stream);

/*
 * pa_decode_append -- one decode step in one launch: each sequence's new token
 * is written at its position context_lens[b] - 1, the slot its block table
 * names there, and then the batch attends as pa_decode ("PyTorch LLM Serving
 * Engine", "Loading": the new K/V goes to its physical slot and the query
 * attends to the whole context, itself included).  The same results, bit for
 * bit, as pa_write_kv of those slots followed by pa_decode.
 *
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim] of kv_dtype: a 16-bit cache
 *                 takes its own type (copied); an int8 cache quantises them as
 *                 pa_write_kv does.  kv_dtype must equal q_dtype.
 *   the rest      as pa_decode (its automatic partitioning and workspace size)
 *
 * The warp that copies the block holding position context_lens[b] - 1 writes
 * the row first.  A sequence with context_lens[b] = 0 writes nothing; one whose
 * block id at that position is outside the pool writes nothing and sets
 * PA_FLAG_BLOCK_ID, as the attention does.  A step whose new tokens go
 * elsewhere than position context_lens[b] - 1 needs pa_write_kv + pa_decode.
 * Errors: pa_decode's, plus PA_ERR_INVALID_ARG for a NULL or misaligned k_new or
 * v_new and PA_ERR_UNSUPPORTED for kv_dtype != q_dtype.
 */
pa_status pa_decode_append(const pa_cache *cache, const void *k_new, const void *v_new,
                           pa_dtype kv_dtype, void *out, const void *q, pa_dtype q_dtype,
                           int num_seqs, int num_q_heads, const int32_t *block_tables,
                           int max_blocks_per_seq, const int32_t *context_lens, float sm_scale,
                           int window, void *workspace, size_t workspace_bytes,
                           int32_t *err_flag, void *stream);

/*
 * Workspace bytes pa_decode / pa_decode_partitioned need for these arguments
 * (partition_blocks as for pa_decode_partitioned; 0 = the automatic choice,
 * evaluated on the current device).  Returns 0 when no workspace is needed (a
 * single pass, or a merge inside the launch), (size_t)-1 on bad arguments.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                 int head_dim, int max_blocks_per_seq, int window,
                                 int partition_blocks);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for code that is
 * handed only its input and output buffers, such as a plugin inside a host
 * engine that owns all allocation, or a serving loop that must never call
 * cudaMalloc/cudaFree because those calls can synchronise the whole device.
 *
 * Same arguments and result as pa_decode, without workspace: when the batch
 * takes pa_decode's workspace merge (very few (sequence, kv head) pairs), the
 * split-K partials live in a scratch array of PA_NOALLOC_SCRATCH_BYTES compiled
 * into the library, which every device that loads the library holds until the
 * process exits; other batches need no scratch.  The call allocates nothing.
 *   - Returns PA_ERR_UNSUPPORTED, launching nothing, when this batch's partials
 *     would exceed PA_NOALLOC_SCRATCH_BYTES (pa_decode_workspace_bytes with
 *     partition_blocks = 0 gives the size); use pa_decode for such batches.
 *   - The first call on each device looks up the scratch's device address with
 *     that device current; make that first call before any stream capture.  A
 *     device reset (cudaDeviceReset) ends the context that address belongs to:
 *     the next call on that device sees a new context and looks the address up
 *     again, so after a reset, too, call once before capturing.
 *   - All calls on a device share the one scratch array and it keeps the last
 *     call's contents (nothing in it needs to start at zero).  Calls that can
 *     run at the same time on the GPU -- on different streams, or from host
 *     threads with no ordering between them -- race on it: serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
pa_status pa_decode_noalloc(const pa_cache *cache, void *out, const void *q, pa_dtype q_dtype,
                            int num_seqs, int num_q_heads, const int32_t *block_tables,
                            int max_blocks_per_seq, const int32_t *context_lens, float sm_scale,
                            int window, int32_t *err_flag, void *stream);

/*
 * pa_prefill_chunk -- chunked prefill: each sequence's chunk of queries attends
 * to the sequence's paged context before the chunk and causally to the chunk
 * itself ("PyTorch LLM Serving Engine", "What is implemented": chunked prefill
 * sharing the step budget with decode).  Decode is the chunk length 1.
 *
 *   q, out        [num_q_tokens][num_q_heads][head_dim]; sequence n owns rows
 *                 cu_q_lens[n] .. cu_q_lens[n+1]-1
 *   cu_q_lens     [num_seqs + 1] int32, cu_q_lens[0] = 0, non-decreasing,
 *                 cu_q_lens[num_seqs] = num_q_tokens
 *   max_q_len     upper bound of every chunk length (sizes the launch)
 *   context_lens  tokens after the write, chunk included: query c of a chunk of C
 *                 sits at position context_lens[n] - C + c
 *   workspace     unused (may be NULL); kept for a uniform signature
 */
pa_status pa_prefill_chunk(const pa_cache *cache, void *out, const void *q, pa_dtype q_dtype,
                           int num_q_tokens, int num_seqs, int num_q_heads,
                           const int32_t *cu_q_lens, int max_q_len,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, float sm_scale, int window,
                           void *workspace, size_t workspace_bytes, int32_t *err_flag,
                           void *stream);

/* Human-readable name of a status. */
const char *pa_status_str(pa_status status);

/* Text of the CUDA runtime error behind the most recent PA_ERR_CUDA returned to
 * the calling thread ("no CUDA error" if there was none).  The string is static:
 * the caller does not free it.  No counterpart in the pages; a diagnostic of the
 * library's own. */
const char *pa_last_cuda_error(void);

/* PA_OK when flags == 0, else PA_ERR_DEVICE_DATA (flags read back by the caller). */
pa_status pa_check_flags(int32_t flags);

/*
 * pa_selftest_bounded_wait -- checks, on the current device, the bounded wait that
 * every in-kernel wait of this library uses (the pages have no counterpart; the
 * library's own failure handling: a wait that runs out reports PA_FLAG_TIMEOUT
 * and the kernel returns instead of hanging).  One small kernel waits, limited to
 * limit_cycles SM clock cycles (1 .. 4e9), on a barrier that nothing completes,
 * once from one thread and once as a whole warp's vote, with no copy in flight;
 * and once on a barrier that has completed.
 *   result    device int64[4]: [0] 1 if the one-thread wait gave up, [1] 1 if the
 *             warp's wait gave up, [2] 1 if the completed barrier's wait returned
 *             at once, [3] SM cycles the one-thread wait took
 *   err_flag  receives PA_FLAG_TIMEOUT from each wait that gave up
 */
pa_status pa_selftest_bounded_wait(long long limit_cycles, long long *result,
                                   int32_t *err_flag, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
