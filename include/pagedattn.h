/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged decode-attention library.
 *
 * One decode step of attention over a block-paged KV cache:
 *
 *   paged_kv_append                 write the step's new K/V row of every
 *                                   (sequence, kv head) into the pool slot
 *                                   that block_table assigns
 *   paged_attention_decode          attention of each query head over the
 *                                   sequence's valid tokens, reading K/V
 *                                   through block_table
 *   paged_attention_decode_append   both in one launch (the usual step)
 *   paged_attention_decode_partial  the same over fixed token partitions,
 *   paged_attention_decode_reduce   then a log-sum-exp merge (split-KV, for
 *                                   long contexts or few sequences)
 *   paged_attention_decode_split_static  the pair with library-owned scratch
 *   paged_attention_decode_shared_prefix split-KV that reads blocks shared
 *                                   by a group of sequences once per group
 *   paged_attention_decode_balanced the same step on a persistent grid with
 *                                   equal work per warp (mixed lengths)
 *   paged_attention_decode_window   attention over the last W tokens only
 *   paged_kv_append_tokens          the prompt write (several tokens per
 *                                   sequence, valid rows only)
 *   paged_kv_append_int8,           the same write and attention over an
 *   paged_attention_decode_int8     int8 cache with per-block scales
 *   paged_kv_append_fp8,            ... over an fp8 (E4M3) cache with
 *   paged_attention_decode_fp8      per-block scales
 *   paged_attention_decode_shared_prefix_int8, _fp8  the shared-prefix
 *                                   split-KV over those two caches
 *   *_workspace, pa_status_string   sizes of caller workspaces, messages
 *
 * Sources (web pages on paged KV caches), cited by title and section:
 *   "KV Cache and BlockManager" (dpshk.com/news/5906718)            [BM]
 *   vLLM memory-management course, ch. 3 "KV Block design"           [KB]
 *   "A strange KV Cache bug" (dpshk.com/news/5937191)                [BUG]
 *   "KV Cache paging in LLM inference" (intelliparadigm.com)         [PG]
 *
 * ---------------------------------------------------------------------------
 * Memory layout (all tensors row-major, element type `dtype`)
 * ---------------------------------------------------------------------------
 *   q, out            [batch][num_heads][head_dim]
 *   k_new, v_new      [batch][num_kv_heads][head_dim]
 *   block_table       int32 [batch][max_blocks_per_seq]; entry j of row b is
 *                     the physical block holding logical block j (tokens
 *                     j*block_size .. j*block_size+block_size-1) of sequence
 *                     b ([BM] s2, [KB] s3.3).  Entries at or past
 *                     ceil(len/block_size) are never read and may be -1, the
 *                     "unallocated" marker of [BM] s5.1.
 *   seq_lens          int32 [batch]: VALID token count of each sequence,
 *                     never the allocated or padded length ([BUG] s2.4).
 *   k_pool, v_pool    element (blk, kv_head, slot, d) of a pool is at
 *                       blk*block_stride + kv_head*block_size*head_dim
 *                         + slot*head_dim + d
 *                     The [num_blocks][2][num_kv_heads][block_size][head_dim]
 *                     cache of [BM] s5.1 (one layer, K and V co-located per
 *                     block as [KB] s3.2 recommends) is passed as
 *                       k_pool = base, v_pool = base + num_kv_heads*block_size*head_dim,
 *                       block_stride = 2*num_kv_heads*block_size*head_dim;
 *                     separate K and V pools use block_stride =
 *                     num_kv_heads*block_size*head_dim.  Each (block, kv
 *                     head) K or V chunk is block_size*head_dim contiguous
 *                     elements.
 *   alignment         The pool pointers, q, out, k_new and v_new must be
 *                     16-byte aligned and block_stride*element_size a multiple
 *                     of 16 bytes: the kernels move rows with 16-byte vector
 *                     and bulk (TMA) copies, which fault on anything less, so
 *                     the host checks reject it with PA_ERR_MISALIGNED.
 *                     Block starts SHOULD be 128-byte aligned ([KB] s3.7: a
 *                     block start off the 128-byte boundary costs bandwidth):
 *                     a pool base on a 128-byte boundary with block_stride and
 *                     the K-to-V offset multiples of 128 bytes keeps every
 *                     block and every (block, kv head) chunk on one.  This is
 *                     a performance expectation, not checked: a pool that is
 *                     16- but not 128-byte aligned gives the same results.
 *
 * Query head h reads kv head h / (num_heads / num_kv_heads) (grouped-query
 * attention; num_heads must be a multiple of num_kv_heads).
 *
 * ---------------------------------------------------------------------------
 * Conventions shared by every entry point
 * ---------------------------------------------------------------------------
 * Ownership   Every data pointer is DEVICE memory owned by the caller.  The
 *             library never allocates or frees memory at run time; the only
 *             device memory it owns is the fixed scratch array of
 *             paged_attention_decode_split_static.
 * Streams     Work is enqueued on `stream` (NULL = legacy default stream) and
 *             runs asynchronously; nothing synchronises the host.  The block
 *             table never round-trips to the host ([BM] s2).
 * Host checks Arguments are validated before anything is enqueued; a failure
 *             returns a PA_ERR_* status synchronously and launches nothing.
 * Device checks
 *             A sequence whose length is negative or exceeds
 *             max_blocks_per_seq*block_size, or whose first
 *             ceil(len/block_size) table entries include one outside
 *             [0, num_blocks), is not read: its output rows are written as
 *             zeros and the matching PA_DEVERR_* bit is OR-ed into *err_word
 *             (when err_word is not NULL).  Kernels never trap; every
 *             device-side wait is bounded and reports PA_DEVERR_TIMEOUT.
 *             This is the "graceful" handling [BM] s4.1 asks for instead of
 *             a silent out-of-range access.
 * Sharing     Several table rows may name the same physical block (prefix
 *             sharing with reference counts, [KB] s3.4); reads from shared
 *             blocks are fine, appends into a shared block are a caller
 *             error (copy on write is the caller's job).
 * Numerics    Scores, softmax and accumulation run in fp32; out is rounded
 *             to `dtype` (round to nearest even).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA
 * include. */
typedef struct CUstream_st *pa_stream_t;

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, inconsistent shape    */
    PA_ERR_UNSUPPORTED = 2,  /* head_dim / dtype combination not compiled in  */
    PA_ERR_MISALIGNED = 3,   /* a pointer or stride breaks the 16-byte rule   */
    PA_ERR_WORKSPACE = 4,    /* split-KV workspace smaller than required      */
    PA_ERR_CUDA = 5          /* the CUDA runtime reported an error at launch  */
} pa_status;

typedef enum pa_dtype {
    PA_F32 = 0,
    PA_F16 = 1,
    PA_BF16 = 2
} pa_dtype;

/* Bits OR-ed into *err_word by the kernels. */
#define PA_DEVERR_BAD_LEN   1  /* seq_len < 0 or > max_blocks_per_seq*block_size */
#define PA_DEVERR_BAD_BLOCK 2  /* a needed table entry is outside [0, num_blocks) */
#define PA_DEVERR_BAD_POS   4  /* append position outside the table row         */
#define PA_DEVERR_TIMEOUT   8  /* a bounded wait for a copy gave up              */
#define PA_DEVERR_BAD_PREFIX 16 /* a declared shared prefix is not shared/held   */

typedef struct pa_shape {
    int32_t batch;              /* sequences B (0 is allowed: nothing to do) */
    int32_t num_heads;          /* query heads H                             */
    int32_t num_kv_heads;       /* kv heads Hkv, H % Hkv == 0                */
    int32_t head_dim;           /* D                                         */
    int32_t block_size;         /* tokens per block                          */
    int32_t max_blocks_per_seq; /* row length MB of block_table              */
    int64_t num_blocks;         /* physical blocks NB in the pool            */
    int64_t block_stride;       /* elements from block j to block j+1        */
    int32_t dtype;              /* pa_dtype of q, out, k/v_new and the pools */
} pa_shape;

/* Supported shapes: head_dim*element_size in {64, 128, 256, 512} bytes
 * (f16/bf16: D = 32, 64, 128, 256; f32: D = 16, 32, 64, 128) and
 * head_dim*element_size a multiple of 16 for the append. */

/* Human-readable name of a status. Never NULL.  (Library housekeeping: no
 * counterpart on the pages.) */
const char *pa_status_string(pa_status status);

/* Library ABI version (major*10000 + minor*100 + patch).  (Library
 * housekeeping: no counterpart on the pages.) */
int32_t pa_version(void);

/*
 * paged_kv_append -- the reshape-and-cache write path.
 *
 * For every sequence b and kv head h, with pos = positions[b] (the valid
 * length before this step), copy k_new[b][h][:] and v_new[b][h][:] into
 * slot pos % block_size of physical block block_table[b][pos / block_size]:
 * tokens keep their logical order inside a block ([BM] s4.4) and the cache
 * grows exactly like the contiguous append of [BUG] s4.1.  The copy is
 * bit-exact.  A sequence with pos outside [0, max_blocks_per_seq*block_size)
 * is skipped with PA_DEVERR_BAD_POS; one whose target entry is outside
 * [0, num_blocks) is skipped with PA_DEVERR_BAD_BLOCK.  positions is not
 * modified (the caller advances seq_lens).
 *
 * k_new, v_new: device [B][Hkv][D]; k_pool, v_pool: device pools (layout
 * above); block_table: device int32 [B][MB]; positions: device int32 [B];
 * err_word: device int32 or NULL.
 */
pa_status paged_kv_append(const pa_shape *shape, const void *k_new, const void *v_new,
                          void *k_pool, void *v_pool, const int32_t *block_table,
                          const int32_t *positions, int32_t *err_word, pa_stream_t stream);

/*
 * paged_attention_decode -- one decode token per sequence.
 *
 * out[b][h][:] = sum_t w_t V[t][:] / sum_t w_t,  w_t = exp(x_t - max x),
 * x_t = scale * <q[b][h][:], K[t][:]>, over t in [0, seq_lens[b]) only, where
 * K[t], V[t] are row t of kv head h/(H/Hkv) found through block_table ([BM]
 * s5.2: the translation happens inside the kernel).  seq_lens[b] == 0 gives
 * out = 0.  The computation is the per-block decomposition of [PG] s2.2:
 * scores per block, running softmax statistics, weighted sum of V blocks.
 *
 * Grouped-query shapes with 16-bit types, D in {64, 128}, and block_size a
 * multiple of 16 (or 8) run on the tensor cores; everything else on the
 * SIMT path.  paged_attention_decode_path() tells which.
 *
 * out, q: device [B][H][D]; pools, block_table as above; seq_lens: device
 * int32 [B]; scale: usually 1/sqrt(D); err_word: device int32 or NULL.
 */
pa_status paged_attention_decode(const pa_shape *shape, void *out, const void *q,
                                 const void *k_pool, const void *v_pool,
                                 const int32_t *block_table, const int32_t *seq_lens,
                                 float scale, int32_t *err_word, pa_stream_t stream);

/*
 * paged_attention_decode_append -- paged_kv_append followed by
 * paged_attention_decode with seq_lens = positions + 1, in one launch.
 *
 * For every sequence b, k_new[b][h][:] and v_new[b][h][:] are written to slot
 * positions[b] % block_size of block block_table[b][positions[b] / block_size]
 * exactly as paged_kv_append writes them, and out[b][:][:] is the attention
 * of q over the positions[b] + 1 tokens that then hold the sequence ([BM]
 * s4.4 and [BUG] s4.1 for the append, [PG] s2.2 for the attention).  The
 * appended token is taken from k_new/v_new directly, so the output does not
 * depend on when the pool write lands.  Results equal the two separate calls
 * (same kernels, same arithmetic).  positions[b] outside
 * [0, max_blocks_per_seq*block_size) gives PA_DEVERR_BAD_POS and zeros; a
 * target entry outside [0, num_blocks) gives PA_DEVERR_BAD_BLOCK and zeros.
 * positions is not modified.
 *
 * k_new, v_new: device [B][Hkv][D]; positions: device int32 [B]; the rest as
 * paged_attention_decode.
 */
pa_status paged_attention_decode_append(const pa_shape *shape, void *out, const void *q,
                                        const void *k_new, const void *v_new, void *k_pool,
                                        void *v_pool, const int32_t *block_table,
                                        const int32_t *positions, float scale,
                                        int32_t *err_word, pa_stream_t stream);

/*
 * paged_kv_append_tokens -- the prompt (prefill) write of several tokens per
 * sequence.
 *
 * k_new, v_new are a padded batch [B][max_tokens][Hkv][D]: rows t <
 * counts[b] of sequence b are written to positions positions[b] + t, each
 * through block_table as paged_kv_append places a single token, and rows t >=
 * counts[b] are padding that never enters the cache -- the valid length, not
 * the padded length, defines the cache contents ([BUG] s2.3-2.4, s4.1).
 * counts[b] outside [0, max_tokens] gives PA_DEVERR_BAD_LEN and
 * positions[b] < 0 or positions[b] + counts[b] past the table row gives
 * PA_DEVERR_BAD_POS, both skipping the sequence; a token whose target entry
 * is outside [0, num_blocks) is skipped with PA_DEVERR_BAD_BLOCK.  The copy
 * is bit-exact.  positions and counts are device int32 [B].
 */
pa_status paged_kv_append_tokens(const pa_shape *shape, const void *k_new, const void *v_new,
                                 int32_t max_tokens, void *k_pool, void *v_pool,
                                 const int32_t *block_table, const int32_t *positions,
                                 const int32_t *counts, int32_t *err_word, pa_stream_t stream);

/*
 * paged_attention_decode_window -- decode over a sliding window.
 *
 * As paged_attention_decode, but each query attends only to the last
 * `window` valid tokens [max(0, L - window), L) of its sequence, the
 * sliding-window cache policy of [BUG] s5.3; blocks wholly before the window
 * are not read.  window must be positive; window >= L gives the full
 * attention.
 */
pa_status paged_attention_decode_window(const pa_shape *shape, void *out, const void *q,
                                        const void *k_pool, const void *v_pool,
                                        const int32_t *block_table, const int32_t *seq_lens,
                                        float scale, int32_t window, int32_t *err_word,
                                        pa_stream_t stream);

/* Which kernel family paged_attention_decode and _partial use for `shape`.
 * (An implementation query: no counterpart on the pages, which leave the
 * kernel to the implementation; [PG] s2.2 gives only its arithmetic.) */
typedef enum pa_path {
    PA_PATH_INVALID = 0,     /* shape rejected                                  */
    PA_PATH_SIMT = 1,        /* fp32 CUDA-core path, one (sequence, head) per CTA */
    PA_PATH_TENSOR_GQA = 2   /* tensor-core path, one (sequence, kv head) per CTA */
} pa_path;
pa_path paged_attention_decode_path(const pa_shape *shape);

/* Which kernel a decode of `shape` runs on the CURRENT device: the single
 * pass of paged_attention_decode / _append (window 0) or _window (window >
 * 0) when partition_tokens is 0, else the partial pass of the split-KV pair
 * with that partition size.  The tensor-core family has two kernels: the
 * warp-level one (mma.sync; few long sequences also spread over
 * thread-block clusters) and, at head_dim 128, one on the fifth-generation
 * tensor cores (tcgen05.mma with accumulators in tensor memory, a
 * persistent grid of at most one CTA per SM, or with few units one unit per
 * thread-block cluster of 2, 4 or 8 CTAs); which one runs depends on how
 * many (sequence, kv head) units the launch has against the SM count.
 * Results agree up to rounding order.  Returns PA_KERNEL_INVALID for a
 * rejected shape, window or partition size.  (An implementation query: no
 * counterpart on the pages.) */
typedef enum pa_kernel {
    PA_KERNEL_INVALID = 0,
    PA_KERNEL_SIMT = 1,       /* CUDA cores                                       */
    PA_KERNEL_MMA_SYNC = 2,   /* tensor cores, warp-level mma.sync                 */
    PA_KERNEL_TCGEN05 = 3     /* tensor cores, tcgen05.mma and tensor memory        */
} pa_kernel;
pa_kernel paged_attention_decode_kernel(const pa_shape *shape, int32_t window, int32_t partition_tokens);

/*
 * Split-KV ("flash decoding") pair for long contexts.
 *
 * [PG] s2.2 computes attention block by block -- scores per block, then the
 * per-block results aggregated before the softmax is normalised and the V
 * blocks summed with their weights.  This pair makes that aggregation
 * explicit across thread blocks: each partition of blocks keeps its own
 * running softmax state, and the reduce combines the states.  The pages do
 * not spell out how partial states combine; the merge below is the
 * log-sum-exp identity (rescale each partition's sum and weighted V by
 * 2^(m_p - M) for the overall maximum M), which makes the result equal to
 * the single-pass attention.
 *
 * paged_attention_decode_partial splits each sequence's valid tokens into
 * partitions of partition_tokens tokens (a positive multiple of 16) and,
 * for every (b, h, partition p) that holds at least one valid token,
 * writes into the workspace
 *   m[b][h][p]      = max over the partition of x_t * log2(e)
 *   l[b][h][p]      = sum over the partition of 2^(x_t*log2(e) - m)
 *   acc[b][h][p][:] = sum over the partition of 2^(x_t*log2(e) - m) V[t][:]
 * in fp32 (x_t as in paged_attention_decode).  paged_attention_decode_reduce
 * then merges the ceil(seq_lens[b]/partition_tokens) partitions of each
 * (b, h):
 *   M = max_p m_p,  out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,
 * which equals paged_attention_decode up to rounding.  Both calls must get the
 * same shape, seq_lens and partition_tokens, on the same stream (or be
 * ordered by the caller).
 *
 * Workspace: device memory of at least paged_attention_partial_workspace()
 * bytes, 16-byte aligned, owned by the caller, holding, with
 * P = ceil(max_blocks_per_seq*block_size / partition_tokens):
 *   float m[B][H][P]; float l[B][H][P]; float acc[B][H][P][D]
 * at byte offsets 0, 4*B*H*P and 8*B*H*P rounded up to 16.  Only the slots
 * of partitions that hold valid tokens are written; the reduce reads only
 * those.  A partition that met a bad table entry stores l = -1, and the
 * reduce then writes zeros for the whole sequence.
 *
 * paged_attention_partial_workspace returns 0 for an invalid shape or
 * partition size.  (A size query for the workspace above: [PG] s2.2's
 * per-block results, one slot per partition.)
 */
size_t paged_attention_partial_workspace(const pa_shape *shape, int32_t partition_tokens);

pa_status paged_attention_decode_partial(const pa_shape *shape, const void *q,
                                         const void *k_pool, const void *v_pool,
                                         const int32_t *block_table, const int32_t *seq_lens,
                                         float scale, int32_t partition_tokens,
                                         void *workspace, size_t workspace_bytes,
                                         int32_t *err_word, pa_stream_t stream);

pa_status paged_attention_decode_reduce(const pa_shape *shape, void *out,
                                        const void *workspace, size_t workspace_bytes,
                                        const int32_t *seq_lens, int32_t partition_tokens,
                                        int32_t *err_word, pa_stream_t stream);

/*
 * paged_attention_decode_shared_prefix -- the split-KV pair for groups of
 * sequences that share a prefix, reading the shared blocks once per group.
 *
 * Sequences forked from one prompt (beam search, parallel sampling) name the
 * same physical blocks for their common prefix ([KB] s3.4: blocks shared by
 * reference count instead of copied).  Group i is the run of sequences
 * [group_first[i], group_first[i+1]) whose table rows agree on the blocks
 * holding their first shared_tokens[i] tokens (group_first and
 * shared_tokens are HOST arrays of num_groups + 1 and num_groups entries;
 * group_first ascends strictly, at most 16 groups; a group whose
 * shared_tokens is below partition_tokens shares nothing and may be any
 * size, the others need members x H/Hkv <= 16).
 * For each group and kv head, the partitions of partition_tokens tokens that
 * lie wholly inside the shared prefix are read once and attended by every
 * member's queries at once (tensor cores; the members are the MMA columns);
 * in the same launch all other partitions are computed per sequence, and
 * the log-sum-exp reduce merges them.  The result is paged_attention_decode's, up to rounding
 * order; it equals the partial + reduce pair's output formula.
 *
 * Device checks: as paged_attention_decode; in addition, a member whose
 * table differs from the group's first member inside a shared partition, or
 * whose length does not cover it, gets zeros and PA_DEVERR_BAD_PREFIX.
 * Workspace: exactly that of the partial/reduce pair
 * (paged_attention_partial_workspace).  Shapes: those of the tensor-core
 * path (paged_attention_decode_path() == PA_PATH_TENSOR_GQA, or the same
 * conditions with num_heads == num_kv_heads) with num_heads/num_kv_heads
 * <= 16; others give PA_ERR_UNSUPPORTED.  Two launches on `stream`.
 */
pa_status paged_attention_decode_shared_prefix(const pa_shape *shape, void *out, const void *q,
                                               const void *k_pool, const void *v_pool,
                                               const int32_t *block_table,
                                               const int32_t *seq_lens, int32_t num_groups,
                                               const int32_t *group_first,
                                               const int32_t *shared_tokens, float scale,
                                               int32_t partition_tokens, void *workspace,
                                               size_t workspace_bytes, int32_t *err_word,
                                               pa_stream_t stream);

/*
 * paged_attention_decode_balanced -- one decode step under a load-balanced,
 * persistent schedule.
 *
 * Computes exactly what the single-pass entry points compute, selected by
 * the arguments:
 *   seq_lens != NULL, positions == NULL   paged_attention_decode (window 0)
 *                                         or paged_attention_decode_window
 *   positions != NULL, seq_lens == NULL   paged_attention_decode_append
 *                                         (k_new, v_new required), over the
 *                                         last `window` tokens when window > 0
 * with the same device checks, zeros and PA_DEVERR_* bits.  k_pool and
 * v_pool are written only in the append mode.
 *
 * The attention is the per-block decomposition of [PG] s2.2; what differs is
 * the schedule, which the sources leave to the implementation: the grid is
 * sized to the GPU (a few CTAs per SM), and the tiles of all
 * (sequence, head) items, laid end to end, are cut into one equal slice per
 * warp, so a batch mixing short and long sequences ([BUG] s2 serves such
 * batches) keeps every SM streaming until the end.  An item cut between
 * warps is finished by the last of them to arrive, which merges their
 * partial softmax states (the log-sum-exp merge of the split-KV pair).
 * Results differ from paged_attention_decode only by fp32 rounding order,
 * and are reproducible run to run for the same inputs and device.
 *
 * Workspace: device memory of at least paged_attention_balanced_workspace()
 * bytes, 16-byte aligned, owned by the caller.  It must be ZERO-FILLED
 * before its first use (e.g. cudaMemsetAsync); every call leaves the
 * counters in it at zero again, so no call after the first needs a fill --
 * unless a call was aborted before completing (a device error that killed
 * the context), after which the workspace must be zero-filled again.  Calls
 * that may overlap on the GPU need separate workspaces.  The size depends on
 * the shape and on the GPU the call runs on (SM count); query it with the
 * target device current.  Returns 0 for a shape this entry point rejects.
 * (paged_attention_balanced_workspace is a size query with no counterpart
 * on the pages.)
 *
 * Rejected shapes (PA_ERR_UNSUPPORTED): the schedule keeps two int32 per
 * sequence in shared memory and counts tiles in int32, which bounds batch
 * and batch*heads*max_blocks_per_seq*block_size/16.
 */
size_t paged_attention_balanced_workspace(const pa_shape *shape);

pa_status paged_attention_decode_balanced(const pa_shape *shape, void *out, const void *q,
                                          void *k_pool, void *v_pool,
                                          const int32_t *block_table, const int32_t *seq_lens,
                                          const int32_t *positions, const void *k_new,
                                          const void *v_new, float scale, int32_t window,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t *err_word, pa_stream_t stream);

/*
 * int8 KV cache: quantised blocks with per-block scales.
 *
 * The sources name int8-quantised cache blocks ([BM] s6.3, and the
 * "quantized" element size of the block-size rule in [BM] s3) without fixing
 * a scheme.  The scheme of these two calls: a pool element is a code c in
 * [-127, 127] (one byte) that stands for c * s, where s is the fp32 scale of
 * its (physical block, kv head) for K, or for V:
 *     kv_scales[(blk*2 + 0)*num_kv_heads + h]   scale of K in block blk, kv head h
 *     kv_scales[(blk*2 + 1)*num_kv_heads + h]   scale of V
 * (device fp32 [num_blocks][2][num_kv_heads], set by whoever allocates the
 * block; scales must be positive and finite).  The pools keep the layout of
 * the 16-bit pools above with one byte per element (block_stride counts
 * bytes; it and head_dim must keep rows and blocks on 16-byte boundaries).
 * shape->dtype is the element type of q, out, k_new and v_new; head_dim must
 * be 64, 128 or 256.
 *
 * paged_kv_append_int8 writes k_new/v_new [B][Hkv][D] like paged_kv_append,
 * each value x as clamp(round_half_even(x / s), -127, 127) with the quotient
 * taken in IEEE binary32 (NaN -> 0), s the scale of the target block; the
 * codes are exactly those of that rule.
 *
 * paged_attention_decode_int8 is paged_attention_decode over the values the
 * codes stand for ([PG] s2.2): x_t = scale * s_K * <q, c_t>, weights w_t as
 * there, out = sum_t w_t s_V c_t / sum_t w_t.  Same device checks, zeros and
 * PA_DEVERR_* bits.  Grouped-query shapes with 16-bit q and head_dim 64 or
 * 128 run on the tensor cores (codes turned into exact fp16 in registers,
 * queries rounded to fp16); the rest on the CUDA cores.
 */
pa_status paged_kv_append_int8(const pa_shape *shape, const void *k_new, const void *v_new,
                               int8_t *k_pool, int8_t *v_pool, const float *kv_scales,
                               const int32_t *block_table, const int32_t *positions,
                               int32_t *err_word, pa_stream_t stream);

pa_status paged_attention_decode_int8(const pa_shape *shape, void *out, const void *q,
                                      const int8_t *k_pool, const int8_t *v_pool,
                                      const float *kv_scales, const int32_t *block_table,
                                      const int32_t *seq_lens, float scale, int32_t *err_word,
                                      pa_stream_t stream);

/*
 * fp8 KV cache: E4M3 blocks with per-block scales.
 *
 * The second scheme for the quantised blocks the sources name ([BM] s6.3,
 * s3) without fixing one: a pool element is an 8-bit floating-point code in
 * the OCP FP8 E4M3 format (sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 holds the subnormals m * 2^-9; no
 * infinities; 0x7F and 0xFF are NaN; largest finite magnitude 448) standing
 * for value(c) * s, with the scales laid out and owned exactly as for the
 * int8 cache above.  The pools have the same byte layout; shape->dtype is
 * the element type of q, out, k_new and v_new (fp32, fp16 or bf16); head_dim
 * must be 64, 128 or 256 (others: PA_ERR_UNSUPPORTED).
 *
 * paged_kv_append_fp8 writes each value x as the E4M3 code of x / s (the
 * quotient in IEEE binary32) nearest to it, ties to the even code,
 * magnitudes beyond 448 saturating to 448 (a NaN quotient gives the NaN code
 * 0x7F).
 *
 * paged_attention_decode_fp8 is paged_attention_decode over the values the
 * codes stand for ([PG] s2.2): x_t = scale * s_K * <q, value(c_t)>, out =
 * sum_t w_t s_V value(c_t) / sum_t w_t.  Same device checks, zeros and
 * PA_DEVERR_* bits.  Grouped-query shapes at head_dim 64 or 128 run on the
 * tensor cores (codes converted to exact fp16 in registers, queries rounded
 * to fp16); the rest on the CUDA cores in fp32.  Results are held to the
 * 16-bit tolerance whatever q's dtype.  A NaN code inside the attended
 * length makes the outputs it meets NaN.
 */
pa_status paged_kv_append_fp8(const pa_shape *shape, const void *k_new, const void *v_new,
                              uint8_t *k_pool, uint8_t *v_pool, const float *kv_scales,
                              const int32_t *block_table, const int32_t *positions,
                              int32_t *err_word, pa_stream_t stream);

pa_status paged_attention_decode_fp8(const pa_shape *shape, void *out, const void *q,
                                     const uint8_t *k_pool, const uint8_t *v_pool,
                                     const float *kv_scales, const int32_t *block_table,
                                     const int32_t *seq_lens, float scale, int32_t *err_word,
                                     pa_stream_t stream);

/*
 * paged_attention_decode_shared_prefix_int8 / _fp8 -- the shared-prefix
 * split-KV pair of paged_attention_decode_shared_prefix over the int8 or fp8
 * cache above ([KB] s3.4 for the sharing, [PG] s2.2 for the per-block
 * decomposition and its merge).
 *
 * Groups, partitions, workspace (paged_attention_partial_workspace), device
 * checks, PA_DEVERR_BAD_PREFIX and the merge are exactly those of
 * paged_attention_decode_shared_prefix; the per-token arithmetic is that of
 * paged_attention_decode_int8 / _fp8 on their tensor-core kernel (codes
 * turned into exact fp16 in registers, queries rounded to fp16), for every
 * unit, with one query column per (member, query head of the kv head), at
 * most 16.  The result is paged_attention_decode_int8's / _fp8's up to
 * rounding order and held to the same tolerance.  Shapes: head_dim 64 or
 * 128; q of fp16 or bf16 (int8), or fp32, fp16 or bf16 (fp8); any block size
 * (tensor boxes where it is 8 or a multiple of 16, row copies otherwise);
 * num_heads/num_kv_heads <= 16.  Others give PA_ERR_UNSUPPORTED.  Two
 * launches on `stream`.
 */
pa_status paged_attention_decode_shared_prefix_int8(const pa_shape *shape, void *out, const void *q,
                                                    const int8_t *k_pool, const int8_t *v_pool,
                                                    const float *kv_scales, const int32_t *block_table,
                                                    const int32_t *seq_lens, int32_t num_groups,
                                                    const int32_t *group_first,
                                                    const int32_t *shared_tokens, float scale,
                                                    int32_t partition_tokens, void *workspace,
                                                    size_t workspace_bytes, int32_t *err_word,
                                                    pa_stream_t stream);

pa_status paged_attention_decode_shared_prefix_fp8(const pa_shape *shape, void *out, const void *q,
                                                   const uint8_t *k_pool, const uint8_t *v_pool,
                                                   const float *kv_scales, const int32_t *block_table,
                                                   const int32_t *seq_lens, int32_t num_groups,
                                                   const int32_t *group_first,
                                                   const int32_t *shared_tokens, float scale,
                                                   int32_t partition_tokens, void *workspace,
                                                   size_t workspace_bytes, int32_t *err_word,
                                                   pa_stream_t stream);

/*
 * paged_attention_decode_split_static -- the split-KV pair without any
 * caller-provided workspace.
 *
 * The sources have no counterpart for this entry point: it exists for
 * callers that cannot allocate device memory, e.g. code running inside a
 * memory pool or allocator callback, a plugin handed only its input and
 * output buffers by a host framework, or a stream being captured where an
 * allocation would break the capture.  It computes exactly what
 * paged_attention_decode_partial followed by paged_attention_decode_reduce
 * compute, but keeps the partial results in a fixed scratch buffer owned by
 * the library: a file-scope device array of PA_STATIC_SCRATCH_BYTES bytes
 * that every GPU which loads the library holds until the process exits.
 * The caller passes only inputs and outputs (same layouts as
 * paged_attention_decode); the call allocates nothing.
 *
 * Limit: a shape whose split-KV workspace (paged_attention_partial_workspace)
 * exceeds PA_STATIC_SCRATCH_BYTES is rejected with PA_ERR_WORKSPACE before
 * anything is enqueued; use the partial/reduce pair with your own workspace
 * for such shapes.
 *
 * Set-up: the first call on each device looks up the device address of the
 * scratch array (with that device current) and caches it together with the
 * identity of the CUDA context that was current; make that first call before
 * any stream capture.  The address belongs to that context: when a later call
 * finds another context current on the device (after cudaDeviceReset, or a
 * context the caller created), it looks the address up again in the new
 * context before launching, so a reset never leaves a stale address behind.
 * A call that has to look the address up is not capturable, so after a
 * reset make one call again before capturing.
 *
 * Sharing: all calls on a device use the same scratch array, and it keeps
 * whatever the previous call left in it.  Nothing in it needs to start at
 * zero: the partial pass writes every slot the reduce pass reads.  Calls
 * that can overlap on the GPU (different streams without ordering, or
 * several host threads) race on the array; order them on one stream or
 * with events.
 */
#define PA_STATIC_SCRATCH_BYTES (8u << 20)
pa_status paged_attention_decode_split_static(const pa_shape *shape, void *out, const void *q,
                                              const void *k_pool, const void *v_pool,
                                              const int32_t *block_table,
                                              const int32_t *seq_lens, float scale,
                                              int32_t partition_tokens, int32_t *err_word,
                                              pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
