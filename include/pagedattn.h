/*
 * pagedattn.h: C ABI of the GB300 (sm_103a) paged KV-cache decode attention
 * library, libpagedattn.so.
 *
 * The operations follow the paging scheme described for vLLM's PagedAttention
 * (web page "vllm-project-vllm" review, §3 Q2, §6 "KV Cache Block Tables",
 * §7): keys and values live in a pool of fixed-size physical blocks; each
 * sequence owns a block table mapping its logical block j to a physical block
 * id, so its blocks need not be contiguous and may be shared by several
 * sequences (prefix / copy-on-write sharing); every decode step appends one
 * token per sequence and attends one query token per sequence over the whole
 * cached context, which makes the step memory-bandwidth bound.
 *
 * Conventions shared by every call
 *  - All array arguments are DEVICE pointers to contiguous row-major data
 *    owned by the caller.  The library never allocates, frees or copies
 *    caller memory, never synchronises the stream (except in check mode, see
 *    pa_set_check_mode) and enqueues its kernels on `stream`.
 *  - Caches: k_cache and v_cache are [num_blocks, num_kv_heads, block_size,
 *    head_dim] of the cache dtype, described by one pa_cache_desc.  Both must
 *    start on a 16-byte boundary.
 *  - Token i of sequence s is in physical block block_tables[s][i / block_size]
 *    at offset i % block_size.  Query head g reads kv head g / G with
 *    G = num_q_heads / num_kv_heads (contiguous grouping).
 *  - context_lens[s] counts every cached token of sequence s including the one
 *    written this step; entries of block_tables past ceil(context_lens[s] /
 *    block_size) are never read.  A context length of 0 gives a zero output.
 *  - FP8 caches use OCP E4M3 with one per-tensor scale: stored =
 *    e4m3_rne_satfinite(x / kv_scale), read back as stored * kv_scale.  For
 *    16-bit caches kv_scale must be 1.
 *  - Supported: head_dim 64 or 128; block_size 8, 16 or 32; G from 1 to 128;
 *    q/out dtype f16 or bf16; cache dtype equal to the q dtype or FP8 E4M3.
 *  - Two kernels serve the decode calls.  When the G query heads of a kv head
 *    times the new tokens per sequence make at most 16 query columns, a
 *    warp-MMA kernel streams each (sequence, kv head) once per CTA.  Wider
 *    groups go to the tensor-core kernel of pa_prefill (query rows packed as
 *    token x head, tcgen05 MMAs with TMEM accumulators), which needs
 *    scale > 0.
 *  - Errors are return codes (pa_status); nothing is thrown across the ABI.
 *    Arguments are checked on the host before anything is launched; a failed
 *    check launches nothing.  Index values in device arrays are not read by
 *    the host.  The kernels never access memory outside the arrays for any
 *    index values: a block id outside the pool reads zeros, a context length
 *    above max_blocks_per_seq * block_size is clamped, a slot outside the pool
 *    is skipped; each such event is recorded in a device error word that
 *    pa_get_device_error() returns, and that check mode turns into
 *    PA_ERR_BAD_INDEX.
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *pa_stream_t;

typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer          */
    PA_ERR_UNSUPPORTED = -2, /* valid but not built: head_dim, block_size, G, dtype  */
    PA_ERR_WORKSPACE = -3,   /* split workspace missing or too small                 */
    PA_ERR_CUDA = -4,        /* a CUDA runtime/driver call or launch failed          */
    PA_ERR_BAD_INDEX = -5,   /* check mode: a kernel saw an out-of-range index       */
    PA_ERR_TIMEOUT = -6,     /* a kernel gave up waiting on its own copy pipeline    */
    PA_ERR_OUT_OF_BLOCKS = -7, /* block manager: not enough free blocks (nothing changed) */
    PA_ERR_NOT_FOUND = -8    /* block manager: unknown sequence id, or id already used */
} pa_status;

/* Device error word bits (pa_get_device_error). */
#define PA_DEVERR_BLOCK_ID 0x1    /* block id outside [0, num_blocks)                 */
#define PA_DEVERR_CONTEXT_LEN 0x2 /* context length < 0 or above the table/partitions */
#define PA_DEVERR_SLOT 0x4        /* slot id outside [0, num_blocks * block_size)     */
#define PA_DEVERR_TIMEOUT 0x8     /* a pipeline wait ran out (about one second)       */
#define PA_DEVERR_LAYOUT 0x10     /* a kernel found its shared memory misaligned and did nothing */

typedef struct {
    int64_t num_blocks;   /* physical blocks in the pool (NB)                 */
    int32_t block_size;   /* tokens per block (8, 16 or 32)                   */
    int32_t num_kv_heads; /* Hkv                                              */
    int32_t head_dim;     /* D (64 or 128)                                    */
    int32_t kv_dtype;     /* pa_dtype of both caches                          */
} pa_cache_desc;

/*
 * pa_reshape_and_cache: writes this step's new K and V rows into the cache
 * slots named by slot_mapping (blocks are extended each decode step, review
 * §6 "KV Cache Block Tables").
 *   key, value    [num_tokens, num_kv_heads, head_dim] of in_dtype (f16/bf16),
 *                 16-byte aligned
 *   slot_mapping  int64 [num_tokens]; slot = block * block_size + offset;
 *                 a negative slot skips the token (padding)
 *   k_cache/v_cache, cache   the pool (cache->kv_dtype == in_dtype, or FP8 E4M3)
 *   kv_scale      FP8 per-tensor scale (> 0); must be 1 for 16-bit caches
 * 16-bit caches receive a bit-exact copy.  FP8 caches receive
 * e4m3_rne_satfinite(float(x) / kv_scale) with an IEEE float32 division.
 * Two tokens naming the same slot in one call leave either row there.
 */
PA_API int pa_reshape_and_cache(const void *key, const void *value, int32_t in_dtype, int32_t num_tokens,
                         void *k_cache, void *v_cache, const pa_cache_desc *cache,
                         const int64_t *slot_mapping, float kv_scale, pa_stream_t stream);

/*
 * pa_decode: one query token per sequence attends over its whole paged
 * context (review §7: decode reads the full KV cache per layer):
 *   out[s][g] = sum_i softmax_i(scale * q[s][g] . k_i) v_i,  i < context_lens[s]
 *   out           [num_seqs, num_q_heads, head_dim] of q_dtype (written)
 *   q             [num_seqs, num_q_heads, head_dim] of q_dtype; q and out 16-byte aligned
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]
 *   context_lens  int32 [num_seqs]
 *   scale         softmax scale (typically 1/sqrt(head_dim)); kv_scale as above
 * One CTA per (sequence, kv head) streams that sequence's K/V blocks once and
 * serves all G query heads that share them.
 */
PA_API int pa_decode(void *out, const void *q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
              const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
              const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
              float scale, float kv_scale, pa_stream_t stream);

/*
 * pa_decode_multi: decode of num_q_tokens (k) new tokens per sequence at once,
 * as when a target model verifies k draft tokens in one pass (speculative
 * decoding: web page "vLLM", speculative decoding paragraph; review §10).
 * New token j of sequence s sits at position context_lens[s] - k + j (all k
 * were written to the cache, e.g. by pa_reshape_and_cache with k slots per
 * sequence) and attends causally to positions 0 .. context_lens[s] - k + j:
 *   out[s][j][g] = sum_{i <= L-k+j} softmax_i(scale * q[s][j][g] . k_i) v_i
 *   out, q   [num_seqs, num_q_tokens, num_q_heads, head_dim] of q_dtype
 * A token whose position is negative (k > L) gets a zero output.  The k
 * tokens of all G query heads of a kv head share each K/V tile loaded: as
 * G * k columns of the warp-MMA kernel when G * k <= 16, as G * k rows of
 * the tensor-core kernel otherwise (then scale > 0).  Other arguments as
 * pa_decode.
 */
PA_API int pa_decode_multi(void *out, const void *q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_tokens,
                           int32_t num_q_heads, const void *k_cache, const void *v_cache,
                           const pa_cache_desc *cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, float scale, float kv_scale, pa_stream_t stream);

/*
 * pa_prefill: the same causal attention as pa_decode_multi for a chunk of C =
 * num_q_tokens new tokens per sequence (positions L - C .. L - 1 of each
 * context; chunked prefill, review §10 table), computed on the tensor cores
 * with tcgen05 MMAs and tensor-memory accumulators: prefill is the
 * compute-bound phase (review §7).  For an even group size G a work item
 * is (sequence, two query heads of one kv head, 128 new tokens): the two
 * query tiles share each K/V tile loaded; for an odd G with head_dim 128 it
 * is (sequence, query head, 128 new tokens).  With E4M3 caches and a
 * workspace (at least pa_prefill_workspace_size bytes, 16-byte aligned, owned
 * by the caller) those calls first widen the batch's blocks exactly to the q
 * dtype (every E4M3 value is a bf16 and an f16 value) into the workspace, a
 * compact pool with its own block table, and kv_scale then multiplies the
 * scores and the output.  The other calls (an odd G with head_dim 64, or
 * E4M3 caches without a workspace) pack the queries of a (sequence, kv head)
 * as rows token * G + head, floor(128 / G) tokens x G heads per 128-row tile,
 * so every K/V tile loaded serves all G heads (the kernel of the wide-group
 * decode calls); there E4M3 tiles are widened to f16 in shared memory and the
 * MMAs run in f16, bf16 q scaled per query row by a power of two 2^e (max|q|
 * 2^e in [2^14, 2^15)) and rounded to f16, exact but for entries below 2^-29
 * of the row's largest.  All kernels are persistent, one CTA per SM walking
 * the items, and stream each item's 128-token K/V tiles through the block
 * table.
 *   out, q   [num_seqs, num_q_tokens, num_q_heads, head_dim] of q_dtype
 *   workspace  device scratch for E4M3 caches, or NULL (ignored for 16-bit
 *              caches); PA_ERR_WORKSPACE if non-NULL and smaller than
 *              pa_prefill_workspace_size or not 16-byte aligned.  Its
 *              contents are not kept between calls.
 * Supported: head_dim 64 or 128, caches of the q dtype or FP8 E4M3, block
 * size 8, 16 or 32, G up to 128, scale > 0.  Other arguments as pa_decode
 * (kv_scale must be 1 for 16-bit caches).
 */
PA_API int pa_prefill(void *out, const void *q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_tokens,
                      int32_t num_q_heads, const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
                      const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                      float scale, float kv_scale, void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Workspace bytes pa_prefill uses with E4M3 caches: 4 * num_kv_heads *
 * block_size * head_dim + 4 per entry of the [num_seqs, max_blocks_per_seq]
 * block tables (the widened K and V blocks and a compact table).  Returns 0
 * for 16-bit caches and for invalid sizes.
 */
PA_API size_t pa_prefill_workspace_size(int32_t num_seqs, int32_t max_blocks_per_seq, const pa_cache_desc *cache);

/*
 * Workspace bytes pa_decode_split needs: num_seqs * num_q_heads *
 * ceil(max_context_len / partition_size) * (head_dim + 2) * 4 (one fp32
 * partial output row plus its (m, l) per partition of each query head; the
 * partition and merge scheme is described at pa_decode_split).  Returns 0 for
 * invalid sizes.
 */
PA_API size_t pa_decode_split_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                      int32_t max_context_len, int32_t partition_size);

/*
 * pa_decode_split: the same result as pa_decode, computed per partition of
 * partition_size tokens (a multiple of 64).  The review's implementation
 * cross-reference (§15, "Paged Attention Kernels": paged attention v1/v2)
 * names a second paged-attention kernel beside the single-pass one without
 * describing it; the pages give no partitioning or merge rule, so the
 * partitions, their partial softmax states and the log-sum-exp merge below
 * are this library's reading of that split-context kernel, chosen so that
 * long contexts spread over many CTAs (decode is bandwidth bound, review
 * §7).  A CTA streams a run of
 * consecutive partitions of one (sequence, kv head), folds their partials
 * (o_p, m_p, l_p) by log-sum-exp in partition order and writes one
 * unnormalised partial per run to the workspace; a second kernel merges the
 * runs the same way:  M = max_p m_p,  L = sum_p l_p 2^(m_p - M),
 * out = sum_p o_p 2^(m_p - M) / L  (scores kept in base 2).  Sequences held
 * by a single run are written directly.
 *   max_context_len  >= every context_lens[s] (the host's own bound; longer
 *                    contexts are clamped and flagged)
 *   workspace        device buffer of at least workspace_bytes =
 *                    pa_decode_split_workspace_size(...), 16-byte aligned,
 *                    owned by the caller; its contents need no initialisation
 *                    and are scratch after the call.  Calls that share a
 *                    workspace must be ordered on one stream.
 */
PA_API int pa_decode_split(void *out, const void *q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
                    const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, float scale, float kv_scale,
                    int32_t max_context_len, int32_t partition_size, void *workspace,
                    size_t workspace_bytes, pa_stream_t stream);

/*
 * Workspace bytes pa_decode_multi_split needs: num_seqs * num_q_tokens *
 * num_q_heads * ceil(max_context_len / partition_size) * (head_dim + 2) * 4.
 * Returns 0 for invalid sizes.
 */
PA_API size_t pa_decode_multi_split_workspace_size(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                                   int32_t head_dim, int32_t max_context_len,
                                                   int32_t partition_size);

/*
 * pa_decode_multi_split: pa_decode_multi (num_q_tokens new tokens per
 * sequence, causal among them) computed per partition of partition_size
 * tokens and merged by log-sum-exp as in pa_decode_split.  Long contexts are
 * spread over several CTAs, so one long sequence no longer sets the time of
 * the whole batch.  A partition that lies wholly after a new token's position
 * contributes nothing to that token.  Arguments as pa_decode_multi plus
 * max_context_len, partition_size and the workspace as pa_decode_split.
 */
PA_API int pa_decode_multi_split(void *out, const void *q, int32_t q_dtype, int32_t num_seqs,
                                 int32_t num_q_tokens, int32_t num_q_heads, const void *k_cache,
                                 const void *v_cache, const pa_cache_desc *cache, const int32_t *block_tables,
                                 int32_t max_blocks_per_seq, const int32_t *context_lens, float scale,
                                 float kv_scale, int32_t max_context_len, int32_t partition_size,
                                 void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_cache_and_decode: pa_reshape_and_cache of this step's new rows followed
 * by pa_decode_multi (partition_size 0) or pa_decode_multi_split
 * (partition_size > 0), in one launch: the CTA that attends over a new
 * token's position writes that token's K and V rows for its kv head into
 * the pool before it loads any tile, so the step needs no separate scatter
 * kernel.  The result and the pool bytes are the same as the two calls'.
 *   key, value    [num_seqs * num_q_tokens, num_kv_heads, head_dim] of q_dtype,
 *                 16-byte aligned; row s * num_q_tokens + j is new token j of
 *                 sequence s (position context_lens[s] - num_q_tokens + j)
 *   slot_mapping  int64 [num_seqs * num_q_tokens]: the slot of that row (as
 *                 pa_reshape_and_cache); negative = skip.  It must be the
 *                 position's slot in the sequence's own block table (a block
 *                 private to the sequence, as copy-on-write makes it); a slot
 *                 outside the pool is skipped, and either case sets
 *                 PA_DEVERR_SLOT.  In check mode a separate kernel first
 *                 scans the live table entries of every other sequence of
 *                 the batch and sets PA_DEVERR_SLOT when one of them names
 *                 the block a new row goes to (copy-on-write skipped: the
 *                 block is shared, so another sequence may read it while it
 *                 is written); the row is still written.
 * Other arguments as pa_decode_multi / pa_decode_multi_split (workspace and
 * max_context_len are read only when partition_size > 0).
 */
PA_API int pa_cache_and_decode(void *out, const void *q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_tokens,
                               int32_t num_q_heads, const void *key, const void *value,
                               const int64_t *slot_mapping, void *k_cache, void *v_cache,
                               const pa_cache_desc *cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                               const int32_t *context_lens, float scale, float kv_scale, int32_t max_context_len,
                               int32_t partition_size, void *workspace, size_t workspace_bytes,
                               pa_stream_t stream);

/*
 * pa_decode_split_noalloc: pa_decode_split without a workspace argument, for
 * callers that cannot allocate device memory when they call (for example a
 * serving process whose KV-cache pool already holds nearly all of HBM, or a
 * host framework that owns every device allocation of its plug-ins).  The
 * pages describe no such call; it exists only for those callers.
 * The partial results go to a 32 MiB scratch array compiled into the library
 * (held on every device that loads it until the process exits).  The
 * arguments, results and errors are those of pa_decode_split given a 32 MiB
 * workspace: argument errors first, then PA_ERR_WORKSPACE when
 * pa_decode_split_workspace_size(num_seqs, num_q_heads, head_dim,
 * max_context_len, partition_size) exceeds 32 MiB; an empty batch returns
 * PA_OK.  The first call on a device (and the first after its context was
 * destroyed and created anew) looks up the scratch address
 * (cudaGetSymbolAddress) and should come before any stream capture.  All calls on a device share the scratch, so
 * calls that can overlap on the GPU (unordered streams) race; calls ordered
 * on one stream are safe.  Allocates nothing.
 */
PA_API int pa_decode_split_noalloc(void *out, const void *q, int32_t q_dtype, int32_t num_seqs,
                                   int32_t num_q_heads, const void *k_cache, const void *v_cache,
                                   const pa_cache_desc *cache, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq, const int32_t *context_lens, float scale,
                                   float kv_scale, int32_t max_context_len, int32_t partition_size,
                                   pa_stream_t stream);

/*
 * Whole-block moves on the pool (all kv heads of a block, K and V).  One
 * block of one cache is num_kv_heads * block_size * head_dim * eb bytes.
 * Index arrays are int64 and, like every buffer here, device-accessible
 * (device memory, or pinned host memory mapped into the device's address
 * space, which is how blocks are swapped to and from the host).  Ids outside
 * the pool are skipped and recorded (PA_DEVERR_BLOCK_ID).  The index array
 * and the buffer are checked with cudaPointerGetAttributes before anything is
 * launched: pinned host memory is used through its device mapping, and
 * memory the device cannot reach returns PA_ERR_INVALID_ARG.
 *
 * pa_copy_blocks: for each pair (src, dst) of block_pairs[num_pairs][2],
 *   k_cache[dst] = k_cache[src] and v_cache[dst] = v_cache[src].  Used for
 *   copy-on-write of a shared, partially filled last block (review §6, §9).
 *   No dst may equal another pair's src or dst.
 * pa_gather_blocks: dst[i][0] = k_cache[block_ids[i]], dst[i][1] =
 *   v_cache[block_ids[i]]; dst is [num][2][Hkv][bs][D] of the cache dtype,
 *   16-byte aligned (swap-out to host memory for preemption, review §9).
 * pa_scatter_blocks: the inverse (swap-in).
 */
PA_API int pa_copy_blocks(void *k_cache, void *v_cache, const pa_cache_desc *cache, const int64_t *block_pairs,
                          int32_t num_pairs, pa_stream_t stream);
PA_API int pa_gather_blocks(void *dst, const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
                            const int64_t *block_ids, int32_t num, pa_stream_t stream);
PA_API int pa_scatter_blocks(void *k_cache, void *v_cache, const pa_cache_desc *cache, const void *src,
                             const int64_t *block_ids, int32_t num, pa_stream_t stream);

/*
 * Host block manager (no device work, not thread-safe: one owner, as the
 * scheduler owns block tables in the review, §6).  Physical blocks come from
 * a free list; a sequence's table only grows; pa_bm_fork shares every block
 * of the parent with the child (a pointer update: reference counts rise, no
 * data moves); pa_bm_append_tokens returns the slot of each new token and,
 * when the sequence's last block is shared and partially filled, first moves
 * the sequence to a private copy of it and reports the (src, dst) pair that
 * the caller copies with pa_copy_blocks.  A full shared block is never
 * copied: the next token starts a fresh block.  Calls that would need more
 * free blocks than exist change nothing and return PA_ERR_OUT_OF_BLOCKS.
 */
typedef struct pa_block_manager pa_block_manager;
PA_API pa_block_manager *pa_bm_create(int64_t num_blocks, int32_t block_size);  /* NULL on bad sizes */
PA_API void pa_bm_destroy(pa_block_manager *bm);
PA_API int pa_bm_add_sequence(pa_block_manager *bm, int64_t seq_id, int64_t num_tokens);
PA_API int pa_bm_fork(pa_block_manager *bm, int64_t parent_id, int64_t child_id);
PA_API int pa_bm_append_tokens(pa_block_manager *bm, int64_t seq_id, int32_t num_new, int64_t *slots_out,
                               int64_t *cow_pair_out /* [2] */, int32_t *num_cow_out);
PA_API int pa_bm_free_sequence(pa_block_manager *bm, int64_t seq_id);
PA_API int pa_bm_block_table(const pa_block_manager *bm, int64_t seq_id, int32_t *out, int32_t capacity,
                             int32_t *num_blocks_out, int64_t *num_tokens_out);
PA_API int64_t pa_bm_num_free_blocks(const pa_block_manager *bm);
PA_API int32_t pa_bm_refcount(const pa_block_manager *bm, int64_t block);  /* -1 for a bad id */
/* Unused slots summed over all sequences (each holds at most block_size - 1). */
PA_API int64_t pa_bm_tail_waste(const pa_block_manager *bm);
/* Violations of the block invariant (0 = consistent): refcount equals the
 * number of table entries naming the block, free exactly when unreferenced,
 * no block twice in one table, ceil(tokens / block_size) blocks per table. */
PA_API int64_t pa_bm_check(const pa_block_manager *bm);

/* Static description of a status code. */
PA_API const char *pa_status_string(int status);

/*
 * Check mode (also enabled by the environment variable PA_CHECK=1 at load):
 * every call synchronises its stream after the launch and returns
 * PA_ERR_BAD_INDEX / PA_ERR_TIMEOUT if a kernel recorded an error.  For
 * debugging; it is process-wide.  Returns the previous setting.
 */
PA_API int pa_set_check_mode(int enable);

/*
 * Synchronises the current device, returns the PA_DEVERR_* bits recorded by
 * kernels on it since the last call, and clears them.  Returns a negative
 * pa_status if the CUDA calls fail.
 */
PA_API int pa_get_device_error(void);

/*
 * pa_selftest_wait_timeout: self-test of the bounded waits in the decode and
 * prefill pipelines (every mbarrier wait there gives up after about one
 * second instead of hanging).  Enqueues on `stream` one kernel whose thread
 * waits, through the same wait helper, on a barrier that nothing arrives at:
 * after about one second the wait gives up, the kernel records
 * PA_DEVERR_TIMEOUT in the device error word and returns, and the context
 * stays usable.  Returns PA_OK, or PA_ERR_CUDA if the launch fails; the bit
 * shows in the next pa_get_device_error().
 */
PA_API int pa_selftest_wait_timeout(pa_stream_t stream);

/*
 * pa_probe_l2_read: measurement utility, not part of the attention path.
 * Enqueues on `stream` one kernel that reads the device buffer `buf` (16-byte
 * aligned, `bytes` long; make it smaller than L2 and read it once beforehand
 * so that it sits in L2) and writes nothing but, when a checksum of the data
 * equals a fixed pattern, 4 bytes at `sink` (device memory): timing the
 * launch with events gives the rate at which the SMs read from L2, the bound
 * of a decode whose K/V blocks are shared by many sequences.
 *   mode 0: `iters` passes over the whole buffer with plain 16-byte loads
 *           cached in L2 only (bytes a multiple of 16);
 *   mode 1: TMA boxes of 16 rows x 128 bytes, the box the attention kernels
 *           load K/V tiles with: one CTA per SM issues `iters` stages of 16
 *           boxes each (bytes a multiple of 2048).
 * *bytes_read (host memory) receives the bytes the launch reads.  Returns
 * PA_OK, PA_ERR_INVALID_ARG for a null pointer, a misaligned buffer, a size
 * the mode cannot use or iters <= 0, or PA_ERR_CUDA if the launch fails.
 */
PA_API int pa_probe_l2_read(const void* buf, size_t bytes, int32_t mode, int32_t iters, void* sink,
                            unsigned long long* bytes_read, pa_stream_t stream);

/* Library version: major * 10000 + minor * 100 + patch. */
PA_API int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */
