/*
 * bsa.h -- C interface of the GB300 (sm_103a) block-skipping causal prefill
 * attention library (libbsa.so).
 *
 * The operation is the one of the dynamic sparse attention deployment guide
 * ("长上下文推理加速方案部署实战：基于动态稀疏注意力机制的推理服务优化指南",
 * cloud.baidu.com article 9427124), §3.2 "dynamic sparse attention kernel":
 * a flash-style forward pass over 128x128 query/key tiles with an online
 * softmax. Key tiles are visited in ascending order; for each one the
 * per-row tile maximum of the scores is compared with the running row
 * maximum, and the tile is skipped -- no exponentials, no V load, no P.V
 * product -- when for every valid row of the query tile
 *
 *        tile_max(row) < running_max(row) + ln(lambda).
 *
 * §3.3 / §6.1 fix the direction (a larger lambda prunes more blocks) and
 * §5 step 3 the defaults (lambda = 0.01, block 128); lambda = 0 turns the
 * rule off and gives exact dense causal attention. GQA support is required
 * by §5 step 4; packed variable-length batches (continuous batching) and FP8
 * are the capabilities the block-sparse prefill monitoring page lists for
 * production prefill kernels.
 *
 * Conventions for every entry point:
 *  - All pointers named "device" must point to memory of the current CUDA
 *    device. The caller owns every buffer; the library never frees them and
 *    never writes to inputs.
 *  - Work is enqueued on `stream` (NULL = legacy default stream) and is fully
 *    asynchronous: no host synchronisation, no host read of device data.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns its status and enqueues nothing. Launch failures
 *    return BSA_ERR_CUDA. Errors found on the device (malformed cu_seqlens, a
 *    pipeline wait that ran out) are recorded in a per-stream status word
 *    that bsa_get_device_status() reads.
 *  - Calls on distinct streams may run concurrently, from any host threads:
 *    each (device, stream) has its own library-owned scratch area (work
 *    queue, tensor maps, status word, tables), grown on demand and kept until
 *    bsa_release_stream() or bsa_release(); host threads meet only briefly on
 *    the lookup of that state. Calls on one stream from several host threads
 *    are serialised by the library (they share its scratch area).
 *  - Per call the one-CTA prologue ranks the sequences longest first in
 *    O(n_seqs^2 / 1024) steps per thread and fills the level table in
 *    O(n_seqs * max_tiles / 1024): about a microsecond at 16 sequences, a
 *    few milliseconds at 10^5.
 *  - Every sequence may have at most 65536 query tiles and 65536 key tiles
 *    (8,388,608 tokens); longer ones are rejected on the device
 *    (BSA_ERR_BAD_SEQLENS, nothing written).
 */
#ifndef BSA_H
#define BSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA. */
typedef struct CUstream_st *bsa_stream_t;

typedef enum {
  BSA_BF16 = 0,     /* q, k, v are bfloat16 */
  BSA_FP8_E4M3 = 1  /* q, k, v are FP8 E4M3 codes with per-head scales */
} bsa_dtype_t;

typedef enum {
  BSA_OK = 0,
  BSA_ERR_INVALID_ARG = 1,  /* a host-checkable argument is out of range   */
  BSA_ERR_UNSUPPORTED = 2,  /* device is not sm_103, or d != 128           */
  BSA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed        */
  BSA_ERR_TIMEOUT = 4,      /* a device-side pipeline wait ran out         */
  BSA_ERR_NO_MEMORY = 5,    /* scratch allocation failed                   */
  BSA_ERR_BAD_SEQLENS = 6   /* device cu_seqlens not a valid prefix sum    */
} bsa_status_t;

/*
 * Block-skipping causal prefill attention, forward.
 *
 * q            device, [total_tokens, Hq, d] row-major (d fastest), 16-byte
 *              aligned; element type from `dtype`.
 * k, v         device, [total_tokens, Hkv, d], same type and alignment.
 * cu_seqlens   device int32 [n_seqs + 1]: cu[0] = 0, non-decreasing,
 *              cu[n_seqs] = total_tokens. Sequence s is rows
 *              cu[s] .. cu[s+1]-1 of q/k/v/out. total_tokens must not exceed
 *              the rows allocated in q, k, v and out (the library cannot
 *              check this). Validated on the device: a violation writes
 *              nothing, and records BSA_ERR_BAD_SEQLENS.
 * n_seqs       >= 1. Hq, Hkv >= 1 with Hq % Hkv == 0; query head h reads
 *              key/value head h / (Hq / Hkv) (grouped-query attention).
 * d            head dimension; 128 is the only supported value.
 * causal       1: causal (key position <= query position); 0: every key of
 *              the sequence is visible (same skip rule, all tiles visited).
 * lambda       skip threshold, 0 <= lambda < 1; 0 disables skipping. NaN
 *              is rejected. With lambda > 0 the decisions are taken first
 *              for every causal key tile (QK^T and the row maxima only; a
 *              skipped tile never raises the running max, so each decision
 *              follows from the maxima of the tiles before it) and then the
 *              kept tiles are computed; lambda = 0 runs one dense pass.
 * dtype        BSA_BF16, or BSA_FP8_E4M3 with scales set by
 *              bsa_set_fp8_scales() on the calling thread.
 * out          device bfloat16 [total_tokens, Hq, d]; must not overlap the
 *              inputs. Every row of every sequence is written.
 * lse          device float32 [Hq, total_tokens] or NULL: natural-log
 *              log-sum-exp of the scaled scores over the kept entries.
 * skip_bitmap  device uint32 or NULL. For sequence s with n_s =
 *              ceil(L_s/128) tiles and W_s = ceil(n_s/32) words per row,
 *              row (s, h, i) starts at word sum_{t<s}(Hq n_t W_t) +
 *              (h n_s + i) W_s; bit j%32 of word j/32 is 1 when key tile j
 *              was skipped for query tile i. Unvisited tiles read 0. Size
 *              in words: bsa_skip_bitmap_words().
 * stream       CUDA stream.
 *
 * The softmax scale is 1/sqrt(d). Scores are accumulated in fp32 on the
 * tensor cores; exponentials are base-2 on the scaled scores.
 */
bsa_status_t bsa_prefill_fwd(const void *q, const void *k, const void *v,
                             const int32_t *cu_seqlens, int32_t n_seqs,
                             int32_t Hq, int32_t Hkv, int32_t d, int32_t causal,
                             float lambda, bsa_dtype_t dtype, void *out,
                             float *lse, uint32_t *skip_bitmap,
                             bsa_stream_t stream);

/*
 * Chunked prefill: the same forward pass when a sequence's queries are only
 * its last Lq positions and its keys/values (earlier chunks included, e.g.
 * read back from a KV cache) number Lk >= Lq -- the chunked prefill that the
 * prefill-acceleration blog (mhpq.cn news 313192, §3.1) and FlowPrefill
 * describe for splitting long prompts. Query row r of sequence s sits at key
 * position Lk - Lq + r (bottom-right causal alignment); key tiles are visited
 * from 0 in order with the same skip rule.
 *
 * q            device [Tq, Hq, d], packed by cu_seqlens_q.
 * k, v         device [Tk, Hkv, d], packed by cu_seqlens_k.
 * cu_seqlens_q, cu_seqlens_k   device int32 [n_seqs + 1] prefix sums (both
 *              start at 0); causal requires Lk >= Lq for every sequence.
 *              Violations are recorded on the device (BSA_ERR_BAD_SEQLENS).
 * out          device bf16 [Tq, Hq, d]; lse device float32 [Hq, Tq] or NULL.
 * skip_bitmap  one row per query tile: n_q = ceil(Lq/128) rows of
 *              W = ceil(ceil(Lk/128)/32) words per (sequence, head);
 *              sequence s starts at word sum_{t<s}(Hq n_q,t W_t), row (s,h,i)
 *              at + (h n_q + i) W; bit j = key tile j. Size:
 *              bsa_skip_bitmap_words_chunked().
 * Other arguments, conventions and errors as bsa_prefill_fwd, which is this
 * call with cu_seqlens_k == cu_seqlens_q.
 */
bsa_status_t bsa_prefill_fwd_chunked(const void *q, const void *k, const void *v,
                                     const int32_t *cu_seqlens_q,
                                     const int32_t *cu_seqlens_k, int32_t n_seqs,
                                     int32_t Hq, int32_t Hkv, int32_t d,
                                     int32_t causal, float lambda,
                                     bsa_dtype_t dtype, void *out, float *lse,
                                     uint32_t *skip_bitmap, bsa_stream_t stream);

/*
 * Paged KV cache: chunked prefill whose keys and values are read from a pool
 * of 128-token pages through a page table -- the paged KV cache that the
 * deployment guide's §5 step 4 recommends for long contexts and that the
 * block-sparse prefill monitoring page lists as a production requirement
 * (FlashPrefill V2). A page holds one 128-key tile, so key tile j of
 * sequence s is page page_table[s * max_pages_per_seq + j] of the pool.
 *
 * k_cache, v_cache  device [num_pages, 128, Hkv, d] (d fastest), 16-byte
 *              aligned; only the pages a sequence uses are read.
 * page_table   device int32 [n_seqs, max_pages_per_seq]; entries for the
 *              ceil(Lk/128) tiles of each sequence must lie in
 *              [0, num_pages) (checked on the device: BSA_ERR_BAD_SEQLENS,
 *              nothing written); later entries are ignored.
 * cu_seqlens_k device int32 [n_seqs + 1]: prefix sums of the key counts Lk
 *              (used for lengths only; keys live in the pages).
 * Everything else as bsa_prefill_fwd_chunked (queries are the last Lq of
 * Lk positions; bitmap layout and size as there).
 */
bsa_status_t bsa_prefill_fwd_paged(const void *q, const void *k_cache,
                                   const void *v_cache, const int32_t *page_table,
                                   int32_t max_pages_per_seq, int32_t num_pages,
                                   const int32_t *cu_seqlens_q,
                                   const int32_t *cu_seqlens_k, int32_t n_seqs,
                                   int32_t Hq, int32_t Hkv, int32_t d,
                                   int32_t causal, float lambda,
                                   bsa_dtype_t dtype, void *out, float *lse,
                                   uint32_t *skip_bitmap, bsa_stream_t stream);

/*
 * Same forward pass as bsa_prefill_fwd, same arguments and results, for
 * callers that may not allocate device memory -- for example a serving
 * engine that reserves nearly all of HBM for its own pool up front and
 * forbids allocations inside kernels' host calls, where a surprise
 * allocation could fail or stall the device. The pages have no counterpart:
 * this is an interface variant, not part of the method.
 *
 * Allocates nothing: its scratch (work queue, tensor maps, scheduling
 * tables, status word) is a fixed array of about 270 KiB compiled into the
 * library and resident on every GPU that loads it until the process exits.
 * Limit: n_seqs <= 1024 (larger batches return BSA_ERR_INVALID_ARG);
 * sequences longer than 8M tokens are rejected on the device as with
 * bsa_prefill_fwd. The first call in a device's context looks up that
 * context's address of the array (and sets the kernels' shared-memory
 * limit); make that first call before any stream capture. All calls share
 * the one array and each call rewrites it: calls whose GPU work overlaps
 * (on different streams) race and must not be issued; calls on one stream
 * are safe. Device-side errors (a malformed cu_seqlens, which leaves the
 * outputs unwritten, or a pipeline time-out) accumulate in the array's
 * status word until bsa_get_noalloc_status() reads and clears them.
 */
bsa_status_t bsa_prefill_fwd_noalloc(const void *q, const void *k, const void *v,
                                     const int32_t *cu_seqlens, int32_t n_seqs,
                                     int32_t Hq, int32_t Hkv, int32_t d,
                                     int32_t causal, float lambda,
                                     bsa_dtype_t dtype, void *out, float *lse,
                                     uint32_t *skip_bitmap, bsa_stream_t stream);

/*
 * Status of the bsa_prefill_fwd_noalloc calls on the current device:
 * synchronises `stream` (the stream those calls were made on), returns the
 * device-side status they recorded since the last read (BSA_OK,
 * BSA_ERR_BAD_SEQLENS or BSA_ERR_TIMEOUT) and clears it. Allocates nothing.
 * BSA_OK if no such call was made in this context yet.
 */
bsa_status_t bsa_get_noalloc_status(bsa_stream_t stream);

/*
 * Per-head dequantisation scales for the next BSA_FP8_E4M3 calls made on this
 * host thread: device float32 arrays q_scale [Hq], k_scale [Hkv],
 * v_scale [Hkv]; a stored code x8 stands for x8 * scale. The pointers are
 * kept (not copied) and must stay valid while such calls run. Passing three
 * NULLs clears them. Returns BSA_ERR_INVALID_ARG if only some are NULL.
 */
bsa_status_t bsa_set_fp8_scales(const float *q_scale, const float *k_scale,
                                const float *v_scale);

/*
 * Per-head FP8 E4M3 quantisation of a bfloat16 tensor x [tokens, H, d]
 * (device, 16-byte aligned): scale[h] = max|x[:, h, :]| / 448 in float32
 * (1.0 for an all-zero head), codes = E4M3(x / scale) rounded to nearest
 * even with saturation to +-448. x_e4m3 device uint8 [tokens, H, d];
 * scale device float32 [H]. d must be a multiple of 8; tokens >= 0.
 */
bsa_status_t bsa_quantize_fp8(const void *x_bf16, int64_t tokens, int32_t H,
                              int32_t d, uint8_t *x_e4m3, float *scale,
                              bsa_stream_t stream);

/*
 * Number of uint32 words of the skip bitmap for a batch, from a HOST copy of
 * cu_seqlens. Returns -1 for a malformed cu_seqlens or n_seqs < 1, Hq < 1.
 */
int64_t bsa_skip_bitmap_words(const int32_t *cu_seqlens_host, int32_t n_seqs,
                              int32_t Hq);

/*
 * Skip-bitmap size in words for bsa_prefill_fwd_chunked, from HOST copies of
 * both boundary arrays. Returns -1 if either is malformed.
 */
int64_t bsa_skip_bitmap_words_chunked(const int32_t *cu_seqlens_q_host,
                                      const int32_t *cu_seqlens_k_host,
                                      int32_t n_seqs, int32_t Hq);

/*
 * Decode with block skipping: a few new queries per sequence (the last Lq of
 * its Lk positions, as bsa_prefill_fwd_chunked) against all its keys, with
 * the key range split across the GPU. Same rule, decisions and outputs as
 * bsa_prefill_fwd_chunked (the deployment guide applies the rule in decoding
 * too, §6.1 suggesting lambda = 0.005 there).
 *
 * The split restates the order rule: a skipped tile never raises the running
 * max (tile_max < m + ln(lambda) < m), so the running max before key tile j
 * is the prefix max of the tile maxima before j. One persistent kernel (one
 * CTA per SM) takes work items (sequence, KV head, split of 8 key tiles, or
 * 4 when (Hq / Hkv) * max_seqlen_q > 16) in order: each publishes its split's
 * tile maxima, reads those of the earlier splits of its (sequence, KV head),
 * decides its tiles and computes P V for the kept ones; the split that
 * finishes last merges the partial results. Outputs are the online softmax
 * over the kept tiles, merged across splits (P and the merge in fp32). A
 * work item waits (bounded by the wait limit) only for items of lower index;
 * a wait that runs out stops the call and records BSA_ERR_TIMEOUT.
 *
 * q, k, v, cu_seqlens_q, cu_seqlens_k, n_seqs, Hq, Hkv, d, causal, lambda,
 * out, lse, skip_bitmap: as bsa_prefill_fwd_chunked (bfloat16 only; the bitmap
 * layout and size are those of bsa_skip_bitmap_words_chunked).
 * max_seqlen_q  >= every Lq (checked on the device); (Hq / Hkv) * max_seqlen_q
 *               <= 32 and Hq / Hkv <= 16.
 * total_k       cu_seqlens_k[n_seqs], the rows of k and v (checked on the
 *               device; a mismatch writes nothing, BSA_ERR_BAD_SEQLENS).
 * Scratch (per-split maxima, per-split partial outputs, per-call counters)
 * is library-owned, per stream, grown stream-ordered, laid out for sizes that
 * only grow and zero-filled whenever it is laid out again; per-call state
 * carries a per-stream call count, so a call that stopped early leaves
 * nothing the next one has to clear.
 */
bsa_status_t bsa_decode_fwd(const void *q, const void *k, const void *v,
                            const int32_t *cu_seqlens_q,
                            const int32_t *cu_seqlens_k, int32_t n_seqs,
                            int32_t max_seqlen_q, int64_t total_k, int32_t Hq,
                            int32_t Hkv, int32_t d, int32_t causal,
                            float lambda, void *out, float *lse,
                            uint32_t *skip_bitmap, bsa_stream_t stream);

/*
 * Token-block importance ("UniPrefill：通过分块动态稀疏化实现通用长上下文预填充
 * 加速", §3.2 Eq. (3)-(4)). For every sequence and query head h, the attention
 * weights A[j, i] of the last n = min(n_window, L) query positions j over
 * the sequence's keys i, with the softmax (scale 1/sqrt(d)) normalised over
 * the whole key range, are averaged over the n rows and summed over blocks
 * of G = 128 keys:
 *
 *        score[h, g] = (1 / (n G)) * sum_{i in block g} sum_j A[j, i].
 *
 * Row j attends the keys i <= j when causal = 1 and every key of the
 * sequence when causal = 0. A sequence's block scores of one head add up to
 * 1/G. Readings where the page is silent: G = 128 (this library's tile), the
 * division by G also for a short last block (as Eq. 4 writes it), one score
 * row per query head (GQA: head h reads key head h / (Hq / Hkv)).
 *
 * q, k         device bfloat16 [total_tokens, Hq | Hkv, d], 16-byte aligned.
 * cu_seqlens   device int32 [n_seqs + 1], as for bsa_prefill_fwd.
 * d            128 only. n_window 1..128. causal 0 or 1.
 * total_blocks sum over sequences of ceil(L_s / 128), from
 *              bsa_importance_blocks(); checked on the device against
 *              cu_seqlens (a mismatch writes nothing and records
 *              BSA_ERR_BAD_SEQLENS).
 * scores       device float32 [Hq, total_blocks]; sequence s's blocks start
 *              at column sum_{t<s} ceil(L_t / 128).
 * mean_scores  device float32 [total_blocks] or NULL: the mean over query
 *              heads, the score the selection below ranks.
 * Scratch (two float tables of Hq x total_blocks x 128) is library-owned,
 * per stream, grown stream-ordered.
 */
bsa_status_t bsa_block_importance(const void *q, const void *k,
                                  const int32_t *cu_seqlens, int32_t n_seqs,
                                  int32_t Hq, int32_t Hkv, int32_t d,
                                  int32_t n_window, int32_t causal,
                                  int64_t total_blocks, float *scores,
                                  float *mean_scores, bsa_stream_t stream);

/*
 * Top-p block selection (same page, §3.3): per sequence, the block indices
 * sorted by descending score (ties: ascending index) and the smallest k*
 * such that the running sum of the first k* sorted scores reaches p times
 * the sum of all of them (running sums in double precision; the total is
 * the running sum at the last block).
 *
 * scores       device float32 [total_blocks] (finite, >= 0), laid out as
 *              bsa_block_importance's mean_scores.
 * cu_seqlens   device int32 [n_seqs + 1]; every sequence may have at most
 *              16384 blocks (2M tokens), else nothing is written and
 *              BSA_ERR_BAD_SEQLENS is recorded.
 * p            0 < p <= 1 (NaN rejected).
 * order        device int32 [total_blocks]: order[off_s + r] = block index
 *              (within sequence s) of rank r.
 * n_selected   device int32 [n_seqs]: k* (0 for an empty sequence).
 * keep         device uint8 [total_blocks] or NULL: 1 for a kept block.
 */
bsa_status_t bsa_top_p_select(const float *scores, const int32_t *cu_seqlens,
                              int32_t n_seqs, int64_t total_blocks, float p,
                              int32_t *order, int32_t *n_selected,
                              uint8_t *keep, bsa_stream_t stream);

/*
 * Number of 128-token blocks of a batch, sum of ceil(L_s / 128), from a HOST
 * copy of cu_seqlens. -1 for a malformed cu_seqlens or n_seqs < 1.
 */
int64_t bsa_importance_blocks(const int32_t *cu_seqlens_host, int32_t n_seqs);

/*
 * Synchronises `stream`, returns the device-side status recorded by the
 * calls made on it since the last read (BSA_OK, BSA_ERR_BAD_SEQLENS or
 * BSA_ERR_TIMEOUT) and clears it. BSA_ERR_CUDA if the synchronisation
 * itself fails.
 */
bsa_status_t bsa_get_device_status(bsa_stream_t stream);

/*
 * Fault drill, for tests of the failure path only. For the calling host
 * thread, later bsa_prefill_fwd*, bsa_decode_fwd and bsa_block_importance
 * calls bound every device pipeline wait by wait_limit_ns, and, when
 * drop_k_load >= 0, the K-tile TMA producer of every CTA (of the forward,
 * decode score or importance score kernel) leaves out its drop_k_load-th K
 * tile load so that the MMA warp's wait for it runs out. The kernel then
 * records BSA_ERR_TIMEOUT (read it with bsa_get_device_status), waits with
 * the same bound for the copies and MMAs it has in flight, frees its tensor
 * memory and returns; the kernels after it in the same call run on whatever
 * the tables hold (the result is meaningless, the status says so) and the
 * context stays usable. bsa_debug_fault_drill(-1, 2000000000) restores the
 * defaults.
 */
bsa_status_t bsa_debug_fault_drill(int32_t drop_k_load, int64_t wait_limit_ns);

/* Static text for a status code. */
const char *bsa_status_string(bsa_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t bsa_version(void);

/*
 * Frees all cached scratch areas. Must not be called while work issued by
 * this library is still running on any stream.
 */
void bsa_release(void);

/*
 * Frees the scratch areas kept for `stream` on the current device
 * (stream-ordered: work already enqueued on it finishes first). Call it
 * before destroying a stream the library was used on; otherwise its scratch
 * stays allocated until bsa_release(). No other host thread may be making
 * calls on that stream at the same time. BSA_ERR_CUDA if a free fails.
 */
bsa_status_t bsa_release_stream(bsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H */
