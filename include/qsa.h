/*
 * qsa.h -- C ABI of libqsa.so, a B300 (sm_103a) implementation of Qwen Sparse
 * Attention (QSA), the global-attention layer of the Qwen3.8-Flash-Next
 * GDN + QSA hybrid.
 *
 * What the layer computes (Qwen3.8-Flash-Next launch post, "Model
 * Architecture / Attention: GDN + QSA for Efficient Memory and Precise
 * Retrieval"; model card "Model Overview / Qwen Sparse Attention"): a
 * lightweight indexer groups the sequence into micro-blocks, scores every
 * past block for every query, the best blocks within a budget are selected,
 * and attention runs over the selected blocks only.  Shapes from the model
 * card: 24 query heads / 2 KV heads of dim 256, rotary dim 64, indexer MQA
 * with 4 query heads and 1 shared key head of dim 128, budget 512 blocks =
 * 2048 tokens (so a micro-block is 4 tokens).  rope_theta 1e7 and
 * partial_rotary_factor 0.25 come from the model card's "Processing
 * Ultra-Long Texts" rope_parameters.
 *
 * Where the pages are silent this library fixes:
 *   - block key  kblk[b] = bf16( (((ki[4b]+ki[4b+1])+ki[4b+2])+ki[4b+3]) / 4 ), sum in fp64;
 *   - block score s[t,b] = sum_h w[t,h] * max(0, qi[t,h] . kblk[b]), b < c(t) = floor(t/4);
 *   - selection: block c(t) always; plus the (budget-1) past blocks with the
 *     highest score (ties: lower block index first); all past blocks if fewer;
 *   - RoPE: rotate-half over dims [0,64) (pairs i, i+32), angle pos*theta^(-2i/64),
 *     rotated values rounded to bf16; dims [64,256) unchanged; no RoPE on the indexer;
 *   - attention: keys j in the selected blocks with j <= t, query head h uses
 *     KV head h/12, softmax scale 1/16 unless configured; fp32 accumulation.
 *
 * Conventions for every call:
 *   - All tensors are dense row-major ("C order"), device pointers unless
 *     stated, and 16-byte aligned.  bf16 values are passed as raw 16-bit
 *     patterns (qsa_bf16).
 *   - The caller owns every buffer, workspaces included.  The library never
 *     allocates or frees device memory and keeps no state between calls
 *     other than a cached per-device property query and a resolved driver
 *     entry point (qsa_sparse_attn_decode_noalloc, at the end, is the one
 *     call that uses a built-in scratch array instead of a workspace).
 *   - Calls run on the current CUDA device: `stream` and every pointer must
 *     belong to it.
 *   - Calls only enqueue work on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and return without synchronising.  One call,
 *     qsa_prefill_overlapped, also forks a helper stream and events of its
 *     own (released by CUDA once their work is done) and joins them back
 *     into `stream` before it returns.
 *   - Argument errors are reported synchronously by the return value, and
 *     then NOTHING is launched and no output is written.  A failed launch
 *     returns QSA_ERR_CUDA (qsa_last_error_detail() says which).
 *   - Problems found on the device (a bounded wait that ran out, an index
 *     range check) are written to the caller's device word *dev_status
 *     (first error wins; the caller sets it to 0 beforehand and reads it
 *     after synchronising).  Kernels never trap.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t qsa_bf16; /* raw bf16 bit pattern */

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size          */
    QSA_ERR_UNSUPPORTED = 2,  /* config or size outside what is compiled in */
    QSA_ERR_WORKSPACE = 3,    /* workspace missing or too small             */
    QSA_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed          */
    QSA_ERR_TIMEOUT = 5,      /* device status: a bounded wait ran out      */
    QSA_ERR_DEVICE_CHECK = 6  /* device status: an in-kernel check failed   */
} qsa_status;

/* The layer's shape.  Only the model card's shapes are compiled in:
 * block_size 4, n_q_heads 24, n_kv_heads 2, head_dim 256, rope_dim 64,
 * n_idx_heads 4, idx_dim 128 (anything else -> QSA_ERR_UNSUPPORTED).
 * budget_blocks may be 1..512.  rope_theta > 0.  softmax_scale <= 0 means
 * 1/sqrt(head_dim).
 * YaRN (model card "Processing Ultra-Long Texts": factor 4 over an original
 * context of 262,144; the published YaRN method): yarn_factor <= 1 turns it
 * off (the default).  With s = yarn_factor > 1 every rotary frequency w of
 * wavelength 2 pi / w becomes (1 - g) w / s + g w, where g ramps linearly
 * from 0 to 1 as r = yarn_original_max_pos / wavelength goes from
 * yarn_alpha to yarn_beta (defaults 1 and 32), and the attention logits are
 * multiplied by (0.1 ln s + 1)^2 on top of softmax_scale.  The same
 * configuration must be used for K-prep (keys) and attention (queries). */
typedef struct {
    int block_size;
    int budget_blocks;
    int n_q_heads;
    int n_kv_heads;
    int head_dim;
    int rope_dim;
    int n_idx_heads;
    int idx_dim;
    double rope_theta;
    float softmax_scale;
    float yarn_factor;
    int yarn_original_max_pos;
    float yarn_alpha;
    float yarn_beta;
} qsa_config;

/* Fills the model card's configuration (budget 512, theta 1e7, scale 1/16,
 * YaRN off with the card's factor-4 settings ready: original context 262,144,
 * alpha 1, beta 32). */
void qsa_default_config(qsa_config *cfg);

/* Human-readable name of a status code (static storage). */
const char *qsa_status_string(qsa_status s);

/* Detail of the last error returned on this host thread (static storage). */
const char *qsa_last_error_detail(void);

/* ------------------------------------------------------------------------
 * K-prep: micro-block keys and RoPE'd keys for `batch` sequences stored with
 * a stride of `max_ctx` tokens (prefill: batch 1, max_ctx = L).
 *   ki     [batch, max_ctx, 128]    per-token indexer keys (in)
 *   k      [batch, max_ctx, 2, 256] keys before RoPE (in); may be NULL
 *   k_rot  [batch, max_ctx, 2, 256] keys after RoPE (out); may equal k;
 *          NULL iff k is NULL (then no RoPE work)
 *   kblk   [batch, max_ctx/4, 128]  block keys (out), rows 0..L/4-1 written
 *   L      tokens per sequence to process, 1 <= L <= max_ctx; key j gets
 *          position j.
 * Block keys: launch post, "Attention: GDN + QSA" (micro-block aggregation);
 * RoPE: model card "Processing Ultra-Long Texts" rope_parameters.
 * ---------------------------------------------------------------------- */
qsa_status qsa_kprep(const qsa_config *cfg, int batch, int64_t L, int64_t max_ctx,
                     const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot,
                     qsa_bf16 *kblk, void *stream);

/* ------------------------------------------------------------------------
 * Prefill indexer + selection for one sequence of L tokens (positions 0..L-1):
 * K-prep, then the block scores of every query against every past block on
 * the tensor cores, fused with a streaming exact top-(budget-1) per query; the
 * score matrix never reaches memory.
 *   qi   [L, 4, 128]   indexer queries        w [L, 4] per-head weights
 *   ki   [L, 128]      indexer keys
 *   k    [L, 2, 256]   keys before RoPE, k_rot [L, 2, 256] after (may alias;
 *                      both NULL to skip the RoPE of K)
 *   idx  [L, budget]   int32 out: selected blocks ascending, the current block
 *                      last among them, then -1 padding
 *   score [L, budget]  float out (may be NULL): the block scores of idx;
 *                      +inf for the current block, -inf for padding
 *   ws   workspace of at least qsa_index_topk_workspace_bytes(cfg, L) bytes
 * Launch post, "Attention: GDN + QSA"; budget: model card "Model Overview /
 * Qwen Sparse Attention".
 * ---------------------------------------------------------------------- */
size_t qsa_index_topk_workspace_bytes(const qsa_config *cfg, int64_t L);
qsa_status qsa_index_topk(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                          const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot, int64_t L,
                          int32_t *idx, float *score, void *ws, size_t ws_bytes,
                          int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Dense block scores, for inspection and testing of the indexer at small L
 * (the same tensor-core kernel as qsa_index_topk with the selection replaced
 * by a store).  scores [L, L/4] float: scores[t, b] for b < floor(t/4);
 * other entries are left untouched.  L <= 65536.
 * ws: at least qsa_index_topk_workspace_bytes(cfg, L) bytes.
 * ---------------------------------------------------------------------- */
qsa_status qsa_index_scores(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                            const qsa_bf16 *ki, int64_t L, float *scores, void *ws,
                            size_t ws_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Prefill block-sparse attention for one sequence of L tokens.
 *   q     [L, 24, 256]  queries before RoPE (rotated in-kernel at position t)
 *   k_rot [L, 2, 256]   keys after RoPE;  v [L, 2, 256]
 *   idx   [L, budget]   selection as written by qsa_index_topk (entries < 0,
 *                       beyond the query's block, or not ascending are ignored
 *                       safely: every gathered row is range-checked)
 *   out   [L, 24, 256]  bf16 out;  lse [L, 24] float out (natural log of the
 *                       softmax denominator of the scaled logits), may be NULL
 * Launch post, "Attention: GDN + QSA" (attention over the selected regions);
 * head layout: model card "Model Overview / Qwen Sparse Attention".
 * ---------------------------------------------------------------------- */
qsa_status qsa_sparse_attn_prefill(const qsa_config *cfg, const qsa_bf16 *q,
                                   const qsa_bf16 *k_rot, const qsa_bf16 *v, const int32_t *idx,
                                   int64_t L, qsa_bf16 *out, float *lse, int32_t *dev_status,
                                   void *stream);

/* ------------------------------------------------------------------------
 * Token-level indexer (the DSA-style variant the launch post contrasts QSA
 * with, "Attention: GDN + QSA": a token-level indexer scores every past
 * position, so its cost grows 4x against 4-token micro-blocks).  The same
 * kernel as qsa_index_topk with one token per selection unit: the unit keys
 * are the indexer keys themselves (no mean), query t sees units 0..t-1 and
 * always keeps its own token t.
 *   qi [L, 4, 128], w [L, 4], ki [L, 128]; idx [L, budget] int32 out: the
 *   selected past tokens ascending, then t, then -1 padding (budget counts
 *   tokens here, 1..512); score [L, budget] or NULL as for qsa_index_topk.
 *   ws: at least qsa_index_topk_tokens_workspace_bytes(cfg, L) bytes.
 * ---------------------------------------------------------------------- */
size_t qsa_index_topk_tokens_workspace_bytes(const qsa_config *cfg, int64_t L);
qsa_status qsa_index_topk_tokens(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                                 const qsa_bf16 *ki, int64_t L, int32_t *idx, float *score, void *ws,
                                 size_t ws_bytes, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Prefill of a new chunk after a cached prefix (prefix-cache serving: the
 * launch post, "Model Architecture / Attention: GDN + QSA for Efficient
 * Memory and Precise Retrieval", measures prefill at a 90% prefix-cache hit
 * rate).  Only the chunk's Lq query rows are computed; they are positions
 * q_offset .. q_offset+Lq-1 of the sequence, and their keys are every block
 * and token before them, cached or new.  The results are those of a full
 * prefill restricted to these rows (same definition, same kernels).
 *
 * qsa_kprep_range: block keys of the complete blocks t_begin/4 .. t_end/4-1
 *   and RoPE'd key rows t_begin .. t_end-1 (the rows and blocks a new chunk
 *   adds; a block straddling t_begin is recomputed from ki, which must hold
 *   every row before t_end).
 *   ki [t_end, 128]; k, k_rot [t_end, 2, 256] (may alias; both NULL to skip
 *   RoPE); kblk [t_end/4, 128] out.
 * qsa_index_topk_cached: qi [Lq, 4, 128], w [Lq, 4] (the chunk's rows; w
 *   needs only 2-byte alignment, so a chunk may start at any row);
 *   kblk [(q_offset+Lq)/4, 128] the block keys so far; idx, score [Lq,
 *   budget] as for qsa_index_topk.  ws: at least
 *   qsa_index_topk_cached_workspace_bytes(cfg, Lq) bytes, 16-byte aligned.
 * qsa_sparse_attn_prefill_cached: q [Lq, 24, 256] (the chunk's rows, before
 *   RoPE); k_rot, v [q_offset+Lq, 2, 256]; idx [Lq, budget]; out [Lq, 24, 256];
 *   lse [Lq, 24] or NULL.
 * Errors as for the full-sequence calls; q_offset + Lq is at most 2^24.
 * ---------------------------------------------------------------------- */
qsa_status qsa_kprep_range(const qsa_config *cfg, const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot,
                           qsa_bf16 *kblk, int64_t t_begin, int64_t t_end, void *stream);
size_t qsa_index_topk_cached_workspace_bytes(const qsa_config *cfg, int64_t Lq);
qsa_status qsa_index_topk_cached(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                                 const qsa_bf16 *kblk, int64_t q_offset, int64_t Lq, int32_t *idx,
                                 float *score, void *ws, size_t ws_bytes, int32_t *dev_status,
                                 void *stream);
/* qsa_index_topk_cached_ctas: qsa_index_topk_cached with the indexer's
 * persistent grid limited to max_ctas CTAs (one per SM; 0 or more than the
 * SM count = every SM), so that other work can run beside it on the other
 * SMs.  Same results for every max_ctas; INVALID_ARG if max_ctas < 0. */
qsa_status qsa_index_topk_cached_ctas(const qsa_config *cfg, const qsa_bf16 *qi, const qsa_bf16 *w,
                                      const qsa_bf16 *kblk, int64_t q_offset, int64_t Lq, int32_t *idx,
                                      float *score, int max_ctas, void *ws, size_t ws_bytes,
                                      int32_t *dev_status, void *stream);
qsa_status qsa_sparse_attn_prefill_cached(const qsa_config *cfg, const qsa_bf16 *q,
                                          const qsa_bf16 *k_rot, const qsa_bf16 *v, const int32_t *idx,
                                          int64_t q_offset, int64_t Lq, qsa_bf16 *out, float *lse,
                                          int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Whole prefill of one sequence with the indexer and the attention running
 * side by side (the launch post, "Attention: GDN + QSA": indexer, selection
 * and attention over the selected regions, with the same definitions as
 * qsa_index_topk followed by qsa_sparse_attn_prefill, and bit-identical
 * results).  The indexer's time goes to instruction issue and the
 * attention's to HBM bytes, so the query rows are cut into chunks and the
 * indexer of chunk j runs on a share of the SMs while the attention of chunk
 * j-1 runs on the rest; the first and the last chunk come in four parts, so
 * the stages run alone (the first indexer, the last attention) for a quarter
 * of a chunk only.
 *   q [L, 24, 256], qi [L, 4, 128], w [L, 4], ki [L, 128], k [L, 2, 256]
 *   (before RoPE), k_rot [L, 2, 256] out (may equal k), v [L, 2, 256];
 *   idx [L, budget] and score [L, budget] (or NULL) as for qsa_index_topk;
 *   out [L, 24, 256], lse [L, 24] (or NULL) as for qsa_sparse_attn_prefill.
 *   ws: at least qsa_prefill_overlapped_workspace_bytes(cfg, L) bytes,
 *   16-byte aligned.
 * The call enqueues on `stream`; internally it forks a higher-priority
 * stream for the indexer and joins it back before the last attention chunk,
 * so work enqueued on `stream` afterwards sees every output.  The split of
 * the SMs adapts while the call runs: before it enqueues chunk j's indexer
 * (j >= 3) the host waits for the indexer of chunk j-1 and the attention of
 * chunk j-2 and rescales the plan's costs by their measured times, so the
 * call returns only when the last chunk is enqueued, about one chunk before
 * the prefill ends.  Errors as for
 * the two calls it combines; QSA_ERR_CUDA if the helper stream or its
 * events cannot be created.
 *
 * Prefills shorter than 262,144 tokens (whose K/V mostly stays in L2, so the
 * attention is bound by its SMs, not by HBM), budget 1, and calls on a stream
 * that is being captured into a CUDA graph run the two stages one after the
 * other on `stream`.
 *
 * qsa_prefill_overlap_plan: the chunking this call uses on a GPU with `sms`
 *   SMs (host only, no GPU needed).  Writes n+1 chunk starts
 *   (chunk_begin[0] = 0, chunk_begin[n] = L; every inner start a multiple of
 *   64) and n indexer grid sizes (index_ctas[0] = sms: the first chunk's
 *   indexer runs alone; the call starts from these and adapts them from the
 *   fourth chunk on), and returns n (1 <= n <= max_chunks), or 0 on
 *   invalid arguments.  chunk_begin needs max_chunks + 1 entries.  The first
 *   and the last four chunks are the parts of the edge chunks when max_chunks
 *   leaves room for them (22 chunks at 1,048,576 tokens).
 * ---------------------------------------------------------------------- */
size_t qsa_prefill_overlapped_workspace_bytes(const qsa_config *cfg, int64_t L);
qsa_status qsa_prefill_overlapped(const qsa_config *cfg, const qsa_bf16 *q, const qsa_bf16 *qi,
                                  const qsa_bf16 *w, const qsa_bf16 *ki, const qsa_bf16 *k, qsa_bf16 *k_rot,
                                  const qsa_bf16 *v, int64_t L, int32_t *idx, float *score, qsa_bf16 *out,
                                  float *lse, void *ws, size_t ws_bytes, int32_t *dev_status, void *stream);
int qsa_prefill_overlap_plan(const qsa_config *cfg, int64_t L, int sms, int max_chunks,
                             int64_t *chunk_begin, int *index_ctas);

/* ------------------------------------------------------------------------
 * Decode: one new token for each of `batch` sequences.  Sequence s holds
 * seq_lens[s] = T tokens in its caches (the new token included, at position
 * T-1, its K/V already written); caches have a stride of max_ctx tokens.
 *   q        [batch, 24, 256]  new queries before RoPE
 *   qi       [batch, 4, 128], w [batch, 4]
 *   k_cache  [batch, max_ctx, 2, 256] keys after RoPE (qsa_kprep output)
 *   v_cache  [batch, max_ctx, 2, 256]
 *   kblk_cache [batch, max_ctx/4, 128] block keys (qsa_kprep output); the
 *            complete blocks before the query's block are read
 *   seq_lens [batch] int32, DEVICE memory, 1 <= T <= max_ctx
 *   out      [batch, 24, 256] bf16 out; lse [batch, 24] float out or NULL
 *   idx_out  [batch, budget] int32 out or NULL: the selection used
 *   ws       at least qsa_decode_workspace_bytes(cfg, batch, max_ctx) bytes
 * Steps: block-key scan (scores and a lower bound of each sequence's
 * (budget-1)-th best score), candidate filter (at small batch it also brings
 * the candidates' K and V rows into L2), exact merge in block order, split
 * attention over the selected blocks, log-sum-exp combine.
 * Launch post, "Attention: GDN + QSA" (decode speed-up at 1M tokens is
 * quoted there); max_ctx <= 3,080,192.
 * ---------------------------------------------------------------------- */
size_t qsa_decode_workspace_bytes(const qsa_config *cfg, int batch, int64_t max_ctx);
qsa_status qsa_sparse_attn_decode(const qsa_config *cfg, int batch, const qsa_bf16 *q,
                                  const qsa_bf16 *qi, const qsa_bf16 *w,
                                  const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                  const qsa_bf16 *kblk_cache, int64_t max_ctx,
                                  const int32_t *seq_lens, qsa_bf16 *out, float *lse,
                                  int32_t *idx_out, void *ws, size_t ws_bytes,
                                  int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Decode without a workspace argument: the same computation as
 * qsa_sparse_attn_decode (same arguments minus ws / ws_bytes), for callers
 * that cannot allocate device memory when they run a decode step -- a C host
 * embedded in a process whose device memory is owned by another runtime, or
 * a serving loop that must not call cudaMalloc/cudaFree (they can
 * synchronise the device and fail under memory pressure mid-request).
 * The pages have no counterpart of this call; it is a property of this
 * library's interface only.
 *   - Scratch is a statically sized device array inside libqsa.so, 16 MiB,
 *     present on every GPU that loads the library until it is unloaded.
 *     batch x max_ctx combinations whose workspace
 *     (qsa_decode_workspace_bytes) exceeds it return QSA_ERR_UNSUPPORTED and
 *     launch nothing (8 x 1,048,576 fits, 12.1 MB; 64 x 262,144, 24.3 MB,
 *     does not).
 *   - Every call looks up the array's device address in the current
 *     context (cudaGetSymbolAddress: a lookup, not an allocation), so a
 *     cudaDeviceReset or a non-primary context is followed correctly.  The
 *     first call in a context may load the library's device code there:
 *     make it before any stream capture.
 *   - Arguments are checked as qsa_sparse_attn_decode checks them, with
 *     the same statuses (batch < 1: QSA_ERR_INVALID_ARG; max_ctx beyond
 *     3,080,192: QSA_ERR_UNSUPPORTED).
 *   - All calls share the array: calls whose GPU work overlaps (other
 *     streams, unordered host threads) race.  Nothing in it needs zeroing.
 *   - Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 * ---------------------------------------------------------------------- */
qsa_status qsa_sparse_attn_decode_noalloc(const qsa_config *cfg, int batch, const qsa_bf16 *q,
                                          const qsa_bf16 *qi, const qsa_bf16 *w,
                                          const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                          const qsa_bf16 *kblk_cache, int64_t max_ctx,
                                          const int32_t *seq_lens, qsa_bf16 *out, float *lse,
                                          int32_t *idx_out, int32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Self-test of the failure path: one kernel waits, with the library's bounded
 * mbarrier wait, on a phase that completes only if `complete` is nonzero.
 * With complete = 0 the wait runs out after limit_ns (1 ns .. 0.1 s) and the
 * kernel writes QSA_ERR_TIMEOUT to *dev_status and returns; with complete = 1
 * it leaves *dev_status untouched.  Every kernel of the library reports a
 * wait that ran out this way (their limit is 2 s).  Returns QSA_ERR_INVALID_ARG
 * for a NULL status or a limit out of range.  The pages have no counterpart.
 * ---------------------------------------------------------------------- */
qsa_status qsa_selftest_bounded_wait(int64_t limit_ns, int complete, int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
