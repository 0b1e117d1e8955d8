/*
 * bsa.h - C ABI of libbsa: radius-rescued block-sparse causal prefill
 * attention for GB300 (sm_103a).
 *
 * The method follows the article "Your 128K Context Is 6x Slower Than It
 * Needs to Be" (articles.phantom-byte.com), sections "Why block-sparse
 * attention underperforms: the mean-dilution trap" and "The rescue branch:
 * two selection paths, one mask".  Per (layer, KV head) a linear-time mask
 * build summarises every key block by its centroid and radius, derives a
 * radius-adaptive rescue coefficient from the median and 90th-percentile
 * radius, thresholds a centroid path and a rescue path independently and ORs
 * the two masks; FlashAttention-style attention with online softmax then runs
 * over the kept blocks only ("attention-kernel-optimization",
 * skill-vault.co.in, section "FlashAttention (1 -> 2 -> 3)").
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers into memory the caller owns; the
 *     library never allocates, frees or synchronises.  Every call is
 *     asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Tensors are dense, contiguous, row-major.  Q is [batch, seq, hq, d],
 *     K and V are [batch, seq, hkv, d], O is [batch, seq, hq, d], all bf16.
 *     Device pointers must be 16-byte aligned.
 *   - Notation: nb = seq / block key (and query) blocks; G = hq / hkv query
 *     heads per KV head; query head h reads KV head g = h / G.
 *   - Host-side argument errors are returned before anything is launched.
 *     A failed launch returns BSA_ERR_CUDA.
 *   - `dev_status` (nullable) is a device int32 the kernels set to a nonzero
 *     bsa_status when a bounded device-side wait gives up (the kernel then
 *     returns without hanging the GPU) or, for packed ragged batches, when a
 *     cu_seqlens entry is inconsistent.  The caller zeroes it and reads it
 *     after its own synchronisation.
 *   - NaN or Inf inputs give undefined (but memory-safe) results.
 */
#ifndef BSA_H_
#define BSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *bsa_stream_t;

typedef enum {
  BSA_OK = 0,
  BSA_ERR_INVALID_ARG = 1,    /* null pointer, misaligned pointer, bad ratio; also written to
                                 *dev_status for an inconsistent cu_seqlens entry */
  BSA_ERR_SHAPE = 2,          /* inconsistent shape (seq % block, hq % hkv, ...) */
  BSA_ERR_UNSUPPORTED = 3,    /* consistent but not implemented (head_dim, block, ...) */
  BSA_ERR_WORKSPACE = 4,      /* workspace missing or too small */
  BSA_ERR_CUDA = 5,           /* a CUDA runtime or driver call failed */
  BSA_ERR_DEVICE_TIMEOUT = 6  /* written to *dev_status by a kernel whose wait gave up */
} bsa_status;

/*
 * Problem shape.  Supported: head_dim in {64, 128}; block in {64, 128, 256};
 * seq % block == 0 with any block count 1 <= nb <= 4096; hq % hkv == 0 with
 * G in {1, 2, 4, 8, 16}; for block 64 the group size G must be even (two heads
 * share one 128-row query tile).
 */
typedef struct {
  int32_t batch, seq, hq, hkv, head_dim, block;
} bsa_shape;

/*
 * Selection parameters (rescue branch section: each of the two paths has its
 * own threshold).  Each path keeps a fraction of the causal row:
 * query block i keeps ceil(ratio * (i + 1)) candidates on each path, computed
 * as (ppm * (i + 1) + 999999) / 1000000 with ppm = floor(ratio * 1e6 + 0.5),
 * clipped to the available candidates.  Ratios must lie in [0, 1].
 * flags: 0 or BSA_SELECT_TOKEN_MAX.
 */
typedef struct {
  float centroid_keep;
  float rescue_keep;
  int32_t flags;
} bsa_select_params;

/*
 * BSA_SELECT_TOKEN_MAX - per-token query aggregation.  The article's selector
 * summarises a query block by its mean query; with this flag a query block is
 * represented by its best single token instead ("The numbers, stated honestly"
 * section: the comparison is between tokens and centroids, done as a tiled
 * reduction so no tokens x blocks tensor is stored):
 *   S_c[i][j] = s * max over the G heads and the tokens t of block i of q_t . c_j
 *   R[i][j]   = s * max over the same (h, t) of (q_t . c_j + alpha_j * |q_t| * r_j)
 * With alpha_j = 1, R bounds every logit of block j.  Ranking, keep counts and
 * outputs are unchanged.  The dot products run on tensor cores with the
 * centroids split into bf16 hi + lo (about 16 significant bits).
 */
#define BSA_SELECT_TOKEN_MAX 1

/* Bits of the optional mask written by bsa_select_mask. */
#define BSA_MASK_FORCED 1u    /* key block 0 or the diagonal block */
#define BSA_MASK_CENTROID 2u  /* kept by the centroid path */
#define BSA_MASK_RESCUE 4u    /* kept by the rescue path */

/*
 * bsa_block_meta - key-block summaries and the rescue coefficient.
 *
 * Rescue branch section: every key block is summarised by its centroid and by
 * the largest distance from one of its keys to that centroid; the rescue
 * coefficient adapts to the distribution of those radii, anchored at their
 * median and 90th percentile, taken per layer and per KV head.
 *
 *   centroid[b][g][j][x]  (fp32, [batch, hkv, nb, head_dim])
 *                         = mean over the block's keys of k[x]          (reading 1)
 *   radius[b][g][j]       = max over the block's keys of |k - centroid|_2 (reading 2)
 *   quant[b][g][0..1]     = median and 90th percentile of radius[b][g][:],
 *                           nearest rank: r_(ceil(p * nb)) of the ascending sort
 *                                                                       (reading 4)
 *   alpha[b][g][j]        = clamp((r_j - med) / (p90 - med), 0, 1), or 0 for
 *                           all j when p90 - med <= 1e-12 * p90          (reading 5)
 * All outputs fp32, caller-allocated.  k: bf16 [batch, seq, hkv, head_dim].
 */
bsa_status bsa_block_meta(const bsa_shape *shape, const void *k, float *centroid, float *radius,
                          float *quant, float *alpha, int32_t *dev_status, bsa_stream_t stream);

/*
 * bsa_select_mask - score every causal key block and emit the kept lists.
 *
 * Rescue branch section: one path ranks the key blocks by their mean-based
 * score and keeps the best; a second path restores blocks with a large radius
 * that this ranking leaves out; the union of the two is kept.  With s = 1/sqrt(head_dim), qbar_{h,i} the mean query of block i
 * for head h and nbar_{h,i} the mean of those queries' L2 norms:
 *   S_c[i][j] = max over the G heads of KV head g of s * qbar_{h,i}.c_j
 *   R[i][j]   = max over those heads of s * (qbar_{h,i}.c_j + alpha_j * nbar_{h,i} * r_j)
 * (readings 6 to 8).  Row i keeps blocks 0 and i (forced, outside both
 * rankings; reading 9), the top ceil(centroid_keep * (i+1)) of 1..i-1 by S_c
 * (readings 10, 11), and the top ceil(rescue_keep * (i+1)) by R of the
 * candidates the centroid path dropped whose alpha_j > 0 (reading 12).  Ties
 * go to the lower block index; the kept set is the union (reading 13).
 *
 * Outputs: kv_idx[b][g][i][0..kv_cnt-1] (int32, [batch, hkv, nb, nb]) holds the
 * kept key blocks of row i in ascending order; entries past kv_cnt are left
 * unspecified.  kv_cnt[b][g][i] (int32, [batch, hkv, nb]).  mask (nullable,
 * uint8 [batch, hkv, nb, nb]) receives the BSA_MASK_* bits of every (i, j).
 * q: bf16 [batch, seq, hq, head_dim]; centroid, radius, alpha as written by
 * bsa_block_meta.  workspace: device scratch of at least
 * bsa_select_workspace_bytes(shape) bytes, 16-byte aligned, owned by the
 * caller (it holds the per-block mean queries and mean query norms, tf32
 * hi / lo splits of the mean queries and centroids, and the two block-score
 * matrices; its contents need no initialisation and are dead after the call's
 * kernels finish).  dev_status (nullable) receives
 * BSA_ERR_DEVICE_TIMEOUT if the score kernel's bounded waits give up.
 */
size_t bsa_select_workspace_bytes(const bsa_shape *shape);
bsa_status bsa_select_mask(const bsa_shape *shape, const bsa_select_params *params, const void *q,
                           const float *centroid, const float *radius, const float *alpha,
                           int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream);

/*
 * bsa_select_mask_noalloc - bsa_select_mask without a caller-provided workspace.
 *
 * The article has no counterpart to this call; it is a library convenience for
 * callers that cannot allocate device memory, such as a host framework that
 * owns the whole device pool and forbids allocations outside it, or a
 * latency-critical caller that must not call cudaMalloc because it can
 * synchronise the device.  The call computes exactly what bsa_select_mask
 * computes (same kernels, same outputs, both query aggregations: flags 0 or
 * BSA_SELECT_TOKEN_MAX), with its scratch in a fixed 12 MiB array inside the
 * library's device image, so it allocates nothing.
 *   - Every GPU that loads libbsa keeps those 12 MiB until the process exits.
 *   - Shapes needing more than 12 MiB of select scratch
 *     (bsa_select_workspace_bytes(shape) > 12 MiB: at 32 query heads,
 *     4 KV heads, head_dim 128 and block 128 that is beyond 35072 tokens;
 *     the 65536- and 131072-token layers need 27.3 MB and 71.4 MB) return
 *     BSA_ERR_WORKSPACE before anything is launched.
 *   - All calls on one device share that array: calls whose kernels overlap on
 *     the GPU (unordered streams) race and give wrong results.  Calls ordered
 *     on one stream are safe.  Nothing in it needs to start at zero.
 *   - The first call on a device, and the first call after that device's
 *     context was reset, looks up the array's device address with that device
 *     current; make that first call before any stream capture.
 * Errors: shape errors as bsa_select_mask, then BSA_ERR_WORKSPACE for shapes
 * beyond the array, then the parameter, pointer and launch errors of
 * bsa_select_mask.  dev_status receives BSA_ERR_DEVICE_TIMEOUT if the score
 * kernels' bounded waits give up.
 */
bsa_status bsa_select_mask_noalloc(const bsa_shape *shape, const bsa_select_params *params,
                                   const void *q, const float *centroid, const float *radius,
                                   const float *alpha, int32_t *kv_idx, int32_t *kv_cnt,
                                   uint8_t *mask, int32_t *dev_status, bsa_stream_t stream);

/*
 * bsa_mask_build - bsa_block_meta followed by bsa_select_mask, in fewer launches.
 *
 * Rescue branch section, the whole mask construction of one layer: the same
 * centroid, radius, quant, alpha, kv_idx, kv_cnt and (nullable) mask as the
 * two calls made one after the other on `stream` with the same arguments, bit
 * for bit.  The key-block summaries and the query-block means are computed in
 * one launch that streams K and Q together, and the quantiles are taken inside
 * it, so the build costs three kernels instead of five.
 * params->flags must be 0 (block-mean queries; per-token aggregation goes
 * through bsa_block_meta and bsa_select_mask).  q: bf16 [batch, seq, hq,
 * head_dim]; k: bf16 [batch, seq, hkv, head_dim]; every output as documented
 * for the two calls, caller-allocated, 16-byte aligned.  workspace: device
 * scratch of at least bsa_mask_build_workspace_bytes(shape) bytes, 16-byte
 * aligned, owned by the caller; its contents need no initialisation (the call
 * zeroes the counters it keeps there) and are dead once the call's kernels
 * finish.  Errors: shape errors, then parameter and pointer errors
 * (BSA_ERR_INVALID_ARG), then BSA_ERR_WORKSPACE, all before any launch;
 * BSA_ERR_CUDA if a launch fails.  dev_status as bsa_select_mask.
 */
size_t bsa_mask_build_workspace_bytes(const bsa_shape *shape);
bsa_status bsa_mask_build(const bsa_shape *shape, const bsa_select_params *params, const void *q,
                          const void *k, float *centroid, float *radius, float *quant, float *alpha,
                          int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, void *workspace,
                          size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream);

/*
 * bsa_prefill_fwd - causal attention over the kept key blocks.
 *
 * Rescue branch section: the combined mask is consumed by an ordinary
 * block-sparse FlashAttention.  For every query token t of block i and head h:
 *   O[t][h] = sum_s softmax_s(scale * q_t . k_s) v_s,  over the tokens s <= t
 *             of the key blocks kv_idx[b][g][i][0..kv_cnt-1], g = h / G;
 *   lse[b][h][t] = natural log of that softmax's normaliser (fp32, nullable).
 * kv_idx rows must be strictly ascending, in [0, i], and contain i; block 0
 * need not be present.  Tiled online softmax gives the explicit softmax's
 * result up to rounding.  o: bf16 [batch, seq, hq, head_dim].
 */
bsa_status bsa_prefill_fwd(const bsa_shape *shape, const void *q, const void *k, const void *v,
                           const int32_t *kv_idx, const int32_t *kv_cnt, float softmax_scale,
                           void *o, float *lse, int32_t *dev_status, bsa_stream_t stream);

/*
 * bsa_prefill_dense_fwd - the same kernel with every causal block kept
 * (the dense baseline every speedup in the article is normalised against).
 */
bsa_status bsa_prefill_dense_fwd(const bsa_shape *shape, const void *q, const void *k,
                                 const void *v, float softmax_scale, void *o, float *lse,
                                 int32_t *dev_status, bsa_stream_t stream);

/*
 * bsa_prefill_layer - one whole layer of the hot path in one call:
 * bsa_mask_build (bsa_block_meta then bsa_select_mask when params->flags is
 * BSA_SELECT_TOKEN_MAX), then bsa_prefill_fwd, all on `stream`.
 * The intermediate tensors live in `workspace` (device, 256-byte aligned, at
 * least bsa_prefill_layer_workspace_bytes(shape) bytes): centroid, radius,
 * quant, alpha, kv_idx, kv_cnt and the mask build scratch.  bsa_prefill_layer_views
 * gives the offsets of the first six.
 */
size_t bsa_prefill_layer_workspace_bytes(const bsa_shape *shape);
bsa_status bsa_prefill_layer(const bsa_shape *shape, const bsa_select_params *params,
                             const void *q, const void *k, const void *v, float softmax_scale,
                             void *o, float *lse, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, bsa_stream_t stream);

/*
 * Byte offsets inside the bsa_prefill_layer workspace of: centroid, radius,
 * quant, alpha, kv_idx, kv_cnt (in that order, 6 entries written to offsets).
 */
bsa_status bsa_prefill_layer_views(const bsa_shape *shape, size_t *offsets);

/* ------------------------------------------------------------------------
 * FP8 (e4m3) inputs.
 *
 * The article's measurements use 8-bit weights and keys (prefill section),
 * and it reports that the radius signal still works with 8-bit keys.
 * These entry points take Q, K and V as OCP e4m3 codes (1 byte per element,
 * same [batch, seq, heads, head_dim] layouts) with one positive scale per
 * tensor: value = e4m3(code) * scale.  They compute exactly what the bf16
 * entry points compute on the dequantised values:
 *   - bsa_block_meta_fp8: centroids, radii, quantiles, alpha of k * k_scale;
 *   - bsa_select_mask_fp8: the selection with q * q_scale (flags must be 0:
 *     BSA_SELECT_TOKEN_MAX returns BSA_ERR_UNSUPPORTED here);
 *   - bsa_prefill_fwd_fp8 / bsa_prefill_dense_fwd_fp8: attention with
 *     S = Q K^T on the tensor cores' e4m3 path (kind::f8f6f4); V is first
 *     widened to bf16 codes of the same values (exact) in the workspace
 *     (bsa_prefill_fp8_workspace_bytes(shape) bytes, 16-byte aligned, owned
 *     by the caller, dead after the call's kernels); O written as bf16;
 *     head_dim 128 only (other head_dims return BSA_ERR_UNSUPPORTED, and the
 *     workspace size function returns 0 for them).
 * Scales must be finite and positive (BSA_ERR_INVALID_ARG otherwise).  Other
 * arguments, layouts and errors as the bf16 entry points.
 * ------------------------------------------------------------------------ */
size_t bsa_prefill_fp8_workspace_bytes(const bsa_shape *shape);
bsa_status bsa_block_meta_fp8(const bsa_shape *shape, const void *k, float k_scale, float *centroid,
                              float *radius, float *quant, float *alpha, int32_t *dev_status,
                              bsa_stream_t stream);
bsa_status bsa_select_mask_fp8(const bsa_shape *shape, const bsa_select_params *params,
                               const void *q, float q_scale, const float *centroid,
                               const float *radius, const float *alpha, int32_t *kv_idx,
                               int32_t *kv_cnt, uint8_t *mask, void *workspace,
                               size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream);
bsa_status bsa_prefill_fwd_fp8(const bsa_shape *shape, const void *q, const void *k, const void *v,
                               float q_scale, float k_scale, float v_scale, const int32_t *kv_idx,
                               const int32_t *kv_cnt, float softmax_scale, void *o, float *lse,
                               void *workspace, size_t workspace_bytes, int32_t *dev_status,
                               bsa_stream_t stream);
bsa_status bsa_prefill_dense_fwd_fp8(const bsa_shape *shape, const void *q, const void *k,
                                     const void *v, float q_scale, float k_scale, float v_scale,
                                     float softmax_scale, void *o, float *lse, void *workspace,
                                     size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Packed ragged batches ("varlen").
 *
 * Serving batches mix prompt lengths (the article's prefill section measures
 * single long prompts; nothing in the method depends on a common length).  A
 * varlen batch packs its sequences along one token axis: sequence b is tokens
 * cu_seqlens[b] .. cu_seqlens[b+1]-1 of q [total_tokens, hq, head_dim] and of
 * k, v [total_tokens, hkv, head_dim]; o is [total_tokens, hq, head_dim] and
 * lse is [hq, total_tokens].  A sequence may have any length >= 0, not only a
 * multiple of the block: its blocks are nb_b = ceil(len_b / block) and the
 * last one holds the remaining len_b - (nb_b - 1) * block tokens, which is
 * then summarised, ranked and attended over those tokens only.  Every
 * sequence is processed exactly as a batch of one.
 *
 * cu_seqlens: DEVICE int32 [batch + 1], 4-byte aligned, with cu_seqlens[0] =
 * 0, non-decreasing, cu_seqlens[batch] <= total_tokens and every length <=
 * max_seqlen.  The host cannot read it without synchronising, so the kernels
 * check each entry: an inconsistent sequence writes BSA_ERR_INVALID_ARG to
 * *dev_status (when given), is treated as empty, and nothing outside the
 * caller's buffers is touched.
 *
 * Per-block arrays use nbs = bsa_varlen_block_stride(shape) =
 * ceil(ceil(max_seqlen / block) / 4) * 4 blocks per sequence:
 *   centroid [batch, hkv, nbs, head_dim], radius and alpha [batch, hkv, nbs],
 *   quant [batch, hkv, 2], kv_idx [batch, hkv, nbs, nbs], kv_cnt [batch, hkv,
 *   nbs], mask [batch, hkv, nbs, nbs].
 * Entries past a sequence's own nb_b blocks are written as zeros (kv_cnt 0);
 * an empty sequence gets quant 0.  Supported head_dim, block and group sizes
 * are those of bsa_shape; ceil(max_seqlen / block) <= 4096.
 * ------------------------------------------------------------------------ */
typedef struct {
  int32_t batch;         /* number of sequences */
  int32_t total_tokens;  /* rows of the packed q, k, v, o (>= 1) */
  int32_t max_seqlen;    /* upper bound of every sequence length (>= 1, <= total_tokens) */
  int32_t hq, hkv, head_dim, block;
} bsa_varlen_shape;

/* nbs of the layouts above, or 0 for an invalid shape. */
int32_t bsa_varlen_block_stride(const bsa_varlen_shape *shape);

/* bsa_block_meta for a packed batch; partial last blocks average their own keys. */
bsa_status bsa_varlen_block_meta(const bsa_varlen_shape *shape, const int32_t *cu_seqlens,
                                 const void *k, float *centroid, float *radius, float *quant,
                                 float *alpha, int32_t *dev_status, bsa_stream_t stream);

/* bsa_select_workspace_bytes / bsa_select_mask for a packed batch: rows i < nb_b of each
 * sequence, keep counts from i + 1 as for a fixed-length sequence. */
size_t bsa_varlen_select_workspace_bytes(const bsa_varlen_shape *shape);
bsa_status bsa_varlen_select_mask(const bsa_varlen_shape *shape, const bsa_select_params *params,
                                  const int32_t *cu_seqlens, const void *q, const float *centroid,
                                  const float *radius, const float *alpha, int32_t *kv_idx,
                                  int32_t *kv_cnt, uint8_t *mask, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status,
                                  bsa_stream_t stream);

/* bsa_prefill_fwd / bsa_prefill_dense_fwd for a packed batch: causal within each sequence;
 * the rows of a partial last block past the sequence end are not written. */
bsa_status bsa_varlen_prefill_fwd(const bsa_varlen_shape *shape, const int32_t *cu_seqlens,
                                  const void *q, const void *k, const void *v,
                                  const int32_t *kv_idx, const int32_t *kv_cnt,
                                  float softmax_scale, void *o, float *lse, int32_t *dev_status,
                                  bsa_stream_t stream);
bsa_status bsa_varlen_prefill_dense_fwd(const bsa_varlen_shape *shape, const int32_t *cu_seqlens,
                                        const void *q, const void *k, const void *v,
                                        float softmax_scale, void *o, float *lse,
                                        int32_t *dev_status, bsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Decode: one new token per sequence (q_len = 1) over a packed cache.
 *
 * The cache of sequence b is tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 of the
 * packed k, v [total_tokens, hkv, head_dim] (varlen layout above); its last
 * token is the new one, already appended, so the new query sits at position
 * len_b - 1 and its row is block i = (len_b - 1) / block.  q_new is bf16
 * [batch, hq, head_dim]; centroid, radius and alpha are those of the cache
 * (bsa_varlen_block_meta on it; a block's summary only matters once the block
 * is complete, since the current block is always kept).
 *
 * bsa_decode_select: the selection of a prefill row for a one-token query
 * block (rescue branch section): scores of the G heads of the new token
 * against the centroids of blocks 1..i-1, S_c = s max_h q_h . c_j and
 * R = s max_h (q_h . c_j + alpha_j |q_h| r_j), forced blocks 0 and i, keep
 * counts from i + 1.  Writes the ascending kept list kv_idx [batch, hkv, nbs]
 * (int32) and kv_cnt [batch, hkv].  params.flags must be 0.  workspace: as
 * for bsa_decode_fwd (the same buffer may serve both calls on one stream).
 *
 * bsa_decode_fwd: attention of the new token over the kept blocks' tokens,
 * split over the kept blocks (a split-KV kernel: decode is bound by memory
 * traffic, and splitting keeps the whole GPU busy at small batch; section on
 * decode in "Your Context Length Decides What a Kernel Is Worth").  o: bf16
 * [batch, hq, head_dim]; lse (nullable) fp32 [batch, hq]; workspace of
 * bsa_decode_workspace_bytes(shape) bytes, 16-byte aligned, for the fp32
 * partial results.  An empty sequence gets o = 0 and lse = -inf.  The kept
 * entries of all rows (b, g) are spread evenly over the GPU's CTAs; batch *
 * hkv above 4096 returns BSA_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------ */
size_t bsa_decode_workspace_bytes(const bsa_varlen_shape *shape);
bsa_status bsa_decode_select(const bsa_varlen_shape *shape, const bsa_select_params *params,
                             const int32_t *cu_seqlens, const void *q_new, const float *centroid,
                             const float *radius, const float *alpha, int32_t *kv_idx,
                             int32_t *kv_cnt, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, bsa_stream_t stream);
bsa_status bsa_decode_fwd(const bsa_varlen_shape *shape, const int32_t *cu_seqlens,
                          const void *q_new, const void *k, const void *v, const int32_t *kv_idx,
                          const int32_t *kv_cnt, float softmax_scale, void *o, float *lse,
                          void *workspace, size_t workspace_bytes, int32_t *dev_status,
                          bsa_stream_t stream);

/*
 * bsa_decode_step - bsa_decode_select followed by bsa_decode_fwd, in one launch.
 *
 * The same selection (kv_idx, kv_cnt written as bsa_decode_select writes them)
 * and the same attention of the new token (o, lse) as the two calls on one
 * stream with the same arguments.  A decode step is a few microseconds of work
 * per phase, so it runs as one cooperative launch whose CTAs are all resident:
 * scores | selection | split-KV attention | merge of the partial results, with
 * a grid-wide barrier between the phases (bounded: a barrier that does not
 * complete within 2 s records BSA_ERR_DEVICE_TIMEOUT in dev_status).  The
 * selection and the partial attention results are those of the two calls; the
 * merge adds the partials in the same order, but the partials themselves
 * depend on how many CTAs the launch has, so O may differ from the two calls
 * in the last bits.  workspace: bsa_decode_workspace_bytes(shape) bytes,
 * 16-byte aligned (it includes the barrier words, which the call zeroes).
 * Errors: shape errors, then the parameter and pointer errors of the two calls
 * (BSA_ERR_INVALID_ARG), BSA_ERR_UNSUPPORTED for batch * hkv above 4096, then
 * BSA_ERR_WORKSPACE, all before any launch; BSA_ERR_CUDA if the launch fails.
 */
bsa_status bsa_decode_step(const bsa_varlen_shape *shape, const bsa_select_params *params,
                           const int32_t *cu_seqlens, const void *q_new, const void *k, const void *v,
                           const float *centroid, const float *radius, const float *alpha,
                           float softmax_scale, int32_t *kv_idx, int32_t *kv_cnt, void *o, float *lse,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           bsa_stream_t stream);

/* ------------------------------------------------------------------------
 * Self-test of the device wait limits (no compute).  Launches `ctas` CTAs
 * (1..8) whose first thread waits, through the bounded wait the attention
 * kernel uses, on an mbarrier that nothing completes.  CTA 0 gives up after
 * limit_ns nanoseconds (1e6 .. 1e9) and writes BSA_ERR_DEVICE_TIMEOUT into
 * *dev_status (int32, caller-owned, 4-byte aligned, 0 before the call); the
 * other CTAs wait with the library's own 4 s limit and stop as soon as they
 * see the status.  Returns BSA_ERR_INVALID_ARG for a null or misaligned
 * status word or out-of-range arguments, BSA_ERR_CUDA if the launch fails.
 * ------------------------------------------------------------------------ */
bsa_status bsa_selftest_wait_timeout(int32_t *dev_status, uint64_t limit_ns, int32_t ctas,
                                     bsa_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *bsa_status_string(bsa_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t bsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H_ */
