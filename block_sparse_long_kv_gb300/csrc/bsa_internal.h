// Internal declarations shared by the libbsa translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsa.h"

namespace bsa {

constexpr int kMaxBlocks = 4096;  // nb limit (select kernel keeps one score row in smem)
constexpr int kMaxDecodeRows = 4096;  // batch * hkv limit of decode (its plan sits in smem)

// A batch is either fixed-length (cu == nullptr: sequence b is tokens
// b*seq .. b*seq+seq-1) or packed ragged (sequence b is tokens cu[b] ..
// cu[b+1]-1 of `total`, each at most `seq` = max_seqlen long).  nb is the
// largest block count of a sequence, nbs the per-sequence stride of every
// caller-visible per-block array (equal to nb when fixed-length, nb rounded up
// to a multiple of 4 when packed), nbw the row stride of the block-score
// matrices in the select workspace (nbs rounded up to a multiple of 4, so
// every score row starts on a 16-byte boundary).
struct MaskShape {
  int batch, seq, hq, hkv, d, block, nb, group;
  const int32_t *cu;
  int total, nbs;
  int fp8;                          // inputs are e4m3 codes: value = code * scale
  float q_scale, k_scale, v_scale;  // used when fp8
  int nbw;
};

__host__ __device__ constexpr int round4(int x) { return (x + 3) / 4 * 4; }

// Token span of sequence b.  Packed entries are checked against total and
// max_seqlen: an inconsistent one records BSA_ERR_INVALID_ARG (if status is
// set) and reads as an empty sequence, so no kernel touches memory outside
// the caller's buffers.
struct SeqSpan {
  int start, len;
};

__device__ __forceinline__ SeqSpan seq_span(const int32_t *cu, int b, int seq, int total,
                                            int32_t *status) {
  if (cu == nullptr) return SeqSpan{b * seq, seq};
  const int s0 = __ldg(cu + b), s1 = __ldg(cu + b + 1);
  if (s0 < 0 || s1 < s0 || s1 > total || s1 - s0 > seq) {
    if (status != nullptr) atomicCAS(status, 0, static_cast<int32_t>(BSA_ERR_INVALID_ARG));
    return SeqSpan{0, 0};
  }
  return SeqSpan{s0, s1 - s0};
}

// Block meta: centroid [b, hkv, nbs, d], radius [b, hkv, nbs] (zero past a sequence's blocks).
cudaError_t launch_block_meta(const MaskShape &s, const void *k, float *centroid, float *radius,
                              int32_t *status, cudaStream_t stream);
// Quantiles [b, hkv, 2] and alpha [b, hkv, nbs] from radius.
cudaError_t launch_quantiles(const MaskShape &s, const float *radius, float *quant, float *alpha,
                             int32_t *status, cudaStream_t stream);
// Bytes of select workspace: tf32 splits of the mean queries [b, hkv, nbs, G, d] and of the
// centroids [b, hkv, nbs, d], mean query norms [b, hkv, nbs, G] and the two score matrices
// [b, hkv, nbs, nbs], all fp32.
size_t select_workspace_bytes(const MaskShape &s);
// Query pooling into the workspace, tensor-core block scores, then top-k + list emission;
// token_max scores every query token instead of the block-mean query.
cudaError_t launch_select(const MaskShape &s, const void *q, const float *centroid,
                          const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                          float scale, bool token_max, int32_t *kv_idx, int32_t *kv_cnt,
                          uint8_t *mask, void *workspace, int32_t *status, cudaStream_t stream);

// The layer path's mask build: key-block meta and query pooling in one launch
// (the quantiles taken by each KV group's last meta CTA), then the scores and the
// selection; `done` holds layer_mask_counter_bytes(s) of counters, zeroed here.
size_t layer_mask_counter_bytes(const MaskShape &s);
cudaError_t launch_layer_mask(const MaskShape &s, const void *q, const void *k, float *centroid, float *radius,
                              float *quant, float *alpha, int64_t ppm_c, int64_t ppm_r, float scale,
                              int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, void *workspace, unsigned *done,
                              int32_t *status, cudaStream_t stream);

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry point.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder(cudaError_t *err);

// Operands of the score GEMM: tf32 hi / lo splits of the centroids [b, hkv, nb, d] and of
// the mean queries [b, hkv, nb, G, d], mean query norms [b, hkv, nb, G], radius, alpha.
struct ScoreOperands {
  const float *c_hi, *c_lo, *q_hi, *q_lo, *nbar, *radius, *alpha;
};
// Block scores S_c and R ([b, hkv, nb, nb] fp32, rows i, columns j < i) on tensor cores.
cudaError_t launch_scores(const MaskShape &s, const ScoreOperands &op, float scale, float *s_c,
                          float *s_r, int32_t *status, cudaStream_t stream);

// Per-token aggregation of the same scores (flag BSA_SELECT_TOKEN_MAX): splits the centroids
// into bf16 hi / lo in c16 (2 * b * hkv * nbs * d bf16) and reduces q . c over every token of
// each query block on tensor cores.
cudaError_t launch_token_scores(const MaskShape &s, const void *q, const float *centroid, void *c16,
                                const float *radius, const float *alpha, float scale, float *s_c,
                                float *s_r, int32_t *status, cudaStream_t stream);

// Decode of one new token per packed sequence (its cache's last token): selection of the
// kept blocks (kv_idx [b, hkv, nbs], kv_cnt [b, hkv]) and split-KV attention (o [b, hq, d],
// lse [b, hq]) with fp32 partials in the workspace.
cudaError_t launch_decode_select(const MaskShape &s, const void *q_new, const float *centroid,
                                 const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                                 float scale, int32_t *kv_idx, int32_t *kv_cnt, void *workspace,
                                 int32_t *status, cudaStream_t stream);
size_t decode_workspace_bytes(const MaskShape &s);
cudaError_t launch_decode(const MaskShape &s, const void *q_new, const void *k, const void *v,
                          const int32_t *kv_idx, const int32_t *kv_cnt, float scale, void *o, float *lse,
                          void *workspace, int32_t *status, cudaStream_t stream);
// bsa_decode_select then bsa_decode_fwd in one cooperative launch (grid barriers between the
// phases; the barrier words in the decode workspace are zeroed here).
cudaError_t launch_decode_step(const MaskShape &s, const void *q_new, const void *k, const void *v,
                               const float *centroid, const float *radius, const float *alpha, int64_t ppm_c,
                               int64_t ppm_r, float select_scale, float softmax_scale, int32_t *kv_idx,
                               int32_t *kv_cnt, void *o, float *lse, void *workspace, int32_t *status,
                               cudaStream_t stream);

// e4m3 codes -> bf16 codes of the same values; n elements, a multiple of 16.
cudaError_t launch_widen_e4m3(const void *src, void *dst, size_t n, cudaStream_t stream);

struct AttnShape {
  int batch, seq, hq, hkv, d, block, nb, group;
  const int32_t *cu;  // packed ragged batch (o [total, hq, d], lse [hq, total]) or null
  int total, nbs;
  int fp8;                          // q, k, v are e4m3 codes (value = code * scale)
  float q_scale, k_scale, v_scale;  // used when fp8
};

// Sparse (kv_idx != nullptr) or dense (kv_idx == nullptr) causal attention.
// Returns BSA_OK or an error code; `cuda_err` receives the CUDA error if any.
bsa_status launch_attention(const AttnShape &s, const void *q, const void *k, const void *v,
                            const int32_t *kv_idx, const int32_t *kv_cnt, float scale, void *o,
                            float *lse, int32_t *dev_status, cudaStream_t stream,
                            cudaError_t *cuda_err);

}  // namespace bsa
