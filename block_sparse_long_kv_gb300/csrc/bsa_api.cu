// libbsa C ABI: argument validation and dispatch.  Every check runs on the
// host before anything is launched; the library never allocates, frees or
// synchronises.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "bsa.h"
#include "bsa_internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by the fixed-length and the packed ragged shapes; nb is the
// largest number of blocks of one sequence.
bsa_status check_common(int batch, int hq, int hkv, int head_dim, int block, int nb) {
  if (hq % hkv != 0) return BSA_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return BSA_ERR_UNSUPPORTED;
  if (block != 64 && block != 128 && block != 256) return BSA_ERR_UNSUPPORTED;
  if (nb > bsa::kMaxBlocks) return BSA_ERR_UNSUPPORTED;
  const long long grp = hq / hkv;
  if (grp != 1 && grp != 2 && grp != 4 && grp != 8 && grp != 16) return BSA_ERR_UNSUPPORTED;
  if (block == 64 && grp % 2 != 0) return BSA_ERR_UNSUPPORTED;
  // grid extents of the widest launch (attention: one CTA per query tile pair)
  const long long items = static_cast<long long>(nb) * batch * hq;
  if (items > (1ll << 30)) return BSA_ERR_UNSUPPORTED;
  return BSA_OK;
}

bsa_status check_shape(const bsa_shape *s) {
  if (s == nullptr) return BSA_ERR_INVALID_ARG;
  if (s->batch < 1 || s->seq < 1 || s->hq < 1 || s->hkv < 1 || s->head_dim < 1 || s->block < 1)
    return BSA_ERR_SHAPE;
  if (s->seq % s->block != 0) return BSA_ERR_SHAPE;
  if (static_cast<long long>(s->batch) * s->seq > INT32_MAX) return BSA_ERR_UNSUPPORTED;
  const int nb = s->seq / s->block;
  return check_common(s->batch, s->hq, s->hkv, s->head_dim, s->block, nb);
}

bsa_status check_varlen(const bsa_varlen_shape *s, const int32_t *cu_seqlens) {
  if (s == nullptr || cu_seqlens == nullptr) return BSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return BSA_ERR_INVALID_ARG;
  if (s->batch < 1 || s->total_tokens < 1 || s->max_seqlen < 1 || s->hq < 1 || s->hkv < 1 ||
      s->head_dim < 1 || s->block < 1)
    return BSA_ERR_SHAPE;
  if (s->max_seqlen > s->total_tokens) return BSA_ERR_SHAPE;
  const long long nb = (static_cast<long long>(s->max_seqlen) + s->block - 1) / s->block;
  if (nb > bsa::kMaxBlocks) return BSA_ERR_UNSUPPORTED;
  return check_common(s->batch, s->hq, s->hkv, s->head_dim, s->block, static_cast<int>(nb));
}

bsa::MaskShape mask_shape(const bsa_shape *s) {
  const int nb = s->seq / s->block;
  return bsa::MaskShape{s->batch, s->seq, s->hq, s->hkv, s->head_dim, s->block,
                        nb, s->hq / s->hkv, nullptr, s->batch * s->seq, nb,
                        0, 1.f, 1.f, 1.f, bsa::round4(nb)};
}

int varlen_blocks(const bsa_varlen_shape *s) { return (s->max_seqlen + s->block - 1) / s->block; }

int varlen_stride(const bsa_varlen_shape *s) { return (varlen_blocks(s) + 3) / 4 * 4; }

bsa::MaskShape mask_shape(const bsa_varlen_shape *s, const int32_t *cu) {
  return bsa::MaskShape{s->batch, s->max_seqlen, s->hq, s->hkv, s->head_dim, s->block,
                        varlen_blocks(s), s->hq / s->hkv, cu, s->total_tokens, varlen_stride(s),
                        0, 1.f, 1.f, 1.f, varlen_stride(s)};
}

bsa::AttnShape attn_shape(const bsa::MaskShape &m) {
  return bsa::AttnShape{m.batch, m.seq, m.hq, m.hkv, m.d, m.block, m.nb, m.group, m.cu, m.total, m.nbs,
                        m.fp8, m.q_scale, m.k_scale, m.v_scale};
}

bool scale_ok(float x) { return x > 0.f && !isinf(x); }  // false for NaN

bsa::MaskShape fp8_shape(const bsa_shape *s, float q_scale, float k_scale, float v_scale) {
  bsa::MaskShape m = mask_shape(s);
  m.fp8 = 1;
  m.q_scale = q_scale;
  m.k_scale = k_scale;
  m.v_scale = v_scale;
  return m;
}

bool ratio_ok(float r) { return r >= 0.f && r <= 1.f; }  // false for NaN

int64_t ratio_ppm(float r) { return static_cast<int64_t>(floor(static_cast<double>(r) * 1e6 + 0.5)); }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace of bsa_mask_build: the select scratch, then the per-(b, g)
// counters of the fused launch.
size_t mask_build_bytes(const bsa::MaskShape &m, size_t *counters_at) {
  const size_t at = round_up(bsa::select_workspace_bytes(m), 256);
  if (counters_at) *counters_at = at;
  return at + bsa::layer_mask_counter_bytes(m);
}

// Workspace layout of bsa_prefill_layer: centroid, radius, quant, alpha,
// kv_idx, kv_cnt, the mask build's workspace, each 256-byte aligned.
constexpr int kLayerRegions = 7;
void layer_views(const bsa::MaskShape &m, size_t off[kLayerRegions], size_t *total) {
  const size_t b = m.batch, h = m.hkv, d = m.d, nb = m.nbs;
  const size_t sizes[kLayerRegions] = {b * h * d * nb * 4, b * h * nb * 4,      b * h * 2 * 4, b * h * nb * 4,
                                       b * h * nb * nb * 4, b * h * nb * 4, mask_build_bytes(m, nullptr)};
  size_t cur = 0;
  for (int x = 0; x < kLayerRegions; ++x) {
    off[x] = cur;
    cur = round_up(cur + sizes[x], 256);
  }
  *total = cur;
}

bsa_status meta_impl(const bsa::MaskShape &ms, const void *k, float *centroid, float *radius,
                     float *quant, float *alpha, int32_t *dev_status, bsa_stream_t stream) {
  if (!k || !centroid || !radius || !quant || !alpha) return BSA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(centroid) || !aligned16(radius) || !aligned16(quant) ||
      !aligned16(alpha))
    return BSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (bsa::launch_block_meta(ms, k, centroid, radius, dev_status, s) != cudaSuccess) return BSA_ERR_CUDA;
  if (bsa::launch_quantiles(ms, radius, quant, alpha, dev_status, s) != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
}

bsa_status select_impl(const bsa::MaskShape &ms, const bsa_select_params *params, const void *q,
                       const float *centroid, const float *radius, const float *alpha,
                       int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, void *workspace,
                       size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream) {
  if (!params || !q || !centroid || !radius || !alpha || !kv_idx || !kv_cnt)
    return BSA_ERR_INVALID_ARG;
  if (!ratio_ok(params->centroid_keep) || !ratio_ok(params->rescue_keep) ||
      (params->flags & ~static_cast<int32_t>(BSA_SELECT_TOKEN_MAX)) != 0)
    return BSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(centroid) || !aligned16(radius) || !aligned16(alpha) ||
      !aligned16(kv_idx) || !aligned16(kv_cnt) || (mask && !aligned16(mask)))
    return BSA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < bsa::select_workspace_bytes(ms))
    return BSA_ERR_WORKSPACE;
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(ms.d)));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool token_max = (params->flags & BSA_SELECT_TOKEN_MAX) != 0;
  if (bsa::launch_select(ms, q, centroid, radius, alpha, ratio_ppm(params->centroid_keep),
                         ratio_ppm(params->rescue_keep), scale, token_max, kv_idx, kv_cnt, mask,
                         workspace, dev_status, s) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

bsa_status mask_build_impl(const bsa::MaskShape &ms, const bsa_select_params *params, const void *q,
                           const void *k, float *centroid, float *radius, float *quant, float *alpha,
                           int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream) {
  if (!params || !q || !k || !centroid || !radius || !quant || !alpha || !kv_idx || !kv_cnt)
    return BSA_ERR_INVALID_ARG;
  if (!ratio_ok(params->centroid_keep) || !ratio_ok(params->rescue_keep) || params->flags != 0)
    return BSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(centroid) || !aligned16(radius) || !aligned16(quant) ||
      !aligned16(alpha) || !aligned16(kv_idx) || !aligned16(kv_cnt) || (mask && !aligned16(mask)))
    return BSA_ERR_INVALID_ARG;
  size_t counters_at = 0;
  if (!workspace || !aligned16(workspace) || workspace_bytes < mask_build_bytes(ms, &counters_at))
    return BSA_ERR_WORKSPACE;
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(ms.d)));
  char *ws = static_cast<char *>(workspace);
  if (bsa::launch_layer_mask(ms, q, k, centroid, radius, quant, alpha, ratio_ppm(params->centroid_keep),
                             ratio_ppm(params->rescue_keep), scale, kv_idx, kv_cnt, mask, ws,
                             reinterpret_cast<unsigned *>(ws + counters_at), dev_status,
                             reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

bsa_status prefill_impl(const bsa::MaskShape &ms, const void *q, const void *k, const void *v,
                        const int32_t *kv_idx, const int32_t *kv_cnt, float softmax_scale, void *o,
                        float *lse, int32_t *dev_status, bsa_stream_t stream) {
  if (!q || !k || !v || !o) return BSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && !aligned16(lse)) || (kv_idx && !aligned16(kv_idx)) ||
      (kv_cnt && !aligned16(kv_cnt)))
    return BSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || isinf(softmax_scale)) return BSA_ERR_INVALID_ARG;
  cudaError_t ce = cudaSuccess;
  return bsa::launch_attention(attn_shape(ms), q, k, v, kv_idx, kv_cnt, softmax_scale, o, lse,
                               dev_status, reinterpret_cast<cudaStream_t>(stream), &ce);
}

bsa_status layer_impl(const bsa::MaskShape &ms, const bsa_select_params *params, const void *q,
                      const void *k, const void *v, float softmax_scale, void *o, float *lse,
                      void *workspace, size_t workspace_bytes, int32_t *dev_status,
                      bsa_stream_t stream) {
  size_t off[kLayerRegions], total = 0;
  layer_views(ms, off, &total);
  if (!workspace || workspace_bytes < total) return BSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BSA_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  float *centroid = reinterpret_cast<float *>(ws + off[0]);
  float *radius = reinterpret_cast<float *>(ws + off[1]);
  float *quant = reinterpret_cast<float *>(ws + off[2]);
  float *alpha = reinterpret_cast<float *>(ws + off[3]);
  int32_t *kv_idx = reinterpret_cast<int32_t *>(ws + off[4]);
  int32_t *kv_cnt = reinterpret_cast<int32_t *>(ws + off[5]);
  bsa_status r;
  if (params != nullptr && (params->flags & BSA_SELECT_TOKEN_MAX) != 0) {
    r = meta_impl(ms, k, centroid, radius, quant, alpha, dev_status, stream);
    if (r != BSA_OK) return r;
    r = select_impl(ms, params, q, centroid, radius, alpha, kv_idx, kv_cnt, nullptr, ws + off[6],
                    total - off[6], dev_status, stream);
  } else {
    r = mask_build_impl(ms, params, q, k, centroid, radius, quant, alpha, kv_idx, kv_cnt, nullptr, ws + off[6],
                        total - off[6], dev_status, stream);
  }
  if (r != BSA_OK) return r;
  return prefill_impl(ms, q, k, v, kv_idx, kv_cnt, softmax_scale, o, lse, dev_status, stream);
}

}  // namespace

extern "C" {

const char *bsa_status_string(bsa_status st) {
  switch (st) {
    case BSA_OK: return "BSA_OK";
    case BSA_ERR_INVALID_ARG: return "BSA_ERR_INVALID_ARG";
    case BSA_ERR_SHAPE: return "BSA_ERR_SHAPE";
    case BSA_ERR_UNSUPPORTED: return "BSA_ERR_UNSUPPORTED";
    case BSA_ERR_WORKSPACE: return "BSA_ERR_WORKSPACE";
    case BSA_ERR_CUDA: return "BSA_ERR_CUDA";
    case BSA_ERR_DEVICE_TIMEOUT: return "BSA_ERR_DEVICE_TIMEOUT";
  }
  return "BSA_ERR_UNKNOWN";
}

int32_t bsa_version(void) { return 100; }

bsa_status bsa_block_meta(const bsa_shape *shape, const void *k, float *centroid, float *radius,
                          float *quant, float *alpha, int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  return meta_impl(mask_shape(shape), k, centroid, radius, quant, alpha, dev_status, stream);
}

size_t bsa_select_workspace_bytes(const bsa_shape *shape) {
  if (check_shape(shape) != BSA_OK) return 0;
  return bsa::select_workspace_bytes(mask_shape(shape));
}

bsa_status bsa_select_mask(const bsa_shape *shape, const bsa_select_params *params, const void *q,
                           const float *centroid, const float *radius, const float *alpha,
                           int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  return select_impl(mask_shape(shape), params, q, centroid, radius, alpha, kv_idx, kv_cnt, mask,
                     workspace, workspace_bytes, dev_status, stream);
}

size_t bsa_mask_build_workspace_bytes(const bsa_shape *shape) {
  if (check_shape(shape) != BSA_OK) return 0;
  return mask_build_bytes(mask_shape(shape), nullptr);
}

bsa_status bsa_mask_build(const bsa_shape *shape, const bsa_select_params *params, const void *q,
                          const void *k, float *centroid, float *radius, float *quant, float *alpha,
                          int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, void *workspace,
                          size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  return mask_build_impl(mask_shape(shape), params, q, k, centroid, radius, quant, alpha, kv_idx, kv_cnt, mask,
                         workspace, workspace_bytes, dev_status, stream);
}

bsa_status bsa_prefill_fwd(const bsa_shape *shape, const void *q, const void *k, const void *v,
                           const int32_t *kv_idx, const int32_t *kv_cnt, float softmax_scale,
                           void *o, float *lse, int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  if (!kv_idx || !kv_cnt) return BSA_ERR_INVALID_ARG;
  return prefill_impl(mask_shape(shape), q, k, v, kv_idx, kv_cnt, softmax_scale, o, lse, dev_status,
                      stream);
}

bsa_status bsa_prefill_dense_fwd(const bsa_shape *shape, const void *q, const void *k,
                                 const void *v, float softmax_scale, void *o, float *lse,
                                 int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  return prefill_impl(mask_shape(shape), q, k, v, nullptr, nullptr, softmax_scale, o, lse,
                      dev_status, stream);
}

size_t bsa_prefill_layer_workspace_bytes(const bsa_shape *shape) {
  if (check_shape(shape) != BSA_OK) return 0;
  size_t off[kLayerRegions], total = 0;
  layer_views(mask_shape(shape), off, &total);
  return total;
}

bsa_status bsa_prefill_layer_views(const bsa_shape *shape, size_t *offsets) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  if (!offsets) return BSA_ERR_INVALID_ARG;
  size_t off[kLayerRegions], total = 0;
  layer_views(mask_shape(shape), off, &total);
  for (int x = 0; x < 6; ++x) offsets[x] = off[x];
  return BSA_OK;
}

bsa_status bsa_prefill_layer(const bsa_shape *shape, const bsa_select_params *params,
                             const void *q, const void *k, const void *v, float softmax_scale,
                             void *o, float *lse, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  return layer_impl(mask_shape(shape), params, q, k, v, softmax_scale, o, lse, workspace,
                    workspace_bytes, dev_status, stream);
}

// ---------------------------------------------------------------- fp8 (e4m3) inputs

bsa_status bsa_block_meta_fp8(const bsa_shape *shape, const void *k, float k_scale, float *centroid,
                              float *radius, float *quant, float *alpha, int32_t *dev_status,
                              bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  if (!scale_ok(k_scale)) return BSA_ERR_INVALID_ARG;
  return meta_impl(fp8_shape(shape, 1.f, k_scale, 1.f), k, centroid, radius, quant, alpha, dev_status,
                   stream);
}

bsa_status bsa_select_mask_fp8(const bsa_shape *shape, const bsa_select_params *params,
                               const void *q, float q_scale, const float *centroid,
                               const float *radius, const float *alpha, int32_t *kv_idx,
                               int32_t *kv_cnt, uint8_t *mask, void *workspace,
                               size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  if (!scale_ok(q_scale)) return BSA_ERR_INVALID_ARG;
  if (params != nullptr && (params->flags & BSA_SELECT_TOKEN_MAX)) return BSA_ERR_UNSUPPORTED;
  return select_impl(fp8_shape(shape, q_scale, 1.f, 1.f), params, q, centroid, radius, alpha, kv_idx,
                     kv_cnt, mask, workspace, workspace_bytes, dev_status, stream);
}

size_t bsa_prefill_fp8_workspace_bytes(const bsa_shape *shape) {
  if (check_shape(shape) != BSA_OK || shape->head_dim != 128) return 0;
  return round_up(static_cast<size_t>(shape->batch) * shape->seq * shape->hkv * shape->head_dim * 2, 256);
}

static bsa_status prefill_fp8_common(const bsa_shape *shape, const void *q, const void *k,
                                     const void *v, float q_scale, float k_scale, float v_scale,
                                     const int32_t *kv_idx, const int32_t *kv_cnt, float softmax_scale,
                                     void *o, float *lse, void *workspace, size_t workspace_bytes,
                                     int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  if (!scale_ok(q_scale) || !scale_ok(k_scale) || !scale_ok(v_scale)) return BSA_ERR_INVALID_ARG;
  if (shape->head_dim != 128) return BSA_ERR_UNSUPPORTED;
  if (!v || !aligned16(v)) return BSA_ERR_INVALID_ARG;
  const size_t need = bsa_prefill_fp8_workspace_bytes(shape);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return BSA_ERR_WORKSPACE;
  const size_t nv = static_cast<size_t>(shape->batch) * shape->seq * shape->hkv * shape->head_dim;
  if (bsa::launch_widen_e4m3(v, workspace, nv, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BSA_ERR_CUDA;
  return prefill_impl(fp8_shape(shape, q_scale, k_scale, v_scale), q, k, workspace, kv_idx, kv_cnt,
                      softmax_scale, o, lse, dev_status, stream);
}

bsa_status bsa_prefill_fwd_fp8(const bsa_shape *shape, const void *q, const void *k, const void *v,
                               float q_scale, float k_scale, float v_scale, const int32_t *kv_idx,
                               const int32_t *kv_cnt, float softmax_scale, void *o, float *lse,
                               void *workspace, size_t workspace_bytes, int32_t *dev_status,
                               bsa_stream_t stream) {
  if (!kv_idx || !kv_cnt) return check_shape(shape) != BSA_OK ? check_shape(shape) : BSA_ERR_INVALID_ARG;
  return prefill_fp8_common(shape, q, k, v, q_scale, k_scale, v_scale, kv_idx, kv_cnt, softmax_scale, o,
                            lse, workspace, workspace_bytes, dev_status, stream);
}

bsa_status bsa_prefill_dense_fwd_fp8(const bsa_shape *shape, const void *q, const void *k,
                                     const void *v, float q_scale, float k_scale, float v_scale,
                                     float softmax_scale, void *o, float *lse, void *workspace,
                                     size_t workspace_bytes, int32_t *dev_status, bsa_stream_t stream) {
  return prefill_fp8_common(shape, q, k, v, q_scale, k_scale, v_scale, nullptr, nullptr, softmax_scale, o,
                            lse, workspace, workspace_bytes, dev_status, stream);
}

// ---------------------------------------------------------------- packed ragged batches

int32_t bsa_varlen_block_stride(const bsa_varlen_shape *shape) {
  if (shape == nullptr) return 0;
  static const int32_t probe = 0;  // any aligned non-null pointer: only the shape is checked
  if (check_varlen(shape, &probe) != BSA_OK) return 0;
  return varlen_stride(shape);
}

bsa_status bsa_varlen_block_meta(const bsa_varlen_shape *shape, const int32_t *cu_seqlens,
                                 const void *k, float *centroid, float *radius, float *quant,
                                 float *alpha, int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_varlen(shape, cu_seqlens);
  if (st != BSA_OK) return st;
  return meta_impl(mask_shape(shape, cu_seqlens), k, centroid, radius, quant, alpha, dev_status,
                   stream);
}

size_t bsa_varlen_select_workspace_bytes(const bsa_varlen_shape *shape) {
  static const int32_t probe = 0;
  if (check_varlen(shape, &probe) != BSA_OK) return 0;
  return bsa::select_workspace_bytes(mask_shape(shape, &probe));
}

bsa_status bsa_varlen_select_mask(const bsa_varlen_shape *shape, const bsa_select_params *params,
                                  const int32_t *cu_seqlens, const void *q, const float *centroid,
                                  const float *radius, const float *alpha, int32_t *kv_idx,
                                  int32_t *kv_cnt, uint8_t *mask, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status,
                                  bsa_stream_t stream) {
  const bsa_status st = check_varlen(shape, cu_seqlens);
  if (st != BSA_OK) return st;
  return select_impl(mask_shape(shape, cu_seqlens), params, q, centroid, radius, alpha, kv_idx,
                     kv_cnt, mask, workspace, workspace_bytes, dev_status, stream);
}

bsa_status bsa_varlen_prefill_fwd(const bsa_varlen_shape *shape, const int32_t *cu_seqlens,
                                  const void *q, const void *k, const void *v,
                                  const int32_t *kv_idx, const int32_t *kv_cnt,
                                  float softmax_scale, void *o, float *lse, int32_t *dev_status,
                                  bsa_stream_t stream) {
  const bsa_status st = check_varlen(shape, cu_seqlens);
  if (st != BSA_OK) return st;
  if (!kv_idx || !kv_cnt) return BSA_ERR_INVALID_ARG;
  return prefill_impl(mask_shape(shape, cu_seqlens), q, k, v, kv_idx, kv_cnt, softmax_scale, o, lse,
                      dev_status, stream);
}

bsa_status bsa_varlen_prefill_dense_fwd(const bsa_varlen_shape *shape, const int32_t *cu_seqlens,
                                        const void *q, const void *k, const void *v,
                                        float softmax_scale, void *o, float *lse,
                                        int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_varlen(shape, cu_seqlens);
  if (st != BSA_OK) return st;
  return prefill_impl(mask_shape(shape, cu_seqlens), q, k, v, nullptr, nullptr, softmax_scale, o,
                      lse, dev_status, stream);
}

// ---------------------------------------------------------------- decode

size_t bsa_decode_workspace_bytes(const bsa_varlen_shape *shape) {
  static const int32_t probe = 0;
  if (check_varlen(shape, &probe) != BSA_OK) return 0;
  return bsa::decode_workspace_bytes(mask_shape(shape, &probe));
}

bsa_status bsa_decode_select(const bsa_varlen_shape *shape, const bsa_select_params *params,
                             const int32_t *cu_seqlens, const void *q_new, const float *centroid,
                             const float *radius, const float *alpha, int32_t *kv_idx,
                             int32_t *kv_cnt, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_varlen(shape, cu_seqlens);
  if (st != BSA_OK) return st;
  if (!params || !q_new || !centroid || !radius || !alpha || !kv_idx || !kv_cnt)
    return BSA_ERR_INVALID_ARG;
  if (!ratio_ok(params->centroid_keep) || !ratio_ok(params->rescue_keep) || params->flags != 0)
    return BSA_ERR_INVALID_ARG;
  if (!aligned16(q_new) || !aligned16(centroid) || !aligned16(radius) || !aligned16(alpha) ||
      !aligned16(kv_idx) || !aligned16(kv_cnt))
    return BSA_ERR_INVALID_ARG;
  const bsa::MaskShape ms = mask_shape(shape, cu_seqlens);
  if (!workspace || !aligned16(workspace) || workspace_bytes < bsa::decode_workspace_bytes(ms))
    return BSA_ERR_WORKSPACE;
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(ms.d)));
  if (bsa::launch_decode_select(ms, q_new, centroid, radius, alpha, ratio_ppm(params->centroid_keep),
                                ratio_ppm(params->rescue_keep), scale, kv_idx, kv_cnt, workspace,
                                dev_status, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

bsa_status bsa_decode_fwd(const bsa_varlen_shape *shape, const int32_t *cu_seqlens,
                          const void *q_new, const void *k, const void *v, const int32_t *kv_idx,
                          const int32_t *kv_cnt, float softmax_scale, void *o, float *lse,
                          void *workspace, size_t workspace_bytes, int32_t *dev_status,
                          bsa_stream_t stream) {
  const bsa_status st = check_varlen(shape, cu_seqlens);
  if (st != BSA_OK) return st;
  if (!q_new || !k || !v || !kv_idx || !kv_cnt || !o) return BSA_ERR_INVALID_ARG;
  if (!aligned16(q_new) || !aligned16(k) || !aligned16(v) || !aligned16(kv_idx) ||
      !aligned16(kv_cnt) || !aligned16(o) || (lse && !aligned16(lse)))
    return BSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || isinf(softmax_scale)) return BSA_ERR_INVALID_ARG;
  const bsa::MaskShape ms = mask_shape(shape, cu_seqlens);
  if (static_cast<long long>(ms.batch) * ms.hkv > bsa::kMaxDecodeRows) return BSA_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) || workspace_bytes < bsa::decode_workspace_bytes(ms))
    return BSA_ERR_WORKSPACE;
  if (bsa::launch_decode(ms, q_new, k, v, kv_idx, kv_cnt, softmax_scale, o, lse, workspace,
                         dev_status, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

bsa_status bsa_decode_step(const bsa_varlen_shape *shape, const bsa_select_params *params,
                           const int32_t *cu_seqlens, const void *q_new, const void *k, const void *v,
                           const float *centroid, const float *radius, const float *alpha,
                           float softmax_scale, int32_t *kv_idx, int32_t *kv_cnt, void *o, float *lse,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           bsa_stream_t stream) {
  const bsa_status st = check_varlen(shape, cu_seqlens);
  if (st != BSA_OK) return st;
  if (!params || !q_new || !k || !v || !centroid || !radius || !alpha || !kv_idx || !kv_cnt || !o)
    return BSA_ERR_INVALID_ARG;
  if (!ratio_ok(params->centroid_keep) || !ratio_ok(params->rescue_keep) || params->flags != 0)
    return BSA_ERR_INVALID_ARG;
  if (!aligned16(q_new) || !aligned16(k) || !aligned16(v) || !aligned16(centroid) || !aligned16(radius) ||
      !aligned16(alpha) || !aligned16(kv_idx) || !aligned16(kv_cnt) || !aligned16(o) || (lse && !aligned16(lse)))
    return BSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || isinf(softmax_scale)) return BSA_ERR_INVALID_ARG;
  const bsa::MaskShape ms = mask_shape(shape, cu_seqlens);
  if (static_cast<long long>(ms.batch) * ms.hkv > bsa::kMaxDecodeRows) return BSA_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) || workspace_bytes < bsa::decode_workspace_bytes(ms))
    return BSA_ERR_WORKSPACE;
  const float select_scale = static_cast<float>(1.0 / sqrt(static_cast<double>(ms.d)));
  if (bsa::launch_decode_step(ms, q_new, k, v, centroid, radius, alpha, ratio_ppm(params->centroid_keep),
                              ratio_ppm(params->rescue_keep), select_scale, softmax_scale, kv_idx, kv_cnt, o, lse,
                              workspace, dev_status, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

}  // extern "C"
