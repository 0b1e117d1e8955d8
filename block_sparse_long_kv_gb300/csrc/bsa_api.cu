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

// Shape checks shared by every entry point.
bsa_status check_shape(const bsa_shape *s) {
  if (s == nullptr) return BSA_ERR_INVALID_ARG;
  if (s->batch < 1 || s->seq < 1 || s->hq < 1 || s->hkv < 1 || s->head_dim < 1 || s->block < 1)
    return BSA_ERR_SHAPE;
  if (s->seq % s->block != 0 || s->hq % s->hkv != 0) return BSA_ERR_SHAPE;
  if (s->head_dim != 64 && s->head_dim != 128) return BSA_ERR_UNSUPPORTED;
  if (s->block != 64 && s->block != 128 && s->block != 256) return BSA_ERR_UNSUPPORTED;
  const int nb = s->seq / s->block;
  if (nb % 4 != 0 || nb > bsa::kMaxBlocks) return BSA_ERR_UNSUPPORTED;
  const long long grp = s->hq / s->hkv;
  if (grp != 1 && grp != 2 && grp != 4 && grp != 8 && grp != 16) return BSA_ERR_UNSUPPORTED;
  if (s->block == 64 && grp % 2 != 0) return BSA_ERR_UNSUPPORTED;
  // grid extents of the widest launch (attention: one CTA per query tile pair)
  const long long items = static_cast<long long>(nb) * s->batch * s->hq;
  if (items > (1ll << 30)) return BSA_ERR_UNSUPPORTED;
  return BSA_OK;
}

bsa::MaskShape mask_shape(const bsa_shape *s) {
  return bsa::MaskShape{s->batch, s->seq, s->hq, s->hkv, s->head_dim, s->block,
                        s->seq / s->block, s->hq / s->hkv};
}

bsa::AttnShape attn_shape(const bsa_shape *s) {
  return bsa::AttnShape{s->batch, s->seq, s->hq, s->hkv, s->head_dim, s->block,
                        s->seq / s->block, s->hq / s->hkv};
}

bool ratio_ok(float r) { return r >= 0.f && r <= 1.f; }  // false for NaN

int64_t ratio_ppm(float r) { return static_cast<int64_t>(floor(static_cast<double>(r) * 1e6 + 0.5)); }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout of bsa_prefill_layer: centroid, radius, quant, alpha,
// kv_idx, kv_cnt, select scratch, each 256-byte aligned.
void layer_views(const bsa_shape *s, size_t off[7], size_t *total) {
  const size_t b = s->batch, h = s->hkv, d = s->head_dim, nb = s->seq / s->block;
  const size_t sizes[7] = {b * h * d * nb * 4, b * h * nb * 4,      b * h * 2 * 4, b * h * nb * 4,
                           b * h * nb * nb * 4, b * h * nb * 4,
                           bsa::select_workspace_bytes(mask_shape(s))};
  size_t cur = 0;
  for (int x = 0; x < 7; ++x) {
    off[x] = cur;
    cur = round_up(cur + sizes[x], 256);
  }
  *total = cur;
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
  (void)dev_status;  // the meta kernels have no waits
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  if (!k || !centroid || !radius || !quant || !alpha) return BSA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(centroid) || !aligned16(radius) || !aligned16(quant) ||
      !aligned16(alpha))
    return BSA_ERR_INVALID_ARG;
  const bsa::MaskShape ms = mask_shape(shape);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (bsa::launch_block_meta(ms, k, centroid, radius, s) != cudaSuccess) return BSA_ERR_CUDA;
  if (bsa::launch_quantiles(ms, radius, quant, alpha, s) != cudaSuccess) return BSA_ERR_CUDA;
  return BSA_OK;
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
  if (!params || !q || !centroid || !radius || !alpha || !kv_idx || !kv_cnt)
    return BSA_ERR_INVALID_ARG;
  if (!ratio_ok(params->centroid_keep) || !ratio_ok(params->rescue_keep) || params->flags != 0)
    return BSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(centroid) || !aligned16(radius) || !aligned16(alpha) ||
      !aligned16(kv_idx) || !aligned16(kv_cnt) || (mask && !aligned16(mask)))
    return BSA_ERR_INVALID_ARG;
  const bsa::MaskShape ms = mask_shape(shape);
  if (!workspace || !aligned16(workspace) || workspace_bytes < bsa::select_workspace_bytes(ms))
    return BSA_ERR_WORKSPACE;
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(shape->head_dim)));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (bsa::launch_select(ms, q, centroid, radius, alpha, ratio_ppm(params->centroid_keep),
                         ratio_ppm(params->rescue_keep), scale, kv_idx, kv_cnt, mask, workspace,
                         dev_status, s) != cudaSuccess)
    return BSA_ERR_CUDA;
  return BSA_OK;
}

static bsa_status prefill_common(const bsa_shape *shape, const void *q, const void *k,
                                 const void *v, const int32_t *kv_idx, const int32_t *kv_cnt,
                                 float softmax_scale, void *o, float *lse, int32_t *dev_status,
                                 bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  if (!q || !k || !v || !o) return BSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && !aligned16(lse)) || (kv_idx && !aligned16(kv_idx)) ||
      (kv_cnt && !aligned16(kv_cnt)))
    return BSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || isinf(softmax_scale)) return BSA_ERR_INVALID_ARG;
  cudaError_t ce = cudaSuccess;
  return bsa::launch_attention(attn_shape(shape), q, k, v, kv_idx, kv_cnt, softmax_scale, o, lse,
                               dev_status, reinterpret_cast<cudaStream_t>(stream), &ce);
}

bsa_status bsa_prefill_fwd(const bsa_shape *shape, const void *q, const void *k, const void *v,
                           const int32_t *kv_idx, const int32_t *kv_cnt, float softmax_scale,
                           void *o, float *lse, int32_t *dev_status, bsa_stream_t stream) {
  if (!kv_idx || !kv_cnt) return BSA_ERR_INVALID_ARG;
  return prefill_common(shape, q, k, v, kv_idx, kv_cnt, softmax_scale, o, lse, dev_status, stream);
}

bsa_status bsa_prefill_dense_fwd(const bsa_shape *shape, const void *q, const void *k,
                                 const void *v, float softmax_scale, void *o, float *lse,
                                 int32_t *dev_status, bsa_stream_t stream) {
  return prefill_common(shape, q, k, v, nullptr, nullptr, softmax_scale, o, lse, dev_status,
                        stream);
}

size_t bsa_prefill_layer_workspace_bytes(const bsa_shape *shape) {
  if (check_shape(shape) != BSA_OK) return 0;
  size_t off[7], total = 0;
  layer_views(shape, off, &total);
  return total;
}

bsa_status bsa_prefill_layer_views(const bsa_shape *shape, size_t *offsets) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  if (!offsets) return BSA_ERR_INVALID_ARG;
  size_t off[7], total = 0;
  layer_views(shape, off, &total);
  for (int x = 0; x < 6; ++x) offsets[x] = off[x];
  return BSA_OK;
}

bsa_status bsa_prefill_layer(const bsa_shape *shape, const bsa_select_params *params,
                             const void *q, const void *k, const void *v, float softmax_scale,
                             void *o, float *lse, void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, bsa_stream_t stream) {
  const bsa_status st = check_shape(shape);
  if (st != BSA_OK) return st;
  size_t off[7], total = 0;
  layer_views(shape, off, &total);
  if (!workspace || workspace_bytes < total) return BSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BSA_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  float *centroid = reinterpret_cast<float *>(ws + off[0]);
  float *radius = reinterpret_cast<float *>(ws + off[1]);
  float *quant = reinterpret_cast<float *>(ws + off[2]);
  float *alpha = reinterpret_cast<float *>(ws + off[3]);
  int32_t *kv_idx = reinterpret_cast<int32_t *>(ws + off[4]);
  int32_t *kv_cnt = reinterpret_cast<int32_t *>(ws + off[5]);
  bsa_status r = bsa_block_meta(shape, k, centroid, radius, quant, alpha, dev_status, stream);
  if (r != BSA_OK) return r;
  r = bsa_select_mask(shape, params, q, centroid, radius, alpha, kv_idx, kv_cnt, nullptr,
                      ws + off[6], total - off[6], dev_status, stream);
  if (r != BSA_OK) return r;
  return bsa_prefill_fwd(shape, q, k, v, kv_idx, kv_cnt, softmax_scale, o, lse, dev_status,
                         stream);
}

}  // extern "C"
