// Internal declarations shared by the libbsa translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsa.h"

namespace bsa {

constexpr int kMaxBlocks = 4096;  // nb limit (select kernel keeps one score row in smem)

struct MaskShape {
  int batch, seq, hq, hkv, d, block, nb, group;
};

// Block meta: centroid [b, hkv, nb, d], radius [b, hkv, nb].
cudaError_t launch_block_meta(const MaskShape &s, const void *k, float *centroid, float *radius,
                              cudaStream_t stream);
// Quantiles [b, hkv, 2] and alpha [b, hkv, nb] from radius.
cudaError_t launch_quantiles(const MaskShape &s, const float *radius, float *quant, float *alpha,
                             cudaStream_t stream);
// Bytes of select workspace: mean query [b, hkv, nb, G, d], mean query norm [b, hkv, nb, G]
// and the two score matrices [b, hkv, nb, nb], all fp32.
size_t select_workspace_bytes(const MaskShape &s);
// Query pooling into the workspace, tensor-core block scores, then top-k + list emission.
cudaError_t launch_select(const MaskShape &s, const void *q, const float *centroid,
                          const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                          float scale, int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask,
                          void *workspace, int32_t *status, cudaStream_t stream);

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

struct AttnShape {
  int batch, seq, hq, hkv, d, block, nb, group;
};

// Sparse (kv_idx != nullptr) or dense (kv_idx == nullptr) causal attention.
// Returns BSA_OK or an error code; `cuda_err` receives the CUDA error if any.
bsa_status launch_attention(const AttnShape &s, const void *q, const void *k, const void *v,
                            const int32_t *kv_idx, const int32_t *kv_cnt, float scale, void *o,
                            float *lse, int32_t *dev_status, cudaStream_t stream,
                            cudaError_t *cuda_err);

}  // namespace bsa
