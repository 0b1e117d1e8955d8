// Block-sparse decode of one new token per sequence (q_len = 1), split over
// the kept key blocks.
//
// Sources: "Your 128K Context Is 6x Slower Than It Needs to Be"
// (articles.phantom-byte.com), section "The rescue branch: two selection
// paths, one mask" (the selection, applied here to a one-token query block);
// "Your Context Length Decides What a Kernel Is Worth" (pub.towardsai.net),
// decode paragraphs: decode attention is bound by memory traffic, and a
// split-KV kernel is what brings a small batch near the card's peak rate.
//
// Three launches per step:
//   decode_select_kernel   one CTA per (b, g): scores of the new token's G
//                          heads against every earlier key block's centroid
//                          (one warp per key block, coalesced centroid rows),
//                          then the same two-path exact top-k as a prefill row
//                          (shared warp code, bsa_topk.cuh)
//   decode_attn_kernel     one CTA per (split of kBlocksPerSplit kept blocks,
//                          b, g): the G heads' logits against each kept key
//                          (one thread per key), an online softmax over the
//                          split, and P V with 2 dims x 2 key halves per thread;
//                          writes the split's unnormalised O, max and sum
//   decode_combine_kernel  one CTA per (b, h): merges the splits (log-sum-exp)
//                          and writes O and LSE
// The cache is a packed batch (sequence b = tokens cu[b] .. cu[b+1]-1, its
// last token the new one), checked like every packed batch (seq_span).

#include <cuda_bf16.h>
#include <stdint.h>

#include "bsa_internal.h"
#include "bsa_topk.cuh"

namespace bsa {
namespace {

using namespace topk;

constexpr int kSelThreads = 256;
constexpr int kAttnThreads = 128;
constexpr int kBlocksPerSplit = 2;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// Dynamic shared memory of the select CTA: q [G][D] fp32, |q| [G], S_c and R
// rows [nbs] fp32, then one warp's row scratch.
size_t decode_select_smem(int group, int d, int nbs) {
  return (static_cast<size_t>(group) * d + 16 + 2 * static_cast<size_t>(nbs)) * 4 + row_scratch_bytes(nbs);
}

template <int D>
__global__ void __launch_bounds__(kSelThreads) decode_select_kernel(
    const uint16_t *__restrict__ q_new, const float *__restrict__ centroid, const float *__restrict__ radius,
    const float *__restrict__ alpha, int32_t *__restrict__ kv_idx, int32_t *__restrict__ kv_cnt,
    const int32_t *__restrict__ cu, int seq, int total, int block, int hq, int hkv, int nbs, long long ppm_c,
    long long ppm_r, float scale, int32_t *status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int g = blockIdx.x, b = blockIdx.y;
  const int grp = hq / hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  float *qs = reinterpret_cast<float *>(smem);           // [G][D]
  float *qn = qs + grp * D;                              // [G] (16 slots)
  float *sc = qn + 16;                                   // [nbs]
  float *sr = sc + nbs;                                  // [nbs]
  const RowScratch w = row_scratch(reinterpret_cast<unsigned char *>(sr + nbs), nbs);

  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  if (sp.len == 0) {
    if (tid == 0) kv_cnt[gb] = 0;
    return;
  }
  const int i = (sp.len - 1) / block;  // the new token's block
  const uint16_t *qrow = q_new + (static_cast<size_t>(b) * hq + static_cast<size_t>(g) * grp) * D;
  for (int e = tid; e < grp * D; e += kSelThreads) qs[e] = bf16f(qrow[e]);
  __syncthreads();
  for (int h = warp; h < grp; h += kSelThreads / 32) {
    float s2 = 0.f;
    for (int x = lane; x < D; x += 32) s2 = fmaf(qs[h * D + x], qs[h * D + x], s2);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    if (lane == 0) qn[h] = sqrtf(s2);
  }
  __syncthreads();

  // S_c[j], R[j] for the candidates 1 <= j < i: one warp per key block
  constexpr int DPL = D / 32;  // dimensions per lane
  for (int j = 1 + warp; j < i; j += kSelThreads / 32) {
    const float *crow = centroid + (gb * nbs + j) * D + lane * DPL;
    float c[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) c[e] = crow[e];
    const float bonus = alpha[gb * nbs + j] * radius[gb * nbs + j];
    float dm = -INFINITY, rm = -INFINITY;
    for (int h = 0; h < grp; ++h) {
      float p = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) p = fmaf(qs[h * D + lane * DPL + e], c[e], p);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
      dm = fmaxf(dm, p);
      rm = fmaxf(rm, fmaf(qn[h], bonus, p));
    }
    if (lane == 0) {
      sc[j] = dm * scale;
      sr[j] = rm * scale;
    }
  }
  __syncthreads();
  if (warp == 0) {
    warp_select_row(sc, sr, alpha + gb * nbs, i, ppm_c, ppm_r, w);
    warp_emit_row(w, i, kv_idx + gb * nbs, kv_cnt + gb, nullptr, nbs);
  }
}

// Split s of row (b, g): kept blocks [s * kBlocksPerSplit, ...) of the list.
// Thread t is key t of a 128-key chunk for the logits and, for P V, owns the
// dimension pair 2 * (t % (D/2)) of key half t / (D/2).
template <int D, int G>
__global__ void __launch_bounds__(kAttnThreads) decode_attn_kernel(
    const uint16_t *__restrict__ q_new, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const int32_t *__restrict__ kv_idx, const int32_t *__restrict__ kv_cnt, float *__restrict__ part_o,
    float *__restrict__ part_ml, const int32_t *__restrict__ cu, int seq, int total, int block, int hkv,
    int nbs, int nsplit, float scale_log2, int32_t *status) {
  constexpr int KCH = 128;          // keys per chunk = threads
  constexpr int DP = D / 2;         // dimension pairs
  constexpr int KH = kAttnThreads / DP;  // key groups in P V (2 for D = 128, 4 for D = 64)
  __shared__ __align__(16) float qs[G][D];
  __shared__ float ps[G][KCH];
  __shared__ float red[G][kAttnThreads / 32];
  __shared__ float mrun[G];
  __shared__ float oacc[KH > 1 ? KH - 1 : 1][G][D];

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const int hq = hkv * G;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const int cnt = sp.len > 0 ? min(kv_cnt[gb], (sp.len - 1) / block + 1) : 0;
  const int e0 = split * kBlocksPerSplit, e1 = min(e0 + kBlocksPerSplit, cnt);
  if (e0 >= e1) return;  // the combine reads only ceil(cnt / kBlocksPerSplit) splits

  const uint16_t *qrow = q_new + (static_cast<size_t>(b) * hq + static_cast<size_t>(g) * G) * D;
  for (int e = tid; e < G * D; e += kAttnThreads) qs[e / D][e % D] = bf16f(qrow[e]) * scale_log2;
  if (tid < G) mrun[tid] = -INFINITY;
  __syncthreads();

  const size_t tok_stride = static_cast<size_t>(hkv) * D;
  const int dp = tid % DP, kh = tid / DP;
  float o[G][2];
  float lsum[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    o[h][0] = o[h][1] = 0.f;
    lsum[h] = 0.f;
  }
  const int last = (sp.len - 1) / block;
  for (int e = e0; e < e1; ++e) {
    int j = kv_idx[gb * nbs + e];
    if (j < 0 || j > last) continue;  // a malformed list entry is skipped
    const int nk = min(block, sp.len - j * block);  // keys of block j
    for (int c0 = 0; c0 < nk; c0 += KCH) {
      const int kk = c0 + tid;
      const bool valid = kk < nk;
      // ---- logits of key kk for the G heads (log2 units)
      float lg[G];
      if (valid) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(
            k + (static_cast<size_t>(sp.start) + static_cast<size_t>(j) * block + kk) * tok_stride +
            static_cast<size_t>(g) * D);
#pragma unroll
        for (int h = 0; h < G; ++h) lg[h] = 0.f;
#pragma unroll 4
        for (int x8 = 0; x8 < D / 8; ++x8) {
          const uint4 u = kr[x8];
          const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
          float kf[8];
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {
            kf[2 * q2] = __uint_as_float(wv[q2] << 16);
            kf[2 * q2 + 1] = __uint_as_float(wv[q2] & 0xFFFF0000u);
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float4 qa = *reinterpret_cast<const float4 *>(&qs[h][x8 * 8]);
            const float4 qb = *reinterpret_cast<const float4 *>(&qs[h][x8 * 8 + 4]);
            lg[h] = fmaf(qa.x, kf[0], lg[h]);
            lg[h] = fmaf(qa.y, kf[1], lg[h]);
            lg[h] = fmaf(qa.z, kf[2], lg[h]);
            lg[h] = fmaf(qa.w, kf[3], lg[h]);
            lg[h] = fmaf(qb.x, kf[4], lg[h]);
            lg[h] = fmaf(qb.y, kf[5], lg[h]);
            lg[h] = fmaf(qb.z, kf[6], lg[h]);
            lg[h] = fmaf(qb.w, kf[7], lg[h]);
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) lg[h] = -INFINITY;
      }
      // ---- chunk max per head, new running max, probabilities
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = lg[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) red[h][warp] = mx;
      }
      __syncthreads();
      float factor[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = red[h][0];
#pragma unroll
        for (int x = 1; x < kAttnThreads / 32; ++x) mx = fmaxf(mx, red[h][x]);
        const float mold = mrun[h];
        const float mnew = fmaxf(mold, mx);
        factor[h] = mold == -INFINITY ? 0.f : exp2f(mold - mnew);
        ps[h][tid] = valid ? exp2f(lg[h] - mnew) : 0.f;
        lg[h] = mnew;  // keep the new max
      }
      __syncthreads();
      if (tid == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) mrun[h] = lg[h];
      }
      // ---- P V for this thread's dimension pair and key half
#pragma unroll
      for (int h = 0; h < G; ++h) {
        o[h][0] *= factor[h];
        o[h][1] *= factor[h];
        lsum[h] *= factor[h];
      }
      const uint32_t *vcol = reinterpret_cast<const uint32_t *>(
          v + (static_cast<size_t>(sp.start) + static_cast<size_t>(j) * block + c0) * tok_stride +
          static_cast<size_t>(g) * D + 2 * dp);
      const int kend = min(KCH, nk - c0);
      for (int s = kh; s < kend; s += KH) {
        const uint32_t vv = vcol[static_cast<size_t>(s) * (tok_stride / 2)];
        const float v0 = __uint_as_float(vv << 16), v1 = __uint_as_float(vv & 0xFFFF0000u);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = ps[h][s];
          o[h][0] = fmaf(p, v0, o[h][0]);
          o[h][1] = fmaf(p, v1, o[h][1]);
          lsum[h] += p;
        }
      }
      __syncthreads();  // ps and mrun are rewritten by the next chunk
    }
  }
  // ---- combine the key halves in a fixed order, write the split's partials
  if (kh > 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      oacc[kh - 1][h][2 * dp] = o[h][0];
      oacc[kh - 1][h][2 * dp + 1] = o[h][1];
    }
  }
  __syncthreads();
  if (kh == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a0 = o[h][0], a1 = o[h][1];
#pragma unroll
      for (int x = 0; x < KH - 1; ++x) {
        a0 += oacc[x][h][2 * dp];
        a1 += oacc[x][h][2 * dp + 1];
      }
      const size_t po = ((static_cast<size_t>(b) * hq + static_cast<size_t>(g) * G + h) * nsplit + split) * D;
      part_o[po + 2 * dp] = a0;
      part_o[po + 2 * dp + 1] = a1;
    }
  }
  // the normaliser: each key half summed its own keys' probabilities; add the halves of
  // dimension pair 0 in the same fixed order
  __syncthreads();
  if (dp == 0 && kh > 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) oacc[kh - 1][h][0] = lsum[h];
  }
  __syncthreads();
  if (tid == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float l = lsum[h];
#pragma unroll
      for (int x = 0; x < KH - 1; ++x) l += oacc[x][h][0];
      const size_t pm = ((static_cast<size_t>(b) * hq + static_cast<size_t>(g) * G + h) * nsplit + split) * 2;
      part_ml[pm] = mrun[h];
      part_ml[pm + 1] = l;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_ml, const int32_t *__restrict__ kv_cnt,
    uint16_t *__restrict__ o, float *__restrict__ lse, const int32_t *__restrict__ cu, int seq, int total,
    int block, int hq, int hkv, int nsplit, int32_t *status) {
  const int h = blockIdx.x, b = blockIdx.y, x = threadIdx.x;
  const int g = h / (hq / hkv);
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const int cnt = sp.len > 0 ? min(kv_cnt[static_cast<size_t>(b) * hkv + g], (sp.len - 1) / block + 1) : 0;
  const int ns = (cnt + kBlocksPerSplit - 1) / kBlocksPerSplit;
  const size_t base = (static_cast<size_t>(b) * hq + h) * nsplit;
  float m = -INFINITY;
  for (int s = 0; s < ns; ++s) m = fmaxf(m, part_ml[(base + s) * 2]);
  float l = 0.f, acc = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float ms = part_ml[(base + s) * 2];
    const float f = ms == -INFINITY ? 0.f : exp2f(ms - m);
    l = fmaf(part_ml[(base + s) * 2 + 1], f, l);
    acc = fmaf(part_o[(base + s) * D + x], f, acc);
  }
  const float r = l > 0.f ? acc / l : 0.f;
  const __nv_bfloat16 rb = __float2bfloat16_rn(r);
  o[(static_cast<size_t>(b) * hq + h) * D + x] = *reinterpret_cast<const uint16_t *>(&rb);
  if (lse != nullptr && x == 0)
    lse[static_cast<size_t>(b) * hq + h] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
}

template <int D, int G>
cudaError_t launch_attn_g(const MaskShape &s, const void *q_new, const void *k, const void *v,
                          const int32_t *kv_idx, const int32_t *kv_cnt, float *po, float *pml, int nsplit,
                          float scale_log2, int32_t *status, cudaStream_t stream) {
  dim3 grid(nsplit, s.hkv, s.batch);
  decode_attn_kernel<D, G><<<grid, kAttnThreads, 0, stream>>>(
      static_cast<const uint16_t *>(q_new), static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v),
      kv_idx, kv_cnt, po, pml, s.cu, s.seq, s.total, s.block, s.hkv, s.nbs, nsplit, scale_log2, status);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_attn_d(const MaskShape &s, const void *q_new, const void *k, const void *v,
                          const int32_t *kv_idx, const int32_t *kv_cnt, float *po, float *pml, int nsplit,
                          float scale_log2, int32_t *status, cudaStream_t st) {
  switch (s.group) {
    case 1: return launch_attn_g<D, 1>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, scale_log2, status, st);
    case 2: return launch_attn_g<D, 2>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, scale_log2, status, st);
    case 4: return launch_attn_g<D, 4>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, scale_log2, status, st);
    case 8: return launch_attn_g<D, 8>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, scale_log2, status, st);
    case 16: return launch_attn_g<D, 16>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, scale_log2, status, st);
    default: return cudaErrorInvalidValue;
  }
}

int decode_splits(const MaskShape &s) { return (s.nbs + kBlocksPerSplit - 1) / kBlocksPerSplit; }

}  // namespace

size_t decode_workspace_bytes(const MaskShape &s) {
  const size_t rows = static_cast<size_t>(s.batch) * s.hq * decode_splits(s);
  return (rows * s.d * 4 + 255) / 256 * 256 + rows * 2 * 4;
}

cudaError_t launch_decode_select(const MaskShape &s, const void *q_new, const float *centroid,
                                 const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                                 float scale, int32_t *kv_idx, int32_t *kv_cnt, int32_t *status,
                                 cudaStream_t stream) {
  const size_t smem = decode_select_smem(s.group, s.d, s.nbs);
  dim3 grid(s.hkv, s.batch);
  cudaError_t e;
  if (s.d == 64) {
    e = cudaFuncSetAttribute(decode_select_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    decode_select_kernel<64><<<grid, kSelThreads, smem, stream>>>(
        static_cast<const uint16_t *>(q_new), centroid, radius, alpha, kv_idx, kv_cnt, s.cu, s.seq, s.total,
        s.block, s.hq, s.hkv, s.nbs, static_cast<long long>(ppm_c), static_cast<long long>(ppm_r), scale, status);
  } else if (s.d == 128) {
    e = cudaFuncSetAttribute(decode_select_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    decode_select_kernel<128><<<grid, kSelThreads, smem, stream>>>(
        static_cast<const uint16_t *>(q_new), centroid, radius, alpha, kv_idx, kv_cnt, s.cu, s.seq, s.total,
        s.block, s.hq, s.hkv, s.nbs, static_cast<long long>(ppm_c), static_cast<long long>(ppm_r), scale, status);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_decode(const MaskShape &s, const void *q_new, const void *k, const void *v,
                          const int32_t *kv_idx, const int32_t *kv_cnt, float scale, void *o, float *lse,
                          void *workspace, int32_t *status, cudaStream_t stream) {
  const int nsplit = decode_splits(s);
  const size_t rows = static_cast<size_t>(s.batch) * s.hq * nsplit;
  float *po = static_cast<float *>(workspace);
  float *pml = reinterpret_cast<float *>(static_cast<char *>(workspace) + (rows * s.d * 4 + 255) / 256 * 256);
  const float sl2 = scale * kLog2e;
  cudaError_t e;
  if (s.d == 64) e = launch_attn_d<64>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, sl2, status, stream);
  else if (s.d == 128) e = launch_attn_d<128>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, sl2, status, stream);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  dim3 grid(s.hq, s.batch);
  if (s.d == 64)
    decode_combine_kernel<64><<<grid, 64, 0, stream>>>(po, pml, kv_cnt, static_cast<uint16_t *>(o), lse, s.cu,
                                                       s.seq, s.total, s.block, s.hq, s.hkv, nsplit, status);
  else
    decode_combine_kernel<128><<<grid, 128, 0, stream>>>(po, pml, kv_cnt, static_cast<uint16_t *>(o), lse, s.cu,
                                                         s.seq, s.total, s.block, s.hq, s.hkv, nsplit, status);
  return cudaGetLastError();
}

}  // namespace bsa
