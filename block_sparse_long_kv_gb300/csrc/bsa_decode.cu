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
// Selection (bsa_decode_select), two launches:
//   decode_score_kernel    64 key blocks per CTA, one warp per key block: the
//                          new token's G heads against the centroid row
//                          (coalesced), S_c and R into the workspace
//   decode_topk_kernel     one warp per (b, g): the same two-path exact top-k
//                          as a prefill row (shared code, bsa_topk.cuh)
// Attention (bsa_decode_fwd), two launches:
//   decode_attn_kernel     one CTA per (kept block, b, g): the block's keys and
//                          values staged in shared memory by cp.async, the G
//                          heads' logits (one thread per key), an online
//                          softmax, and P V with 2 dimensions x one key group
//                          per thread; writes the split's unnormalised O, max
//                          and sum
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

constexpr int kAttnThreads = 128;
constexpr int kBlocksPerSplit = 1;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// ---------------------------------------------------------------- selection

constexpr int kScoreWarps = 8;
constexpr int kScoreBlocksPerWarp = 8;  // key blocks per warp: 64 per CTA

// S_c[j] and R[j] of the new token of (b, g) for the candidates 1 <= j < i, one
// warp per key block (a coalesced centroid row per lane group), 64 key blocks
// per CTA so every SM takes part even at batch 1.
template <int D>
__global__ void __launch_bounds__(kScoreWarps * 32) decode_score_kernel(
    const uint16_t *__restrict__ q_new, const float *__restrict__ centroid, const float *__restrict__ radius,
    const float *__restrict__ alpha, float *__restrict__ s_c, float *__restrict__ s_r,
    const int32_t *__restrict__ cu, int seq, int total, int block, int hq, int hkv, int nbs, float scale,
    int32_t *status) {
  __shared__ __align__(16) float qs[16 * D];
  __shared__ float qn[16];
  const int jt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int grp = hq / hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  if (sp.len == 0) return;
  const int i = (sp.len - 1) / block;  // the new token's block
  const int j0 = jt * kScoreWarps * kScoreBlocksPerWarp;
  if (j0 >= i) return;
  const uint16_t *qrow = q_new + (static_cast<size_t>(b) * hq + static_cast<size_t>(g) * grp) * D;
  for (int e = tid; e < grp * D; e += kScoreWarps * 32) qs[e] = bf16f(qrow[e]);
  __syncthreads();
  for (int h = warp; h < grp; h += kScoreWarps) {
    float s2 = 0.f;
    for (int x = lane; x < D; x += 32) s2 = fmaf(qs[h * D + x], qs[h * D + x], s2);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    if (lane == 0) qn[h] = sqrtf(s2);
  }
  __syncthreads();
  constexpr int DPL = D / 32;  // dimensions per lane
  for (int r = 0; r < kScoreBlocksPerWarp; ++r) {
    const int j = j0 + warp * kScoreBlocksPerWarp + r;
    if (j < 1 || j >= i) continue;  // warp-uniform
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
      s_c[gb * nbs + j] = dm * scale;
      s_r[gb * nbs + j] = rm * scale;
    }
  }
}

// One warp per (b, g): the two-path exact top-k of the new token's row (the
// prefill row code, bsa_topk.cuh) and the ascending kept list.
__global__ void __launch_bounds__(32) decode_topk_kernel(
    const float *__restrict__ s_c, const float *__restrict__ s_r, const float *__restrict__ alpha,
    int32_t *__restrict__ kv_idx, int32_t *__restrict__ kv_cnt, const int32_t *__restrict__ cu, int seq,
    int total, int block, int hkv, int nbs, long long ppm_c, long long ppm_r, int32_t *status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int g = blockIdx.x, b = blockIdx.y;
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  if (sp.len == 0) {
    if (threadIdx.x == 0) kv_cnt[gb] = 0;
    return;
  }
  const int i = (sp.len - 1) / block;
  const RowScratch w = row_scratch(smem, nbs);
  warp_select_row(s_c + gb * nbs, s_r + gb * nbs, alpha + gb * nbs, i, ppm_c, ppm_r, w);
  warp_emit_row(w, i, kv_idx + gb * nbs, kv_cnt + gb, nullptr, nbs);
}

// ---------------------------------------------------------------- attention

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <int D, int G>
struct DecCfg {
  static constexpr int KCH = 128;                    // keys per chunk = threads
  static constexpr int KROW = D * 2 + 16;            // padded key row (bytes): conflict-free row reads
  static constexpr int DP = D / 2;                   // dimension pairs
  static constexpr int KH = kAttnThreads / DP;       // key groups in P V
  static constexpr size_t OFF_K = 0;
  static constexpr size_t OFF_V = OFF_K + static_cast<size_t>(KCH) * KROW;
  static constexpr size_t OFF_Q = OFF_V + static_cast<size_t>(KCH) * D * 2;
  static constexpr size_t OFF_P = OFF_Q + static_cast<size_t>(G) * D * 4;
  static constexpr size_t SMEM = OFF_P + static_cast<size_t>(G) * KCH * 4;
  // the key-half O partials reuse the key buffer after the last chunk
  static_assert(static_cast<size_t>(KH > 1 ? KH - 1 : 1) * G * D * 4 <= static_cast<size_t>(KCH) * KROW,
                "O partials fit in the key buffer");
};

// Split s of row (b, g): kept blocks [s * kBlocksPerSplit, ...) of the list.
// Each 128-key chunk is staged in shared memory by cp.async (key rows padded,
// value rows dense); thread t takes key t for the G logits and, for P V, the
// dimension pair 2 * (t % (D/2)) of key group t / (D/2).
template <int D, int G>
__global__ void __launch_bounds__(kAttnThreads) decode_attn_kernel(
    const uint16_t *__restrict__ q_new, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const int32_t *__restrict__ kv_idx, const int32_t *__restrict__ kv_cnt, float *__restrict__ part_o,
    float *__restrict__ part_ml, const int32_t *__restrict__ cu, int seq, int total, int block, int hkv,
    int nbs, int nsplit, float scale_log2, int32_t *status) {
  using C = DecCfg<D, G>;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char *ks = smem + C::OFF_K;
  const uint16_t *vs = reinterpret_cast<const uint16_t *>(smem + C::OFF_V);
  float (*qs)[D] = reinterpret_cast<float (*)[D]>(smem + C::OFF_Q);
  float (*ps)[C::KCH] = reinterpret_cast<float (*)[C::KCH]>(smem + C::OFF_P);
  __shared__ float red[G][kAttnThreads / 32];
  __shared__ float mrun[G];

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

  const size_t tok_stride = static_cast<size_t>(hkv) * D;
  const int dp = tid % C::DP, kh = tid / C::DP;
  float o[G][2];
  float lsum[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    o[h][0] = o[h][1] = 0.f;
    lsum[h] = 0.f;
  }
  const int last = (sp.len - 1) / block;
  for (int e = e0; e < e1; ++e) {
    const int j = kv_idx[gb * nbs + e];
    if (j < 0 || j > last) continue;  // a malformed list entry is skipped (CTA-uniform)
    const int nk = min(block, sp.len - j * block);  // keys of block j
    for (int c0 = 0; c0 < nk; c0 += C::KCH) {
      const int kend = min(C::KCH, nk - c0);
      __syncthreads();  // the previous chunk's K, V and P are no longer read
      {
        // stage the chunk's key and value rows: D*2/16 pieces of 16 bytes per row
        constexpr int PR = D * 2 / 16;
        const uint16_t *kg = k + (static_cast<size_t>(sp.start) + static_cast<size_t>(j) * block + c0) * tok_stride +
                             static_cast<size_t>(g) * D;
        const uint16_t *vg = v + (static_cast<size_t>(sp.start) + static_cast<size_t>(j) * block + c0) * tok_stride +
                             static_cast<size_t>(g) * D;
        for (int x = tid; x < kend * PR; x += kAttnThreads) {
          const int r = x / PR, pc = x - r * PR;
          cp_async16(ks + r * C::KROW + pc * 16, kg + static_cast<size_t>(r) * tok_stride + pc * 8);
          cp_async16(smem + C::OFF_V + (static_cast<size_t>(r) * D + pc * 8) * 2,
                     vg + static_cast<size_t>(r) * tok_stride + pc * 8);
        }
        cp_async_wait_all();
      }
      __syncthreads();
      const bool valid = tid < kend;
      // ---- logits of key c0 + tid for the G heads (log2 units)
      float lg[G];
#pragma unroll
      for (int h = 0; h < G; ++h) lg[h] = valid ? 0.f : -INFINITY;
      if (valid) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(ks + tid * C::KROW);
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
            float a = lg[h];
            a = fmaf(qa.x, kf[0], a);
            a = fmaf(qa.y, kf[1], a);
            a = fmaf(qa.z, kf[2], a);
            a = fmaf(qa.w, kf[3], a);
            a = fmaf(qb.x, kf[4], a);
            a = fmaf(qb.y, kf[5], a);
            a = fmaf(qb.z, kf[6], a);
            a = fmaf(qb.w, kf[7], a);
            lg[h] = a;
          }
        }
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
      // ---- P V for this thread's dimension pair and key group
#pragma unroll
      for (int h = 0; h < G; ++h) {
        o[h][0] *= factor[h];
        o[h][1] *= factor[h];
        lsum[h] *= factor[h];
      }
      const uint32_t *vcol = reinterpret_cast<const uint32_t *>(vs) + dp;
#pragma unroll 4
      for (int s = kh; s < kend; s += C::KH) {
        const uint32_t vv = vcol[s * (D / 2)];
        const float v0 = __uint_as_float(vv << 16), v1 = __uint_as_float(vv & 0xFFFF0000u);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = ps[h][s];
          o[h][0] = fmaf(p, v0, o[h][0]);
          o[h][1] = fmaf(p, v1, o[h][1]);
          lsum[h] += p;
        }
      }
    }
  }
  __syncthreads();  // the key buffer becomes the key groups' O partials
  float (*oacc)[G][D] = reinterpret_cast<float (*)[G][D]>(ks);
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
      for (int x = 0; x < C::KH - 1; ++x) {
        a0 += oacc[x][h][2 * dp];
        a1 += oacc[x][h][2 * dp + 1];
      }
      const size_t po = ((static_cast<size_t>(b) * hq + static_cast<size_t>(g) * G + h) * nsplit + split) * D;
      part_o[po + 2 * dp] = a0;
      part_o[po + 2 * dp + 1] = a1;
    }
  }
  // the normaliser: each key group summed its own keys' probabilities; add the groups of
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
      for (int x = 0; x < C::KH - 1; ++x) l += oacc[x][h][0];
      const size_t pm = ((static_cast<size_t>(b) * hq + static_cast<size_t>(g) * G + h) * nsplit + split) * 2;
      part_ml[pm] = mrun[h];
      part_ml[pm + 1] = l;
    }
  }
}

// One CTA per (b, h): the splits' maxima and sums reduced across the CTA, then
// O = sum_s w_s O_s / sum_s w_s l_s with w_s = 2^(m_s - max m), 8 splits'
// partial rows in flight per thread.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_ml, const int32_t *__restrict__ kv_cnt,
    uint16_t *__restrict__ o, float *__restrict__ lse, const int32_t *__restrict__ cu, int seq, int total,
    int block, int hq, int hkv, int nsplit, int32_t *status) {
  extern __shared__ float wsm[];  // [nsplit] weights
  __shared__ float redm[D / 32], redl[D / 32];
  const int h = blockIdx.x, b = blockIdx.y, x = threadIdx.x, lane = x & 31, warp = x >> 5;
  const int g = h / (hq / hkv);
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const int cnt = sp.len > 0 ? min(kv_cnt[static_cast<size_t>(b) * hkv + g], (sp.len - 1) / block + 1) : 0;
  const int ns = (cnt + kBlocksPerSplit - 1) / kBlocksPerSplit;
  const size_t base = (static_cast<size_t>(b) * hq + h) * nsplit;
  float m = -INFINITY;
  for (int s = x; s < ns; s += D) m = fmaxf(m, part_ml[(base + s) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) redm[warp] = m;
  __syncthreads();
  m = redm[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) m = fmaxf(m, redm[w]);
  float l = 0.f;
  for (int s = x; s < ns; s += D) {
    const float ms = part_ml[(base + s) * 2];
    const float wgt = ms == -INFINITY ? 0.f : exp2f(ms - m);
    wsm[s] = wgt;
    l = fmaf(part_ml[(base + s) * 2 + 1], wgt, l);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  if (lane == 0) redl[warp] = l;
  __syncthreads();
  l = 0.f;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) l += redl[w];
  float acc = 0.f;
  int s = 0;
  for (; s + 8 <= ns; s += 8) {
    float pv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) pv[u] = part_o[(base + s + u) * D + x];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc = fmaf(pv[u], wsm[s + u], acc);
  }
  for (; s < ns; ++s) acc = fmaf(part_o[(base + s) * D + x], wsm[s], acc);
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
  using C = DecCfg<D, G>;
  auto kern = decode_attn_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  dim3 grid(nsplit, s.hkv, s.batch);
  kern<<<grid, kAttnThreads, C::SMEM, stream>>>(
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

// Workspace regions (each 256-byte aligned): partial O [b, hq, nsplit, d], partial (max, sum)
// [b, hq, nsplit, 2], then the selection's S_c and R rows [b, hkv, nbs].
struct DecRegions {
  size_t po, pml, sc, sr, total;
};

DecRegions decode_regions(const MaskShape &s) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(s.batch) * s.hq * decode_splits(s);
  const size_t srow = static_cast<size_t>(s.batch) * s.hkv * s.nbs * 4;
  DecRegions r;
  r.po = 0;
  r.pml = r.po + r256(rows * s.d * 4);
  r.sc = r.pml + r256(rows * 2 * 4);
  r.sr = r.sc + r256(srow);
  r.total = r.sr + r256(srow);
  return r;
}

}  // namespace

size_t decode_workspace_bytes(const MaskShape &s) { return decode_regions(s).total; }

cudaError_t launch_decode_select(const MaskShape &s, const void *q_new, const float *centroid,
                                 const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                                 float scale, int32_t *kv_idx, int32_t *kv_cnt, void *workspace,
                                 int32_t *status, cudaStream_t stream) {
  const DecRegions r = decode_regions(s);
  float *sc = reinterpret_cast<float *>(static_cast<char *>(workspace) + r.sc);
  float *sr = reinterpret_cast<float *>(static_cast<char *>(workspace) + r.sr);
  dim3 grid((s.nbs + kScoreWarps * kScoreBlocksPerWarp - 1) / (kScoreWarps * kScoreBlocksPerWarp), s.hkv, s.batch);
  if (s.d == 64)
    decode_score_kernel<64><<<grid, kScoreWarps * 32, 0, stream>>>(
        static_cast<const uint16_t *>(q_new), centroid, radius, alpha, sc, sr, s.cu, s.seq, s.total, s.block,
        s.hq, s.hkv, s.nbs, scale, status);
  else if (s.d == 128)
    decode_score_kernel<128><<<grid, kScoreWarps * 32, 0, stream>>>(
        static_cast<const uint16_t *>(q_new), centroid, radius, alpha, sc, sr, s.cu, s.seq, s.total, s.block,
        s.hq, s.hkv, s.nbs, scale, status);
  else
    return cudaErrorInvalidValue;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = row_scratch_bytes(s.nbs);
  e = cudaFuncSetAttribute(decode_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  decode_topk_kernel<<<dim3(s.hkv, s.batch), 32, smem, stream>>>(sc, sr, alpha, kv_idx, kv_cnt, s.cu, s.seq, s.total,
                                                                 s.block, s.hkv, s.nbs, static_cast<long long>(ppm_c),
                                                                 static_cast<long long>(ppm_r), status);
  return cudaGetLastError();
}

cudaError_t launch_decode(const MaskShape &s, const void *q_new, const void *k, const void *v,
                          const int32_t *kv_idx, const int32_t *kv_cnt, float scale, void *o, float *lse,
                          void *workspace, int32_t *status, cudaStream_t stream) {
  const int nsplit = decode_splits(s);
  const DecRegions r = decode_regions(s);
  float *po = reinterpret_cast<float *>(static_cast<char *>(workspace) + r.po);
  float *pml = reinterpret_cast<float *>(static_cast<char *>(workspace) + r.pml);
  const float sl2 = scale * kLog2e;
  cudaError_t e;
  if (s.d == 64) e = launch_attn_d<64>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, sl2, status, stream);
  else if (s.d == 128) e = launch_attn_d<128>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, nsplit, sl2, status, stream);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  dim3 grid(s.hq, s.batch);
  const size_t csmem = static_cast<size_t>(nsplit) * 4;
  if (s.d == 64)
    decode_combine_kernel<64><<<grid, 64, csmem, stream>>>(po, pml, kv_cnt, static_cast<uint16_t *>(o), lse, s.cu,
                                                           s.seq, s.total, s.block, s.hq, s.hkv, nsplit, status);
  else
    decode_combine_kernel<128><<<grid, 128, csmem, stream>>>(po, pml, kv_cnt, static_cast<uint16_t *>(o), lse,
                                                             s.cu, s.seq, s.total, s.block, s.hq, s.hkv, nsplit,
                                                             status);
  return cudaGetLastError();
}

}  // namespace bsa
