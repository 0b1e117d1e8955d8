// Mask build for radius-rescued block-sparse prefill (HBM-bound kernels).
//
// Source: "Your 128K Context Is 6x Slower Than It Needs to Be"
// (articles.phantom-byte.com), section "The rescue branch: two selection
// paths, one mask": per key block a centroid and a max key-to-centroid radius,
// the median / 90th-percentile radius per (layer, KV head) as the reference
// points of a radius-adaptive coefficient, two independently thresholded
// selection paths, OR-combined.  The build reads every token a fixed number of
// times, so it is linear in the sequence length.
//
// Five launches:
//   meta_kernel     one CTA per (b, g, j): centroid and radius of key block j
//                   (streams K once, the block held in registers)
//   quant_kernel    one CTA per (b, g): bitonic sort of the nb radii in
//                   registers, nearest-rank median / p90, rescue coefficient alpha
//   qpool_kernel    one CTA per (b, i, head chunk): mean query and mean query
//                   norm of block i (streams Q once: the dominant HBM bytes),
//                   written as tf32 hi / lo splits; one more CTA row splits the
//                   centroids the same way
//   score_kernel    (bsa_score.cu) centroid / rescue scores of every causal key
//                   block on tensor cores
//   select_kernel   one warp per (b, g, i): per-path exact top-k (a linear
//                   value histogram, then a radix threshold inside its
//                   threshold bin), OR, ascending kept-list emission
// Every reduction runs in a fixed order, so results are deterministic.

#include <cuda_bf16.h>
#include <stdint.h>

#include "bsa_fp8.cuh"
#include "bsa_internal.h"
#include "bsa_topk.cuh"

namespace bsa {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void unpack_bf16x8(const uint4 &u, float f[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(w[e] << 16);
    f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
  }
}

// Eight consecutive input elements: bf16 (16 bytes) or e4m3 (8 bytes, F8).
template <bool F8>
__device__ __forceinline__ uint4 load8(const unsigned char *p) {
  if constexpr (F8) {
    const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(p));
    return make_uint4(x.x, x.y, 0u, 0u);
  } else {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
  }
}

template <bool F8>
__device__ __forceinline__ void unpack8(const uint4 &u, float f[8]) {
  if constexpr (F8) e4m3x8_to_f32(make_uint2(u.x, u.y), f);
  else unpack_bf16x8(u, f);
}

// ---------------------------------------------------------------- block meta

// One CTA per (b, g, j), the key block held in registers: thread t owns the
// 8 dimensions v = t % (D/8) of the tokens u, u + TL, u + 2 TL, ... with
// u = t / (D/8) and TL = 256 / (D/8) token lanes.  Pass 1 sums the tokens into
// the centroid (lane shuffles, then 8 warp partials in a fixed order); pass 2
// takes each token's squared distance to it from the same registers, so K is
// read from HBM once and never staged in shared memory.
// A partial last block (a packed sequence whose length is not a multiple of
// BLK) averages over its own tokens; CTAs past a sequence's last block write
// zeros.
template <int D, int BLK, bool F8>
__global__ void __launch_bounds__(kThreads, (D * BLK > 128 * 128 ? 1 : 3)) meta_kernel(const unsigned char *__restrict__ k,
                                                        float *__restrict__ centroid,
                                                        float *__restrict__ radius,
                                                        const int32_t *__restrict__ cu, int seq,
                                                        int total, int hkv, int nbs, float scale,
                                                        int32_t *status) {
  constexpr int EB = F8 ? 1 : 2;      // bytes per input element
  constexpr int VPR = D / 8;          // 16-byte vectors per key row
  constexpr int TL = kThreads / VPR;  // token lanes
  constexpr int TPT = BLK / TL;       // tokens per thread
  constexpr int NW = kThreads / 32;
  static_assert(TPT >= 1 && TPT * TL == BLK, "block must be a multiple of the token lanes");
  __shared__ __align__(16) float part[NW][D];
  __shared__ __align__(16) float sc[D];
  __shared__ float wmax[NW];

  const int j = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int v = tid % VPR, u = tid / VPR;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const size_t ob = (static_cast<size_t>(b) * hkv + g) * nbs + j;
  const int cnt = min(BLK, sp.len - j * BLK);  // keys in this block
  if (cnt <= 0) {
    if (tid < D) centroid[ob * D + tid] = 0.f;
    if (tid == 0) radius[ob] = 0.f;
    return;
  }
  const size_t tok_stride = static_cast<size_t>(hkv) * D * EB;  // bytes
  const unsigned char *base = k + (static_cast<size_t>(sp.start) + static_cast<size_t>(j) * BLK + u) * tok_stride +
                              (static_cast<size_t>(g) * D + v * 8) * EB;
  uint4 raw[TPT];
  if (cnt == BLK) {
#pragma unroll
    for (int r = 0; r < TPT; ++r) raw[r] = load8<F8>(base + static_cast<size_t>(r) * TL * tok_stride);
  } else {  // partial last block of a packed sequence
#pragma unroll
    for (int r = 0; r < TPT; ++r)
      raw[r] = (r * TL + u < cnt) ? load8<F8>(base + static_cast<size_t>(r) * TL * tok_stride)
                                  : make_uint4(0u, 0u, 0u, 0u);
  }

  // ---- pass 1: centroid
  float s[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) s[e] = 0.f;
#pragma unroll
  for (int r = 0; r < TPT; ++r) {
    float f[8];
    unpack8<F8>(raw[r], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] += f[e];
  }
#pragma unroll
  for (int off = VPR; off < 32; off <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] += __shfl_xor_sync(0xffffffffu, s[e], off);
  if (lane < VPR) {
    float4 *pp = reinterpret_cast<float4 *>(&part[warp][v * 8]);
    pp[0] = make_float4(s[0], s[1], s[2], s[3]);
    pp[1] = make_float4(s[4], s[5], s[6], s[7]);
  }
  __syncthreads();
  if (tid < D) {
    float c = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) c += part[w][tid];
    c /= static_cast<float>(cnt);
    sc[tid] = c;
    centroid[ob * D + tid] = c * scale;  // in the inputs' units (scale 1 for bf16)
  }
  __syncthreads();

  // ---- pass 2: max squared distance to the centroid
  float c[8];
  {
    const float4 c0 = reinterpret_cast<const float4 *>(sc)[2 * v];
    const float4 c1 = reinterpret_cast<const float4 *>(sc)[2 * v + 1];
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
    c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
  }
  float best = 0.f;
#pragma unroll
  for (int r = 0; r < TPT; ++r) {
    float f[8];
    unpack8<F8>(raw[r], f);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float dl = f[e] - c[e];
      acc = fmaf(dl, dl, acc);
    }
#pragma unroll
    for (int off = 1; off < VPR; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (r * TL + u < cnt) best = fmaxf(best, acc);
  }
#pragma unroll
  for (int off = VPR; off < 32; off <<= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, off));
  if (lane == 0) wmax[warp] = best;
  __syncthreads();
  if (tid == 0) {
    float m = wmax[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) m = fmaxf(m, wmax[w]);
    radius[ob] = sqrtf(m) * scale;
  }
}

// ---------------------------------------------------------------- quantiles

// Bitonic sort of the nb radii (padded with +inf to npow2 >= 32 E entries),
// then nearest-rank median / p90 and alpha.  Thread t holds entries
// t E .. t E + E - 1 in registers: exchange distances below E stay in the
// thread, those below 32 E go through warp shuffles, and only the longer ones
// through shared memory.
template <int E>
__global__ void __launch_bounds__(1024) quant_kernel(const float *__restrict__ radius,
                                                     float *__restrict__ quant,
                                                     float *__restrict__ alpha,
                                                     const int32_t *__restrict__ cu, int seq,
                                                     int total, int block, int nbs, int npow2,
                                                     int32_t *status) {
  extern __shared__ float sr[];
  __shared__ float sq[2];
  const int g = blockIdx.x, b = blockIdx.y, hkv = gridDim.x;
  const int tid = threadIdx.x;
  const size_t base = (static_cast<size_t>(b) * hkv + g) * nbs;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const int nb = (sp.len + block - 1) / block;  // this sequence's blocks
  for (int j = nb + tid; j < nbs; j += blockDim.x) alpha[base + j] = 0.f;
  if (nb == 0) {
    if (tid == 0) {
      quant[(static_cast<size_t>(b) * hkv + g) * 2 + 0] = 0.f;
      quant[(static_cast<size_t>(b) * hkv + g) * 2 + 1] = 0.f;
    }
    return;
  }
  float x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int idx = tid * E + e;
    x[e] = idx < nb ? radius[base + idx] : INFINITY;
  }
  for (int kk = 2; kk <= npow2; kk <<= 1) {
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      if (jj >= 32 * E) {
        // partner in another warp: exchange through shared memory
#pragma unroll
        for (int e = 0; e < E; ++e) sr[tid * E + e] = x[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int idx = tid * E + e;
          const float p = sr[idx ^ jj];
          const bool up = (idx & kk) == 0, lower = (idx & jj) == 0;
          x[e] = (lower == up) ? fminf(x[e], p) : fmaxf(x[e], p);
        }
        __syncthreads();
      } else if (jj >= E) {
        const int lj = jj / E;  // partner lane distance
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int idx = tid * E + e;
          const float p = __shfl_xor_sync(0xffffffffu, x[e], lj);
          const bool up = (idx & kk) == 0, lower = (idx & jj) == 0;
          x[e] = (lower == up) ? fminf(x[e], p) : fmaxf(x[e], p);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int pe = e ^ jj;
          if (pe > e) {
            const int idx = tid * E + e;
            const bool up = (idx & kk) == 0;
            const float a = x[e], c = x[pe];
            x[e] = up ? fminf(a, c) : fmaxf(a, c);
            x[pe] = up ? fmaxf(a, c) : fminf(a, c);
          }
        }
      }
    }
  }
  // nearest rank (1-based): ceil(nb / 2) and ceil(9 nb / 10)
  const int r_med = (nb + 1) / 2 - 1, r_p90 = (9 * nb + 9) / 10 - 1;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int idx = tid * E + e;
    if (idx == r_med) sq[0] = x[e];
    if (idx == r_p90) sq[1] = x[e];
  }
  __syncthreads();
  const float med = sq[0], p90 = sq[1];
  const float span = p90 - med;
  const bool degenerate = span <= 1e-12f * p90;
  if (tid == 0) {
    quant[(static_cast<size_t>(b) * hkv + g) * 2 + 0] = med;
    quant[(static_cast<size_t>(b) * hkv + g) * 2 + 1] = p90;
  }
  for (int j = tid; j < nb; j += blockDim.x) {
    float a = 0.f;
    if (!degenerate) a = fminf(fmaxf((radius[base + j] - med) / span, 0.f), 1.f);
    alpha[base + j] = a;
  }
}

// ---------------------------------------------------------------- query pooling

// tf32 split of an fp32 value: hi keeps the top 10 mantissa bits (exact in
// tf32), lo = x - hi is exact in fp32.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// Sums a full block's queries (8 dimensions per lane) and their norms, 8 (bf16)
// or 16 (e4m3) loads in flight per thread.
template <int D, bool F8>
__device__ __forceinline__ void pool_full(const unsigned char *__restrict__ base, size_t tok_stride,
                                          int cnt, unsigned wmask, float acc[8], float &nsum) {
  constexpr int VH = D / 8;        // lanes per head
  constexpr int TB = F8 ? 16 : 8;  // tokens in flight per lane (8-byte e4m3 loads: twice as many)
  for (int t0 = 0; t0 < cnt; t0 += TB) {
    uint4 u[TB];
#pragma unroll
    for (int r = 0; r < TB; ++r) u[r] = load8<F8>(base + static_cast<size_t>(t0 + r) * tok_stride);
#pragma unroll
    for (int r = 0; r < TB; ++r) {
      float f[8];
      unpack8<F8>(u[r], f);
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc[e] += f[e];
        sq = fmaf(f[e], f[e], sq);
      }
#pragma unroll
      for (int off = VH / 2; off > 0; off >>= 1) sq += __shfl_xor_sync(wmask, sq, off);
      nsum += sqrtf(sq);
    }
  }
}

// The same over the cnt < block queries of a packed sequence's partial last
// block, one token at a time (one such block per sequence).
template <int D, bool F8>
__device__ __forceinline__ void pool_partial(const unsigned char *__restrict__ base, size_t tok_stride,
                                             int cnt, unsigned wmask, float acc[8], float &nsum) {
  constexpr int VH = D / 8;
#pragma unroll 1
  for (int t = 0; t < cnt; ++t) {
    float f[8];
    unpack8<F8>(load8<F8>(base + static_cast<size_t>(t) * tok_stride), f);
    float sq = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      acc[e] += f[e];
      sq = fmaf(f[e], f[e], sq);
    }
#pragma unroll
    for (int off = VH / 2; off > 0; off >>= 1) sq += __shfl_xor_sync(wmask, sq, off);
    nsum += sqrtf(sq);
  }
}

// One thread per (head, 8 dimensions); the token loop keeps 8 16-byte loads in
// flight per thread.  Writes the mean query as tf32 hi / lo splits,
// q_hi/q_lo[b][g][i][hh][x] (one K-major row per (query block, head): the B
// operand of the score GEMM), and nbar[b][g][i][hh].  The extra row of CTAs
// (blockIdx.y == nhc) splits the centroids of key block blockIdx.x of every KV
// head into c_hi / c_lo, the GEMM's A operand.
template <int D, bool F8>
__global__ void __launch_bounds__(kThreads) qpool_kernel(const unsigned char *__restrict__ q,
                                                         float *__restrict__ q_hi,
                                                         float *__restrict__ q_lo,
                                                         float *__restrict__ nbar,
                                                         const float *__restrict__ centroid,
                                                         float *__restrict__ c_hi,
                                                         float *__restrict__ c_lo,
                                                         const int32_t *__restrict__ cu, int seq,
                                                         int total, int hq, int hkv, int block,
                                                         int nbs, int hpc, int nhc, float scale,
                                                         int32_t *status) {
  constexpr int VH = D / 8;  // lanes per head
  constexpr int EB = F8 ? 1 : 2;  // bytes per input element
  const int i = blockIdx.x, hc = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  if (hc == nhc) {
    for (int e = tid; e < hkv * D; e += blockDim.x) {
      const int g = e / D, x = e - g * D;
      const size_t o = ((static_cast<size_t>(b) * hkv + g) * nbs + i) * D + x;
      const float v = centroid[o], h = tf32_hi(v);
      c_hi[o] = h;
      c_lo[o] = v - h;
    }
    return;
  }
  const int hl = tid / VH, xv = tid - hl * VH;
  const int h = hc * hpc + hl;
  const int grp = hq / hkv, g = h / grp, hh = h - g * grp;
  const size_t row = (static_cast<size_t>(b) * hkv + g) * nbs + i;
  const size_t qo = (row * grp + hh) * D + xv * 8;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const int cnt = min(block, sp.len - i * block);  // queries in this block
  if (cnt <= 0) {  // past the sequence's last block: zero rows
    float4 *qh = reinterpret_cast<float4 *>(q_hi + qo);
    float4 *ql = reinterpret_cast<float4 *>(q_lo + qo);
    qh[0] = qh[1] = ql[0] = ql[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (xv == 0) nbar[row * grp + hh] = 0.f;
    return;
  }
  const size_t tok_stride = static_cast<size_t>(hq) * D * EB;  // bytes
  const unsigned char *base = q + (static_cast<size_t>(sp.start) + static_cast<size_t>(i) * block) * tok_stride +
                              (static_cast<size_t>(h) * D + xv * 8) * EB;
  // lanes present in this warp (the last warp may be partial); a head's lanes never straddle warps
  const int present = min(32, static_cast<int>(blockDim.x) - (tid & ~31));
  const unsigned wmask = present >= 32 ? 0xffffffffu : ((1u << present) - 1u);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  float nsum = 0.f;
  if (cnt == block) pool_full<D, F8>(base, tok_stride, cnt, wmask, acc, nsum);
  else pool_partial<D, F8>(base, tok_stride, cnt, wmask, acc, nsum);
  const float inv = scale / static_cast<float>(cnt);  // exact for a full bf16 block (scale 1, cnt 2^k)
  float m[8], hi[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    m[e] = acc[e] * inv;
    hi[e] = tf32_hi(m[e]);
  }
  float4 *qh = reinterpret_cast<float4 *>(q_hi + qo);
  float4 *ql = reinterpret_cast<float4 *>(q_lo + qo);
  qh[0] = make_float4(hi[0], hi[1], hi[2], hi[3]);
  qh[1] = make_float4(hi[4], hi[5], hi[6], hi[7]);
  ql[0] = make_float4(m[0] - hi[0], m[1] - hi[1], m[2] - hi[2], m[3] - hi[3]);
  ql[1] = make_float4(m[4] - hi[4], m[5] - hi[5], m[6] - hi[6], m[7] - hi[7]);
  if (xv == 0) nbar[row * grp + hh] = nsum * inv;
}

// ---------------------------------------------------------------- select

using namespace topk;

constexpr int kSelWarps = 8;   // rows per select CTA, one warp each


// One warp per (b, g, i) row, longest rows first; kSelWarps rows per CTA.
// Loads the row's centroid-path keys (scores from the tensor-core score
// kernel), selects the top kc, then the rescue-path keys of the candidates the
// centroid path dropped and whose alpha is positive, selects the top kr, ORs in
// the forced sink and diagonal blocks and writes the ascending kept list.
// nbs is the row stride of alpha, kv_idx, kv_cnt and mask (the caller's arrays),
// nbw the row stride of the score matrices and of the per-warp shared scratch.
// When nbs is not a multiple of 4 (a fixed-length batch whose block count is
// not), alpha and mask rows are not 16- / 4-byte aligned and are accessed
// element by element.
template <bool ALIGNED>
__global__ void __launch_bounds__(kSelWarps * 32) select_kernel(
    const float *__restrict__ s_c, const float *__restrict__ s_r, const float *__restrict__ alpha,
    int32_t *__restrict__ kv_idx, int32_t *__restrict__ kv_cnt, uint8_t *__restrict__ mask,
    const int32_t *__restrict__ cu, int seq, int total, int block, int hkv, int nbs, int nbw,
    long long ppm_c, long long ppm_r, int32_t *status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = nbs - 1 - (static_cast<int>(blockIdx.x) * kSelWarps + warp);
  if (i < 0) return;
  const int g = blockIdx.y, b = blockIdx.z;
  {
    // rows past the sequence's last block: empty list, zero mask row
    const SeqSpan sp = seq_span(cu, b, seq, total, status);
    if (i >= (sp.len + block - 1) / block) {
      const size_t row = (static_cast<size_t>(b) * hkv + g) * nbs + i;
      if (lane == 0) kv_cnt[row] = 0;
      if (mask != nullptr) {
        if constexpr (ALIGNED) {
          uint32_t *mrow = reinterpret_cast<uint32_t *>(mask + row * static_cast<size_t>(nbs));
          for (int j4 = lane * 4; j4 < nbs; j4 += 128) mrow[j4 >> 2] = 0u;
        } else {
          for (int j = lane; j < nbs; j += 32) mask[row * static_cast<size_t>(nbs) + j] = 0u;
        }
      }
      return;
    }
  }
  const RowScratch w = row_scratch(smem + static_cast<size_t>(warp) * row_scratch_bytes(nbw), nbw);
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const size_t row = gb * nbs + i;
  warp_select_row<ALIGNED>(s_c + row * nbw, s_r + row * nbw, alpha + gb * nbs, i, ppm_c, ppm_r, w);
  warp_emit_row<ALIGNED>(w, i, kv_idx + row * static_cast<size_t>(nbs), kv_cnt + row,
                         mask != nullptr ? mask + row * static_cast<size_t>(nbs) : nullptr, nbs);
}

template <int D, int BLK>
cudaError_t launch_meta_t(const MaskShape &s, const void *k, float *centroid, float *radius,
                          int32_t *status, cudaStream_t stream) {
  dim3 grid(s.nbs, s.hkv, s.batch);
  const unsigned char *kb = static_cast<const unsigned char *>(k);
  if (s.fp8)
    meta_kernel<D, BLK, true><<<grid, kThreads, 0, stream>>>(kb, centroid, radius, s.cu, s.seq, s.total, s.hkv,
                                                             s.nbs, s.k_scale, status);
  else
    meta_kernel<D, BLK, false><<<grid, kThreads, 0, stream>>>(kb, centroid, radius, s.cu, s.seq, s.total, s.hkv,
                                                              s.nbs, 1.f, status);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_meta_d(const MaskShape &s, const void *k, float *centroid, float *radius,
                          int32_t *status, cudaStream_t stream) {
  switch (s.block) {
    case 64: return launch_meta_t<D, 64>(s, k, centroid, radius, status, stream);
    case 128: return launch_meta_t<D, 128>(s, k, centroid, radius, status, stream);
    case 256: return launch_meta_t<D, 256>(s, k, centroid, radius, status, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Heads per query-pooling CTA: the largest divisor of hq with <= 256 threads.
int qpool_heads(int hq, int d) {
  int best = 1;
  for (int h = 1; h <= hq; ++h)
    if (hq % h == 0 && h * (d / 8) <= kThreads) best = h;
  return best;
}

template <int D>
cudaError_t launch_qpool_d(const MaskShape &s, const void *q, float *q_hi, float *q_lo, float *nbar,
                           const float *centroid, float *c_hi, float *c_lo, int32_t *status,
                           cudaStream_t stream) {
  const int hpc = qpool_heads(s.hq, D);
  const int nhc = s.hq / hpc;
  dim3 grid(s.nbs, nhc + 1, s.batch);
  const unsigned char *qb = static_cast<const unsigned char *>(q);
  if (s.fp8)
    qpool_kernel<D, true><<<grid, hpc * (D / 8), 0, stream>>>(qb, q_hi, q_lo, nbar, centroid, c_hi, c_lo, s.cu,
                                                              s.seq, s.total, s.hq, s.hkv, s.block, s.nbs, hpc,
                                                              nhc, s.q_scale, status);
  else
    qpool_kernel<D, false><<<grid, hpc * (D / 8), 0, stream>>>(qb, q_hi, q_lo, nbar, centroid, c_hi, c_lo, s.cu,
                                                               s.seq, s.total, s.hq, s.hkv, s.block, s.nbs, hpc,
                                                               nhc, 1.f, status);
  return cudaGetLastError();
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }


// Select workspace regions, each 256-byte aligned: q_hi, q_lo [b, hkv, nbs, G, d],
// nbar [b, hkv, nbs, G], c_hi, c_lo [b, hkv, nbs, d], S_c, R [b, hkv, nbs, nbw], all fp32.
struct SelectRegions {
  size_t off[7];
  size_t total;
};

SelectRegions select_regions(const MaskShape &s) {
  const size_t rows = static_cast<size_t>(s.batch) * s.hq * s.nbs;  // (b, g, i, h) rows
  const size_t blocks = static_cast<size_t>(s.batch) * s.hkv * s.nbs;
  const size_t sizes[7] = {rows * s.d * 4, rows * s.d * 4, rows * 4, blocks * s.d * 4, blocks * s.d * 4,
                           blocks * s.nbw * 4, blocks * s.nbw * 4};
  SelectRegions r{};
  size_t at = 0;
  for (int x = 0; x < 7; ++x) {
    r.off[x] = at;
    at += round256(sizes[x]);
  }
  r.total = at;
  return r;
}

}  // namespace

size_t select_workspace_bytes(const MaskShape &s) { return select_regions(s).total; }

cudaError_t launch_block_meta(const MaskShape &s, const void *k, float *centroid, float *radius,
                              int32_t *status, cudaStream_t stream) {
  if (s.d == 64) return launch_meta_d<64>(s, k, centroid, radius, status, stream);
  if (s.d == 128) return launch_meta_d<128>(s, k, centroid, radius, status, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_quantiles(const MaskShape &s, const float *radius, float *quant, float *alpha,
                             int32_t *status, cudaStream_t stream) {
  // E entries per thread, at most 1024 threads, and at least one full warp
  const int e = s.nb > 2048 ? 4 : (s.nb > 1024 ? 2 : 1);
  int npow2 = 32 * e;
  while (npow2 < s.nb) npow2 <<= 1;
  const int threads = npow2 / e;
  dim3 grid(s.hkv, s.batch);
  const size_t smem = static_cast<size_t>(npow2) * 4;
  if (e == 4)
    quant_kernel<4><<<grid, threads, smem, stream>>>(radius, quant, alpha, s.cu, s.seq, s.total, s.block,
                                                     s.nbs, npow2, status);
  else if (e == 2)
    quant_kernel<2><<<grid, threads, smem, stream>>>(radius, quant, alpha, s.cu, s.seq, s.total, s.block,
                                                     s.nbs, npow2, status);
  else
    quant_kernel<1><<<grid, threads, smem, stream>>>(radius, quant, alpha, s.cu, s.seq, s.total, s.block,
                                                     s.nbs, npow2, status);
  return cudaGetLastError();
}

cudaError_t launch_select(const MaskShape &s, const void *q, const float *centroid,
                          const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                          float scale, bool token_max, int32_t *kv_idx, int32_t *kv_cnt,
                          uint8_t *mask, void *workspace, int32_t *status, cudaStream_t stream) {
  const SelectRegions r = select_regions(s);
  char *ws = static_cast<char *>(workspace);
  float *reg[7];
  for (int x = 0; x < 7; ++x) reg[x] = reinterpret_cast<float *>(ws + r.off[x]);
  float *q_hi = reg[0], *q_lo = reg[1], *nbar = reg[2], *c_hi = reg[3], *c_lo = reg[4];
  float *s_c = reg[5], *s_r = reg[6];
  cudaError_t e;
  if (token_max) {
    // the bf16 centroid splits (2 bytes each, hi then lo) fit in the fp32 c_hi region
    e = launch_token_scores(s, q, centroid, c_hi, radius, alpha, scale, s_c, s_r, status, stream);
  } else {
    if (s.d == 64) e = launch_qpool_d<64>(s, q, q_hi, q_lo, nbar, centroid, c_hi, c_lo, status, stream);
    else if (s.d == 128) e = launch_qpool_d<128>(s, q, q_hi, q_lo, nbar, centroid, c_hi, c_lo, status, stream);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    e = launch_scores(s, ScoreOperands{c_hi, c_lo, q_hi, q_lo, nbar, radius, alpha}, scale, s_c, s_r,
                      status, stream);
  }
  if (e != cudaSuccess) return e;
  const size_t smem = kSelWarps * row_scratch_bytes(s.nbw);
  const bool aligned = s.nbs % 4 == 0;
  auto kern = aligned ? select_kernel<true> : select_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((s.nbs + kSelWarps - 1) / kSelWarps, s.hkv, s.batch);
  kern<<<grid, kSelWarps * 32, smem, stream>>>(s_c, s_r, alpha, kv_idx, kv_cnt, mask, s.cu, s.seq, s.total,
                                               s.block, s.hkv, s.nbs, s.nbw, static_cast<long long>(ppm_c),
                                               static_cast<long long>(ppm_r), status);
  return cudaGetLastError();
}

}  // namespace bsa
