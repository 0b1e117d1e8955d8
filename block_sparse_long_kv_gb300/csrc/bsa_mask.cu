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
// Kernels:
//   meta_kernel     one CTA per (b, g, j): centroid and radius of key block j
//                   (streams K once, the block held in registers)
//   quant_kernel    one CTA per (b, g): bitonic sort of the nb radii in
//                   registers, nearest-rank median / p90, rescue coefficient alpha
//   qpool_kernel    one CTA per (b, i, head chunk): mean query and mean query
//                   norm of block i (streams Q once: the dominant HBM bytes),
//                   written as tf32 hi / lo splits; one more CTA row splits the
//                   centroids the same way
//   meta_pool_kernel  the three above in one grid (bsa_mask_build and the
//                   layer call): meta CTAs, then pooling CTAs; each KV group's
//                   last meta CTA takes the quantiles
//   score_kernel    (bsa_score.cu) centroid / rescue scores of every causal key
//                   block on tensor cores
//   select_kernel   a team of 1 to 8 warps per (b, g, i) row, sized to the
//                   row: per-path exact top-k (a linear value histogram, then a
//                   radix threshold inside its threshold bin), OR, ascending
//                   kept-list emission
// Every reduction runs in a fixed order, so results are deterministic.

#include <cuda_bf16.h>
#include <stdint.h>

#include "bsa_fp8.cuh"
#include "bsa_internal.h"
#include "bsa_topk.cuh"
#include "sm103_ptx.cuh"

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

// tf32 split of an fp32 value: hi keeps the top 10 mantissa bits (exact in
// tf32), lo = x - hi is exact in fp32.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }


// One CTA per (b, g, j), the key block held in registers: thread t owns the
// 8 dimensions v = t % (D/8) of the tokens u, u + TL, u + 2 TL, ... with
// u = t / (D/8) and TL = 256 / (D/8) token lanes.  Pass 1 sums the tokens into
// the centroid (lane shuffles, then 8 warp partials in a fixed order); pass 2
// takes each token's squared distance to it from the same registers, so K is
// read from HBM once and never staged in shared memory.
// A partial last block (a packed sequence whose length is not a multiple of
// BLK) averages over its own tokens; CTAs past a sequence's last block write
// zeros.
template <int D, int BLK>
constexpr int meta_min_blocks() { return D * BLK > 128 * 128 ? 1 : 3; }

// Centroid and radius of key block j of (b, g); with c_hi / c_lo (nullable) also
// the centroid's tf32 hi / lo split (the score GEMM's A operand).
template <int D, int BLK, bool F8>
__device__ __forceinline__ void meta_block(int j, int g, int b, const unsigned char *__restrict__ k,
                                           float *__restrict__ centroid, float *__restrict__ radius,
                                           float *__restrict__ c_hi, float *__restrict__ c_lo,
                                           const int32_t *__restrict__ cu, int seq, int total, int hkv,
                                           int nbs, float scale, int32_t *status) {
  constexpr int EB = F8 ? 1 : 2;      // bytes per input element
  constexpr int VPR = D / 8;          // 16-byte vectors per key row
  constexpr int TL = kThreads / VPR;  // token lanes
  constexpr int TPT = BLK / TL;       // tokens per thread
  constexpr int NW = kThreads / 32;
  static_assert(TPT >= 1 && TPT * TL == BLK, "block must be a multiple of the token lanes");
  __shared__ __align__(16) float part[NW][D];
  __shared__ __align__(16) float sc[D];
  __shared__ float wmax[NW];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int v = tid % VPR, u = tid / VPR;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const size_t ob = (static_cast<size_t>(b) * hkv + g) * nbs + j;
  const int cnt = min(BLK, sp.len - j * BLK);  // keys in this block
  if (cnt <= 0) {
    if (tid < D) {
      centroid[ob * D + tid] = 0.f;
      if (c_hi != nullptr) c_hi[ob * D + tid] = c_lo[ob * D + tid] = 0.f;
    }
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
    const float cv = c * scale;  // in the inputs' units (scale 1 for bf16)
    centroid[ob * D + tid] = cv;
    if (c_hi != nullptr) {
      const float h = tf32_hi(cv);
      c_hi[ob * D + tid] = h;
      c_lo[ob * D + tid] = cv - h;
    }
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

template <int D, int BLK, bool F8>
__global__ void __launch_bounds__(kThreads, (meta_min_blocks<D, BLK>())) meta_kernel(
    const unsigned char *__restrict__ k, float *__restrict__ centroid, float *__restrict__ radius,
    const int32_t *__restrict__ cu, int seq, int total, int hkv, int nbs, float scale, int32_t *status) {
  meta_block<D, BLK, F8>(blockIdx.x, blockIdx.y, blockIdx.z, k, centroid, radius, nullptr, nullptr, cu, seq,
                         total, hkv, nbs, scale, status);
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

// Sixteen consecutive elements of one query token for one lane: bf16 (two
// 16-byte loads) or e4m3 (one).
template <bool F8>
struct Vec16 {
  uint4 u[F8 ? 1 : 2];
};

template <bool F8>
__device__ __forceinline__ Vec16<F8> load16(const unsigned char *p) {
  Vec16<F8> v;
  v.u[0] = __ldcs(reinterpret_cast<const uint4 *>(p));
  if constexpr (!F8) v.u[1] = __ldcs(reinterpret_cast<const uint4 *>(p + 16));
  return v;
}

// The sixteen elements as eight packed fp32 pairs (elements 2 e, 2 e + 1).
template <bool F8>
__device__ __forceinline__ void unpack16(const Vec16<F8> &v, uint64_t p[8]) {
  if constexpr (F8) {
    float f[16];
    e4m3x8_to_f32(make_uint2(v.u[0].x, v.u[0].y), f);
    e4m3x8_to_f32(make_uint2(v.u[0].z, v.u[0].w), f + 8);
#pragma unroll
    for (int e = 0; e < 8; ++e) p[e] = ptx::f32x2(f[2 * e], f[2 * e + 1]);
  } else {
    const uint32_t w[8] = {v.u[0].x, v.u[0].y, v.u[0].z, v.u[0].w, v.u[1].x, v.u[1].y, v.u[1].z, v.u[1].w};
#pragma unroll
    for (int e = 0; e < 8; ++e) p[e] = ptx::f32x2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
  }
}

// Adds one token's sixteen elements to the lane's pair sums and its L2 norm
// (the head's D / 16 lanes combine their partial squares) to nsum.
template <int D, bool F8>
__device__ __forceinline__ void pool_token(const Vec16<F8> &v, unsigned wmask, uint64_t acc[8], float &nsum) {
  constexpr int VH = D / 16;  // lanes per head
  uint64_t f[8];
  unpack16<F8>(v, f);
  uint64_t sq2 = 0ull;  // (+0.0f, +0.0f)
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    acc[e] = ptx::add_f32x2(acc[e], f[e]);
    sq2 = ptx::fma_f32x2(f[e], f[e], sq2);
  }
  float s0, s1;
  ptx::f32x2_split(sq2, s0, s1);
  float sq = s0 + s1;
#pragma unroll
  for (int off = VH / 2; off > 0; off >>= 1) sq += __shfl_xor_sync(wmask, sq, off);
  nsum += sqrtf(sq);
}

// Sums a full block's queries (16 dimensions per lane, on packed fp32 pairs)
// and their norms, 4 (bf16) or 8 (e4m3) tokens in flight per thread.
template <int D, bool F8>
__device__ __forceinline__ void pool_full(const unsigned char *__restrict__ base, size_t tok_stride,
                                          int cnt, unsigned wmask, uint64_t acc[8], float &nsum) {
  constexpr int TB = F8 ? 8 : 4;  // tokens in flight (32 or 16 bytes each per lane)
  for (int t0 = 0; t0 < cnt; t0 += TB) {
    Vec16<F8> u[TB];
#pragma unroll
    for (int r = 0; r < TB; ++r) u[r] = load16<F8>(base + static_cast<size_t>(t0 + r) * tok_stride);
#pragma unroll
    for (int r = 0; r < TB; ++r) pool_token<D, F8>(u[r], wmask, acc, nsum);
  }
}

// The same over the cnt < block queries of a packed sequence's partial last
// block, one token at a time (one such block per sequence).
template <int D, bool F8>
__device__ __forceinline__ void pool_partial(const unsigned char *__restrict__ base, size_t tok_stride,
                                             int cnt, unsigned wmask, uint64_t acc[8], float &nsum) {
#pragma unroll 1
  for (int t = 0; t < cnt; ++t) pool_token<D, F8>(load16<F8>(base + static_cast<size_t>(t) * tok_stride), wmask, acc, nsum);
}

// One thread per (head, 16 dimensions); the token loop keeps 4 (bf16) or 8
// (e4m3) tokens of loads in flight per thread.  Writes the mean query as tf32 hi / lo splits,
// q_hi/q_lo[b][g][i][hh][x] (one K-major row per (query block, head): the B
// operand of the score GEMM), and nbar[b][g][i][hh].  The extra row of CTAs
// (blockIdx.y == nhc) splits the centroids of key block blockIdx.x of every KV
// head into c_hi / c_lo, the GEMM's A operand.
template <int D, bool F8>
__device__ __forceinline__ void qpool_block(int i, int hc, int b, int nthreads, const unsigned char *__restrict__ q,
                                            float *__restrict__ q_hi, float *__restrict__ q_lo,
                                            float *__restrict__ nbar, const int32_t *__restrict__ cu, int seq,
                                            int total, int hq, int hkv, int block, int nbs, int hpc, float scale,
                                            int32_t *status) {
  constexpr int VH = D / 16;  // lanes per head
  constexpr int EB = F8 ? 1 : 2;  // bytes per input element
  const int tid = threadIdx.x;
  const int hl = tid / VH, xv = tid - hl * VH;
  const int h = hc * hpc + hl;
  const int grp = hq / hkv, g = h / grp, hh = h - g * grp;
  const size_t row = (static_cast<size_t>(b) * hkv + g) * nbs + i;
  const size_t qo = (row * grp + hh) * D + xv * 16;
  float4 *qh = reinterpret_cast<float4 *>(q_hi + qo);
  float4 *ql = reinterpret_cast<float4 *>(q_lo + qo);
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const int cnt = min(block, sp.len - i * block);  // queries in this block
  if (cnt <= 0) {  // past the sequence's last block: zero rows
#pragma unroll
    for (int x = 0; x < 4; ++x) qh[x] = ql[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (xv == 0) nbar[row * grp + hh] = 0.f;
    return;
  }
  const size_t tok_stride = static_cast<size_t>(hq) * D * EB;  // bytes
  const unsigned char *base = q + (static_cast<size_t>(sp.start) + static_cast<size_t>(i) * block) * tok_stride +
                              (static_cast<size_t>(h) * D + xv * 16) * EB;
  // lanes present in this warp (the last warp may be partial); a head's lanes never straddle warps
  const int present = min(32, nthreads - (tid & ~31));
  const unsigned wmask = present >= 32 ? 0xffffffffu : ((1u << present) - 1u);
  uint64_t acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0ull;
  float nsum = 0.f;
  if (cnt == block) pool_full<D, F8>(base, tok_stride, cnt, wmask, acc, nsum);
  else pool_partial<D, F8>(base, tok_stride, cnt, wmask, acc, nsum);
  const float inv = scale / static_cast<float>(cnt);  // exact for a full bf16 block (scale 1, cnt 2^k)
  float m[16], hi[16];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ptx::f32x2_split(acc[e], m[2 * e], m[2 * e + 1]);
    m[2 * e] *= inv;
    m[2 * e + 1] *= inv;
    hi[2 * e] = tf32_hi(m[2 * e]);
    hi[2 * e + 1] = tf32_hi(m[2 * e + 1]);
  }
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    qh[x] = make_float4(hi[4 * x], hi[4 * x + 1], hi[4 * x + 2], hi[4 * x + 3]);
    ql[x] = make_float4(m[4 * x] - hi[4 * x], m[4 * x + 1] - hi[4 * x + 1], m[4 * x + 2] - hi[4 * x + 2],
                        m[4 * x + 3] - hi[4 * x + 3]);
  }
  if (xv == 0) nbar[row * grp + hh] = nsum * inv;
}

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
  const int i = blockIdx.x, hc = blockIdx.y, b = blockIdx.z;
  if (hc == nhc) {
    for (int e = threadIdx.x; e < hkv * D; e += blockDim.x) {
      const int g = e / D, x = e - g * D;
      const size_t o = ((static_cast<size_t>(b) * hkv + g) * nbs + i) * D + x;
      const float v = centroid[o], h = tf32_hi(v);
      c_hi[o] = h;
      c_lo[o] = v - h;
    }
    return;
  }
  qpool_block<D, F8>(i, hc, b, static_cast<int>(blockDim.x), q, q_hi, q_lo, nbar, cu, seq, total, hq, hkv, block,
                     nbs, hpc, scale, status);
}

// ---------------------------------------------------------------- meta + pooling in one launch

// Nearest-rank median / p90 of the nb radii of one (b, g) and every block's
// alpha, by one CTA: the radii (read through L2: other CTAs wrote them) sorted
// ascending in shared memory by a bitonic network over npow2 entries (+inf
// padding).  Same values as quant_kernel: the sort is exact and alpha takes the
// same operations.
__device__ __forceinline__ void quant_smem(const float *radius, float *quant, float *alpha, float *buf, int nb,
                                           int nbs, size_t base, size_t qo) {
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int j = nb + tid; j < nbs; j += nt) alpha[base + j] = 0.f;
  if (nb == 0) {
    if (tid == 0) quant[qo] = quant[qo + 1] = 0.f;
    return;
  }
  int npow2 = 2;
  while (npow2 < nb) npow2 <<= 1;
  for (int x = tid; x < npow2; x += nt) buf[x] = x < nb ? __ldcg(radius + base + x) : INFINITY;
  __syncthreads();
  for (int kk = 2; kk <= npow2; kk <<= 1) {
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      for (int x = tid; x < npow2; x += nt) {
        const int p = x ^ jj;
        if (p > x) {
          const float a = buf[x], c = buf[p];
          if ((a > c) == ((x & kk) == 0)) {  // ascending where bit kk of x is clear
            buf[x] = c;
            buf[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const float med = buf[(nb + 1) / 2 - 1], p90 = buf[(9 * nb + 9) / 10 - 1];
  const float span = p90 - med;
  const bool degenerate = span <= 1e-12f * p90;
  if (tid == 0) {
    quant[qo] = med;
    quant[qo + 1] = p90;
  }
  for (int j = tid; j < nb; j += nt) {
    float a = 0.f;
    if (!degenerate) a = fminf(fmaxf((__ldcg(radius + base + j) - med) / span, 0.f), 1.f);
    alpha[base + j] = a;
  }
}

// The layer path's first launch: the key-block meta CTAs (b, g, j) and the
// query-pooling CTAs (b, head chunk, i) in one grid, so K and Q stream with no
// launch boundary between them.  Meta CTAs also write the centroids' tf32
// splits; the last meta CTA of each (b, g) to finish (counted in done[b][g],
// zero before the launch) takes that group's quantiles and alpha, so no launch
// waits on the radii.
template <int D, int BLK>
__global__ void __launch_bounds__(kThreads, (meta_min_blocks<D, BLK>())) meta_pool_kernel(
    const unsigned char *__restrict__ k, const unsigned char *__restrict__ q, float *__restrict__ centroid,
    float *__restrict__ radius, float *__restrict__ quant, float *__restrict__ alpha, float *__restrict__ c_hi,
    float *__restrict__ c_lo, float *__restrict__ q_hi, float *__restrict__ q_lo, float *__restrict__ nbar,
    unsigned *__restrict__ done, const int32_t *__restrict__ cu, int batch, int seq, int total, int hq, int hkv,
    int block, int nbs, int hpc, int nhc, int32_t *status) {
  extern __shared__ float sort_buf[];
  __shared__ unsigned last;
  // Grid order: unit u < nbs / 2 holds the pooling CTAs of query block u and the meta CTAs of key
  // blocks 2u and 2u + 1 (for every sequence); an odd nbs adds one unit with the last key block;
  // the remaining units pool query blocks ceil(nbs / 2) .. nbs - 1.  K streams beside Q instead of
  // ahead of it, and every key block is summarised by the middle of the Q stream, so the
  // quantiles are taken while the pooling goes on.
  int kind = 0, idx = 0, sub = 0, b = 0;  // kind 0: pooling (i, head chunk), 1: meta (j, g)
  {
    int x = static_cast<int>(blockIdx.x);
    const int hf = nbs / 2, s2 = nhc + 2 * hkv;
    const int l1 = hf * batch * s2;
    if (x < l1) {
      const int u = x / (batch * s2), rem = x - u * (batch * s2);
      b = rem / s2;
      const int o = rem - b * s2;
      if (o < nhc) {
        idx = u;
        sub = o;
      } else {
        kind = 1;
        idx = 2 * u + (o - nhc) / hkv;
        sub = (o - nhc) % hkv;
      }
    } else {
      x -= l1;
      bool placed = false;
      if (nbs & 1) {
        const int s1 = nhc + hkv;
        if (x < batch * s1) {
          b = x / s1;
          const int o = x - b * s1;
          if (o < nhc) {
            idx = hf;
            sub = o;
          } else {
            kind = 1;
            idx = 2 * hf;
            sub = o - nhc;
          }
          placed = true;
        } else {
          x -= batch * s1;
        }
      }
      if (!placed) {
        const int q = x / (batch * nhc), rem = x - q * (batch * nhc);
        idx = (nbs + 1) / 2 + q;
        b = rem / nhc;
        sub = rem - b * nhc;
      }
    }
  }
  if (kind == 1) {
    const int j = idx, g = sub;
    meta_block<D, BLK, false>(j, g, b, k, centroid, radius, c_hi, c_lo, cu, seq, total, hkv, nbs, 1.f, status);
    __threadfence();  // this CTA's radius before its count
    __syncthreads();
    const size_t bg = static_cast<size_t>(b) * hkv + g;
    if (threadIdx.x == 0) last = atomicAdd(done + bg, 1u) == static_cast<unsigned>(nbs - 1);
    __syncthreads();
    if (last) {
      __threadfence();
      const SeqSpan sp = seq_span(cu, b, seq, total, status);
      quant_smem(radius, quant, alpha, sort_buf, (sp.len + block - 1) / block, nbs, bg * nbs, bg * 2);
    }
    return;
  }
  const int i = idx, hc = sub;
  const int nthreads = hpc * (D / 16);
  if (static_cast<int>(threadIdx.x) < nthreads)
    qpool_block<D, false>(i, hc, b, nthreads, q, q_hi, q_lo, nbar, cu, seq, total, hq, hkv, block, nbs, hpc, 1.f,
                          status);
}

// ---------------------------------------------------------------- select

using namespace topk;

// Rows go to teams of W warps (topk::Team), W the smallest power of two with
// 32 W P >= i + 1, packed kTeamMaxWarps / W teams to a CTA of kTeamMaxWarps
// warps.  Class W holds the rows with 16 P W < i + 1 <= 32 P W (those with
// i + 1 <= 32 P for W = 1).  The grid runs class by class, widest first, and
// within a class group by group (b, g) and longest row first, so the CTAs
// resident at one time mostly run one team width's code.  Returns the CTAs of
// `groups` row sets of nbs rows each; with cta >= 0 also the class, the
// group, the first (longest) row and the team count of CTA `cta`.
struct TeamPlan {
  int w, group, first_row, teams;
};

template <int P>
__host__ __device__ inline int team_plan(int nbs, int groups, int cta, TeamPlan *plan) {
  int total = 0;
  for (int w = kTeamMaxWarps; w >= 1; w >>= 1) {
    const int hi_n = nbs < 32 * P * w ? nbs : 32 * P * w;
    const int lo_n = w == 1 ? 1 : 16 * P * w + 1;
    if (hi_n < lo_n) continue;
    const int rows = hi_n - lo_n + 1, tpc = kTeamMaxWarps / w;
    const int ctas = (rows + tpc - 1) / tpc;  // per group
    if (cta >= total && cta < total + ctas * groups) {
      const int k = (cta - total) % ctas;
      plan->w = w;
      plan->group = (cta - total) / ctas;
      plan->first_row = hi_n - 1 - k * tpc;
      plan->teams = rows - k * tpc < tpc ? rows - k * tpc : tpc;
    }
    total += ctas * groups;
  }
  return total;
}

struct SelectArgs {
  const float *s_c, *s_r, *alpha;
  int32_t *kv_idx, *kv_cnt;
  uint8_t *mask;
  const int32_t *cu;
  int batch, seq, total, block, hkv, nbs, nbw;
  long long ppm_c, ppm_r;
  int32_t *status;
};

template <int P, bool ALIGNED>
__device__ __forceinline__ void select_team_row(TeamScratch &sh, int team, int w, int i, int b, int g,
                                                const SelectArgs &a) {
  TeamRT tm(sh, w, 1 + team, static_cast<int>(threadIdx.x) - team * 32 * w);
  const size_t gb = static_cast<size_t>(b) * a.hkv + g;
  const size_t row = gb * a.nbs + i;
  {
    // rows past the sequence's last block: empty list, zero mask row
    const SeqSpan sp = seq_span(a.cu, b, a.seq, a.total, a.status);
    if (i >= (sp.len + a.block - 1) / a.block) {
      if (tm.t == 0) a.kv_cnt[row] = 0;
      if (a.mask != nullptr) {
        uint8_t *mrow = a.mask + row * static_cast<size_t>(a.nbs);
        if constexpr (ALIGNED) {
          for (int j4 = tm.t * 4; j4 < a.nbs; j4 += 4 * tm.T) reinterpret_cast<uint32_t *>(mrow)[j4 >> 2] = 0u;
        } else {
          for (int j = tm.t; j < a.nbs; j += tm.T) mrow[j] = 0u;
        }
      }
      return;
    }
  }
  tm.clear_hist();
  tm.sync();
  uint32_t fl[P / 4];
  team_select_row<TeamRT, P, ALIGNED>(tm, a.s_c + row * a.nbw, a.s_r + row * a.nbw, a.alpha + gb * a.nbs, i,
                                      a.ppm_c, a.ppm_r, fl);
  team_emit_row<TeamRT, P, ALIGNED>(tm, fl, i, a.kv_idx + row * static_cast<size_t>(a.nbs), a.kv_cnt + row,
                                    a.mask != nullptr ? a.mask + row * static_cast<size_t>(a.nbs) : nullptr, a.nbs);
}

// Per-path exact top-k, OR and kept-list emission for every (b, g, i) row:
// loads the row's centroid-path scores (from the tensor-core score kernel),
// selects the top kc, then the rescue-path scores of the candidates the
// centroid path dropped and whose alpha is positive, selects the top kr, ORs in
// the forced sink and diagonal blocks and writes the ascending kept list.
// P entries per lane (32 kTeamMaxWarps P >= nbw).  nbs is the row stride of
// alpha, kv_idx, kv_cnt and mask (the caller's arrays), nbw the row stride of
// the score matrices.  When nbs is not a multiple of 4 (a fixed-length batch
// whose block count is not), alpha and mask rows are not 16- / 4-byte aligned
// and are accessed element by element.
template <int P, bool ALIGNED>
__global__ void __launch_bounds__(kTeamMaxWarps * 32, (P <= 8 ? 4 : 2)) select_kernel(const __grid_constant__ SelectArgs a) {
  __shared__ TeamScratch sh[kTeamMaxWarps];
  TeamPlan plan{1, 0, 0, 0};
  team_plan<P>(a.nbs, a.batch * a.hkv, static_cast<int>(blockIdx.x), &plan);
  const int team = static_cast<int>(threadIdx.x >> 5) / plan.w;
  if (team >= plan.teams) return;  // whole teams leave; barriers are per team
  const int i = plan.first_row - team, g = plan.group % a.hkv, b = plan.group / a.hkv;
  select_team_row<P, ALIGNED>(sh[team], team, plan.w, i, b, g, a);  // one code path for every team width
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

// Heads per query-pooling CTA: the largest divisor of hq with <= 256 threads
// (d / 16 of them per head).
int qpool_heads(int hq, int d) {
  int best = 1;
  for (int h = 1; h <= hq; ++h)
    if (hq % h == 0 && h * (d / 16) <= kThreads) best = h;
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
    qpool_kernel<D, true><<<grid, hpc * (D / 16), 0, stream>>>(qb, q_hi, q_lo, nbar, centroid, c_hi, c_lo, s.cu,
                                                              s.seq, s.total, s.hq, s.hkv, s.block, s.nbs, hpc,
                                                              nhc, s.q_scale, status);
  else
    qpool_kernel<D, false><<<grid, hpc * (D / 16), 0, stream>>>(qb, q_hi, q_lo, nbar, centroid, c_hi, c_lo, s.cu,
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

namespace {

template <int P>
cudaError_t launch_select_p(const SelectArgs &a, bool aligned, cudaStream_t stream) {
  const int ctas = team_plan<P>(a.nbs, a.batch * a.hkv, -1, nullptr);
  dim3 grid(ctas > 0 ? ctas : 1);
  auto kern = aligned ? select_kernel<P, true> : select_kernel<P, false>;
  kern<<<grid, kTeamMaxWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t select_rows(const MaskShape &s, const float *s_c, const float *s_r, const float *alpha, int64_t ppm_c,
                        int64_t ppm_r, int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, int32_t *status,
                        cudaStream_t stream) {
  const bool al = s.nbs % 4 == 0;
  const SelectArgs a{s_c, s_r, alpha, kv_idx, kv_cnt, mask, s.cu, s.batch, s.seq, s.total, s.block, s.hkv, s.nbs, s.nbw,
                     static_cast<long long>(ppm_c), static_cast<long long>(ppm_r), status};
  if (s.nbw <= 32 * kTeamMaxWarps * 8) return launch_select_p<8>(a, al, stream);
  if (s.nbw <= 32 * kTeamMaxWarps * 16) return launch_select_p<16>(a, al, stream);
  return cudaErrorInvalidValue;
}

struct Regions {
  float *q_hi, *q_lo, *nbar, *c_hi, *c_lo, *s_c, *s_r;
};

Regions regions(const MaskShape &s, void *workspace) {
  const SelectRegions r = select_regions(s);
  char *ws = static_cast<char *>(workspace);
  float *reg[7];
  for (int x = 0; x < 7; ++x) reg[x] = reinterpret_cast<float *>(ws + r.off[x]);
  return Regions{reg[0], reg[1], reg[2], reg[3], reg[4], reg[5], reg[6]};
}

template <int D, int BLK>
cudaError_t launch_meta_pool_t(const MaskShape &s, const void *q, const void *k, float *centroid, float *radius,
                               float *quant, float *alpha, const Regions &w, unsigned *done, int32_t *status,
                               cudaStream_t stream) {
  const int hpc = qpool_heads(s.hq, D);
  const int nhc = s.hq / hpc;
  const long long nmeta = static_cast<long long>(s.nbs) * s.hkv * s.batch;
  const long long npool = static_cast<long long>(s.nbs) * nhc * s.batch;
  int npow2 = 2;
  while (npow2 < s.nbs) npow2 <<= 1;
  const size_t smem = static_cast<size_t>(npow2) * 4;
  meta_pool_kernel<D, BLK><<<static_cast<unsigned>(nmeta + npool), kThreads, smem, stream>>>(
      static_cast<const unsigned char *>(k), static_cast<const unsigned char *>(q), centroid, radius, quant, alpha,
      w.c_hi, w.c_lo, w.q_hi, w.q_lo, w.nbar, done, s.cu, s.batch, s.seq, s.total, s.hq, s.hkv, s.block, s.nbs, hpc,
      nhc, status);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_meta_pool_d(const MaskShape &s, const void *q, const void *k, float *centroid, float *radius,
                               float *quant, float *alpha, const Regions &w, unsigned *done, int32_t *status,
                               cudaStream_t stream) {
  switch (s.block) {
    case 64: return launch_meta_pool_t<D, 64>(s, q, k, centroid, radius, quant, alpha, w, done, status, stream);
    case 128: return launch_meta_pool_t<D, 128>(s, q, k, centroid, radius, quant, alpha, w, done, status, stream);
    case 256: return launch_meta_pool_t<D, 256>(s, q, k, centroid, radius, quant, alpha, w, done, status, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_select(const MaskShape &s, const void *q, const float *centroid,
                          const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                          float scale, bool token_max, int32_t *kv_idx, int32_t *kv_cnt,
                          uint8_t *mask, void *workspace, int32_t *status, cudaStream_t stream) {
  const Regions w = regions(s, workspace);
  cudaError_t e;
  if (token_max) {
    // the bf16 centroid splits (2 bytes each, hi then lo) fit in the fp32 c_hi region
    e = launch_token_scores(s, q, centroid, w.c_hi, radius, alpha, scale, w.s_c, w.s_r, status, stream);
  } else {
    if (s.d == 64) e = launch_qpool_d<64>(s, q, w.q_hi, w.q_lo, w.nbar, centroid, w.c_hi, w.c_lo, status, stream);
    else if (s.d == 128) e = launch_qpool_d<128>(s, q, w.q_hi, w.q_lo, w.nbar, centroid, w.c_hi, w.c_lo, status, stream);
    else return cudaErrorInvalidValue;
    if (e != cudaSuccess) return e;
    e = launch_scores(s, ScoreOperands{w.c_hi, w.c_lo, w.q_hi, w.q_lo, w.nbar, radius, alpha}, scale, w.s_c, w.s_r,
                      status, stream);
  }
  if (e != cudaSuccess) return e;
  return select_rows(s, w.s_c, w.s_r, alpha, ppm_c, ppm_r, kv_idx, kv_cnt, mask, status, stream);
}

size_t layer_mask_counter_bytes(const MaskShape &s) { return static_cast<size_t>(s.batch) * s.hkv * 4; }

cudaError_t launch_layer_mask(const MaskShape &s, const void *q, const void *k, float *centroid, float *radius,
                              float *quant, float *alpha, int64_t ppm_c, int64_t ppm_r, float scale,
                              int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask, void *workspace, unsigned *done,
                              int32_t *status, cudaStream_t stream) {
  if (s.fp8 || (s.d != 64 && s.d != 128)) return cudaErrorInvalidValue;
  const Regions w = regions(s, workspace);
  cudaError_t e = cudaMemsetAsync(done, 0, layer_mask_counter_bytes(s), stream);
  if (e != cudaSuccess) return e;
  e = s.d == 64 ? launch_meta_pool_d<64>(s, q, k, centroid, radius, quant, alpha, w, done, status, stream)
                : launch_meta_pool_d<128>(s, q, k, centroid, radius, quant, alpha, w, done, status, stream);
  if (e != cudaSuccess) return e;
  e = launch_scores(s, ScoreOperands{w.c_hi, w.c_lo, w.q_hi, w.q_lo, w.nbar, radius, alpha}, scale, w.s_c, w.s_r,
                    status, stream);
  if (e != cudaSuccess) return e;
  return select_rows(s, w.s_c, w.s_r, alpha, ppm_c, ppm_r, kv_idx, kv_cnt, mask, status, stream);
}

}  // namespace bsa
