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
// Three launches:
//   meta_kernel     one CTA per (b, g, j): centroid and radius of key block j
//   quant_kernel    one CTA per (b, g): nearest-rank median / p90 and alpha
//   select_kernel   one CTA per (b, g, i): mean query and mean query norm of
//                   block i for the G heads of group g (the dominant HBM
//                   stream), then centroid / rescue scores for every causal
//                   key block, per-path top-k by radix select, OR, emission
//                   of the ascending kept list.
// Every reduction runs in a fixed order, so results are deterministic.

#include <cuda_bf16.h>
#include <stdint.h>

#include "bsa_internal.h"

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

__device__ __forceinline__ float bf16_at(const uint16_t *p, int idx) {
  return __uint_as_float(static_cast<uint32_t>(p[idx]) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// ---------------------------------------------------------------- block meta

template <int D>
__global__ void __launch_bounds__(kThreads) meta_kernel(const uint16_t *__restrict__ k,
                                                        float *__restrict__ centroid,
                                                        float *__restrict__ radius, int seq,
                                                        int hkv, int block, int nb) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int VPR = D / 8;       // 16-byte vectors per key row
  constexpr int P = kThreads / D;  // partial sums per centroid coordinate
  uint4 *sk = reinterpret_cast<uint4 *>(smem);
  float *part = reinterpret_cast<float *>(smem + static_cast<size_t>(block) * D * 2);
  __shared__ float sc[D];
  __shared__ float wmax[kThreads / 32];

  const int j = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const size_t tok_stride = static_cast<size_t>(hkv) * D;
  const uint16_t *base =
      k + (static_cast<size_t>(b) * seq + static_cast<size_t>(j) * block) * tok_stride +
      static_cast<size_t>(g) * D;

  const int nvec = block * VPR;
  for (int e = tid; e < nvec; e += kThreads) {
    const int t = e / VPR, v = e - t * VPR;
    sk[e] = __ldcs(reinterpret_cast<const uint4 *>(base + static_cast<size_t>(t) * tok_stride) + v);
  }
  __syncthreads();

  const uint16_t *skh = reinterpret_cast<const uint16_t *>(sk);
  {
    const int x = tid % D, p = tid / D;
    float s = 0.f;
    for (int t = p; t < block; t += P) s += bf16_at(skh, t * D + x);
    part[p * D + x] = s;
  }
  __syncthreads();
  if (tid < D) {
    float s = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) s += part[p * D + tid];
    const float c = s / static_cast<float>(block);
    sc[tid] = c;
    centroid[((static_cast<size_t>(b) * hkv + g) * D + tid) * nb + j] = c;
  }
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31;
  float best = 0.f;
  for (int t = warp; t < block; t += kThreads / 32) {
    float acc = 0.f;
#pragma unroll
    for (int x = lane; x < D; x += 32) {
      const float dl = bf16_at(skh, t * D + x) - sc[x];
      acc = fmaf(dl, dl, acc);
    }
    best = fmaxf(best, warp_sum(acc));
  }
  if (lane == 0) wmax[warp] = best;
  __syncthreads();
  if (tid == 0) {
    float m = wmax[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, wmax[w]);
    radius[(static_cast<size_t>(b) * hkv + g) * nb + j] = sqrtf(m);
  }
}

// ---------------------------------------------------------------- quantiles

__global__ void __launch_bounds__(1024) quant_kernel(const float *__restrict__ radius,
                                                     float *__restrict__ quant,
                                                     float *__restrict__ alpha, int nb) {
  extern __shared__ float sr[];
  __shared__ float s_med, s_p90;
  const int g = blockIdx.x, b = blockIdx.y, hkv = gridDim.x;
  const size_t base = (static_cast<size_t>(b) * hkv + g) * nb;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) sr[j] = radius[base + j];
  __syncthreads();
  // nearest rank (1-based): ceil(nb / 2) and ceil(9 nb / 10)
  const int i_med = (nb + 1) / 2 - 1;
  const int i_p90 = (9 * nb + 9) / 10 - 1;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) {
    const float rj = sr[j];
    int pos = 0;  // position of j in the (value, index)-ordered ascending sort
    for (int q = 0; q < nb; ++q) {
      const float rq = sr[q];
      pos += (rq < rj) || (rq == rj && q < j);
    }
    if (pos == i_med) s_med = rj;
    if (pos == i_p90) s_p90 = rj;
  }
  __syncthreads();
  const float med = s_med, p90 = s_p90;
  const float span = p90 - med;
  const bool degenerate = span <= 1e-12f * p90;
  if (threadIdx.x == 0) {
    quant[(static_cast<size_t>(b) * hkv + g) * 2 + 0] = med;
    quant[(static_cast<size_t>(b) * hkv + g) * 2 + 1] = p90;
  }
  for (int j = threadIdx.x; j < nb; j += blockDim.x) {
    float a = 0.f;
    if (!degenerate) a = fminf(fmaxf((sr[j] - med) / span, 0.f), 1.f);
    alpha[base + j] = a;
  }
}

// ---------------------------------------------------------------- select

// Order-preserving 48-bit key: score bits on top (higher score = larger key),
// then 0xFFFF - j so that equal scores rank the lower block index first.
// Keys are unique within a row, so the k-th largest is a single element.
__device__ __forceinline__ uint64_t rank_key(float s, int j) {
  uint32_t u = __float_as_uint(s);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(u) << 16) | static_cast<uint64_t>(0xFFFFu - static_cast<uint32_t>(j));
}

struct SelectSmem {
  unsigned hist[256];
  unsigned long long bc_digit;
  unsigned bc_above;
  int wsum[kThreads / 32];
  int total;
};

// Exclusive prefix sum over the block; every thread passes its count.
__device__ int block_exclusive_scan(int v, SelectSmem &sm, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) sm.wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kThreads / 32 ? sm.wsum[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    if (lane < kThreads / 32) sm.wsum[lane] = wi - w;
    if (lane == kThreads / 32 - 1) sm.total = wi;
  }
  __syncthreads();
  const int res = sm.wsum[warp] + incl - v;
  *total = sm.total;
  __syncthreads();
  return res;
}

// Key of the k-th largest (1-based) eligible element of score[jlo, jhi).
// Requires 1 <= k <= number of eligible elements.  Radix select, 8-bit digits
// from the most significant end; called by the whole block.
template <typename Elig>
__device__ uint64_t radix_kth_largest(const float *score, int jlo, int jhi, Elig elig, int k,
                                      SelectSmem &sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t prefix = 0, pmask = 0;
  unsigned krem = static_cast<unsigned>(k);
  for (int shift = 40; shift >= 0; shift -= 8) {
    sm.hist[tid] = 0;  // kThreads == 256 bins
    __syncthreads();
    for (int base = jlo; base < jhi; base += kThreads) {
      const int j = base + tid;
      bool ok = j < jhi && elig(j);
      const uint64_t key = ok ? rank_key(score[j], j) : 0ull;
      ok = ok && ((key & pmask) == prefix);
      const unsigned digit = static_cast<unsigned>(key >> shift) & 255u;
      const unsigned peers = __match_any_sync(0xffffffffu, ok ? digit : 256u);
      if (ok && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[digit], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      unsigned c[8];
      unsigned s = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        c[e] = sm.hist[8 * lane + e];
        s += c[e];
      }
      unsigned suf = s;  // sum over lanes >= this lane
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned o = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += o;
      }
      unsigned acc = suf - s;  // elements in bins above this lane's bins
#pragma unroll
      for (int e = 7; e >= 0; --e) {
        if (acc < krem && krem <= acc + c[e]) {
          sm.bc_digit = static_cast<unsigned long long>(8 * lane + e);
          sm.bc_above = acc;
        }
        acc += c[e];
      }
    }
    __syncthreads();
    krem -= sm.bc_above;
    prefix |= static_cast<uint64_t>(sm.bc_digit) << shift;
    pmask |= 0xFFull << shift;
    __syncthreads();
  }
  return prefix;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) select_kernel(
    const uint16_t *__restrict__ q, const float *__restrict__ centroid,
    const float *__restrict__ radius, const float *__restrict__ alpha, int32_t *__restrict__ kv_idx,
    int32_t *__restrict__ kv_cnt, uint8_t *__restrict__ mask, int seq, int hq, int hkv, int block,
    int nb, long long ppm_c, long long ppm_r, float scale) {
  constexpr int VH = D / 8;    // 16-byte vectors per head row
  constexpr int VR = G * VH;   // vectors per token row of the group
  static_assert(VR <= kThreads && kThreads % VR == 0, "group row must fit the block");
  constexpr int RPP = kThreads / VR;  // token rows per pass

  extern __shared__ __align__(16) unsigned char smem[];
  float *psum = reinterpret_cast<float *>(smem);   // [RPP][G*D]
  float *pn = psum + RPP * G * D;                   // [RPP][G]
  float *qbt = pn + ((RPP * G + 3) & ~3);           // [D][G]  mean query, dimension-major
  float *nbar = qbt + D * G;                        // [G]
  float *sS = nbar + ((G + 3) & ~3);                // [nb] centroid-path score
  float *sR = sS + nb;                              // [nb] rescue-path score
  uint8_t *flags = reinterpret_cast<uint8_t *>(sR + nb);  // [nb]
  __shared__ SelectSmem sm;

  const int i = nb - 1 - static_cast<int>(blockIdx.x);  // longest rows first
  const int g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- query pooling: block i, heads g*G .. g*G+G-1 (G*D contiguous bf16 per token)
  {
    const int v = tid % VR, r0 = tid / VR, hh = v / VH;
    const size_t tok_stride = static_cast<size_t>(hq) * D;
    const uint16_t *base = q + (static_cast<size_t>(b) * seq + static_cast<size_t>(i) * block) * tok_stride +
                           static_cast<size_t>(g) * G * D + static_cast<size_t>(v) * 8;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    float nsum = 0.f;
    const int nrow = block / RPP;
#pragma unroll 4
    for (int it = 0; it < nrow; ++it) {
      const int t = r0 + it * RPP;
      const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(base + static_cast<size_t>(t) * tok_stride));
      float f[8];
      unpack_bf16x8(u, f);
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc[e] += f[e];
        sq = fmaf(f[e], f[e], sq);
      }
#pragma unroll
      for (int off = VH / 2; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      nsum += sqrtf(sq);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) psum[r0 * G * D + v * 8 + e] = acc[e];
    if (v % VH == 0) pn[r0 * G + hh] = nsum;
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += kThreads) {
    float s = 0.f;
    for (int r = 0; r < RPP; ++r) s += psum[r * G * D + e];
    const int hh = e / D, x = e - hh * D;
    qbt[x * G + hh] = s / static_cast<float>(block);
  }
  if (tid < G) {
    float s = 0.f;
    for (int r = 0; r < RPP; ++r) s += pn[r * G + tid];
    nbar[tid] = s / static_cast<float>(block);
  }
  for (int j = tid; j < nb; j += kThreads) flags[j] = 0;
  __syncthreads();

  // ---- scores for candidates j in [1, i-1]; thread tile = 4 key blocks x G heads
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const float *cbase = centroid + gb * D * nb;
  const float *rb = radius + gb * nb;
  const float *ab = alpha + gb * nb;
  for (int j0 = warp * 128; j0 < i; j0 += kThreads / 32 * 128) {
    const int jq = j0 + lane * 4;
    if (jq < i) {
      float acc[G][4];
#pragma unroll
      for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[hh][c] = 0.f;
      const float *cp = cbase + jq;
#pragma unroll 4
      for (int x = 0; x < D; ++x) {
        const float4 c4 = __ldg(reinterpret_cast<const float4 *>(cp + static_cast<size_t>(x) * nb));
        float qv[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int h4 = 0; h4 < G / 4; ++h4) {
            const float4 t = reinterpret_cast<const float4 *>(qbt + x * G)[h4];
            qv[4 * h4] = t.x;
            qv[4 * h4 + 1] = t.y;
            qv[4 * h4 + 2] = t.z;
            qv[4 * h4 + 3] = t.w;
          }
        } else {
#pragma unroll
          for (int hh = 0; hh < G; ++hh) qv[hh] = qbt[x * G + hh];
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          acc[hh][0] = fmaf(qv[hh], c4.x, acc[hh][0]);
          acc[hh][1] = fmaf(qv[hh], c4.y, acc[hh][1]);
          acc[hh][2] = fmaf(qv[hh], c4.z, acc[hh][2]);
          acc[hh][3] = fmaf(qv[hh], c4.w, acc[hh][3]);
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = jq + c;
        if (j >= 1 && j < i) {
          const float bonus = ab[j] * rb[j];
          float dm = acc[0][c];
          float rm = fmaf(nbar[0], bonus, acc[0][c]);
#pragma unroll
          for (int hh = 1; hh < G; ++hh) {
            dm = fmaxf(dm, acc[hh][c]);
            rm = fmaxf(rm, fmaf(nbar[hh], bonus, acc[hh][c]));
          }
          sS[j] = dm * scale;
          sR[j] = rm * scale;
        }
      }
    }
  }
  if (tid == 0) {
    flags[0] |= BSA_MASK_FORCED;
    flags[i] |= BSA_MASK_FORCED;
  }
  __syncthreads();

  // ---- centroid path: top kc of candidates 1..i-1 by S_c
  const int ncand = i > 1 ? i - 1 : 0;
  const long long kc_full = (ppm_c * (i + 1) + 999999LL) / 1000000LL;
  const int kc = static_cast<int>(kc_full < ncand ? kc_full : ncand);
  if (kc > 0) {
    uint64_t thr = 0;
    if (kc < ncand) thr = radix_kth_largest(sS, 1, i, [](int) { return true; }, kc, sm);
    for (int j = 1 + tid; j < i; j += kThreads)
      if (kc == ncand || rank_key(sS[j], j) >= thr) flags[j] |= BSA_MASK_CENTROID;
  }
  __syncthreads();

  // ---- rescue path: among the dropped candidates with alpha > 0, top kr by R
  auto eligible = [&](int j) { return !(flags[j] & BSA_MASK_CENTROID) && ab[j] > 0.f; };
  int my = 0;
  for (int j = 1 + tid; j < i; j += kThreads) my += eligible(j) ? 1 : 0;
  int nelig = 0;
  (void)block_exclusive_scan(my, sm, &nelig);
  const long long kr_full = (ppm_r * (i + 1) + 999999LL) / 1000000LL;
  const int kr = static_cast<int>(kr_full < nelig ? kr_full : nelig);
  if (kr > 0) {
    uint64_t thr = 0;
    if (kr < nelig) thr = radix_kth_largest(sR, 1, i, eligible, kr, sm);
    __syncthreads();  // every thread has evaluated eligible() before flags change
    for (int j = 1 + tid; j < i; j += kThreads)
      if (eligible(j) && (kr == nelig || rank_key(sR[j], j) >= thr)) flags[j] |= 0x80;
    __syncthreads();
    for (int j = 1 + tid; j < i; j += kThreads)
      if (flags[j] & 0x80) flags[j] = static_cast<uint8_t>((flags[j] & 0x7F) | BSA_MASK_RESCUE);
  }
  __syncthreads();

  // ---- emit the ascending kept list of row i and the optional mask row
  const int n = i + 1;
  const int chunk = (n + kThreads - 1) / kThreads;
  const int lo = min(tid * chunk, n), hi = min(lo + chunk, n);
  int cnt = 0;
  for (int j = lo; j < hi; ++j) cnt += flags[j] != 0;
  int total = 0;
  int off = block_exclusive_scan(cnt, sm, &total);
  int32_t *row = kv_idx + (gb * nb + i) * static_cast<size_t>(nb);
  for (int j = lo; j < hi; ++j)
    if (flags[j]) row[off++] = j;
  if (tid == 0) kv_cnt[gb * nb + i] = total;
  if (mask != nullptr) {
    uint8_t *mrow = mask + (gb * nb + i) * static_cast<size_t>(nb);
    for (int j = tid; j < nb; j += kThreads) mrow[j] = j <= i ? flags[j] : 0;
  }
}

template <int D, int G>
size_t select_smem_bytes(int nb) {
  constexpr int RPP = kThreads / (G * D / 8);
  size_t floats = static_cast<size_t>(RPP) * G * D + ((RPP * G + 3) & ~3) + D * G + ((G + 3) & ~3) +
                  2 * static_cast<size_t>(nb);
  return floats * 4 + static_cast<size_t>(nb);
}

template <int D, int G>
cudaError_t launch_select_t(const MaskShape &s, const void *q, const float *centroid,
                            const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                            float scale, int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask,
                            cudaStream_t stream) {
  const size_t smem = select_smem_bytes<D, G>(s.nb);
  cudaError_t e = cudaFuncSetAttribute(select_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(s.nb, s.hkv, s.batch);
  select_kernel<D, G><<<grid, kThreads, smem, stream>>>(
      static_cast<const uint16_t *>(q), centroid, radius, alpha, kv_idx, kv_cnt, mask, s.seq, s.hq,
      s.hkv, s.block, s.nb, static_cast<long long>(ppm_c), static_cast<long long>(ppm_r), scale);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_select_d(const MaskShape &s, const void *q, const float *c, const float *r,
                            const float *a, int64_t pc, int64_t pr, float scale, int32_t *idx,
                            int32_t *cnt, uint8_t *mask, cudaStream_t st) {
  switch (s.group) {
    case 1: return launch_select_t<D, 1>(s, q, c, r, a, pc, pr, scale, idx, cnt, mask, st);
    case 2: return launch_select_t<D, 2>(s, q, c, r, a, pc, pr, scale, idx, cnt, mask, st);
    case 4: return launch_select_t<D, 4>(s, q, c, r, a, pc, pr, scale, idx, cnt, mask, st);
    case 8: return launch_select_t<D, 8>(s, q, c, r, a, pc, pr, scale, idx, cnt, mask, st);
    case 16: return launch_select_t<D, 16>(s, q, c, r, a, pc, pr, scale, idx, cnt, mask, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_meta_d(const MaskShape &s, const void *k, float *centroid, float *radius,
                          cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(s.block) * D * 2 + static_cast<size_t>(kThreads / D) * D * 4;
  cudaError_t e = cudaFuncSetAttribute(meta_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(s.nb, s.hkv, s.batch);
  meta_kernel<D><<<grid, kThreads, smem, stream>>>(static_cast<const uint16_t *>(k), centroid, radius,
                                                   s.seq, s.hkv, s.block, s.nb);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_meta(const MaskShape &s, const void *k, float *centroid, float *radius,
                              cudaStream_t stream) {
  if (s.d == 64) return launch_meta_d<64>(s, k, centroid, radius, stream);
  if (s.d == 128) return launch_meta_d<128>(s, k, centroid, radius, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_quantiles(const MaskShape &s, const float *radius, float *quant, float *alpha,
                             cudaStream_t stream) {
  dim3 grid(s.hkv, s.batch);
  quant_kernel<<<grid, 1024, static_cast<size_t>(s.nb) * 4, stream>>>(radius, quant, alpha, s.nb);
  return cudaGetLastError();
}

cudaError_t launch_select(const MaskShape &s, const void *q, const float *centroid,
                          const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                          float scale, int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask,
                          cudaStream_t stream) {
  if (s.d == 64)
    return launch_select_d<64>(s, q, centroid, radius, alpha, ppm_c, ppm_r, scale, kv_idx, kv_cnt,
                               mask, stream);
  if (s.d == 128)
    return launch_select_d<128>(s, q, centroid, radius, alpha, ppm_c, ppm_r, scale, kv_idx, kv_cnt,
                                mask, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bsa
