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
//                   (streams K once)
//   quant_kernel    one CTA per (b, g): bitonic sort of the nb radii,
//                   nearest-rank median / p90, rescue coefficient alpha
//   qpool_kernel    one CTA per (b, i, head chunk): mean query and mean query
//                   norm of block i (streams Q once: the dominant HBM bytes)
//   score_kernel    (bsa_score.cu) centroid / rescue scores of every causal key
//                   block on tensor cores
//   select_kernel   one CTA per (b, g, i): per-path top-k by radix select, OR,
//                   ascending kept-list emission
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

  // block * VPR vectors, a multiple of kThreads for every supported (block, D)
  const int nvec = block * VPR;
  for (int e0 = 0; e0 < nvec; e0 += 8 * kThreads) {
    uint4 u[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int e = e0 + r * kThreads + tid;
      const int t = e / VPR, v = e - t * VPR;
      if (e < nvec)
        u[r] = __ldcs(reinterpret_cast<const uint4 *>(base + static_cast<size_t>(t) * tok_stride) + v);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int e = e0 + r * kThreads + tid;
      if (e < nvec) sk[e] = u[r];
    }
  }
  __syncthreads();

  const uint16_t *skh = reinterpret_cast<const uint16_t *>(sk);
  {
    // four interleaved partial sums per thread, combined in a fixed order
    const int x = tid % D, p = tid / D;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int t = p; t < block; t += 4 * P) {
      s0 += bf16_at(skh, t * D + x);
      s1 += bf16_at(skh, (t + P) * D + x);
      s2 += bf16_at(skh, (t + 2 * P) * D + x);
      s3 += bf16_at(skh, (t + 3 * P) * D + x);
    }
    part[p * D + x] = (s0 + s1) + (s2 + s3);
  }
  __syncthreads();
  if (tid < D) {
    float s = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) s += part[p * D + tid];
    const float c = s / static_cast<float>(block);
    sc[tid] = c;
    centroid[((static_cast<size_t>(b) * hkv + g) * nb + j) * D + tid] = c;
  }
  __syncthreads();

  const int warp = tid >> 5, lane = tid & 31;
  float best = 0.f;
  for (int t = warp * 4; t < block; t += kThreads / 32 * 4) {  // four rows per warp at a time
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int x = lane; x < D; x += 32) {
      const float cx = sc[x];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float dl = bf16_at(skh, (t + r) * D + x) - cx;
        acc[r] = fmaf(dl, dl, acc[r]);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
    best = fmaxf(best, fmaxf(fmaxf(acc[0], acc[1]), fmaxf(acc[2], acc[3])));
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

// Bitonic sort of the nb radii (padded with +inf to a power of two), then
// nearest-rank median / p90 and alpha.
__global__ void __launch_bounds__(1024) quant_kernel(const float *__restrict__ radius,
                                                     float *__restrict__ quant,
                                                     float *__restrict__ alpha, int nb, int npow2) {
  extern __shared__ float sr[];
  const int g = blockIdx.x, b = blockIdx.y, hkv = gridDim.x;
  const size_t base = (static_cast<size_t>(b) * hkv + g) * nb;
  for (int j = threadIdx.x; j < npow2; j += blockDim.x) sr[j] = j < nb ? radius[base + j] : INFINITY;
  __syncthreads();
  for (int kk = 2; kk <= npow2; kk <<= 1) {
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      for (int idx = threadIdx.x; idx < npow2; idx += blockDim.x) {
        const int ixj = idx ^ jj;
        if (ixj > idx) {
          const bool up = (idx & kk) == 0;
          const float a = sr[idx], c = sr[ixj];
          if ((a > c) == up) {
            sr[idx] = c;
            sr[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  // nearest rank (1-based): ceil(nb / 2) and ceil(9 nb / 10)
  const float med = sr[(nb + 1) / 2 - 1];
  const float p90 = sr[(9 * nb + 9) / 10 - 1];
  const float span = p90 - med;
  const bool degenerate = span <= 1e-12f * p90;
  if (threadIdx.x == 0) {
    quant[(static_cast<size_t>(b) * hkv + g) * 2 + 0] = med;
    quant[(static_cast<size_t>(b) * hkv + g) * 2 + 1] = p90;
  }
  for (int j = threadIdx.x; j < nb; j += blockDim.x) {
    float a = 0.f;
    if (!degenerate) a = fminf(fmaxf((radius[base + j] - med) / span, 0.f), 1.f);
    alpha[base + j] = a;
  }
}

// ---------------------------------------------------------------- query pooling

// One thread per (head, 8 dimensions); the token loop keeps 8 16-byte loads in
// flight per thread.  Writes qbar[b][g][i][hh][x] (one K-major row per (query
// block, head), the A operand of the score GEMM) and nbar[b][g][i][hh].
template <int D>
__global__ void __launch_bounds__(kThreads) qpool_kernel(const uint16_t *__restrict__ q,
                                                         float *__restrict__ qbar,
                                                         float *__restrict__ nbar, int seq,
                                                         int hq, int hkv, int block, int nb,
                                                         int hpc) {
  constexpr int VH = D / 8;  // lanes per head
  const int i = blockIdx.x, hc = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int hl = tid / VH, xv = tid - hl * VH;
  const int h = hc * hpc + hl;
  const size_t tok_stride = static_cast<size_t>(hq) * D;
  const uint16_t *base = q + (static_cast<size_t>(b) * seq + static_cast<size_t>(i) * block) * tok_stride +
                         static_cast<size_t>(h) * D + xv * 8;
  // lanes present in this warp (the last warp may be partial); a head's lanes never straddle warps
  const int present = min(32, static_cast<int>(blockDim.x) - (tid & ~31));
  const unsigned wmask = present >= 32 ? 0xffffffffu : ((1u << present) - 1u);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  float nsum = 0.f;
  for (int t0 = 0; t0 < block; t0 += 8) {
    uint4 u[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      u[r] = __ldcs(reinterpret_cast<const uint4 *>(base + static_cast<size_t>(t0 + r) * tok_stride));
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float f[8];
      unpack_bf16x8(u[r], f);
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
  const int grp = hq / hkv, g = h / grp, hh = h - g * grp;
  const size_t row = (static_cast<size_t>(b) * hkv + g) * nb + i;
  float4 *qb = reinterpret_cast<float4 *>(qbar + ((row * grp + hh) * D + xv * 8));
  const float inv_b = 1.f / static_cast<float>(block);  // exact: block is a power of two
  qb[0] = make_float4(acc[0] * inv_b, acc[1] * inv_b, acc[2] * inv_b, acc[3] * inv_b);
  qb[1] = make_float4(acc[4] * inv_b, acc[5] * inv_b, acc[6] * inv_b, acc[7] * inv_b);
  if (xv == 0) nbar[row * grp + hh] = nsum * inv_b;
}

// ---------------------------------------------------------------- select

// Order-preserving key of a float score: a higher score gives a larger key.
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelectSmem {
  unsigned hist[256];
  unsigned bc_digit, bc_above, bc_count;
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
    const int w = lane < kThreads / 32 ? sm.wsum[lane] : 0;
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

// Marks (flags |= bit) the k best eligible entries of score[1, i): higher score
// first, ties to the lower index.  Requires 1 <= k < number eligible.  Radix
// select over the 32-bit score key, 8-bit digits from the top; the rare case of
// several entries sharing the threshold key is settled by index order.
__device__ void mark_top_k(const float *score, const uint8_t *flags_in, uint8_t elig_bit,
                           uint8_t *flags, uint8_t bit, int i, int k, SelectSmem &sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, pmask = 0;
  unsigned krem = static_cast<unsigned>(k), n_eq = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    sm.hist[tid] = 0;  // kThreads == 256 bins
    __syncthreads();
    for (int base = 1; base < i; base += kThreads) {
      const int j = base + tid;
      bool ok = j < i && (flags_in[j] & elig_bit);
      const uint32_t key = ok ? score_key(score[j]) : 0u;
      ok = ok && ((key & pmask) == prefix);
      const unsigned digit = (key >> shift) & 255u;
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
      unsigned suf = s;  // elements in the bins of lanes >= this lane
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned o = __shfl_down_sync(0xffffffffu, suf, off);
        if (lane + off < 32) suf += o;
      }
      unsigned acc = suf - s;  // elements in bins above this lane's bins
#pragma unroll
      for (int e = 7; e >= 0; --e) {
        if (acc < krem && krem <= acc + c[e]) {
          sm.bc_digit = 8 * lane + e;
          sm.bc_above = acc;
          sm.bc_count = c[e];
        }
        acc += c[e];
      }
    }
    __syncthreads();
    krem -= sm.bc_above;
    n_eq = sm.bc_count;
    prefix |= sm.bc_digit << shift;
    pmask |= 0xFFu << shift;
    __syncthreads();
  }
  // keys above the threshold are in; krem of the n_eq keys equal to it are in
  if (n_eq == krem) {
    for (int j = 1 + tid; j < i; j += kThreads)
      if ((flags_in[j] & elig_bit) && score_key(score[j]) >= prefix) flags[j] |= bit;
  } else {
    for (int j = 1 + tid; j < i; j += kThreads)
      if ((flags_in[j] & elig_bit) && score_key(score[j]) > prefix) flags[j] |= bit;
    const int n = i - 1;
    const int chunk = (n + kThreads - 1) / kThreads;
    const int lo = 1 + min(tid * chunk, n), hi = min(lo + chunk, i);
    int cnt = 0;
    for (int j = lo; j < hi; ++j) cnt += (flags_in[j] & elig_bit) && score_key(score[j]) == prefix;
    int total = 0;
    int rank = block_exclusive_scan(cnt, sm, &total);
    for (int j = lo; j < hi; ++j)
      if ((flags_in[j] & elig_bit) && score_key(score[j]) == prefix) {
        if (rank < static_cast<int>(krem)) flags[j] |= bit;
        ++rank;
      }
  }
  __syncthreads();
}

constexpr uint8_t kCand = 0x40;  // candidate of the centroid path (1 <= j < i)
constexpr uint8_t kElig = 0x20;  // candidate of the rescue path

// One CTA per (b, g, i), longest rows first: load the row's scores (computed on
// tensor cores by the score kernel), rank each path, OR, emit the kept list.
__global__ void __launch_bounds__(kThreads) select_kernel(
    const float *__restrict__ s_c, const float *__restrict__ s_r, const float *__restrict__ alpha,
    int32_t *__restrict__ kv_idx, int32_t *__restrict__ kv_cnt, uint8_t *__restrict__ mask, int hkv,
    int nb, long long ppm_c, long long ppm_r) {
  extern __shared__ __align__(16) unsigned char smem[];
  float *sS = reinterpret_cast<float *>(smem);           // [nb] centroid-path score
  float *sR = sS + nb;                                   // [nb] rescue-path score
  uint8_t *flags = reinterpret_cast<uint8_t *>(sR + nb);  // [nb]
  __shared__ SelectSmem sm;

  const int i = nb - 1 - static_cast<int>(blockIdx.x);
  const int g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const size_t row = gb * nb + i;
  const float *ab = alpha + gb * nb;
  const float *rc = s_c + row * nb, *rr = s_r + row * nb;
  for (int j = tid; j < nb; j += kThreads) {
    uint8_t f = 0;
    if (j >= 1 && j < i) {
      sS[j] = rc[j];
      sR[j] = rr[j];
      f = kCand | (ab[j] > 0.f ? kElig : 0);  // eligibility is provisional: cleared if the centroid path keeps j
    }
    if (j == 0 || j == i) f |= BSA_MASK_FORCED;
    flags[j] = f;
  }
  __syncthreads();

  // ---- centroid path: top kc of candidates 1..i-1 by S_c
  const int ncand = i > 1 ? i - 1 : 0;
  const long long kc_full = (ppm_c * (i + 1) + 999999LL) / 1000000LL;
  const int kc = static_cast<int>(kc_full < ncand ? kc_full : ncand);
  if (kc == ncand) {
    for (int j = 1 + tid; j < i; j += kThreads) flags[j] |= BSA_MASK_CENTROID;
    __syncthreads();
  } else if (kc > 0) {
    mark_top_k(sS, flags, kCand, flags, BSA_MASK_CENTROID, i, kc, sm);
  }

  // ---- rescue path: among the dropped candidates with alpha > 0, top kr by R
  int my = 0;
  for (int j = 1 + tid; j < i; j += kThreads) {
    if (flags[j] & BSA_MASK_CENTROID) flags[j] &= static_cast<uint8_t>(~kElig);
    my += (flags[j] & kElig) ? 1 : 0;
  }
  int nelig = 0;
  (void)block_exclusive_scan(my, sm, &nelig);
  const long long kr_full = (ppm_r * (i + 1) + 999999LL) / 1000000LL;
  const int kr = static_cast<int>(kr_full < nelig ? kr_full : nelig);
  if (kr == nelig && kr > 0) {
    for (int j = 1 + tid; j < i; j += kThreads)
      if (flags[j] & kElig) flags[j] |= BSA_MASK_RESCUE;
    __syncthreads();
  } else if (kr > 0) {
    mark_top_k(sR, flags, kElig, flags, BSA_MASK_RESCUE, i, kr, sm);
  }

  // ---- emit the ascending kept list of row i and the optional mask row
  constexpr uint8_t kKeep = BSA_MASK_FORCED | BSA_MASK_CENTROID | BSA_MASK_RESCUE;
  const int n = i + 1;
  const int chunk = (n + kThreads - 1) / kThreads;
  const int lo = min(tid * chunk, n), hi = min(lo + chunk, n);
  int cnt = 0;
  for (int j = lo; j < hi; ++j) cnt += (flags[j] & kKeep) != 0;
  int total = 0;
  int off = block_exclusive_scan(cnt, sm, &total);
  int32_t *dst = kv_idx + row * static_cast<size_t>(nb);
  for (int j = lo; j < hi; ++j)
    if (flags[j] & kKeep) dst[off++] = j;
  if (tid == 0) kv_cnt[row] = total;
  if (mask != nullptr) {
    uint8_t *mrow = mask + row * static_cast<size_t>(nb);
    for (int j = tid; j < nb; j += kThreads) mrow[j] = j <= i ? (flags[j] & kKeep) : 0;
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


// Heads per query-pooling CTA: the largest divisor of hq with <= 256 threads.
int qpool_heads(int hq, int d) {
  int best = 1;
  for (int h = 1; h <= hq; ++h)
    if (hq % h == 0 && h * (d / 8) <= kThreads) best = h;
  return best;
}

template <int D>
cudaError_t launch_qpool_d(const MaskShape &s, const void *q, float *qbar, float *nbar,
                           cudaStream_t stream) {
  const int hpc = qpool_heads(s.hq, D);
  dim3 grid(s.nb, s.hq / hpc, s.batch);
  qpool_kernel<D><<<grid, hpc * (D / 8), 0, stream>>>(static_cast<const uint16_t *>(q), qbar, nbar,
                                                      s.seq, s.hq, s.hkv, s.block, s.nb, hpc);
  return cudaGetLastError();
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t select_workspace_bytes(const MaskShape &s) {
  const size_t rows = static_cast<size_t>(s.batch) * s.hq * s.nb;  // (b, g, i, h) rows
  const size_t scores = static_cast<size_t>(s.batch) * s.hkv * s.nb * s.nb;
  return round256(rows * s.d * 4) + round256(rows * 4) + 2 * round256(scores * 4);
}

cudaError_t launch_block_meta(const MaskShape &s, const void *k, float *centroid, float *radius,
                              cudaStream_t stream) {
  if (s.d == 64) return launch_meta_d<64>(s, k, centroid, radius, stream);
  if (s.d == 128) return launch_meta_d<128>(s, k, centroid, radius, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_quantiles(const MaskShape &s, const float *radius, float *quant, float *alpha,
                             cudaStream_t stream) {
  int npow2 = 1;
  while (npow2 < s.nb) npow2 <<= 1;
  dim3 grid(s.hkv, s.batch);
  const int threads = npow2 < 1024 ? (npow2 < 32 ? 32 : npow2) : 1024;
  quant_kernel<<<grid, threads, static_cast<size_t>(npow2) * 4, stream>>>(radius, quant, alpha, s.nb, npow2);
  return cudaGetLastError();
}

cudaError_t launch_select(const MaskShape &s, const void *q, const float *centroid,
                          const float *radius, const float *alpha, int64_t ppm_c, int64_t ppm_r,
                          float scale, int32_t *kv_idx, int32_t *kv_cnt, uint8_t *mask,
                          void *workspace, int32_t *status, cudaStream_t stream) {
  const size_t rows = static_cast<size_t>(s.batch) * s.hq * s.nb;
  const size_t scores = static_cast<size_t>(s.batch) * s.hkv * s.nb * s.nb;
  char *ws = static_cast<char *>(workspace);
  float *qbar = reinterpret_cast<float *>(ws);
  float *nbar = reinterpret_cast<float *>(ws + round256(rows * s.d * 4));
  float *s_c = reinterpret_cast<float *>(ws + round256(rows * s.d * 4) + round256(rows * 4));
  float *s_r = reinterpret_cast<float *>(reinterpret_cast<char *>(s_c) + round256(scores * 4));
  cudaError_t e;
  if (s.d == 64) e = launch_qpool_d<64>(s, q, qbar, nbar, stream);
  else if (s.d == 128) e = launch_qpool_d<128>(s, q, qbar, nbar, stream);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  e = launch_scores(s, qbar, nbar, centroid, radius, alpha, scale, s_c, s_r, status, stream);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(s.nb) * 9;
  e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(s.nb, s.hkv, s.batch);
  select_kernel<<<grid, kThreads, smem, stream>>>(s_c, s_r, alpha, kv_idx, kv_cnt, mask, s.hkv, s.nb,
                                                  static_cast<long long>(ppm_c),
                                                  static_cast<long long>(ppm_r));
  return cudaGetLastError();
}

}  // namespace bsa
