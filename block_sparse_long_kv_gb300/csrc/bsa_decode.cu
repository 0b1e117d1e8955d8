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
//   decode_score_kernel    32 key blocks per CTA, one warp per key block: the
//                          new token's G heads against the centroid row
//                          (coalesced), S_c and R into the workspace
//   decode_select_kernel   one 256-thread CTA per (b, g): the two-path exact
//                          top-k of a prefill row, CTA-wide (a histogram of
//                          the values, then radix digits of the keys in the
//                          threshold bin, as the prefill row code in
//                          bsa_topk.cuh does per warp; ties by index)
// Attention (bsa_decode_fwd), two launches:
//   decode_attn_kernel     as many CTAs as fit on the GPU (up to 1024): the kept
//                          entries of all rows (b, g) laid end to end and cut
//                          into equal runs, one per CTA, so a short batch and a
//                          mix of long and short sequences load every SM alike.
//                          A CTA streams its entries in 64-key chunks through a
//                          two-stage cp.async ring, computes the G heads'
//                          logits, an online softmax and P V on CUDA cores, and
//                          writes one unnormalised partial (O, max, sum) per row
//                          it touches
//   decode_combine_kernel  one CTA per (b, h): merges the row's partials
//                          (log-sum-exp) and writes O and LSE
// The cache is a packed batch (sequence b = tokens cu[b] .. cu[b+1]-1, its
// last token the new one), checked like every packed batch (seq_span).

#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "bsa_internal.h"
#include "bsa_topk.cuh"
#include "sm103_ptx.cuh"

namespace bsa {
namespace {

using namespace topk;

constexpr int kAttnThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// ---------------------------------------------------------------- selection

constexpr int kScoreWarps = 8;
constexpr int kScoreBlocksPerWarp = 4;  // key blocks per warp: 32 per CTA

// S_c[j] and R[j] of the new token of (b, g) for the candidates 1 <= j < i, one
// warp per key block (a coalesced centroid row per lane group), NW * R key
// blocks per chunk jt, so every SM takes part even at batch 1.  Each warp
// issues the loads of all its centroid rows before it reads the query, so a
// CTA waits for memory about once.  A key block's scores do not depend on NW.
template <int D, int NW>
__device__ __forceinline__ void decode_score_chunk(
    int jt, int g, int b, const uint16_t *__restrict__ q_new, const float *__restrict__ centroid,
    const float *__restrict__ radius, const float *__restrict__ alpha, float *__restrict__ s_c,
    float *__restrict__ s_r, const int32_t *__restrict__ cu, int seq, int total, int block, int hq, int hkv,
    int nbs, float scale, int32_t *status) {
  constexpr int DPL = D / 32;  // dimensions per lane
  constexpr int R = kScoreBlocksPerWarp;
  __shared__ __align__(16) float qs[16 * D];
  __shared__ float qn[16];
  const int grp = hq / hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  if (sp.len == 0) return;
  const int i = (sp.len - 1) / block;  // the new token's block
  const int j0 = jt * NW * R;
  if (j0 >= i) return;  // CTA-uniform
  const int jw = j0 + warp * R;
  float c[R][DPL];
  float bonus[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = jw + r;
    bonus[r] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) c[r][e] = 0.f;
    if (j >= 1 && j < i) {  // warp-uniform
      const float *crow = centroid + (gb * nbs + j) * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 v4 = *reinterpret_cast<const float4 *>(crow);
        c[r][0] = v4.x; c[r][1] = v4.y; c[r][2] = v4.z; c[r][3] = v4.w;
      } else {
        const float2 v2 = *reinterpret_cast<const float2 *>(crow);
        c[r][0] = v2.x; c[r][1] = v2.y;
      }
      bonus[r] = alpha[gb * nbs + j] * radius[gb * nbs + j];
    }
  }
  const uint16_t *qrow = q_new + (static_cast<size_t>(b) * hq + static_cast<size_t>(g) * grp) * D;
  for (int e = tid; e < grp * D; e += NW * 32) qs[e] = bf16f(qrow[e]);
  __syncthreads();
  for (int h = warp; h < grp; h += NW) {
    float s2 = 0.f;
    for (int x = lane; x < D; x += 32) s2 = fmaf(qs[h * D + x], qs[h * D + x], s2);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
    if (lane == 0) qn[h] = sqrtf(s2);
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = jw + r;
    if (j < 1 || j >= i) continue;  // warp-uniform
    float dm = -INFINITY, rm = -INFINITY;
    for (int h = 0; h < grp; ++h) {
      float p = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) p = fmaf(qs[h * D + lane * DPL + e], c[r][e], p);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
      dm = fmaxf(dm, p);
      rm = fmaxf(rm, fmaf(qn[h], bonus[r], p));
    }
    if (lane == 0) {
      s_c[gb * nbs + j] = dm * scale;
      s_r[gb * nbs + j] = rm * scale;
    }
  }
  __syncthreads();  // qs / qn are reused by the next chunk
}

template <int D>
__global__ void __launch_bounds__(kScoreWarps * 32) decode_score_kernel(
    const uint16_t *__restrict__ q_new, const float *__restrict__ centroid, const float *__restrict__ radius,
    const float *__restrict__ alpha, float *__restrict__ s_c, float *__restrict__ s_r,
    const int32_t *__restrict__ cu, int seq, int total, int block, int hq, int hkv, int nbs, float scale,
    int32_t *status) {
  decode_score_chunk<D, kScoreWarps>(blockIdx.x, blockIdx.y, blockIdx.z, q_new, centroid, radius, alpha, s_c, s_r,
                                     cu, seq, total, block, hq, hkv, nbs, scale, status);
}

// ---------------------------------------------------------------- CTA-wide selection
//
// One CTA of kSelThreads threads per (b, g).  Thread t holds the row entries
// j = t * E .. t * E + E - 1 (blocked order, so a CTA prefix sum over threads
// is a prefix sum in index order).  The exact top-k is the same two-stage
// select as the warp code: a 256-bin histogram of the candidates' values finds
// the threshold bin, then 8-bit radix digits of the order-preserving keys
// inside that bin; equal keys at the threshold are ranked by index.

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
static_assert(kMaxBlocks <= 16 * kSelThreads, "a row fits in sixteen entries per thread");

struct SelShared {
  unsigned hist[256];
  unsigned wsum[kSelWarps];
  float wlo[kSelWarps], whi[kSelWarps];
  unsigned bc[3];
};

// Sum over the CTA; every thread gets it.
__device__ __forceinline__ unsigned cta_sum(unsigned v, SelShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) sh.wsum[warp] = v;
  __syncthreads();
  unsigned t = lane < kSelWarps ? sh.wsum[lane] : 0u;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  __syncthreads();
  return t;
}

// Minimum and maximum over the CTA; every thread gets them.
__device__ __forceinline__ void cta_minmax(float &lo, float &hi, SelShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_minmax(lo, hi);
  if (lane == 0) {
    sh.wlo[warp] = lo;
    sh.whi[warp] = hi;
  }
  __syncthreads();
  lo = lane < kSelWarps ? sh.wlo[lane] : INFINITY;
  hi = lane < kSelWarps ? sh.whi[lane] : -INFINITY;
  warp_minmax(lo, hi);
  __syncthreads();
}

// Exclusive prefix sum over the threads in thread order; *total gets the sum.
__device__ __forceinline__ unsigned cta_exclusive_scan(unsigned c, unsigned *total, SelShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned wt;
  const unsigned ex = warp_exclusive_scan(c, &wt);
  if (lane == 0) sh.wsum[warp] = wt;
  __syncthreads();
  unsigned tot;
  const unsigned wex = warp_exclusive_scan(lane < kSelWarps ? sh.wsum[lane] : 0u, &tot);
  const unsigned off = __shfl_sync(0xffffffffu, wex, warp);
  __syncthreads();
  *total = tot;
  return off + ex;
}

// Warp 0 finds the bin of the take-th largest entry of sh.hist; every thread
// gets (bin, entries above it, its count) back.
__device__ __forceinline__ void cta_find_bin(unsigned take, unsigned *bin, unsigned *above, unsigned *count,
                                             SelShared &sh) {
  if (threadIdx.x < 32) {
    unsigned bn, ab, ct;
    warp_find_bin(sh.hist, take, &bn, &ab, &ct);
    if (threadIdx.x == 0) {
      sh.bc[0] = bn;
      sh.bc[1] = ab;
      sh.bc[2] = ct;
    }
  }
  __syncthreads();
  *bin = sh.bc[0];
  *above = sh.bc[1];
  *count = sh.bc[2];
}

__device__ __forceinline__ void cta_zero_hist(SelShared &sh) {
  if (threadIdx.x < 256) sh.hist[threadIdx.x] = 0u;
  __syncthreads();
}

// Bit e of the result: entry e of this thread is among the k best nonzero keys
// of the CTA (1 <= k < number of nonzero keys).  lo / hi: the CTA's range of the
// candidates' values.
template <int E>
__device__ unsigned cta_topk(const uint32_t (&key)[E], unsigned k, float lo, float hi, SelShared &sh) {
  float inv = 0.f;
  if (hi > lo) {
    const float x = 256.f / (hi - lo);
    if (x <= 1.0e38f) inv = x;
  }
  int bin[E];
#pragma unroll
  for (int e = 0; e < E; ++e) bin[e] = key[e] == 0u ? -1 : (inv > 0.f ? value_bin(key[e], lo, inv) : 0);
  cta_zero_hist(sh);
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (bin[e] >= 0) atomicAdd(&sh.hist[bin[e]], 1u);
  __syncthreads();
  unsigned bstar, above, count;
  cta_find_bin(k, &bstar, &above, &count, sh);
  unsigned take = k - above;
  unsigned sel = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (bin[e] > static_cast<int>(bstar) || (bin[e] == static_cast<int>(bstar) && count == take)) sel |= 1u << e;
  if (count == take) return sel;  // the whole threshold bin is in
  // radix digits of the keys inside the threshold bin, from the top
  uint32_t prefix = 0u, pmask = 0u;
  unsigned n_eq = count;
  for (int shift = 24; shift >= 0; shift -= 8) {
    cta_zero_hist(sh);
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (bin[e] == static_cast<int>(bstar) && (key[e] & pmask) == prefix)
        atomicAdd(&sh.hist[(key[e] >> shift) & 255u], 1u);
    __syncthreads();
    unsigned digit, ab2, ct2;
    cta_find_bin(take, &digit, &ab2, &ct2, sh);
    take -= ab2;
    n_eq = ct2;
    prefix |= digit << shift;
    pmask |= 0xFFu << shift;
    if (n_eq == take) break;  // CTA-uniform: every thread read the same values
  }
  unsigned eq = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (bin[e] != static_cast<int>(bstar)) continue;
    const uint32_t top = key[e] & pmask;
    if (top > prefix) sel |= 1u << e;
    else if (top == prefix) eq |= 1u << e;
  }
  if (n_eq == take) return sel | eq;
  // equal full keys at the threshold: the lowest indices first
  unsigned tot;
  unsigned rank = cta_exclusive_scan(__popc(eq), &tot, sh);
#pragma unroll
  for (int e = 0; e < E; ++e)
    if ((eq >> e) & 1u) {
      if (rank < take) sel |= 1u << e;
      ++rank;
    }
  return sel;
}

// The selection of one decode row per CTA: candidates 1..i-1, the top kc by
// S_c, then among the dropped candidates with alpha > 0 the top kr by R,
// blocks 0 and i forced; writes the ascending kept list and its length.
template <int E>
__global__ void __launch_bounds__(kSelThreads) decode_select_kernel(
    const float *__restrict__ s_c, const float *__restrict__ s_r, const float *__restrict__ alpha,
    int32_t *__restrict__ kv_idx, int32_t *__restrict__ kv_cnt, const int32_t *__restrict__ cu, int seq,
    int total, int block, int hkv, int nbs, long long ppm_c, long long ppm_r, int32_t *status) {
  __shared__ __align__(16) SelShared sh;
  const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  if (sp.len == 0) {
    if (tid == 0) kv_cnt[gb] = 0;
    return;
  }
  const int i = (sp.len - 1) / block;
  const float *rc = s_c + gb * nbs, *rr = s_r + gb * nbs, *ab = alpha + gb * nbs;
  const int jb = tid * E;

  // ---- centroid path
  uint32_t key[E];
  float lo = INFINITY, hi = -INFINITY;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = jb + e;
    const bool cand = j >= 1 && j < i;
    const float x = cand ? rc[j] : 0.f;
    key[e] = cand ? score_key(x) : 0u;
    if (cand) {
      lo = fminf(lo, x);
      hi = fmaxf(hi, x);
    }
  }
  const int ncand = i > 1 ? i - 1 : 0;
  const long long kc_full = (ppm_c * (i + 1) + 999999LL) / 1000000LL;
  const int kc = static_cast<int>(kc_full < ncand ? kc_full : ncand);
  unsigned cent = 0u;
  if (kc == ncand) {
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (key[e] != 0u) cent |= 1u << e;
  } else if (kc > 0) {
    cta_minmax(lo, hi, sh);
    cent = cta_topk<E>(key, static_cast<unsigned>(kc), lo, hi, sh);
  }

  // ---- rescue path
  lo = INFINITY;
  hi = -INFINITY;
  unsigned ne = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = jb + e;
    const bool elig = j >= 1 && j < i && ((cent >> e) & 1u) == 0u && ab[j] > 0.f;
    const float x = elig ? rr[j] : 0.f;
    key[e] = elig ? score_key(x) : 0u;
    ne += elig ? 1u : 0u;
    if (elig) {
      lo = fminf(lo, x);
      hi = fmaxf(hi, x);
    }
  }
  const int nelig = static_cast<int>(cta_sum(ne, sh));
  const long long kr_full = (ppm_r * (i + 1) + 999999LL) / 1000000LL;
  const int kr = static_cast<int>(kr_full < nelig ? kr_full : nelig);
  unsigned resc = 0u;
  if (kr > 0 && kr == nelig) {
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (key[e] != 0u) resc |= 1u << e;
  } else if (kr > 0) {
    cta_minmax(lo, hi, sh);
    resc = cta_topk<E>(key, static_cast<unsigned>(kr), lo, hi, sh);
  }

  // ---- emit the ascending list: forced 0 and i, then the two paths
  unsigned keep = cent | resc;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int j = jb + e;
    if (j == 0 || j == i) keep |= 1u << e;
  }
  unsigned kept;
  unsigned pos = cta_exclusive_scan(__popc(keep), &kept, sh);
  int32_t *dst = kv_idx + gb * nbs;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if ((keep >> e) & 1u) dst[pos++] = jb + e;
  if (tid == 0) kv_cnt[gb] = static_cast<int32_t>(kept);
}

// ---------------------------------------------------------------- attention

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's most recent cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kChunk = 64;       // keys per chunk
constexpr int kStages = 2;       // chunks in shared memory: the current one and the next in flight;
                                 // small enough for two CTAs per SM
constexpr int kMaxDecodeCtas = 1024;

template <int D, int G>
struct DecCfg {
  static constexpr int ROW = D * 2 + 16;   // padded key / value row (bytes): conflict-free fragment loads
  static constexpr int NKS = D / 16;       // k-steps of S = Q K^T
  static constexpr int NNT = D / 8;        // n-tiles of O = P V
  static constexpr size_t STAGE = static_cast<size_t>(kChunk) * ROW;  // keys or values of one chunk
  static constexpr size_t OFF_K = 0;
  static constexpr size_t OFF_V = OFF_K + kStages * STAGE;
  static constexpr size_t OFF_O = OFF_V + kStages * STAGE;                 // [warps][G][D] fp32
  static constexpr size_t OFF_ML = OFF_O + static_cast<size_t>(kAttnThreads / 32) * G * D * 4;  // [2][warps][16]
  static constexpr size_t OFF_ROWS = OFF_ML + 2 * (kAttnThreads / 32) * 16 * 4;
  // + (rows + 1) prefix counts and (rows + 1) partial offsets (int32)
  static size_t smem(int rows) { return OFF_ROWS + static_cast<size_t>(rows + 1) * 2 * 4; }
  static_assert(kChunk == 16 * (kAttnThreads / 32), "one 16-key slice of a chunk per warp");
  static_assert(G <= 16, "the heads of a group fill at most the 16 rows of one MMA");
};

// D = A B + C on the tensor cores, one warp, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 bf16 matrices from shared memory, transposed (lane l names row l % 8 of matrix l / 8).
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(row))));
}

// cp.async of 16 bytes that fills the destination with zeros (reads nothing).
__device__ __forceinline__ void cp_async16_zero(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

// CTA-wide exclusive prefix sum over the threads (kAttnThreads) in thread order.
__device__ __forceinline__ int block_exclusive_scan(int c, int *total, int *wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned wt;
  const unsigned ex = warp_exclusive_scan(static_cast<unsigned>(c), &wt);
  if (lane == 0) wsum[warp] = static_cast<int>(wt);
  __syncthreads();
  int off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kAttnThreads / 32; ++w) {
    off += w < warp ? wsum[w] : 0;
    tot += wsum[w];
  }
  __syncthreads();
  *total = tot;
  return off + static_cast<int>(ex);
}

// The kept entries of the rows (b, g) laid end to end: row r holds entries
// pre[r] .. pre[r+1]-1.  CTA c of C takes the W = ceil(N / C) entries c W ..,
// so each row is covered by a run of consecutive CTAs; the partial of (row r,
// CTA c) goes to slot off[r] + c - pre[r] / W.  Every CTA builds pre and off in
// shared memory (rows <= kMaxDecodeRows); CTA 0 also stores W and off for the
// combine.  Returns W (0 when no row keeps anything).
__device__ int decode_plan(const int32_t *kv_cnt, const int32_t *cu, int seq, int total, int block, int hkv,
                           int rows, int *pre, int *off, int *plan, int32_t *status, int *wsum) {
  const int tid = threadIdx.x;
  const int per = (rows + kAttnThreads - 1) / kAttnThreads;
  const int r0 = min(rows, tid * per), r1 = min(rows, r0 + per);
  int local = 0;
  for (int r = r0; r < r1; ++r) {
    const SeqSpan sp = seq_span(cu, r / hkv, seq, total, status);
    const int c = sp.len > 0 ? min(kv_cnt[r], (sp.len - 1) / block + 1) : 0;
    pre[r] = max(c, 0);  // the count for now; the prefix below
    local += max(c, 0);
  }
  int n;
  int run = block_exclusive_scan(local, &n, wsum);
  for (int r = r0; r < r1; ++r) {
    const int c = pre[r];
    pre[r] = run;
    run += c;
  }
  if (tid == 0) pre[rows] = n;
  __syncthreads();
  const int W = n > 0 ? (n + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) : 0;
  int parts = 0;
  for (int r = r0; r < r1; ++r) {
    const int a = pre[r], b = pre[r + 1];
    off[r] = b > a ? (b - 1) / W - a / W + 1 : 0;
    parts += off[r];
  }
  int np;
  run = block_exclusive_scan(parts, &np, wsum);
  for (int r = r0; r < r1; ++r) {
    const int c = off[r];
    off[r] = run;
    run += c;
  }
  if (tid == 0) off[rows] = np;
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int r = tid; r <= rows; r += kAttnThreads) plan[1 + r] = off[r];
    if (tid == 0) plan[0] = W;
  }
  return W;
}

// One chunk of keys: row r, first token (in the packed k / v) and key count.
struct DChunk {
  int r, tok, n;
};

// Walks the chunks of entries [x, x1) in order, skipping list entries that
// name no block of the row's sequence.  Every thread walks the same sequence.
struct DecWalk {
  int x, x1, r, c0, nk, jtok;
  int e0, rend, start, len, last;  // the row's first entry number, end, sequence and last block
  const int32_t *list;             // the row's kept list
  int pfx, pf;                     // entry pfx's block index, loaded ahead (pfx = -1: none)
};

__device__ __forceinline__ void walk_row(DecWalk &w, const int *pre, const int32_t *kv_idx, const int32_t *cu,
                                         int seq, int total, int block, int hkv, int nbs, int32_t *status) {
  while (w.x >= pre[w.r + 1]) ++w.r;  // rows with no entries are passed over
  w.e0 = pre[w.r];
  w.rend = pre[w.r + 1];
  const SeqSpan sp = seq_span(cu, w.r / hkv, seq, total, status);
  w.start = sp.start;
  w.len = sp.len;
  w.last = (sp.len - 1) / block;
  w.list = kv_idx + static_cast<size_t>(w.r) * nbs;
}

// Moves w to the next valid entry at or after w.x (c0 = 0); w.x == w.x1 when none is left.
// The block index of the entry after it is requested at once, so that its load is in flight
// while this entry's chunks stream.
__device__ __forceinline__ void walk_entry(DecWalk &w, const int *pre, const int32_t *kv_idx, const int32_t *cu,
                                           int seq, int total, int block, int hkv, int nbs, int32_t *status) {
  for (; w.x < w.x1; ++w.x) {
    if (w.x >= w.rend) walk_row(w, pre, kv_idx, cu, seq, total, block, hkv, nbs, status);
    const int j = w.x == w.pfx ? w.pf : w.list[w.x - w.e0];
    w.pfx = -1;
    if (w.x + 1 < w.x1 && w.x + 1 < w.rend) {
      w.pfx = w.x + 1;
      w.pf = w.list[w.x + 1 - w.e0];
    }
    if (j >= 0 && j <= w.last) {
      w.c0 = 0;
      w.nk = min(block, w.len - j * block);
      w.jtok = w.start + j * block;
      return;
    }
  }
}

// The chunk at w, then w advanced past it; r = -1 when the walk is over.
__device__ __forceinline__ DChunk walk_next(DecWalk &w, const int *pre, const int32_t *kv_idx, const int32_t *cu,
                                            int seq, int total, int block, int hkv, int nbs, int32_t *status) {
  if (w.x >= w.x1) return DChunk{-1, 0, 0};
  const DChunk c{w.r, w.jtok + w.c0, min(kChunk, w.nk - w.c0)};
  w.c0 += kChunk;
  if (w.c0 >= w.nk) {
    ++w.x;
    walk_entry(w, pre, kv_idx, cu, seq, total, block, hkv, nbs, status);
  }
  return c;
}

// Split-KV decode attention over the plan above.  CTA c walks its entries in
// chunks of 64 keys through a two-stage cp.async ring (a chunk's keys and
// values are one group; the next chunk is in flight while one is computed,
// and the ring is small enough for two CTAs per SM).
// Each warp owns 16 keys of a chunk and keeps its own online softmax: the G
// heads of the row are the rows of a 16 x 8 x 16 bf16 tensor-core MMA, so
// S = Q K^T is two n-tiles of 8 keys over D / 16 k-steps (Q held as A
// fragments in registers), and O += P V is one k-step of the warp's 16 keys
// over D / 8 n-tiles (P repacked from the S accumulators, V fragments by
// transposing matrix loads).  When the walk enters a new row (b, g) the
// warps' partials of the previous row are merged in shared memory and written
// to its slot (unnormalised O, max and sum in log2 units).  A slot whose
// entries name no valid block keeps max -inf, which the combine skips.
template <int D, int G>
__device__ __forceinline__ void decode_attn_run(
    const uint16_t *__restrict__ q_new, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const int32_t *__restrict__ kv_idx, const int32_t *__restrict__ kv_cnt, float *__restrict__ part_o,
    float *__restrict__ part_ml, int *__restrict__ plan, const int32_t *__restrict__ cu, int seq, int total,
    int block, int hkv, int nbs, int rows, float scale_log2, int32_t *status, unsigned char *smem) {
  using C = DecCfg<D, G>;
  constexpr int NW = kAttnThreads / 32;
  float (*oacc)[G][D] = reinterpret_cast<float (*)[G][D]>(smem + C::OFF_O);
  float (*wm)[16] = reinterpret_cast<float (*)[16]>(smem + C::OFF_ML);  // [warp][head]: max
  float (*wl)[16] = wm + NW;                                             // [warp][head]: sum
  int *pre = reinterpret_cast<int *>(smem + C::OFF_ROWS);
  int *off = pre + rows + 1;
  __shared__ int wsum[NW];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;  // MMA fragment row group and column pair
  const int hq = hkv * G;
  const int c = blockIdx.x;
  const int W = decode_plan(kv_cnt, cu, seq, total, block, hkv, rows, pre, off, plan, status, wsum);
  const int n_all = pre[rows];
  const int x0 = c * W, x1 = min(n_all, x0 + W);
  if (x0 >= x1) return;  // CTA-uniform

  // the row holding entry x0: the last r with pre[r] <= x0
  int lo = 0, hi = rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x0) lo = mid;
    else hi = mid - 1;
  }
  auto slot_of = [&](int r) { return off[r] + c - pre[r] / W; };
  // every slot of this CTA starts empty (a flush below overwrites it)
  for (int r = lo + tid; r < rows && pre[r] < x1; r += kAttnThreads)
    if (pre[r + 1] > pre[r])
      for (int h = 0; h < G; ++h)
        *reinterpret_cast<float2 *>(part_ml + (static_cast<size_t>(slot_of(r)) * G + h) * 2) =
            make_float2(-INFINITY, 0.f);

  DecWalk w;
  w.x = x0;
  w.x1 = x1;
  w.r = lo;
  w.pfx = -1;
  walk_row(w, pre, kv_idx, cu, seq, total, block, hkv, nbs, status);
  walk_entry(w, pre, kv_idx, cu, seq, total, block, hkv, nbs, status);

  constexpr int PR = D * 2 / 16;  // 16-byte pieces per key or value row
  auto issue = [&](const DChunk &ch, int stage) {
    if (ch.r >= 0) {
      const size_t gofs = static_cast<size_t>(ch.r % hkv) * D;
      unsigned char *kst = smem + C::OFF_K + stage * C::STAGE;
      unsigned char *vst = smem + C::OFF_V + stage * C::STAGE;
      for (int x = tid; x < kChunk * PR; x += kAttnThreads) {
        const int r = x / PR, pc = x - r * PR;
        if (r < ch.n) {
          const size_t src = (static_cast<size_t>(ch.tok) + r) * hkv * D + gofs + pc * 8;
          cp_async16(kst + r * C::ROW + pc * 16, k + src);
          cp_async16(vst + r * C::ROW + pc * 16, v + src);
        } else {
          // past the chunk's keys: zero values, so that P = 0 meets finite numbers in P V
          cp_async16_zero(vst + r * C::ROW + pc * 16, v);
        }
      }
    }
    cp_async_commit();  // one group per chunk, empty past the end of the walk
  };

  uint32_t qa[C::NKS][4];  // Q as A fragments: rows gq and gq + 8 are heads of the group
  float o[C::NNT][4];      // O accumulators: heads gq (0, 1) and gq + 8 (2, 3), dims 8 nt + 2 tq
  float m_lo = -INFINITY, m_hi = -INFINITY;  // running max (log2 units) over this warp's keys
  float l_lo = 0.f, l_hi = 0.f;              // this thread's share of the sums
  int arow = -1;

  auto start_row = [&](int r) {
    const uint16_t *qb = q_new + (static_cast<size_t>(r / hkv) * hq + static_cast<size_t>(r % hkv) * G) * D;
    auto ld = [&](int h, int col) -> uint32_t {
      return h < G ? *reinterpret_cast<const uint32_t *>(qb + static_cast<size_t>(h) * D + col) : 0u;
    };
#pragma unroll
    for (int ks = 0; ks < C::NKS; ++ks) {
      const int col = 16 * ks + 2 * tq;
      qa[ks][0] = ld(gq, col);
      qa[ks][1] = ld(gq + 8, col);
      qa[ks][2] = ld(gq, col + 8);
      qa[ks][3] = ld(gq + 8, col + 8);
    }
#pragma unroll
    for (int nt = 0; nt < C::NNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    m_lo = m_hi = -INFINITY;
    l_lo = l_hi = 0.f;
  };

  auto flush = [&](int r) {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    if (tq == 0) {
      wm[warp][gq] = m_lo;
      wm[warp][gq + 8] = m_hi;
      wl[warp][gq] = l_lo;
      wl[warp][gq + 8] = l_hi;
    }
    __syncthreads();
    float mlo = -INFINITY, mhi = -INFINITY;
#pragma unroll
    for (int x = 0; x < NW; ++x) {
      mlo = fmaxf(mlo, wm[x][gq]);
      mhi = fmaxf(mhi, wm[x][gq + 8]);
    }
    const float slo = m_lo == -INFINITY ? 0.f : exp2f(m_lo - mlo);
    const float shi = m_hi == -INFINITY ? 0.f : exp2f(m_hi - mhi);
#pragma unroll
    for (int nt = 0; nt < C::NNT; ++nt) {
      if (gq < G)
        *reinterpret_cast<float2 *>(&oacc[warp][gq][8 * nt + 2 * tq]) = make_float2(o[nt][0] * slo, o[nt][1] * slo);
      if (gq + 8 < G)
        *reinterpret_cast<float2 *>(&oacc[warp][gq + 8][8 * nt + 2 * tq]) =
            make_float2(o[nt][2] * shi, o[nt][3] * shi);
    }
    __syncthreads();
    const size_t sl = static_cast<size_t>(slot_of(r));
    for (int e = tid; e < G * D / 2; e += kAttnThreads) {
      const int h = e / (D / 2), d2 = 2 * (e % (D / 2));
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int x = 0; x < NW; ++x) {
        a0 += oacc[x][h][d2];
        a1 += oacc[x][h][d2 + 1];
      }
      *reinterpret_cast<float2 *>(part_o + (sl * G + h) * D + d2) = make_float2(a0, a1);
    }
    if (tid < G) {
      float m = -INFINITY, l = 0.f;
#pragma unroll
      for (int x = 0; x < NW; ++x) m = fmaxf(m, wm[x][tid]);
#pragma unroll
      for (int x = 0; x < NW; ++x)
        if (wm[x][tid] != -INFINITY) l = fmaf(exp2f(wm[x][tid] - m), wl[x][tid], l);
      *reinterpret_cast<float2 *>(part_ml + (sl * G + tid) * 2) = make_float2(m, l);
    }
    __syncthreads();
  };

  // this lane's row addresses for the transposing value loads: matrix lane / 8 of a pair of
  // n-tiles is keys (lane / 8) % 2 * 8 .. + 7 of the warp's 16, dims (lane / 16) * 8 .. + 7
  const int vkey = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
  const int vcol = (lane >> 4) * 8;

  // chunks u .. u + kStages - 2 are in flight at the top of step u; ring[] holds their rows
  DChunk ring[kStages - 1];
#pragma unroll
  for (int x = 0; x < kStages - 1; ++x) {
    ring[x] = walk_next(w, pre, kv_idx, cu, seq, total, block, hkv, nbs, status);
    issue(ring[x], x);
  }
  for (int u = 0; ring[0].r >= 0; ++u) {  // CTA-uniform: every thread walks the same chunks
    const DChunk cur = ring[0];
#pragma unroll
    for (int x = 0; x < kStages - 2; ++x) ring[x] = ring[x + 1];
    ring[kStages - 2] = walk_next(w, pre, kv_idx, cu, seq, total, block, hkv, nbs, status);
    issue(ring[kStages - 2], (u + kStages - 1) % kStages);  // the stage of chunk u-1, free since its step
    cp_async_wait<kStages - 1>();  // chunk u has landed (the later ones may be in flight)
    __syncthreads();
    if (cur.r != arow) {
      if (arow >= 0) flush(arow);
      start_row(cur.r);
      arow = cur.r;
    }
    const int stage = u % kStages;
    const unsigned char *kst = smem + C::OFF_K + stage * C::STAGE;
    const unsigned char *vst = smem + C::OFF_V + stage * C::STAGE;

    // ---- S = Q K^T for this warp's 16 keys (two n-tiles of 8)
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    const unsigned char *krow = kst + (warp * 16 + gq) * C::ROW + 4 * tq;
#pragma unroll
    for (int ks = 0; ks < C::NKS; ++ks) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const unsigned char *kp = krow + nt * 8 * C::ROW + 32 * ks;
        mma_bf16_16816(s[nt], qa[ks], *reinterpret_cast<const uint32_t *>(kp),
                       *reinterpret_cast<const uint32_t *>(kp + 16));
      }
    }

    // ---- online softmax per head over the warp's keys (log2 units)
    float x[2][4];
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = warp * 16 + nt * 8 + 2 * tq + (e & 1);
        x[nt][e] = key < cur.n ? s[nt][e] * scale_log2 : -INFINITY;
        if (e < 2) mx_lo = fmaxf(mx_lo, x[nt][e]);
        else mx_hi = fmaxf(mx_hi, x[nt][e]);
      }
#pragma unroll
    for (int offs = 1; offs <= 2; offs <<= 1) {
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, offs));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, offs));
    }
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float f_lo = m_lo == -INFINITY ? 0.f : exp2f(m_lo - mn_lo);
    const float f_hi = m_hi == -INFINITY ? 0.f : exp2f(m_hi - mn_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    float p[2][4];
    float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mref = e < 2 ? mn_lo : mn_hi;
        p[nt][e] = x[nt][e] == -INFINITY ? 0.f : exp2f(x[nt][e] - mref);
        if (e < 2) ps_lo += p[nt][e];
        else ps_hi += p[nt][e];
      }
    l_lo = fmaf(l_lo, f_lo, ps_lo);
    l_hi = fmaf(l_hi, f_hi, ps_hi);
    if (f_lo != 1.f || f_hi != 1.f) {
#pragma unroll
      for (int nt = 0; nt < C::NNT; ++nt) {
        o[nt][0] *= f_lo;
        o[nt][1] *= f_lo;
        o[nt][2] *= f_hi;
        o[nt][3] *= f_hi;
      }
    }

    // ---- O += P V over the warp's 16 keys
    const uint32_t pa[4] = {ptx::pack_bf16x2(p[0][0], p[0][1]), ptx::pack_bf16x2(p[0][2], p[0][3]),
                            ptx::pack_bf16x2(p[1][0], p[1][1]), ptx::pack_bf16x2(p[1][2], p[1][3])};
    const unsigned char *vrow = vst + vkey * C::ROW + vcol * 2;
#pragma unroll
    for (int np = 0; np < C::NNT / 2; ++np) {
      uint32_t vb[4];
      ldmatrix_x4_trans(vb, vrow + np * 32);
      mma_bf16_16816(o[2 * np], pa, vb[0], vb[1]);
      mma_bf16_16816(o[2 * np + 1], pa, vb[2], vb[3]);
    }
    __syncthreads();  // every warp is done with the stage before it is refilled
  }
  cp_async_wait<0>();  // only empty groups can remain
  if (arow >= 0) flush(arow);
}

template <int D, int G>
__global__ void __launch_bounds__(kAttnThreads) decode_attn_kernel(
    const uint16_t *__restrict__ q_new, const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
    const int32_t *__restrict__ kv_idx, const int32_t *__restrict__ kv_cnt, float *__restrict__ part_o,
    float *__restrict__ part_ml, int *__restrict__ plan, const int32_t *__restrict__ cu, int seq, int total,
    int block, int hkv, int nbs, int rows, float scale_log2, int32_t *status) {
  extern __shared__ __align__(16) unsigned char smem[];
  decode_attn_run<D, G>(q_new, k, v, kv_idx, kv_cnt, part_o, part_ml, plan, cu, seq, total, block, hkv, nbs, rows,
                        scale_log2, status, smem);
}

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;  // the merge order: 8 warp partials

// O and LSE of head h of sequence b: O = sum_s w_s O_s / sum_s w_s l_s over the
// slots of the head's row, w_s = 2^(m_s - max m) (slots with max -inf are
// empty).  The merge runs in a fixed order of kCombineWarps partials: partial
// w takes the slots w, w + 8, w + 16, ... (each lane D/32 dimensions), and the
// partials are added in order 0..7.  A CTA of NWR warps computes the partials
// w = warp, warp + NWR, ..., so the result does not depend on NWR.
template <int D, int NWR>
__device__ __forceinline__ void combine_head(int b, int h, const float *__restrict__ part_o,
                                             const float *__restrict__ part_ml, const int *__restrict__ plan,
                                             uint16_t *__restrict__ o, float *__restrict__ lse, int hq, int hkv) {
  constexpr int VL = D / 32;  // dimensions per lane
  __shared__ __align__(16) float red_o[kCombineWarps][D];
  __shared__ float red_l[kCombineWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = hq / hkv;
  const int r = b * hkv + h / grp, hl = h % grp;
  const int s0 = plan[1 + r], ns = plan[2 + r] - s0;
  float m = -INFINITY;
  for (int s = lane; s < ns; s += 32) m = fmaxf(m, part_ml[(static_cast<size_t>(s0 + s) * grp + hl) * 2]);
#pragma unroll
  for (int offs = 16; offs > 0; offs >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, offs));
  for (int vw = warp; vw < kCombineWarps; vw += NWR) {
    float acc[VL];
#pragma unroll
    for (int x = 0; x < VL; ++x) acc[x] = 0.f;
    float l = 0.f;
    for (int sb = vw; sb < ns; sb += 4 * kCombineWarps) {
      float2 ml[4];
      float pv[4][VL];
#pragma unroll
      for (int uu = 0; uu < 4; ++uu) {
        const int s = sb + uu * kCombineWarps;
        ml[uu] = make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int x = 0; x < VL; ++x) pv[uu][x] = 0.f;
        if (s < ns) {
          const size_t at = static_cast<size_t>(s0 + s) * grp + hl;
          ml[uu] = *reinterpret_cast<const float2 *>(part_ml + at * 2);
          const float *src = part_o + at * D + lane * VL;
          if constexpr (VL == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(src);
            pv[uu][0] = t.x; pv[uu][1] = t.y; pv[uu][2] = t.z; pv[uu][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2 *>(src);
            pv[uu][0] = t.x; pv[uu][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int uu = 0; uu < 4; ++uu) {
        if (ml[uu].x == -INFINITY) continue;  // an empty slot (or past ns)
        const float wgt = exp2f(ml[uu].x - m);
        l = fmaf(ml[uu].y, wgt, l);
#pragma unroll
        for (int x = 0; x < VL; ++x) acc[x] = fmaf(pv[uu][x], wgt, acc[x]);
      }
    }
#pragma unroll
    for (int x = 0; x < VL; ++x) red_o[vw][lane * VL + x] = acc[x];
    if (lane == 0) red_l[vw] = l;
  }
  __syncthreads();
  for (int d = tid; d < D; d += NWR * 32) {
    float a = 0.f, ls = 0.f;
#pragma unroll
    for (int wi = 0; wi < kCombineWarps; ++wi) {
      a += red_o[wi][d];
      ls += red_l[wi];
    }
    const float rr = ls > 0.f ? a / ls : 0.f;
    const __nv_bfloat16 rb = __float2bfloat16_rn(rr);
    o[(static_cast<size_t>(b) * hq + h) * D + d] = *reinterpret_cast<const uint16_t *>(&rb);
    if (lse != nullptr && d == 0)
      lse[static_cast<size_t>(b) * hq + h] = ls > 0.f ? (m + log2f(ls)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();  // red_o / red_l are reused by the next head
}

// One CTA per (b, h).
template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_ml, const int *__restrict__ plan,
    uint16_t *__restrict__ o, float *__restrict__ lse, int hq, int hkv) {
  combine_head<D, kCombineWarps>(blockIdx.y, blockIdx.x, part_o, part_ml, plan, o, lse, hq, hkv);
}

// ---------------------------------------------------------------- the whole step in one launch

// Grid-wide barrier k (k = 1, 2, ...) of a cooperative launch (every CTA is
// resident): each CTA adds 1 to bar[0] with release semantics and waits until
// it reads k * gridDim.x with acquire semantics, so every write before the
// barrier is visible to every CTA after it.  bar[0] is zero before the launch
// and is never reset inside it (barrier k's target follows from k).  The wait is
// bounded: after kGridWaitNs it records BSA_ERR_DEVICE_TIMEOUT and returns, so
// no CTA hangs.
constexpr uint64_t kGridWaitNs = 2000000000ull;

__device__ __forceinline__ void grid_sync(unsigned *bar, unsigned k, int32_t *status) {
  __threadfence();  // every thread's writes, before the CTA's arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
    const unsigned target = k * gridDim.x;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
      unsigned seen;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(seen) : "l"(bar) : "memory");
      if (seen >= target) break;
      __nanosleep(32);
      if (ptx::globaltimer_ns() - t0 > kGridWaitNs) {
        if (status != nullptr) atomicCAS(status, 0, BSA_ERR_DEVICE_TIMEOUT);
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
}

struct DecStepArgs {
  const uint16_t *q_new, *k, *v;
  const float *centroid, *radius, *alpha;
  int32_t *kv_idx, *kv_cnt;
  float *s_c, *s_r, *part_o, *part_ml;
  int *plan;
  unsigned *bar;
  uint16_t *o;
  float *lse;
  const int32_t *cu;
  int batch, seq, total, block, hq, hkv, nbs;
  long long ppm_c, ppm_r;
  float scale, scale_log2;
  int32_t *status;
};

// The selection of row r = (b, g) by the CTA as one team of warps (P row entries
// per lane, 32 NW P >= nbs): topk::team_select_row, exactly the selection of a
// prefill row i = (len - 1) / B.
template <int NW, int P>
__device__ __forceinline__ void decode_select_team(int r, const DecStepArgs &a) {
  __shared__ __align__(16) TeamScratch tsh;
  Team<NW> tm(tsh, 1, static_cast<int>(threadIdx.x));
  const int b = r / a.hkv;
  const size_t gb = static_cast<size_t>(r);
  const SeqSpan sp = seq_span(a.cu, b, a.seq, a.total, a.status);
  if (sp.len == 0) {
    if (threadIdx.x == 0) a.kv_cnt[gb] = 0;
    return;
  }
  const int i = (sp.len - 1) / a.block;
  tm.clear_hist();
  tm.sync();
  uint32_t fl[P / 4];
  team_select_row<Team<NW>, P, true>(tm, a.s_c + gb * a.nbs, a.s_r + gb * a.nbs, a.alpha + gb * a.nbs, i, a.ppm_c,
                               a.ppm_r, fl);
  team_emit_row<Team<NW>, P, true>(tm, fl, i, a.kv_idx + gb * a.nbs, a.kv_cnt + gb, nullptr, a.nbs);
  tm.sync();  // the scratch is reused by the next row
}

// One decode step in one cooperative launch:
//   scores     chunks of key blocks of every row (b, g) over every CTA; the CTA
//              that finishes a row's last chunk with candidates (counted in
//              bar[1 + r]) runs that row's selection, so no barrier separates
//              the two
//   | barrier 1 | split-KV attention (the even cut of decode_attn_run)
//   | barrier 2 | merge (one head per CTA).
// The same arithmetic as the four-launch path.  bar holds 1 + rows zeroed words.
template <int D, int G>
__global__ void __launch_bounds__(kAttnThreads) decode_step_kernel(const __grid_constant__ DecStepArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int row_done;
  constexpr int NW = kAttnThreads / 32;
  const int rows = a.batch * a.hkv;
  // the rows' chunks that hold candidates (j0 < i; always chunk 0), laid end to end: row r owns
  // items pre[r] .. pre[r+1]-1, and CTA c takes items c, c + gridDim.x, ..., so the work of short
  // and long rows spreads over all CTAs at once
  int *pre = reinterpret_cast<int *>(smem);  // rows + 1 entries; the attention phase reuses it
  __shared__ int wsum[NW];
  {
    const int per = (rows + kAttnThreads - 1) / kAttnThreads;
    const int r0 = min(rows, static_cast<int>(threadIdx.x) * per), r1 = min(rows, r0 + per);
    int local = 0;
    for (int r = r0; r < r1; ++r) {
      const SeqSpan sp = seq_span(a.cu, r / a.hkv, a.seq, a.total, a.status);
      const int i = sp.len > 0 ? (sp.len - 1) / a.block : -1;
      pre[r] = max(1, (i + NW * kScoreBlocksPerWarp - 1) / (NW * kScoreBlocksPerWarp));
      local += pre[r];
    }
    int n;
    int run = block_exclusive_scan(local, &n, wsum);
    for (int r = r0; r < r1; ++r) {
      const int c = pre[r];
      pre[r] = run;
      run += c;
    }
    if (threadIdx.x == 0) pre[rows] = n;
    __syncthreads();
  }
  for (int item = blockIdx.x; item < pre[rows]; item += gridDim.x) {
    int lo = 0, hi = rows - 1;  // the row holding item: the last r with pre[r] <= item
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= item) lo = mid;
      else hi = mid - 1;
    }
    const int r = lo, jt = item - pre[r], counted = pre[r + 1] - pre[r];
    decode_score_chunk<D, NW>(jt, r % a.hkv, r / a.hkv, a.q_new, a.centroid, a.radius, a.alpha, a.s_c, a.s_r,
                              a.cu, a.seq, a.total, a.block, a.hq, a.hkv, a.nbs, a.scale, a.status);
    __threadfence();  // this chunk's scores before its count
    __syncthreads();
    if (threadIdx.x == 0) row_done = atomicAdd(a.bar + 1 + r, 1u) == static_cast<unsigned>(counted - 1);
    __syncthreads();
    if (row_done) {  // CTA-uniform
      __threadfence();
      if (a.nbs <= 32 * NW * 8) decode_select_team<NW, 8>(r, a);
      else if (a.nbs <= 32 * NW * 16) decode_select_team<NW, 16>(r, a);
      else decode_select_team<NW, 32>(r, a);
    }
  }
  grid_sync(a.bar, 1, a.status);
  decode_attn_run<D, G>(a.q_new, a.k, a.v, a.kv_idx, a.kv_cnt, a.part_o, a.part_ml, a.plan, a.cu, a.seq, a.total,
                        a.block, a.hkv, a.nbs, rows, a.scale_log2, a.status, smem);
  grid_sync(a.bar, 2, a.status);
  for (int item = blockIdx.x; item < a.batch * a.hq; item += gridDim.x)
    combine_head<D, NW>(item / a.hq, item % a.hq, a.part_o, a.part_ml, a.plan, a.o, a.lse, a.hq, a.hkv);
}

template <int D, int G>
cudaError_t launch_attn_g(const MaskShape &s, const void *q_new, const void *k, const void *v,
                          const int32_t *kv_idx, const int32_t *kv_cnt, float *po, float *pml, int *plan,
                          float scale_log2, int32_t *status, cudaStream_t stream) {
  using C = DecCfg<D, G>;
  auto kern = decode_attn_kernel<D, G>;
  const int rows = s.batch * s.hkv;
  const size_t smem = C::smem(rows);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kAttnThreads, smem)) != cudaSuccess)
    return e;
  const int ctas = std::max(1, std::min(kMaxDecodeCtas, sms * std::max(per_sm, 1)));
  kern<<<ctas, kAttnThreads, smem, stream>>>(
      static_cast<const uint16_t *>(q_new), static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v),
      kv_idx, kv_cnt, po, pml, plan, s.cu, s.seq, s.total, s.block, s.hkv, s.nbs, rows, scale_log2, status);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_attn_d(const MaskShape &s, const void *q_new, const void *k, const void *v,
                          const int32_t *kv_idx, const int32_t *kv_cnt, float *po, float *pml, int *plan,
                          float scale_log2, int32_t *status, cudaStream_t st) {
  switch (s.group) {
    case 1: return launch_attn_g<D, 1>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, plan, scale_log2, status, st);
    case 2: return launch_attn_g<D, 2>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, plan, scale_log2, status, st);
    case 4: return launch_attn_g<D, 4>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, plan, scale_log2, status, st);
    case 8: return launch_attn_g<D, 8>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, plan, scale_log2, status, st);
    case 16: return launch_attn_g<D, 16>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, plan, scale_log2, status, st);
    default: return cudaErrorInvalidValue;
  }
}

// Workspace regions (each 256-byte aligned): partial O [slots, G, d] and partial (max, sum)
// [slots, G, 2] with slots = kMaxDecodeCtas + b * hkv (each row's run of CTAs adds at most one
// slot to the CTA count), the plan [b * hkv + 2] int32, then the selection's S_c and R rows
// [b, hkv, nbs].
struct DecRegions {
  size_t po, pml, plan, sc, sr, bar, total;
};

DecRegions decode_regions(const MaskShape &s) {
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(s.batch) * s.hkv;
  const size_t slots = (kMaxDecodeCtas + rows) * static_cast<size_t>(s.group);
  const size_t srow = rows * s.nbs * 4;
  DecRegions r;
  r.po = 0;
  r.pml = r.po + r256(slots * s.d * 4);
  r.plan = r.pml + r256(slots * 2 * 4);
  r.sc = r.plan + r256((rows + 2) * 4);
  r.sr = r.sc + r256(srow);
  r.bar = r.sr + r256(srow);  // the fused step's barrier and per-row counters
  r.total = r.bar + r256((rows + 1) * 4);
  return r;
}

// The CTAs of one decode step: as many as are resident at once (a cooperative launch), at most
// kMaxDecodeCtas.  The kernel's dynamic shared-memory limit is set once, to what the largest row
// count needs (it is one setting per kernel, so it must cover every shape), and the occupancy is
// looked up once per (device, rows) and kept, so a step costs the host one memset and one launch.
template <int D, int G>
cudaError_t step_ctas(const void *kern, size_t smem, int rows, int *ctas) {
  using C = DecCfg<D, G>;
  struct Entry {
    int dev, rows, ctas;
  };
  static std::mutex mu;
  static Entry cache[16] = {};
  static int used = 0;
  static bool limit_set[64] = {};  // per device (the setting belongs to the device's context)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (int x = 0; x < used; ++x)
    if (cache[x].dev == dev && cache[x].rows == rows) {
      *ctas = cache[x].ctas;
      return cudaSuccess;
    }
  if (dev < 0 || dev >= 64 || !limit_set[dev]) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(C::smem(kMaxDecodeRows)))) != cudaSuccess)
      return e;
    if (dev >= 0 && dev < 64) limit_set[dev] = true;
  }
  int sms = 0, per_sm = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kAttnThreads, smem)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  *ctas = std::max(1, std::min(kMaxDecodeCtas, sms * per_sm));
  if (used < 16) cache[used++] = Entry{dev, rows, *ctas};
  return cudaSuccess;
}

template <int D, int G>
cudaError_t launch_step_g(const MaskShape &s, const DecStepArgs &a, cudaStream_t stream) {
  using C = DecCfg<D, G>;
  auto kern = decode_step_kernel<D, G>;
  const int rows = s.batch * s.hkv;
  const size_t smem = C::smem(rows);
  int ctas = 0;
  cudaError_t e = step_ctas<D, G>(reinterpret_cast<const void *>(kern), smem, rows, &ctas);
  if (e != cudaSuccess) return e;
  // the barrier counter and the per-row score counters start at zero
  if ((e = cudaMemsetAsync(a.bar, 0, (static_cast<size_t>(rows) + 1) * sizeof(unsigned), stream)) != cudaSuccess)
    return e;
  DecStepArgs args = a;
  void *params[] = {&args};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(ctas), dim3(kAttnThreads), params,
                                     smem, stream);
}

template <int D>
cudaError_t launch_step_d(const MaskShape &s, const DecStepArgs &a, cudaStream_t st) {
  switch (s.group) {
    case 1: return launch_step_g<D, 1>(s, a, st);
    case 2: return launch_step_g<D, 2>(s, a, st);
    case 4: return launch_step_g<D, 4>(s, a, st);
    case 8: return launch_step_g<D, 8>(s, a, st);
    case 16: return launch_step_g<D, 16>(s, a, st);
    default: return cudaErrorInvalidValue;
  }
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
  const dim3 rows(s.hkv, s.batch);
  const long long pc = static_cast<long long>(ppm_c), pr = static_cast<long long>(ppm_r);
  if (s.nbs <= 4 * kSelThreads)
    decode_select_kernel<4><<<rows, kSelThreads, 0, stream>>>(sc, sr, alpha, kv_idx, kv_cnt, s.cu, s.seq, s.total,
                                                              s.block, s.hkv, s.nbs, pc, pr, status);
  else if (s.nbs <= 8 * kSelThreads)
    decode_select_kernel<8><<<rows, kSelThreads, 0, stream>>>(sc, sr, alpha, kv_idx, kv_cnt, s.cu, s.seq, s.total,
                                                              s.block, s.hkv, s.nbs, pc, pr, status);
  else if (s.nbs <= 16 * kSelThreads)
    decode_select_kernel<16><<<rows, kSelThreads, 0, stream>>>(sc, sr, alpha, kv_idx, kv_cnt, s.cu, s.seq,
                                                               s.total, s.block, s.hkv, s.nbs, pc, pr, status);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_decode(const MaskShape &s, const void *q_new, const void *k, const void *v,
                          const int32_t *kv_idx, const int32_t *kv_cnt, float scale, void *o, float *lse,
                          void *workspace, int32_t *status, cudaStream_t stream) {
  if (static_cast<long long>(s.batch) * s.hkv > kMaxDecodeRows) return cudaErrorInvalidValue;
  const DecRegions r = decode_regions(s);
  float *po = reinterpret_cast<float *>(static_cast<char *>(workspace) + r.po);
  float *pml = reinterpret_cast<float *>(static_cast<char *>(workspace) + r.pml);
  int *plan = reinterpret_cast<int *>(static_cast<char *>(workspace) + r.plan);
  const float sl2 = scale * kLog2e;
  cudaError_t e;
  if (s.d == 64) e = launch_attn_d<64>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, plan, sl2, status, stream);
  else if (s.d == 128) e = launch_attn_d<128>(s, q_new, k, v, kv_idx, kv_cnt, po, pml, plan, sl2, status, stream);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  dim3 grid(s.hq, s.batch);
  if (s.d == 64)
    decode_combine_kernel<64><<<grid, kCombineThreads, 0, stream>>>(po, pml, plan, static_cast<uint16_t *>(o), lse,
                                                                   s.hq, s.hkv);
  else
    decode_combine_kernel<128><<<grid, kCombineThreads, 0, stream>>>(po, pml, plan, static_cast<uint16_t *>(o),
                                                                    lse, s.hq, s.hkv);
  return cudaGetLastError();
}

cudaError_t launch_decode_step(const MaskShape &s, const void *q_new, const void *k, const void *v,
                               const float *centroid, const float *radius, const float *alpha, int64_t ppm_c,
                               int64_t ppm_r, float select_scale, float softmax_scale, int32_t *kv_idx,
                               int32_t *kv_cnt, void *o, float *lse, void *workspace, int32_t *status,
                               cudaStream_t stream) {
  if (static_cast<long long>(s.batch) * s.hkv > kMaxDecodeRows) return cudaErrorInvalidValue;
  const DecRegions r = decode_regions(s);
  char *ws = static_cast<char *>(workspace);
  DecStepArgs a;
  a.q_new = static_cast<const uint16_t *>(q_new);
  a.k = static_cast<const uint16_t *>(k);
  a.v = static_cast<const uint16_t *>(v);
  a.centroid = centroid;
  a.radius = radius;
  a.alpha = alpha;
  a.kv_idx = kv_idx;
  a.kv_cnt = kv_cnt;
  a.s_c = reinterpret_cast<float *>(ws + r.sc);
  a.s_r = reinterpret_cast<float *>(ws + r.sr);
  a.part_o = reinterpret_cast<float *>(ws + r.po);
  a.part_ml = reinterpret_cast<float *>(ws + r.pml);
  a.plan = reinterpret_cast<int *>(ws + r.plan);
  a.bar = reinterpret_cast<unsigned *>(ws + r.bar);
  a.o = static_cast<uint16_t *>(o);
  a.lse = lse;
  a.cu = s.cu;
  a.batch = s.batch;
  a.seq = s.seq;
  a.total = s.total;
  a.block = s.block;
  a.hq = s.hq;
  a.hkv = s.hkv;
  a.nbs = s.nbs;
  a.ppm_c = static_cast<long long>(ppm_c);
  a.ppm_r = static_cast<long long>(ppm_r);
  a.scale = select_scale;
  a.scale_log2 = softmax_scale * kLog2e;
  a.status = status;
  if (s.d == 64) return launch_step_d<64>(s, a, stream);
  if (s.d == 128) return launch_step_d<128>(s, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bsa
