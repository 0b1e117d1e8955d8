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
//   decode_select_kernel   one 1024-thread CTA per (b, g): the two-path exact
//                          top-k of a prefill row, CTA-wide (a histogram of
//                          the values, then radix digits of the keys in the
//                          threshold bin, as the prefill row code in
//                          bsa_topk.cuh does per warp; ties by index)
// Attention (bsa_decode_fwd), two launches:
//   decode_attn_kernel     P CTAs per (b, g), about 456 in all: CTA s takes the
//                          kept entries s, s + P, ... in chunks of 128 keys
//                          staged by cp.async (keys and values as separate
//                          groups, the next keys in flight during P V), the G
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
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// ---------------------------------------------------------------- selection

constexpr int kScoreWarps = 8;
constexpr int kScoreBlocksPerWarp = 4;  // key blocks per warp: 32 per CTA

// S_c[j] and R[j] of the new token of (b, g) for the candidates 1 <= j < i, one
// warp per key block (a coalesced centroid row per lane group), 32 key blocks
// per CTA so every SM takes part even at batch 1.  Each warp issues the loads
// of all its centroid rows before it reads the query, so a CTA waits for
// memory about once.
template <int D>
__global__ void __launch_bounds__(kScoreWarps * 32) decode_score_kernel(
    const uint16_t *__restrict__ q_new, const float *__restrict__ centroid, const float *__restrict__ radius,
    const float *__restrict__ alpha, float *__restrict__ s_c, float *__restrict__ s_r,
    const int32_t *__restrict__ cu, int seq, int total, int block, int hq, int hkv, int nbs, float scale,
    int32_t *status) {
  constexpr int DPL = D / 32;  // dimensions per lane
  constexpr int R = kScoreBlocksPerWarp;
  __shared__ __align__(16) float qs[16 * D];
  __shared__ float qn[16];
  const int jt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int grp = hq / hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const size_t gb = static_cast<size_t>(b) * hkv + g;
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  if (sp.len == 0) return;
  const int i = (sp.len - 1) / block;  // the new token's block
  const int j0 = jt * kScoreWarps * R;
  if (j0 >= i) return;
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
}

// ---------------------------------------------------------------- CTA-wide selection
//
// One CTA of kSelThreads threads per (b, g).  Thread t holds the row entries
// j = t * E .. t * E + E - 1 (blocked order, so a CTA prefix sum over threads
// is a prefix sum in index order).  The exact top-k is the same two-stage
// select as the warp code: a 256-bin histogram of the candidates' values finds
// the threshold bin, then 8-bit radix digits of the order-preserving keys
// inside that bin; equal keys at the threshold are ranked by index.

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
static_assert(kMaxBlocks <= 4 * kSelThreads, "a row fits in four entries per thread");

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
  unsigned t = sh.wsum[lane];
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
  lo = sh.wlo[lane];
  hi = sh.whi[lane];
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
  const unsigned wex = warp_exclusive_scan(sh.wsum[lane], &tot);
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
  // the key-group O partials reuse the key buffer after the last chunk
  static_assert(static_cast<size_t>(KH > 1 ? KH - 1 : 1) * G * D * 4 <= static_cast<size_t>(KCH) * KROW,
                "O partials fit in the key buffer");
};

// The work of one split: kept entries e = split, split + P, ... of the list,
// each cut into chunks of up to KCH keys.  A chunk is (entry, first key, keys).
struct Chunk {
  int e, j, c0, n;
};

// The first chunk at entry e or later (stepping by P) whose block index is a
// valid block of the sequence; e == cnt when there is none.
__device__ __forceinline__ Chunk first_chunk(const int32_t *list, int e, int cnt, int step, int last, int len,
                                             int block) {
  for (; e < cnt; e += step) {
    const int j = list[e];
    if (j >= 0 && j <= last) return Chunk{e, j, 0, min(min(block, len - j * block), 128)};
  }
  return Chunk{cnt, 0, 0, 0};
}

__device__ __forceinline__ Chunk next_chunk(const Chunk &c, const int32_t *list, int cnt, int step, int last,
                                            int len, int block) {
  const int nk = min(block, len - c.j * block);
  if (c.c0 + 128 < nk) return Chunk{c.e, c.j, c.c0 + 128, min(128, nk - c.c0 - 128)};
  return first_chunk(list, c.e + step, cnt, step, last, len, block);
}

// Split `split` of row (b, g) (P splits per row): the G heads of the new token
// over its kept entries, one chunk of up to 128 keys at a time.  A chunk's
// keys and values are two cp.async groups into one key and one value buffer:
// the logits wait only for the keys, and the next chunk's keys are requested
// as soon as the logits are done, so they arrive while this chunk's P V runs
// (its values requested after P V).  Thread t takes key t for the logits and,
// for P V, the dimension pair t % (D/2) of key group t / (D/2).  Writes the
// split's unnormalised O, running max and sum (log2 units); a split with no
// valid entry writes an empty partial (max -inf, sum 0, O 0).
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
  if (split >= cnt) return;  // the combine reads the partials of splits < min(P, cnt) only
  const int last = (sp.len - 1) / block;
  const int32_t *list = kv_idx + gb * nbs;

  const size_t tok_stride = static_cast<size_t>(hkv) * D;
  const uint16_t *kbase = k + static_cast<size_t>(sp.start) * tok_stride + static_cast<size_t>(g) * D;
  const uint16_t *vbase = v + static_cast<size_t>(sp.start) * tok_stride + static_cast<size_t>(g) * D;
  constexpr int PR = D * 2 / 16;  // 16-byte pieces per row
  auto stage_k = [&](const Chunk &c) {
    const uint16_t *kg = kbase + (static_cast<size_t>(c.j) * block + c.c0) * tok_stride;
    for (int x = tid; x < c.n * PR; x += kAttnThreads) {
      const int r = x / PR, pc = x - r * PR;
      cp_async16(ks + r * C::KROW + pc * 16, kg + static_cast<size_t>(r) * tok_stride + pc * 8);
    }
    cp_async_commit();
  };
  auto stage_v = [&](const Chunk &c) {
    const uint16_t *vg = vbase + (static_cast<size_t>(c.j) * block + c.c0) * tok_stride;
    for (int x = tid; x < c.n * PR; x += kAttnThreads) {
      const int r = x / PR, pc = x - r * PR;
      cp_async16(smem + C::OFF_V + (static_cast<size_t>(r) * D + pc * 8) * 2,
                 vg + static_cast<size_t>(r) * tok_stride + pc * 8);
    }
    cp_async_commit();
  };

  Chunk cur = first_chunk(list, split, cnt, nsplit, last, sp.len, block);
  if (cur.e < cnt) {
    stage_k(cur);
    stage_v(cur);
  }
  const uint16_t *qrow = q_new + (static_cast<size_t>(b) * hq + static_cast<size_t>(g) * G) * D;
  for (int e = tid; e < G * D; e += kAttnThreads) qs[e / D][e % D] = bf16f(qrow[e]) * scale_log2;
  if (tid < G) mrun[tid] = -INFINITY;

  const int dp = tid % C::DP, kh = tid / C::DP;
  float o[G][2];
  float lsum[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    o[h][0] = o[h][1] = 0.f;
    lsum[h] = 0.f;
  }
  while (cur.e < cnt) {  // CTA-uniform: every thread walks the same list
    const Chunk nxt = next_chunk(cur, list, cnt, nsplit, last, sp.len, block);
    const bool more = nxt.e < cnt;
    cp_async_wait<1>();  // this chunk's keys (its values may still be in flight)
    __syncthreads();
    const bool valid = tid < cur.n;
    // ---- logits of key cur.c0 + tid for the G heads (log2 units)
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
    __syncthreads();  // ps written; every thread is done with the key buffer
    if (tid == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) mrun[h] = lg[h];
    }
    if (more) {
      stage_k(nxt);
      cp_async_wait<1>();  // this chunk's values (the next keys may still be in flight)
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    // ---- P V for this thread's dimension pair and key group
#pragma unroll
    for (int h = 0; h < G; ++h) {
      o[h][0] *= factor[h];
      o[h][1] *= factor[h];
      lsum[h] *= factor[h];
    }
    const uint32_t *vcol = reinterpret_cast<const uint32_t *>(vs) + dp;
#pragma unroll 4
    for (int s = kh; s < cur.n; s += C::KH) {
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
    __syncthreads();  // the value buffer and ps are free
    if (more) stage_v(nxt);
    cur = nxt;
  }
  __syncthreads();  // no copy is in flight; the key buffer becomes the key groups' O partials
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
      *reinterpret_cast<float2 *>(part_o + po + 2 * dp) = make_float2(a0, a1);
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
      *reinterpret_cast<float2 *>(part_ml + pm) = make_float2(mrun[h], l);
    }
  }
}

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;

// One CTA per (b, h): O = sum_s w_s O_s / sum_s w_s l_s over the ns = min(P, cnt)
// splits, w_s = 2^(m_s - max m).  Warp w takes the splits s = w, w + 8, ...
// (every warp first finds max m itself), each lane D/32 dimensions; the warps'
// sums meet in shared memory in a fixed order.
template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_ml, const int32_t *__restrict__ kv_cnt,
    uint16_t *__restrict__ o, float *__restrict__ lse, const int32_t *__restrict__ cu, int seq, int total,
    int block, int hq, int hkv, int nsplit, int32_t *status) {
  constexpr int VL = D / 32;  // dimensions per lane
  __shared__ __align__(16) float red_o[kCombineWarps][D];
  __shared__ float red_l[kCombineWarps];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = h / (hq / hkv);
  const SeqSpan sp = seq_span(cu, b, seq, total, status);
  const int cnt = sp.len > 0 ? min(kv_cnt[static_cast<size_t>(b) * hkv + g], (sp.len - 1) / block + 1) : 0;
  const int ns = max(0, min(nsplit, cnt));
  const size_t base = (static_cast<size_t>(b) * hq + h) * nsplit;
  float m = -INFINITY;
  for (int s = lane; s < ns; s += 32) m = fmaxf(m, part_ml[(base + s) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float acc[VL];
#pragma unroll
  for (int x = 0; x < VL; ++x) acc[x] = 0.f;
  float l = 0.f;
  for (int s0 = warp; s0 < ns; s0 += 4 * kCombineWarps) {
    float2 ml[4];
    float pv[4][VL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int s = s0 + u * kCombineWarps;
      ml[u] = make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int x = 0; x < VL; ++x) pv[u][x] = 0.f;
      if (s < ns) {
        ml[u] = *reinterpret_cast<const float2 *>(part_ml + (base + s) * 2);
        const float *src = part_o + (base + s) * D + lane * VL;
        if constexpr (VL == 4) {
          const float4 t = *reinterpret_cast<const float4 *>(src);
          pv[u][0] = t.x; pv[u][1] = t.y; pv[u][2] = t.z; pv[u][3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2 *>(src);
          pv[u][0] = t.x; pv[u][1] = t.y;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (ml[u].x == -INFINITY) continue;  // an empty split (or past ns)
      const float w = exp2f(ml[u].x - m);
      l = fmaf(ml[u].y, w, l);
#pragma unroll
      for (int x = 0; x < VL; ++x) acc[x] = fmaf(pv[u][x], w, acc[x]);
    }
  }
#pragma unroll
  for (int x = 0; x < VL; ++x) red_o[warp][lane * VL + x] = acc[x];
  if (lane == 0) red_l[warp] = l;
  __syncthreads();
  if (tid < D) {
    float a = 0.f, ls = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      a += red_o[w][tid];
      ls += red_l[w];
    }
    const float r = ls > 0.f ? a / ls : 0.f;
    const __nv_bfloat16 rb = __float2bfloat16_rn(r);
    o[(static_cast<size_t>(b) * hq + h) * D + tid] = *reinterpret_cast<const uint16_t *>(&rb);
    if (lse != nullptr && tid == 0)
      lse[static_cast<size_t>(b) * hq + h] = ls > 0.f ? (m + log2f(ls)) * 0.69314718055994531f : -INFINITY;
  }
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

// Splits per (b, g) row: enough CTAs for about kDecodeCtas in all (152 SMs x 3
// resident CTAs), at most one per block of the row.
constexpr int kDecodeCtas = 456;

int decode_splits(const MaskShape &s) {
  const long long rows = static_cast<long long>(s.hkv) * s.batch;
  const long long p = (kDecodeCtas + rows - 1) / rows;
  return static_cast<int>(p < s.nbs ? p : s.nbs);
}

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
  const dim3 rows(s.hkv, s.batch);
  const long long pc = static_cast<long long>(ppm_c), pr = static_cast<long long>(ppm_r);
  if (s.nbs <= kSelThreads)
    decode_select_kernel<1><<<rows, kSelThreads, 0, stream>>>(sc, sr, alpha, kv_idx, kv_cnt, s.cu, s.seq, s.total,
                                                              s.block, s.hkv, s.nbs, pc, pr, status);
  else if (s.nbs <= 2 * kSelThreads)
    decode_select_kernel<2><<<rows, kSelThreads, 0, stream>>>(sc, sr, alpha, kv_idx, kv_cnt, s.cu, s.seq, s.total,
                                                              s.block, s.hkv, s.nbs, pc, pr, status);
  else if (s.nbs <= 4 * kSelThreads)
    decode_select_kernel<4><<<rows, kSelThreads, 0, stream>>>(sc, sr, alpha, kv_idx, kv_cnt, s.cu, s.seq, s.total,
                                                              s.block, s.hkv, s.nbs, pc, pr, status);
  else
    return cudaErrorInvalidValue;
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
  if (s.d == 64)
    decode_combine_kernel<64><<<grid, kCombineThreads, 0, stream>>>(po, pml, kv_cnt, static_cast<uint16_t *>(o),
                                                                   lse, s.cu, s.seq, s.total, s.block, s.hq, s.hkv,
                                                                   nsplit, status);
  else
    decode_combine_kernel<128><<<grid, kCombineThreads, 0, stream>>>(po, pml, kv_cnt, static_cast<uint16_t *>(o),
                                                                    lse, s.cu, s.seq, s.total, s.block, s.hq, s.hkv,
                                                                    nsplit, status);
  return cudaGetLastError();
}

}  // namespace bsa
