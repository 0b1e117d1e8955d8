// Warp-level exact top-k over 32-bit order-preserving score keys, shared by
// the prefill select kernel and the decode select kernel.
//
// A row's candidates are keys[0, n) with key 0 marking a non-candidate.  The
// k best are found by a linear 256-bin histogram of the candidates' values
// (bins above the threshold bin are in), then an 8-bit-digit radix select over
// the threshold bin's keys; equal keys at the threshold are ranked by index.
#pragma once

#include <stdint.h>

#include "bsa.h"

namespace bsa {
namespace topk {

constexpr int kCompact = 256;  // capacity of the per-warp list of threshold-bin keys

// Order-preserving key of a float score: a higher score gives a larger key.
// Every non-NaN score maps to a key >= 1, so key 0 marks "not a candidate".
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inverse of score_key for a nonzero key.
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Exclusive prefix sum of c over the lanes of a warp; *total receives the sum.
__device__ __forceinline__ unsigned warp_exclusive_scan(unsigned c, unsigned *total) {
  const int lane = threadIdx.x & 31;
  unsigned incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return incl - c;
}

// In a 256-bin histogram (lane l reads bins 8l .. 8l+7), the bin holding the
// take-th largest entry counting down from the top bin, the number of entries
// in the bins above it, and its own count.  Requires 1 <= take <= total.
__device__ __forceinline__ void warp_find_bin(const unsigned *hist, unsigned take, unsigned *bin,
                                              unsigned *above, unsigned *count) {
  const int lane = threadIdx.x & 31;
  const uint4 h0 = reinterpret_cast<const uint4 *>(hist)[2 * lane];
  const uint4 h1 = reinterpret_cast<const uint4 *>(hist)[2 * lane + 1];
  const unsigned c[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
  unsigned s = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) s += c[e];
  unsigned suf = s;  // entries in the bins of lanes >= this lane
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned o = __shfl_down_sync(0xffffffffu, suf, off);
    if (lane + off < 32) suf += o;
  }
  unsigned acc = suf - s, my_bin = 0, my_above = 0, my_count = 0;
  bool hit = false;
#pragma unroll
  for (int e = 7; e >= 0; --e) {
    if (!hit && acc < take && take <= acc + c[e]) {
      hit = true;
      my_bin = 8 * lane + e;
      my_above = acc;
      my_count = c[e];
    }
    acc += c[e];
  }
  const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
  *bin = __shfl_sync(0xffffffffu, my_bin, src);
  *above = __shfl_sync(0xffffffffu, my_above, src);
  *count = __shfl_sync(0xffffffffu, my_count, src);
  __syncwarp();
}

// Radix threshold of the k largest nonzero keys of keys[0, n) (1 <= k < number
// of nonzero keys), one warp, 8-bit digits from the top.  The selection is:
// every key with (key & pmask) > prefix, plus the first `take` in index order
// of the `n_eq` nonzero keys with (key & pmask) == prefix.
struct Threshold {
  uint32_t prefix, pmask;
  unsigned take, n_eq;
};

__device__ inline Threshold warp_radix_threshold(const uint32_t *keys, int n, unsigned k, unsigned *hist) {
  const int lane = threadIdx.x & 31;
  Threshold t{0u, 0u, k, 0u};
  for (int shift = 24; shift >= 0; shift -= 8) {
    reinterpret_cast<uint4 *>(hist)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(hist)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    for (int j0 = 0; j0 < n; j0 += 32) {  // warp-uniform trip count: every lane reaches the match
      const int j = j0 + lane;
      const uint32_t key = j < n ? keys[j] : 0u;
      const bool ok = key != 0u && (key & t.pmask) == t.prefix;
      const unsigned digit = (key >> shift) & 255u;
      const unsigned peers = __match_any_sync(0xffffffffu, ok ? digit : 256u);
      if (ok && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
    }
    __syncwarp();
    unsigned digit, above, count;
    warp_find_bin(hist, t.take, &digit, &above, &count);
    t.take -= above;
    t.n_eq = count;
    t.prefix |= digit << shift;
    t.pmask |= 0xFFu << shift;
    if (t.n_eq == t.take) break;  // the whole bin is in: no finer digit needed
  }
  return t;
}

// The k best candidates of a row.  A linear 256-bin histogram of the
// candidates' values over [lo, hi] finds the bin holding the threshold; bins
// above it are in, and inside it the radix threshold t over the bin's keys
// (gathered into a short list) decides, unless the whole bin is in.  The bin
// map is monotone in the value, so this is the exact top-k of the keys.  With
// no usable value range, or a threshold bin too crowded for the list, every
// candidate falls in bin 0 and t is taken over the whole row.
struct RowSelect {
  float lo, inv;  // bin(v) = min(255, trunc((v - lo) * inv)); inv == 0 maps everything to bin 0
  int bstar;
  bool whole;
  Threshold t;
};

__device__ __forceinline__ int value_bin(uint32_t key, float lo, float inv) {
  return min(255, static_cast<int>((key_value(key) - lo) * inv));
}

// keys[0, n) are readable 4 at a time: the entries from n up to the next
// multiple of 4 are zero.
__device__ inline RowSelect warp_select(const uint32_t *keys, int n, unsigned k, float lo, float hi,
                                 unsigned *hist, uint32_t *ckeys) {
  const int lane = threadIdx.x & 31;
  RowSelect r;
  r.lo = lo;
  r.inv = 0.f;
  r.bstar = 0;
  r.whole = false;
  if (hi > lo) {
    const float inv = 256.f / (hi - lo);
    if (inv <= 1.0e38f) r.inv = inv;
  }
  if (r.inv > 0.f) {
    reinterpret_cast<uint4 *>(hist)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(hist)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    for (int j = 4 * lane; j < n; j += 128) {
      const uint4 kk = reinterpret_cast<const uint4 *>(keys)[j >> 2];
      const uint32_t kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (kv[e] != 0u) atomicAdd(&hist[value_bin(kv[e], r.lo, r.inv)], 1u);
    }
    __syncwarp();
    unsigned bstar, above, count;
    warp_find_bin(hist, k, &bstar, &above, &count);
    r.bstar = static_cast<int>(bstar);
    const unsigned take = k - above;
    if (count == take) {
      r.whole = true;
      return r;
    }
    if (count <= static_cast<unsigned>(kCompact)) {
      unsigned base = 0;
      for (int j0 = 0; j0 < n; j0 += 128) {  // warp-uniform trip count for the scan
        const int j = j0 + 4 * lane;
        uint32_t kv[4] = {0u, 0u, 0u, 0u};
        unsigned m = 0;
        if (j < n) {
          const uint4 kk = reinterpret_cast<const uint4 *>(keys)[j >> 2];
          kv[0] = kk.x; kv[1] = kk.y; kv[2] = kk.z; kv[3] = kk.w;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (kv[e] != 0u && value_bin(kv[e], r.lo, r.inv) == r.bstar) m |= 1u << e;
        }
        unsigned tot;
        unsigned pos = base + warp_exclusive_scan(__popc(m), &tot);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((m >> e) & 1u) ckeys[pos++] = kv[e];
        base += tot;
      }
      __syncwarp();
      r.t = warp_radix_threshold(ckeys, static_cast<int>(count), take, hist);
      return r;
    }
  }
  r.inv = 0.f;
  r.bstar = 0;
  r.t = warp_radix_threshold(keys, n, k, hist);
  return r;
}

// flags[j] |= bit for the candidates RowSelect r keeps among keys[0, n).  Each
// lane owns 4 consecutive entries (one flags word); equal keys at the
// threshold are ranked in index order.
__device__ inline void warp_mark(const uint32_t *keys, int n, const RowSelect &r, uint8_t *flags, uint8_t bit) {
  const int lane = threadIdx.x & 31;
  const bool ranked = !r.whole && r.t.n_eq != r.t.take;
  unsigned taken = 0;
  for (int j0 = 0; j0 < n; j0 += 128) {  // warp-uniform trip count for the scan
    const int j = j0 + 4 * lane;
    unsigned in = 0, eq = 0;  // bit e: entry j + e
    if (j < n) {
      const uint4 kk = reinterpret_cast<const uint4 *>(keys)[j >> 2];
      const uint32_t kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (kv[e] == 0u) continue;
        const int bn = value_bin(kv[e], r.lo, r.inv);
        if (bn > r.bstar || (bn == r.bstar && r.whole)) {
          in |= 1u << e;
        } else if (bn == r.bstar) {
          const uint32_t top = kv[e] & r.t.pmask;
          if (top > r.t.prefix) in |= 1u << e;
          else if (top == r.t.prefix) eq |= 1u << e;
        }
      }
    }
    if (ranked) {
      unsigned tot;
      unsigned rank = taken + warp_exclusive_scan(__popc(eq), &tot);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((eq >> e) & 1u) {
          if (rank < r.t.take) in |= 1u << e;
          ++rank;
        }
      taken += tot;
    } else {
      in |= eq;
    }
    if (in != 0u) {
      uint32_t *fw = reinterpret_cast<uint32_t *>(flags) + (j >> 2);
      uint32_t w = *fw;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((in >> e) & 1u) w |= static_cast<uint32_t>(bit) << (8 * e);
      *fw = w;
    }
  }
}

__device__ __forceinline__ void warp_minmax(float &lo, float &hi) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
  }
}


// Per-warp scratch of one row: keys [nbs] u32, hist [256] u32, ckeys [kCompact]
// u32, flags [nbs] u8 (nbs % 4 == 0 keeps each 16-byte aligned).
struct RowScratch {
  uint32_t *keys;
  unsigned *hist;
  uint32_t *ckeys;
  uint8_t *flags;
};

__host__ __device__ constexpr size_t row_scratch_bytes(int nbs) {
  return static_cast<size_t>(nbs) * 4 + 1024 + kCompact * 4 +
         ((static_cast<size_t>(nbs) + 15) & ~static_cast<size_t>(15));
}

__device__ __forceinline__ RowScratch row_scratch(unsigned char *base, int nbs) {
  RowScratch w;
  w.keys = reinterpret_cast<uint32_t *>(base);
  w.hist = reinterpret_cast<unsigned *>(base + static_cast<size_t>(nbs) * 4);
  w.ckeys = reinterpret_cast<uint32_t *>(base + static_cast<size_t>(nbs) * 4 + 1024);
  w.flags = base + static_cast<size_t>(nbs) * 4 + 1024 + kCompact * 4;
  return w;
}

// Selection of one row i by one warp: key blocks 0 and i forced, the top kc
// of the candidates 1..i-1 by rc, then among the candidates the centroid path
// dropped whose alpha is positive the top kr by rr; keep counts
// ceil(ratio * (i + 1)) from ppm, clipped to the candidates.  rc and rr point
// at 16-byte aligned rows readable for round_up(i + 1, 4) entries (shared or
// global memory); so does ab (alpha) when AB_ALIGNED, otherwise ab is read one
// entry at a time and only for j < i.  Leaves the BSA_MASK_* bits in
// w.flags[0..i] and zeros up to round_up(i + 1, 4).
template <bool AB_ALIGNED = true>
__device__ inline void warp_select_row(const float *rc, const float *rr, const float *ab, int i,
                                       long long ppm_c, long long ppm_r, const RowScratch &w) {
  const int lane = threadIdx.x & 31;
  uint32_t *keys = w.keys;
  uint8_t *flags = w.flags;
  const int n4 = (i + 4) & ~3;  // keys / flags [0, n4) cover 0..i; entries j >= i are never candidates

  // ---- centroid path: top kc of candidates 1..i-1 by S_c
  // (the row is read in batches of eight 16-byte loads per lane, all issued before any is used)
  constexpr int LB = 4;
  float lo = INFINITY, hi = -INFINITY;
  for (int jb = lane * 4; jb < n4; jb += 128 * LB) {
    float4 v[LB];
#pragma unroll
    for (int u = 0; u < LB; ++u) {
      const int j4 = jb + u * 128;
      v[u] = j4 < n4 ? reinterpret_cast<const float4 *>(rc)[j4 >> 2] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < LB; ++u) {
      const int j4 = jb + u * 128;
      if (j4 >= n4) continue;
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t kp[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j4 + e;
        const bool cand = j >= 1 && j < i;
        kp[e] = cand ? score_key(x[e]) : 0u;
        if (cand) {
          lo = fminf(lo, x[e]);
          hi = fmaxf(hi, x[e]);
        }
      }
      reinterpret_cast<uint4 *>(keys)[j4 >> 2] = make_uint4(kp[0], kp[1], kp[2], kp[3]);
      reinterpret_cast<uint32_t *>(flags)[j4 >> 2] = 0u;
    }
  }
  warp_minmax(lo, hi);
  __syncwarp();
  const int ncand = i > 1 ? i - 1 : 0;
  const long long kc_full = (ppm_c * (i + 1) + 999999LL) / 1000000LL;
  const int kc = static_cast<int>(kc_full < ncand ? kc_full : ncand);
  if (kc == ncand) {
    for (int j = 1 + lane; j < i; j += 32) flags[j] = BSA_MASK_CENTROID;
  } else if (kc > 0) {
    const RowSelect r = warp_select(keys, i, static_cast<unsigned>(kc), lo, hi, w.hist, w.ckeys);
    warp_mark(keys, i, r, flags, BSA_MASK_CENTROID);
  }
  __syncwarp();

  // ---- rescue path: among the dropped candidates with alpha > 0, top kr by R
  int nelig = 0;
  lo = INFINITY;
  hi = -INFINITY;
  for (int jb = lane * 4; jb < n4; jb += 128 * (LB / 2)) {
    float4 v[LB / 2], a[LB / 2];
#pragma unroll
    for (int u = 0; u < LB / 2; ++u) {
      const int j4 = jb + u * 128;
      const bool in = j4 < n4;
      v[u] = in ? reinterpret_cast<const float4 *>(rr)[j4 >> 2] : make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (AB_ALIGNED) {
        a[u] = in ? reinterpret_cast<const float4 *>(ab)[j4 >> 2] : make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        a[u] = make_float4(j4 < i ? ab[j4] : 0.f, j4 + 1 < i ? ab[j4 + 1] : 0.f,
                           j4 + 2 < i ? ab[j4 + 2] : 0.f, j4 + 3 < i ? ab[j4 + 3] : 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < LB / 2; ++u) {
      const int j4 = jb + u * 128;
      if (j4 >= n4) continue;
      const uint32_t f4 = reinterpret_cast<const uint32_t *>(flags)[j4 >> 2];
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w}, al[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
      uint32_t kp[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j4 + e;
        const bool elig = j >= 1 && j < i && al[e] > 0.f && ((f4 >> (8 * e)) & BSA_MASK_CENTROID) == 0;
        kp[e] = elig ? score_key(x[e]) : 0u;
        nelig += elig ? 1 : 0;
        if (elig) {
          lo = fminf(lo, x[e]);
          hi = fmaxf(hi, x[e]);
        }
      }
      reinterpret_cast<uint4 *>(keys)[j4 >> 2] = make_uint4(kp[0], kp[1], kp[2], kp[3]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) nelig += __shfl_xor_sync(0xffffffffu, nelig, off);
  warp_minmax(lo, hi);
  __syncwarp();
  const long long kr_full = (ppm_r * (i + 1) + 999999LL) / 1000000LL;
  const int kr = static_cast<int>(kr_full < nelig ? kr_full : nelig);
  if (kr > 0 && kr == nelig) {
    for (int j = lane; j < i; j += 32)
      if (keys[j] != 0u) flags[j] |= BSA_MASK_RESCUE;
  } else if (kr > 0) {
    const RowSelect r = warp_select(keys, i, static_cast<unsigned>(kr), lo, hi, w.hist, w.ckeys);
    warp_mark(keys, i, r, flags, BSA_MASK_RESCUE);
  }
  __syncwarp();
  if (lane == 0) {
    flags[0] |= BSA_MASK_FORCED;
    flags[i] |= BSA_MASK_FORCED;
  }
  __syncwarp();
}

// Writes the ascending kept list of row i (w.flags[0..i]) to dst and its
// length to *cnt; with mrow, also the row's mask bits (nbs bytes, zero past i),
// four bytes per store when MROW_ALIGNED (mrow 4-byte aligned, nbs % 4 == 0),
// else byte by byte.
template <bool MROW_ALIGNED = true>
__device__ inline void warp_emit_row(const RowScratch &w, int i, int32_t *dst, int32_t *cnt,
                                     uint8_t *mrow, int nbs) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  int kept = 0;
  for (int j0 = 0; j0 <= i; j0 += 32) {
    const int j = j0 + lane;
    const bool keep = j <= i && w.flags[j] != 0;
    const unsigned bl = __ballot_sync(0xffffffffu, keep);
    if (keep) dst[kept + __popc(bl & lt)] = j;
    kept += __popc(bl);
  }
  if (lane == 0) *cnt = kept;
  if (!MROW_ALIGNED && mrow != nullptr) {
    for (int j = lane; j < nbs; j += 32) mrow[j] = j <= i ? w.flags[j] : 0u;
    return;
  }
  if (mrow != nullptr) {
    uint32_t *m4 = reinterpret_cast<uint32_t *>(mrow);
    for (int j4 = lane * 4; j4 < nbs; j4 += 128) {
      uint32_t m = 0;
      if (j4 <= i) {
        m = reinterpret_cast<const uint32_t *>(w.flags)[j4 >> 2];
        if (j4 + 3 > i) m &= 0xFFFFFFFFu >> (8 * (j4 + 3 - i));  // zero the bytes past i
      }
      m4[j4 >> 2] = m;
    }
  }
}

}  // namespace topk
}  // namespace bsa
