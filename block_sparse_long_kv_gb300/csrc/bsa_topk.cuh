// Exact top-k over 32-bit order-preserving score keys: warp-level helpers (used
// by the decode select kernel) and the team-of-warps row selection of the
// prefill select kernel.
//
// A row's candidates carry a nonzero key (key 0 marks a non-candidate).  The k
// best are found by a linear 256-bin histogram of the candidates' values (bins
// above the threshold bin are in), then a radix select over the threshold
// bin's keys; equal keys at the threshold are ranked by index.
#pragma once

#include <stdint.h>

#include "bsa.h"

namespace bsa {
namespace topk {

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

// Linear value bin of a key over [lo, lo + 256 / inv] (0 .. 255; everything in bin 0 when
// inv is 0): monotone in the key.
__device__ __forceinline__ int value_bin(uint32_t key, float lo, float inv) {
  return min(255, static_cast<int>((key_value(key) - lo) * inv));
}

__device__ __forceinline__ void warp_minmax(float &lo, float &hi) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
  }
}


// ------------------------------------------------------------------ one team of warps per row
//
// The selection of a prefill row, spread over a team of W warps (W a power of two, up to 8), the
// row's entries held in registers: team thread t owns entries P t .. P t + P - 1, so index order
// is thread order and every rank is a team-wide prefix sum.  Rows get the smallest team that
// holds them (32 W P >= the row's length), so short rows cost one warp and long rows finish in
// a few dozen team barriers instead of one warp walking every entry through each phase.
// Within the threshold bin the radix digits start at the highest bit on which the bin's keys
// differ (the bits above it are shared by all of them), so a bin of near-equal values needs
// one or two passes, not four.  Value bins are computed once per path and kept in registers.

constexpr int kTeamMaxWarps = 8;

struct BinHit {
  unsigned bin, above, count;
};

struct TeamScratch {
  unsigned hist[2][256];                 // alternating histograms; each is zeroed after its search
  unsigned wsum[2][kTeamMaxWarps];       // alternating per-warp partials of scans and reductions
  float wlo[2][kTeamMaxWarps], whi[2][kTeamMaxWarps];
  unsigned res[3];                       // bin search result: bin, entries above, its count
  uint32_t gkey[32];                     // the keys of a small threshold bin, gathered to be ranked
  unsigned gcnt;                         // how many are gathered (zero outside a gather)
  unsigned gres[3];                      // their ranking: threshold key, take among equals, equals
};

template <int W>
struct Team {
  static constexpr int T = 32 * W;       // threads
  static constexpr int B = 256 / T;      // histogram bins per thread
  static_assert(W >= 1 && W <= kTeamMaxWarps && (W & (W - 1)) == 0, "team of 1, 2, 4 or 8 warps");
  TeamScratch &sh;
  int bar_id;                            // named barrier of the team (W > 1)
  int t, lane, warp;                     // team-local thread, lane, warp
  int rot = 0, hrot = 0;                 // alternation of the scratch buffers (team-uniform)

  __device__ Team(TeamScratch &s, int id, int tid) : sh(s), bar_id(id), t(tid), lane(tid & 31), warp(tid >> 5) {}

  __device__ __forceinline__ void sync() const {
    if constexpr (W == 1) __syncwarp();
    else asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(T) : "memory");
  }

  // Exclusive prefix sum over the team in thread order; *total receives the sum.  One barrier;
  // the alternating partial buffers make back-to-back calls safe.
  __device__ __forceinline__ unsigned scan(unsigned v, unsigned *total) {
    unsigned incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if constexpr (W == 1) {
      *total = __shfl_sync(0xffffffffu, incl, 31);
      return incl - v;
    } else {
      unsigned *wb = sh.wsum[rot];
      rot ^= 1;
      if (lane == 31) wb[warp] = incl;
      sync();
      unsigned pre = 0, tot = 0;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const unsigned x = wb[w];
        pre += w < warp ? x : 0u;
        tot += x;
      }
      *total = tot;
      return pre + incl - v;
    }
  }

  // Team-wide min / max of lo / hi and sum of n.
  __device__ __forceinline__ void minmax_count(float &lo, float &hi, unsigned &n) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
      n += __shfl_xor_sync(0xffffffffu, n, off);
    }
    if constexpr (W > 1) {
      const int r = rot;
      rot ^= 1;
      if (lane == 0) {
        sh.wlo[r][warp] = lo;
        sh.whi[r][warp] = hi;
        sh.wsum[r][warp] = n;
      }
      sync();
      lo = sh.wlo[r][0];
      hi = sh.whi[r][0];
      n = sh.wsum[r][0];
#pragma unroll
      for (int w = 1; w < W; ++w) {
        lo = fminf(lo, sh.wlo[r][w]);
        hi = fmaxf(hi, sh.whi[r][w]);
        n += sh.wsum[r][w];
      }
    }
  }

  // Team-wide AND and OR.
  __device__ __forceinline__ void and_or(uint32_t &a, uint32_t &o) {
    a = __reduce_and_sync(0xffffffffu, a);
    o = __reduce_or_sync(0xffffffffu, o);
    if constexpr (W > 1) {
      const int r = rot;
      rot ^= 1;
      if (lane == 0) {
        sh.wsum[r][warp] = a;
        reinterpret_cast<uint32_t *>(sh.wlo[r])[warp] = o;
      }
      sync();
      a = 0xFFFFFFFFu;
      o = 0u;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        a &= sh.wsum[r][w];
        o |= reinterpret_cast<const uint32_t *>(sh.wlo[r])[w];
      }
    }
  }

  // In histogram h (256 bins), the bin holding the take-th largest entry counting down from the
  // top bin, the entries in the bins above it and its own count (1 <= take <= total).  Thread t
  // reads bins 255 - B t - e, e < B (thread order = descending bins); afterwards it zeroes them
  // for the histogram's next use (every team thread has read its bins by then).
  __device__ __forceinline__ BinHit find_bin(unsigned *h, unsigned take) {
    unsigned c[B], sum = 0;
#pragma unroll
    for (int e = 0; e < B; ++e) {
      c[e] = h[255 - B * t - e];
      sum += c[e];
    }
    unsigned tot;
    unsigned before = scan(sum, &tot);
#pragma unroll
    for (int e = 0; e < B; ++e) {
      if (before < take && take <= before + c[e]) {
        sh.res[0] = 255u - B * t - e;
        sh.res[1] = before;
        sh.res[2] = c[e];
      }
      before += c[e];
    }
    sync();
    const BinHit r{sh.res[0], sh.res[1], sh.res[2]};
#pragma unroll
    for (int e = 0; e < B; ++e) h[255 - B * t - e] = 0u;
    return r;
  }

  // Both histograms and the gather count to zero (before the row's first barrier).
  __device__ __forceinline__ void clear_hist() {
#pragma unroll
    for (int e = 0; e < B; ++e) {
      sh.hist[0][B * t + e] = 0u;
      sh.hist[1][B * t + e] = 0u;
    }
    if (t == 0) sh.gcnt = 0u;
  }
};

// The same team with its width w chosen at run time (1, 2, 4 or 8 warps): one code path
// serves every row length, so a kernel whose resident CTAs run teams of different widths keeps
// a single copy of the selection code in the instruction cache.
struct TeamRT {
  TeamScratch &sh;
  int W, T, B;                           // warps, threads, histogram bins per thread
  int bar_id;
  int t, lane, warp;
  int rot = 0, hrot = 0;

  __device__ TeamRT(TeamScratch &s, int w, int id, int tid)
      : sh(s), W(w), T(32 * w), B(256 / (32 * w)), bar_id(id), t(tid), lane(tid & 31), warp(tid >> 5) {}

  __device__ __forceinline__ void sync() const {
    if (W == 1) __syncwarp();
    else asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(T) : "memory");
  }

  __device__ __forceinline__ unsigned scan(unsigned v, unsigned *total) {
    unsigned incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (W == 1) {
      *total = __shfl_sync(0xffffffffu, incl, 31);
      return incl - v;
    }
    unsigned *wb = sh.wsum[rot];
    rot ^= 1;
    if (lane == 31) wb[warp] = incl;
    sync();
    unsigned pre = 0, tot = 0;
    for (int w = 0; w < W; ++w) {
      const unsigned x = wb[w];
      pre += w < warp ? x : 0u;
      tot += x;
    }
    *total = tot;
    return pre + incl - v;
  }

  __device__ __forceinline__ void minmax_count(float &lo, float &hi, unsigned &n) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
      n += __shfl_xor_sync(0xffffffffu, n, off);
    }
    if (W == 1) return;
    const int r = rot;
    rot ^= 1;
    if (lane == 0) {
      sh.wlo[r][warp] = lo;
      sh.whi[r][warp] = hi;
      sh.wsum[r][warp] = n;
    }
    sync();
    lo = sh.wlo[r][0];
    hi = sh.whi[r][0];
    n = sh.wsum[r][0];
    for (int w = 1; w < W; ++w) {
      lo = fminf(lo, sh.wlo[r][w]);
      hi = fmaxf(hi, sh.whi[r][w]);
      n += sh.wsum[r][w];
    }
  }

  __device__ __forceinline__ void and_or(uint32_t &a, uint32_t &o) {
    a = __reduce_and_sync(0xffffffffu, a);
    o = __reduce_or_sync(0xffffffffu, o);
    if (W == 1) return;
    const int r = rot;
    rot ^= 1;
    if (lane == 0) {
      sh.wsum[r][warp] = a;
      reinterpret_cast<uint32_t *>(sh.wlo[r])[warp] = o;
    }
    sync();
    a = 0xFFFFFFFFu;
    o = 0u;
    for (int w = 0; w < W; ++w) {
      a &= sh.wsum[r][w];
      o |= reinterpret_cast<const uint32_t *>(sh.wlo[r])[w];
    }
  }

  __device__ __forceinline__ BinHit find_bin(unsigned *h, unsigned take) {
    unsigned c[8], sum = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = e < B ? h[255 - B * t - e] : 0u;
      sum += c[e];
    }
    unsigned tot;
    unsigned before = scan(sum, &tot);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (e < B && before < take && take <= before + c[e]) {
        sh.res[0] = 255u - B * t - e;
        sh.res[1] = before;
        sh.res[2] = c[e];
      }
      before += c[e];
    }
    sync();
    const BinHit r{sh.res[0], sh.res[1], sh.res[2]};
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (e < B) h[255 - B * t - e] = 0u;
    return r;
  }

  __device__ __forceinline__ void clear_hist() {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (e < B) {
        sh.hist[0][B * t + e] = 0u;
        sh.hist[1][B * t + e] = 0u;
      }
    if (t == 0) sh.gcnt = 0u;
  }
};

// Outcome of one path's selection: value bins above bstar are in (all of bstar when whole);
// inside bstar a key is in when (key & pmask) > prefix, and of the keys with (key & pmask) ==
// prefix the first `take` in index order.
struct TeamSel {
  int bstar;
  bool whole;
  uint32_t prefix, pmask;
  unsigned take, n_eq;
};

// The k best of the nonzero keys among the team's registers (1 <= k < number of nonzero keys);
// bin[x]: value bin of key x (monotone in the key).  Both histograms are zero on entry and exit.
template <class TM, int P>
__device__ inline TeamSel team_select(TM &tm, const uint32_t (&key)[P], const uint8_t (&bin)[P], unsigned k) {
  TeamSel r;
  r.whole = false;
  r.prefix = 0u;
  r.pmask = 0u;
  {
    unsigned *h = tm.sh.hist[tm.hrot];
    tm.hrot ^= 1;
#pragma unroll
    for (int x = 0; x < P; ++x)
      if (key[x] != 0u) atomicAdd(&h[bin[x]], 1u);
    tm.sync();
    const BinHit b = tm.find_bin(h, k);
    r.bstar = static_cast<int>(b.bin);
    r.take = k - b.above;
    r.n_eq = b.count;
    if (b.count == r.take) {
      r.whole = true;
      return r;
    }
  }
  if (r.n_eq <= 32u) {
    // A small threshold bin (the common case): its keys are gathered and one warp ranks them,
    // instead of radix passes over every entry.  The threshold is the key K whose count of
    // larger keys is below take and whose count of larger-or-equal keys reaches it; the keys
    // equal to K are then ranked by index as after the radix passes.  Every thread has read the
    // bin search's result before the barrier below.
#pragma unroll
    for (int x = 0; x < P; ++x)
      if (key[x] != 0u && bin[x] == r.bstar) tm.sh.gkey[atomicAdd(&tm.sh.gcnt, 1u)] = key[x];
    tm.sync();
    if (tm.warp == 0) {
      const int n = static_cast<int>(r.n_eq);
      const uint32_t kl = tm.lane < n ? tm.sh.gkey[tm.lane] : 0u;
      unsigned above = 0u, equal = 0u;
      for (int c = 0; c < n; ++c) {
        const uint32_t kc = tm.sh.gkey[c];
        above += kc > kl ? 1u : 0u;
        equal += kc == kl ? 1u : 0u;
      }
      const bool hit = tm.lane < n && above < r.take && r.take <= above + equal;
      const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;  // some lane holds K
      const uint32_t kt = __shfl_sync(0xffffffffu, kl, src);
      const unsigned at = __shfl_sync(0xffffffffu, above, src), eq = __shfl_sync(0xffffffffu, equal, src);
      if (tm.lane == 0) {
        tm.sh.gres[0] = kt;
        tm.sh.gres[1] = r.take - at;
        tm.sh.gres[2] = eq;
        tm.sh.gcnt = 0u;
      }
    }
    tm.sync();
    r.prefix = tm.sh.gres[0];
    r.pmask = 0xFFFFFFFFu;
    r.take = tm.sh.gres[1];
    r.n_eq = tm.sh.gres[2];
    return r;
  }
  // the bits every key of the threshold bin shares need no pass
  uint32_t a = 0xFFFFFFFFu, o = 0u;
#pragma unroll
  for (int x = 0; x < P; ++x)
    if (key[x] != 0u && bin[x] == r.bstar) {
      a &= key[x];
      o |= key[x];
    }
  tm.and_or(a, o);
  const uint32_t diff = a ^ o;
  if (diff == 0u) {  // every key of the bin is equal: index order decides
    r.prefix = a;
    r.pmask = 0xFFFFFFFFu;
    return r;
  }
  int top = 31 - __clz(diff);
  r.pmask = ~((2u << top) - 1u);  // bits above top (none when top is 31)
  r.prefix = a & r.pmask;
  while (top >= 0) {
    const int shift = top >= 7 ? top - 7 : 0;
    const uint32_t dmask = (2u << (top - shift)) - 1u;  // digit width top - shift + 1 <= 8
    unsigned *h = tm.sh.hist[tm.hrot];
    tm.hrot ^= 1;
#pragma unroll
    for (int x = 0; x < P; ++x) {
      const uint32_t kv = key[x];
      const bool ok = kv != 0u && bin[x] == r.bstar && (kv & r.pmask) == r.prefix;
      if (ok) atomicAdd(&h[(kv >> shift) & dmask], 1u);
    }
    tm.sync();
    const BinHit d = tm.find_bin(h, r.take);
    r.take -= d.above;
    r.n_eq = d.count;
    r.prefix |= d.bin << shift;
    r.pmask |= dmask << shift;
    if (r.n_eq == r.take) break;  // the whole digit bin is in
    top = shift - 1;
  }
  return r;
}

// Sets `bit` in the flag bytes of the entries TeamSel r keeps (entry x: byte x % 4 of
// fl[x / 4]); equal keys at the threshold are ranked in index order.
template <class TM, int P>
__device__ inline void team_mark(TM &tm, const uint32_t (&key)[P], const uint8_t (&bin)[P], const TeamSel &r,
                                 uint32_t (&fl)[P / 4], uint32_t bit) {
  unsigned in = 0u, eq = 0u;  // bit x: entry x
#pragma unroll
  for (int x = 0; x < P; ++x) {
    const uint32_t kv = key[x];
    if (kv == 0u) continue;
    const int bn = bin[x];
    if (bn > r.bstar || (bn == r.bstar && r.whole)) {
      in |= 1u << x;
    } else if (bn == r.bstar) {
      const uint32_t tp = kv & r.pmask;
      if (tp > r.prefix) in |= 1u << x;
      else if (tp == r.prefix) eq |= 1u << x;
    }
  }
  if (!r.whole && r.n_eq != r.take) {  // team-uniform
    unsigned tot;
    unsigned rank = tm.scan(__popc(eq), &tot);
#pragma unroll
    for (int x = 0; x < P; ++x)
      if ((eq >> x) & 1u) {
        if (rank < r.take) in |= 1u << x;
        ++rank;
      }
  } else {
    in |= eq;
  }
#pragma unroll
  for (int x = 0; x < P; ++x)
    if ((in >> x) & 1u) fl[x / 4] |= bit << (8 * (x % 4));
}

// Value bins of the keys over [lo, hi] (256 linear bins; everything in bin 0 without a usable
// range).  Monotone in the key, so the top-k of the keys is decided bin by bin.
template <int P>
__device__ __forceinline__ void value_bins(const uint32_t (&key)[P], float lo, float hi, uint8_t (&bin)[P]) {
  float inv = 0.f;
  if (hi > lo) {
    const float x = 256.f / (hi - lo);
    if (x <= 1.0e38f) inv = x;
  }
#pragma unroll
  for (int x = 0; x < P; ++x) bin[x] = key[x] != 0u ? static_cast<uint8_t>(value_bin(key[x], lo, inv)) : 0;
}

// Selection of row i by a team: key blocks 0 and i forced, the top kc of candidates 1..i-1 by
// rc, then the top kr by rr among the candidates the centroid path dropped whose alpha is
// positive; keep counts ceil(ratio (i + 1)) from ppm, clipped to the candidates.  rc and rr:
// 16-byte aligned rows readable for round_up(i + 1, 4) entries; ab (alpha) likewise when
// AB_ALIGNED, else read one entry at a time for j < i.  32 W P >= i + 1.  Leaves the BSA_MASK_*
// bits of entry P t + x in byte x % 4 of fl[x / 4] (zero past i).  Both histograms must be zero
// and ordered before the team's first barrier.
template <class TM, int P, bool AB_ALIGNED>
__device__ inline void team_select_row(TM &tm, const float *rc, const float *rr, const float *ab, int i,
                                       long long ppm_c, long long ppm_r, uint32_t (&fl)[P / 4]) {
  static_assert(P % 4 == 0 && P <= 32, "whole 16-byte groups, one mask bit per entry");
  const int j0 = P * tm.t;
  const int n4 = (i + 4) & ~3;
  uint32_t key[P];
  uint8_t bin[P];
#pragma unroll
  for (int x = 0; x < P / 4; ++x) fl[x] = 0u;

  // ---- centroid path: top kc of candidates 1..i-1 by S_c
  float lo = INFINITY, hi = -INFINITY;
  {
    float4 v[P / 4];
#pragma unroll
    for (int u = 0; u < P / 4; ++u) {
      const int j4 = j0 + 4 * u;
      v[u] = j4 < n4 ? reinterpret_cast<const float4 *>(rc)[j4 >> 2] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < P / 4; ++u) {
      const float xs[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j0 + 4 * u + e;
        const bool cand = j >= 1 && j < i;
        key[4 * u + e] = cand ? score_key(xs[e]) : 0u;
        if (cand) {
          lo = fminf(lo, xs[e]);
          hi = fmaxf(hi, xs[e]);
        }
      }
    }
  }
  const int ncand = i > 1 ? i - 1 : 0;
  const long long kc_full = (ppm_c * (i + 1) + 999999LL) / 1000000LL;
  const int kc = static_cast<int>(kc_full < ncand ? kc_full : ncand);
  if (kc == ncand) {
#pragma unroll
    for (int x = 0; x < P; ++x)
      if (key[x] != 0u) fl[x / 4] |= BSA_MASK_CENTROID << (8 * (x % 4));
  } else if (kc > 0) {
    unsigned dummy = 0u;
    tm.minmax_count(lo, hi, dummy);
    value_bins<P>(key, lo, hi, bin);
    const TeamSel r = team_select<TM, P>(tm, key, bin, static_cast<unsigned>(kc));
    team_mark<TM, P>(tm, key, bin, r, fl, BSA_MASK_CENTROID);
  }

  // ---- rescue path: among the dropped candidates with alpha > 0, top kr by R
  unsigned nelig = 0u;
  lo = INFINITY;
  hi = -INFINITY;
  {
    float4 v[P / 4], a[P / 4];
#pragma unroll
    for (int u = 0; u < P / 4; ++u) {
      const int j4 = j0 + 4 * u;
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
    for (int u = 0; u < P / 4; ++u) {
      const float xs[4] = {v[u].x, v[u].y, v[u].z, v[u].w}, al[4] = {a[u].x, a[u].y, a[u].z, a[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int x = 4 * u + e;
        const int j = j0 + x;
        const bool elig = j >= 1 && j < i && al[e] > 0.f && ((fl[u] >> (8 * e)) & BSA_MASK_CENTROID) == 0u;
        key[x] = elig ? score_key(xs[e]) : 0u;
        nelig += elig ? 1u : 0u;
        if (elig) {
          lo = fminf(lo, xs[e]);
          hi = fmaxf(hi, xs[e]);
        }
      }
    }
  }
  tm.minmax_count(lo, hi, nelig);
  const long long kr_full = (ppm_r * (i + 1) + 999999LL) / 1000000LL;
  const int kr = static_cast<int>(kr_full < static_cast<long long>(nelig) ? kr_full : static_cast<long long>(nelig));
  if (kr > 0 && kr == static_cast<int>(nelig)) {
#pragma unroll
    for (int x = 0; x < P; ++x)
      if (key[x] != 0u) fl[x / 4] |= BSA_MASK_RESCUE << (8 * (x % 4));
  } else if (kr > 0) {
    value_bins<P>(key, lo, hi, bin);
    const TeamSel r = team_select<TM, P>(tm, key, bin, static_cast<unsigned>(kr));
    team_mark<TM, P>(tm, key, bin, r, fl, BSA_MASK_RESCUE);
  }
#pragma unroll
  for (int x = 0; x < P; ++x) {
    const int j = j0 + x;
    if (j == 0 || j == i) fl[x / 4] |= BSA_MASK_FORCED << (8 * (x % 4));
  }
}

// Writes row i's ascending kept list (entries whose flag byte is nonzero) to dst and its length
// to *cnt; with mrow, also the mask bytes (nbs of them, zero past i), a word per store when
// MROW_ALIGNED (mrow 4-byte aligned, nbs % 4 == 0), else byte by byte.  32 W P >= nbs is not
// required: entries past the team's reach are zero-filled by the lanes that reach them.
template <class TM, int P, bool MROW_ALIGNED>
__device__ inline void team_emit_row(TM &tm, const uint32_t (&fl)[P / 4], int i, int32_t *dst, int32_t *cnt,
                                     uint8_t *mrow, int nbs) {
  const int j0 = P * tm.t;
  unsigned mine = 0u;
#pragma unroll
  for (int x = 0; x < P; ++x) mine += ((fl[x / 4] >> (8 * (x % 4))) & 0xFFu) != 0u ? 1u : 0u;
  unsigned tot;
  unsigned pos = tm.scan(mine, &tot);
#pragma unroll
  for (int x = 0; x < P; ++x)
    if (((fl[x / 4] >> (8 * (x % 4))) & 0xFFu) != 0u) dst[pos++] = j0 + x;
  if (tm.t == 0) *cnt = static_cast<int32_t>(tot);
  if (mrow == nullptr) return;
  // the row's mask: the team's own entries, then zeros up to nbs (past 32 W P)
#pragma unroll
  for (int u = 0; u < P / 4; ++u) {
    const int j4 = j0 + 4 * u;
    if (j4 >= nbs) continue;
    if constexpr (MROW_ALIGNED) {
      reinterpret_cast<uint32_t *>(mrow)[j4 >> 2] = fl[u];
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (j4 + e < nbs) mrow[j4 + e] = static_cast<uint8_t>(fl[u] >> (8 * e));
    }
  }
  if constexpr (MROW_ALIGNED) {
    for (int j4 = tm.T * P + 4 * tm.t; j4 < nbs; j4 += 4 * tm.T)
      reinterpret_cast<uint32_t *>(mrow)[j4 >> 2] = 0u;
  } else {
    for (int j = tm.T * P + tm.t; j < nbs; j += tm.T) mrow[j] = 0u;
  }
}

}  // namespace topk
}  // namespace bsa
