// Per-token query aggregation of the block scores on tcgen05 tensor cores (sm_103a).
//
// Source: "Your 128K Context Is 6x Slower Than It Needs to Be"
// (articles.phantom-byte.com), section "The numbers, stated honestly": a
// selector that compares every token with every block centroid needs a table
// of tokens x blocks in memory, unless the comparison is reduced tile by tile
// as it is computed.  This kernel is that tiled reduction.  For one (batch, KV head g), query block i
// and key block j:
//   S_c[i][j] = s * max over the G heads h and the tokens t of block i of q_{h,t} . c_j
//   R[i][j]   = s * max_{h,t} (q_{h,t} . c_j + alpha_j * |q_{h,t}| * r_j)
// With alpha_j = 1, R bounds every logit q_{h,t} . k of block j (Cauchy-Schwarz),
// so it is an upper bound of the block's largest attention score.
//
// One CTA owns 256 consecutive tokens of one sequence (the N side of the MMA)
// and walks the 128-key-block tiles below them (the M side, one TMEM lane per
// key block); for each tile it runs the G heads of the group:
//   D = C_hi Q_h^T + C_lo Q_h^T      (kind::f16, bf16 operands, f32 accumulate)
// Q is bf16 and exact as an operand; the centroids are split into bf16
// hi + lo, which keeps about 16 significant bits (error below 2^-16 of
// |q||c| per product).  The epilogue thread of key block j takes the max
// over its 256 columns per query block straight from its own TMEM lane, so no
// N x nb tensor exists anywhere; the max over heads stays in registers, and
// S_c and R are written once per (i, j).
//
// Warp roles: warp 0 issues the TMA loads (a centroid tile per key-block tile,
// a Q tile per head through a 2-stage ring); warp 1 owns two 256-column TMEM
// accumulators and issues the MMAs; warps 2-3 compute the token norms |q_{h,t}|
// from the first pass's Q tiles; warps 4-7 run the epilogue.  Every wait is
// bounded.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsa_internal.h"
#include "sm103_ptx.cuh"

namespace bsa {
namespace {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: no legitimate wait comes close

template <int D, int BLK, int G>
struct TokCfg {
  static constexpr int ROWS = 128;                 // key blocks per tile (M, TMEM lanes)
  static constexpr int TT = 256;                   // tokens per CTA (N)
  static constexpr int QB = TT / BLK;              // query blocks per CTA
  static constexpr int NCH = D / 64;               // 128-byte K chunks
  static constexpr uint32_t A_CHUNK = ROWS * 128;  // 16 KB
  static constexpr uint32_t A_SPLIT = NCH * A_CHUNK;
  static constexpr uint32_t A_BYTES = 2 * A_SPLIT;  // hi + lo
  static constexpr uint32_t B_CHUNK = TT * 128;     // 32 KB
  static constexpr uint32_t B_BYTES = NCH * B_CHUNK;
  static constexpr int BS = 2;  // Q stages
  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_B = OFF_A + A_BYTES;
  static constexpr uint32_t OFF_NRM = OFF_B + BS * B_BYTES;  // [G][TT] token norms
  static constexpr uint32_t OFF_BAR = OFF_NRM + G * TT * 4;
  // barriers: A full / empty, Q full[BS] / empty[BS], TMEM full[2] / empty[2],
  // norms ready[G] (each used once), final drain
  static constexpr int B_AF = 0, B_AE = 1, B_BF = 2, B_BE = B_BF + BS, B_TF = B_BE + BS,
                       B_TE = B_TF + 2, B_NR = B_TE + 2, B_FIN = B_NR + G, NBARS = B_FIN + 1;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + NBARS * 8 + 16 + 1024;
  static constexpr int THREADS = 256;
  static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(ROWS, TT, false);
  static_assert(BLK >= 32 && TT % BLK == 0, "a 32-column TMEM chunk must lie in one query block");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared-memory budget");
};

__device__ __forceinline__ bool wait_b(uint32_t bar, uint32_t parity, int32_t *status, bool &ok) {
  if (!ok) return false;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kWaitNs) {
      if (status != nullptr) atomicCAS(status, 0, BSA_ERR_DEVICE_TIMEOUT);
      ok = false;
      return false;
    }
  }
  return true;
}

struct TokMaps {
  CUtensorMap q, c_hi, c_lo;
};

struct TokArgs {
  const float *radius, *alpha;
  float *s_c, *s_r;
  const int32_t *cu;
  int seq, total, hkv, nbs, ntt;
  int nbw;  // row stride of s_c and s_r
  float scale;
  int32_t *status;
};

template <int D, int BLK, int G>
__global__ void __launch_bounds__(256, 1)
    token_score_kernel(const __grid_constant__ TokMaps maps, const TokArgs a) {
  using C = TokCfg<D, BLK, G>;
  const int tt = a.ntt - 1 - static_cast<int>(blockIdx.x);  // longest causal rows first
  const int g = blockIdx.y, b = blockIdx.z;
  const int gb = b * a.hkv + g;
  const SeqSpan sp = seq_span(a.cu, b, a.seq, a.total, a.status);
  const int tok0 = tt * C::TT;  // first token of the tile within its sequence
  if (tok0 >= sp.len) return;
  const int nbb = (sp.len + BLK - 1) / BLK;
  const int i0 = tok0 / BLK;
  const int i_last = min(i0 + C::QB, nbb) - 1;        // last query block of the tile
  const int njt = i_last >= 1 ? (i_last - 1) / C::ROWS + 1 : 0;  // key-block tiles with j < i_last
  if (njt == 0) return;
  const int nvalid = min(C::TT, sp.len - tok0);       // token columns inside the sequence

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char *sb = smem_raw + (base - raw);
  float *nrm = reinterpret_cast<float *>(sb + C::OFF_NRM);
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int x) { return bar0 + 8u * static_cast<uint32_t>(x); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::OFF_BAR + C::NBARS * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int x = 0; x < C::NBARS; ++x) {
      uint32_t count = 1;
      if (x >= C::B_BE && x < C::B_BE + C::BS) count = 3;  // MMA commit + both norm warps
      if (x >= C::B_TE && x < C::B_TE + 2) count = 4;      // the four epilogue warps
      if (x >= C::B_NR && x < C::B_NR + G) count = 2;      // both norm warps
      ptx::mbar_init(bar(x), count);
    }
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  const int total_n = njt * G;  // (key-block tile, head) steps

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&maps.q);
      ptx::tma_prefetch_desc(&maps.c_hi);
      ptx::tma_prefetch_desc(&maps.c_lo);
      int a_issued = 0, b_issued = 0;
      for (int n = 0; ok && n < total_n; ++n) {
        const int jt = n / G, h = n - jt * G, s = n % C::BS, u = n / C::BS;
        // the Q tile goes first, so it is in flight while the previous key-block tile drains
        if (u > 0 && !wait_b(bar(C::B_BE + s), (u - 1) & 1, a.status, ok)) break;
        ptx::mbar_arrive_expect_tx(bar(C::B_BF + s), C::B_BYTES);
        for (int c = 0; c < C::NCH; ++c)
          ptx::tma_load_4d(base + C::OFF_B + s * C::B_BYTES + c * C::B_CHUNK, &maps.q, bar(C::B_BF + s),
                           c * 64, g * G + h, sp.start + tok0, 0);
        b_issued = n + 1;
        if (h == 0) {
          if (jt > 0 && !wait_b(bar(C::B_AE), (jt - 1) & 1, a.status, ok)) break;
          ptx::mbar_arrive_expect_tx(bar(C::B_AF), C::A_BYTES);
          const int arow = gb * a.nbs + jt * C::ROWS;
          for (int c = 0; c < C::NCH; ++c) {
            ptx::tma_load_2d(base + C::OFF_A + c * C::A_CHUNK, &maps.c_hi, bar(C::B_AF), c * 64, arow);
            ptx::tma_load_2d(base + C::OFF_A + C::A_SPLIT + c * C::A_CHUNK, &maps.c_lo, bar(C::B_AF),
                             c * 64, arow);
          }
          a_issued = jt + 1;
        }
      }
      if (!ok) {  // let the copies in flight land before shared memory is released
        bool dok = true;
        if (a_issued > 0) wait_b(bar(C::B_AF), (a_issued - 1) & 1, nullptr, dok);
        dok = true;
        for (int n = b_issued - C::BS > 0 ? b_issued - C::BS : 0; n < b_issued; ++n) {
          wait_b(bar(C::B_BF + n % C::BS), (n / C::BS) & 1, nullptr, dok);
          dok = true;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint64_t da_hi = ptx::sdesc_sw128(base + C::OFF_A, 16, 1024);
      const uint64_t da_lo = ptx::sdesc_sw128(base + C::OFF_A + C::A_SPLIT, 16, 1024);
      const uint64_t db0 = ptx::sdesc_sw128(base + C::OFF_B, 16, 1024);
      for (int jt = 0; ok && jt < njt; ++jt) {
        if (!wait_b(bar(C::B_AF), jt & 1, a.status, ok)) break;
        ptx::tc_fence_after();
        for (int h = 0; h < G; ++h) {
          const int n = jt * G + h, s = n % C::BS, buf = n & 1;
          if (!wait_b(bar(C::B_BF + s), (n / C::BS) & 1, a.status, ok)) break;
          if (n >= 2 && !wait_b(bar(C::B_TE + buf), ((n >> 1) - 1) & 1, a.status, ok)) break;
          ptx::tc_fence_after();
          const uint32_t dst = tmem + buf * C::TT;
          const uint64_t db = db0 + ((static_cast<uint64_t>(s) * C::B_BYTES) >> 4);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ao = (c * C::A_CHUNK + kk * 32) >> 4, bo = (c * C::B_CHUNK + kk * 32) >> 4;
              ptx::mma_ss(dst, da_hi + ao, db + bo, C::IDESC, (c > 0 || kk > 0) ? 1u : 0u);
            }
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ao = (c * C::A_CHUNK + kk * 32) >> 4, bo = (c * C::B_CHUNK + kk * 32) >> 4;
              ptx::mma_ss(dst, da_lo + ao, db + bo, C::IDESC, 1u);
            }
          ptx::mma_commit(bar(C::B_BE + s));
          ptx::mma_commit(bar(C::B_TF + buf));
        }
        ptx::mma_commit(bar(C::B_AE));
      }
      // every MMA issued so far completes before TMEM is released
      ptx::mma_commit(bar(C::B_FIN));
      bool dok = true;
      wait_b(bar(C::B_FIN), 0, nullptr, dok);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ================================================================ token norms
    const int nt = threadIdx.x - 64;  // 0..63: tokens nt, nt + 64, nt + 128, nt + 192
    for (int n = 0; n < total_n; ++n) {
      const int s = n % C::BS;
      if (!wait_b(bar(C::B_BF + s), (n / C::BS) & 1, a.status, ok)) break;
      if (n < G) {  // the first key-block tile brings every head's Q tile once
        const unsigned char *tile = sb + C::OFF_B + s * C::B_BYTES;
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
          const int r = nt + 64 * m;
          float sq = 0.f;
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              // 128-byte swizzle: 16-byte unit u of row r sits at unit u ^ (r % 8)
              const uint4 x = *reinterpret_cast<const uint4 *>(tile + c * C::B_CHUNK + r * 128 +
                                                               ((u ^ (r & 7)) << 4));
              const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
                sq = fmaf(lo, lo, sq);
                sq = fmaf(hi, hi, sq);
              }
            }
          nrm[n * C::TT + r] = sqrtf(sq);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(C::B_NR + n));
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::B_BE + s));
    }
  } else {
    // ================================================================ epilogue
    const int sub = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(sub << 5) << 16;
    for (int jt = 0; ok && jt < njt; ++jt) {
      const int j = jt * C::ROWS + (sub << 5) + lane;  // this thread's key block
      const bool jv = j < nbb;
      const float bonus =
          jv ? a.alpha[static_cast<size_t>(gb) * a.nbs + j] * a.radius[static_cast<size_t>(gb) * a.nbs + j]
             : 0.f;
      float dm[C::QB], rm[C::QB];
#pragma unroll
      for (int q = 0; q < C::QB; ++q) dm[q] = rm[q] = -INFINITY;
      for (int h = 0; h < G; ++h) {
        const int n = jt * G + h, buf = n & 1;
        if (!wait_b(bar(C::B_TF + buf), (n >> 1) & 1, a.status, ok)) break;
        if (jt == 0 && !wait_b(bar(C::B_NR + h), 0, a.status, ok)) break;
        ptx::tc_fence_after();
        const float *nr = nrm + h * C::TT;
#pragma unroll
        for (int cc = 0; cc < C::TT / 32; ++cc) {
          uint32_t v[32];
          ptx::tmem_ld32(tmem + lane_off + buf * C::TT + cc * 32, v);
          ptx::tmem_wait_ld();
          const int q = (cc * 32) / BLK;  // query block of these 32 columns
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = cc * 32 + e;
            const float x = col < nvalid ? __uint_as_float(v[e]) : -INFINITY;
            dm[q] = fmaxf(dm[q], x);
            rm[q] = fmaxf(rm[q], fmaf(nr[col], bonus, x));
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(C::B_TE + buf));
      }
      if (!ok) break;
#pragma unroll
      for (int q = 0; q < C::QB; ++q) {
        const int i = i0 + q;
        if (jv && j < i && i < nbb) {
          const size_t o = (static_cast<size_t>(gb) * a.nbs + i) * a.nbw + j;
          a.s_c[o] = dm[q] * a.scale;
          a.s_r[o] = rm[q] * a.scale;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// bf16 hi / lo split of the centroids: hi = bf16(c), lo = bf16(c - hi).
__global__ void centroid_split16_kernel(const float *__restrict__ centroid, __nv_bfloat16 *__restrict__ hi,
                                        __nv_bfloat16 *__restrict__ lo, size_t n) {
  for (size_t e = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float c = centroid[e];
    const __nv_bfloat16 h = __float2bfloat16_rn(c);
    hi[e] = h;
    lo[e] = __float2bfloat16_rn(c - __bfloat162float(h));
  }
}

bool map_c16(EncodeTiledFn fn, CUtensorMap *map, const void *ptr, int d, uint64_t rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {64u, 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map_q(EncodeTiledFn fn, CUtensorMap *map, const void *ptr, int total, int hq, int d) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hq),
                              static_cast<cuuint64_t>(total), 1};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(hq) * d * 2,
                                 static_cast<cuuint64_t>(total) * hq * d * 2};
  const cuuint32_t box[4] = {64u, 1u, 256u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int BLK, int G>
cudaError_t launch_t(const MaskShape &s, const TokMaps &maps, const TokArgs &args, cudaStream_t stream) {
  using C = TokCfg<D, BLK, G>;
  auto kern = token_score_kernel<D, BLK, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(args.ntt, s.hkv, s.batch);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(maps, args);
  return cudaGetLastError();
}

template <int D, int BLK>
cudaError_t launch_g(const MaskShape &s, const TokMaps &m, const TokArgs &a, cudaStream_t st) {
  switch (s.group) {
    case 1: return launch_t<D, BLK, 1>(s, m, a, st);
    case 2: return launch_t<D, BLK, 2>(s, m, a, st);
    case 4: return launch_t<D, BLK, 4>(s, m, a, st);
    case 8: return launch_t<D, BLK, 8>(s, m, a, st);
    case 16: return launch_t<D, BLK, 16>(s, m, a, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
cudaError_t launch_blk(const MaskShape &s, const TokMaps &m, const TokArgs &a, cudaStream_t st) {
  switch (s.block) {
    case 64: return launch_g<D, 64>(s, m, a, st);
    case 128: return launch_g<D, 128>(s, m, a, st);
    case 256: return launch_g<D, 256>(s, m, a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_token_scores(const MaskShape &s, const void *q, const float *centroid, void *c16,
                                const float *radius, const float *alpha, float scale, float *s_c,
                                float *s_r, int32_t *status, cudaStream_t stream) {
  const size_t n = static_cast<size_t>(s.batch) * s.hkv * s.nbs * s.d;
  __nv_bfloat16 *hi = static_cast<__nv_bfloat16 *>(c16);
  __nv_bfloat16 *lo = hi + n;
  centroid_split16_kernel<<<static_cast<unsigned>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096), 256, 0,
                            stream>>>(centroid, hi, lo, n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  EncodeTiledFn fn = tensor_map_encoder(&e);
  if (fn == nullptr || e != cudaSuccess) return e == cudaSuccess ? cudaErrorNotSupported : e;
  TokMaps maps;
  const uint64_t rows = static_cast<uint64_t>(s.batch) * s.hkv * s.nbs;
  if (!map_q(fn, &maps.q, q, s.total, s.hq, s.d) || !map_c16(fn, &maps.c_hi, hi, s.d, rows) ||
      !map_c16(fn, &maps.c_lo, lo, s.d, rows))
    return cudaErrorInvalidValue;
  TokArgs a{radius, alpha, s_c, s_r, s.cu, s.seq, s.total, s.hkv, s.nbs, (s.seq + 255) / 256, s.nbw, scale,
            status};
  if (s.d == 64) return launch_blk<64>(s, maps, a, stream);
  if (s.d == 128) return launch_blk<128>(s, maps, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bsa
