// Centroid-path and rescue-path block scores on tcgen05 tensor cores (sm_103a).
//
// Source: "Your 128K Context Is 6x Slower Than It Needs to Be"
// (articles.phantom-byte.com), section "The rescue branch: two selection
// paths, one mask".  For one (batch, KV head g) the scores of query block i and
// key block j are
//   S_c[i][j] = s * max_h qbar_{h,i} . c_j
//   R[i][j]   = s * max_h (qbar_{h,i} . c_j + nbar_{h,i} * alpha_j * r_j)
// over the G query heads h of group g.  The dot products are a dense product;
// one CTA computes D = C Qbar^T for 128 key blocks (rows j, the TMEM lanes)
// against 256 (query block, head) columns, so each thread holds every head of
// a (j, i) pair in its own registers: the max over heads needs no shuffles and
// the stores of consecutive j coalesce.  fp32 precision comes from tf32 MMAs
// on hi / lo splits: x = hi + lo with hi = x with its low 13 mantissa bits
// cleared (exact in tf32) and lo = x - hi, and
//   D = A_hi B_hi + A_hi B_lo + A_lo B_hi,
// whose error (the dropped A_lo B_lo term and lo's own rounding) stays below
// 2^-20 of |a||b| per product.  The splits are written by the query-pooling
// launch, so this kernel is TMA loads plus MMAs plus the epilogue.
//
// Warp roles: warp 0 issues TMA loads of 32-dimension chunks (one 128-byte
// swizzle row) of the four operands; warp 1 owns 256 TMEM columns and issues
// the MMAs; then all eight warps read the accumulator (one TMEM lane per key
// block, each warp half of the columns) and write S_c and R.  Every wait is
// bounded.  One stage of shared memory (96 KB) per CTA, so two CTAs share an
// SM (256 TMEM columns and 128 registers a thread each): one CTA's loads and
// epilogue overlap the other's MMAs, which a second stage inside one CTA did
// less well (29 against 35 us per 128K layer).

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsa_internal.h"
#include "sm103_ptx.cuh"

namespace bsa {
namespace {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: no legitimate wait comes close

template <int D, int G>
struct ScoreCfg {
  static constexpr int ROWS = 128;     // key blocks per tile (TMEM lanes)
  static constexpr int COLS = 256;     // (query block, head) columns per tile
  static constexpr int NI = COLS / G;  // query blocks per tile
  static constexpr int KC = 32;        // fp32 elements per K-chunk
  static constexpr int NKC = D / KC;
  static constexpr int NS = 1;       // stages (see the note on occupancy above)
  static constexpr uint32_t A_BYTES = ROWS * KC * 4;  // 16 KB
  static constexpr uint32_t B_BYTES = COLS * KC * 4;  // 32 KB
  // stage layout: A_hi, A_lo, B_hi, B_lo
  static constexpr uint32_t STAGE = 2 * (A_BYTES + B_BYTES);
  static constexpr uint32_t OFF_NBAR = NS * STAGE;
  static constexpr uint32_t OFF_BAR = OFF_NBAR + COLS * 4;
  // barriers: full[NS] (TMA), empty[NS] (MMAs done with the stage), done
  static constexpr int B_FULL = 0, B_EMPTY = NS, B_DONE = 2 * NS, NBARS = 2 * NS + 1;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + NBARS * 8 + 16 + 1024;
  static constexpr int THREADS = 256;
  // kind::tf32: D f32, A and B tf32, both K-major, M = 128, N = 256
  static constexpr uint32_t IDESC = (1u << 4) | (2u << 7) | (2u << 10) |
                                    (static_cast<uint32_t>(COLS >> 3) << 17) |
                                    (static_cast<uint32_t>(ROWS >> 4) << 24);
  static_assert(SMEM_BYTES <= 227 * 1024, "shared-memory budget");
};

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

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

struct ScoreMaps {
  CUtensorMap c_hi, c_lo, q_hi, q_lo;
};

struct ScoreSeq {
  const int32_t *cu;  // packed ragged batch, or null
  int seq, total, block, hkv;
};

template <int D, int G>
__global__ void __launch_bounds__(256, 2)
    score_kernel(const __grid_constant__ ScoreMaps maps, const float *__restrict__ nbar,
                 const float *__restrict__ radius, const float *__restrict__ alpha,
                 float *__restrict__ s_c, float *__restrict__ s_r, int nb, int nbw, const ScoreSeq sq,
                 float scale, int32_t *status) {
  using C = ScoreCfg<D, G>;
  const int jt = blockIdx.x, it = blockIdx.y, gb = blockIdx.z;  // gb = b * hkv + g
  // nb: per-sequence stride of the per-block arrays; nbw: row stride of S_c and R
  const int j0 = jt * C::ROWS, i0 = it * C::NI;
  // this sequence's blocks (nb is the per-sequence stride of every per-block array)
  const SeqSpan sp = seq_span(sq.cu, gb / sq.hkv, sq.seq, sq.total, status);
  const int nbb = (sp.len + sq.block - 1) / sq.block;
  // only tiles with some key block j below some query block i < nbb carry work
  if (i0 >= nbb || j0 >= min(i0 + C::NI, nbb) - 1) return;

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char *sb = smem_raw + (base - raw);
  float *snbar = reinterpret_cast<float *>(sb + C::OFF_NBAR);
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int x) { return bar0 + 8u * static_cast<uint32_t>(x); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::OFF_BAR + C::NBARS * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int x = 0; x < C::NBARS; ++x) ptx::mbar_init(bar(x), 1);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::COLS);
    ptx::tmem_relinquish();
  }
  for (int c = threadIdx.x; c < C::COLS; c += C::THREADS) {
    const int i = i0 + c / G;
    snbar[c] = i < nb ? nbar[(static_cast<size_t>(gb) * nb + i0) * G + c] : 0.f;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&maps.c_hi);
      ptx::tma_prefetch_desc(&maps.c_lo);
      ptx::tma_prefetch_desc(&maps.q_hi);
      ptx::tma_prefetch_desc(&maps.q_lo);
      const int arow = gb * nb + j0, brow = (gb * nb + i0) * G;
      int issued = 0;
      for (int kc = 0; kc < C::NKC; ++kc) {
        const int s = kc % C::NS;
        if (kc >= C::NS && !wait_b(bar(C::B_EMPTY + s), (kc / C::NS - 1) & 1, status, ok)) break;
        const uint32_t st = base + s * C::STAGE;
        ptx::mbar_arrive_expect_tx(bar(C::B_FULL + s), 2 * (C::A_BYTES + C::B_BYTES));
        ptx::tma_load_2d(st, &maps.c_hi, bar(C::B_FULL + s), kc * C::KC, arow);
        ptx::tma_load_2d(st + C::A_BYTES, &maps.c_lo, bar(C::B_FULL + s), kc * C::KC, arow);
        ptx::tma_load_2d(st + 2 * C::A_BYTES, &maps.q_hi, bar(C::B_FULL + s), kc * C::KC, brow);
        ptx::tma_load_2d(st + 2 * C::A_BYTES + C::B_BYTES, &maps.q_lo, bar(C::B_FULL + s), kc * C::KC, brow);
        issued = kc + 1;
      }
      if (!ok) {  // let the copies in flight land before shared memory is released
        bool dok = true;
        for (int kc = issued - C::NS > 0 ? issued - C::NS : 0; kc < issued; ++kc)
          wait_b(bar(C::B_FULL + kc % C::NS), (kc / C::NS) & 1, nullptr, dok);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint64_t da = ptx::sdesc_sw128(base, 16, 1024);
      const uint64_t db = ptx::sdesc_sw128(base + 2 * C::A_BYTES, 16, 1024);
      constexpr uint64_t LO_A = C::A_BYTES >> 4, LO_B = C::B_BYTES >> 4, STG = C::STAGE >> 4;
      for (int kc = 0; kc < C::NKC; ++kc) {
        const int s = kc % C::NS;
        if (!wait_b(bar(C::B_FULL + s), (kc / C::NS) & 1, status, ok)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < C::KC / 8; ++ks) {
          const uint64_t a = da + s * STG + ((ks * 32) >> 4), b = db + s * STG + ((ks * 32) >> 4);
          mma_tf32(tmem, a, b, C::IDESC, (kc > 0 || ks > 0) ? 1u : 0u);  // hi * hi
          mma_tf32(tmem, a, b + LO_B, C::IDESC, 1u);                       // hi * lo
          mma_tf32(tmem, a + LO_A, b, C::IDESC, 1u);                       // lo * hi
        }
        ptx::mma_commit(bar(C::B_EMPTY + s));
      }
      ptx::mma_commit(bar(C::B_DONE));  // also on abort: every issued MMA completes first
    }
    __syncwarp();
  }
  // ---- epilogue, all eight warps: warp w reads TMEM lanes 32 (w % 4) .. + 31 (its key blocks)
  // and the column half w / 4; the producer and MMA warps join once their work is issued
  {
    bool dok = true;
    wait_b(bar(C::B_DONE), 0, status, dok);
    ptx::tc_fence_after();
    const int r = ((warp & 3) << 5) + lane;  // TMEM lane = key block row
    const int j = j0 + r;
    const bool row_ok = dok && j < nbb;
    const float bonus = row_ok ? alpha[static_cast<size_t>(gb) * nb + j] * radius[static_cast<size_t>(gb) * nb + j] : 0.f;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    constexpr int HALF = C::COLS / 2;
    const int cbase = (warp >> 2) * HALF;
#pragma unroll 1
    for (int cc = 0; cc < HALF / 64; ++cc) {
      uint32_t v[64];
      // two 32-column loads in flight before the wait
      ptx::tmem_ld32(tmem + lane_off + cbase + cc * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      ptx::tmem_ld32(tmem + lane_off + cbase + cc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      ptx::tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 64 / G; ++q) {
        // columns cbase + cc*64 + q*G .. + G-1 hold the G heads of one query block
        const int c0 = q * G;
        const int col = cbase + cc * 64 + c0;
        const int i = i0 + col / G;
        float dm = __uint_as_float(v[c0]);
        float rm = fmaf(snbar[col], bonus, dm);
#pragma unroll
        for (int h = 1; h < G; ++h) {
          const float x = __uint_as_float(v[c0 + h]);
          dm = fmaxf(dm, x);
          rm = fmaxf(rm, fmaf(snbar[col + h], bonus, x));
        }
        if (row_ok && j < i && i < nbb) {
          const size_t o = (static_cast<size_t>(gb) * nb + i) * nbw + j;
          s_c[o] = dm * scale;
          s_r[o] = rm * scale;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::COLS);
  }
}

bool make_map_2d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  cudaError_t e;
  EncodeTiledFn fn = tensor_map_encoder(&e);
  if (fn == nullptr || e != cudaSuccess) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 4};
  const cuuint32_t box[2] = {32u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_t(const MaskShape &s, const ScoreOperands &op, float scale, float *s_c, float *s_r,
                     int32_t *status, cudaStream_t stream) {
  using C = ScoreCfg<D, G>;
  ScoreMaps maps;
  const uint64_t groups = static_cast<uint64_t>(s.batch) * s.hkv;
  if (!make_map_2d(&maps.c_hi, op.c_hi, D, groups * s.nbs, C::ROWS) ||
      !make_map_2d(&maps.c_lo, op.c_lo, D, groups * s.nbs, C::ROWS) ||
      !make_map_2d(&maps.q_hi, op.q_hi, D, groups * s.nbs * G, C::COLS) ||
      !make_map_2d(&maps.q_lo, op.q_lo, D, groups * s.nbs * G, C::COLS))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(score_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid((s.nbs + C::ROWS - 1) / C::ROWS, (s.nbs + C::NI - 1) / C::NI, static_cast<unsigned>(groups));
  const ScoreSeq sq{s.cu, s.seq, s.total, s.block, s.hkv};
  score_kernel<D, G><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(maps, op.nbar, op.radius, op.alpha,
                                                                  s_c, s_r, s.nbs, s.nbw, sq, scale, status);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const MaskShape &s, const ScoreOperands &op, float scale, float *sc, float *sr,
                     int32_t *st, cudaStream_t stream) {
  switch (s.group) {
    case 1: return launch_t<D, 1>(s, op, scale, sc, sr, st, stream);
    case 2: return launch_t<D, 2>(s, op, scale, sc, sr, st, stream);
    case 4: return launch_t<D, 4>(s, op, scale, sc, sr, st, stream);
    case 8: return launch_t<D, 8>(s, op, scale, sc, sr, st, stream);
    case 16: return launch_t<D, 16>(s, op, scale, sc, sr, st, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_scores(const MaskShape &s, const ScoreOperands &op, float scale, float *s_c,
                          float *s_r, int32_t *status, cudaStream_t stream) {
  if (s.d == 64) return launch_d<64>(s, op, scale, s_c, s_r, status, stream);
  if (s.d == 128) return launch_d<128>(s, op, scale, s_c, s_r, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bsa
