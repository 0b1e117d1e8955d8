// Block-sparse causal prefill attention on tcgen05 tensor cores (sm_103a).
//
// Source: "Your 128K Context Is 6x Slower Than It Needs to Be"
// (articles.phantom-byte.com), section "The rescue branch": the combined mask
// runs as regular block-sparse FlashAttention; and "attention-kernel-
// optimization" (skill-vault.co.in), section "FlashAttention (1 -> 2 -> 3)":
// Q/K/V tiles streamed through on-chip memory with online-softmax rescaling,
// so the N x N score matrix never reaches HBM.
//
// One CTA owns NT query tiles of 128 rows that share one kept-block list: the
// rows are 128 tokens of one head (block 128 / 256) or 64 tokens x 2 heads of
// the same KV group (block 64), so K and V tiles are loaded once per CTA for
// NT tiles (GQA sharing).  Key tiles are always 128 keys wide: with block 64
// a tile holds two kept blocks (two TMA boxes into one tile; an odd count
// leaves the last tile's second half masked), so every S MMA is N = 128.
// Warp roles:
//   warp 0      TMA producer: Q tiles once, then K and V tiles of every kept
//               block through mbarrier rings (KS K stages, VS V stages)
//   warp 1      TMEM owner and single-thread MMA issuer:
//                 S_t = Q_t K^T   (SS form, both operands in shared memory)
//                 O_t += P_t V    (TS form, P read from TMEM)
//               in the ping-pong order S_0(n), PV_1(n-1), S_1(n), PV_0(n), so
//               the tensor core works on one tile while the other tile's
//               softmax runs
//   warps 4..   softmax warps: for 128-column key tiles two warps per 32-row
//               TMEM sub-partition, each thread owning half of a query row's
//               columns (the halves exchange partial maxima through shared
//               memory); read S_t from TMEM, causal mask on the diagonal tile
//               only, online softmax in registers (exp2), P_t as bf16 back into
//               TMEM over S_t, rare O_t rescale, then the epilogue (O / l, LSE)
// setmaxnreg moves registers from the producer / MMA warpgroup to the softmax
// warps; the host refuses to launch if the compiled register count differs
// from the budget the split assumes.
// FP8 inputs (F8): Q and K arrive as e4m3 codes with per-tensor scales and
// S = Q K^T runs as kind::f8f6f4 (both operands K-major, K = 32 per MMA).  V
// is widened to bf16 codes once per layer by a streaming pass (exact: every
// e4m3 value is a bf16 value) and read by the unchanged P V path, so P stays
// bf16 in TMEM and O matches the bf16 path's accuracy on the dequantised
// inputs.  The scales fold into the softmax scale and the final 1 / l.
// TMEM columns: S_t at t*KT, O_t at NT*KT + t*D (fp32 accumulators, one TMEM
// lane per query row).  Every mbarrier wait is bounded: on timeout the kernel
// records BSA_ERR_DEVICE_TIMEOUT, drains its in-flight copies and MMAs, frees
// TMEM and returns.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "bsa_fp8.cuh"
#include "bsa_internal.h"
#include "bsa_wait.cuh"
#include "sm103_ptx.cuh"

namespace bsa {
namespace {

using wait::Ctl;
using wait::drain_bar;
using wait::report;
using wait::wait_bar;

struct AttnParams {
  const int32_t *kv_idx;  // [b, hkv, nbs, nbs] (sparse) or null (dense)
  const int32_t *kv_cnt;  // [b, hkv, nbs]
  uint16_t *o;            // bf16 [total, hq, d] (= [b, seq, hq, d] when fixed-length)
  float *lse;             // [b, hq, seq] (fixed-length) or [hq, total] (packed), or null
  int32_t *dev_status;    // nullable
  const int32_t *cu;      // packed ragged batch: sequence b is tokens cu[b] .. cu[b+1]-1; or null
  int batch, seq, hq, hkv, nb, group;  // seq: fixed length, or max_seqlen when packed
  int total, nbs;         // tokens in q / k / v / o; per-sequence stride of per-block arrays
  float scale_log2;       // softmax scale * log2(e) (times q_scale * k_scale for fp8 inputs)
  float v_scale;          // 1, or the fp8 value scale
};

template <int D, int BLK, int NT, bool F8 = false>
struct Cfg {
  static constexpr int KT = 128;                    // key-tile rows
  static constexpr bool PAIR = BLK == 64;           // a key tile holds two kept 64-key blocks
  static constexpr int KBOX = PAIR ? 64 : KT;       // key rows per TMA box
  static constexpr int QH = BLK == 64 ? 2 : 1;      // heads stacked in one 128-row Q tile
  static constexpr int QTOK = 128 / QH;             // tokens per Q tile
  static constexpr int NQS = BLK == 256 ? 2 : 1;    // Q tiles along one query block
  static constexpr int SUB = PAIR ? 1 : BLK / KT;   // key tiles per key block (pairs: half a tile each)
  static constexpr int QKB = F8 ? 1 : 2;            // bytes per Q / K element
  static constexpr int CE = 128 / QKB;              // Q / K elements per 128-byte swizzle row
  static constexpr int NCH = D * QKB / 128;         // 128-byte swizzle chunks per Q / K row
  static constexpr int NCHV = D / 64;               // chunks per bf16 V row
  static constexpr int NKK = D * QKB / 32;          // 32-byte K steps of one S = Q K^T
  static_assert(NCH >= 1 && D * QKB % 128 == 0, "Q / K rows are whole 128-byte swizzle rows");
  static_assert(NCHV >= 1, "V rows are whole 128-byte swizzle rows");
  static constexpr uint32_t Q_TILE = 128u * D * QKB;
  static constexpr uint32_t K_TILE = static_cast<uint32_t>(KT) * D * QKB;
  static constexpr uint32_t KV_TILE = static_cast<uint32_t>(KT) * D * 2;  // a bf16 V tile
  static constexpr uint32_t Q_CHUNK = 128u * 128;
  static constexpr uint32_t KV_CHUNK = static_cast<uint32_t>(KT) * 128;
  // Softmax threads per query row: with 128-column key tiles two warps share each
  // 32-row TMEM sub-partition, one per 64-column half, so a tile's softmax takes
  // half as long; they exchange partial row maxima through shared memory.
  static constexpr int CH = KT == 128 ? 2 : 1;
  static constexpr int CW = KT / CH;                 // S columns per softmax thread
  static constexpr uint32_t RED_BYTES = NT * CH * 128 * 2;  // bf16 partial maxima
  // A softmax thread releases its P columns to the P V MMAs in NCHK chunks of 32 S columns
  // (16 key rows of V per MMA, two MMAs per chunk and column half), so the tensor core
  // starts on the first chunk while the second is still being exponentiated.
  static constexpr int NCHK = CW / 32;
  static constexpr int KS = 2;  // K stages: K(n+KS) only needs S(n) done
  // V stages: V(n+VS) needs PV_1(n) done, which comes late; use 3 when they fit
  static constexpr int VS =
      (NT * Q_TILE + KS * K_TILE + 3 * KV_TILE + RED_BYTES + 1024 + 512 <= 227u * 1024) ? 3 : 2;
  static constexpr int TM_O = NT * KT;
  static constexpr int TM_NEED = NT * (KT + D);
  static constexpr uint32_t TM_COLS =
      TM_NEED <= 32 ? 32 : TM_NEED <= 64 ? 64 : TM_NEED <= 128 ? 128 : TM_NEED <= 256 ? 256 : 512;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NT * Q_TILE;
  static constexpr uint32_t OFF_V = OFF_K + KS * K_TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + VS * KV_TILE;
  // barriers: Q, K full/empty, V full/empty, S full[NT], P ready[NT][NCHK], O done[NT],
  // final drain
  static constexpr int B_Q = 0, B_KF = 1, B_KE = B_KF + KS, B_VF = B_KE + KS, B_VE = B_VF + VS,
                       B_SF = B_VE + VS, B_PR = B_SF + NT, B_OD = B_PR + NT * NCHK, B_FIN = B_OD + NT,
                       NBARS = B_FIN + 1;
  static constexpr uint32_t OFF_RED = (OFF_BAR + NBARS * 8 + 16 + 15) / 16 * 16;
  static constexpr uint32_t SMEM_BYTES = OFF_RED + RED_BYTES + 1024;  // + 1 KB alignment slack
  static constexpr int THREADS = 128 + 128 * NT * CH;
  // setmaxnreg split between the producer / MMA warpgroup and the softmax
  // warpgroups; each sum equals the launch allocation (threads x registers):
  //   640 threads x 96 = 128 x 56 + 512 x 104,  384 threads x 168 = 128 x 72 + 256 x 216
  static constexpr int REG_LAUNCH = THREADS == 640 ? 96 : THREADS == 384 ? 168 : 0;
  static constexpr int REG_LOW = THREADS == 640 ? 56 : 72;
  static constexpr int REG_HIGH = THREADS == 640 ? 104 : 216;
  static_assert(REG_LAUNCH == 0 || 128 * REG_LOW + (THREADS - 128) * REG_HIGH <= THREADS * REG_LAUNCH,
                "register split exceeds the launch allocation");
  static constexpr uint32_t IDESC_S = F8 ? ptx::idesc_e4m3_f32(128, KT) : ptx::idesc_bf16_f32(128, KT, false);
  static constexpr uint32_t IDESC_O = ptx::idesc_bf16_f32(128, D, true);
  static_assert(TM_NEED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared-memory budget");
};

template <int D, int BLK, int NT, bool DENSE, bool F8>
__global__ void __launch_bounds__(Cfg<D, BLK, NT, F8>::THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D, BLK, NT, F8>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char *sb = smem_raw + (base - raw);
  const uint32_t sQ = base + C::OFF_Q, sK = base + C::OFF_K, sV = base + C::OFF_V;
  const uint32_t bar0 = base + C::OFF_BAR;
  auto bar = [&](int idx) { return bar0 + 8u * static_cast<uint32_t>(idx); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sb + C::OFF_BAR + C::NBARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const Ctl ctl{abort_flag, p.dev_status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: one (KV head, sequence) after another, so the CTAs running at any time
  // share one head's K and V (64 MB at 128K tokens, inside L2) and re-read it from L2, not
  // HBM; within it heavy rows first (i descending), the head tiles of one row adjacent
  const int nhp = p.group / C::QH / NT;
  int item = blockIdx.x;
  const int hp = item % nhp;
  item /= nhp;
  const int qs = item % C::NQS;
  item /= C::NQS;
  const int i = p.nb - 1 - item % p.nb;
  item /= p.nb;
  const int b = item % p.batch;
  const int g = item / p.batch;
  const int qtok0 = i * BLK + qs * 128;  // first query token of the CTA's tiles (in its sequence)
  const SeqSpan sp = seq_span(p.cu, b, p.seq, p.total, p.dev_status);
  if (qtok0 >= sp.len) return;           // past the end of a shorter sequence: no rows
  const size_t row = (static_cast<size_t>(b) * p.hkv + g) * p.nbs + i;
  int cnt;
  if constexpr (DENSE) {
    cnt = i + 1;
  } else {
    cnt = p.kv_cnt[row];
    cnt = cnt < 0 ? 0 : (cnt > i + 1 ? i + 1 : cnt);
  }
  const int32_t *kvrow = DENSE ? nullptr : p.kv_idx + row * p.nbs;
  // the diagonal block of the first half of a 256-row block has an all-masked second key tile;
  // 64-key blocks go two to a tile (an odd count leaves the last tile's second half empty)
  const int T = C::PAIR ? (cnt + 1) / 2 : cnt * C::SUB - ((C::NQS == 2 && qs == 0 && cnt > 0) ? 1 : 0);
  auto entry_block = [&](int e) -> int { return DENSE ? e : __ldg(kvrow + e); };
  auto key_block = [&](int n) -> int { return entry_block(n / C::SUB); };

  if (threadIdx.x == 0) {
    for (int x = 0; x < C::NBARS; ++x) {
      uint32_t count = 1;
      if (x >= C::B_PR && x < C::B_PR + NT * C::NCHK) count = 4 * C::CH;  // one arrive per softmax warp
      ptx::mbar_init(bar(x), count);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::TM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
  // the producer / MMA warpgroup needs few registers; the softmax warpgroups take the rest
  if constexpr (C::REG_LAUNCH != 0) ptx::setmaxnreg_dec<C::REG_LOW>();
  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0 && T > 0) {
      ptx::tma_prefetch_desc(&tm_q);
      ptx::tma_prefetch_desc(&tm_k);
      ptx::tma_prefetch_desc(&tm_v);
      // L2 priorities: every Q tile is read by one CTA only, while the CTAs running at the
      // same time re-read one KV head's K and V tiles, so Q goes first and K / V stay
      const uint64_t once = ptx::l2_policy_evict_first(), keep = ptx::l2_policy_evict_last();
      ptx::mbar_arrive_expect_tx(bar(C::B_Q), NT * C::Q_TILE);
      for (int t = 0; t < NT; ++t) {
        const int h0 = g * p.group + (hp * NT + t) * C::QH;
        for (int c = 0; c < C::NCH; ++c)
          ptx::tma_load_4d_hint(sQ + t * C::Q_TILE + c * C::Q_CHUNK, &tm_q, bar(C::B_Q), c * C::CE, h0,
                                sp.start + qtok0, 0, once);
      }
      int k_issued = 0, v_issued = 0;  // tiles whose K / V copies were issued
      // first key token of each TMA box of tile n: one box of 128 keys, or (pairs) two
      // boxes of 64, the second a copy of the first when the tile holds one block
      int kt0[2];
      auto tile_tokens = [&](int n) {
        if constexpr (C::PAIR) {
          kt0[0] = sp.start + entry_block(2 * n) * BLK;
          kt0[1] = 2 * n + 1 < cnt ? sp.start + entry_block(2 * n + 1) * BLK : kt0[0];
        } else {
          kt0[0] = sp.start + key_block(n) * BLK + (n % C::SUB) * C::KT;
        }
      };
      constexpr int NBOX = C::PAIR ? 2 : 1;
      constexpr uint32_t BOX_ROWS_BYTES = static_cast<uint32_t>(C::KBOX) * 128;  // one box within a chunk
      for (int n = 0; n < T; ++n) {
        tile_tokens(n);
        const int ks = n % C::KS, ku = n / C::KS;
        if (ku > 0 && !wait_bar(bar(C::B_KE + ks), (ku - 1) & 1, ctl)) break;
        ptx::mbar_arrive_expect_tx(bar(C::B_KF + ks), C::K_TILE);
        for (int x = 0; x < NBOX; ++x)
          for (int c = 0; c < C::NCH; ++c)
            ptx::tma_load_4d_hint(sK + ks * C::K_TILE + c * C::KV_CHUNK + x * BOX_ROWS_BYTES, &tm_k,
                                  bar(C::B_KF + ks), c * C::CE, g, kt0[x], 0, keep);
        k_issued = n + 1;
        const int vs = n % C::VS, vu = n / C::VS;
        if (vu > 0 && !wait_bar(bar(C::B_VE + vs), (vu - 1) & 1, ctl)) break;
        ptx::mbar_arrive_expect_tx(bar(C::B_VF + vs), C::KV_TILE);
        for (int x = 0; x < NBOX; ++x)
          for (int c = 0; c < C::NCHV; ++c)
            ptx::tma_load_4d_hint(sV + vs * C::KV_TILE + c * C::KV_CHUNK + x * BOX_ROWS_BYTES, &tm_v,
                                  bar(C::B_VF + vs), c * 64, g, kt0[x], 0, keep);
        v_issued = n + 1;
      }
      if (*abort_flag) {
        // let every copy still in flight land before the CTA's shared memory is released
        drain_bar(bar(C::B_Q), 0);
        for (int n = k_issued - C::KS > 0 ? k_issued - C::KS : 0; n < k_issued; ++n)
          drain_bar(bar(C::B_KF + n % C::KS), (n / C::KS) & 1);
        for (int n = v_issued - C::VS > 0 ? v_issued - C::VS : 0; n < v_issued; ++n)
          drain_bar(bar(C::B_VF + n % C::VS), (n / C::VS) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0 && T > 0) {
      // descriptors are linear in the start address (14-bit field, shared addresses
      // < 256 KB): each MMA adds a constant to a base built once here
      const uint64_t dq0 = ptx::sdesc_sw128(sQ, 16, 1024);
      const uint64_t dk0 = ptx::sdesc_sw128(sK, 16, 1024);
      const uint64_t dv0 = ptx::sdesc_sw128(sV, C::KV_CHUNK, 1024);
      auto issue_s = [&](int t, int ks) {
        const uint64_t dq = dq0 + static_cast<uint64_t>(t) * (C::Q_TILE >> 4);
        const uint64_t dk = dk0 + static_cast<uint64_t>(ks) * (C::K_TILE >> 4);
        const uint32_t dst = tmem + t * C::KT;
#pragma unroll
        for (int kk = 0; kk < C::NKK; ++kk) {  // 32 bytes of K per MMA (16 bf16 or 32 e4m3)
          const uint64_t qo = ((kk / 4) * C::Q_CHUNK + (kk % 4) * 32) >> 4;
          const uint64_t ko = ((kk / 4) * C::KV_CHUNK + (kk % 4) * 32) >> 4;
          if constexpr (F8) ptx::mma_ss_f8(dst, dq + qo, dk + ko, C::IDESC_S, kk > 0 ? 1u : 0u);
          else ptx::mma_ss(dst, dq + qo, dk + ko, C::IDESC_S, kk > 0 ? 1u : 0u);
        }
        ptx::mma_commit(bar(C::B_SF + t));
      };
      // O_t += P_t V over the key rows of P chunk c: in every column half hf the 32 keys
      // hf * CW + 32 c .. + 31, two MMAs of 16 keys each; the first MMA of a tile's first
      // chunk overwrites O (n == 0) or accumulates into it.  Returns false if a wait gave up.
      auto issue_pv = [&](int t, int vs, int n) -> bool {
        const uint64_t dv = dv0 + static_cast<uint64_t>(vs) * (C::KV_TILE >> 4);
        const uint32_t dst = tmem + C::TM_O + t * D, src = tmem + t * C::KT;
#pragma unroll
        for (int c = 0; c < C::NCHK; ++c) {
          if (!wait_bar(bar(C::B_PR + t * C::NCHK + c), n & 1, ctl)) return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int hf = 0; hf < C::CH; ++hf)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int kk = (hf * C::CW + c * 32) / 16 + e;  // 16 keys of V per MMA
              ptx::mma_ts(dst, src + kk * 8, dv + ((kk * 2048) >> 4), C::IDESC_O,
                          (n > 0 || c > 0 || hf > 0 || e > 0) ? 1u : 0u);
            }
        }
        ptx::mma_commit(bar(C::B_OD + t));
        return true;
      };
      bool ok = wait_bar(bar(C::B_Q), 0, ctl);
      ptx::tc_fence_after();
      for (int n = 0; ok && n < T; ++n) {
        const int ks = n % C::KS;
        if (!(ok = wait_bar(bar(C::B_KF + ks), (n / C::KS) & 1, ctl))) break;
        ptx::tc_fence_after();
        // S_0(n) overwrites the columns PV_0(n-1) reads P_0 from.  tcgen05.mma
        // operations issued by one thread execute in issue order, so S_0(n) is
        // queued right behind PV_0(n-1) without waiting for it to complete.
        issue_s(0, ks);
        // V(n) is waited for here, while the tensor core still works on S_0(n) and the issue
        // of this tile's MMAs is held back by it anyway, so no wait but P_0's stands between
        // S_1(n) and PV_0(n)
        const int vs = n % C::VS;
        if (!(ok = wait_bar(bar(C::B_VF + vs), (n / C::VS) & 1, ctl))) break;
        if constexpr (NT == 2) {
          if (n > 0) {
            // PV_1(n-1) overlaps softmax_0(n); S_1(n) follows it in issue order
            const int pv = n - 1, pvs = pv % C::VS;
            if (!(ok = issue_pv(1, pvs, pv))) break;
            ptx::mma_commit(bar(C::B_VE + pvs));
          }
          issue_s(1, ks);
        }
        if (!(ok = issue_pv(0, vs, n))) break;
        // K(n)'s slot is released only now, so nothing but the wait for P_0 separates S_1(n)
        // from PV_0(n); K(n + KS) still has a whole key tile to arrive
        ptx::mma_commit(bar(C::B_KE + ks));
        if constexpr (NT == 1) ptx::mma_commit(bar(C::B_VE + vs));
      }
      if constexpr (NT == 2) {
        if (ok) {
          const int pv = T - 1, vs = pv % C::VS;
          if ((ok = issue_pv(1, vs, pv))) ptx::mma_commit(bar(C::B_VE + vs));
        }
      }
      if (!ok) {
        // every MMA issued so far must finish before TMEM is released
        ptx::mma_commit(bar(C::B_FIN));
        drain_bar(bar(C::B_FIN), 0);
      }
    }
    __syncwarp();
  }
  } else {
    // ================================================================ softmax + epilogue
    if constexpr (C::REG_LAUNCH != 0) ptx::setmaxnreg_inc<C::REG_HIGH>();
    const int sw = warp - 4;
    const int t = sw / (4 * C::CH);             // query tile of this warp
    const int hf = (sw >> 2) % C::CH;           // column half of the key tile
    const int sub = warp & 3;                   // TMEM sub-partition: rows 32*sub .. 32*sub+31
    const int r = (sub << 5) + lane;            // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(sub << 5) << 16;
    const uint32_t tS = tmem + lane_off + t * C::KT + hf * C::CW;         // this thread's S columns
    const uint32_t tP = tmem + lane_off + t * C::KT + hf * (C::CW / 2);   // its P columns (bf16 pairs)
    constexpr int OD_COLS = D / C::CH;                                    // O columns it rescales / writes
    const uint32_t tO = tmem + lane_off + C::TM_O + t * D + hf * OD_COLS;
    uint16_t *red = reinterpret_cast<uint16_t *>(sb + C::OFF_RED) + (t * C::CH) * 128;
    const int pair_bar = 1 + t * 4 + sub;       // the two warps that share rows 32*sub ..
    const int tok = r / C::QH;
    const int head = g * p.group + (hp * NT + t) * C::QH + (r % C::QH);
    const int qtok = qtok0 + tok;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;               // l: this thread's share of the normaliser
    bool ok = true;

    for (int n = 0; n < T; ++n) {
      // the tile's key block is read before the wait for S, so the read overlaps the wait
      int ktok0;        // key of this thread's column 0
      bool half = true;  // pairs: this thread's half of the tile holds a kept block
      if constexpr (C::PAIR) {
        half = 2 * n + hf < cnt;
        ktok0 = entry_block(half ? 2 * n + hf : 2 * n) * BLK;
      } else {
        ktok0 = key_block(n) * BLK + (n % C::SUB) * C::KT + hf * C::CW;
      }
      if (!(ok = wait_bar(bar(C::B_SF + t), n & 1, ctl))) break;
      ptx::tc_fence_after();
      uint32_t sr[C::CW];
      float pm[C::CW / 32];  // the max of each 32 loaded columns, from the load itself
#pragma unroll
      for (int c = 0; c < C::CW / 32; ++c)
        ptx::tmem_ld32_max(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]), pm[c]);
      ptx::tmem_wait_ld();
      float mx;
      if (!half || ktok0 + C::CW - 1 > qtok0) {
        // columns that overlap the diagonal: key ktok0 + c is visible iff ktok0 + c <= qtok;
        // an empty half masks every column.  The loaded maxima include the masked columns,
        // so the max is taken again over the visible ones (one tile per row at most)
        const int lim = half ? qtok - ktok0 : -1;
#pragma unroll
        for (int c = 0; c < C::CW; ++c)
          if (c > lim) sr[c] = __float_as_uint(-INFINITY);
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = __uint_as_float(sr[e]);
#pragma unroll
        for (int c = 8; c < C::CW; c += 8)
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], __uint_as_float(sr[c + e]));
        mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      } else {
        mx = pm[0];
#pragma unroll
        for (int c = 1; c < C::CW / 32; ++c) mx = fmaxf(mx, pm[c]);
      }
      // the row max of both halves: each half's partial max rounded up to bf16 (any upper
      // bound of the row max is a valid reference, and both halves then hold the same
      // value).  The slot is rewritten only after the partner has arrived on P ready, which
      // the next S tile waits for.
      auto row_max = [&](float part) -> float {
        if constexpr (C::CH == 2) {
          uint32_t u = __float_as_uint(part);
          if ((u & 0xFFFFu) != 0u && !(u >> 31)) u += 0x10000u;
          const uint16_t mine = static_cast<uint16_t>(u >> 16);
          red[hf * 128 + r] = mine;
          ptx::named_barrier(pair_bar, 64);
          const uint16_t other = red[(1 - hf) * 128 + r];
          return fmaxf(__uint_as_float(static_cast<uint32_t>(mine) << 16),
                       __uint_as_float(static_cast<uint32_t>(other) << 16));
        } else {
          return part;
        }
      };
      // the running max moves only when the tile's row max exceeds it by more than 2^8
      // (exact: O and the normaliser share whatever reference is used); the first tile
      // always takes its own.  The decision is the same in both halves of a row (same m,
      // same exchanged max); the O rescale is warp-wide since TMEM accesses are
      // warp-collective, and lanes that keep their max scale by 1.
      const float mt = row_max(mx) * sl2;
      float factor = 1.f;
      bool resc = false;
      if (mt > m + 8.f) {
        factor = m == -INFINITY ? 0.f : ptx::ex2_approx(m - mt);
        resc = m != -INFINITY;  // O holds partial sums only once a finite max was taken
        m = mt;
      }
      // P = 2^(s * scale - m) as bf16 pairs into TMEM over S, with the row sums.  Column
      // pairs go through packed fp32 FMAs and adds (one instruction per pair, each element
      // rounded as the scalar operation would be), the sums in four partial chains.  Each
      // chunk of 32 columns is released to the P V MMAs as soon as its stores (and, in the
      // first chunk, any O rescale) have landed.  The rescale follows the first chunk's
      // stores, when that chunk's S registers are free again.
      const float mb = m == -INFINITY ? 0.f : m;  // (no max yet only after fully masked tiles)
      uint64_t acc[2] = {0ull, 0ull};             // (+0.0f, +0.0f) pairs
      const uint64_t scl = ptx::f32x2(sl2, sl2), neg = ptx::f32x2(-mb, -mb);
#pragma unroll
      for (int c16 = 0; c16 < C::NCHK; ++c16) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t x = ptx::fma_f32x2(
              ptx::f32x2(__uint_as_float(sr[c16 * 32 + 2 * e]), __uint_as_float(sr[c16 * 32 + 2 * e + 1])),
              scl, neg);
          float x0, x1;
          ptx::f32x2_split(x, x0, x1);
          const float p0 = ptx::ex2_approx(x0), p1 = ptx::ex2_approx(x1);
          acc[e & 1] = ptx::add_f32x2(acc[e & 1], ptx::f32x2(p0, p1));
          pk[e] = ptx::pack_bf16x2(p0, p1);
        }
        ptx::tmem_st16(tP + c16 * 16, pk);
        if (c16 == 0 && __any_sync(0xffffffffu, resc)) {
          // eight columns at a time: the second chunk's S values are still live
#pragma unroll 1
          for (int c = 0; c < OD_COLS / 8; ++c) {
            uint32_t ov[8];
            ptx::tmem_ld8(tO + c * 8, ov);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
            ptx::tmem_st8(tO + c * 8, ov);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(C::B_PR + t * C::NCHK + c16));
      }
      float rs4[4];
      ptx::f32x2_split(acc[0], rs4[0], rs4[1]);
      ptx::f32x2_split(acc[1], rs4[2], rs4[3]);
      l = l * factor + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
    }

    if (ok && T > 0) ok = wait_bar(bar(C::B_OD + t), (T - 1) & 1, ctl);
    ptx::tc_fence_after();
    if constexpr (C::CH == 2) {
      // full normaliser = the two halves' shares, added in a fixed order; the Q tiles'
      // shared memory is free once every MMA has completed
      float *lsh = reinterpret_cast<float *>(sb + C::OFF_Q) + (t * C::CH) * 128;
      lsh[hf * 128 + r] = l;
      ptx::named_barrier(pair_bar, 64);
      l = lsh[r] + lsh[128 + r];
    }
    const float inv = (ok && l > 0.f) ? p.v_scale / l : 0.f;
    const bool row_valid = qtok < sp.len;  // a partial last block's tile rows past the sequence end
    const uint64_t o_policy = ptx::l2_policy_evict_first();
    uint16_t *orow = p.o + ((static_cast<size_t>(sp.start) + qtok) * p.hq + head) * D + hf * OD_COLS;
#pragma unroll
    for (int c = 0; c < OD_COLS / 32; ++c) {
      uint32_t ov[32];
      if (T > 0) {
        ptx::tmem_ld32(tO + c * 32, ov);
        ptx::tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) ov[e] = 0u;
      }
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = ptx::pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
      uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
      if (row_valid) {
#pragma unroll
        for (int v = 0; v < 4; ++v)  // O is written once: it leaves L2 first
          ptx::st_global_v4_hint(dst + v, make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]),
                                 o_policy);
      }
    }
    if (p.lse != nullptr && hf == 0 && row_valid) {
      const float lse = (ok && l > 0.f) ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      const size_t at = p.cu == nullptr
                            ? (static_cast<size_t>(b) * p.hq + head) * p.seq + qtok
                            : static_cast<size_t>(head) * p.total + sp.start + qtok;
      p.lse[at] = lse;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TM_COLS);
  }
}

// ---------------------------------------------------------------- host side

// [batch, seq, heads, d] viewed as a 4-D tensor (d innermost), tile box
// {box_inner, box_heads, box_tokens, 1}: bf16 or e4m3 (fp8) elements, 128-byte
// swizzling or none.
bool make_map(EncodeTiledFn fn, CUtensorMap *map, const void *ptr, int batch, int seq, int heads,
              int d, int box_heads, int box_tokens, bool fp8, int box_inner, bool swizzle) {
  const cuuint64_t eb = fp8 ? 1 : 2;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(seq), static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * eb,
                                 static_cast<cuuint64_t>(heads) * d * eb,
                                 static_cast<cuuint64_t>(seq) * heads * d * eb};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_heads),
                             static_cast<cuuint32_t>(box_tokens), 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
            const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int BLK, int NT, bool DENSE, bool F8>
bsa_status launch_t(const AttnShape &s, const void *q, const void *k, const void *v,
                    const AttnParams &prm, cudaStream_t stream, cudaError_t *cerr) {
  using C = Cfg<D, BLK, NT, F8>;
  cudaError_t e = cudaSuccess;
  EncodeTiledFn fn = tensor_map_encoder(&e);
  if (fn == nullptr || e != cudaSuccess) {
    *cerr = e == cudaSuccess ? cudaErrorNotSupported : e;
    return BSA_ERR_CUDA;
  }
  // one token axis over the whole batch: sequence b starts at token b * seq, or at cu[b] when packed
  CUtensorMap mq, mk, mv;
  const bool maps_ok =
      make_map(fn, &mq, q, 1, s.total, s.hq, D, C::QH, C::QTOK, F8, C::CE, true) &&
      make_map(fn, &mk, k, 1, s.total, s.hkv, D, 1, C::KBOX, F8, C::CE, true) &&
      make_map(fn, &mv, v, 1, s.total, s.hkv, D, 1, C::KBOX, false, 64, true);  // bf16 V (widened if fp8)
  if (!maps_ok) {
    *cerr = cudaErrorInvalidValue;
    return BSA_ERR_CUDA;
  }
  auto kern = attn_kernel<D, BLK, NT, DENSE, F8>;
  if constexpr (C::REG_LAUNCH != 0) {
    // setmaxnreg.inc waits until the registers it asks for are free: the split is only
    // safe if the kernel really launches with REG_LAUNCH registers per thread
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) {
      *cerr = e;
      return BSA_ERR_CUDA;
    }
    if (fa.numRegs != C::REG_LAUNCH) return BSA_ERR_UNSUPPORTED;
  }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) {
    *cerr = e;
    return BSA_ERR_CUDA;
  }
  const long long nitems = static_cast<long long>(s.nb) * C::NQS * s.batch * s.hkv * (s.group / C::QH / NT);
  kern<<<static_cast<unsigned>(nitems), C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    *cerr = e;
    return BSA_ERR_CUDA;
  }
  return BSA_OK;
}

template <int D, int BLK, bool DENSE, bool F8>
bsa_status launch_nt(const AttnShape &s, const void *q, const void *k, const void *v,
                     const AttnParams &prm, cudaStream_t st, cudaError_t *cerr) {
  constexpr int QH = BLK == 64 ? 2 : 1;
  if ((s.group / QH) % 2 == 0) return launch_t<D, BLK, 2, DENSE, F8>(s, q, k, v, prm, st, cerr);
  return launch_t<D, BLK, 1, DENSE, F8>(s, q, k, v, prm, st, cerr);
}

template <int D, bool DENSE, bool F8>
bsa_status launch_blk(const AttnShape &s, const void *q, const void *k, const void *v,
                      const AttnParams &prm, cudaStream_t st, cudaError_t *cerr) {
  switch (s.block) {
    case 64: return launch_nt<D, 64, DENSE, F8>(s, q, k, v, prm, st, cerr);
    case 128: return launch_nt<D, 128, DENSE, F8>(s, q, k, v, prm, st, cerr);
    case 256: return launch_nt<D, 256, DENSE, F8>(s, q, k, v, prm, st, cerr);
    default: return BSA_ERR_UNSUPPORTED;
  }
}

// e4m3 codes -> bf16 codes of the same values (exact), 16 per thread per step.
__global__ void __launch_bounds__(256) widen_e4m3_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                         size_t n16) {
  for (size_t e = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; e < n16;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 u = __ldcs(src + e);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[8];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      float f[8];
      e4m3x8_to_f32(make_uint2(w[x], 0u), f);  // the low four bytes of each word
      o[2 * x] = ptx::pack_bf16x2(f[0], f[1]);
      o[2 * x + 1] = ptx::pack_bf16x2(f[2], f[3]);
    }
    __stcs(dst + 2 * e, make_uint4(o[0], o[1], o[2], o[3]));
    __stcs(dst + 2 * e + 1, make_uint4(o[4], o[5], o[6], o[7]));
  }
}

}  // namespace

cudaError_t launch_widen_e4m3(const void *src, void *dst, size_t n, cudaStream_t stream) {
  const size_t n16 = n / 16;  // n is a multiple of 16 (head_dim 128 rows)
  const unsigned grid = static_cast<unsigned>(n16 / 256 + 1 < 152 * 16 ? n16 / 256 + 1 : 152 * 16);
  widen_e4m3_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
  return cudaGetLastError();
}

EncodeTiledFn tensor_map_encoder(cudaError_t *err) {
  static EncodeTiledFn fn = nullptr;
  static cudaError_t status = cudaSuccess;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                              cudaEnableDefault, &q);
    if (status == cudaSuccess && q != cudaDriverEntryPointSuccess) status = cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  *err = status;
  return fn;
}

bsa_status launch_attention(const AttnShape &s, const void *q, const void *k, const void *v,
                            const int32_t *kv_idx, const int32_t *kv_cnt, float scale, void *o,
                            float *lse, int32_t *dev_status, cudaStream_t stream,
                            cudaError_t *cuda_err) {
  *cuda_err = cudaSuccess;
  AttnParams prm{};
  prm.kv_idx = kv_idx;
  prm.kv_cnt = kv_cnt;
  prm.o = static_cast<uint16_t *>(o);
  prm.lse = lse;
  prm.dev_status = dev_status;
  prm.cu = s.cu;
  prm.batch = s.batch;
  prm.seq = s.seq;
  prm.hq = s.hq;
  prm.hkv = s.hkv;
  prm.nb = s.nb;
  prm.group = s.group;
  prm.total = s.total;
  prm.nbs = s.nbs;
  const double qk = s.fp8 ? static_cast<double>(s.q_scale) * s.k_scale : 1.0;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * qk * 1.4426950408889634);
  prm.v_scale = s.fp8 ? s.v_scale : 1.f;
  const bool dense = kv_idx == nullptr;
  if (s.fp8) {
    // e4m3 Q / K rows must fill whole 128-byte swizzle rows: head_dim 128
    if (s.d != 128) return BSA_ERR_UNSUPPORTED;
    return dense ? launch_blk<128, true, true>(s, q, k, v, prm, stream, cuda_err)
                 : launch_blk<128, false, true>(s, q, k, v, prm, stream, cuda_err);
  }
  if (s.d == 64)
    return dense ? launch_blk<64, true, false>(s, q, k, v, prm, stream, cuda_err)
                 : launch_blk<64, false, false>(s, q, k, v, prm, stream, cuda_err);
  if (s.d == 128)
    return dense ? launch_blk<128, true, false>(s, q, k, v, prm, stream, cuda_err)
                 : launch_blk<128, false, false>(s, q, k, v, prm, stream, cuda_err);
  return BSA_ERR_UNSUPPORTED;
}

}  // namespace bsa
