// prefill_tc.cu -- tensor-core prefill for sm_103a: TMA-staged Q/K/V tiles,
// S = Q K^T and O += P V as tcgen05 MMAs with TMEM accumulators, online
// softmax in warp-specialised registers.
//
// What it computes: O = softmax(scale * Q K^T + mask) V with the online
// normaliser of "Attention" (recursiveai.org OneGPU docs), opening paragraph,
// and the per-tile steps of "attention_forward -- Causal Multi-Head Attention
// with Online Softmax" (llm.istanbul), section "Online Softmax Algoritmasi".
// Two refinements from "Attention", section "Apple simdgroup kernel": each
// row keeps a reference maximum that is raised only when a tile's maximum
// exceeds it by more than a slack (here 8 in log2 units, so exp2(x - m) <= 256
// in the probabilities), and the accumulator is rescaled only on a raise; and
// from section "Matrix hardware": the probabilities are rounded to the element
// type before the P V product.
//
// CTA: 384 threads (three warpgroups), two 128-row query tiles (256 rows) of
// one (batch, head).
//   warps 0-3  softmax for query tile 0 (thread = one row = one TMEM lane)
//   warps 4-7  softmax for query tile 1
//   warp 8     TMA producer (Q once, then K and V tiles through a ring)
//   warp 9     TMEM owner and MMA issuer (one elected lane issues)
//   warps 10-11 idle: they complete the third warpgroup so that it can hand
//              its registers to the softmax warpgroups (setmaxnreg: 216 per
//              softmax thread, which holds a 128-column row of S without
//              spilling, and 56 per producer thread)
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 and O1 after them; the
// probabilities P overwrite the first BN/2 columns of their S tile as packed
// 16-bit pairs and feed the second MMA straight from TMEM.
//
// The two query tiles ping-pong: while the softmax warps of one tile work on
// S, the tensor core runs P V and the next Q K^T of the other tile.
//
// Every wait is bounded: after ~2 s a waiter raises a CTA abort flag and the
// library status word (ATTN_ERR_DEVICE_TIMEOUT); every role then leaves its
// loop, waits (bounded) for its own copies and MMAs in flight, and the TMEM
// owner frees TMEM before the CTA exits.
#include <string.h>

#include <type_traits>

#include "prefill_tc.h"
#include "tc_ptx.cuh"
#include "tma.h"

namespace attn {
namespace tc {

constexpr int BM = 128;            // query rows per tile
constexpr int BN = 128;            // keys per tile
constexpr int kThreads = 384;  // softmax warpgroups 0-1, producer warpgroup 2 (TMA warp, MMA warp, two idle)
// Per-thread registers after the split.  The block is launched with 168
// (65536 / 384, rounded down to the allocation unit); 8 warps x 216 plus
// 4 warps x 56 is 62464 <= 384 x 168 = 64512, so the increase never waits.
constexpr int kSoftmaxRegs = 216;
constexpr int kProducerRegs = 56;
constexpr int kSplitRegs = 8 * 32 * kSoftmaxRegs + 4 * 32 * kProducerRegs;
static_assert(kSplitRegs <= kThreads * ((65536 / kThreads) & ~7), "register split exceeds the block's registers");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kSlack = 8.0f;     // log2 units

struct Bars {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  int lo_u, hi_u;
  int first_live, last_live;   // a broadcast mask's first / last key with a value other than -inf in the CTA's span
};

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;                  // 64-column (128-byte) chunks
  static constexpr int kStages = D <= 64 ? 4 : 2;
  static constexpr int kQTile = BM * D * 2;               // bytes
  static constexpr int kKTile = BN * D * 2;
  static constexpr int kMaskTile = BN * 4;                // a key tile's broadcast mask values (f32)
  static constexpr int kSmem = 2 * kQTile + 2 * kStages * kKTile + kStages * kMaskTile;
  static constexpr int kS0 = 0, kS1 = BN, kO0 = 2 * BN, kO1 = 2 * BN + D;
  static_assert(2 * BN + 2 * D <= 512, "TMEM budget");
};

// Scores of a tile's keys e outside [a, z) (key offsets within the tile)
// become -inf.  Most tiles that need it are cut at one end only (the causal
// diagonal, a key length), which takes one comparison an element.
template <int N>
__device__ __forceinline__ void hide_outside(uint32_t* x, int a, int z) {
  if (a <= 0) {
#pragma unroll
    for (int e = 0; e < N; ++e)
      if (e >= z) x[e] = __float_as_uint(-INFINITY);
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e)
      if (e < a || e >= z) x[e] = __float_as_uint(-INFINITY);
  }
}

template <int D, bool BF16, bool MASK, bool XF>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Problem p, const int n_qblocks,
                      const int pair_heads, const int mask_bcast, const int drop_first_copy, const Split sp) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* k_s = q_s + 2 * C::kQTile;
  uint8_t* v_s = k_s + C::kStages * C::kKTile;
  // A mask broadcast over heads and rows ([B,1,1,K], 16-byte aligned) is staged
  // per key tile with the V copy and read from here by every softmax thread.
  float* m_s = reinterpret_cast<float*>(v_s + C::kStages * C::kKTile);
  __shared__ Bars sb;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Launch order.  Causal or segmented problems: heaviest query blocks first
  // (block L covers query block n_qblocks-1-L/(H*B)).  Otherwise every block
  // does the same work, and the query blocks of one (batch, head) run side by
  // side so that its K and V come from DRAM once and from L2 after that.
  // With key ranges (sp.n_splits > 1) the ranges of one query block are
  // adjacent in the launch order and each CTA takes one.
  const int HB = p.H * p.B;
  const bool lpt = p.causal || p.seg != nullptr;
  const int blk = sp.n_splits > 1 ? (int)(blockIdx.x / sp.n_splits) : (int)blockIdx.x;
  const int64_t kr0 = sp.n_splits > 1 ? (int64_t)(blockIdx.x % sp.n_splits) * sp.split_len : 0;
  const int64_t kr1 = sp.n_splits > 1 ? min((int64_t)p.Sk, kr0 + sp.split_len) : (int64_t)p.Sk;
  // The two query tiles are rows [q0, q0 + 256) of one head, or with
  // pair_heads (q_len <= 128 and at least two query heads a kv head) rows
  // [0, q_len) of two query heads of one kv head, which then share every K
  // and V tile instead of one tile holding no row.
  int h, b, g, q0;
  if (pair_heads) {
    const int npg = (p.qpg + 1) / 2;
    const int pr = blk % npg;
    g = (blk / npg) % p.G;
    b = blk / (npg * p.G);
    h = g * p.qpg + 2 * pr;
    q0 = 0;
  } else {
    const int hb = lpt ? blk % HB : blk / n_qblocks;
    const int qb = lpt ? n_qblocks - 1 - blk / HB : blk % n_qblocks;
    h = hb % p.H;
    b = hb / p.H;
    g = h / p.qpg;
    q0 = qb * 2 * BM;
  }
  const int ht_step = pair_heads ? 1 : 0;    // query tile 1: head h + ht_step,
  const int rt_step = pair_heads ? 0 : BM;   // rows from q0 + rt_step
  // Without a window or segment starts every row's keys start at the key
  // range's start (kr0, a multiple of BN), so the CTA's first K and V tiles
  // are known before any key length is read from global memory: their copies
  // start at once, with Q's, into stage 0.  (Not with the test hook, which
  // drops the producer's first K copy.)
  // (Nor with a staged broadcast mask, whose -inf keys can move the first tile.)
  const bool early = !(p.causal && p.window >= 0) && p.seg == nullptr && !(drop_first_copy && blockIdx.x == 0) &&
                     !(MASK && mask_bcast);

  if (threadIdx.x == 0) {
    // The copies' descriptors start on their way before anything else.
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    sb.lo_u = 0x7fffffff;
    sb.hi_u = -1;
    sb.first_live = 0x7fffffff;
    sb.last_live = -1;
    sb.abort = 0;
    mbar_init(&sb.q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sb.k_full[s], 1);
      mbar_init(&sb.k_empty[s], 1);
      mbar_init(&sb.v_full[s], 1);
      mbar_init(&sb.v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], BM);
      mbar_init(&sb.o_done[i], 1);
    }
    mbar_init(&sb.mma_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // Q does not depend on the key range: its copy starts at once.
    mbar_expect_tx(&sb.q_full, 2 * C::kQTile);
    for (int tt = 0; tt < 2; ++tt)
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_4d(q_s + tt * C::kQTile + c * BM * 128, &tm_q, &sb.q_full, c * 64, q0 + tt * rt_step,
                    h + tt * ht_step, b);
    if (early) {
      const int krow = (int)kr0;
      mbar_expect_tx(&sb.k_full[0], C::kKTile);
      for (int c = 0; c < C::kChunks; ++c) tma_load_4d(k_s + c * BN * 128, &tm_k, &sb.k_full[0], c * 64, krow, g, b);
      const uint32_t mbytes = MASK && mask_bcast ? (uint32_t)min(BN, p.Sk - krow) * 4u : 0u;
      mbar_expect_tx(&sb.v_full[0], C::kKTile + mbytes);
      if (mbytes) bulk_load(m_s, p.M + p.m.off + (int64_t)b * p.m.bs + krow, mbytes, &sb.v_full[0]);
      for (int c = 0; c < C::kChunks; ++c) tma_load_4d(v_s + c * BN * 128, &tm_v, &sb.v_full[0], c * 64, krow, g, b);
    }
  }
  // ---- row ranges and their union ----
  const int t = warp / 4;                       // query tile of a softmax thread
  const int r = (warp % 4) * 32 + lane;         // row within the tile = TMEM lane
  const int qrow = q0 + t * rt_step + r;
  // (pair_heads with an odd count of query heads: tile 1 may have no head)
  int lo = 0, hi = 0;
  if (warp < 8 && qrow < p.Sq && h + t * ht_step < (g + 1) * p.qpg) {
    int64_t lo64, hi64;
    row_range(p, b, qrow, lo64, hi64);
    lo64 = max(lo64, kr0);
    hi64 = min(hi64, kr1);
    lo = (int)lo64;
    hi = (int)(hi64 > lo64 ? hi64 : lo64);
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&sb.tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  // The union of the rows' visible key ranges.  Without segment starts both
  // ends of a row's range are non-decreasing in the row (the window's left end
  // moves with the diagonal), so [lo of the first row, hi of the last row)
  // covers the union; otherwise reduce over rows.
  // hi_0: the end of query tile 0's visible keys (without segment starts);
  // under a causal bound tile 0 stops one key tile short of tile 1.
  int lo_u, hi_u, hi_0 = 0x7fffffff;
  if (p.seg == nullptr) {
    const int last = min(q0 + 2 * BM, p.Sq) - 1;
    int64_t l64 = 0, h64 = 0, f_lo = 0, f_hi = 0, t_lo = 0, t_hi = 0;
    if (last >= q0) {
      row_range(p, b, last, l64, h64);
      row_range(p, b, q0, f_lo, f_hi);
      row_range(p, b, min(q0 + BM, p.Sq) - 1, t_lo, t_hi);
      f_lo = max(f_lo, kr0);
      h64 = min(h64, kr1);
      hi_0 = (int)min(t_hi, kr1);
    }
    lo_u = (int)f_lo;
    hi_u = h64 > f_lo ? (int)h64 : -1;
  } else {
    if (warp < 8 && hi > lo) {
      atomicMin(&sb.lo_u, lo);
      atomicMax(&sb.hi_u, hi);
    }
    __syncthreads();
    lo_u = sb.lo_u;
    hi_u = sb.hi_u;
  }
  // A broadcast mask whose first or last keys are -inf throughout (key
  // padding, left or right) starts and ends the CTA's key span at its first
  // and last keys with another value: the tiles outside would hold only -inf
  // scores.  NaN and +inf entries count as keys with a value (they make rows
  // NaN).  Spans up to kTrimSpan keys.
  constexpr int kTrimSpan = 4096;
  if (MASK && mask_bcast && hi_u > lo_u && hi_u - lo_u <= kTrimSpan) {
    const float* mr = p.M + p.m.off + (int64_t)b * p.m.bs;
    constexpr int kPer = (kTrimSpan + kThreads - 1) / kThreads;
    float mv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int k = lo_u + (int)threadIdx.x + j * kThreads;
      mv[j] = k < hi_u ? __ldg(mr + k) : -INFINITY;
    }
    int first = 0x7fffffff, last = -1;
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (!(mv[j] == -INFINITY)) {
        const int k = lo_u + (int)threadIdx.x + j * kThreads;
        first = min(first, k);
        last = k;
      }
    first = __reduce_min_sync(0xffffffffu, first);
    last = __reduce_max_sync(0xffffffffu, last);
    if (lane == 0 && last >= 0) {
      atomicMin(&sb.first_live, first);
      atomicMax(&sb.last_live, last);
    }
    __syncthreads();
    if (sb.last_live >= 0) {
      lo_u = sb.first_live;
      hi_u = sb.last_live + 1;
    } else {
      hi_u = lo_u;   // no key with a value: nothing to compute
    }
    hi_0 = min(hi_0, hi_u);
  }
  const uint32_t tmem = sb.tmem_base;
  const bool any = hi_u > lo_u;
  const int j0 = any ? lo_u / BN : 0;
  const int n_tiles = any ? (hi_u + BN - 1) / BN - j0 : 0;
  // Key tiles of query tile 0: a prefix of the CTA's tiles (tile 1 sees at
  // least as far), so the key tiles beyond its last visible key are not
  // computed for it.
  const int n0 = hi_0 >= hi_u ? n_tiles : (hi_0 > lo_u ? (hi_0 + BN - 1) / BN - j0 : 0);

  // Registers move from the producer warpgroup to the softmax warpgroups.
  // Each role sets its own count inside its branch, so no code after the
  // change is compiled under both limits.
  if (warp == 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int issued = early ? 1 : 0;   // tiles whose K and V copies were both issued
      int k_only = -1;              // a tile whose K copy was issued but not its V copy
      for (int i = issued; i < n_tiles; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
        const int krow = (j0 + i) * BN;
        if (!wait_bar(&sb.k_empty[s], ph ^ 1u, &sb.abort, p.status)) break;
        mbar_expect_tx(&sb.k_full[s], C::kKTile);
        // Test hook (attn_test_inject): the first CTA's first K copy is
        // announced but never issued, so the MMA warp's wait runs out.
        const bool dropped = drop_first_copy && i == 0 && blockIdx.x == 0;
        for (int c = 0; c < C::kChunks && !dropped; ++c)
          tma_load_4d(k_s + s * C::kKTile + c * BN * 128, &tm_k, &sb.k_full[s], c * 64, krow, g, b);
        if (!wait_bar(&sb.v_empty[s], ph ^ 1u, &sb.abort, p.status)) {
          k_only = i;
          break;
        }
        const uint32_t mbytes = MASK && mask_bcast ? (uint32_t)min(BN, p.Sk - krow) * 4u : 0u;
        mbar_expect_tx(&sb.v_full[s], C::kKTile + mbytes);
        if (mbytes)
          bulk_load(m_s + s * BN, p.M + p.m.off + (int64_t)b * p.m.bs + krow, mbytes, &sb.v_full[s]);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(v_s + s * C::kKTile + c * BN * 128, &tm_v, &sb.v_full[s], c * 64, krow, g, b);
        issued = i + 1;
      }
      // Copies still in flight land before the CTA can exit.  A stage's
      // earlier copies completed before it was refilled, so the last kStages
      // tiles are the only ones to wait for.
      drain_bar(&sb.q_full, 0, p.status);
      for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
        drain_bar(&sb.k_full[s], ph, p.status);
        drain_bar(&sb.v_full[s], ph, p.status);
      }
      if (k_only >= 0) drain_bar(&sb.k_full[k_only % C::kStages], (uint32_t)(k_only / C::kStages) & 1u, p.status);
    }
  } else if (warp == 9) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    // ---------------- MMA issuer ----------------
    // The whole warp runs this loop (warp-uniform control flow); one elected
    // lane issues each tcgen05 instruction.  Each barrier the issuer needs is
    // first tested without blocking a batch of MMAs ahead of its use, so a
    // phase that has already completed costs no barrier round trip there.
    constexpr uint32_t kIdQK = idesc_f16(BF16, false, BM, BN);
    constexpr uint32_t kIdPV = idesc_f16(BF16, true, BM, D);
    const uint32_t q_addr = su32(q_s), k_addr = su32(k_s), v_addr = su32(v_s);
    bool ok = n_tiles > 0;
    if (ok) ok = wait_warp(&sb.q_full, 0, &sb.abort, p.status);
    // Descriptors of each operand tile's start; the K-steps add constants.
    const uint64_t qd0 = sdesc(q_addr, 16, 1024), qd1 = sdesc(q_addr + C::kQTile, 16, 1024);
    const uint64_t kd0 = sdesc(k_addr, 16, 1024), vd0 = sdesc(v_addr, BN * 128, 1024);
    auto issue_qk = [&](int tt, int s) {
      fence_after();
      const uint64_t ad = tt ? qd1 : qd0;
      const uint64_t bd0 = sdesc_add(kd0, (uint32_t)(s * C::kKTile));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t a = sdesc_add(ad, (uint32_t)((kk / 4) * BM * 128 + (kk % 4) * 32));
        const uint64_t bd = sdesc_add(bd0, (uint32_t)((kk / 4) * BN * 128 + (kk % 4) * 32));
        mma_ss_w(tmem + (tt ? C::kS1 : C::kS0), a, bd, kIdQK, kk > 0);
      }
    };
    auto issue_pv = [&](int tt, int s, bool first) {
      fence_after();
      const uint64_t bd0 = sdesc_add(vd0, (uint32_t)(s * C::kKTile));
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t bd = sdesc_add(bd0, (uint32_t)(kk * 16 * 128));
        mma_ts_w(tmem + (tt ? C::kO1 : C::kO0), tmem + (tt ? C::kS1 : C::kS0) + kk * 8, bd, kIdPV,
                 (!first || kk > 0) ? 1u : 0u);
      }
    };
    // Prologue: S0 and S1 of tile 0.
    if (ok) ok = wait_warp(&sb.k_full[0], 0, &sb.abort, p.status);
    if (ok) {
      if (n0 > 0) {
        issue_qk(0, 0);
        mma_commit_w(&sb.s_full[0]);
      }
      issue_qk(1, 0);
      mma_commit_w(&sb.s_full[1]);
      mma_commit_w(&sb.k_empty[0]);
    }
    bool rv = ok && mbar_test(&sb.v_full[0], 0);   // V(0) landed?
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int s = i % C::kStages;
      const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
      const int k0 = (j0 + i) * BN;
      const bool more = i + 1 < n_tiles;
      const bool has0 = i < n0, more0 = i + 1 < n0;
      const int s1 = (i + 1) % C::kStages;
      const uint32_t ph1 = (uint32_t)((i + 1) / C::kStages) & 1u;
      bool rp0 = !has0 || mbar_test(&sb.p_full[0], (uint32_t)i & 1u);
      if (!(ok = wait_ready(rv, &sb.v_full[s], ph, &sb.abort, p.status))) break;
      // Zero the V rows of keys no row of this CTA sees (they may hold anything).
      if (k0 < lo_u || k0 + BN > hi_u) {
        for (int u = lane; u < BN * C::kChunks * 8; u += 32) {
          const int row = u / (C::kChunks * 8);
          const int rest = u % (C::kChunks * 8);
          const int kk = k0 + row;
          if (kk < lo_u || kk >= hi_u) {
            uint4* dst = reinterpret_cast<uint4*>(v_s + s * C::kKTile + (rest / 8) * BN * 128 + row * 128 +
                                                  (rest % 8) * 16);
            *dst = make_uint4(0, 0, 0, 0);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      const bool rk = !more || mbar_test(&sb.k_full[s1], ph1);
      // Query tile 0: P0 V, then the next S0.
      if (has0) {
        if (!(ok = wait_ready(rp0, &sb.p_full[0], (uint32_t)i & 1u, &sb.abort, p.status))) break;
        issue_pv(0, s, i == 0);
        mma_commit_w(&sb.o_done[0]);
      }
      const bool rp1 = mbar_test(&sb.p_full[1], (uint32_t)i & 1u);
      if (more) {
        if (!(ok = wait_ready(rk, &sb.k_full[s1], ph1, &sb.abort, p.status))) break;
        if (more0) {
          issue_qk(0, s1);
          mma_commit_w(&sb.s_full[0]);
        }
      }
      rv = more && mbar_test(&sb.v_full[s1], ph1);   // for the next tile
      // Query tile 1: P1 V, then the next S1.
      if (!(ok = wait_ready(rp1, &sb.p_full[1], (uint32_t)i & 1u, &sb.abort, p.status))) break;
      issue_pv(1, s, i == 0);
      mma_commit_w(&sb.o_done[1]);
      mma_commit_w(&sb.v_empty[s]);
      if (more) {
        issue_qk(1, s1);
        mma_commit_w(&sb.s_full[1]);
        mma_commit_w(&sb.k_empty[s1]);
      }
    }
    // Every MMA issued above has completed before TMEM is freed.
    if (n_tiles > 0) {
      mma_commit_w(&sb.mma_done);
      if (lane == 0) drain_bar(&sb.mma_done, 0, p.status);
    }
    __syncwarp();
  } else if (warp >= 10) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ---------------- softmax: one thread per query row ----------------
    const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + (t ? C::kS1 : C::kS0);
    const uint32_t o_tm = tmem + lane_off + (t ? C::kO1 : C::kO0);
    const float sc = p.scale * kLog2e;
    // Soft-capping: the scaled product s becomes cap2 * tanh(s_raw * kinv) in log2 units.
    const bool capped = p.softcap > 0.f;
    const float kinv = capped ? p.scale / p.softcap : 0.f, cap2 = p.softcap * kLog2e;
    // Without softcap and with a positive scale the scores of a masked problem
    // stay in natural units, s * scale + mask (one packed FMA for two keys),
    // and the exponent's multiplier takes log2(e).  Scores under a softcap or a
    // scale that is not positive are formed in log2 units one at a time, in an
    // instantiation of their own (XF, chosen by the launcher from the same
    // test), so that the common kernels do not carry that path's registers.
    const bool mask_nat = MASK && !capped && sc > 0.f;
    const bool explicit_x = XF;
    const float c_eff = mask_nat ? kLog2e : (explicit_x ? 1.f : sc);
    const uint64_t scale2 = f2u(p.scale, p.scale);
    const float* mrow = nullptr;
    if (MASK && qrow < p.Sq)
      mrow = p.M + p.m.off + (int64_t)b * p.m.bs + (int64_t)(h + t * ht_step) * p.m.hs + (int64_t)qrow * p.m.rs;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    uint32_t x[BN];
    const int n_my = t ? n_tiles : n0;   // this query tile's key tiles
    // A mask with a row per query (not staged): all 128 values of the tile
    // are loaded into x at once (one memory round trip a tile, not one per
    // few keys), and S is then added to them 32 columns at a time.  Mask
    // values of hidden keys inside the key axis are read and then replaced by
    // -inf with the rest of the hidden scores.  (Issuing these loads before
    // the wait for S keeps x live across it, and the compiler then spills.)
    const bool mask_pf = MASK && mask_nat && !mask_bcast;
    auto load_mask = [&](int i) {
      const int k0 = (j0 + i) * BN;
      const float* mp = mrow ? mrow + k0 : nullptr;
      if (mp && k0 + BN <= p.Sk && ((uintptr_t)mp & 15) == 0) {
#pragma unroll
        for (int j = 0; j < BN / 4; ++j) {
          const float4 v4 = __ldg(reinterpret_cast<const float4*>(mp) + j);
          x[4 * j] = __float_as_uint(v4.x);
          x[4 * j + 1] = __float_as_uint(v4.y);
          x[4 * j + 2] = __float_as_uint(v4.z);
          x[4 * j + 3] = __float_as_uint(v4.w);
        }
      } else {
#pragma unroll
        for (int e = 0; e < BN; ++e) x[e] = __float_as_uint((mp && k0 + e < p.Sk) ? __ldg(mp + e) : 0.f);
      }
    };
    for (int i = 0; i < n_my; ++i) {
      if (!wait_warp(&sb.s_full[t], (uint32_t)i & 1u, &sb.abort, p.status)) {
        ok = false;
        break;
      }
      // The staged mask values arrive with V(i); its stage is freed only after
      // P V(i), so they stay in place while this tile's softmax reads them.
      if (MASK && mask_bcast &&
          !wait_warp(&sb.v_full[i % C::kStages], (uint32_t)(i / C::kStages) & 1u, &sb.abort, p.status)) {
        ok = false;
        break;
      }
      fence_after();
      const int k0 = (j0 + i) * BN;
      const float* ms = m_s + (i % C::kStages) * BN;   // staged mask values of this key tile
      // With a finite reference maximum the tile's P is computed against it
      // directly, without scanning for the tile maximum; a row whose tile sum
      // reaches kLagMax (so some score rose that far above the reference) makes
      // the warp redo the tile with the scan.  Below that bound P keeps its
      // relative precision in its own type (bf16 up to 2^127, f16 up to 65504)
      // and in the f32 sums, so only overflow needs the scan.
      constexpr float kLagMax = BF16 ? 0x1p64f : 0x1p15f;
      bool scan = __any_sync(0xffffffffu, !(m_ref > -INFINITY));
      bool rescale = false;
      float corr = 1.f;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        if (mask_pf) {
          load_mask(i);
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t sv[32];
            tmem_ld32(s_tm + c * 32, sv);
            tmem_ld_wait_regs<1>(sv);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int xe = c * 32 + e;
              float v0, v1;
              fma2(v0, v1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), scale2,
                   f2u(__uint_as_float(x[xe]), __uint_as_float(x[xe + 1])));
              x[xe] = __float_as_uint(v0);
              x[xe + 1] = __float_as_uint(v1);
            }
          }
          if (!(k0 >= lo && k0 + BN <= hi)) {
#pragma unroll
            for (int e = 0; e < BN; ++e) {
              const int kk = k0 + e;
              if (kk < lo || kk >= hi) x[e] = __float_as_uint(-INFINITY);
            }
          }
        } else if (mask_nat) {
          // Staged broadcast mask (out-of-range keys are hidden below).
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            tmem_ld32(s_tm + c * 32, x + c * 32);
            tmem_ld_wait_regs<1>(x + c * 32);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int xe = c * 32 + e;
              float v0, v1;
              fma2(v0, v1, __uint_as_float(x[xe]), __uint_as_float(x[xe + 1]), scale2, f2u(ms[xe], ms[xe + 1]));
              x[xe] = __float_as_uint(v0);
              x[xe + 1] = __float_as_uint(v1);
            }
          }
          if (!(k0 >= lo && k0 + BN <= hi)) {
#pragma unroll
            for (int e = 0; e < BN; ++e) {
              const int kk = k0 + e;
              if (kk < lo || kk >= hi) x[e] = __float_as_uint(-INFINITY);
            }
          }
        } else if (explicit_x) {
          // Scores to log2 units with the additive mask, one 32-column chunk at a
          // time (the wait's memory clobber keeps at most 32 mask loads live).
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            tmem_ld32(s_tm + c * 32, x + c * 32);
            tmem_ld_wait_regs<1>(x + c * 32);
#pragma unroll
            for (int e = c * 32; e < c * 32 + 32; ++e) {
              const int kk = k0 + e;
              float v = -INFINITY;
              if (kk >= lo && kk < hi) {
                const float s = __uint_as_float(x[e]);
                const float t = capped ? cap2 * tanh_exp2(s * kinv) : s * sc;
                v = MASK ? fmaf(mrow[kk], kLog2e, t) : t;
              }
              x[e] = __float_as_uint(v);
              if ((e & 7) == 7) asm volatile("" ::: "memory");  // at most 8 mask loads in flight
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_tm + c * 32, x + c * 32);
          tmem_ld_wait_regs<BN / 32>(x);
          if (!(k0 >= lo && k0 + BN <= hi)) hide_outside<BN>(x, lo - k0, hi - k0);
        }
        if (scan) {
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int e = 0; e < BN; e += 4) {
            mx0 = max3(mx0, __uint_as_float(x[e]), __uint_as_float(x[e + 1]));
            mx1 = max3(mx1, __uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]));
          }
          const float mt = fmaxf(mx0, mx1) * c_eff;
          const bool raise = mt > m_ref + kSlack;     // also true for the first tile with a visible key
          if (raise) corr = ex2(m_ref - mt);          // 0 when m_ref = -inf
          // O holds earlier tiles' sums only if m_ref was finite; it is rescaled
          // below, after P is stored (warp-uniform TMEM traffic).
          rescale = raise && m_ref > -INFINITY;
          if (raise) {
            l *= corr;
            m_ref = mt;
          }
        }
        const float neg = -(m_ref == -INFINITY ? 0.f : m_ref);
        const uint64_t c2 = f2u(c_eff, c_eff), n2 = f2u(neg, neg);
        float la0 = 0.f, la1 = 0.f, lb0 = 0.f, lb1 = 0.f;
#pragma unroll
        for (int e = 0; e < BN; e += 4) {
          float a0, a1, b0, b1;
          fma2(a0, a1, __uint_as_float(x[e]), __uint_as_float(x[e + 1]), c2, n2);
          fma2(b0, b1, __uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]), c2, n2);
          a0 = ex2(a0);
          a1 = ex2(a1);
          b0 = ex2(b0);
          b1 = ex2(b1);
          add2(la0, la1, a0, a1);
          add2(lb0, lb1, b0, b1);
          x[e / 2] = pack2<BF16>(a0, a1);
          x[e / 2 + 1] = pack2<BF16>(b0, b1);
        }
        const float lt = (la0 + la1) + (lb0 + lb1);
        if (scan || !__any_sync(0xffffffffu, lt >= kLagMax)) {   // NaN sums stay (a NaN row)
          l += lt;
          break;
        }
        scan = true;
      }
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) tmem_st32(s_tm + c * 32, x + c * 32);
      if (__any_sync(0xffffffffu, rescale)) {
        // P V of the previous tile must have landed in O before it is scaled.
        if (!wait_warp(&sb.o_done[t], (uint32_t)(i - 1) & 1u, &sb.abort, p.status)) {
          ok = false;
          break;
        }
        fence_after();
        const float f = rescale ? corr : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_tm + c * 32, o);
          tmem_ld_wait_regs<1>(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
          tmem_st32(o_tm + c * 32, o);
        }
      }
      tmem_st_wait();
      fence_before();
      mbar_arrive(&sb.p_full[t]);
    }
    // ---- epilogue: O / l, special rows, LSE ----
    if (ok && n_my > 0) ok = wait_warp(&sb.o_done[t], (uint32_t)(n_my - 1) & 1u, &sb.abort, p.status);
    if (ok) {
      fence_after();
      const int ht = h + t * ht_step;   // this thread's query head
      const bool valid = qrow < p.Sq && ht < (g + 1) * p.qpg;
      // The sink logit joins the denominator (and rescales the accumulated O);
      // with key ranges the merge adds it once.
      const float o_mul = p.sink_on && sp.n_splits == 1 ? fold_sink<true>(m_ref, l, sink_logit(p, ht) * kLog2e) : 1.f;
      const bool hidden_row = (l == 0.f);         // no visible key; a NaN l stays a NaN row
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      T* orow = valid ? static_cast<T*>(p.O) + p.o.off + (int64_t)b * p.o.bs + (int64_t)ht * p.o.hs +
                            (int64_t)qrow * p.o.rs
                      : nullptr;
      const float inv = o_mul / l;
      const float fill = p.masked_zero ? 0.f : NAN;
      if (sp.n_splits > 1) {
        // This key range's partial: O / l in float32 and its LSE (-inf when
        // the range has no visible key; the merge then gives it no weight).
        const int split = (int)(blockIdx.x % sp.n_splits);
        const int64_t prow = ((int64_t)b * p.H + ht) * p.Sq + qrow;
        float4* po = reinterpret_cast<float4*>(sp.part_o + (prow * sp.n_splits + split) * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          if (n_my > 0) {
            tmem_ld32(o_tm + c * 32, o);
            tmem_ld_wait_regs<1>(o);
          }
          if (valid && !hidden_row) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              po[c * 8 + e / 4] = make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                                              __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
          }
        }
        if (valid) sp.part_lse[prow * sp.n_splits + split] = hidden_row ? -INFINITY : (m_ref + __log2f(l)) * kLn2;
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          if (n_my > 0) {
            tmem_ld32(o_tm + c * 32, o);
            tmem_ld_wait_regs<1>(o);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float a = hidden_row ? fill : __uint_as_float(o[e]) * inv;
            float bb = hidden_row ? fill : __uint_as_float(o[e + 1]) * inv;
            w[e / 2] = pack2<BF16>(a, bb);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        }
        if (valid && p.lse)
          p.lse[(int64_t)b * p.lse_bs + (int64_t)ht * p.lse_hs + qrow] =
              hidden_row ? -INFINITY : (m_ref + __log2f(l)) * kLn2;
      }
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 9) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// ---- host side -----------------------------------------------------------------------

template <int D, bool BF16, bool MASK, bool XF>
int launch(const Problem& p, const Split& sp, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!tma_map_bhsd(&mq, p.Q, p.dtype, D, p.Sq, p.H, p.B, p.q, BM) ||
      !tma_map_bhsd(&mk, p.K, p.dtype, D, p.Sk, p.G, p.B, p.k, BN) ||
      !tma_map_bhsd(&mv, p.V, p.dtype, D, p.Sk, p.G, p.B, p.v, BN))
    return -1;  // not describable: caller falls back
  const int nqb = (p.Sq + 2 * BM - 1) / (2 * BM);
  // q_len <= 128 with two or more query heads a kv head: a CTA takes two
  // heads (one query tile each) of one kv head.
  const int pair = (p.Sq <= BM && p.qpg >= 2) ? 1 : 0;
  const int64_t blocks = (pair ? (int64_t)p.B * p.G * ((p.qpg + 1) / 2) : (int64_t)nqb * p.H * p.B) * sp.n_splits;
  if (blocks > 0x7fffffff) return -1;
  const int smem = Cfg<D>::kSmem + 1024;
  auto kern = prefill_tc_kernel<D, BF16, MASK, XF>;
  // setmaxnreg.inc waits until the block's register pool holds the larger
  // count, so the pool the kernel is launched with must cover the split.
  static const bool regs_ok = [] {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, (const void*)prefill_tc_kernel<D, BF16, MASK, XF>) != cudaSuccess) return false;
    return a.numRegs * kThreads >= kSplitRegs;
  }();
  if (!regs_ok) return -1;
  cudaError_t e = ensure_smem((const void*)kern, smem);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  // Broadcast mask rows are copied in bulk: 16-byte aligned rows and tiles
  // whose byte counts are multiples of 16 (key tiles start at multiples of
  // BN, so k_len divisible by 4 suffices).
  const int mask_bcast = (MASK && p.m.hs == 0 && p.m.rs == 0 && p.m.off % 4 == 0 && p.m.bs % 4 == 0 &&
                          (reinterpret_cast<uintptr_t>(p.M) & 15) == 0 && p.Sk % 4 == 0)
                             ? 1
                             : 0;
  const int drop = take_injection() == ATTN_INJECT_DROP_FIRST_COPY ? 1 : 0;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(mq, mk, mv, p, nqb, pair, mask_bcast, drop, sp);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D, bool XF>
int launch_x(const Problem& p, const Split& sp, cudaStream_t st) {
  const bool m = p.M != nullptr;
  if (p.dtype == ATTN_BF16) return m ? launch<D, true, true, XF>(p, sp, st) : launch<D, true, false, XF>(p, sp, st);
  return m ? launch<D, false, true, XF>(p, sp, st) : launch<D, false, false, XF>(p, sp, st);
}

template <int D>
int launch_d(const Problem& p, const Split& sp, cudaStream_t st) {
  const bool xf = p.softcap > 0.f || !(p.scale * kLog2e > 0.f);
  return xf ? launch_x<D, true>(p, sp, st) : launch_x<D, false>(p, sp, st);
}

}  // namespace tc

int prefill_tc_try(const Problem& p, const Split& sp, cudaStream_t st, int* used) {
  *used = 0;
  if (p.dtype != ATTN_BF16 && p.dtype != ATTN_F16) return ATTN_OK;
  if (p.kv_int8) return ATTN_OK;  // int8 caches: the CUDA-core path
  if (p.D != 64 && p.D != 128 && p.D != 256) return ATTN_OK;
  if (p.Sk < 1 || p.Sq < 1) return ATTN_OK;
  if (p.Sk > 0x3fffffff || p.Sq > 0x3fffffff) return ATTN_OK;
  const float sc = p.scale * tc::kLog2e;
  if (!(sc == sc) || isinf(sc)) return ATTN_OK;
  if (!tma_layout_ok(p.Q, p.q, p.Sq, p.H, p.B) || !tma_layout_ok(p.K, p.k, p.Sk, p.G, p.B) ||
      !tma_layout_ok(p.V, p.v, p.Sk, p.G, p.B) || !tma_layout_ok(p.O, p.o, p.Sq, p.H, p.B))
    return ATTN_OK;
  int rc = -1;
  if (p.D == 256) {
    rc = prefill_tc2_launch(p, sp, st);      // CTA pairs
    if (rc < 0) rc = prefill_tc1_launch(p, sp, st);
  } else {
    rc = p.D == 64 ? tc::launch_d<64>(p, sp, st) : tc::launch_d<128>(p, sp, st);
  }
  if (rc < 0) return ATTN_OK;  // tensor map refused: generic path
  *used = 1;
  return rc;
}

}  // namespace attn
