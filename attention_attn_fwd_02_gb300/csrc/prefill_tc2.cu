// prefill_tc2.cu -- tensor-core prefill for head_dim 256 (f16/bf16) on CTA
// pairs: two CTAs of a cluster, each with its own 128 query rows of one
// (batch, head), share every K and V tile through pair MMAs
// (tcgen05.mma.cta_group::2, M = 256).
//
// What it computes is the same as prefill_tc1.cu: O = softmax(scale * Q K^T +
// mask) V with the online normaliser of "Attention" (recursiveai.org OneGPU
// docs), opening paragraph, the reference-maximum slack and rounded P of that
// page's sections "Apple simdgroup kernel" and "Matrix hardware", and the
// per-tile steps of "attention_forward -- Causal Multi-Head Attention with
// Online Softmax", section "Online Softmax Algoritmasi".
//
// Why pairs.  At head_dim 256 one CTA needs 128 KB of K and V per 128-key
// tile against 2048 cycles of MMA work: 64 bytes a cycle from L2 into shared
// memory, the whole of what an SM sustains, plus the tensor core's own reads
// of shared memory.  Measured on GB300, the single-CTA kernel's MMA warp
// waited ~30% of every tile for K/V data.  In a pair MMA the B operand is
// split between the two CTAs (each holds N/2 columns at the same
// shared-memory address) and A and D are per CTA (each its own 128 rows):
// for Q K^T (N = keys) a CTA holds 64 keys of the K tile, for P V (N =
// channels) 128 channels of the V tile, so each SM moves half the bytes per
// tile and the ring of four 32 KB units holds two tiles ahead instead of one.
// One thread of the leader CTA (cluster rank 0) issues every MMA of the pair;
// completions arrive on the barrier at the same offset in both CTAs
// (multicast commit).  TMEM is allocated collectively (one warp in each CTA,
// same address in both).
//
// Readiness across the pair.  The leader's MMA needs both CTAs' data: each
// CTA's producer copies its halves into its own ring and its own barrier
// completes; in the follower a relay warp (warp 9, which issues nothing)
// waits for each of its units and for its Q, zeroes V rows of keys the pair
// does not see, and arrives remotely on the leader's barrier for that unit,
// which counts two arrivals (its own copy's and the relay's).  P is ready when
// the leader's 256 softmax threads and the follower's 8 softmax warps (one
// remote arrival each) have arrived.  Waits on barriers that the other CTA or
// the pair's tensor cores arrive on acquire at cluster scope.  The remote
// arrivals for P and for copied units carry no release: the data they
// announce is complete before them (P's TMEM stores waited for, a unit's
// bytes counted in by its own barrier), and a release at cluster scope cost
// each arrival ~1000 cycles (C5: 135.8 us with release arrivals, 109.2 us
// without).  An arrival after the relay's own shared-memory stores (zeroed V
// rows) keeps the release.
//
// CTA: 320 threads.  Warps 0-7: softmax (two threads per query row, as in
// prefill_tc1.cu); warp 8: TMA producer; warp 9: MMA issuer (leader) or relay
// (follower).  TMEM (per CTA): S0 [0, 128), S1 [128, 256), O [256, 512).
// Segment starts are not taken here (the union of the pair's key ranges is
// formed from its first and last rows).  All waits are bounded; every thread
// of both CTAs reaches the final cluster barrier.
#include <string.h>

#include <type_traits>

#include "prefill_tc.h"
#include "tc_ptx.cuh"
#include "tma.h"

namespace attn {
namespace tc2 {

using namespace tc;

constexpr int BM = 128;                 // query rows per CTA
constexpr int BN = 128;                 // keys per tile
constexpr int kThreads = 320;
constexpr int kHalf = BN / 2;           // keys per softmax thread per tile
constexpr int kUnits = 4;               // ring units
constexpr int kUnit = 32768;            // bytes per unit: a CTA's half of a K or V tile
constexpr int kKHalf = BN / 2;          // keys of a K tile each CTA holds
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kSlack = 8.0f;          // log2 units
constexpr int kMaskCap = 4096;
constexpr int kMaxListTiles = kMaskCap / BN;

struct Bars {
  uint64_t q_full;
  uint64_t full[kUnits], empty[kUnits];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done, mma_done;
  uint64_t pair[4];          // per softmax warp pair (w, w + 4): one phase per exchange
  uint32_t tmem_base;
  int abort;
  uint32_t live;             // staged mask: bit t set when key tile j0 + t has a key of non -inf mask
  int n_live;
  uint8_t list[kMaxListTiles];
  float red_max[2][2][BM];   // [tile parity][key half][row]: partial tile maxima
  float red_l[2][BM];        // [key half][row]: partial sums for the epilogue
};

template <int D, bool MASK>
struct Cfg {
  static_assert(D == 256, "this kernel is laid out for head_dim 256");
  static constexpr int kQTile = BM * D * 2;                      // 64 KB
  static constexpr int kMaskBytes = MASK ? kMaskCap * 4 : 0;     // staged broadcast mask (16 KB)
  static constexpr int kSmem = kQTile + kUnits * kUnit + kMaskBytes;
  static constexpr int kS0 = 0, kS1 = BN, kO = 2 * BN;
  static_assert(kO + D <= 512, "TMEM budget");
  // A K unit: 4 chunks of [64 keys][128 B] (head-dim quarters of this CTA's 64 keys).
  // A V unit: 2 chunks of [128 keys][128 B] (this CTA's 128 channels, 64 each).
  static_assert(4 * kKHalf * 128 == kUnit && 2 * BN * 128 == kUnit, "unit layout");
};

// Unit sequence shared by the producer, the MMA issuer and the relay: K(0),
// K(1), then for every tile i: V(i), and K(i+2) when it exists (one unit each).
struct UnitSeq {
  int n_tiles, step = 0;
  __device__ bool next(int& kind, int& tile) {
    const int pre = n_tiles >= 2 ? 2 : n_tiles;
    if (step < pre) {
      kind = 0;
      tile = step;
    } else {
      int s = step - pre;
      const int full_groups = n_tiles > 2 ? n_tiles - 2 : 0;
      if (s < 2 * full_groups) {
        kind = s % 2 == 0 ? 1 : 0;
        tile = s % 2 == 0 ? s / 2 : s / 2 + 2;
      } else {
        s -= 2 * full_groups;
        const int i = full_groups + s;
        if (i >= n_tiles) return false;
        kind = 1;
        tile = i;
      }
    }
    ++step;
    return true;
  }
};

template <int D, bool BF16, bool MASK, bool XF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const Problem p, const int n_qblocks, const int pair_heads, const int drop_first_copy,
                       const int mask_stage,
                       const int o_tma, const Split sp) {
  using C = Cfg<D, MASK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* ring = q_s + C::kQTile;
  float* m_s = reinterpret_cast<float*>(ring + kUnits * kUnit);   // staged mask values (MASK only)
  __shared__ Bars sb;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_rank();
  // Launch order, by pairs (256-row query blocks): heaviest first under a
  // causal bound, otherwise the query blocks of one (batch, head) side by side.
  // With key ranges (sp.n_splits > 1) each pair takes one range.
  const int pair = (int)(blockIdx.x / 2);
  const int HB = p.H * p.B;
  const bool lpt = p.causal != 0;
  const int blk = sp.n_splits > 1 ? pair / sp.n_splits : pair;
  const int64_t kr0 = sp.n_splits > 1 ? (int64_t)(pair % sp.n_splits) * sp.split_len : 0;
  const int64_t kr1 = sp.n_splits > 1 ? min((int64_t)p.Sk, kr0 + sp.split_len) : (int64_t)p.Sk;
  // The pair's CTAs hold rows [qp0, qp0 + 128) and [qp0 + 128, qp0 + 256) of
  // one head, or with pair_heads (q_len <= 128 and at least two query heads a
  // kv head) rows [0, q_len) of two query heads of one kv head, which then
  // share every K and V tile instead of the follower holding no row.
  int h, b, g, qp0, q0;
  if (pair_heads) {
    const int npg = (p.qpg + 1) / 2;
    const int pr = blk % npg;
    g = (blk / npg) % p.G;
    b = blk / (npg * p.G);
    h = g * p.qpg + 2 * pr + (int)rank;     // this CTA's head
    qp0 = 0;
    q0 = 0;
  } else {
    const int hb = lpt ? blk % HB : blk / n_qblocks;
    const int qb = lpt ? n_qblocks - 1 - blk / HB : blk % n_qblocks;
    h = hb % p.H;
    b = hb / p.H;
    g = h / p.qpg;
    qp0 = qb * 2 * BM;                       // the pair's first row
    q0 = qp0 + (int)rank * BM;               // this CTA's first row
  }
  // (pair_heads with an odd count of query heads: the follower of a group's
  // last pair has no head; it computes along and writes nothing)
  const bool head_ok = h < (g + 1) * p.qpg;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    if (o_tma) prefetch_tmap(&tm_o);
    sb.live = 0u;
    sb.n_live = 0;
    sb.abort = 0;
    // The leader's data barriers also count the follower relay's arrival.
    const uint32_t peers = rank == 0 ? 2u : 1u;
    mbar_init(&sb.q_full, peers);
    for (int u = 0; u < kUnits; ++u) {
      mbar_init(&sb.full[u], peers);
      mbar_init(&sb.empty[u], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], 2 * BM + 8);   // leader: its 256 threads + the follower's 8 warps
    }
    mbar_init(&sb.o_done, 1);
    mbar_init(&sb.mma_done, 1);
    for (int w = 0; w < 4; ++w) mbar_init(&sb.pair[w], 64);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // Q does not depend on the key plan: its copy starts at once (local
    // barrier; the follower forwards its completion to the leader later).
    mbar_expect_tx(&sb.q_full, C::kQTile);
    for (int c = 0; c < D / 64; ++c) tma_load_4d(q_s + c * BM * 128, &tm_q, &sb.q_full, c * 64, q0, h, b);
  }
  const int r = (warp % 4) * 32 + lane;  // softmax row = TMEM lane (warps 0-7)
  const int ch = warp / 4;                // key half / O half of a softmax thread
  const int qrow = q0 + r;
  int lo = 0, hi = 0;
  if (warp < 8 && qrow < p.Sq) {
    int64_t lo64, hi64;
    row_range(p, b, qrow, lo64, hi64);
    lo64 = max(lo64, kr0);
    hi64 = min(hi64, kr1);
    lo = (int)lo64;
    hi = (int)(hi64 > lo64 ? hi64 : lo64);
  }
  // The pair's union of visible key ranges: both ends of a row's range are
  // non-decreasing in the row (no segment starts), so [lo of the pair's first
  // row, hi of its last row) covers it.  Both CTAs compute the same plan.
  int lo_u, hi_u;
  {
    const int last = min(qp0 + 2 * BM, p.Sq) - 1;
    int64_t l64 = 0, h64 = 0, f_lo = 0, f_hi = 0;
    row_range(p, b, last, l64, h64);
    row_range(p, b, qp0, f_lo, f_hi);
    f_lo = max(f_lo, kr0);
    h64 = min(h64, kr1);
    lo_u = (int)f_lo;
    hi_u = h64 > f_lo ? (int)h64 : -1;
  }
  const bool any = hi_u > lo_u;
  const int j0 = any ? lo_u / BN : 0;
  const int n_span = any ? (hi_u + BN - 1) / BN - j0 : 0;   // key tiles spanning the union
  // The first key tiles' halves start their way into L2 while the pair
  // starts up and the mask is scanned (their copies into the ring wait for
  // the live-tile list).
  if (warp == 8 && lane == 0) {
    for (int t = 0; t < 2 && t < n_span; ++t) {
      const int krow = (j0 + t) * BN;
      for (int c = 0; c < 4; ++c) tma_prefetch_4d(&tm_k, c * 64, krow + (int)rank * kKHalf, g, b);
      for (int c = 0; c < 2; ++c) tma_prefetch_4d(&tm_v, ((int)rank * 2 + c) * 64, krow, g, b);
    }
  }
  // A broadcast mask over a span of at most kMaskCap keys is copied to shared
  // memory once (every softmax thread reads it there), and key tiles whose
  // visible keys all have mask -inf are dropped from the CTA's work: their
  // probabilities are zero, so neither the maximum, the sum nor O sees them.
  // NaN or +inf entries keep their tile (they make rows NaN).  Every thread
  // issues its loads (16-byte vectors when the row is aligned) before the
  // pair's start-up barriers, so their latency overlaps them.
  const int mbase = j0 * BN;
  const bool staged = MASK && mask_stage && n_span > 0 && n_span <= kMaxListTiles;
  const int mlen = staged ? min(p.Sk, (j0 + n_span) * BN) - mbase : 0;
  const float* msrc = MASK ? p.M + p.m.off + (int64_t)b * p.m.bs + mbase : nullptr;
  const bool mvec = staged && (reinterpret_cast<uintptr_t>(msrc) & 15) == 0;
  constexpr int kVec = MASK ? (kMaskCap / 4 + kThreads - 1) / kThreads : 1;
  float4 mv4[kVec];
  if (mvec) {
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int k = 4 * (threadIdx.x + j * kThreads);
      mv4[j] = k + 3 < mlen ? __ldg(reinterpret_cast<const float4*>(msrc + k)) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (k < mlen && k + 3 >= mlen) {   // the ragged end
        mv4[j].x = msrc[k];
        mv4[j].y = k + 1 < mlen ? msrc[k + 1] : -INFINITY;
        mv4[j].z = k + 2 < mlen ? msrc[k + 2] : -INFINITY;
        mv4[j].w = -INFINITY;
      }
    }
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&sb.tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  // Both CTAs' barriers exist before either CTA arrives on the other's (their
  // initialisation was released to the cluster by its own fence, so the
  // arrival is relaxed and does not wait for the mask loads in flight).
  cluster_sync_relaxed();
  fence_after();
  const uint32_t tmem = sb.tmem_base;
  if (staged) {
    // Store the values and mark the tiles of this thread's keys that are live.
    uint32_t mine = 0u;
    if (mvec) {
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        const int k = 4 * (threadIdx.x + j * kThreads);
        if (k >= mlen) continue;
        reinterpret_cast<float4*>(m_s)[k / 4] = mv4[j];
        const float e[4] = {mv4[j].x, mv4[j].y, mv4[j].z, mv4[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int key = mbase + k + q;
          if (k + q < mlen && key >= lo_u && key < hi_u && !(e[q] == -INFINITY)) mine |= 1u << ((k + q) / BN);
        }
      }
    } else {
      constexpr int kSc = (kMaskCap + kThreads - 1) / kThreads;
      float v[kSc];
#pragma unroll
      for (int j = 0; j < kSc; ++j) {
        const int k = threadIdx.x + j * kThreads;
        v[j] = k < mlen ? msrc[k] : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < kSc; ++j) {
        const int k = threadIdx.x + j * kThreads;
        if (k >= mlen) continue;
        m_s[k] = v[j];
        const int key = mbase + k;
        if (key >= lo_u && key < hi_u && !(v[j] == -INFINITY)) mine |= 1u << (k / BN);
      }
    }
    mine = __reduce_or_sync(0xffffffffu, mine);
    if (lane == 0 && mine) atomicOr(&sb.live, mine);
    __syncthreads();
    // The i-th live tile is the i-th set bit of the live mask.
    const uint32_t live = sb.live;
    if (threadIdx.x < (unsigned)n_span && ((live >> threadIdx.x) & 1u))
      sb.list[__popc(live & ((1u << threadIdx.x) - 1u))] = (uint8_t)threadIdx.x;
    if (threadIdx.x == 0) sb.n_live = __popc(live);
    __syncthreads();
  }
  const int n_tiles = staged ? sb.n_live : n_span;
  // Key tile (relative to j0) of the CTA's i-th tile of work.
  auto tile_of = [&](int i) -> int { return staged ? (int)sb.list[i] : i; };

  if (warp == 8) {
    // ---------------- TMA producer: this CTA's Q and halves ----------------
    if (lane == 0) {
      UnitSeq seq{n_tiles};
      int kind, tile, issued = 0;
      while (seq.next(kind, tile)) {
        const int u = issued % kUnits;
        const uint32_t ph = (uint32_t)(issued / kUnits) & 1u;
        if (!wait_bar_cl(&sb.empty[u], ph ^ 1u, &sb.abort, p.status)) break;
        mbar_expect_tx(&sb.full[u], kUnit);
        uint8_t* dst = ring + u * kUnit;
        const int krow = (j0 + tile_of(tile)) * BN;
        if (drop_first_copy && issued == 0 && blockIdx.x == 0) {
          // Test hook (attn_test_inject): the leader's first unit is announced
          // but never copied, so the MMA warp's wait runs out.
        } else if (kind == 0) {
          // this CTA's 64 keys of K rows [krow, krow + 128): four 64-column chunks
          for (int c = 0; c < 4; ++c)
            tma_load_4d(dst + c * kKHalf * 128, &tm_k, &sb.full[u], c * 64, krow + (int)rank * kKHalf, g, b);
        } else {
          // this CTA's 128 channels of V rows [krow, krow + 128): two 64-column chunks
          for (int c = 0; c < 2; ++c)
            tma_load_4d(dst + c * BN * 128, &tm_v, &sb.full[u], ((int)rank * 2 + c) * 64, krow, g, b);
        }
        ++issued;
      }
      // Copies still in flight land before the CTA can exit: the last kUnits
      // units issued are the only ones not known to have been consumed.
      drain_bar_cl(&sb.q_full, 0, p.status);
      for (int j = issued > kUnits ? issued - kUnits : 0; j < issued; ++j)
        drain_bar_cl(&sb.full[j % kUnits], (uint32_t)(j / kUnits) & 1u, p.status);
    }
  } else if (warp == 9 && rank == 1) {
    // ---------------- relay (follower): this CTA's data is ready ----------------
    // Waits for its Q and each of its units in the issuer's order, zeroes the
    // V rows of keys the pair does not see, and arrives on the leader's barrier.
    // Q is forwarded even when the pair has no key tile: the leader's
    // producer waits for its Q barrier's phase before it exits.
    bool ok = wait_warp_cl(&sb.q_full, 0, &sb.abort, p.status);
    if (ok && lane == 0) mbar_arrive_remote(&sb.q_full, 0u);
    UnitSeq seq{n_tiles};
    int kind, tile, taken = 0;
    while (ok && seq.next(kind, tile)) {
      const int u = taken % kUnits;
      const uint32_t ph = (uint32_t)(taken / kUnits) & 1u;
      ++taken;
      if (!(ok = wait_warp_cl(&sb.full[u], ph, &sb.abort, p.status))) break;
      const int k0 = (j0 + tile_of(tile)) * BN;
      const bool zeroed = kind == 1 && (k0 < lo_u || k0 + BN > hi_u);
      if (zeroed) {
        uint8_t* vp = ring + u * kUnit;
        for (int w = lane; w < BN * 2 * 8; w += 32) {
          const int row = w / 16, rest = w % 16;   // 2 chunks x 8 16-byte pieces per row
          const int kk = k0 + row;
          if (kk < lo_u || kk >= hi_u)
            *reinterpret_cast<uint4*>(vp + (rest / 8) * BN * 128 + row * 128 + (rest % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      // The unit's bytes are complete in shared memory once its phase
      // completed, so the arrival needs no release, except after this warp's
      // own stores (the zeroed rows).
      if (lane == 0) {
        if (zeroed) mbar_arrive_remote(&sb.full[u], 0u);
        else mbar_arrive_remote_relaxed(&sb.full[u], 0u);
      }
    }
    // The pair's last MMAs write this CTA's TMEM too: they complete before it is freed.
    if (n_tiles > 0 && lane == 0) drain_bar_cl(&sb.mma_done, 0, p.status);
    __syncwarp();
  } else if (warp == 9) {
    // ---------------- MMA issuer (leader): pair MMAs, one elected lane ----------------
    constexpr uint32_t kIdQK = idesc_f16(BF16, false, 2 * BM, BN);
    constexpr uint32_t kIdPV = idesc_f16(BF16, true, 2 * BM, D);
    const uint32_t q_addr = su32(q_s), ring_addr = su32(ring);
    const uint64_t qd = sdesc(q_addr, 16, 1024), ud = sdesc(ring_addr, 16, 1024),
                   vd = sdesc(ring_addr, BN * 128, 1024);
    int taken = 0;
    bool next_ready = false;
    bool ok = n_tiles > 0;
    auto take = [&]() -> uint32_t {
      const int u = taken % kUnits;
      const uint32_t ph = (uint32_t)(taken / kUnits) & 1u;
      ++taken;
      if (!wait_ready_cl(next_ready, &sb.full[u], ph, &sb.abort, p.status)) return 0u;
      next_ready = mbar_test_cl(&sb.full[taken % kUnits], (uint32_t)(taken / kUnits) & 1u);
      return ring_addr + (uint32_t)(u * kUnit);
    };
    // The unit just taken is released in both CTAs when the MMAs issued so far complete.
    auto give = [&]() { mma2_commit_both_w(&sb.empty[(taken - 1) % kUnits]); };
    // S[slot] = Q K^T over the pair: 16 MMAs of K = 16 (head-dim steps), N = 128 keys.
    auto issue_qk = [&](int slot) -> bool {
      const uint32_t ku = take();
      if (!ku) return false;
      fence_after();
      const uint64_t bd0 = sdesc_add(ud, ku - ring_addr);
#pragma unroll
      for (int kq = 0; kq < 16; ++kq) {
        const uint64_t a = sdesc_add(qd, (uint32_t)((kq / 4) * BM * 128 + (kq % 4) * 32));
        const uint64_t bd = sdesc_add(bd0, (uint32_t)((kq / 4) * kKHalf * 128 + (kq % 4) * 32));
        mma2_ss_w(tmem + (slot ? C::kS1 : C::kS0), a, bd, kIdQK, kq > 0);
      }
      give();
      mma2_commit_both_w(&sb.s_full[slot]);
      return true;
    };
    // O += P[slot] V over the pair: 8 MMAs of K = 16 keys, N = 256 channels.
    auto issue_pv = [&](int slot, int tile, bool first) -> bool {
      const uint32_t vu = take();
      if (!vu) return false;
      const int k0 = (j0 + tile_of(tile)) * BN;
      if (k0 < lo_u || k0 + BN > hi_u) {
        uint8_t* vp = ring + (vu - ring_addr);
        for (int w = lane; w < BN * 2 * 8; w += 32) {
          const int row = w / 16, rest = w % 16;
          const int kk = k0 + row;
          if (kk < lo_u || kk >= hi_u)
            *reinterpret_cast<uint4*>(vp + (rest / 8) * BN * 128 + row * 128 + (rest % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      fence_after();
      const uint64_t bd0 = sdesc_add(vd, vu - ring_addr);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t bd = sdesc_add(bd0, (uint32_t)(kk * 16 * 128));
        mma2_ts_w(tmem + C::kO, tmem + (slot ? C::kS1 : C::kS0) + kk * 8, bd, kIdPV, (!first || kk > 0) ? 1u : 0u);
      }
      give();
      mma2_commit_both_w(&sb.o_done);
      return true;
    };
    if (ok) ok = wait_warp_cl(&sb.q_full, 0, &sb.abort, p.status);
    for (int j = 0; ok && j < 2 && j < n_tiles; ++j) ok = issue_qk(j);
    bool rp = ok && mbar_test_cl(&sb.p_full[0], 0u);
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int slot = i & 1;
      if (!(ok = wait_ready_cl(rp, &sb.p_full[slot], (uint32_t)(i >> 1) & 1u, &sb.abort, p.status))) break;
      if (!(ok = issue_pv(slot, i, i == 0))) break;
      if (i + 1 < n_tiles) rp = mbar_test_cl(&sb.p_full[slot ^ 1], (uint32_t)((i + 1) >> 1) & 1u);
      if (i + 2 < n_tiles && !(ok = issue_qk(slot))) break;
    }
    if (taken > 0) {
      mma2_commit_both_w(&sb.mma_done);
      if (lane == 0) drain_bar_cl(&sb.mma_done, 0, p.status);
    }
    __syncwarp();
  } else {
    // ---------------- softmax: two threads per query row ----------------
    const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t o_tm = tmem + lane_off + C::kO + ch * (D / 2);
    // Exchange point of warps w and w + 4: both arrive, then wait (bounded)
    // for the phase; the arrive releases and the wait acquires the shared
    // memory written before it.
    uint64_t* pair_bar = &sb.pair[warp % 4];
    auto pair_sync = [&](int phase) -> bool {
      mbar_arrive(pair_bar);
      return wait_warp(pair_bar, (uint32_t)phase & 1u, &sb.abort, p.status);
    };
    const float sc = p.scale * kLog2e;
    // Soft-capping: the scaled product s becomes cap2 * tanh(s_raw * kinv) in log2 units.
    const bool capped = p.softcap > 0.f;
    const float kinv = capped ? p.scale / p.softcap : 0.f, cap2 = p.softcap * kLog2e;
    // With a mask, no softcap and a positive scale the scores stay in natural
    // units, s * scale + mask (one packed FMA for two keys), and the exponent's
    // multiplier takes log2(e); scores under a softcap or a scale that is not
    // positive are formed in log2 units, in an instantiation of their own (XF,
    // chosen by the launcher from the same test) so that the common kernels do
    // not carry that path.
    const bool mask_nat = MASK && !capped && sc > 0.f;
    const bool explicit_x = XF;
    const float c_eff = mask_nat ? kLog2e : (explicit_x ? 1.f : sc);
    const uint64_t scale2 = f2u(p.scale, p.scale);
    const float* mrow = nullptr;
    if (MASK && qrow < p.Sq)
      mrow = p.M + p.m.off + (int64_t)b * p.m.bs + (int64_t)h * p.m.hs + (int64_t)qrow * p.m.rs;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    uint32_t x[kHalf];
    for (int i = 0; i < n_tiles; ++i) {
      const int slot = i & 1;
      const uint32_t s_tm = tmem + lane_off + (slot ? C::kS1 : C::kS0);
      const int k0 = (j0 + tile_of(i)) * BN + ch * kHalf;   // this thread's first key
      float mv[kHalf];
      if (MASK && staged) {
        // Staged values (keys past k_len hold whatever was there; they are hidden below).
        const float4* ms4 = reinterpret_cast<const float4*>(m_s + (k0 - mbase));
#pragma unroll
        for (int j = 0; j < kHalf / 4; ++j) {
          const float4 v4 = ms4[j];
          mv[4 * j] = v4.x;
          mv[4 * j + 1] = v4.y;
          mv[4 * j + 2] = v4.z;
          mv[4 * j + 3] = v4.w;
        }
      } else if (MASK) {
        // Mask values of this thread's 64 keys (vector loads when the slice is
        // in range and 16-byte aligned; hidden keys read as 0).  Issued before
        // the wait for S so their latency overlaps it.
        const float* mp = mrow ? mrow + k0 : nullptr;
        if (mp && k0 + kHalf <= p.Sk && ((uintptr_t)mp & 15) == 0) {
#pragma unroll
          for (int j = 0; j < kHalf / 4; ++j) {
            const float4 v4 = __ldg(reinterpret_cast<const float4*>(mp) + j);
            mv[4 * j] = v4.x;
            mv[4 * j + 1] = v4.y;
            mv[4 * j + 2] = v4.z;
            mv[4 * j + 3] = v4.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < kHalf; ++e) mv[e] = (mp && k0 + e >= lo && k0 + e < hi) ? mp[e] : 0.f;
        }
      }
      if (!wait_warp_cl(&sb.s_full[slot], (uint32_t)(i >> 1) & 1u, &sb.abort, p.status)) {
        ok = false;
        break;
      }
      fence_after();
      tmem_ld32(s_tm + ch * kHalf, x);
      tmem_ld32(s_tm + ch * kHalf + 32, x + 32);
      tmem_ld_wait_regs<2>(x);
      const bool inside = k0 >= lo && k0 + kHalf <= hi;
      if (mask_nat) {
#pragma unroll
        for (int e = 0; e < kHalf; e += 2) {
          float v0, v1;
          fma2(v0, v1, __uint_as_float(x[e]), __uint_as_float(x[e + 1]), scale2, f2u(mv[e], mv[e + 1]));
          x[e] = __float_as_uint(v0);
          x[e + 1] = __float_as_uint(v1);
        }
        if (!inside) {
#pragma unroll
          for (int e = 0; e < kHalf; ++e) {
            const int kk = k0 + e;
            if (kk < lo || kk >= hi) x[e] = __float_as_uint(-INFINITY);
          }
        }
      } else if (explicit_x) {
        // Scores to log2 units plus the additive mask.
#pragma unroll
        for (int e = 0; e < kHalf; ++e) {
          const int kk = k0 + e;
          const float s = __uint_as_float(x[e]);
          const float t = capped ? cap2 * tanh_exp2(s * kinv) : s * sc;
          const float v = MASK ? fmaf(mv[e], kLog2e, t) : t;
          x[e] = __float_as_uint((kk >= lo && kk < hi) ? v : -INFINITY);
        }
      } else if (!inside) {
#pragma unroll
        for (int e = 0; e < kHalf; ++e) {
          const int kk = k0 + e;
          if (kk < lo || kk >= hi) x[e] = __float_as_uint(-INFINITY);
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int e = 0; e < kHalf; e += 4) {
        mx0 = max3(mx0, __uint_as_float(x[e]), __uint_as_float(x[e + 1]));
        mx1 = max3(mx1, __uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]));
      }
      // Swap partial maxima with the other thread of this row.  The barrier
      // also orders both threads' loads of S before either stores P over it
      // (P of keys 64..127 lands on columns that held S of keys 32..63).
      sb.red_max[slot][ch][r] = fmaxf(mx0, mx1);
      fence_before();
      if (!pair_sync(i)) {
        ok = false;
        break;
      }
      fence_after();
      const float mt = fmaxf(sb.red_max[slot][0][r], sb.red_max[slot][1][r]) * c_eff;
      const bool raise = mt > m_ref + kSlack;  // also true for the first tile with a visible key
      float corr = 1.f;
      if (raise) corr = ex2(m_ref - mt);       // 0 when m_ref = -inf
      const bool rescale = raise && m_ref > -INFINITY;
      if (raise) {
        l *= corr;
        m_ref = mt;
      }
      const float neg = -(m_ref == -INFINITY ? 0.f : m_ref);
      const uint64_t c2 = f2u(c_eff, c_eff), n2 = f2u(neg, neg);
      float la0 = 0.f, la1 = 0.f, lb0 = 0.f, lb1 = 0.f;
#pragma unroll
      for (int e = 0; e < kHalf; e += 4) {
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
      l += (la0 + la1) + (lb0 + lb1);
      tmem_st32(s_tm + ch * (kHalf / 2), x);  // P of this thread's 64 keys: 32 packed columns
      if (__any_sync(0xffffffffu, rescale)) {
        // P V of the previous tile must have landed in O before it is scaled.
        if (!wait_warp_cl(&sb.o_done, (uint32_t)(i - 1) & 1u, &sb.abort, p.status)) {
          ok = false;
          break;
        }
        fence_after();
        const float f = rescale ? corr : 1.f;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
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
      // P(i) of this CTA's rows is in its TMEM: the leader's threads arrive on
      // its P barrier themselves, the follower's warps once each, remotely.
      // The follower's stores of P have completed (tcgen05.wait::st above), so
      // its arrival needs no release; a release arrival at cluster scope costs
      // the warp ~1000 cycles a tile (measured), on the softmax's critical path.
      if (rank == 0) {
        mbar_arrive(&sb.p_full[slot]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(&sb.p_full[slot], 0u);
      }
    }
    // ---- epilogue: O / l, special rows, LSE ----
    // A parity wait only tells the current phase from the one before it.
    // S of the last tile being ready implies only that P V of the tile three
    // back has completed (S is double-buffered, so Q K^T of tile i is issued
    // before P V of tile i-1), so o_done may still be two phases short of the
    // final one: wait for the second-to-last phase first, then the last.
    if (ok && n_tiles > 1) ok = wait_warp_cl(&sb.o_done, (uint32_t)(n_tiles - 2) & 1u, &sb.abort, p.status);
    if (ok && n_tiles > 0) ok = wait_warp_cl(&sb.o_done, (uint32_t)(n_tiles - 1) & 1u, &sb.abort, p.status);
    // The row's sum is the two threads' partial sums (same reference maximum).
    sb.red_l[ch][r] = l;
    if (ok) ok = pair_sync(n_tiles);
    l = sb.red_l[0][r] + sb.red_l[1][r];
    if (ok) {
      fence_after();
      const bool valid = qrow < p.Sq && head_ok;
      // The sink logit joins the denominator (and rescales the accumulated O);
      // with key ranges the merge adds it once.
      const float o_mul = p.sink_on && sp.n_splits == 1 ? fold_sink<true>(m_ref, l, sink_logit(p, h) * kLog2e) : 1.f;
      const bool hidden_row = (l == 0.f);  // no visible key; a NaN l stays a NaN row
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      T* orow = valid ? static_cast<T*>(p.O) + p.o.off + (int64_t)b * p.o.bs + (int64_t)h * p.o.hs +
                            (int64_t)qrow * p.o.rs + ch * (D / 2)
                      : nullptr;
      const float inv = o_mul / l;
      const float fill = p.masked_zero ? 0.f : NAN;
      if (sp.n_splits > 1) {
        // This key range's partial: O / l in float32 (each thread its half of
        // the columns) and its LSE (-inf when the range has no visible key).
        const int split = (int)((blockIdx.x / 2) % sp.n_splits);
        const int64_t prow = ((int64_t)b * p.H + h) * p.Sq + qrow;
        float4* po = reinterpret_cast<float4*>(sp.part_o + (prow * sp.n_splits + split) * D + ch * (D / 2));
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          if (n_tiles > 0) {
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
        if (valid && ch == 0)
          sp.part_lse[prow * sp.n_splits + split] = hidden_row ? -INFINITY : (m_ref + __log2f(l)) * kLn2;
      } else {
        // With a tensor map for O, each warp stages its 32 rows x 128 channels
        // in the ring, in the map's box layout (two boxes of 64 channels, rows
        // of 128 bytes, 16-byte chunks swizzled by the row), and one lane
        // stores them with two tiled copies: full 128-byte lines instead of
        // 16 bytes of 32 rows per store instruction.  The ring is free here:
        // no unit is copied after the last one, and the last P V (which
        // read it) has completed.  Rows past the end of Q are not written.
        const int wr0 = (warp % 4) * 32;   // the warp's first row in the CTA
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          if (n_tiles > 0) {
            tmem_ld32(o_tm + c * 32, o);
            tmem_ld_wait_regs<1>(o);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float a = hidden_row ? fill : __uint_as_float(o[e]) * inv;
            const float bb = hidden_row ? fill : __uint_as_float(o[e + 1]) * inv;
            w[e / 2] = pack2<BF16>(a, bb);
          }
          if (o_tma) {
            uint8_t* rowp = ring + (ch * 2 + c / 2) * (BM * 128) + r * 128;
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              *reinterpret_cast<uint4*>(rowp + ((((c % 2) * 4 + v4) ^ (r & 7)) * 16)) =
                  make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          } else if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        }
        if (o_tma) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0 && q0 + wr0 < p.Sq && head_ok) {
            for (int cc = 0; cc < 2; ++cc)
              tma_store_4d(&tm_o, ring + (ch * 2 + cc) * (BM * 128) + wr0 * 128, (ch * 2 + cc) * 64, q0 + wr0, h, b);
            bulk_store_commit_wait_read();
          }
          __syncwarp();
        }
        if (valid && p.lse && ch == 0)
          p.lse[(int64_t)b * p.lse_bs + (int64_t)h * p.lse_hs + qrow] =
              hidden_row ? -INFINITY : (m_ref + __log2f(l)) * kLn2;
      }
    }
  }

  fence_before();
  __syncthreads();
  // No CTA leaves (or frees TMEM) while the other may still arrive on its barriers.
  cluster_sync();
  if (warp == 9) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

template <int D, bool BF16, bool MASK, bool XF>
int launch(const Problem& p, const Split& sp, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mo;
  if (!tma_map_bhsd(&mq, p.Q, p.dtype, D, p.Sq, p.H, p.B, p.q, BM) ||
      !tma_map_bhsd(&mk, p.K, p.dtype, D, p.Sk, p.G, p.B, p.k, kKHalf) ||
      !tma_map_bhsd(&mv, p.V, p.dtype, D, p.Sk, p.G, p.B, p.v, BN))
    return -1;  // not describable: caller falls back
  // O is stored by tiled copies of 32 rows when TMA can describe it (the
  // final output only: key-range partials are float32 rows of their own).
  const int o_tma = sp.n_splits == 1 && tma_map_bhsd(&mo, p.O, p.dtype, D, p.Sq, p.H, p.B, p.o, 32) ? 1 : 0;
  if (!o_tma) memset(&mo, 0, sizeof mo);
  const int npq = (p.Sq + 2 * BM - 1) / (2 * BM);   // pairs per (batch, head)
  // q_len <= 128 with two or more query heads a kv head: a pair takes two
  // heads of one kv head (one CTA each).
  const int ph = (p.Sq <= BM && p.qpg >= 2) ? 1 : 0;
  const int64_t blocks =
      2 * (ph ? (int64_t)p.B * p.G * ((p.qpg + 1) / 2) : (int64_t)npq * p.H * p.B) * sp.n_splits;
  if (blocks > 0x7fffffff) return -1;
  const int smem = Cfg<D, MASK>::kSmem + 1024;
  auto kern = prefill_tc2_kernel<D, BF16, MASK, XF>;
  cudaError_t e = ensure_smem((const void*)kern, smem);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  const int drop = take_injection() == ATTN_INJECT_DROP_FIRST_COPY ? 1 : 0;
  const int mask_stage = (MASK && p.m.hs == 0 && p.m.rs == 0) ? 1 : 0;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(mq, mk, mv, mo, p, npq, ph, drop, mask_stage, o_tma, sp);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace tc2

namespace tc2 {
template <bool XF>
int launch_x(const Problem& p, const Split& sp, cudaStream_t st) {
  const bool m = p.M != nullptr;
  if (p.dtype == ATTN_BF16)
    return m ? launch<256, true, true, XF>(p, sp, st) : launch<256, true, false, XF>(p, sp, st);
  return m ? launch<256, false, true, XF>(p, sp, st) : launch<256, false, false, XF>(p, sp, st);
}
}  // namespace tc2

int prefill_tc2_launch(const Problem& p, const Split& sp, cudaStream_t st) {
  if (p.D != 256 || p.seg != nullptr) return -1;
  const bool xf = p.softcap > 0.f || !(p.scale * tc2::kLog2e > 0.f);
  return xf ? tc2::launch_x<true>(p, sp, st) : tc2::launch_x<false>(p, sp, st);
}

}  // namespace attn
