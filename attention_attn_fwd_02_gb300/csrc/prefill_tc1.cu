// prefill_tc1.cu -- tensor-core prefill for head_dim 256 (f16/bf16): one
// 128-row query tile per CTA, 128-key tiles, S double-buffered in TMEM, K and
// V streamed through a ring of 32 KB shared-memory units.
//
// What it computes is the same as prefill_tc.cu: O = softmax(scale * Q K^T +
// mask) V with the online normaliser of "Attention" (recursiveai.org OneGPU
// docs), opening paragraph, the reference-maximum slack and rounded P of that
// page's sections "Apple simdgroup kernel" and "Matrix hardware", and the
// per-tile steps of "attention_forward -- Causal Multi-Head Attention with
// Online Softmax", section "Online Softmax Algoritmasi".
//
// Why a separate shape: at head_dim 256 one accumulator O takes 256 TMEM
// columns, so two query tiles (the ping-pong of the head_dim <= 128 kernel)
// do not fit the 512 columns.  Instead the overlap comes from two S buffers:
// while the softmax warps turn S(i) into P(i), the tensor core runs P(i-1) V
// and S(i+1) = Q K(i+1)^T.
//
// Tile sizes.  A tcgen05.mma costs its issuing thread about 48 cycles
// whatever its size, and an M128 x N64 x K16 product runs in 32, so 64-key
// tiles leave the tensor core waiting on issue; each tile also pays a fixed
// few hundred cycles of barrier and TMEM round trips in the softmax.  Tiles
// of 128 keys give N = 128 for Q K^T (64 cycles per instruction) and halve
// the per-key fixed cost.  With S at 2 x 128 columns and O at 256, TMEM is
// full, so Q stays in shared memory (64 KB); K and V pass through a ring of
// four 32 KB units: a K tile is two units (head-dim halves), a V tile two
// units (key halves), each freed as soon as the MMAs that read it complete.
// The producer fills units in exactly the order the MMA warp consumes them:
// K(0), K(1), then per tile i: V(i), K(i+2).
//
// Softmax: two threads per query row.  Warps w and w + 4 read the same 32
// TMEM lanes (rows); warp w takes keys [0, 64) of every tile and O columns
// [0, 128), warp w + 4 keys [64, 128) and O columns [128, 256).  The two
// threads of a row swap their partial tile maxima through shared memory (an
// mbarrier per warp pair, one phase per exchange), so both hold the same reference
// maximum and make the same rescale decisions; their partial sums l are added
// once, in the epilogue.  Two softmax warps per SM sub-partition hide each
// other's latencies, and each thread's unrolled tile code is half as long.
//
// CTA: 320 threads.  Warps 0-7: softmax; warp 8: TMA producer; warp 9: TMEM
// owner and MMA issuer.  TMEM: S0 [0, 128), S1 [128, 256), O [256, 512).
// All waits are bounded.
#include <string.h>

#include <type_traits>

#include "prefill_tc.h"
#include "tc_ptx.cuh"
#include "tma.h"

namespace attn {
namespace tc1 {

using namespace tc;

constexpr int BM = 128;                 // query rows per CTA
constexpr int BN = 128;                 // keys per tile
constexpr int kThreads = 320;
constexpr int kHalf = BN / 2;           // keys per softmax thread per tile
constexpr int kUnits = 4;               // ring units
constexpr int kUnit = 32768;            // bytes per unit
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kSlack = 8.0f;          // log2 units
// A mask broadcast over heads and rows ([B,1,1,K]) is staged for the CTA's
// whole key range when that range holds at most this many keys.
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
  int lo_u, hi_u;
  uint32_t live;             // staged mask: bit t set when key tile j0 + t has a key of non -inf mask
  int n_live;
  uint8_t list[kMaxListTiles];   // staged mask: the live key tiles, relative to j0, in order
  float red_max[2][2][BM];   // [tile parity][key half][row]: partial tile maxima
  float red_l[2][BM];        // [key half][row]: partial sums for the epilogue
};

template <int D, bool MASK>
struct Cfg {
  static_assert(D == 256, "this kernel is laid out for head_dim 256");
  static constexpr int kQTile = BM * D * 2;                      // 64 KB
  static constexpr int kMaskBytes = MASK ? kMaskCap * 4 : 0;     // staged broadcast mask (16 KB)
  static constexpr int kSmem = kQTile + kUnits * kUnit + kMaskBytes;   // 192 or 208 KB
  static constexpr int kS0 = 0, kS1 = BN, kO = 2 * BN;
  static_assert(kO + D <= 512, "TMEM budget");
  // A K unit holds one head-dim half of a key tile: 2 chunks of [128 keys][128 B].
  // A V unit holds one key half of a value tile: 4 chunks of [64 keys][128 B].
  static_assert(2 * BN * 128 == kUnit && 4 * (BN / 2) * 128 == kUnit, "unit layout");
};

// Unit sequence shared by the producer and the MMA warp: K(0), K(1), then for
// every tile i: V(i), and K(i+2) when it exists.  Each K or V tile is two units.
struct UnitSeq {
  int n_tiles, step = 0;
  // Returns false at the end; otherwise (kind, tile, half): kind 0 = K, 1 = V.
  __device__ bool next(int& kind, int& tile, int& half) {
    const int pre = n_tiles >= 2 ? 4 : 2 * n_tiles;  // prologue units
    if (step < pre) {
      kind = 0;
      tile = step / 2;
      half = step % 2;
    } else {
      // after the prologue: groups of V(i) (2 units) and K(i+2) (2 units if i+2 < n)
      int s = step - pre, i = 0;
      // units per tile i: 2 + (i + 2 < n_tiles ? 2 : 0); the first n_tiles-2 tiles have 4
      const int full_groups = n_tiles > 2 ? n_tiles - 2 : 0;
      if (s < 4 * full_groups) {
        i = s / 4;
        const int r = s % 4;
        kind = r < 2 ? 1 : 0;
        tile = r < 2 ? i : i + 2;
        half = r % 2;
      } else {
        s -= 4 * full_groups;
        i = full_groups + s / 2;
        if (i >= n_tiles) return false;
        kind = 1;
        tile = i;
        half = s % 2;
      }
    }
    ++step;
    return true;
  }
};

template <int D, bool BF16, bool MASK, bool XF>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc1_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const Problem p, const int n_qblocks,
                       const int drop_first_copy, const int mask_stage, const Split sp) {
  using C = Cfg<D, MASK>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* ring = q_s + C::kQTile;
  float* m_s = reinterpret_cast<float*>(ring + kUnits * kUnit);   // staged mask values (MASK only)
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
  const int hb = lpt ? blk % HB : blk / n_qblocks;
  const int qb = lpt ? n_qblocks - 1 - blk / HB : blk % n_qblocks;
  const int h = hb % p.H, b = hb / p.H;
  const int g = h / p.qpg;
  const int q0 = qb * BM;

  if (threadIdx.x == 0) {
    // The copies' descriptors start on their way before anything else.
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    sb.lo_u = 0x7fffffff;
    sb.hi_u = -1;
    sb.live = 0u;
    sb.n_live = 0;
    sb.abort = 0;
    mbar_init(&sb.q_full, 1);
    for (int u = 0; u < kUnits; ++u) {
      mbar_init(&sb.full[u], 1);
      mbar_init(&sb.empty[u], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sb.s_full[i], 1);
      mbar_init(&sb.p_full[i], 2 * BM);
    }
    mbar_init(&sb.o_done, 1);
    mbar_init(&sb.mma_done, 1);
    for (int w = 0; w < 4; ++w) mbar_init(&sb.pair[w], 64);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // Q does not depend on the key range: its copy starts at once.
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
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&sb.tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp < 4 && hi > lo) {   // the rows' ranges (warps 4-7 hold the same rows)
    atomicMin(&sb.lo_u, lo);
    atomicMax(&sb.hi_u, hi);
  }
  __syncthreads();
  const uint32_t tmem = sb.tmem_base;
  const int lo_u = sb.lo_u, hi_u = sb.hi_u;
  const bool any = hi_u > lo_u;
  const int j0 = any ? lo_u / BN : 0;
  const int n_span = any ? (hi_u + BN - 1) / BN - j0 : 0;   // key tiles spanning the union
  // A broadcast mask over a span of at most kMaskCap keys is copied to shared
  // memory once (every softmax thread reads it there), and key tiles whose
  // visible keys all have mask -inf are dropped from the CTA's work: their
  // probabilities are zero, so neither the maximum, the sum nor O sees them.
  // NaN or +inf entries keep their tile (they make rows NaN).
  const int mbase = j0 * BN;
  const bool staged = MASK && mask_stage && n_span > 0 && n_span <= kMaxListTiles;
  if (staged) {
    // Every thread issues all of its loads before using any (one memory round
    // trip), stores the values and marks the tiles of its keys that are live.
    const int mlen = min(p.Sk, (j0 + n_span) * BN) - mbase;
    const float* src = p.M + p.m.off + (int64_t)b * p.m.bs + mbase;
    uint32_t mine = 0u;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      constexpr int kVec = (kMaskCap / 4 + kThreads - 1) / kThreads;
      float4 v[kVec];
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        const int k = 4 * (threadIdx.x + j * kThreads);
        v[j] = k + 3 < mlen ? __ldg(reinterpret_cast<const float4*>(src + k)) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < mlen && k + 3 >= mlen) {   // the ragged end
          v[j].x = src[k];
          v[j].y = k + 1 < mlen ? src[k + 1] : -INFINITY;
          v[j].z = k + 2 < mlen ? src[k + 2] : -INFINITY;
          v[j].w = -INFINITY;
        }
      }
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        const int k = 4 * (threadIdx.x + j * kThreads);
        if (k >= mlen) continue;
        reinterpret_cast<float4*>(m_s)[k / 4] = v[j];
        const float e[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
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
        v[j] = k < mlen ? src[k] : -INFINITY;
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
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      UnitSeq seq{n_tiles};
      int kind, tile, half, issued = 0;
      while (seq.next(kind, tile, half)) {
        const int u = issued % kUnits;
        const uint32_t ph = (uint32_t)(issued / kUnits) & 1u;
        if (!wait_bar(&sb.empty[u], ph ^ 1u, &sb.abort, p.status)) break;
        mbar_expect_tx(&sb.full[u], kUnit);
        uint8_t* dst = ring + u * kUnit;
        const int krow = (j0 + tile_of(tile)) * BN;
        if (drop_first_copy && issued == 0 && blockIdx.x == 0) {
          // Test hook (attn_test_inject): the first CTA's first unit is
          // announced but never copied, so the MMA warp's wait runs out.
        } else if (kind == 0) {
          // head-dim half `half` of K rows [krow, krow + 128): two 64-column chunks
          for (int c = 0; c < 2; ++c)
            tma_load_4d(dst + c * BN * 128, &tm_k, &sb.full[u], (2 * half + c) * 64, krow, g, b);
        } else {
          // key half `half` of V rows: four 64-column chunks of 64 rows
          for (int c = 0; c < 4; ++c)
            tma_load_4d(dst + c * (BN / 2) * 128, &tm_v, &sb.full[u], c * 64, krow + half * (BN / 2), g, b);
        }
        ++issued;
      }
      // Copies still in flight land before the CTA can exit: the last kUnits
      // units issued are the only ones not known to have been consumed.
      drain_bar(&sb.q_full, 0, p.status);
      for (int j = issued > kUnits ? issued - kUnits : 0; j < issued; ++j)
        drain_bar(&sb.full[j % kUnits], (uint32_t)(j / kUnits) & 1u, p.status);
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    // The whole warp runs this code (warp-uniform control flow); one elected
    // lane issues each tcgen05 instruction.  The next ring unit's barrier and
    // the next P's barrier are tested without blocking a batch of MMAs ahead
    // of their use, so a phase that has already completed costs no barrier
    // round trip where the unit or P is taken.
    constexpr uint32_t kIdQK = idesc_f16(BF16, false, BM, BN);
    constexpr uint32_t kIdPV = idesc_f16(BF16, true, BM, D);
    const uint32_t q_addr = su32(q_s), ring_addr = su32(ring);
    // Descriptors of the operand tiles' starts; the K-steps add constants.
    const uint64_t qd = sdesc(q_addr, 16, 1024), ud = sdesc(ring_addr, 16, 1024),
                   vd = sdesc(ring_addr, (BN / 2) * 128, 1024);
    int taken = 0;        // units consumed so far (ring position)
    bool next_ready = false;   // early test of unit `taken`
    bool ok = n_tiles > 0;
    // Waits for the next unit; returns its shared address (0 on abort), and
    // tests the unit after it.
    auto take = [&]() -> uint32_t {
      const int u = taken % kUnits;
      const uint32_t ph = (uint32_t)(taken / kUnits) & 1u;
      ++taken;
      if (!wait_ready(next_ready, &sb.full[u], ph, &sb.abort, p.status)) return 0u;
      next_ready = mbar_test(&sb.full[taken % kUnits], (uint32_t)(taken / kUnits) & 1u);
      return ring_addr + (uint32_t)(u * kUnit);
    };
    // The unit just taken is released when the MMAs issued so far complete.
    auto give = [&]() { mma_commit_w(&sb.empty[(taken - 1) % kUnits]); };
    // S[slot] = Q K(tile)^T: 16 MMAs of K = 16, the first 8 from the low
    // head-dim half of K, the rest from the high half.
    auto issue_qk = [&](int slot) -> bool {
      for (int hf = 0; hf < 2; ++hf) {
        const uint32_t ku = take();
        if (!ku) return false;
        fence_after();
        const uint64_t bd0 = sdesc_add(ud, ku - ring_addr);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int kq = hf * 8 + kk;  // K-step over head_dim
          const uint64_t a = sdesc_add(qd, (uint32_t)((kq / 4) * BM * 128 + (kq % 4) * 32));
          const uint64_t bd = sdesc_add(bd0, (uint32_t)((kk / 4) * BN * 128 + (kk % 4) * 32));
          mma_ss_w(tmem + (slot ? C::kS1 : C::kS0), a, bd, kIdQK, kq > 0);
        }
        give();
      }
      mma_commit_w(&sb.s_full[slot]);
      return true;
    };
    // O += P[slot] V(tile): 8 MMAs of K = 16 keys, 4 per V unit.
    auto issue_pv = [&](int slot, int tile, bool first) -> bool {
      const int k0 = (j0 + tile_of(tile)) * BN;
      for (int hf = 0; hf < 2; ++hf) {
        const uint32_t vu = take();
        if (!vu) return false;
        const int kb = k0 + hf * (BN / 2);
        // Zero the V rows of keys no row of this CTA sees (they may hold anything).
        if (kb < lo_u || kb + BN / 2 > hi_u) {
          uint8_t* vp = ring + (vu - ring_addr);
          for (int w = lane; w < (BN / 2) * 4 * 8; w += 32) {
            const int row = w / 32, rest = w % 32;   // 4 chunks x 8 16-byte pieces per row
            const int kk = kb + row;
            if (kk < lo_u || kk >= hi_u)
              *reinterpret_cast<uint4*>(vp + (rest / 8) * (BN / 2) * 128 + row * 128 + (rest % 8) * 16) =
                  make_uint4(0, 0, 0, 0);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        fence_after();
        const uint64_t bd0 = sdesc_add(vd, vu - ring_addr);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = sdesc_add(bd0, (uint32_t)(kk * 16 * 128));
          mma_ts_w(tmem + C::kO, tmem + (slot ? C::kS1 : C::kS0) + (hf * 4 + kk) * 8, bd, kIdPV,
                   (!first || hf > 0 || kk > 0) ? 1u : 0u);
        }
        give();
      }
      mma_commit_w(&sb.o_done);
      return true;
    };
    if (ok) ok = wait_warp(&sb.q_full, 0, &sb.abort, p.status);
    // Prologue: S of the first two key tiles.
    for (int j = 0; ok && j < 2 && j < n_tiles; ++j) ok = issue_qk(j);
    bool rp = ok && mbar_test(&sb.p_full[0], 0u);
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int slot = i & 1;
      if (!(ok = wait_ready(rp, &sb.p_full[slot], (uint32_t)(i >> 1) & 1u, &sb.abort, p.status))) break;
      if (!(ok = issue_pv(slot, i, i == 0))) break;
      if (i + 1 < n_tiles) rp = mbar_test(&sb.p_full[slot ^ 1], (uint32_t)((i + 1) >> 1) & 1u);
      // Q K^T of tile i+2 into the S buffer P(i) just left (the tensor core
      // runs a thread's MMAs in issue order, so P V(i) reads P first).
      if (i + 2 < n_tiles && !(ok = issue_qk(slot))) break;
    }
    // Every MMA issued above has completed before TMEM is freed.
    if (taken > 0) {
      mma_commit_w(&sb.mma_done);
      if (lane == 0) drain_bar(&sb.mma_done, 0, p.status);
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
    // chosen by the launcher from the same test).
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
      if (!wait_warp(&sb.s_full[slot], (uint32_t)(i >> 1) & 1u, &sb.abort, p.status)) {
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
        if (!wait_warp(&sb.o_done, (uint32_t)(i - 1) & 1u, &sb.abort, p.status)) {
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
      mbar_arrive(&sb.p_full[slot]);
    }
    // ---- epilogue: O / l, special rows, LSE ----
    // A parity wait only tells the current phase from the one before it.
    // S of the last tile being ready implies only that P V of the tile three
    // back has completed (S is double-buffered, so Q K^T of tile i is issued
    // before P V of tile i-1), so o_done may still be two phases short of the
    // final one: wait for the second-to-last phase first, then the last.
    if (ok && n_tiles > 1) ok = wait_warp(&sb.o_done, (uint32_t)(n_tiles - 2) & 1u, &sb.abort, p.status);
    if (ok && n_tiles > 0) ok = wait_warp(&sb.o_done, (uint32_t)(n_tiles - 1) & 1u, &sb.abort, p.status);
    // The row's sum is the two threads' partial sums (same reference maximum).
    sb.red_l[ch][r] = l;
    if (ok) ok = pair_sync(n_tiles);
    l = sb.red_l[0][r] + sb.red_l[1][r];
    if (ok) {
      fence_after();
      const bool valid = qrow < p.Sq;
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
        const int split = (int)(blockIdx.x % sp.n_splits);
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
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
          }
        }
        if (valid && p.lse && ch == 0)
          p.lse[(int64_t)b * p.lse_bs + (int64_t)h * p.lse_hs + qrow] =
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

template <int D, bool BF16, bool MASK, bool XF>
int launch(const Problem& p, const Split& sp, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!tma_map_bhsd(&mq, p.Q, p.dtype, D, p.Sq, p.H, p.B, p.q, BM) ||
      !tma_map_bhsd(&mk, p.K, p.dtype, D, p.Sk, p.G, p.B, p.k, BN) ||
      !tma_map_bhsd(&mv, p.V, p.dtype, D, p.Sk, p.G, p.B, p.v, BN / 2))
    return -1;  // not describable: caller falls back
  const int nqb = (p.Sq + BM - 1) / BM;
  const int64_t blocks = (int64_t)nqb * p.H * p.B * sp.n_splits;
  if (blocks > 0x7fffffff) return -1;
  const int smem = Cfg<D, MASK>::kSmem + 1024;
  auto kern = prefill_tc1_kernel<D, BF16, MASK, XF>;
  cudaError_t e = ensure_smem((const void*)kern, smem);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  const int drop = take_injection() == ATTN_INJECT_DROP_FIRST_COPY ? 1 : 0;
  // A mask broadcast over heads and rows is staged in shared memory.
  const int mask_stage = (MASK && p.m.hs == 0 && p.m.rs == 0) ? 1 : 0;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(mq, mk, mv, p, nqb, drop, mask_stage, sp);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace tc1

namespace tc1 {
template <bool XF>
int launch_x(const Problem& p, const Split& sp, cudaStream_t st) {
  const bool m = p.M != nullptr;
  if (p.dtype == ATTN_BF16)
    return m ? launch<256, true, true, XF>(p, sp, st) : launch<256, true, false, XF>(p, sp, st);
  return m ? launch<256, false, true, XF>(p, sp, st) : launch<256, false, false, XF>(p, sp, st);
}
}  // namespace tc1

int prefill_tc1_launch(const Problem& p, const Split& sp, cudaStream_t st) {
  if (p.D != 256) return -1;
  const bool xf = p.softcap > 0.f || !(p.scale * tc1::kLog2e > 0.f);
  return xf ? tc1::launch_x<true>(p, sp, st) : tc1::launch_x<false>(p, sp, st);
}

}  // namespace attn
