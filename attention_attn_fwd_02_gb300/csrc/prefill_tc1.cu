// prefill_tc1.cu -- tensor-core prefill for head_dim 256 (f16/bf16): one
// 128-row query tile per CTA, 64-key tiles, S double-buffered in TMEM.
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
// and S(i+1) = Q K(i+1)^T.  Shared memory holds Q (64 KB) and a two-stage
// ring of 64-key K and V tiles (32 KB each).
//
// CTA: 192 threads.  Warps 0-3: softmax, one thread per query row (= TMEM
// lane); warp 4: TMA producer; warp 5: TMEM owner and MMA issuer.
// TMEM: S0 [0, 64), S1 [64, 128), O [128, 128 + D).  All waits are bounded.
#include <string.h>

#include <type_traits>

#include "prefill_tc.h"
#include "tc_ptx.cuh"
#include "tma.h"

namespace attn {
namespace tc1 {

using namespace tc;

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 64;   // keys per tile
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kSlack = 8.0f;  // log2 units

struct Bars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done, mma_done;
  uint32_t tmem_base;
  int abort;
  int lo_u, hi_u;
};

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kStages = 2;
  static constexpr int kQTile = BM * D * 2;
  static constexpr int kKTile = BN * D * 2;
  static constexpr int kSmem = kQTile + 2 * kStages * kKTile;
  static constexpr int kS0 = 0, kS1 = BN, kO = 2 * BN;
  static_assert(2 * BN + D <= 512, "TMEM budget");
};

template <int D, bool BF16, bool MASK>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc1_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const Problem p, const int n_qblocks) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* k_s = q_s + C::kQTile;
  uint8_t* v_s = k_s + C::kStages * C::kKTile;
  __shared__ Bars sb;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Launch order.  Causal or segmented problems: heaviest query blocks first
  // (block L covers query block n_qblocks-1-L/(H*B)).  Otherwise every block
  // does the same work, and the query blocks of one (batch, head) run side by
  // side so that its K and V come from DRAM once and from L2 after that.
  const int HB = p.H * p.B;
  const bool lpt = p.causal || p.seg != nullptr;
  const int hb = lpt ? (int)(blockIdx.x % HB) : (int)(blockIdx.x / n_qblocks);
  const int qb = lpt ? n_qblocks - 1 - (int)(blockIdx.x / HB) : (int)(blockIdx.x % n_qblocks);
  const int h = hb % p.H, b = hb / p.H;
  const int g = h / p.qpg;
  const int q0 = qb * BM;

  const int r = warp * 32 + lane;  // softmax row = TMEM lane (warps 0-3)
  const int qrow = q0 + r;
  int lo = 0, hi = 0;
  if (warp < 4 && qrow < p.Sq) {
    int64_t lo64, hi64;
    row_range(p, b, qrow, lo64, hi64);
    lo = (int)lo64;
    hi = (int)(hi64 > lo64 ? hi64 : lo64);
  }
  if (threadIdx.x == 0) {
    sb.lo_u = 0x7fffffff;
    sb.hi_u = -1;
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
    }
    mbar_init(&sb.o_done, 1);
    mbar_init(&sb.mma_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&sb.tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp < 4 && hi > lo) {
    atomicMin(&sb.lo_u, lo);
    atomicMax(&sb.hi_u, hi);
  }
  __syncthreads();
  const uint32_t tmem = sb.tmem_base;
  const int lo_u = sb.lo_u, hi_u = sb.hi_u;
  const bool any = hi_u > lo_u;
  const int j0 = any ? lo_u / BN : 0;
  const int n_tiles = any ? (hi_u + BN - 1) / BN - j0 : 0;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_tiles > 0) {
      int issued = 0, k_only = -1;
      mbar_expect_tx(&sb.q_full, C::kQTile);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_4d(q_s + c * BM * 128, &tm_q, &sb.q_full, c * 64, q0, h, b);
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % C::kStages;
        const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
        const int krow = (j0 + i) * BN;
        if (!wait_bar(&sb.k_empty[s], ph ^ 1u, &sb.abort, p.status)) break;
        mbar_expect_tx(&sb.k_full[s], C::kKTile);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(k_s + s * C::kKTile + c * BN * 128, &tm_k, &sb.k_full[s], c * 64, krow, g, b);
        if (!wait_bar(&sb.v_empty[s], ph ^ 1u, &sb.abort, p.status)) {
          k_only = i;
          break;
        }
        mbar_expect_tx(&sb.v_full[s], C::kKTile);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_4d(v_s + s * C::kKTile + c * BN * 128, &tm_v, &sb.v_full[s], c * 64, krow, g, b);
        issued = i + 1;
      }
      // Copies still in flight land before the CTA can exit.
      drain_bar(&sb.q_full, 0, p.status);
      for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i) {
        drain_bar(&sb.k_full[i % C::kStages], (uint32_t)(i / C::kStages) & 1u, p.status);
        drain_bar(&sb.v_full[i % C::kStages], (uint32_t)(i / C::kStages) & 1u, p.status);
      }
      if (k_only >= 0)
        drain_bar(&sb.k_full[k_only % C::kStages], (uint32_t)(k_only / C::kStages) & 1u, p.status);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t kIdQK = idesc_f16(BF16, false, BM, BN);
    constexpr uint32_t kIdPV = idesc_f16(BF16, true, BM, D);
    const uint32_t q_addr = su32(q_s), k_addr = su32(k_s), v_addr = su32(v_s);
    auto issue_qk = [&](int slot, int s) {  // S[slot] = Q K(stage s)^T
      fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t a = sdesc(q_addr + (uint32_t)((kk / 4) * BM * 128 + (kk % 4) * 32), 16, 1024);
        const uint64_t bd = sdesc(k_addr + s * C::kKTile + (uint32_t)((kk / 4) * BN * 128 + (kk % 4) * 32), 16, 1024);
        mma_ss(tmem + (slot ? C::kS1 : C::kS0), a, bd, kIdQK, kk > 0);
      }
    };
    auto issue_pv = [&](int slot, int s, bool first) {  // O += P[slot] V(stage s)
      fence_after();
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t bd = sdesc(v_addr + s * C::kKTile + kk * 16 * 128, BN * 128, 1024);
        mma_ts(tmem + C::kO, tmem + (slot ? C::kS1 : C::kS0) + kk * 8, bd, kIdPV, (!first || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = n_tiles > 0;
    if (ok) ok = wait_warp(&sb.q_full, 0, &sb.abort, p.status);
    // Prologue: S of the first two key tiles.
    for (int j = 0; ok && j < 2 && j < n_tiles; ++j) {
      if (!(ok = wait_warp(&sb.k_full[j], 0, &sb.abort, p.status))) break;
      if (lane == 0) {
        issue_qk(j, j);
        mma_commit(&sb.s_full[j]);
        mma_commit(&sb.k_empty[j]);
      }
      __syncwarp();
    }
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int s = i % C::kStages;  // stage and S slot coincide
      const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
      const int k0 = (j0 + i) * BN;
      if (!wait_warp(&sb.v_full[s], ph, &sb.abort, p.status)) break;
      // Zero the V rows of keys no row of this CTA sees (they may hold anything).
      if (k0 < lo_u || k0 + BN > hi_u) {
        for (int u = lane; u < BN * C::kChunks * 8; u += 32) {
          const int row = u / (C::kChunks * 8);
          const int rest = u % (C::kChunks * 8);
          const int kk = k0 + row;
          if (kk < lo_u || kk >= hi_u)
            *reinterpret_cast<uint4*>(v_s + s * C::kKTile + (rest / 8) * BN * 128 + row * 128 + (rest % 8) * 16) =
                make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();
      if (!wait_warp(&sb.p_full[s], ph, &sb.abort, p.status)) break;
      if (lane == 0) {
        issue_pv(s, s, i == 0);
        mma_commit(&sb.o_done);
        mma_commit(&sb.v_empty[s]);
      }
      __syncwarp();
      if (i + 2 < n_tiles) {
        if (!wait_warp(&sb.k_full[s], (uint32_t)((i + 2) / C::kStages) & 1u, &sb.abort, p.status)) break;
        if (lane == 0) {
          issue_qk(s, s);
          mma_commit(&sb.s_full[s]);
          mma_commit(&sb.k_empty[s]);
        }
        __syncwarp();
      }
    }
    if (lane == 0 && n_tiles > 0) {
      mma_commit(&sb.mma_done);
      drain_bar(&sb.mma_done, 0, p.status);
    }
    __syncwarp();
  } else {
    // ---------------- softmax: one thread per query row ----------------
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t o_tm = tmem + lane_off + C::kO;
    const float sc = p.scale * kLog2e;
    const bool explicit_x = MASK || !(sc > 0.f);
    const float c_eff = explicit_x ? 1.f : sc;
    const float* mrow = nullptr;
    if (MASK && qrow < p.Sq)
      mrow = p.M + p.m.off + (int64_t)b * p.m.bs + (int64_t)h * p.m.hs + (int64_t)qrow * p.m.rs;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    uint32_t x[BN];
    // The mask slice of a key tile is loaded one tile ahead, so its latency
    // overlaps the current tile's softmax.  A whole in-range, 16-byte-aligned
    // slice is read with vector loads.
    float mv[BN];
    auto load_mask = [&](int k0) {
      const float* mp = mrow ? mrow + k0 : nullptr;
      if (mp && k0 + BN <= p.Sk && ((uintptr_t)mp & 15) == 0) {
#pragma unroll
        for (int j = 0; j < BN / 4; ++j) {
          const float4 v4 = __ldg(reinterpret_cast<const float4*>(mp) + j);
          mv[4 * j] = v4.x;
          mv[4 * j + 1] = v4.y;
          mv[4 * j + 2] = v4.z;
          mv[4 * j + 3] = v4.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < BN; ++e) mv[e] = (mp && k0 + e >= lo && k0 + e < hi) ? mp[e] : 0.f;
      }
    };
    if (MASK && n_tiles > 0) load_mask(j0 * BN);
    for (int i = 0; i < n_tiles; ++i) {
      const int slot = i & 1;
      const uint32_t s_tm = tmem + lane_off + (slot ? C::kS1 : C::kS0);
      if (!wait_warp(&sb.s_full[slot], (uint32_t)(i >> 1) & 1u, &sb.abort, p.status)) {
        ok = false;
        break;
      }
      fence_after();
      const int k0 = (j0 + i) * BN;
      if (explicit_x) {
        // Scores to log2 units plus the additive mask.
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_tm + c * 32, x + c * 32);
        tmem_ld_wait_regs<BN / 32>(x);
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          const int kk = k0 + e;
          const float s = __uint_as_float(x[e]);
          const float v = MASK ? fmaf(s, sc, mv[e] * kLog2e) : s * sc;
          x[e] = __float_as_uint((kk >= lo && kk < hi) ? v : -INFINITY);
        }
        if (MASK && i + 1 < n_tiles) load_mask(k0 + BN);
      } else {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_tm + c * 32, x + c * 32);
        tmem_ld_wait_regs<BN / 32>(x);
        if (!(k0 >= lo && k0 + BN <= hi)) {
#pragma unroll
          for (int e = 0; e < BN; ++e) {
            const int kk = k0 + e;
            if (kk < lo || kk >= hi) x[e] = __float_as_uint(-INFINITY);
          }
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int e = 0; e < BN; e += 4) {
        mx0 = max3(mx0, __uint_as_float(x[e]), __uint_as_float(x[e + 1]));
        mx1 = max3(mx1, __uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]));
      }
      const float mt = fmaxf(mx0, mx1) * c_eff;
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
      l += (la0 + la1) + (lb0 + lb1);
      tmem_st32(s_tm, x);  // P of the 64 keys: 32 packed columns
      if (__any_sync(0xffffffffu, rescale)) {
        // P V of the previous tile must have landed in O before it is scaled.
        if (!wait_warp(&sb.o_done, (uint32_t)(i - 1) & 1u, &sb.abort, p.status)) {
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
    if (ok) {
      fence_after();
      const bool valid = qrow < p.Sq;
      const bool hidden_row = (l == 0.f);  // no visible key; a NaN l stays a NaN row
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      T* orow = valid ? static_cast<T*>(p.O) + p.o.off + (int64_t)b * p.o.bs + (int64_t)h * p.o.hs +
                            (int64_t)qrow * p.o.rs
                      : nullptr;
      const float inv = 1.f / l;
      const float fill = p.masked_zero ? 0.f : NAN;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
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
      if (valid && p.lse)
        p.lse[(int64_t)b * p.lse_bs + (int64_t)h * p.lse_hs + qrow] =
            hidden_row ? -INFINITY : (m_ref + __log2f(l)) * kLn2;
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 5) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

template <int D, bool BF16, bool MASK>
int launch(const Problem& p, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!tma_map_bhsd(&mq, p.Q, p.dtype, D, p.Sq, p.H, p.B, p.q, BM) ||
      !tma_map_bhsd(&mk, p.K, p.dtype, D, p.Sk, p.G, p.B, p.k, BN) ||
      !tma_map_bhsd(&mv, p.V, p.dtype, D, p.Sk, p.G, p.B, p.v, BN))
    return -1;  // not describable: caller falls back
  const int nqb = (p.Sq + BM - 1) / BM;
  const int64_t blocks = (int64_t)nqb * p.H * p.B;
  if (blocks > 0x7fffffff) return -1;
  const int smem = Cfg<D>::kSmem + 1024;
  auto kern = prefill_tc1_kernel<D, BF16, MASK>;
  cudaError_t e = ensure_smem((const void*)kern, smem);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(mq, mk, mv, p, nqb);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace tc1

int prefill_tc1_launch(const Problem& p, cudaStream_t st) {
  const bool m = p.M != nullptr;
  if (p.D != 256) return -1;
  if (p.dtype == ATTN_BF16) return m ? tc1::launch<256, true, true>(p, st) : tc1::launch<256, true, false>(p, st);
  return m ? tc1::launch<256, false, true>(p, st) : tc1::launch<256, false, false>(p, st);
}

}  // namespace attn
