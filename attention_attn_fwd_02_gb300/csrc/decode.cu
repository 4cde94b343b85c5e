// decode.cu -- bandwidth-bound split-range decode pass for head_dim 128
// f16/bf16 caches whose rows are contiguous (a BNSH cache [B, G, cap, 128]).
//
// What it computes: for one query row per (batch, head) against the cached
// keys, the partial softmax-attention result of one contiguous key range --
// LSE_r and O_r = sum_k exp(s_k - LSE_r) V_k -- which the combine kernel
// merges in range order ("Attention" (recursiveai.org OneGPU docs), section
// "Accuracy at long key lengths": key ranges whose cut depends only on the
// shape, merged in range order; "com.microsoft.GroupQueryAttention", section
// "Implementation variants": split-K decode; "attention_forward -- Causal
// Multi-Head Attention with Online Softmax", section "attention_decode Farki":
// one query row per head against the cache).
//
// One CTA (4 warps) owns one (batch, kv head, key range) and up to 16 query
// heads of that kv head, so each cache byte is read once.  The range streams
// through shared memory in 64-key stages, two deep (64 KB, so three CTAs
// share an SM: more resident warps beat a deeper ring, measured against three
// and four stages), copied by TMA with 128-byte swizzle; warp w takes keys
// 16w..16w+15 of a stage.  The per-group
// contractions run on the tensor cores with mma.sync (m16n8k16, f32
// accumulation) only to keep instruction issue far below the HBM rate: with
// the CTA's query heads as the 16 MMA rows (zero-padded), S[head][key] = Q K^T
// takes K through conflict-free ldmatrix reads, and P (rounded to the element
// type) -- whose accumulator layout is the A-operand layout of the next MMA --
// multiplies V read through ldmatrix.trans.  Each warp keeps its own
// online-softmax state (reference maximum with a slack of 8 in log2 units,
// as in "Attention", section "Apple simdgroup kernel"); the four warps merge
// in warp order at the end.  All sums have a fixed order.  Waits are bounded
// (status word on timeout).
//
// Test hook: with the one-shot fault of attn_test_inject armed, the first CTA
// announces but never issues its first stage copy, so its waits run out; the
// kernel then records ATTN_ERR_DEVICE_TIMEOUT, drains its other copies and
// exits (a test reads the status word).  Nothing else changes.
#include <limits.h>

#include <type_traits>

#include "decode.h"
#include "tma.h"

namespace attn {
namespace dec {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kRowBytes = kD * 2;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kSlack = 8.0f;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; on timeout raises the CTA abort flag and the status word.
__device__ __forceinline__ bool wait_bar(uint64_t* b, uint32_t parity, int* abort_flag, int* status) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!mbar_try(b, parity)) {
    if (*(volatile int*)abort_flag) return false;
    if (gtimer() - t0 > kTimeoutNs) {
      *(volatile int*)abort_flag = 1;
      atomicExch(status, ATTN_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void drain_bar(uint64_t* b, uint32_t parity, int* status) {
  const uint64_t t0 = gtimer();
  while (!mbar_try(b, parity))
    if (gtimer() - t0 > kTimeoutNs) {
      atomicExch(status, ATTN_ERR_DEVICE_TIMEOUT);
      return;
    }
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- tensor-core (mma.sync) variant ------------------------------------------------------
//
// The same split pass with the per-group contractions on the tensor cores, to
// cut instruction issue so the pass can run at the HBM rate.  Stages of 64
// keys arrive by TMA (128-byte swizzle, so ldmatrix reads are conflict-free);
// warp w takes keys 16w..16w+15 of a stage.  With the query heads of the CTA
// as the M = 16 rows (zero-padded):  S[head][key] = Q K^T by m16n8k16 MMAs
// (B = K rows through ldmatrix), then P (rounded to the element type) is the
// A operand of O[head][d] += P V (B = V rows through ldmatrix.trans); the S
// accumulator layout is the P operand layout, so P never leaves registers.

constexpr int kMStageKeys = 64;
constexpr int kMStages = 2;
constexpr int kMTile = kMStageKeys * kRowBytes;  // K or V tile of a stage (two 64-column chunks)
constexpr int kMHeads = 16;                      // query heads per CTA (MMA rows)

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}
// Byte offset of (row, element d) in a 64-row tile written by TMA with
// 128-byte swizzle: 64-element chunks of 8 KB; in a row the 16-byte unit u
// sits at u ^ (row % 8).
__device__ __forceinline__ uint32_t sw_off(int row, int d) {
  return (uint32_t)((d >> 6) * (kMStageKeys * 128) + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4));
}

// XF: scores under a softcap or an additive mask (an instantiation of its
// own, so that the plain kernel carries neither path).
template <bool BF16, bool XF>
__global__ void __launch_bounds__(kThreads) decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                              const __grid_constant__ CUtensorMap tm_v,
                                                              const Problem p, const Split sp, const int n_hc,
                                                              const int drop_first_copy) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kMStages], empty[kMStages];
  __shared__ int abort_flag;
  __shared__ float red_m[kWarps][kMHeads], red_l[kWarps][kMHeads];

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, gid = lane >> 2, tig = lane & 3;
  int64_t blk = blockIdx.x;
  const int split = (int)(blk % sp.n_splits);
  blk /= sp.n_splits;
  const int hc = (int)(blk % n_hc);
  blk /= n_hc;
  const int g = (int)(blk % p.G);
  const int b = (int)(blk / p.G);
  const int h0 = g * p.qpg + hc * kMHeads;
  const int nh = min(kMHeads, p.qpg - hc * kMHeads);

  // Decode with append: the CTAs of the range holding the new row write it
  // first; the proxy fence orders those writes before this CTA's TMA reads.
  if (p.k_new) {
    const int64_t row = append_target(p, b);
    if (row >= 0 && row / sp.split_len == split) {
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      append_row<T>(p, b, g, row);
      __syncthreads();
      if (tid == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  }
  int64_t lo, hi;
  row_range(p, b, 0, lo, hi);
  const int64_t k_begin = (int64_t)split * sp.split_len;
  const int64_t start = max(lo, k_begin);
  const int64_t end = min(hi, k_begin + sp.split_len);
  if (start >= end) {  // empty range: the combine ignores it
    for (int i = tid; i < nh * kD; i += kThreads) {
      const int64_t row = (int64_t)b * p.H + h0 + i / kD;
      sp.part_o[(row * sp.n_splits + split) * kD + i % kD] = 0.f;
    }
    if (tid < nh) sp.part_lse[((int64_t)b * p.H + h0 + tid) * sp.n_splits + split] = -INFINITY;
    return;
  }

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kMStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int n_chunks = (int)((end - start + kMStageKeys - 1) / kMStageKeys);
  auto issue = [&](int ch) {
    const int s = ch % kMStages;
    const int row0 = (int)(start + (int64_t)ch * kMStageKeys);
    uint8_t* ks = smem + s * 2 * kMTile;
    mbar_expect_tx(&full[s], 2 * kMTile);
    if (drop_first_copy && ch == 0 && blockIdx.x == 0) return;  // test hook: the stage never lands
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      tma_load_4d(ks + c * (kMStageKeys * 128), &tm_k, &full[s], c * 64, row0, g, b);
      tma_load_4d(ks + kMTile + c * (kMStageKeys * 128), &tm_v, &full[s], c * 64, row0, g, b);
    }
  };
  int issued = 0;
  if (tid == 0)
    for (; issued < min(kMStages, n_chunks); ++issued) issue(issued);

  // Q as the A operand: rows = heads (gid, gid + 8), k = 16-element slices of D.
  uint32_t qa[8][4];
  {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    const T* Q = static_cast<const T*>(p.Q);
    auto ld2 = [&](int hh, int d) -> uint32_t {
      if (hh >= nh) return 0u;
      const int64_t base = p.q.off + (int64_t)b * p.q.bs + (int64_t)(h0 + hh) * p.q.hs + d;
      const uint16_t lo16 = reinterpret_cast<const uint16_t*>(Q)[base];
      const uint16_t hi16 = reinterpret_cast<const uint16_t*>(Q)[base + 1];
      return (uint32_t)lo16 | ((uint32_t)hi16 << 16);
    };
#pragma unroll
    for (int ds = 0; ds < 8; ++ds) {
      qa[ds][0] = ld2(gid, ds * 16 + tig * 2);
      qa[ds][1] = ld2(gid + 8, ds * 16 + tig * 2);
      qa[ds][2] = ld2(gid, ds * 16 + 8 + tig * 2);
      qa[ds][3] = ld2(gid + 8, ds * 16 + 8 + tig * 2);
    }
  }
  const float c = p.scale * kLog2e;
  const bool capped = XF && p.softcap > 0.f;
  const float kinv = capped ? p.scale / p.softcap : 0.f, cap2 = p.softcap * kLog2e;
  const float* mrow = XF && p.M ? p.M + p.m.off + (int64_t)b * p.m.bs : nullptr;

  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
  float m_ref[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const uint32_t sbase = su32(smem);
  const int mi = lane >> 3, ri = lane & 7;

  bool ok = true;
  int consumed = 0;
  for (int ch = 0; ch < n_chunks; ++ch) {
    const int s = ch % kMStages;
    const uint32_t ph = (uint32_t)(ch / kMStages) & 1u;
    ok = __all_sync(0xffffffffu, wait_bar(&full[s], ph, &abort_flag, p.status));
    if (!ok) break;
    consumed = ch + 1;
    const int64_t k0 = start + (int64_t)ch * kMStageKeys + warp * 16;  // first key of this warp
    const uint32_t ks = sbase + s * 2 * kMTile;
    const uint32_t vs = ks + kMTile;
    uint8_t* vgen = smem + s * 2 * kMTile + kMTile;
    const int rbase = warp * 16;  // warp's first row in the stage tile
    // Rows past the range end may hold anything (they can be NaN): zero their V.
    if (k0 + 16 > end) {
      for (int u = lane; u < 16 * 16; u += 32) {
        const int rr = u >> 4, unit = u & 15;
        if (k0 + rr >= end)
          *reinterpret_cast<uint4*>(vgen + (unit >> 3) * (kMStageKeys * 128) + (rbase + rr) * 128 +
                                    (((unit & 7) ^ ((rbase + rr) & 7)) << 4)) = make_uint4(0, 0, 0, 0);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    // S = Q K^T for the warp's 16 keys (two n-tiles of 8 keys).
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ds = 0; ds < 8; ++ds) {
      uint32_t kb[4];
      ldsm4(ks + sw_off(rbase + (mi >> 1) * 8 + ri, ds * 16 + (mi & 1) * 8), kb);
      mma16816<BF16>(sc[0], qa[ds], kb[0], kb[1]);
      mma16816<BF16>(sc[1], qa[ds], kb[2], kb[3]);
    }
    // Scores in log2 units; keys past the end are hidden.
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t key = k0 + nt * 8 + tig * 2 + (e & 1);
        const int hh = gid + (e >> 1) * 8;
        float x = capped ? cap2 * tanh_exp2(sc[nt][e] * kinv) : sc[nt][e] * c;
        if (mrow && key < end && hh < nh) x = fmaf(mrow[(int64_t)(h0 + hh) * p.m.hs + key], kLog2e, x);
        sc[nt][e] = key < end ? x : -INFINITY;
      }
    // Per head row: maximum over the 16 keys (a quad of lanes shares a row).
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = fmaxf(fmaxf(sc[0][2 * r], sc[0][2 * r + 1]), fmaxf(sc[1][2 * r], sc[1][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (mx > m_ref[r] + kSlack) {
        const float corr = ex2(m_ref[r] - mx);
        l[r] *= corr;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          o[nt][2 * r] *= corr;
          o[nt][2 * r + 1] *= corr;
        }
        m_ref[r] = mx;
      }
    }
    uint32_t pa[4];
    {
      const float mu0 = m_ref[0] == -INFINITY ? 0.f : m_ref[0];
      const float mu1 = m_ref[1] == -INFINITY ? 0.f : m_ref[1];
      float pv[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pv[nt][0] = ex2(sc[nt][0] - mu0);
        pv[nt][1] = ex2(sc[nt][1] - mu0);
        pv[nt][2] = ex2(sc[nt][2] - mu1);
        pv[nt][3] = ex2(sc[nt][3] - mu1);
      }
      l[0] += (pv[0][0] + pv[0][1]) + (pv[1][0] + pv[1][1]);
      l[1] += (pv[0][2] + pv[0][3]) + (pv[1][2] + pv[1][3]);
      pa[0] = pack2<BF16>(pv[0][0], pv[0][1]);
      pa[1] = pack2<BF16>(pv[0][2], pv[0][3]);
      pa[2] = pack2<BF16>(pv[1][0], pv[1][1]);
      pa[3] = pack2<BF16>(pv[1][2], pv[1][3]);
    }
    // O += P V over the 128 columns (16 n-tiles of 8).
#pragma unroll
    for (int dn = 0; dn < 8; ++dn) {
      uint32_t vb[4];
      ldsm4t(vs + sw_off(rbase + (mi & 1) * 8 + ri, dn * 16 + (mi >> 1) * 8), vb);
      mma16816<BF16>(o[2 * dn], pa, vb[0], vb[1]);
      mma16816<BF16>(o[2 * dn + 1], pa, vb[2], vb[3]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (tid == 0 && issued < n_chunks) {
      if (!wait_bar(&empty[s], ph, &abort_flag, p.status)) {
        ok = false;
      } else {
        issue(issued);
        ++issued;
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
  }
  if (tid == 0)
    for (int ch = consumed; ch < issued; ++ch) drain_bar(&full[ch % kMStages], (uint32_t)(ch / kMStages) & 1u, p.status);
  ok = __syncthreads_and(ok && !*(volatile int*)&abort_flag);
  if (!ok) return;

  // Row sums over the quad, then merge the four warps in order.
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  float* red_acc = reinterpret_cast<float*>(smem);  // [kWarps][kMHeads][kD]
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int hh = gid + 8 * r;
    if (hh < nh) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        red_acc[(warp * kMHeads + hh) * kD + nt * 8 + tig * 2] = o[nt][2 * r];
        red_acc[(warp * kMHeads + hh) * kD + nt * 8 + tig * 2 + 1] = o[nt][2 * r + 1];
      }
      if (tig == 0) {
        red_m[warp][hh] = m_ref[r];
        red_l[warp][hh] = l[r];
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < nh * kD; i += kThreads) {
    const int hh = i / kD, d = i % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][hh]);
    const int64_t row = (int64_t)b * p.H + h0 + hh;
    float ov = 0.f, lse = -INFINITY;
    if (M != -INFINITY) {
      float L = 0.f, a = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ex2(red_m[w][hh] - M);
        L = fmaf(f, red_l[w][hh], L);
        a = fmaf(f, red_acc[(w * kMHeads + hh) * kD + d], a);
      }
      ov = a / L;
      lse = (M + __log2f(L)) * kLn2;
    }
    sp.part_o[(row * sp.n_splits + split) * kD + d] = ov;
    if (d == 0) sp.part_lse[row * sp.n_splits + split] = lse;
  }
}

template <bool BF16, bool XF>
int launch_mma(const Problem& p, const Split& s, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!tma_map_bhsd(&mk, p.K, p.dtype, kD, p.Sk, p.G, p.B, p.k, kMStageKeys) ||
      !tma_map_bhsd(&mv, p.V, p.dtype, kD, p.Sk, p.G, p.B, p.v, kMStageKeys))
    return -1;
  const int n_hc = (p.qpg + kMHeads - 1) / kMHeads;
  const int64_t blocks = (int64_t)s.n_splits * n_hc * p.G * p.B;
  if (blocks <= 0 || blocks > 0x7fffffff) return -1;
  const int smem = kMStages * 2 * kMTile + 1024;
  auto kern = decode_mma_kernel<BF16, XF>;
  if (ensure_smem((const void*)kern, smem) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const int drop = take_injection() == ATTN_INJECT_DROP_FIRST_COPY ? 1 : 0;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(mk, mv, p, s, n_hc, drop);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace dec
}  // namespace attn

namespace attn {

int decode_fast_try(const Problem& p, const Split& s, cudaStream_t st, int* used) {
  *used = 0;
  if (p.dtype != ATTN_BF16 && p.dtype != ATTN_F16) return ATTN_OK;
  if (p.kv_int8) return ATTN_OK;
  if (p.D != dec::kD || p.Sq != 1 || s.n_splits < 1) return ATTN_OK;
  if (!tma_layout_ok(p.K, p.k, p.Sk, p.G, p.B) || !tma_layout_ok(p.V, p.v, p.Sk, p.G, p.B)) return ATTN_OK;
  const bool xf = p.softcap > 0.f || p.M != nullptr;
  const int rc = p.dtype == ATTN_BF16 ? (xf ? dec::launch_mma<true, true>(p, s, st) : dec::launch_mma<true, false>(p, s, st))
                                      : (xf ? dec::launch_mma<false, true>(p, s, st) : dec::launch_mma<false, false>(p, s, st));
  if (rc < 0) return ATTN_OK;
  *used = 1;
  return rc;
}

}  // namespace attn
