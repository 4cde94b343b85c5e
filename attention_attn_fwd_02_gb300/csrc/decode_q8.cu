// decode_q8.cu -- split-range decode pass over an int8 key/value cache
// (head_dim 128, f16/bf16 queries), bandwidth-bound like decode.cu but with
// half the cache bytes per key.
//
// What it computes: the same partial results as decode.cu -- for one query
// row per (batch, head) and one contiguous key range, LSE_r and
// O_r = sum_k exp(s_k - LSE_r) V_k, merged in range order by the combine
// kernel ("Attention" (recursiveai.org OneGPU docs), section "Accuracy at
// long key lengths"; "com.microsoft.GroupQueryAttention", section
// "Implementation variants": the int8 split-K decode) -- with the cache
// values K = k8 * k_scale and V = v8 * v_scale ("com.microsoft.GroupQueryAttention",
// inputs k_scale and v_scale: one scale per cache or one per (kv head,
// channel)).
//
// The scales leave the loop: Q . (k8 * s_k) = (Q * s_k) . k8, so Q is scaled
// by the key scales once (per channel) and rounded to f16; and
// sum p (v8 * s_v) = s_v * sum p v8, so the value scale multiplies the finished
// partial O.  The integers themselves enter the tensor cores as f16, which
// holds every int8 exactly: a byte x becomes the f16 with bits 0x6400 | (x ^
// 0x80), whose value is 1024 + x + 128, minus 1152.
//
// Fragment layouts (mma.sync m16n8k16, f16 in, f32 accumulate; g = lane / 4,
// t = lane % 4).  The cache bytes are read with ldmatrix as if they were
// 16-bit elements, two int8 values each.  Q K^T sums over head-dim channels,
// so any permutation of the 16 channels of a K-step that Q and K share gives
// the same S: thread t takes channels 4t .. 4t+3 of each 16 -- the 32-bit word
// ldmatrix hands it from row g of an 8-key, 16-channel block -- where the
// operand layout asks for channels 2t, 2t+1, 2t+8, 2t+9.  P V sums over keys
// in their natural order (the S accumulators of two 8-key tiles are the A
// operand).  ldmatrix.trans of an 8-key, 16-channel block hands thread (g, t)
// keys 2t and 2t+1 of channels 2g and 2g+1; the even channel's pair is the B
// operand of one n-tile and the odd channel's of another, so n-tile (c, q) of
// channel block c has channel 16 c + 2 n + q in its column n.
//
// CTA: 4 warps; one (batch, kv head, key range) and up to 16 query heads of
// that kv head (the MMA rows), so each cache byte is read once.  The range
// streams through shared memory in 64-key stages, three deep (48 KB, so four
// CTAs share an SM), copied by TMA with 128-byte swizzle (conflict-free
// 32-bit reads); warp w takes keys 16w .. 16w+15 of a stage.  Waits are
// bounded (status word on timeout).
#include <stdlib.h>

#include <type_traits>

#include "decode.h"
#include "tc_ptx.cuh"
#include "tma.h"

namespace attn {
namespace dq8 {

using tc::drain_bar;
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::su32;
using tc::tma_load_4d;
using tc::wait_bar;

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStageKeys = 64;
constexpr int kStages = 3;
constexpr int kTile = kStageKeys * kD;   // bytes of the K (or V) tile of a stage
constexpr int kHeads = 16;               // query heads per CTA (MMA rows)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kSlack = 8.0f;

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// Two biased bytes (already XOR 0x80) at the byte slots picked by sel, placed
// as the low halves of an f16 pair with exponent byte 0x64, minus 1152: the
// original signed integers as an exact f16 pair.
__device__ __forceinline__ uint32_t bytes_to_h2(uint32_t biased, uint32_t sel) {
  const uint32_t w = prmt(biased, 0x64646464u, sel);
  __half2 h = *reinterpret_cast<const __half2*>(&w);
  h = __hsub2(h, __half2half2(__ushort_as_half((unsigned short)0x6480)));  // 1152
  return *reinterpret_cast<uint32_t*>(&h);
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
__global__ void __launch_bounds__(kThreads) decode_q8_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                             const __grid_constant__ CUtensorMap tm_v,
                                                             const Problem p, const Split sp, const int n_hc) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ int abort_flag;
  __shared__ float red_m[kWarps][kHeads], red_l[kWarps][kHeads];

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, gid = lane >> 2, tig = lane & 3;
  int64_t blk = blockIdx.x;
  const int split = (int)(blk % sp.n_splits);
  blk /= sp.n_splits;
  const int hc = (int)(blk % n_hc);
  blk /= n_hc;
  const int g = (int)(blk % p.G);
  const int b = (int)(blk / p.G);
  const int h0 = g * p.qpg + hc * kHeads;
  const int nh = min(kHeads, p.qpg - hc * kHeads);

  // Decode with append: the CTAs of the range holding the new row quantise
  // and write it first; the proxy fence orders those writes before this
  // CTA's TMA reads.
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int n_chunks = (int)((end - start + kStageKeys - 1) / kStageKeys);
  auto issue = [&](int ch) {
    const int s = ch % kStages;
    const int row0 = (int)(start + (int64_t)ch * kStageKeys);
    uint8_t* ks = smem + s * 2 * kTile;
    mbar_expect_tx(&full[s], 2 * kTile);
    tma_load_4d(ks, &tm_k, &full[s], 0, row0, g, b);
    tma_load_4d(ks + kTile, &tm_v, &full[s], 0, row0, g, b);
  };
  int issued = 0;
  if (tid == 0)
    for (; issued < min(kStages, n_chunks); ++issued) issue(issued);

  const bool per_channel = p.kv_per_channel != 0;
  // Q scaled by the key scales, as f16 A operands: rows = heads (gid, gid + 8),
  // K-step ds covers channels 16 ds .. 16 ds + 15, thread tig takes channels
  // 16 ds + 4 tig .. + 3 (see the layout note above).
  uint32_t qa[8][4];
  {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    const T* Q = static_cast<const T*>(p.Q);
    auto q2 = [&](int hh, int d) -> uint32_t {
      if (hh >= nh) return 0u;
      const int64_t base = p.q.off + (int64_t)b * p.q.bs + (int64_t)(h0 + hh) * p.q.hs + d;
      const float s0 = p.k_scale[per_channel ? g * kD + d : 0];
      const float s1 = p.k_scale[per_channel ? g * kD + d + 1 : 0];
      __half2 v = __floats2half2_rn(to_f32(Q[base]) * s0, to_f32(Q[base + 1]) * s1);
      return *reinterpret_cast<uint32_t*>(&v);
    };
#pragma unroll
    for (int ds = 0; ds < 8; ++ds) {
      const int d = ds * 16 + tig * 4;
      qa[ds][0] = q2(gid, d);
      qa[ds][1] = q2(gid + 8, d);
      qa[ds][2] = q2(gid, d + 2);
      qa[ds][3] = q2(gid + 8, d + 2);
    }
  }
  const float c = p.scale * kLog2e;
  const bool capped = p.softcap > 0.f;
  const float kinv = capped ? p.scale / p.softcap : 0.f, cap2 = p.softcap * kLog2e;
  const float* mrow = p.M ? p.M + p.m.off + (int64_t)b * p.m.bs : nullptr;

  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
  float m_ref[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

  bool ok = true;
  int consumed = 0;
  for (int ch = 0; ch < n_chunks; ++ch) {
    const int s = ch % kStages;
    const uint32_t ph = (uint32_t)(ch / kStages) & 1u;
    ok = __all_sync(0xffffffffu, wait_bar(&full[s], ph, &abort_flag, p.status));
    if (!ok) break;
    consumed = ch + 1;
    const int64_t k0 = start + (int64_t)ch * kStageKeys + warp * 16;  // first key of this warp
    // ldmatrix row addresses: lane L supplies row (L % 8) of block L / 8 in a
    // 128-byte-swizzled tile (16-byte unit u of row r at u ^ (r % 8)).
    const uint32_t kt = su32(smem + s * 2 * kTile), vt = kt + kTile;
    const int lrow = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);   // blocks alternate key halves
    const uint32_t krow = kt + lrow * 128, vrow = vt + lrow * 128;
    const int ublk = lane >> 4;                                       // blocks 2, 3: the next 16 channels
    // Rows past the range end need no clearing: their probabilities are 0 and
    // every int8 value is finite (rows past the capacity are zero-filled).
    // S = Q K^T for the warp's 16 keys (two n-tiles of 8 keys).
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int dp = 0; dp < 4; ++dp) {   // channel blocks 2 dp and 2 dp + 1
      uint32_t kw[4];                  // (block 2dp, keys 0-7), (2dp, 8-15), (2dp+1, 0-7), (2dp+1, 8-15)
      ldsm4(krow + (((2 * dp + ublk) ^ (lane & 7)) << 4), kw);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = kw[j] ^ 0x80808080u;
        mma_f16(sc[j & 1], qa[2 * dp + (j >> 1)], bytes_to_h2(w, 0x4140u), bytes_to_h2(w, 0x4342u));
      }
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
        const float corr = ex2_approx(m_ref[r] - mx);
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
        pv[nt][0] = ex2_approx(sc[nt][0] - mu0);
        pv[nt][1] = ex2_approx(sc[nt][1] - mu0);
        pv[nt][2] = ex2_approx(sc[nt][2] - mu1);
        pv[nt][3] = ex2_approx(sc[nt][3] - mu1);
      }
      l[0] += (pv[0][0] + pv[0][1]) + (pv[1][0] + pv[1][1]);
      l[1] += (pv[0][2] + pv[0][3]) + (pv[1][2] + pv[1][3]);
      auto h2 = [](float lo_, float hi_) {
        __half2 v = __floats2half2_rn(lo_, hi_);
        return *reinterpret_cast<uint32_t*>(&v);
      };
      pa[0] = h2(pv[0][0], pv[0][1]);
      pa[1] = h2(pv[0][2], pv[0][3]);
      pa[2] = h2(pv[1][0], pv[1][1]);
      pa[3] = h2(pv[1][2], pv[1][3]);
    }
    // O += P V over channel blocks of 16: ldmatrix.trans gives each thread
    // [V(2t, 2g), V(2t, 2g+1), V(2t+1, 2g), V(2t+1, 2g+1)] of a block's keys
    // 0-7 (and 8-15 in the next register); bytes 0 and 2 are the even
    // channel's key pair, bytes 1 and 3 the odd channel's.
#pragma unroll
    for (int cp = 0; cp < 4; ++cp) {   // channel blocks 2 cp and 2 cp + 1
      uint32_t vw[4];                  // (block 2cp, keys 0-7), (2cp, 8-15), (2cp+1, 0-7), (2cp+1, 8-15)
      ldsm4t(vrow + (((2 * cp + ublk) ^ (lane & 7)) << 4), vw);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo8 = vw[2 * j] ^ 0x80808080u, hi8 = vw[2 * j + 1] ^ 0x80808080u;
        const int c = 2 * cp + j;
        mma_f16(o[2 * c], pa, bytes_to_h2(lo8, 0x4240u), bytes_to_h2(hi8, 0x4240u));
        mma_f16(o[2 * c + 1], pa, bytes_to_h2(lo8, 0x4341u), bytes_to_h2(hi8, 0x4341u));
      }
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
    for (int ch = consumed; ch < issued; ++ch) drain_bar(&full[ch % kStages], (uint32_t)(ch / kStages) & 1u, p.status);
  ok = __syncthreads_and(ok && !*(volatile int*)&abort_flag);
  if (!ok) return;

  // Row sums over the quad, then merge the four warps in order.
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  float* red_acc = reinterpret_cast<float*>(smem);  // [kWarps][kHeads][kD], by channel
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int hh = gid + 8 * r;
    if (hh < nh) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        // accumulator column n of n-tile nt = (block c, parity q) is channel 16 c + 2 n + q
        const int d0 = 16 * (nt >> 1) + 2 * (tig * 2) + (nt & 1);
        red_acc[(warp * kHeads + hh) * kD + d0] = o[nt][2 * r];
        red_acc[(warp * kHeads + hh) * kD + d0 + 2] = o[nt][2 * r + 1];
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
        const float f = ex2_approx(red_m[w][hh] - M);
        L = fmaf(f, red_l[w][hh], L);
        a = fmaf(f, red_acc[(w * kHeads + hh) * kD + d], a);
      }
      ov = a / L * p.v_scale[per_channel ? g * kD + d : 0];
      lse = (M + __log2f(L)) * kLn2;
    }
    sp.part_o[(row * sp.n_splits + split) * kD + d] = ov;
    if (d == 0) sp.part_lse[row * sp.n_splits + split] = lse;
  }
}

template <bool BF16>
int launch(const Problem& p, const Split& s, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!tma_map_bhsd_u8(&mk, p.K, kD, p.Sk, p.G, p.B, p.k, kStageKeys) ||
      !tma_map_bhsd_u8(&mv, p.V, kD, p.Sk, p.G, p.B, p.v, kStageKeys))
    return -1;
  const int n_hc = (p.qpg + kHeads - 1) / kHeads;
  const int64_t blocks = (int64_t)s.n_splits * n_hc * p.G * p.B;
  if (blocks <= 0 || blocks > 0x7fffffff) return -1;
  const int smem = kStages * 2 * kTile + 1024;
  auto kern = decode_q8_kernel<BF16>;
  if (ensure_smem((const void*)kern, smem) != cudaSuccess) return ATTN_ERR_CUDA;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(mk, mv, p, s, n_hc);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace dq8

int decode_q8_try(const Problem& p, const Split& s, cudaStream_t st, int* used) {
  *used = 0;
  if (!p.kv_int8) return ATTN_OK;
  if (p.dtype != ATTN_BF16 && p.dtype != ATTN_F16) return ATTN_OK;
  if (p.D != dq8::kD || p.Sq != 1 || s.n_splits < 1) return ATTN_OK;
  if (!tma_layout_ok_es(p.K, p.k, p.Sk, p.G, p.B, 1) || !tma_layout_ok_es(p.V, p.v, p.Sk, p.G, p.B, 1))
    return ATTN_OK;
  const int rc = p.dtype == ATTN_BF16 ? dq8::launch<true>(p, s, st) : dq8::launch<false>(p, s, st);
  if (rc < 0) return ATTN_OK;
  *used = 1;
  return rc;
}

}  // namespace attn
