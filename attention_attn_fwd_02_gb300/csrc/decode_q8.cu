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
// by the key scales once (per channel), and by scale * log2(e) so that scores
// come out in log2 units, then rounded to f16; and
// sum p (v8 * s_v) = s_v * sum p v8, so the value scale multiplies the finished
// partial O.  The integers enter the tensor cores as exact f16 values with a
// bias: a byte x becomes the f16 with bits 0x6400 | (x ^ 0x80), whose value is
// x + 1152, one logic operation for two bytes.  The bias is taken out once, not
// per element: S = sum Q'(x + 1152) - 1152 sum Q' (the accumulators start at
// -1152 sum Q'), and O = sum p (x + 1152) - 1152 sum p, with sum p the sum of
// the same rounded probabilities, accumulated by an MMA against ones.
//
// The query heads of a kv head are few (often 4 or 8), so the MMA puts the
// keys on its 16 rows and the heads on its 8 columns: S^T = K Q'^T and
// O^T = V^T P^T (mma.sync m16n8k16, f16 in, f32 accumulate; g = lane / 4,
// t = lane % 4).  The cache bytes are read with ldmatrix as if they were
// 16-bit elements, two int8 values each.  S^T sums over head-dim channels, so
// any permutation of the 16 channels of a K-step that K and Q share gives the
// same S: ldmatrix hands thread t the word of channels 4t .. 4t+3 of key rows
// g and g + 8, whose bytes 0 and 2 are the operand's k = 2t, 2t + 1 and bytes 1
// and 3 its k = 2t + 8, 2t + 9; Q' follows the same order.  The S^T
// accumulator (keys g, g+8 x heads 2t, 2t+1), rounded to f16, is moved into
// the B operand of P^T (keys 2t, 2t+1 (+8) x head g) by movmatrix.trans.
// ldmatrix.trans of an 8-key, 16-channel block hands thread (g, t) keys 2t
// and 2t+1 of channels 2g and 2g+1: the even channel's pair is row g of the
// V^T operand, the odd channel's row g + 8.
//
// CTA: 4 warps; one (batch, kv head, key range) and up to 8 (or 16, two MMA
// column tiles) query heads of that kv head, so each cache byte is read once.
// The range streams through shared memory in 64-key stages, two deep (32 KB,
// so five CTAs share an SM at 96 registers a thread: more resident warps beat
// a deeper ring here, measured against three and four stages), copied by TMA
// with 128-byte swizzle (conflict-free ldmatrix);
// warp w takes keys 16w .. 16w+15 of a stage.  Waits are bounded (status word
// on timeout).
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
constexpr int kStages = 2;
constexpr int kTile = kStageKeys * kD;   // bytes of the K (or V) tile of a stage
constexpr float kBias = 1152.f;          // the f16 value of a biased int8 0
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
// Two int8 values of a word (bytes 0 and 2, or 1 and 3) as an f16 pair with
// exponent byte 0x64 and the byte XOR 0x80 as its low mantissa bits: the
// value 1024 + (x + 128) = x + kBias, exact, in one logic operation.
__device__ __forceinline__ uint32_t bias_lo(uint32_t w) { return (w & 0x00FF00FFu) ^ 0x64806480u; }
__device__ __forceinline__ uint32_t bias_hi(uint32_t w) { return ((w >> 8) & 0x00FF00FFu) ^ 0x64806480u; }
// Transpose of an 8x8 matrix of 16-bit values held one row pair per thread.
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
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

// XF: scores under a softcap or an additive mask (an instantiation of its
// own, so that the plain kernel carries neither path).
template <bool BF16, int NT, bool XF>
__global__ void __launch_bounds__(kThreads) decode_q8_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                             const __grid_constant__ CUtensorMap tm_v,
                                                             const Problem p, const Split sp, const int n_hc,
                                                             const int drop_first_copy) {
  constexpr int kHc = 8 * NT;   // query heads per CTA (MMA columns)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ int abort_flag;
  __shared__ float red_m[kWarps][kHc], red_l[kWarps][kHc];

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, gid = lane >> 2, tig = lane & 3;
  int64_t blk = blockIdx.x;
  const int split = (int)(blk % sp.n_splits);
  blk /= sp.n_splits;
  const int hc = (int)(blk % n_hc);
  blk /= n_hc;
  const int g = (int)(blk % p.G);
  const int b = (int)(blk / p.G);
  const int h0 = g * p.qpg + hc * kHc;
  const int nh = min(kHc, p.qpg - hc * kHc);

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
    if (drop_first_copy && ch == 0 && blockIdx.x == 0) return;  // test hook: the stage never lands
    tma_load_4d(ks, &tm_k, &full[s], 0, row0, g, b);
    tma_load_4d(ks + kTile, &tm_v, &full[s], 0, row0, g, b);
  };
  int issued = 0;
  if (tid == 0)
    for (; issued < min(kStages, n_chunks); ++issued) issue(issued);

  const bool per_channel = p.kv_per_channel != 0;
  // Q' = Q * k_scale * scale * log2(e) as f16 B operands (n = head, k =
  // channel): head 8j + gid, channel block c; b0 holds channels 16c + 4tig and
  // + 2, b1 channels + 1 and + 3 (the order the K bytes arrive in).  qs sums
  // the thread's rounded Q' values, for the bias correction below.
  uint32_t qb[NT][8][2];
  float kinit[NT][2];
  {
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    const T* Q = static_cast<const T*>(p.Q);
    const float cs = p.scale * kLog2e;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int hh = 8 * j + gid;
      float qs = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int d = 16 * c + 4 * tig;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (hh < nh) {
          const int64_t base = p.q.off + (int64_t)b * p.q.bs + (int64_t)(h0 + hh) * p.q.hs + d;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            v[e] = __half2float(__float2half_rn(to_f32(Q[base + e]) * p.k_scale[per_channel ? g * kD + d + e : 0] * cs));
        }
        qs += (v[0] + v[1]) + (v[2] + v[3]);
        __half2 h02 = __floats2half2_rn(v[0], v[2]), h13 = __floats2half2_rn(v[1], v[3]);
        qb[j][c][0] = *reinterpret_cast<uint32_t*>(&h02);
        qb[j][c][1] = *reinterpret_cast<uint32_t*>(&h13);
      }
      qs += __shfl_xor_sync(0xffffffffu, qs, 1);
      qs += __shfl_xor_sync(0xffffffffu, qs, 2);
      // The accumulator columns of this thread are heads 8j + 2tig and + 1.
      const float q0 = __shfl_sync(0xffffffffu, qs, 8 * tig);
      const float q1 = __shfl_sync(0xffffffffu, qs, 8 * tig + 4);
      kinit[j][0] = -kBias * q0;
      kinit[j][1] = -kBias * q1;
    }
  }
  const bool capped = XF && p.softcap > 0.f;
  const float kinv = capped ? 1.f / (p.softcap * kLog2e) : 0.f, cap2 = p.softcap * kLog2e;
  const float* mrow = XF && p.M ? p.M + p.m.off + (int64_t)b * p.m.bs : nullptr;
  const bool plain = !XF;

  // O^T accumulators: o[c][j] rows = channels 16c + 2gid (rows gid) and
  // 16c + 2gid + 1 (rows gid + 8), columns = heads 8j + 2tig, + 1.  ls[j]
  // accumulates the rounded probabilities themselves (same columns).
  float o[8][NT][4], ls[NT][4];
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[c][j][e] = 0.f;
  float m_ref[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    m_ref[j][0] = m_ref[j][1] = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) ls[j][e] = 0.f;
  }
  const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};

  // ldmatrix row addresses: lane L supplies row (L % 8) of block L / 8 in a
  // 128-byte-swizzled tile (16-byte unit u of row r at u ^ (r % 8)); blocks
  // alternate the warp's two 8-key halves, blocks 2 and 3 take the next 16
  // channels.
  const int lrow = warp * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
  const int ublk = lane >> 4;

  bool ok = true;
  int consumed = 0;
  for (int ch = 0; ch < n_chunks; ++ch) {
    const int s = ch % kStages;
    const uint32_t ph = (uint32_t)(ch / kStages) & 1u;
    ok = __all_sync(0xffffffffu, wait_bar(&full[s], ph, &abort_flag, p.status));
    if (!ok) break;
    consumed = ch + 1;
    const int64_t k0 = start + (int64_t)ch * kStageKeys + warp * 16;  // first key of this warp
    const uint32_t krow = su32(smem + s * 2 * kTile) + lrow * 128, vrow = krow + kTile;
    // Rows past the range end need no clearing: their probabilities are 0 and
    // every int8 value is finite (rows past the capacity are zero-filled).
    // S^T = K Q'^T for the warp's 16 keys (MMA rows: keys gid, gid + 8),
    // started at the bias correction so that it holds the scores in log2 units.
    float st[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      st[j][0] = st[j][2] = kinit[j][0];
      st[j][1] = st[j][3] = kinit[j][1];
    }
#pragma unroll
    for (int dp = 0; dp < 4; ++dp) {   // channel blocks 2 dp and 2 dp + 1
      uint32_t kw[4];                  // (block 2dp, keys 0-7), (2dp, 8-15), (2dp+1, 0-7), (2dp+1, 8-15)
      ldsm4(krow + (((2 * dp + ublk) ^ (lane & 7)) << 4), kw);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint32_t a[4] = {bias_lo(kw[2 * jj]), bias_lo(kw[2 * jj + 1]), bias_hi(kw[2 * jj]),
                               bias_hi(kw[2 * jj + 1])};
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_f16(st[j], a, qb[j][2 * dp + jj][0], qb[j][2 * dp + jj][1]);
      }
    }
    // Transforms and hiding of keys past the end (warp-uniform skip for whole
    // in-range tiles without softcap or mask).
    if (!plain || k0 + 16 > end) {
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t key = k0 + gid + 8 * (e >> 1);
          const int hh = 8 * j + 2 * tig + (e & 1);
          float x = capped ? cap2 * tanh_exp2(st[j][e] * kinv) : st[j][e];
          if (mrow && key < end && hh < nh) x = fmaf(mrow[(int64_t)(h0 + hh) * p.m.hs + key], kLog2e, x);
          st[j][e] = key < end ? x : -INFINITY;
        }
    }
    uint32_t pb[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      // Per head column: maximum over the 16 keys (the eight lanes of a tig).
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float mx = fmaxf(st[j][q], st[j][q + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (mx > m_ref[j][q] + kSlack) {
          const float corr = ex2_approx(m_ref[j][q] - mx);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            o[c][j][q] *= corr;
            o[c][j][q + 2] *= corr;
          }
          ls[j][q] *= corr;
          ls[j][q + 2] *= corr;
          m_ref[j][q] = mx;
        }
      }
      const float mu0 = m_ref[j][0] == -INFINITY ? 0.f : m_ref[j][0];
      const float mu1 = m_ref[j][1] == -INFINITY ? 0.f : m_ref[j][1];
      __half2 p01 = __floats2half2_rn(ex2_approx(st[j][0] - mu0), ex2_approx(st[j][1] - mu1));
      __half2 p23 = __floats2half2_rn(ex2_approx(st[j][2] - mu0), ex2_approx(st[j][3] - mu1));
      // P as an 8-key x 8-head matrix per key half; transposed, it is the B
      // operand (k = keys 2tig, 2tig + 1 (+ 8), n = head gid).
      pb[j][0] = movtrans(*reinterpret_cast<uint32_t*>(&p01));
      pb[j][1] = movtrans(*reinterpret_cast<uint32_t*>(&p23));
    }
    // O^T += V^T P^T over channel blocks of 16: ldmatrix.trans gives each thread
    // [V(2t, 2g), V(2t, 2g+1), V(2t+1, 2g), V(2t+1, 2g+1)] of a block's keys
    // 0-7 (and 8-15 in the next register); bytes 0 and 2 are channel 2g's key
    // pair (MMA row gid), bytes 1 and 3 channel 2g+1's (row gid + 8).
#pragma unroll
    for (int cp = 0; cp < 4; ++cp) {   // channel blocks 2 cp and 2 cp + 1
      uint32_t vw[4];                  // (block 2cp, keys 0-7), (2cp, 8-15), (2cp+1, 0-7), (2cp+1, 8-15)
      ldsm4t(vrow + (((2 * cp + ublk) ^ (lane & 7)) << 4), vw);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const uint32_t a[4] = {bias_lo(vw[2 * jj]), bias_hi(vw[2 * jj]), bias_lo(vw[2 * jj + 1]),
                               bias_hi(vw[2 * jj + 1])};
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_f16(o[2 * cp + jj][j], a, pb[j][0], pb[j][1]);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) mma_f16(ls[j], ones, pb[j][0], pb[j][1]);
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

  // Per warp: the biased values sum to O + 1152 * l, so subtract the bias
  // times the probability sum; then merge the four warps in order.
  float* red_acc = reinterpret_cast<float*>(smem);  // [kWarps][kHc][kD], by channel
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int hh = 8 * j + 2 * tig + q;
      if (hh < nh) {
        const float corr = kBias * ls[j][q];
        float* dst = red_acc + (warp * kHc + hh) * kD + 2 * gid;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          dst[16 * c] = o[c][j][q] - corr;
          dst[16 * c + 1] = o[c][j][q + 2] - corr;
        }
        if (gid == 0) {
          red_m[warp][hh] = m_ref[j][q];
          red_l[warp][hh] = ls[j][q];
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
        a = fmaf(f, red_acc[(w * kHc + hh) * kD + d], a);
      }
      ov = a / L * p.v_scale[per_channel ? g * kD + d : 0];
      lse = (M + __log2f(L)) * kLn2;
    }
    sp.part_o[(row * sp.n_splits + split) * kD + d] = ov;
    if (d == 0) sp.part_lse[row * sp.n_splits + split] = lse;
  }
}

template <bool BF16, int NT, bool XF>
int launch(const Problem& p, const Split& s, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!tma_map_bhsd_u8(&mk, p.K, kD, p.Sk, p.G, p.B, p.k, kStageKeys) ||
      !tma_map_bhsd_u8(&mv, p.V, kD, p.Sk, p.G, p.B, p.v, kStageKeys))
    return -1;
  const int n_hc = (p.qpg + 8 * NT - 1) / (8 * NT);
  const int64_t blocks = (int64_t)s.n_splits * n_hc * p.G * p.B;
  if (blocks <= 0 || blocks > 0x7fffffff) return -1;
  const int smem = kStages * 2 * kTile + 1024;
  auto kern = decode_q8_kernel<BF16, NT, XF>;
  if (ensure_smem((const void*)kern, smem) != cudaSuccess) return ATTN_ERR_CUDA;
  const int drop = take_injection() == ATTN_INJECT_DROP_FIRST_COPY ? 1 : 0;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(mk, mv, p, s, n_hc, drop);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <bool BF16, bool XF>
int launch_x(const Problem& p, const Split& s, cudaStream_t st) {
  return p.qpg <= 8 ? launch<BF16, 1, XF>(p, s, st) : launch<BF16, 2, XF>(p, s, st);
}

template <bool BF16>
int launch(const Problem& p, const Split& s, cudaStream_t st) {
  const bool xf = p.softcap > 0.f || p.M != nullptr;
  return xf ? launch_x<BF16, true>(p, s, st) : launch_x<BF16, false>(p, s, st);
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
