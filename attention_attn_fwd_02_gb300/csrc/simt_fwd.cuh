// simt_fwd.cuh -- the CUDA-core forward kernel and its launcher, included by
// simt.cu (the general layout) and simt_full.cu (the chunked form), so that
// the two sets of template instances compile in parallel.
//
// The forward follows the online normaliser of "Attention" (recursiveai.org
// OneGPU docs), opening paragraph, and the per-block steps of
// "attention_forward -- Causal Multi-Head Attention with Online Softmax"
// (llm.istanbul), section "Online Softmax Algoritmasi": per tile of keys take
// the tile maximum, rescale the running sum and accumulator by
// exp(m_old - m_new), add the tile's exp(s - m_new) terms.  Each tile's
// products go into a fresh accumulator that is added after the one rescale
// ("Attention", section "Accuracy at long key lengths": blockwise summation).
//
// Layout of the work: a CTA of 128 threads owns 128/TPR query rows of one
// (batch, kv head) pair; TPR threads (4 to 32) share a row, each holding up to
// 8 of its head_dim elements (element d lives in lane d % TPR, slot d / TPR;
// when head_dim is exactly 8 * TPR, the kernel takes a form in which a
// lane holds the two 4-element chunks lr and lr + TPR of the row, read from
// shared memory as one 16-byte load each: a quarter of the load instructions
// and no per-slot bounds tests).  Rows are
// ordered (query, head-in-group), so the heads that share a key/value head
// read each staged key tile once.  Dot products are reduced over the TPR lanes
// with an xor butterfly, which gives every lane the same bits; every sum has a
// fixed order, so results are deterministic.
#pragma once

#include <float.h>
#include <limits.h>
#include <math.h>

#include "common.cuh"

namespace attn {

// The chunked form (head_dim 32, 64, 128 or 256, i.e. 8 x threads-per-row), in simt_full.cu.
cudaError_t launch_simt_full(const Problem& p, const Split& s, cudaStream_t st);

namespace {

constexpr int kThreads = 128;
constexpr int kSlots = 8;    // head_dim elements per thread
constexpr int kTile = 32;    // keys per staged tile

// KV8: K and V are int8 (value = integer * scale) instead of T.  Two CTAs an
// SM's worth of registers (up to 255 a thread): the tile's 32 dot products
// then stay in flight together without spilling (measured on GB300: the tiny
// float32 problem 15.0 -> 13.0 us a call against three CTAs' 168 registers,
// larger problems 10-15 % slower than with three, still 1.1-1.4x faster than
// the per-key branching form).
template <typename T, int TPR, bool KV8, bool FULL>
__global__ void __launch_bounds__(kThreads, 2) simt_attn_kernel(Problem p, Split sp, int64_t row_blocks) {
  constexpr int RPC = kThreads / TPR;  // rows per CTA
  extern __shared__ __align__(16) float smem[];
  float* Ks = smem;
  float* Vs = smem + kTile * p.D;
  __shared__ int s_lo, s_hi;

  // Linear block index -> (split, batch*kv_head, row block).
  int64_t blk = blockIdx.x;
  const int rb = (int)(blk % row_blocks);
  blk /= row_blocks;
  const int bg = (int)(blk % ((int64_t)p.B * p.G));
  const int split = (int)(blk / ((int64_t)p.B * p.G));
  const int b = bg / p.G, g = bg % p.G;
  const int D = p.D;
  // Decode with append: every CTA of the range holding the new row writes it
  // (the same values) before the first barrier below, so its own staging
  // reads see it.
  if (p.k_new) {
    const int64_t row = append_target(p, b);
    if (row >= 0 && row / sp.split_len == split) append_row<T>(p, b, g, row);
  }

  const int64_t k0 = (int64_t)split * sp.split_len;
  const int64_t k1 = min((int64_t)p.Sk, k0 + (int64_t)sp.split_len);
  const int rl = threadIdx.x / TPR, lr = threadIdx.x % TPR;
  // The head_dim element in slot s of this lane, and whether it exists.
  auto dim_of = [&](int s) { return FULL ? 4 * (lr + TPR * (s / 4)) + s % 4 : lr + TPR * s; };
  auto has = [&](int s) { return FULL || (TPR * s < D && lr + TPR * s < D); };
  const int64_t r = (int64_t)rb * RPC + rl;
  const bool valid = r < (int64_t)p.Sq * p.qpg;
  const int i = valid ? (int)(r / p.qpg) : 0;
  const int h = g * p.qpg + (valid ? (int)(r % p.qpg) : 0);

  int64_t lo = 0, hi = 0;
  if (valid) {
    row_range(p, b, i, lo, hi);
    lo = max(lo, k0);
    hi = min(hi, k1);
    if (hi < lo) hi = lo;
  }
  if (threadIdx.x == 0) {
    s_lo = INT_MAX;
    s_hi = INT_MIN;
  }
  __syncthreads();
  if (valid && lr == 0 && hi > lo) {
    atomicMin(&s_lo, (int)lo);
    atomicMax(&s_hi, (int)hi);
  }
  __syncthreads();
  const int u_lo = s_lo, u_hi = s_hi;  // union of the CTA's row ranges (empty: u_lo > u_hi)

  const T* Q = static_cast<const T*>(p.Q);
  const T* K = static_cast<const T*>(p.K);
  const T* V = static_cast<const T*>(p.V);
  const int64_t qb = p.q.off + (int64_t)b * p.q.bs + (int64_t)h * p.q.hs + (int64_t)i * p.q.rs;
  const int64_t kb = p.k.off + (int64_t)b * p.k.bs + (int64_t)g * p.k.hs;
  const int64_t vb = p.v.off + (int64_t)b * p.v.bs + (int64_t)g * p.v.hs;
  const int64_t mrow = p.M ? p.m.off + (int64_t)b * p.m.bs + (int64_t)h * p.m.hs + (int64_t)i * p.m.rs : 0;

  float qr[kSlots], acc[kSlots];
#pragma unroll
  for (int s = 0; s < kSlots; ++s) {
    qr[s] = (valid && has(s)) ? to_f32(Q[qb + dim_of(s)]) : 0.f;
    acc[s] = 0.f;
  }
  float m = -INFINITY, l = 0.f;

  for (int t0 = (u_lo / kTile) * kTile; t0 < u_hi; t0 += kTile) {
    __syncthreads();
    // Stage the tile; keys outside the CTA's union are zero (never read from
    // memory).  Each thread issues the loads of kBatch elements before it
    // stores any, so a tile costs about one memory latency, not kBatch.
    constexpr int kBatch = 8;
    for (int e0 = threadIdx.x; e0 < kTile * D; e0 += kThreads * kBatch) {
      float kv[kBatch], vv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads;
        const int j = e / D, d = e - j * D;
        const int kk = t0 + j;
        kv[u] = 0.f;
        vv[u] = 0.f;
        if (e < kTile * D && kk >= u_lo && kk < u_hi) {
          if constexpr (KV8) {
            const int si = p.kv_per_channel ? g * D + d : 0;
            kv[u] = (float)reinterpret_cast<const int8_t*>(p.K)[kb + (int64_t)kk * p.k.rs + d] * p.k_scale[si];
            vv[u] = (float)reinterpret_cast<const int8_t*>(p.V)[vb + (int64_t)kk * p.v.rs + d] * p.v_scale[si];
          } else {
            kv[u] = to_f32(K[kb + (int64_t)kk * p.k.rs + d]);
            vv[u] = to_f32(V[vb + (int64_t)kk * p.v.rs + d]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads;
        if (e < kTile * D) {
          Ks[e] = kv[u];
          Vs[e] = vv[u];
        }
      }
    }
    __syncthreads();

    // The tile's dot products first, with no branch between keys, so that the
    // 32 independent products and reductions overlap; then the score
    // transforms, each behind one test for the whole tile.
    float sc[kTile];
#pragma unroll
    for (int j = 0; j < kTile; ++j) {
      float part = 0.f;
      if constexpr (FULL) {
        const float4* kr = reinterpret_cast<const float4*>(Ks + j * D);
        const float4 a = kr[lr], c = kr[lr + TPR];
        const float kx[kSlots] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int s = 0; s < kSlots; ++s) part = fmaf(qr[s], kx[s], part);
      } else {
#pragma unroll
        for (int s = 0; s < kSlots; ++s)
          if (has(s)) part = fmaf(qr[s], Ks[j * D + dim_of(s)], part);
      }
#pragma unroll
      for (int off = TPR / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      sc[j] = p.scale * part;
    }
    if (p.softcap > 0.f) {
#pragma unroll
      for (int j = 0; j < kTile; ++j) sc[j] = p.softcap * tanhf(sc[j] / p.softcap);
    }
    if (p.M && valid) {
#pragma unroll
      for (int j = 0; j < kTile; ++j) {
        const int kk = t0 + j;
        if (kk >= lo && kk < hi) sc[j] += p.M[mrow + kk];
      }
    }
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < kTile; ++j) {
      const int kk = t0 + j;
      const bool vis = valid && kk >= lo && kk < hi;
      sc[j] = vis ? sc[j] : -INFINITY;
      mt = fmaxf(mt, sc[j]);
    }
    const float m_new = fmaxf(m, mt);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no exp(-inf - -inf)
    const float corr = expf(m - m_use);
    float lt = 0.f;
#pragma unroll
    for (int j = 0; j < kTile; ++j) {
      sc[j] = expf(sc[j] - m_use);
      lt += sc[j];
    }
    l = fmaf(l, corr, lt);
    if constexpr (FULL) {
      float t[kSlots];
#pragma unroll
      for (int s = 0; s < kSlots; ++s) t[s] = 0.f;
#pragma unroll
      for (int j = 0; j < kTile; ++j) {
        const float4* vr = reinterpret_cast<const float4*>(Vs + j * D);
        const float4 a = vr[lr], c = vr[lr + TPR];
        const float vx[kSlots] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int s = 0; s < kSlots; ++s) t[s] = fmaf(sc[j], vx[s], t[s]);
      }
#pragma unroll
      for (int s = 0; s < kSlots; ++s) acc[s] = fmaf(acc[s], corr, t[s]);
    } else {
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        if (has(s)) {
          const int d = dim_of(s);
          float t = 0.f;
#pragma unroll
          for (int j = 0; j < kTile; ++j) t = fmaf(sc[j], Vs[j * D + d], t);
          acc[s] = fmaf(acc[s], corr, t);
        }
      }
    }
    m = m_new;
  }

  if (!valid) return;
  // Direct output (prefill) or one key range's partial result (decode: the
  // combine merges the ranges and adds the sink term once).
  const bool direct = sp.part_o == nullptr;
  if (direct && p.sink_on) {
    const float f = fold_sink<false>(m, l, sink_logit(p, h));
#pragma unroll
    for (int s = 0; s < kSlots; ++s) acc[s] *= f;
  }
  const bool hidden = (l == 0.f);  // no key with non-zero weight; NaN l is a NaN row
  if (direct) {
    T* O = static_cast<T*>(p.O);
    const int64_t ob = p.o.off + (int64_t)b * p.o.bs + (int64_t)h * p.o.hs + (int64_t)i * p.o.rs;
    const float fill = p.masked_zero ? 0.f : NAN;
#pragma unroll
    for (int s = 0; s < kSlots; ++s)
      if (has(s)) O[ob + dim_of(s)] = from_f32<T>(hidden ? fill : acc[s] / l);
    if (p.lse && lr == 0)
      p.lse[(int64_t)b * p.lse_bs + (int64_t)h * p.lse_hs + i] = hidden ? -INFINITY : m + logf(l);
  } else {
    const int64_t row = ((int64_t)b * p.H + h) * p.Sq + i;
    float* po = sp.part_o + (row * sp.n_splits + split) * D;
#pragma unroll
    for (int s = 0; s < kSlots; ++s)
      if (has(s)) po[dim_of(s)] = hidden ? 0.f : acc[s] / l;
    if (lr == 0) sp.part_lse[row * sp.n_splits + split] = hidden ? -INFINITY : m + logf(l);
  }
}

template <typename T, int TPR, bool KV8, bool FULL>
cudaError_t launch_simt_f(const Problem& p, const Split& s, cudaStream_t st) {
  constexpr int RPC = kThreads / TPR;
  const int64_t rows = (int64_t)p.Sq * p.qpg;
  const int64_t row_blocks = (rows + RPC - 1) / RPC;
  const int64_t blocks = row_blocks * p.B * p.G * s.n_splits;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > INT_MAX) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)2 * kTile * p.D * sizeof(float);
  cudaError_t e = ensure_smem((const void*)simt_attn_kernel<T, TPR, KV8, FULL>, (int)smem);
  if (e != cudaSuccess) return e;
  simt_attn_kernel<T, TPR, KV8, FULL><<<(unsigned)blocks, kThreads, smem, st>>>(p, s, row_blocks);
  return cudaGetLastError();
}

// Threads per row from head_dim: 4 up to 32, 8 up to 64, 16 up to 128, else 32.
// FULL requires head_dim == 8 * threads-per-row.
template <typename T, bool KV8, bool FULL>
cudaError_t launch_simt_k(const Problem& p, const Split& s, cudaStream_t st) {
  if (p.D <= 32) return launch_simt_f<T, 4, KV8, FULL>(p, s, st);
  if (p.D <= 64) return launch_simt_f<T, 8, KV8, FULL>(p, s, st);
  if (p.D <= 128) return launch_simt_f<T, 16, KV8, FULL>(p, s, st);
  return launch_simt_f<T, 32, KV8, FULL>(p, s, st);
}

template <bool FULL>
cudaError_t launch_simt_all(const Problem& p, const Split& s, cudaStream_t st) {
  switch (p.dtype) {
    case ATTN_F32:
      return p.kv_int8 ? launch_simt_k<float, true, FULL>(p, s, st) : launch_simt_k<float, false, FULL>(p, s, st);
    case ATTN_F16:
      return p.kv_int8 ? launch_simt_k<__half, true, FULL>(p, s, st) : launch_simt_k<__half, false, FULL>(p, s, st);
    default:
      return p.kv_int8 ? launch_simt_k<__nv_bfloat16, true, FULL>(p, s, st)
                       : launch_simt_k<__nv_bfloat16, false, FULL>(p, s, st);
  }
}

}  // namespace

}  // namespace attn
