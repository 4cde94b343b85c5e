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
// One CTA (4 warps) owns one (batch, kv head, key range) and every query head
// of that kv head (up to 8 per CTA), so each cache byte is read once.  The
// range streams through shared memory in 32-key stages with 1-D bulk copies
// (cp.async.bulk, completion on an mbarrier) four stages deep.  In a stage,
// warp w takes keys 8w..8w+7 as four pairs: lanes 0-15 read one 256-byte key
// row and lanes 16-31 the next, 16 bytes (8 elements) each, so every shared
// load is conflict-free.  The per-head dot products are reduced over the 16
// lanes of a row with a transposing butterfly (each step halves the values a
// lane carries) and gathered back, so every lane ends with the scores of its
// key for all heads.  Each warp keeps its own online-softmax state (reference
// maximum with a slack of 8 in log2 units, as in "Attention", section "Apple
// simdgroup kernel"); the four warps merge in warp order at the end.  All
// sums have a fixed order.  Waits are bounded (status word on timeout).
#include <limits.h>

#include <type_traits>

#include "decode.h"

namespace attn {
namespace dec {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kStageKeys = 32;
constexpr int kStages = 4;
constexpr int kRowBytes = kD * 2;
constexpr int kStageBytes = kStageKeys * kRowBytes;  // one of K or V
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
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 8 elements (16 bytes) of a 16-bit row to float.
template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

// Sum v[0..HG) over the 16 lanes that share a key row and return, in every
// lane, the sums of all HG heads in head order.  Reduce-scatter: at lane bits
// 3, 2, ... a lane that still carries n > 1 values keeps the half selected by
// its bit (upper half for bit = 1) and sends the other half, so after log2(HG)
// splits it carries one head, whose index has the split bits as digits (bit 3
// most significant); the remaining bits are plain butterfly adds.  Gather:
// the splits are undone from the lowest split bit up, each step concatenating
// [lower lane's values, upper lane's values], which restores head order.
template <int HG>
__device__ __forceinline__ void row_reduce_gather(float (&v)[HG], int lane) {
  constexpr int kSplits = HG == 1 ? 0 : (HG == 2 ? 1 : (HG == 4 ? 2 : 3));
  float cur[HG];
#pragma unroll
  for (int i = 0; i < HG; ++i) cur[i] = v[i];
#pragma unroll
  for (int step = 0; step < 4; ++step) {
    const int bit = 3 - step;
    const int m = 1 << bit;
    if (step < kSplits) {
      const int h = HG >> (step + 1);
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < HG / 2; ++i) {
        if (i < h) {
          const float send = upper ? cur[i] : cur[i + h];
          const float keep = upper ? cur[i + h] : cur[i];
          cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
    } else {
      cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], m);
    }
  }
  float all[HG];
  all[0] = cur[0];
#pragma unroll
  for (int s = 0; s < kSplits; ++s) {
    const int m = 1 << (4 - kSplits + s);
    const int have = 1 << s;
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < HG / 2; ++i) {
      if (i < have) {
        const float other = __shfl_xor_sync(0xffffffffu, all[i], m);
        const float lo = upper ? other : all[i];
        const float hi = upper ? all[i] : other;
        all[i] = lo;
        all[i + have] = hi;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < HG; ++i) v[i] = all[i];
}

template <int HG, bool BF16>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const Problem p, const Split sp, const int n_hc) {
  extern __shared__ __align__(128) uint8_t smem[];  // kStages x (K stage, V stage); reused for the merge
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ int abort_flag;
  __shared__ float red_m[kWarps][HG], red_l[kWarps][HG];

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32, half = lane >> 4, sub = lane & 15;
  int64_t blk = blockIdx.x;
  const int split = (int)(blk % sp.n_splits);
  blk /= sp.n_splits;
  const int hc = (int)(blk % n_hc);
  blk /= n_hc;
  const int g = (int)(blk % p.G);
  const int b = (int)(blk / p.G);
  const int h0 = g * p.qpg + hc * HG;
  const int nh = min(HG, p.qpg - hc * HG);

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

  // Query rows of the heads of this CTA, pre-scaled to log2 units.
  const float c = p.scale * kLog2e;
  float q[HG][8];
  {
    const auto* Q = static_cast<const typename std::conditional<BF16, __nv_bfloat16, __half>::type*>(p.Q);
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      const int64_t base = p.q.off + (int64_t)b * p.q.bs + (int64_t)(h0 + hh) * p.q.hs + sub * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) q[hh][e] = hh < nh ? to_f32(Q[base + e]) * c : 0.f;
    }
  }
  const float* mrow = nullptr;
  if (p.M) mrow = p.M + p.m.off + (int64_t)b * p.m.bs;

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
  const char* kbase = static_cast<const char*>(p.K) + (p.k.off + (int64_t)b * p.k.bs + (int64_t)g * p.k.hs) * 2;
  const char* vbase = static_cast<const char*>(p.V) + (p.v.off + (int64_t)b * p.v.bs + (int64_t)g * p.v.hs) * 2;
  auto issue = [&](int ch) {
    const int s = ch % kStages;
    const int64_t c0 = start + (int64_t)ch * kStageKeys;
    const uint32_t nr = (uint32_t)min((int64_t)kStageKeys, end - c0);
    uint8_t* ks = smem + s * 2 * kStageBytes;
    mbar_expect_tx(&full[s], 2 * nr * kRowBytes);
    bulk_g2s(ks, kbase + c0 * kRowBytes, nr * kRowBytes, &full[s]);
    bulk_g2s(ks + kStageBytes, vbase + c0 * kRowBytes, nr * kRowBytes, &full[s]);
  };
  int issued = 0;
  if (tid == 0) {
    for (; issued < min(kStages, n_chunks); ++issued) issue(issued);
  }

  float m_ref[HG], l[HG], acc[HG][8];
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    m_ref[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[hh][e] = 0.f;
  }
  bool ok = true;
  int consumed = 0;
  for (int ch = 0; ch < n_chunks; ++ch) {
    const int s = ch % kStages;
    const uint32_t ph = (uint32_t)(ch / kStages) & 1u;
    ok = __all_sync(0xffffffffu, wait_bar(&full[s], ph, &abort_flag, p.status));
    if (!ok) break;
    consumed = ch + 1;
    const int64_t c0 = start + (int64_t)ch * kStageKeys;
    const int nr = (int)min((int64_t)kStageKeys, end - c0);
    const uint8_t* ks = smem + s * 2 * kStageBytes;
    const uint8_t* vs = ks + kStageBytes;

    float sc[4][HG];
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      const int row = warp * 8 + pr * 2 + half;
      float kf[8];
      unpack8<BF16>(*reinterpret_cast<const uint4*>(ks + row * kRowBytes + sub * 16), kf);
      float part[HG];
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) a = fmaf(q[hh][e], kf[e], a);
        part[hh] = a;
      }
      row_reduce_gather<HG>(part, lane);
      const bool valid = row < nr;
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        float x = part[hh];
        if (mrow && valid && hh < nh) x = fmaf(mrow[(int64_t)(h0 + hh) * p.m.hs + c0 + row], kLog2e, x);
        sc[pr][hh] = valid ? x : -INFINITY;
      }
    }
    // Chunk maximum per head (the same in every lane after the exchange across halves).
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      float mx = fmaxf(fmaxf(sc[0][hh], sc[1][hh]), fmaxf(sc[2][hh], sc[3][hh]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      if (mx > m_ref[hh] + kSlack) {  // raise the reference and rescale (warp-uniform)
        const float corr = ex2(m_ref[hh] - mx);
        l[hh] *= corr;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[hh][e] *= corr;
        m_ref[hh] = mx;
      }
    }
#pragma unroll
    for (int pr = 0; pr < 4; ++pr) {
      const int row = warp * 8 + pr * 2 + half;
      const bool valid = row < nr;
      float vf[8];
      unpack8<BF16>(*reinterpret_cast<const uint4*>(vs + row * kRowBytes + sub * 16), vf);
#pragma unroll
      for (int e = 0; e < 8; ++e) vf[e] = valid ? vf[e] : 0.f;
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        const float pv = ex2(sc[pr][hh] - (m_ref[hh] == -INFINITY ? 0.f : m_ref[hh]));
        l[hh] += pv;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[hh][e] = fmaf(pv, vf[e], acc[hh][e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (tid == 0 && issued < n_chunks) {
      // the stage is refilled once all warps are done with it
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
  // Copies still in flight land before the CTA exits.
  if (tid == 0)
    for (int ch = consumed; ch < issued; ++ch) drain_bar(&full[ch % kStages], (uint32_t)(ch / kStages) & 1u, p.status);
  ok = __syncthreads_and(ok && !*(volatile int*)&abort_flag);
  if (!ok) return;

  // Merge the two key halves of each warp, then the four warps in order.
#pragma unroll
  for (int hh = 0; hh < HG; ++hh) {
    l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 16);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[hh][e] += __shfl_xor_sync(0xffffffffu, acc[hh][e], 16);
  }
  float* red_acc = reinterpret_cast<float*>(smem);  // [kWarps][HG][kD]
  if (half == 0) {
#pragma unroll
    for (int hh = 0; hh < HG; ++hh)
#pragma unroll
      for (int e = 0; e < 8; ++e) red_acc[(warp * HG + hh) * kD + sub * 8 + e] = acc[hh][e];
  }
  if (lane == 0) {
#pragma unroll
    for (int hh = 0; hh < HG; ++hh) {
      red_m[warp][hh] = m_ref[hh];
      red_l[warp][hh] = l[hh];
    }
  }
  __syncthreads();
  for (int i = tid; i < nh * kD; i += kThreads) {
    const int hh = i / kD, d = i % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][hh]);
    const int64_t row = (int64_t)b * p.H + h0 + hh;
    float o = 0.f, lse = -INFINITY;
    if (M != -INFINITY) {
      float L = 0.f, a = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = ex2(red_m[w][hh] - M);
        L = fmaf(f, red_l[w][hh], L);
        a = fmaf(f, red_acc[(w * HG + hh) * kD + d], a);
      }
      o = a / L;
      lse = (M + __log2f(L)) * kLn2;
    }
    sp.part_o[(row * sp.n_splits + split) * kD + d] = o;
    if (d == 0) sp.part_lse[row * sp.n_splits + split] = lse;
  }
}

template <int HG, bool BF16>
int launch(const Problem& p, const Split& s, cudaStream_t st) {
  const int n_hc = (p.qpg + HG - 1) / HG;
  const int64_t blocks = (int64_t)s.n_splits * n_hc * p.G * p.B;
  if (blocks <= 0 || blocks > 0x7fffffff) return -1;
  const int smem = kStages * 2 * kStageBytes;
  auto kern = decode_split_kernel<HG, BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_ERR_CUDA;
  kern<<<(unsigned)blocks, kThreads, smem, st>>>(p, s, n_hc);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <bool BF16>
int launch_hg(const Problem& p, const Split& s, cudaStream_t st) {
  if (p.qpg <= 1) return launch<1, BF16>(p, s, st);
  if (p.qpg <= 2) return launch<2, BF16>(p, s, st);
  if (p.qpg <= 4) return launch<4, BF16>(p, s, st);
  return launch<8, BF16>(p, s, st);
}

}  // namespace dec
}  // namespace attn

namespace attn {

int decode_fast_try(const Problem& p, const Split& s, cudaStream_t st, int* used) {
  *used = 0;
  if (p.dtype != ATTN_BF16 && p.dtype != ATTN_F16) return ATTN_OK;
  if (p.D != dec::kD || p.Sq != 1 || s.n_splits < 1) return ATTN_OK;
  // contiguous 256-byte cache rows starting on 16-byte boundaries
  if (p.k.rs != dec::kD || p.v.rs != dec::kD) return ATTN_OK;
  auto al = [](const void* base, const Layout& l) {
    return ((uintptr_t)base % 16 == 0) && (l.off % 8 == 0) && (l.bs % 8 == 0) && (l.hs % 8 == 0);
  };
  if (!al(p.K, p.k) || !al(p.V, p.v)) return ATTN_OK;
  const int rc = p.dtype == ATTN_BF16 ? dec::launch_hg<true>(p, s, st) : dec::launch_hg<false>(p, s, st);
  if (rc < 0) return ATTN_OK;
  *used = 1;
  return rc;
}

}  // namespace attn
