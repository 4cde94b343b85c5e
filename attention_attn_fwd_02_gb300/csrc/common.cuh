// common.cuh -- types shared by the kernels and the host planner of libattn.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "attn.h"

namespace attn {

struct Layout {
  int64_t off, bs, hs, rs;  // elements: offset, batch, head, row strides
};

// A validated problem with defaults resolved, passed by value to kernels.
struct Problem {
  int B, H, G, Sq, Sk, D, qpg;   // qpg = heads / kv_heads
  int dtype;                     // ATTN_F32 / ATTN_F16 / ATTN_BF16
  float scale;
  int causal;
  int64_t coff;                  // causal offset (resolved)
  int masked_zero;
  int window;                    // left window (keys behind the diagonal), -1 = none
  int align_klens;               // 1: causal offset of entry b is L_b - Sq
  int klens_plus;                // added to k_lens[b] (1 for last-index lengths)
  float softcap;                 // 0: off; > 0: scores are softcap * tanh(scale q.k / softcap)
  int sink_on;                   // 1: a sink logit joins every row's denominator
  const float* sink;             // per-head sink logits (nullptr: 0 for every head)
  int kv_int8;                   // 1: K and V are int8, value = integer * scale
  int kv_per_channel;            // 1: scales per (kv head, channel); 0: one scale each
  const float* k_scale;
  const float* v_scale;
  const void* k_new;             // decode with append: new rows [B][G][D] in dtype (nullptr: none)
  const void* v_new;
  Layout q, k, v, o, m;
  int64_t seg_bs, lse_bs, lse_hs;
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  const float* M;
  const int32_t* seg;
  const int32_t* klens;
  float* lse;
  int* status;                   // device status word (ATTN_ERR_DEVICE_TIMEOUT on a given-up wait)
};

// Key range [k_begin, k_end) cut out of [0, Sk) for split passes, and where the
// per-range partial results go.
struct Split {
  int n_splits;      // 1 = no split: write O / LSE directly
  int split_len;     // keys per range (multiple of 32)
  float* part_o;     // [rows][n_splits][D], rows = B*H*Sq in (b, h, i) order
  float* part_lse;   // [rows][n_splits]
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__host__ __device__ __forceinline__ int64_t clamp64(int64_t x, int64_t lo, int64_t hi) {
  return x < lo ? lo : (x > hi ? hi : x);
}

// Visible key range [lo, hi) of query row i of batch entry b: the structural
// rules (key length, causal bound with its optional left window, segment
// start) intersect to one interval.  L_b is the entry's valid key count; the
// causal diagonal of row i is key i + off with off the problem's offset, or
// L_b - Sq when the bound is right-aligned to the entry's length.
__device__ __forceinline__ void row_range(const Problem& p, int b, int i, int64_t& lo, int64_t& hi) {
  int64_t kl = p.Sk;
  if (p.klens) kl = clamp64((int64_t)p.klens[b] + p.klens_plus, 0, p.Sk);
  hi = kl;
  lo = 0;
  if (p.causal) {
    const int64_t diag = (int64_t)i + (p.align_klens ? kl - p.Sq : p.coff);
    hi = diag + 1 < hi ? diag + 1 : hi;
    if (hi < 0) hi = 0;
    if (p.window >= 0 && diag - p.window > lo) lo = diag - p.window;
  }
  if (p.seg) {
    const int64_t s = clamp64((int64_t)p.seg[(int64_t)b * p.seg_bs + i], 0, p.Sk);
    if (s > lo) lo = s;
  }
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh(y) from its definition with a single base-2 exponential:
// tanh(|y|) = (1 - e) / (1 + e) with e = exp(-2|y|) = 2^(-2 log2(e) |y|), and
// the sign of y restored.  The subtraction 1 - e costs at most one float32
// ulp of 1 in absolute error near y = 0; large |y| gives e = 0 and +-1; NaN
// stays NaN.  Used by the half-precision kernels' soft-capping.
__device__ __forceinline__ float tanh_exp2(float y) {
  const float e = ex2_approx(-2.8853900817779268f * fabsf(y));
  return copysignf(__fdividef(1.f - e, 1.f + e), y);
}

// The sink logit of head h in natural-log units.
__device__ __forceinline__ float sink_logit(const Problem& p, int h) { return p.sink ? p.sink[h] : 0.f; }

// Folds a sink logit s (same units and base as m) into a row's running
// maximum m and sum l, where the row's sum is l relative to m and base is 2
// (exp2) or e (exp): afterwards l and m describe the row including the sink,
// and the returned factor rescales the row's accumulated numerator.  A NaN or
// +inf sink makes the row NaN; a -inf sink changes nothing.
template <bool BASE2>
__device__ __forceinline__ float fold_sink(float& m, float& l, float s) {
  if (s != s || s == INFINITY) {
    l = NAN;
    return 1.f;
  }
  if (s == -INFINITY) return 1.f;
  const float mx = fmaxf(m, s);   // m = -inf (no visible key): the sink alone
  const float f = BASE2 ? ex2_approx(m - mx) : expf(m - mx);
  l = fmaf(l, f, BASE2 ? ex2_approx(s - mx) : expf(s - mx));
  m = mx;
  return f;
}

// The cache update before a decode step with append: the new key and value
// rows of (batch b, kv head g) go to cache row `row` (the entry's last valid
// row).  Float caches take a copy; an int8 cache takes x / scale rounded to
// the nearest integer (ties to even, IEEE float32 division) and saturated to
// [-128, 127].  The block's threads share the D elements; the caller
// synchronises before any of its threads or copies read the row.
template <typename T>
__device__ __forceinline__ void append_row(const Problem& p, int b, int g, int64_t row) {
  const int64_t src = ((int64_t)b * p.G + g) * p.D;
  const int64_t kd = p.k.off + (int64_t)b * p.k.bs + (int64_t)g * p.k.hs + row * p.k.rs;
  const int64_t vd = p.v.off + (int64_t)b * p.v.bs + (int64_t)g * p.v.hs + row * p.v.rs;
  const T* kn = static_cast<const T*>(p.k_new);
  const T* vn = static_cast<const T*>(p.v_new);
  for (int d = threadIdx.x; d < p.D; d += blockDim.x) {
    if (p.kv_int8) {
      const int si = p.kv_per_channel ? g * p.D + d : 0;
      const float ck = fminf(fmaxf(rintf(to_f32(kn[src + d]) / p.k_scale[si]), -128.f), 127.f);
      const float cv = fminf(fmaxf(rintf(to_f32(vn[src + d]) / p.v_scale[si]), -128.f), 127.f);
      const_cast<int8_t*>(static_cast<const int8_t*>(p.K))[kd + d] = (int8_t)ck;
      const_cast<int8_t*>(static_cast<const int8_t*>(p.V))[vd + d] = (int8_t)cv;
    } else {
      const_cast<T*>(static_cast<const T*>(p.K))[kd + d] = kn[src + d];
      const_cast<T*>(static_cast<const T*>(p.V))[vd + d] = vn[src + d];
    }
  }
}

// Row of the cache update for batch entry b (its clamped length minus one),
// or -1 when the entry has no valid row.
__device__ __forceinline__ int64_t append_target(const Problem& p, int b) {
  const int64_t L = p.klens ? clamp64((int64_t)p.klens[b] + p.klens_plus, 0, p.Sk) : p.Sk;
  return L - 1;
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device once; the setting lasts for the process, so later launches only look
// it up (the attribute call costs microseconds, which small problems feel).
inline cudaError_t ensure_smem(const void* kern, int bytes) {
  struct Entry {
    const void* k;
    int dev, bytes;
  };
  static std::mutex mu;
  static Entry tab[256];
  static int n = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (tab[i].k == kern && tab[i].dev == dev && tab[i].bytes >= bytes) return cudaSuccess;
  }
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> lock(mu);
    if (n < 256) tab[n++] = {kern, dev, bytes};
  }
  return e;
}

// Device addresses of a __device__ symbol, per (device, context).  A host
// program's name for a __device__ variable is a host-side stand-in, so the
// address kernels need is looked up with cudaGetSymbolAddress once for each
// device and context: after a cudaDeviceReset the device gets a new context
// whose copy of the symbol may sit elsewhere, and the id changes with it.
struct SymbolCache {
  static constexpr int kSlots = 64;
  std::mutex mu;
  int dev[kSlots];
  unsigned long long ctx[kSlots];
  void* ptr[kSlots];
  int n = 0;
};
// Address of `symbol` (the host stand-in's address) on the current device;
// returns an ATTN_* status.
int symbol_address(SymbolCache& cache, const void* symbol, void** out);

// Takes (and clears) the one-shot test fault armed by attn_test_inject;
// ATTN_INJECT_NONE when none is armed.  Host side, called right before a
// launch of a kernel that supports the fault.
int take_injection();

// Host-side launchers (defined in the kernel translation units).
cudaError_t launch_simt(const Problem& p, const Split& s, cudaStream_t st);
cudaError_t launch_combine(const Problem& p, const Split& s, int32_t out_dtype, cudaStream_t st);
cudaError_t launch_ex2_probe(int blocks, int iters, float* sink, cudaStream_t st);
cudaError_t launch_combine_flat(int n_splits, int rows, int D, const float* part_o, const float* part_lse,
                                int32_t out_dtype, void* o, int64_t o_row_stride, float* lse,
                                int masked_zero, cudaStream_t st);

}  // namespace attn
