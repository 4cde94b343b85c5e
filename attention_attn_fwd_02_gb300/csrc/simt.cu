// simt.cu -- CUDA-core kernels: the exact float32 forward (also the generic
// fallback for half/bfloat16 layouts the tensor-core path cannot take), the
// generic split-range decode pass, and the partial-result combine.  The
// forward kernel itself is in simt_fwd.cuh; this file launches its general
// layout and hands head_dim 8 x threads-per-row to the chunked form
// (simt_full.cu).
#include "simt_fwd.cuh"

namespace attn {

namespace {

// One warp per row: merge the row's range partials in range order.
// With sink_on the head's sink logit enters as one more range with an
// empty numerator (the sink term of the denominator, added once per row).
// The lanes read the ranges' LSEs in parallel (lane r: ranges r, r + 32, ...)
// and broadcast the weights; the partial rows of four ranges are loaded
// before they are summed, so the loads overlap instead of queueing behind one
// another.  Ranges with weight 0 (empty, or underflowed) are left out of the
// sum by a select, so an unwritten partial never reaches it.
template <typename T>
__global__ void __launch_bounds__(128) combine_kernel(int n_splits, int64_t rows, int D, const float* part_o,
                                                      const float* part_lse, T* O, Layout ol, int H, int Sq,
                                                      float* lse, int64_t lse_bs, int64_t lse_hs,
                                                      int64_t lse_rs, int masked_zero, int sink_on,
                                                      const float* sink) {
  constexpr unsigned kAll = 0xffffffffu;
  const int64_t row = (int64_t)blockIdx.x * 4 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  const float* pl = part_lse + row * n_splits;
  const int i = (int)(row % Sq);
  const int h = (int)((row / Sq) % H);
  const float sg = sink_on ? (sink ? sink[h] : 0.f) : -INFINITY;
  bool bad = isnan(sg) || sg == INFINITY;
  float M = bad ? -INFINITY : sg;
  for (int r = lane; r < n_splits; r += 32) {
    const float x = pl[r];
    if (isnan(x) || x == INFINITY) bad = true;
    else M = fmaxf(M, x);
  }
  bad = __any_sync(kAll, bad);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kAll, M, o));
  const int64_t b = row / ((int64_t)Sq * H);
  const int64_t ob = ol.off + b * ol.bs + (int64_t)h * ol.hs + (int64_t)i * ol.rs;
  const bool normal = !bad && M != -INFINITY;
  float acc[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) acc[s] = 0.f;
  float ws = 0.f;
  if (normal) {
    for (int base = 0; base < n_splits; base += 32) {
      const int r = base + lane;
      const float x = r < n_splits ? pl[r] : -INFINITY;
      const float wr = x == -INFINITY ? 0.f : expf(x - M);
      ws += wr;
      const int nr = min(32, n_splits - base);
      for (int k = 0; k < nr; k += 4) {
        float w[4], v[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          w[u] = __shfl_sync(kAll, wr, k + u);   // lanes past the last range hold 0
          const float* src = part_o + (row * n_splits + min(base + k + u, n_splits - 1)) * D;
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const int d = lane + 32 * s;
            v[u][s] = d < D ? src[d] : 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int s = 0; s < 8; ++s) acc[s] = w[u] != 0.f ? fmaf(w[u], v[u][s], acc[s]) : acc[s];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(kAll, ws, o);
    if (sg > -INFINITY) ws += expf(sg - M);
  }
  const float val_fill = (!bad && M == -INFINITY) ? (masked_zero ? 0.f : NAN) : NAN;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int d = lane + 32 * s;
    if (d < D) O[ob + d] = from_f32<T>(normal ? acc[s] / ws : val_fill);
  }
  if (lse && lane == 0)
    lse[b * lse_bs + (int64_t)h * lse_hs + (int64_t)i * lse_rs] =
        bad ? NAN : (M == -INFINITY ? -INFINITY : M + logf(ws));
}

template <typename T>
cudaError_t launch_combine_t(int n_splits, int64_t rows, int D, const float* po, const float* pl, void* o,
                             Layout ol, int H, int Sq, float* lse, int64_t lbs, int64_t lhs, int64_t lrs,
                             int masked_zero, int sink_on, const float* sink, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + 3) / 4;
  if (blocks > INT_MAX) return cudaErrorInvalidConfiguration;
  combine_kernel<T><<<(unsigned)blocks, 128, 0, st>>>(n_splits, rows, D, po, pl, static_cast<T*>(o), ol, H, Sq,
                                                      lse, lbs, lhs, lrs, masked_zero, sink_on, sink);
  return cudaGetLastError();
}

cudaError_t combine_dispatch(int32_t dt, int n_splits, int64_t rows, int D, const float* po, const float* pl,
                             void* o, Layout ol, int H, int Sq, float* lse, int64_t lbs, int64_t lhs,
                             int64_t lrs, int masked_zero, int sink_on, const float* sink, cudaStream_t st) {
  switch (dt) {
    case ATTN_F32:
      return launch_combine_t<float>(n_splits, rows, D, po, pl, o, ol, H, Sq, lse, lbs, lhs, lrs, masked_zero,
                                     sink_on, sink, st);
    case ATTN_F16:
      return launch_combine_t<__half>(n_splits, rows, D, po, pl, o, ol, H, Sq, lse, lbs, lhs, lrs, masked_zero,
                                      sink_on, sink, st);
    default:
      return launch_combine_t<__nv_bfloat16>(n_splits, rows, D, po, pl, o, ol, H, Sq, lse, lbs, lhs, lrs,
                                             masked_zero, sink_on, sink, st);
  }
}

}  // namespace

cudaError_t launch_simt(const Problem& p, const Split& s, cudaStream_t st) {
  if (p.D == 32 || p.D == 64 || p.D == 128 || p.D == 256) return launch_simt_full(p, s, st);
  return launch_simt_all<false>(p, s, st);
}

cudaError_t launch_combine(const Problem& p, const Split& s, int32_t out_dtype, cudaStream_t st) {
  const int64_t rows = (int64_t)p.B * p.H * p.Sq;
  return combine_dispatch(out_dtype, s.n_splits, rows, p.D, s.part_o, s.part_lse, p.O, p.o, p.H, p.Sq, p.lse,
                          p.lse_bs, p.lse_hs, 1, p.masked_zero, p.sink_on, p.sink, st);
}

cudaError_t launch_combine_flat(int n_splits, int rows, int D, const float* part_o, const float* part_lse,
                                int32_t out_dtype, void* o, int64_t o_row_stride, float* lse, int masked_zero,
                                cudaStream_t st) {
  Layout ol{0, 0, 0, o_row_stride};
  return combine_dispatch(out_dtype, n_splits, rows, D, part_o, part_lse, o, ol, 1, rows, lse, 0, 0, 1,
                          masked_zero, 0, nullptr, st);
}

}  // namespace attn
