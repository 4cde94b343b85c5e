// probe.cu -- exponential-throughput micro-kernel (a measurement utility, not
// part of the attention path).
//
// The softmax evaluates one base-2 exponential per visible query-key pair
// ("Attention" (recursiveai.org OneGPU docs), opening paragraph: p = exp(s - m)
// for every score), so the rate of the hardware exponential bounds the
// prefill beside the tensor cores.  This kernel measures that rate: every
// thread runs eight independent chains x <- ex2(-x), which stay in [-1, -0.5]
// after the first step, so each step is one approximate exponential with no
// other arithmetic on its path.  The caller times it with events.
#include "common.cuh"

namespace attn {
namespace {

constexpr int kProbeThreads = 256;

__global__ void __launch_bounds__(kProbeThreads) ex2_probe_kernel(int iters, float* sink) {
  float x[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = -0.5f - 0.0625f * j - 1e-6f * threadIdx.x;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = -ex2_approx(x[j]);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += x[j];
  // One value per CTA keeps the chains alive.
  __shared__ float red[kProbeThreads / 32];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kProbeThreads / 32; ++w) t += red[w];
    sink[blockIdx.x] = t;
  }
}

}  // namespace

cudaError_t launch_ex2_probe(int blocks, int iters, float* sink, cudaStream_t st) {
  ex2_probe_kernel<<<(unsigned)blocks, kProbeThreads, 0, st>>>(iters, sink);
  return cudaGetLastError();
}

}  // namespace attn
