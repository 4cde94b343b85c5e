// simt_full.cu -- the chunked form of the CUDA-core forward (head_dim equal
// to 8 x threads-per-row: 32, 64, 128, 256), compiled apart from the general
// layout's instances in simt.cu.
#include "simt_fwd.cuh"

namespace attn {

cudaError_t launch_simt_full(const Problem& p, const Split& s, cudaStream_t st) {
  return launch_simt_all<true>(p, s, st);
}

}  // namespace attn
