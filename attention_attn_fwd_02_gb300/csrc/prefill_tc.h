// prefill_tc.h -- tensor-core (tcgen05 + TMEM + TMA) prefill path.
#pragma once
#include "common.cuh"

namespace attn {
// Launches the tensor-core kernel when the problem fits it (f16/bf16, a
// head_dim it is built for, a layout TMA can describe).  Sets *used = 1 when
// it launched; returns an ATTN_* status.
// With s.n_splits > 1 every CTA also takes one key range and writes that
// range's partial (O / l in float32, and its LSE) to s.part_o / s.part_lse.
int prefill_tc_try(const Problem& p, const Split& s, cudaStream_t st, int* used);

// The head_dim 256 kernel (one query tile per CTA, double-buffered S).
// Returns -1 when TMA cannot describe the layout, else an ATTN_* status.
int prefill_tc1_launch(const Problem& p, const Split& s, cudaStream_t st);

// The head_dim 256 kernel on CTA pairs (cta_group::2): each pair shares its K
// and V tiles.  Returns -1 when it does not apply (segment starts) or TMA
// cannot describe the layout, else an ATTN_* status.
int prefill_tc2_launch(const Problem& p, const Split& s, cudaStream_t st);
}  // namespace attn
