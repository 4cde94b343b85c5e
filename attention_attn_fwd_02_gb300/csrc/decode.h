// decode.h -- bandwidth-bound split-range decode pass.
#pragma once
#include "common.cuh"

namespace attn {
// Launches the specialised decode split pass when the problem fits it
// (f16/bf16, head_dim 128, a cache layout TMA can describe).
// Sets *used = 1 when it launched; returns an ATTN_* status.
int decode_fast_try(const Problem& p, const Split& s, cudaStream_t st, int* used);
// The same for an int8 key/value cache (f16/bf16 queries, head_dim 128).
int decode_q8_try(const Problem& p, const Split& s, cudaStream_t st, int* used);
}  // namespace attn
