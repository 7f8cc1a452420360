// The rank-r side products of the LoRA linear (tcgen05, one launch each).
#pragma once
#include "common.cuh"

namespace sl {

// out [M, r] fp32 = Q [M, C] * W^T, W = A [r, C] (wt = 0) or B [C, r] (wt = 1).
sl_status skinny_down(const uint16_t* Q, int64_t M, int C, const uint16_t* W, int wt, int r, float* out,
                      cudaStream_t stream);
// out = (accumulate ? out : 0) + s * P^T Q, P [M, r] fp32, Q [M, C] bf16;
// stored [r, C] (transpose = 1, dA) or [C, r] (transpose = 0, dB).
sl_status skinny_grad(const float* P, const uint16_t* Q, int64_t M, int C, int r, float s, float* out, int transpose,
                      int accumulate, cudaStream_t stream);

}  // namespace sl
