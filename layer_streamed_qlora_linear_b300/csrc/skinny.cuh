// The rank-r side products of the LoRA linear (tcgen05, one launch each).
#pragma once
#include "common.cuh"

namespace sl {

constexpr int kSkMaxGroups = 4;

// out [M, G r] fp32 = Q [M, C] * W^T for a group of G adapters of rank r
// (G = 1: a single adapter):
//   wt = 0: W = A_cat [G r, C] (the adapters' A stacked);
//   wt = 1: W = blockdiag(B_g)^T with B_cat [C, r] (the adapters' B stacked
//           along C; columns [bounds[g], bounds[g+1]) of Q belong to adapter g).
// bounds: G + 1 increasing column offsets, multiples of 128, bounds[G] = C;
// nullptr when G == 1.
sl_status skinny_down(const uint16_t* Q, int64_t M, int C, const uint16_t* W, int wt, int r, int G, const int* bounds,
                      float* out, cudaStream_t stream);
// out = (accumulate ? out : 0) + s * P'^T Q with P [M, G r] fp32 and Q [M, C] bf16:
//   select = 0: P' = P, out [G r, C] (transpose = 1, dA_cat) or [C, G r];
//   select = 1: columns of Q in adapter g use P' = P[:, g r .. g r + r),
//               out [C, r] (transpose = 0, dB_cat).
sl_status skinny_grad(const float* P, const uint16_t* Q, int64_t M, int C, int r, int G, const int* bounds, int select,
                      float s, float* out, int transpose, int accumulate, cudaStream_t stream);
// dA and dB of one backward (two skinny_grad passes sharing M, r, G, s and
// accumulate) as one launch.
struct GradPass {
  const float* P;
  const uint16_t* Q;
  int C;
  const int* bounds;
  int select;
  float* out;
  int transpose;
};
sl_status skinny_grad_pair(const GradPass& p0, const GradPass& p1, int64_t M, int r, int G, float s, int accumulate,
                           cudaStream_t stream);
// The SwiGLU backward fused with the gate/up group's U pass (dg, du bitwise
// glue_swiglu_bwd's): dg, du [M, F] (row stride ld_out) from dm [M, F]
// (dense) and g, u (row stride ld_in), and U [M, 2 r] = [dg | du]
// blockdiag(B_g, B_u) with B_cat = [B_g; B_u] [2F, r].
sl_status skinny_swiglu_u(const uint16_t* dm, const uint16_t* g, const uint16_t* u, int64_t ld_in, uint16_t* dg,
                          uint16_t* du, int64_t ld_out, int64_t M, int F, const uint16_t* B_cat, int r, float* U,
                          cudaStream_t stream);

}  // namespace sl
