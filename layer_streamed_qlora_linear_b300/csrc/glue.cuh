// Row-wise / elementwise kernels of the synthetic decoder layer (see glue.cu).
#pragma once
#include "common.cuh"

namespace sl {

// w: the norm's fp32 weight [D] or nullptr
sl_status glue_rms_fwd(const float* h, const uint16_t* add, float* h_out, uint16_t* x, float* rstd,
                       const float* w, int64_t M, int D, cudaStream_t s);
// q at row stride ldq, k and v at row stride ldkv (column blocks of a
// projection group's output or dense arrays); a dense [M, D].
sl_status glue_mix_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* a, int64_t M, int D,
                       int Dkv, int64_t ldq, int64_t ldkv, cudaStream_t s);
// g, u at row stride ld; m dense [M, F].
sl_status glue_swiglu_fwd(const uint16_t* g, const uint16_t* u, uint16_t* m, int64_t M, int F, int64_t ld,
                          cudaStream_t s);
sl_status glue_resid_add(const float* h, const uint16_t* add, float* out, int64_t n, cudaStream_t s);
sl_status glue_to_bf16(const float* x, uint16_t* y, int64_t n, cudaStream_t s);
sl_status glue_swiglu_bwd(const uint16_t* dm, const uint16_t* g, const uint16_t* u, uint16_t* dg, uint16_t* du,
                          int64_t M, int F, int64_t ld, cudaStream_t s);
// dx = dxf (fp32) or dx0 + dx1 + dx2 (bf16, dx1/dx2 nullable); dh_in, w nullable
sl_status glue_rms_bwd(const float* dh_in, const uint16_t* dx0, const uint16_t* dx1, const uint16_t* dx2,
                       const float* dxf, const float* h, const float* rstd, const float* w, float* dh_out,
                       uint16_t* dh_bf16, int64_t M, int D, cudaStream_t s);
sl_status glue_embed(const int32_t* tokens, const uint16_t* embed, int64_t V, float* h0, int64_t M, int D, int* err,
                     cudaStream_t s);
sl_status glue_mix_bwd(const uint16_t* da, const uint16_t* q, const uint16_t* k, uint16_t* dq, uint16_t* dk,
                       uint16_t* dv, int64_t M, int D, int Dkv, int64_t ldq, int64_t ldkv, cudaStream_t s);

}  // namespace sl
