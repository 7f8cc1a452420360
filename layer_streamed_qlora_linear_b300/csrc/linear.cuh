// Internal entry points of the LoRA linear, shared by the C ABI and the
// stack scheduler (same kernels, same order, in both resident and streamed
// runs).
#pragma once
#include "common.cuh"

namespace sl {

sl_status linear_fwd(const sl_weight* w, const void* X, int64_t M, const void* A, const void* B, int r,
                     float alpha, void* Y, void* T_save, void* ws, size_t ws_bytes, cudaStream_t stream);
// The forward with the GEMM's split-K scratch given directly (nullptr: none).
sl_status linear_fwd_x(const sl_weight* w, const void* X, int64_t M, const void* A, const void* B, int r,
                       float alpha, void* Y, void* T_save, void* split_ws, size_t split_bytes, cudaStream_t stream);
sl_status linear_bwd(const sl_weight* w, const void* X, const void* dY, int64_t M, const void* A, const void* B,
                     int r, float alpha, const void* T_save, void* dX, float* dA, float* dB, int accumulate,
                     void* ws, size_t ws_bytes, cudaStream_t stream);
// Where a backward runs its adapter-gradient passes (dA, dB): on `stream`
// after waiting for `fork`, which the main stream records once U is
// written; `done` (optional) is recorded on `stream` after them.  With no
// side (nullptr) they run in order on the main stream.
struct GradSide {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t done = nullptr;
};
// The backward with U and the dX GEMM on `main` and dA, dB on `side`.
sl_status linear_bwd_split(const sl_weight* w, const void* X, const void* dY, int64_t M, const void* A, const void* B,
                           int r, float alpha, const void* T_save, void* dX, float* dA, float* dB, int accumulate,
                           void* ws, size_t ws_bytes, cudaStream_t main, const GradSide* side, void* split_ws,
                           size_t split_bytes);
size_t linear_ws_bytes(int64_t M, int64_t N, int64_t K, int r);
// Projection groups (sl_lora_group_fwd / _bwd).
sl_status group_fwd(const sl_weight* w, int G, const int64_t* N_g, const void* X, int64_t M, const void* A_cat,
                    const void* B_cat, int r, float alpha, void* Y_cat, void* T_cat, cudaStream_t stream);
sl_status group_fwd_x(const sl_weight* w, int G, const int64_t* N_g, const void* X, int64_t M, const void* A_cat,
                      const void* B_cat, int r, float alpha, void* Y_cat, void* T_cat, void* split_ws,
                      size_t split_bytes, cudaStream_t stream);
sl_status group_bwd(const sl_weight* w, int G, const int64_t* N_g, const void* X, const void* dY_cat, int64_t M,
                    const void* A_cat, const void* B_cat, int r, float alpha, const void* T_cat, void* dX, float* dA_cat,
                    float* dB_cat, int accumulate, void* ws, size_t ws_bytes, cudaStream_t stream);
// u_ready: the workspace's U_cat region already holds dY_cat blockdiag(B_g)
// (written by a fused producer), so the U pass is skipped.
sl_status group_bwd_split(const sl_weight* w, int G, const int64_t* N_g, const void* X, const void* dY_cat, int64_t M,
                          const void* A_cat, const void* B_cat, int r, float alpha, const void* T_cat, void* dX,
                          float* dA_cat, float* dB_cat, int accumulate, void* ws, size_t ws_bytes, cudaStream_t main,
                          const GradSide* side, void* split_ws, size_t split_bytes, bool u_ready = false);
size_t group_ws_bytes(int64_t M, int G, int r);

}  // namespace sl
