// The frozen-base LoRA linear, forward and backward (steps a3, a4, a6).
//
// "Exact Layer Streaming ..." (abstract): LoRA training with the base frozen
// in NF4; only the adapters A [r, K] and B [N, r] learn.
//   forward   T = X A^T (K2, here);  Y = X W^T + s T B^T (one fused tcgen05 GEMM)
//   backward  U = dY B (K4, here);   dX = dY W + s U A (one fused GEMM)
//             dA = s U^T X, dB = s dY^T T (K6, here; fp32, fixed-order sums)
// The skinny kernels are HBM-bound streams over X / dY; the rank-r operand
// is staged in shared memory and every reduction runs in a fixed order so
// that results are bitwise reproducible.
#include "common.cuh"
#include "gemm.cuh"
#include "linear.cuh"

namespace sl {

// out[m, i] = sum_k X[m, k] * W(i, k)  (fp32),  W(i, k) = Wp[i * w_si + k * w_sk]
// 8 warps x 2 rows per block; W staged 256 columns at a time.
template <int R>
__global__ void __launch_bounds__(256) lora_down_kernel(const uint16_t* __restrict__ X, int64_t M, int K,
                                                        const uint16_t* __restrict__ Wp, int64_t w_si,
                                                        int64_t w_sk, int r, float* __restrict__ out) {
  __shared__ __align__(16) uint16_t wsm[R][256 + 8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * 16 + warp * 2;
  float acc[2][R];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int i = 0; i < R; ++i) acc[a][i] = 0.0f;
  for (int k0 = 0; k0 < K; k0 += 256) {
    __syncthreads();
    if (w_sk == 1) {
      for (int idx = threadIdx.x; idx < R * 256; idx += 256) {
        const int i = idx >> 8, kk = idx & 255;
        wsm[i][kk] = (i < r && k0 + kk < K) ? Wp[i * w_si + (k0 + kk)] : 0;
      }
    } else {
      for (int idx = threadIdx.x; idx < R * 256; idx += 256) {
        const int kk = idx / R, i = idx % R;
        wsm[i][kk] = (i < r && k0 + kk < K) ? Wp[i * w_si + static_cast<int64_t>(k0 + kk) * w_sk] : 0;
      }
    }
    __syncthreads();
    const int kk = lane * 8;
    if (k0 + kk < K) {
      float xv[2][8];
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int64_t row = row0 + a;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < M) v = *reinterpret_cast<const uint4*>(X + row * K + k0 + kk);
        const uint32_t p[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xv[a][2 * e] = bf16_lo(p[e]);
          xv[a][2 * e + 1] = bf16_hi(p[e]);
        }
      }
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const uint4 wv = *reinterpret_cast<const uint4*>(&wsm[i][kk]);
        const uint32_t p[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float w0 = bf16_lo(p[e]), w1 = bf16_hi(p[e]);
#pragma unroll
          for (int a = 0; a < 2; ++a) acc[a][i] = fmaf(xv[a][2 * e + 1], w1, fmaf(xv[a][2 * e], w0, acc[a][i]));
        }
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int64_t row = row0 + a;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      float v = acc[a][i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && row < M && i < r) out[row * r + i] = v;
    }
  }
}

// part[split][i][k] = sum_{m in split} P[m, i] * Q[m, k]   (fixed m order)
template <int R>
__global__ void __launch_bounds__(256) lora_grad_partial_kernel(const float* __restrict__ P,
                                                                const uint16_t* __restrict__ Q, int64_t M, int Kq,
                                                                int r, int64_t m_per_split,
                                                                float* __restrict__ part) {
  constexpr int RG = R / 4;
  __shared__ float psm[64][R + 1];
  const int c = threadIdx.x & 63, g = threadIdx.x >> 6;
  const int col = blockIdx.x * 64 + c;
  const int split = blockIdx.y;
  const int64_t mb = split * m_per_split;
  const int64_t me = (mb + m_per_split < M) ? mb + m_per_split : M;
  float acc[RG];
#pragma unroll
  for (int j = 0; j < RG; ++j) acc[j] = 0.0f;
  for (int64_t mc = mb; mc < me; mc += 64) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < 64 * R; idx += 256) {
      const int mm = idx / R, i = idx % R;
      psm[mm][i] = (mc + mm < me && i < r) ? P[(mc + mm) * r + i] : 0.0f;
    }
    __syncthreads();
    const int nrow = static_cast<int>((me - mc) < 64 ? (me - mc) : 64);
    if (col < Kq) {
      for (int mm = 0; mm < nrow; ++mm) {
        const float q = bf16_to_f32(Q[(mc + mm) * Kq + col]);
#pragma unroll
        for (int j = 0; j < RG; ++j) acc[j] = fmaf(psm[mm][g * RG + j], q, acc[j]);
      }
    }
  }
  if (col < Kq) {
#pragma unroll
    for (int j = 0; j < RG; ++j) {
      const int i = g * RG + j;
      if (i < r) part[(static_cast<int64_t>(split) * r + i) * Kq + col] = acc[j];
    }
  }
}

// out = (accumulate ? out : 0) + s * sum_split part[split]   (fixed split order)
// transpose: out[k * r + i] (dB [N, r]) instead of out[i * Kq + k] (dA [r, K]).
__global__ void lora_grad_reduce_kernel(const float* __restrict__ part, int splits, int r, int Kq, float s,
                                        float* __restrict__ out, int transpose, int accumulate) {
  const int64_t total = static_cast<int64_t>(r) * Kq;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t i = idx / Kq, k = idx % Kq;
    float v = 0.0f;
    for (int sp = 0; sp < splits; ++sp) v += part[(static_cast<int64_t>(sp) * r + i) * Kq + k];
    v *= s;
    const int64_t o = transpose ? k * r + i : idx;
    out[o] = accumulate ? out[o] + v : v;
  }
}

int grad_splits(int64_t M) {
  int64_t s = ceil_div(M, 256);
  return static_cast<int>(s < 1 ? 1 : (s > 16 ? 16 : s));
}

sl_status lora_down(const uint16_t* X, int64_t M, int K, const uint16_t* W, int64_t w_si, int64_t w_sk, int r,
                    float* out, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(ceil_div(M, 16));
#define SL_DOWN(RR) lora_down_kernel<RR><<<grid, 256, 0, stream>>>(X, M, K, W, w_si, w_sk, r, out)
  if (r <= 8) SL_DOWN(8);
  else if (r <= 16) SL_DOWN(16);
  else SL_DOWN(32);
#undef SL_DOWN
  return check_launch("lora_down_kernel");
}

sl_status lora_grad(const float* P, const uint16_t* Q, int64_t M, int Kq, int r, float s, float* out,
                    int transpose, int accumulate, float* part, cudaStream_t stream) {
  const int splits = grad_splits(M);
  const int64_t mps = ceil_div(ceil_div(M, splits), 64) * 64;
  dim3 grid(static_cast<unsigned>(ceil_div(Kq, 64)), static_cast<unsigned>(splits));
#define SL_GRAD(RR) lora_grad_partial_kernel<RR><<<grid, 256, 0, stream>>>(P, Q, M, Kq, r, mps, part)
  if (r <= 8) SL_GRAD(8);
  else if (r <= 16) SL_GRAD(16);
  else SL_GRAD(32);
#undef SL_GRAD
  sl_status st = check_launch("lora_grad_partial_kernel");
  if (st != SL_OK) return st;
  const int64_t total = static_cast<int64_t>(r) * Kq;
  int grid2 = static_cast<int>(ceil_div(total, 256));
  if (grid2 > num_sms() * 8) grid2 = num_sms() * 8;
  lora_grad_reduce_kernel<<<grid2, 256, 0, stream>>>(part, splits, r, Kq, s, out, transpose, accumulate);
  return check_launch("lora_grad_reduce_kernel");
}

size_t linear_bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int r) {
  if (r <= 0) return 0;
  const int splits = grad_splits(M);
  return align_up(static_cast<size_t>(M) * r * 4, 256) + align_up(static_cast<size_t>(splits) * r * K * 4, 256) +
         align_up(static_cast<size_t>(splits) * r * N * 4, 256);
}

static sl_status check_weight(const sl_weight* w) {
  SL_REQUIRE(w, "null sl_weight");
  SL_REQUIRE(w->N > 0 && w->K > 0, "sl_weight: N and K must be positive");
  SL_REQUIRE(w->N % 32 == 0, "sl_weight: N must be a multiple of 32");
  if (w->kind == SL_WEIGHT_NF4) {
    SL_REQUIRE(w->codes && w->absmax, "sl_weight: NF4 needs codes and absmax");
    SL_REQUIRE(w->K % 256 == 0, "sl_weight: NF4 needs K % 256 == 0");
  } else if (w->kind == SL_WEIGHT_BF16) {
    SL_REQUIRE(w->w, "sl_weight: BF16 needs w");
    SL_REQUIRE(w->K % 64 == 0, "sl_weight: BF16 needs K % 64 == 0");
  } else {
    return set_error(SL_ERR_INVALID, "sl_weight: unknown kind");
  }
  return SL_OK;
}

sl_status linear_fwd(const sl_weight* w, const void* X, int64_t M, const void* A, const void* B, int r,
                     float alpha, void* Y, void* T_save, cudaStream_t stream) {
  sl_status st = check_weight(w);
  if (st != SL_OK) return st;
  SL_REQUIRE(X && Y && M > 0, "sl_lora_linear_fwd: null X/Y or M <= 0");
  const bool lora = r > 0 && A && B;
  SL_REQUIRE(!lora || (r % 8 == 0 && r <= 32 && T_save), "sl_lora_linear_fwd: need r % 8 == 0, r <= 32, T_save");
  SL_REQUIRE(M < (1LL << 31), "sl_lora_linear_fwd: M too large");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  if (lora) {
    st = lora_down(static_cast<const uint16_t*>(X), M, static_cast<int>(w->K), static_cast<const uint16_t*>(A),
                   w->K, 1, r, static_cast<float*>(T_save), stream);
    if (st != SL_OK) return st;
  }
  GemmLaunch g{};
  g.bsrc = (w->kind == SL_WEIGHT_NF4) ? kBSrcNF4 : kBSrcBF16;
  g.bmn = 0;
  g.epi = kEpiStoreBF16;
  g.A = X;
  g.lda = w->K;
  g.w = w->w;
  g.codes = w->codes;
  g.absmax = w->absmax;
  g.ldw = w->K;
  g.args.M = static_cast<int>(M);
  g.args.N = static_cast<int>(w->N);
  g.args.K = static_cast<int>(w->K);
  g.args.lora_x = lora ? static_cast<const float*>(T_save) : nullptr;
  g.args.lora_w = lora ? static_cast<const uint16_t*>(B) : nullptr;
  g.args.r = lora ? r : 0;
  g.args.s = lora ? alpha / static_cast<float>(r) : 0.0f;
  g.args.out = Y;
  g.args.ld_out = w->N;
  g.args.err = err;
  return launch_gemm(g, stream);
}

sl_status linear_bwd(const sl_weight* w, const void* X, const void* dY, int64_t M, const void* A, const void* B,
                     int r, float alpha, const void* T_save, void* dX, float* dA, float* dB, int accumulate,
                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  sl_status st = check_weight(w);
  if (st != SL_OK) return st;
  SL_REQUIRE(dY && M > 0, "sl_lora_linear_bwd: null dY or M <= 0");
  const bool lora = r > 0 && A && B;
  SL_REQUIRE(!lora || (r % 8 == 0 && r <= 32), "sl_lora_linear_bwd: need r % 8 == 0 and r <= 32");
  SL_REQUIRE(!lora || (X && T_save && dA && dB), "sl_lora_linear_bwd: LoRA backward needs X, T_save, dA, dB");
  SL_REQUIRE(M < (1LL << 31), "sl_lora_linear_bwd: M too large");
  const size_t need = lora ? linear_bwd_ws_bytes(M, w->N, w->K, r) : 0;
  SL_REQUIRE(ws_bytes >= need && (need == 0 || ws), "sl_lora_linear_bwd: workspace too small");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255) == 0, "sl_lora_linear_bwd: workspace must be 256-byte aligned");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  uint8_t* p = static_cast<uint8_t*>(ws);
  float* U = nullptr;
  float* partA = nullptr;
  float* partB = nullptr;
  if (lora) {
    const int splits = grad_splits(M);
    U = reinterpret_cast<float*>(p);
    p += align_up(static_cast<size_t>(M) * r * 4, 256);
    partA = reinterpret_cast<float*>(p);
    p += align_up(static_cast<size_t>(splits) * r * w->K * 4, 256);
    partB = reinterpret_cast<float*>(p);
    // U = dY B : W(i, n) = B[n * r + i]
    st = lora_down(static_cast<const uint16_t*>(dY), M, static_cast<int>(w->N), static_cast<const uint16_t*>(B), 1,
                   r, r, U, stream);
    if (st != SL_OK) return st;
  }
  if (dX) {
    GemmLaunch g{};
    g.bsrc = (w->kind == SL_WEIGHT_NF4) ? kBSrcNF4 : kBSrcBF16;
    g.bmn = 1;
    g.epi = kEpiStoreBF16;
    g.A = dY;
    g.lda = w->N;
    g.w = w->w;
    g.codes = w->codes;
    g.absmax = w->absmax;
    g.ldw = w->K;
    g.args.M = static_cast<int>(M);
    g.args.N = static_cast<int>(w->K);
    g.args.K = static_cast<int>(w->N);
    g.args.lora_x = lora ? U : nullptr;
    g.args.lora_w = lora ? static_cast<const uint16_t*>(A) : nullptr;
    g.args.r = lora ? r : 0;
    g.args.s = lora ? alpha / static_cast<float>(r) : 0.0f;
    g.args.out = dX;
    g.args.ld_out = w->K;
    g.args.err = err;
    SL_REQUIRE(w->K % 32 == 0, "sl_lora_linear_bwd: K must be a multiple of 32");
    st = launch_gemm(g, stream);
    if (st != SL_OK) return st;
  }
  if (lora) {
    const float s = alpha / static_cast<float>(r);
    st = lora_grad(U, static_cast<const uint16_t*>(X), M, static_cast<int>(w->K), r, s, dA, 0, accumulate, partA,
                   stream);
    if (st != SL_OK) return st;
    st = lora_grad(static_cast<const float*>(T_save), static_cast<const uint16_t*>(dY), M,
                   static_cast<int>(w->N), r, s, dB, 1, accumulate, partB, stream);
    if (st != SL_OK) return st;
  }
  return SL_OK;
}

}  // namespace sl

using namespace sl;

extern "C" sl_status sl_lora_linear_fwd(const sl_weight* w, const void* X, int64_t M, const void* A, const void* B,
                                        int32_t r, float alpha, void* Y, void* T_save, void* ws, size_t ws_bytes,
                                        cudaStream_t stream) {
  (void)ws;
  (void)ws_bytes;
  return linear_fwd(w, X, M, A, B, r, alpha, Y, T_save, stream);
}

extern "C" sl_status sl_lora_linear_bwd(const sl_weight* w, const void* X, const void* dY, int64_t M, const void* A,
                                        const void* B, int32_t r, float alpha, const void* T_save, void* dX,
                                        float* dA, float* dB, int32_t accumulate, void* ws, size_t ws_bytes,
                                        cudaStream_t stream) {
  return linear_bwd(w, X, dY, M, A, B, r, alpha, T_save, dX, dA, dB, accumulate, ws, ws_bytes, stream);
}

extern "C" size_t sl_lora_linear_workspace_size(int64_t M, int64_t N, int64_t K, int32_t r) {
  return linear_bwd_ws_bytes(M, N, K, r);
}
