// The frozen-base LoRA linear, forward and backward (steps a3, a4, a6).
//
// "Exact Layer Streaming ..." (abstract): LoRA training with the base frozen
// in NF4; only the adapters A [r, K] and B [N, r] learn.
//   forward   T = X A^T;  Y = X W^T + s T B^T (one fused tcgen05 GEMM)
//   backward  U = dY B;   dX = dY W + s U A (one fused GEMM)
//             dA = s U^T X, dB = s dY^T T
// The rank-r products run as single tcgen05 launches (skinny.cu) with
// fixed-order cluster reductions, so results are bitwise reproducible.  The
// CUDA-core rank-r kernels below serve only the allocation-free forward,
// whose K-split partials live in a fixed device array.
#include <algorithm>
#include <mutex>
#include <string>

#include "common.cuh"
#include "gemm.cuh"
#include "linear.cuh"
#include "skinny.cuh"

namespace sl {

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------- CUDA-core T (allocation-free forward)
// part[split][m][i] = sum_{k in split} X[m, k] * W(i, k), fp32.
// W(i, k) = Wp[i * K + k] (kWT == 0: A [r, K]) or Wp[k * r + i] (kWT == 1: B [N, r]).
// Block: 128 threads, 32 rows x 512 columns of X staged in shared memory by
// cp.async (all loads in flight at once); thread = (row, quarter of the rank).
constexpr int kDnRows = 32;
constexpr int kDnCols = 512;
constexpr int kDnPad = 8;

template <int R, int kWT>
__global__ void __launch_bounds__(128) lora_down_kernel(const uint16_t* __restrict__ X, int64_t M, int K,
                                                        const uint16_t* __restrict__ Wp, int r,
                                                        float* __restrict__ part) {
  extern __shared__ __align__(16) uint8_t dsm[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(dsm);                            // [32][512 + 8]
  uint16_t* ws = xs + kDnRows * (kDnCols + kDnPad);                           // [R][512 + 8] or [512][R]
  const int tid = threadIdx.x;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kDnRows;
  const int k0 = blockIdx.y * kDnCols;
  const int kn = (K - k0 < kDnCols) ? (K - k0) : kDnCols;  // multiple of 8
  // X tile: 32 rows x 64 chunks of 16 bytes
  for (int c = tid; c < kDnRows * (kDnCols / 8); c += 128) {
    const int row = c / (kDnCols / 8), ch = c % (kDnCols / 8);
    const bool ok = (m0 + row < M) && (ch * 8 < kn);
    const uint16_t* src = ok ? X + (m0 + row) * K + k0 + ch * 8 : X;
    cp_async16(xs + row * (kDnCols + kDnPad) + ch * 8, src, ok);
  }
  if (kWT == 0) {
    for (int c = tid; c < R * (kDnCols / 8); c += 128) {
      const int i = c / (kDnCols / 8), ch = c % (kDnCols / 8);
      const bool ok = (i < r) && (ch * 8 < kn);
      const uint16_t* src = ok ? Wp + static_cast<int64_t>(i) * K + k0 + ch * 8 : Wp;
      cp_async16(ws + i * (kDnCols + kDnPad) + ch * 8, src, ok);
    }
  } else {
    // contiguous [kn, r] slice of B; smem layout [k][R]
    for (int c = tid; c < kDnCols * R / 8; c += 128) {
      const int kk = (c * 8) / R, i0 = (c * 8) % R;
      const bool ok = (kk < kn) && (i0 < r);
      const uint16_t* src = ok ? Wp + static_cast<int64_t>(k0 + kk) * r + i0 : Wp;
      cp_async16(ws + kk * R + i0, src, ok);
    }
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  constexpr int RQ = R / 4;
  const int row = tid >> 2, g = tid & 3;
  float acc[RQ];
#pragma unroll
  for (int j = 0; j < RQ; ++j) acc[j] = 0.0f;
  const uint16_t* xr = xs + row * (kDnCols + kDnPad);
  for (int k = 0; k < kn; k += 8) {
    const uint4 xv = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = bf16_lo(xw[e]);
      x[2 * e + 1] = bf16_hi(xw[e]);
    }
    if (kWT == 0) {
#pragma unroll
      for (int j = 0; j < RQ; ++j) {
        const uint4 wv = *reinterpret_cast<const uint4*>(ws + (g * RQ + j) * (kDnCols + kDnPad) + k);
        const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          acc[j] = fmaf(x[2 * e + 1], bf16_hi(w[e]), fmaf(x[2 * e], bf16_lo(w[e]), acc[j]));
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint16_t* wk = ws + (k + e) * R + g * RQ;
#pragma unroll
        for (int j = 0; j < RQ; j += 2) {
          const uint32_t w2 = *reinterpret_cast<const uint32_t*>(wk + j);
          acc[j] = fmaf(x[e], bf16_lo(w2), acc[j]);
          acc[j + 1] = fmaf(x[e], bf16_hi(w2), acc[j + 1]);
        }
      }
    }
  }
  const int64_t gm = m0 + row;
  if (gm < M) {
    float* dst = part + (static_cast<int64_t>(blockIdx.y) * M + gm) * r;
#pragma unroll
    for (int j = 0; j < RQ; ++j) {
      const int i = g * RQ + j;
      if (i < r) dst[i] = acc[j];
    }
  }
}

// out[m][i] = sum over splits (fixed order) of part[split][m][i]
__global__ void sum_splits_kernel(const float* __restrict__ part, int splits, int64_t n, float* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n; idx += stride) {
    float v = 0.0f;
    for (int sp = 0; sp < splits; ++sp) v += part[static_cast<int64_t>(sp) * n + idx];
    out[idx] = v;
  }
}

static int rank_bucket(int r) { return r <= 8 ? 8 : (r <= 16 ? 16 : 32); }

int down_splits(int64_t K) { return static_cast<int>(ceil_div(K, kDnCols)); }

static size_t down_smem(int R) {
  return (static_cast<size_t>(kDnRows) * (kDnCols + kDnPad) + static_cast<size_t>(R) * (kDnCols + kDnPad)) * 2;
}
// Set on every call (a cheap host-side call), so the attribute holds on
// whichever device is current.
template <typename Kern>
static sl_status set_smem(Kern k, size_t bytes) {
  SL_CHECK_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)));
  return SL_OK;
}

// out [M, r] fp32 = X [M, K] * W^T; W given as A [r, K] (wt = 0) or B [K, r] (wt = 1).
// part: scratch of down_splits(K) * M * r floats (unused when one split).
sl_status lora_down(const uint16_t* X, int64_t M, int K, const uint16_t* W, int wt, int r, float* out, float* part,
                    cudaStream_t stream) {
  const int splits = down_splits(K);
  float* dst = splits == 1 ? out : part;
  dim3 grid(static_cast<unsigned>(ceil_div(M, kDnRows)), static_cast<unsigned>(splits));
  const int R = rank_bucket(r);
  const size_t sm = down_smem(R);
#define SL_DOWN(RR, WT)                                                                           \
  do {                                                                                            \
    sl_status st_ = set_smem(lora_down_kernel<RR, WT>, sm);                                       \
    if (st_ != SL_OK) return st_;                                                                 \
    lora_down_kernel<RR, WT><<<grid, 128, sm, stream>>>(X, M, K, W, r, dst);                      \
  } while (0)
  if (R == 8) { if (wt) SL_DOWN(8, 1); else SL_DOWN(8, 0); }
  else if (R == 16) { if (wt) SL_DOWN(16, 1); else SL_DOWN(16, 0); }
  else { if (wt) SL_DOWN(32, 1); else SL_DOWN(32, 0); }
#undef SL_DOWN
  sl_status st = check_launch("lora_down_kernel");
  if (st != SL_OK || splits == 1) return st;
  const int64_t n = M * r;
  int g = static_cast<int>(ceil_div(n, 256));
  if (g > num_sms() * 4) g = num_sms() * 4;
  sum_splits_kernel<<<g, 256, 0, stream>>>(part, splits, n, out);
  return check_launch("sum_splits_kernel");
}

// Workspace of one linear: U [M, r] fp32 (backward only), then, when the
// CTA-pair GEMM runs (M > 128), the scratch that lets its last partial wave
// split along K (either direction).
struct LinWs {
  size_t U, U_bytes, split, total;
};

static LinWs lin_ws(int64_t M, int64_t N, int64_t K, int r) {
  (void)N;
  (void)K;
  LinWs w{};
  if (r <= 0) return w;
  w.U = 0;
  w.U_bytes = align_up(static_cast<size_t>(M) * r * 4, 256);
  w.split = w.U_bytes;
  w.total = w.U_bytes + (M > 128 ? split_scratch_bytes() : 0);
  return w;
}

// The split scratch inside a caller's workspace laid out as [U | split], if it is there.
static void* split_in(void* ws, size_t ws_bytes, size_t U_bytes) {
  if (!ws || ws_bytes < U_bytes + split_scratch_bytes() || (reinterpret_cast<uintptr_t>(ws) & 255)) return nullptr;
  return static_cast<uint8_t*>(ws) + U_bytes;
}

size_t linear_ws_bytes(int64_t M, int64_t N, int64_t K, int r) { return lin_ws(M, N, K, r).total; }

static sl_status check_weight(const sl_weight* w) {
  SL_REQUIRE(w, "null sl_weight");
  SL_REQUIRE(w->N > 0 && w->K > 0, "sl_weight: N and K must be positive");
  SL_REQUIRE(w->N % 32 == 0, "sl_weight: N must be a multiple of 32");
  if (w->kind == SL_WEIGHT_NF4) {
    SL_REQUIRE(w->codes && w->absmax, "sl_weight: NF4 needs codes and absmax");
    SL_REQUIRE(w->K % 256 == 0, "sl_weight: NF4 needs K % 256 == 0");
  } else if (w->kind == SL_WEIGHT_NF4_DQ) {
    SL_REQUIRE(w->codes && w->qabsmax && w->absmax2, "sl_weight: NF4_DQ needs codes, qabsmax and absmax2");
    SL_REQUIRE(w->K % 256 == 0 && w->N % 256 == 0, "sl_weight: NF4_DQ needs N % 256 == 0 and K % 256 == 0");
    SL_REQUIRE(w->dq_col0 >= 0 && w->dq_col0 % 256 == 0, "sl_weight: NF4_DQ needs dq_col0 a multiple of 256");
    SL_REQUIRE(w->qabsmax_ld % 16 == 0 && w->qabsmax_ld >= w->dq_col0 + w->N,
               "sl_weight: NF4_DQ needs qabsmax_ld % 16 == 0 and >= dq_col0 + N");
    SL_REQUIRE(w->absmax2_ld % 4 == 0 && w->absmax2_ld >= 2 * ((w->dq_col0 + w->N) / 256),
               "sl_weight: NF4_DQ needs absmax2_ld % 4 == 0 and >= 2 (dq_col0 + N) / 256");
  } else if (w->kind == SL_WEIGHT_BF16) {
    SL_REQUIRE(w->w, "sl_weight: BF16 needs w");
    SL_REQUIRE(w->K % 64 == 0, "sl_weight: BF16 needs K % 64 == 0");
  } else {
    return set_error(SL_ERR_INVALID, "sl_weight: unknown kind");
  }
  return SL_OK;
}

// The frozen weight as the GEMM's B operand.
static void bind_weight(GemmLaunch& g, const sl_weight* w) {
  g.bsrc = (w->kind == SL_WEIGHT_BF16) ? kBSrcBF16 : kBSrcNF4;
  g.w = w->w;
  g.codes = w->codes;
  g.absmax = w->absmax;
  g.ldw = w->K;
  if (w->kind == SL_WEIGHT_NF4_DQ) {
    g.args.dq = 1;
    g.args.dq_col0 = static_cast<int>(w->dq_col0);
    g.qabsmax = w->qabsmax;
    g.q_ld = w->qabsmax_ld;
    g.absmax2 = w->absmax2;
    g.a2_ld = w->absmax2_ld;
  }
}

// The double-quantised absmax is read by the persistent CTA-pair GEMM only.
static sl_status check_rows(const sl_weight* w, int64_t M, const char* who) {
  if (w->kind == SL_WEIGHT_NF4_DQ && M <= 128)
    return set_error(SL_ERR_UNSUPPORTED, std::string(who) + ": NF4_DQ weights need M > 128");
  return SL_OK;
}

sl_status linear_fwd(const sl_weight* w, const void* X, int64_t M, const void* A, const void* B, int r,
                     float alpha, void* Y, void* T_save, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const size_t U_bytes = r > 0 ? lin_ws(M, 0, 0, r).U_bytes : 0;
  void* split = split_in(ws, ws_bytes, U_bytes);
  return linear_fwd_x(w, X, M, A, B, r, alpha, Y, T_save, split, split ? split_scratch_bytes() : 0, stream);
}

sl_status linear_fwd_x(const sl_weight* w, const void* X, int64_t M, const void* A, const void* B, int r,
                       float alpha, void* Y, void* T_save, void* split_ws, size_t split_bytes, cudaStream_t stream) {
  sl_status st = check_weight(w);
  if (st != SL_OK) return st;
  SL_REQUIRE(X && Y && M > 0, "sl_lora_linear_fwd: null X/Y or M <= 0");
  const bool lora = r > 0 && A && B;
  SL_REQUIRE(!lora || (r % 8 == 0 && r <= 32 && T_save), "sl_lora_linear_fwd: need r % 8 == 0, r <= 32, T_save");
  SL_REQUIRE(M < (1LL << 31), "sl_lora_linear_fwd: M too large");
  st = check_rows(w, M, "sl_lora_linear_fwd");
  if (st != SL_OK) return st;
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  if (lora) {
    st = skinny_down(static_cast<const uint16_t*>(X), M, static_cast<int>(w->K), static_cast<const uint16_t*>(A), 0, r,
                     1, nullptr, static_cast<float*>(T_save), stream);
    if (st != SL_OK) return st;
  }
  GemmLaunch g{};
  g.split_ws = split_ws;
  g.split_ws_bytes = split_bytes;
  bind_weight(g, w);
  g.bmn = 0;
  g.epi = kEpiStoreBF16;
  g.A = X;
  g.lda = w->K;
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

sl_status linear_bwd_split(const sl_weight* w, const void* X, const void* dY, int64_t M, const void* A, const void* B,
                           int r, float alpha, const void* T_save, void* dX, float* dA, float* dB, int accumulate,
                           void* ws, size_t ws_bytes, cudaStream_t stream, const GradSide* side, void* split_ws,
                           size_t split_bytes) {
  sl_status st = check_weight(w);
  if (st != SL_OK) return st;
  SL_REQUIRE(dY && M > 0, "sl_lora_linear_bwd: null dY or M <= 0");
  const bool lora = r > 0 && A && B;
  SL_REQUIRE(!lora || (r % 8 == 0 && r <= 32), "sl_lora_linear_bwd: need r % 8 == 0 and r <= 32");
  SL_REQUIRE(!lora || (X && T_save && dA && dB), "sl_lora_linear_bwd: LoRA backward needs X, T_save, dA, dB");
  SL_REQUIRE(M < (1LL << 31), "sl_lora_linear_bwd: M too large");
  if (dX) {
    st = check_rows(w, M, "sl_lora_linear_bwd");
    if (st != SL_OK) return st;
  }
  const LinWs L = lin_ws(M, w->N, w->K, lora ? r : 0);
  SL_REQUIRE(ws_bytes >= L.U_bytes && (L.U_bytes == 0 || ws), "sl_lora_linear_bwd: workspace too small");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255) == 0, "sl_lora_linear_bwd: workspace must be 256-byte aligned");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  uint8_t* p = static_cast<uint8_t*>(ws);
  float* U = nullptr;
  if (lora) {
    U = reinterpret_cast<float*>(p + L.U);
    // U = dY B
    st = skinny_down(static_cast<const uint16_t*>(dY), M, static_cast<int>(w->N), static_cast<const uint16_t*>(B), 1,
                     r, 1, nullptr, U, stream);
    if (st != SL_OK) return st;
    if (side) {  // dA and dB go to the side stream once U is written
      SL_CHECK_CUDA(cudaEventRecord(side->fork, stream));
      SL_CHECK_CUDA(cudaStreamWaitEvent(side->stream, side->fork, 0));
    }
  }
  if (dX) {
    GemmLaunch g{};
    g.split_ws = split_ws;
    g.split_ws_bytes = split_bytes;
    bind_weight(g, w);
    g.bmn = 1;
    g.epi = kEpiStoreBF16;
    g.A = dY;
    g.lda = w->N;
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
    cudaStream_t gs = side ? side->stream : stream;
    // dA [r, K] = s U^T X;  dB [N, r] = s dY^T T  (one launch)
    const GradPass pa{U, static_cast<const uint16_t*>(X), static_cast<int>(w->K), nullptr, 0, dA, 1};
    const GradPass pb{static_cast<const float*>(T_save), static_cast<const uint16_t*>(dY), static_cast<int>(w->N),
                      nullptr, 1, dB, 0};
    st = skinny_grad_pair(pa, pb, M, r, 1, s, accumulate, gs);
    if (st != SL_OK) return st;
    if (side && side->done) SL_CHECK_CUDA(cudaEventRecord(side->done, gs));
  }
  return SL_OK;
}

// The caller's stream waits for `main` after running `body` there with the
// adapter-gradient passes on the caller's stream itself: U and the dX GEMM
// run on the high-priority library stream, whose blocks the GPU dispatches
// first, and dA / dB take the SMs the GEMM leaves idle.  Without that
// stream everything runs in order on the caller's stream.
template <typename Body>
static sl_status run_bwd_split(cudaStream_t stream, bool lora, Body body) {
  cudaStream_t hi = lora ? hi_stream() : nullptr;
  cudaEvent_t e_in = hi ? fork_event(0) : nullptr, e_fork = hi ? fork_event(1) : nullptr,
              e_out = hi ? fork_event(2) : nullptr;
  if (!hi || !e_in || !e_fork || !e_out) return body(stream, nullptr);
  SL_CHECK_CUDA(cudaEventRecord(e_in, stream));
  SL_CHECK_CUDA(cudaStreamWaitEvent(hi, e_in, 0));
  const GradSide side{stream, e_fork, nullptr};
  const sl_status st = body(hi, &side);
  // join even after a failure, so that the caller's stream stays ordered after all of it
  const cudaError_t e1 = cudaEventRecord(e_out, hi);
  const cudaError_t e2 = e1 == cudaSuccess ? cudaStreamWaitEvent(stream, e_out, 0) : e1;
  if (st != SL_OK) return st;
  if (e2 != cudaSuccess) return cuda_error(e2, "backward: joining the library stream");
  return SL_OK;
}

sl_status linear_bwd(const sl_weight* w, const void* X, const void* dY, int64_t M, const void* A, const void* B,
                     int r, float alpha, const void* T_save, void* dX, float* dA, float* dB, int accumulate,
                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  const size_t U_bytes = r > 0 ? lin_ws(M, 0, 0, r).U_bytes : 0;
  void* split = split_in(ws, ws_bytes, U_bytes);
  return run_bwd_split(stream, r > 0 && A && B, [&](cudaStream_t main, const GradSide* side) {
    return linear_bwd_split(w, X, dY, M, A, B, r, alpha, T_save, dX, dA, dB, accumulate, ws, ws_bytes, main, side,
                            split, split ? split_scratch_bytes() : 0);
  });
}

// ---------------------------------------------------------- projection groups
// G projections that read the same input (q, k, v or gate, up), frozen
// weights stored back to back along N (one sl_weight of N = sum N_g rows),
// adapters back to back (A_cat [G r, K], B_cat [sum N_g, r]).  One fused GEMM
// and one rank-r pass of each kind for the whole group.

static sl_status check_group(const sl_weight* w, int G, const int64_t* N_g, int64_t M, int r, int bounds[5]) {
  sl_status st = check_weight(w);
  if (st != SL_OK) return st;
  SL_REQUIRE(w->kind != SL_WEIGHT_BF16, "projection group: NF4 weights only");
  SL_REQUIRE(M > 128 && M < (1LL << 31), "projection group: need 128 < M < 2^31");
  SL_REQUIRE(G >= 1 && G <= kSkMaxGroups && N_g, "projection group: need 1 <= G <= 4 projections");
  SL_REQUIRE(r >= 0 && r % 8 == 0 && r <= 32 && G * r <= 64, "projection group: need r % 8 == 0, r <= 32, G r <= 64");
  int64_t off = 0;
  bounds[0] = 0;
  for (int g = 0; g < G; ++g) {
    SL_REQUIRE(N_g[g] > 0 && N_g[g] % 256 == 0, "projection group: every N_g must be a positive multiple of 256");
    off += N_g[g];
    bounds[g + 1] = static_cast<int>(off);
  }
  SL_REQUIRE(off == w->N, "projection group: the N_g must add up to the weight's N");
  for (int g = G + 1; g < 5; ++g) bounds[g] = bounds[G];
  return SL_OK;
}

// U_cat [M, G r] fp32, then the split-K scratch of the CTA-pair GEMM (M > 128).
static size_t group_U_bytes(int64_t M, int G, int r) {
  return r > 0 ? align_up(static_cast<size_t>(M) * G * r * 4, 256) : 0;
}
size_t group_ws_bytes(int64_t M, int G, int r) {
  return r > 0 ? group_U_bytes(M, G, r) + (M > 128 ? split_scratch_bytes() : 0) : 0;
}

sl_status group_fwd(const sl_weight* w, int G, const int64_t* N_g, const void* X, int64_t M, const void* A_cat,
                    const void* B_cat, int r, float alpha, void* Y_cat, void* T_cat, cudaStream_t stream) {
  return group_fwd_x(w, G, N_g, X, M, A_cat, B_cat, r, alpha, Y_cat, T_cat, nullptr, 0, stream);
}

sl_status group_fwd_x(const sl_weight* w, int G, const int64_t* N_g, const void* X, int64_t M, const void* A_cat,
                      const void* B_cat, int r, float alpha, void* Y_cat, void* T_cat, void* split_ws,
                      size_t split_bytes, cudaStream_t stream) {
  int bounds[5];
  sl_status st = check_group(w, G, N_g, M, r, bounds);
  if (st != SL_OK) return st;
  const bool lora = r > 0;
  SL_REQUIRE(X && Y_cat && (!lora || (A_cat && B_cat && T_cat)), "sl_lora_group_fwd: null argument");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  if (lora) {
    // T_cat [M, G r] = X A_cat^T
    st = skinny_down(static_cast<const uint16_t*>(X), M, static_cast<int>(w->K), static_cast<const uint16_t*>(A_cat), 0,
                     r, G, nullptr, static_cast<float*>(T_cat), stream);
    if (st != SL_OK) return st;
  }
  GemmLaunch g{};
  g.split_ws = split_ws;
  g.split_ws_bytes = split_bytes;
  bind_weight(g, w);
  g.bmn = 0;
  g.epi = kEpiStoreBF16;
  g.grouped = 1;
  g.A = X;
  g.lda = w->K;
  g.args.M = static_cast<int>(M);
  g.args.N = static_cast<int>(w->N);
  g.args.K = static_cast<int>(w->K);
  g.args.lora_x = lora ? static_cast<const float*>(T_cat) : nullptr;
  g.args.lora_w = lora ? static_cast<const uint16_t*>(B_cat) : nullptr;
  g.args.r = r;
  g.args.lora_ld = G * r;
  g.args.lora_G = G;
  for (int i = 0; i < 5; ++i) g.args.lora_bounds[i] = bounds[i];
  g.args.s = lora ? alpha / static_cast<float>(r) : 0.0f;
  g.args.out = Y_cat;
  g.args.ld_out = w->N;
  g.args.err = err;
  return launch_gemm(g, stream);
}

sl_status group_bwd_split(const sl_weight* w, int G, const int64_t* N_g, const void* X, const void* dY_cat, int64_t M,
                          const void* A_cat, const void* B_cat, int r, float alpha, const void* T_cat, void* dX,
                          float* dA_cat, float* dB_cat, int accumulate, void* ws, size_t ws_bytes,
                          cudaStream_t stream, const GradSide* side, void* split_ws, size_t split_bytes,
                          bool u_ready) {
  int bounds[5];
  sl_status st = check_group(w, G, N_g, M, r, bounds);
  if (st != SL_OK) return st;
  const bool lora = r > 0;
  SL_REQUIRE(dY_cat && (!lora || (X && A_cat && B_cat && T_cat && dA_cat && dB_cat)),
             "sl_lora_group_bwd: null argument");
  SL_REQUIRE(!lora || (ws && ws_bytes >= group_U_bytes(M, G, r) && (reinterpret_cast<uintptr_t>(ws) & 255) == 0),
             "sl_lora_group_bwd: workspace too small or not 256-byte aligned");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  const int NN = static_cast<int>(w->N), K = static_cast<int>(w->K);
  const float s = lora ? alpha / static_cast<float>(r) : 0.0f;
  float* U = lora ? static_cast<float*>(ws) : nullptr;
  if (lora) {
    // U_cat [M, G r] = dY_cat blockdiag(B_g)
    if (!u_ready) {
      st = skinny_down(static_cast<const uint16_t*>(dY_cat), M, NN, static_cast<const uint16_t*>(B_cat), 1, r, G,
                       bounds, U, stream);
      if (st != SL_OK) return st;
    }
    if (side) {  // dA and dB go to the side stream once U is written
      SL_CHECK_CUDA(cudaEventRecord(side->fork, stream));
      SL_CHECK_CUDA(cudaStreamWaitEvent(side->stream, side->fork, 0));
    }
  }
  if (dX) {
    // dX = dY_cat W_cat + s U_cat A_cat: the plain dX GEMM at rank G r
    GemmLaunch g{};
    g.split_ws = split_ws;
    g.split_ws_bytes = split_bytes;
    bind_weight(g, w);
    g.bmn = 1;
    g.epi = kEpiStoreBF16;
    g.grouped = 1;
    g.A = dY_cat;
    g.lda = NN;
    g.args.M = static_cast<int>(M);
    g.args.N = K;
    g.args.K = NN;
    g.args.lora_x = U;
    g.args.lora_w = lora ? static_cast<const uint16_t*>(A_cat) : nullptr;
    g.args.r = G * r;
    g.args.s = s;
    g.args.out = dX;
    g.args.ld_out = K;
    g.args.err = err;
    st = launch_gemm(g, stream);
    if (st != SL_OK) return st;
  }
  if (!lora) return SL_OK;
  cudaStream_t gs = side ? side->stream : stream;
  // dA_cat [G r, K] = s U_cat^T X;  dB_cat [sum N_g, r]: rows of projection g = s dY_g^T T_g  (one launch)
  const GradPass pa{U, static_cast<const uint16_t*>(X), K, nullptr, 0, dA_cat, 1};
  const GradPass pb{static_cast<const float*>(T_cat), static_cast<const uint16_t*>(dY_cat), NN, bounds, 1, dB_cat, 0};
  st = skinny_grad_pair(pa, pb, M, r, G, s, accumulate, gs);
  if (st != SL_OK) return st;
  if (side && side->done) SL_CHECK_CUDA(cudaEventRecord(side->done, gs));
  return SL_OK;
}

sl_status group_bwd(const sl_weight* w, int G, const int64_t* N_g, const void* X, const void* dY_cat, int64_t M,
                    const void* A_cat, const void* B_cat, int r, float alpha, const void* T_cat, void* dX, float* dA_cat,
                    float* dB_cat, int accumulate, void* ws, size_t ws_bytes, cudaStream_t stream) {
  void* split = split_in(ws, ws_bytes, group_U_bytes(M, G, r));
  return run_bwd_split(stream, r > 0, [&](cudaStream_t main, const GradSide* side) {
    return group_bwd_split(w, G, N_g, X, dY_cat, M, A_cat, B_cat, r, alpha, T_cat, dX, dA_cat, dB_cat, accumulate, ws,
                           ws_bytes, main, side, split, split ? split_scratch_bytes() : 0);
  });
}

// ------------------------------------------------ allocation-free forward
// Some callers cannot hand libsl a workspace: they run under a memory
// manager that owns all device memory (a framework caching allocator with a
// hard budget, an embedding application that forbids cudaMalloc because it
// synchronises the device and fragments its pool).  For them the forward
// keeps its only scratch -- the K-split partial sums of T = X A^T -- in this
// file-scope device array, so the call allocates nothing.  Every device that
// loads libsl holds the array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, looked up once per device (with that device
// current): in host code the symbol is only a host-side stand-in.
static sl_status noalloc_scratch_ptr(void** out) {
  static std::mutex mu;
  static void* ptrs[64] = {nullptr};
  int dev = 0;
  SL_CHECK_CUDA(cudaGetDevice(&dev));
  SL_REQUIRE(dev >= 0 && dev < 64, "sl_lora_linear_fwd_noalloc: device index out of range");
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_error(e, "sl_lora_linear_fwd_noalloc: cudaGetSymbolAddress");
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return SL_OK;
}

// Bytes of scratch the forward needs: one fp32 [M, r] partial per 512-column
// split of K (none when K fits one split).
static size_t noalloc_need(int64_t M, int64_t K, int r) {
  const int splits = down_splits(K);
  return splits > 1 ? static_cast<size_t>(splits) * M * r * 4 : 0;
}

sl_status linear_fwd_noalloc(const sl_weight* w, const void* X, int64_t M, const void* A, const void* B, int r,
                             float alpha, void* Y, void* T_save, cudaStream_t stream) {
  sl_status st = check_weight(w);
  if (st != SL_OK) return st;
  SL_REQUIRE(X && Y && M > 0, "sl_lora_linear_fwd_noalloc: null X/Y or M <= 0");
  const bool lora = r > 0 && A && B;
  SL_REQUIRE(!lora || (r % 8 == 0 && r <= 32 && T_save),
             "sl_lora_linear_fwd_noalloc: need r % 8 == 0, r <= 32, T_save");
  SL_REQUIRE(M < (1LL << 31), "sl_lora_linear_fwd_noalloc: M too large");
  st = check_rows(w, M, "sl_lora_linear_fwd_noalloc");
  if (st != SL_OK) return st;
  // The rank-r pass reads X and A with 16-byte cp.async loads and the GEMM
  // moves X, B, T_save and Y by TMA: check every base up front, so that a
  // misaligned pointer is an error status before anything is launched.
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  SL_REQUIRE(al16(X) && al16(Y) && (w->K * 2) % 16 == 0 && (w->N * 2) % 16 == 0,
             "sl_lora_linear_fwd_noalloc: X and Y must be 16-byte aligned");
  SL_REQUIRE(!lora || (al16(A) && al16(B) && al16(T_save)),
             "sl_lora_linear_fwd_noalloc: A, B and T_save must be 16-byte aligned");
  const size_t need = lora ? noalloc_need(M, w->K, r) : 0;
  if (need > kNoAllocScratchBytes)
    return set_error(SL_ERR_INVALID, "sl_lora_linear_fwd_noalloc: needs " + std::to_string(need) +
                                         " bytes of scratch (ceil(K/512) * M * r * 4), above the fixed " +
                                         std::to_string(kNoAllocScratchBytes) +
                                         "-byte maximum; use sl_lora_linear_fwd with a workspace");
  void* scratch = nullptr;
  st = noalloc_scratch_ptr(&scratch);
  if (st != SL_OK) return st;
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  if (lora) {
    // Every partial element that the split sum reads is written first by
    // this call, so the array needs no clearing between calls.
    st = lora_down(static_cast<const uint16_t*>(X), M, static_cast<int>(w->K), static_cast<const uint16_t*>(A), 0, r,
                   static_cast<float*>(T_save), static_cast<float*>(scratch), stream);
    if (st != SL_OK) return st;
  }
  GemmLaunch g{};
  bind_weight(g, w);
  g.bmn = 0;
  g.epi = kEpiStoreBF16;
  g.A = X;
  g.lda = w->K;
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

}  // namespace sl

using namespace sl;

extern "C" sl_status sl_lora_linear_fwd(const sl_weight* w, const void* X, int64_t M, const void* A, const void* B,
                                        int32_t r, float alpha, void* Y, void* T_save, void* ws, size_t ws_bytes,
                                        cudaStream_t stream) {
  return linear_fwd(w, X, M, A, B, r, alpha, Y, T_save, ws, ws_bytes, stream);
}

extern "C" sl_status sl_lora_linear_bwd(const sl_weight* w, const void* X, const void* dY, int64_t M, const void* A,
                                        const void* B, int32_t r, float alpha, const void* T_save, void* dX,
                                        float* dA, float* dB, int32_t accumulate, void* ws, size_t ws_bytes,
                                        cudaStream_t stream) {
  return linear_bwd(w, X, dY, M, A, B, r, alpha, T_save, dX, dA, dB, accumulate, ws, ws_bytes, stream);
}

extern "C" size_t sl_lora_linear_workspace_size(int64_t M, int64_t N, int64_t K, int32_t r) {
  return linear_ws_bytes(M, N, K, r);
}

extern "C" sl_status sl_lora_group_fwd(const sl_weight* w_cat, int32_t G, const int64_t* N_g, const void* X, int64_t M,
                                       const void* A_cat, const void* B_cat, int32_t r, float alpha, void* Y_cat,
                                       void* T_cat, cudaStream_t stream) {
  return group_fwd(w_cat, G, N_g, X, M, A_cat, B_cat, r, alpha, Y_cat, T_cat, stream);
}

extern "C" sl_status sl_lora_group_bwd(const sl_weight* w_cat, int32_t G, const int64_t* N_g, const void* X,
                                       const void* dY_cat, int64_t M, const void* A_cat, const void* B_cat, int32_t r,
                                       float alpha, const void* T_cat, void* dX, float* dA_cat, float* dB_cat,
                                       int32_t accumulate, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return group_bwd(w_cat, G, N_g, X, dY_cat, M, A_cat, B_cat, r, alpha, T_cat, dX, dA_cat, dB_cat, accumulate, ws,
                   ws_bytes, stream);
}

extern "C" size_t sl_lora_group_workspace_size(int64_t M, int32_t G, int32_t r) { return group_ws_bytes(M, G, r); }

extern "C" sl_status sl_lora_linear_fwd_noalloc(const sl_weight* w, const void* X, int64_t M, const void* A,
                                                const void* B, int32_t r, float alpha, void* Y, void* T_save,
                                                cudaStream_t stream) {
  return linear_fwd_noalloc(w, X, M, A, B, r, alpha, Y, T_save, stream);
}
