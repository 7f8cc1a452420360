// K0 / K1: NF4 quantise and dequantise (blocksize 64, fp32 absmax).
//
// "Exact Layer Streaming ..." (abstract) keeps the frozen base in NF4; the
// code of an element is the nearest NF4 level to x = w / absmax (IEEE fp32
// division), ties to the lower level; absmax == 0 gives the zero level.
// Both kernels are HBM-bound streams: one warp per 64-element block for the
// quantiser (coalesced 128-byte reads, a shuffle max), one thread per 8
// elements for the dequantiser.
#include <cstring>

#include "common.cuh"
#include "nf4.cuh"

namespace sl {


__device__ __forceinline__ uint32_t nf4_code_of(float x) {
  uint32_t c = 0;
#pragma unroll
  for (int j = 0; j < 15; ++j) c += (x >= __uint_as_float(d_nf4_thresh_bits[j])) ? 1u : 0u;
  return c;
}

template <bool kF32>
__global__ void __launch_bounds__(256) nf4_quantize_kernel(const void* __restrict__ W, int64_t nblocks,
                                                           uint8_t* __restrict__ codes,
                                                           float* __restrict__ absmax, int* __restrict__ bad) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t b = warp; b < nblocks; b += nwarps) {
    float w0, w1;
    if (kF32) {
      const float2 v = reinterpret_cast<const float2*>(W)[b * 32 + lane];
      w0 = v.x;
      w1 = v.y;
    } else {
      const uint32_t v = reinterpret_cast<const uint32_t*>(W)[b * 32 + lane];
      w0 = bf16_lo(v);
      w1 = bf16_hi(v);
    }
    const bool nonfinite = !isfinite(w0) || !isfinite(w1);
    float a = fmaxf(fabsf(w0), fabsf(w1));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (__any_sync(0xffffffffu, nonfinite) && lane == 0) atomicOr(bad, 1);
    uint32_t c0 = 7, c1 = 7;
    if (a > 0.0f) {
      c0 = nf4_code_of(__fdiv_rn(w0, a));
      c1 = nf4_code_of(__fdiv_rn(w1, a));
    }
    codes[b * 32 + lane] = static_cast<uint8_t>((c0 << 4) | c1);
    if (lane == 0) absmax[b] = a;
  }
}

// The double-quantised absmax of a weight (see sl_weight, SL_WEIGHT_NF4_DQ).
struct DqAbsmax {
  const int8_t* q;
  int64_t q_ld;
  const float* a2;
  int64_t a2_ld;
  int64_t col0;
  int64_t blocks_per_row;  // K / 64
};

// absmax of 64-block `blk` (row-major block index n * K/64 + j): fma(s, q, c)
__device__ __forceinline__ float dq_absmax(const DqAbsmax& d, int64_t blk) {
  const int64_t n = blk / d.blocks_per_row, j = blk % d.blocks_per_row;
  const int64_t col = d.col0 + n;
  const float q = static_cast<float>(d.q[j * d.q_ld + col]);
  const float* cs = d.a2 + j * d.a2_ld + 2 * (col / 256);
  return fmaf(cs[1], q, cs[0]);
}

template <bool kF32, bool kDQ>
__global__ void __launch_bounds__(256) nf4_dequantize_kernel(const uint32_t* __restrict__ codes,
                                                             const float* __restrict__ absmax, DqAbsmax dq,
                                                             int64_t nwords, void* __restrict__ out) {
  __shared__ float tab[16];
  if (threadIdx.x < 16) tab[threadIdx.x] = __uint_as_float(d_nf4_level_bits[threadIdx.x]);
  __syncthreads();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nwords; i += stride) {
    const uint32_t w = codes[i];
    const float a = kDQ ? dq_absmax(dq, i >> 3) : absmax[i >> 3];  // 8 words (64 elements) per block
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t byte = (w >> (8 * j)) & 0xFFu;
      v[2 * j] = __fmul_rn(tab[byte >> 4], a);
      v[2 * j + 1] = __fmul_rn(tab[byte & 15u], a);
    }
    if (kF32) {
      float4* o = reinterpret_cast<float4*>(out) + 2 * i;
      o[0] = make_float4(v[0], v[1], v[2], v[3]);
      o[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      uint4 p;
      p.x = pack_bf16x2(v[0], v[1]);
      p.y = pack_bf16x2(v[2], v[3]);
      p.z = pack_bf16x2(v[4], v[5]);
      p.w = pack_bf16x2(v[6], v[7]);
      reinterpret_cast<uint4*>(out)[i] = p;
    }
  }
}

// Double quantisation of the absmax: one thread per (64-block column j,
// 256 consecutive rows n).  Every step is the stated IEEE operation, so the
// result is bit-identical to its definition (float64 sum in ascending n).
__global__ void nf4_double_quantize_kernel(const float* __restrict__ absmax, int64_t N, int64_t nbj,
                                           int8_t* __restrict__ q, int64_t q_ld, float* __restrict__ a2,
                                           int64_t a2_ld) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nb = N / 256;
  if (t >= nbj * nb) return;
  const int64_t j = t / nb, b = t % nb;
  const float* src = absmax + (b * 256) * nbj + j;  // absmax[n][j] for n = 256 b ..
  double sum = 0.0;
  for (int i = 0; i < 256; ++i) sum += static_cast<double>(src[i * nbj]);
  const float c = __double2float_rn(sum / 256.0);
  float m = 0.0f;
  for (int i = 0; i < 256; ++i) m = fmaxf(m, fabsf(__fsub_rn(src[i * nbj], c)));
  const float sc = __fdiv_rn(m, 127.0f);
  int8_t* qo = q + j * q_ld + b * 256;
  for (int i = 0; i < 256; ++i) {
    float v = 0.0f;
    if (sc > 0.0f) v = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(src[i * nbj], c), sc)), -127.0f), 127.0f);
    qo[i] = static_cast<int8_t>(v);
  }
  a2[j * a2_ld + 2 * b] = c;
  a2[j * a2_ld + 2 * b + 1] = sc;
}

static int grid_for(int64_t items, int per_block) {
  int64_t g = ceil_div(items, per_block);
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  return static_cast<int>(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace sl

using namespace sl;

extern "C" sl_status sl_nf4_quantize(const void* W, int32_t dtype, int64_t N, int64_t K, uint8_t* codes,
                                     float* absmax, cudaStream_t stream) {
  SL_REQUIRE(W && codes && absmax, "sl_nf4_quantize: null pointer");
  SL_REQUIRE(N > 0 && K > 0 && K % 64 == 0, "sl_nf4_quantize: need N > 0 and K a positive multiple of 64");
  SL_REQUIRE(dtype == SL_DTYPE_BF16 || dtype == SL_DTYPE_F32, "sl_nf4_quantize: dtype must be BF16 or F32");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(W) & 15) == 0 && (reinterpret_cast<uintptr_t>(codes) & 15) == 0 &&
                 (reinterpret_cast<uintptr_t>(absmax) & 15) == 0,
             "sl_nf4_quantize: pointers must be 16-byte aligned");
  sl_status st = SL_OK;
  int* word = device_error_word();
  if (!word) return SL_ERR_CUDA;
  // word + 1 is reserved for the timeout probe; use a private flag instead.
  static int* flags[64] = {nullptr};
  int dev = 0;
  SL_CHECK_CUDA(cudaGetDevice(&dev));
  SL_REQUIRE(dev >= 0 && dev < 64, "sl_nf4_quantize: device index out of range");
  if (!flags[dev]) SL_CHECK_CUDA(cudaMalloc(&flags[dev], sizeof(int)));
  int* bad = flags[dev];
  SL_CHECK_CUDA(cudaMemsetAsync(bad, 0, sizeof(int), stream));
  const int64_t nblocks = N * K / 64;
  const int grid = grid_for(nblocks, 8);
  if (dtype == SL_DTYPE_F32)
    nf4_quantize_kernel<true><<<grid, 256, 0, stream>>>(W, nblocks, codes, absmax, bad);
  else
    nf4_quantize_kernel<false><<<grid, 256, 0, stream>>>(W, nblocks, codes, absmax, bad);
  st = check_launch("nf4_quantize_kernel");
  if (st != SL_OK) return st;
  int h = 0;
  SL_CHECK_CUDA(cudaMemcpyAsync(&h, bad, sizeof(int), cudaMemcpyDeviceToHost, stream));
  SL_CHECK_CUDA(cudaStreamSynchronize(stream));
  if (h) return set_error(SL_ERR_NONFINITE, "sl_nf4_quantize: non-finite weight");
  return SL_OK;
}

extern "C" sl_status sl_nf4_dequantize(const uint8_t* codes, const float* absmax, int64_t N, int64_t K,
                                       int32_t out_dtype, void* out, cudaStream_t stream) {
  SL_REQUIRE(codes && absmax && out, "sl_nf4_dequantize: null pointer");
  SL_REQUIRE(N > 0 && K > 0 && K % 64 == 0, "sl_nf4_dequantize: need K a positive multiple of 64");
  SL_REQUIRE(out_dtype == SL_DTYPE_BF16 || out_dtype == SL_DTYPE_F32, "sl_nf4_dequantize: bad out_dtype");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(codes) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0 &&
                 (reinterpret_cast<uintptr_t>(absmax) & 3) == 0,
             "sl_nf4_dequantize: misaligned pointer");
  const int64_t nwords = N * K / 8;
  const int grid = grid_for(nwords, 256);
  const DqAbsmax none{};
  if (out_dtype == SL_DTYPE_F32)
    nf4_dequantize_kernel<true, false><<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(codes), absmax,
                                                                 none, nwords, out);
  else
    nf4_dequantize_kernel<false, false><<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(codes),
                                                                  absmax, none, nwords, out);
  return check_launch("nf4_dequantize_kernel");
}

extern "C" sl_status sl_nf4_double_quantize(const float* absmax, int64_t N, int64_t K, int8_t* qabsmax,
                                            int64_t qabsmax_ld, float* absmax2, int64_t absmax2_ld,
                                            cudaStream_t stream) {
  SL_REQUIRE(absmax && qabsmax && absmax2, "sl_nf4_double_quantize: null pointer");
  SL_REQUIRE(N > 0 && N % 256 == 0 && K > 0 && K % 64 == 0,
             "sl_nf4_double_quantize: need N a positive multiple of 256 and K of 64");
  SL_REQUIRE(qabsmax_ld >= N && absmax2_ld >= 2 * (N / 256), "sl_nf4_double_quantize: output row stride too small");
  const int64_t nbj = K / 64, tasks = nbj * (N / 256);
  nf4_double_quantize_kernel<<<static_cast<unsigned>(ceil_div(tasks, 128)), 128, 0, stream>>>(
      absmax, N, nbj, qabsmax, qabsmax_ld, absmax2, absmax2_ld);
  return check_launch("nf4_double_quantize_kernel");
}

extern "C" sl_status sl_weight_dequantize(const sl_weight* w, int32_t out_dtype, void* out, cudaStream_t stream) {
  SL_REQUIRE(w && out, "sl_weight_dequantize: null pointer");
  if (w->kind == SL_WEIGHT_NF4) return sl_nf4_dequantize(w->codes, w->absmax, w->N, w->K, out_dtype, out, stream);
  SL_REQUIRE(w->kind == SL_WEIGHT_NF4_DQ, "sl_weight_dequantize: NF4 or NF4_DQ weights only");
  SL_REQUIRE(w->codes && w->qabsmax && w->absmax2, "sl_weight_dequantize: null pointer");
  SL_REQUIRE(w->N > 0 && w->K > 0 && w->K % 64 == 0 && w->dq_col0 >= 0 && w->dq_col0 % 256 == 0,
             "sl_weight_dequantize: bad shape or column offset");
  SL_REQUIRE(out_dtype == SL_DTYPE_BF16 || out_dtype == SL_DTYPE_F32, "sl_weight_dequantize: bad out_dtype");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(w->codes) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0,
             "sl_weight_dequantize: misaligned pointer");
  const DqAbsmax dq{w->qabsmax, w->qabsmax_ld, w->absmax2, w->absmax2_ld, w->dq_col0, w->K / 64};
  const int64_t nwords = w->N * w->K / 8;
  const int grid = grid_for(nwords, 256);
  if (out_dtype == SL_DTYPE_F32)
    nf4_dequantize_kernel<true, true><<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(w->codes), nullptr,
                                                                dq, nwords, out);
  else
    nf4_dequantize_kernel<false, true><<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(w->codes),
                                                                 nullptr, dq, nwords, out);
  return check_launch("nf4_dequantize_kernel");
}
