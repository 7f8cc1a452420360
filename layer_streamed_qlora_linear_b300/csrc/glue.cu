// K8: the elementwise / row-wise parts of the synthetic decoder layer
// (steps a5 and a7).  The pages stream decoder layers ("Soup CLI ...", "How
// Layer Streaming Works") without stating their internals; the layer here is
// the token-local pre-norm layer of the library's design:
//   x1 = RMS(h); a = q*rep(k) + rep(v); h1 = h + o; x2 = RMS(h1);
//   m = SiLU(g)*u; h2 = h1 + d          (RMS(h) = h / sqrt(mean(h^2) + 1e-5))
// fp32 arithmetic; the residual stream and its gradient are fp32, every GEMM
// input/output is bf16 (rounded once).  Row reductions use a fixed-order
// block reduction, so results are bitwise reproducible.
// All kernels are HBM-bound streams over [M, D] / [M, F] tensors.
#include "common.cuh"
#include "glue.cuh"

namespace sl {

constexpr int kRowThreads = 256;
constexpr float kRmsEps = 1e-5f;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ void load8_bf16(const uint16_t* p, float (&f)[8]) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = bf16_lo(w[e]);
    f[2 * e + 1] = bf16_hi(w[e]);
  }
}

__device__ __forceinline__ void store8_bf16(uint16_t* p, const float (&f)[8]) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  *reinterpret_cast<uint4*>(p) = v;
}

__device__ __forceinline__ void load8_f32(const float* p, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void store8_f32(float* p, const float (&f)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// hs = h (+ add);  x = bf16(hs * rstd (* w));  rstd = 1 / sqrt(mean(hs^2) + eps)
// h_out receives hs when `add` is given (the residual update h1 = h + o);
// w (nullable) is the norm's fp32 weight [D].
__global__ void __launch_bounds__(kRowThreads) rms_fwd_kernel(const float* __restrict__ h,
                                                              const uint16_t* __restrict__ add,
                                                              float* __restrict__ h_out, uint16_t* __restrict__ x,
                                                              float* __restrict__ rstd, const float* __restrict__ w,
                                                              int D) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kRowThreads / 32];
  const int64_t row = blockIdx.x;
  const float* hr = h + row * D;
  float ss = 0.0f;
  for (int i = threadIdx.x * 8; i < D; i += kRowThreads * 8) {
    float f[8];
    load8_f32(hr + i, f);
    if (add) {
      float a[8];
      load8_bf16(add + row * D + i, a);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] += a[e];
      store8_f32(h_out + row * D + i, f);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
  }
  const float tot = block_sum(ss, red);
  const float r = 1.0f / sqrtf(tot / static_cast<float>(D) + kRmsEps);
  if (threadIdx.x == 0) rstd[row] = r;
  const float* src = add ? h_out + row * D : hr;
  for (int i = threadIdx.x * 8; i < D; i += kRowThreads * 8) {
    float f[8];
    load8_f32(src + i, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] *= r;
    if (w) {
      float fw[8];
      load8_f32(w + i, fw);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] *= fw[e];
    }
    store8_bf16(x + row * D + i, f);
  }
}

// a[m, j] = bf16(q[m, j] * k[m, kv(j)] + v[m, kv(j)]); kv(j): head j/128 reads kv head (j/128)/g.
__global__ void mix_fwd_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                               const uint16_t* __restrict__ v, uint16_t* __restrict__ a, int64_t M, int D,
                               int Dkv, int64_t ldq, int64_t ldkv) {
  pdl_trigger();
  pdl_wait();
  const int g = D / Dkv;
  const int64_t n8 = M * D / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    const int64_t e0 = t * 8;
    const int64_t m = e0 / D;
    const int j = static_cast<int>(e0 % D);
    const int c = (j / 128 / g) * 128 + (j % 128);
    float fq[8], fk[8], fv[8], fa[8];
    load8_bf16(q + m * ldq + j, fq);
    load8_bf16(k + m * ldkv + c, fk);
    load8_bf16(v + m * ldkv + c, fv);
#pragma unroll
    for (int e = 0; e < 8; ++e) fa[e] = fmaf(fq[e], fk[e], fv[e]);
    store8_bf16(a + e0, fa);
  }
}

// Logistic function with the fast exponential and division (relative error
// ~1e-6, far below the bf16 rounding of every result that uses it); the
// fused SwiGLU rank-r kernels (skinny.cu) compute it the same way.
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// m = bf16(SiLU(g) * u)
// g, u: rows of F elements at row stride ld; m dense [M, F].
__global__ void swiglu_fwd_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ u,
                                  uint16_t* __restrict__ m, int64_t M, int F, int64_t ld) {
  pdl_trigger();
  pdl_wait();
  const int64_t n8 = M * F / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    const int64_t row = t * 8 / F, off = row * ld + t * 8 % F;
    float fg[8], fu[8], fm[8];
    load8_bf16(g + off, fg);
    load8_bf16(u + off, fu);
#pragma unroll
    for (int e = 0; e < 8; ++e) fm[e] = fg[e] * sigmoidf_(fg[e]) * fu[e];
    store8_bf16(m + t * 8, fm);
  }
}

// out = h + add (fp32 residual update), optional bf16 copy of nothing.
__global__ void resid_add_kernel(const float* __restrict__ h, const uint16_t* __restrict__ add,
                                 float* __restrict__ out, int64_t n) {
  pdl_trigger();
  pdl_wait();
  const int64_t n8 = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    float f[8], a[8];
    load8_f32(h + t * 8, f);
    load8_bf16(add + t * 8, a);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] += a[e];
    store8_f32(out + t * 8, f);
  }
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ x, uint16_t* __restrict__ y, int64_t n) {
  pdl_trigger();
  pdl_wait();
  const int64_t n8 = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    float f[8];
    load8_f32(x + t * 8, f);
    store8_bf16(y + t * 8, f);
  }
}

// dg = bf16(dm * u * s * (1 + g (1 - s))), du = bf16(dm * g * s), s = sigmoid(g)
// dm dense [M, F]; g, u, dg, du: rows of F elements at row stride ld.
__global__ void swiglu_bwd_kernel(const uint16_t* __restrict__ dm, const uint16_t* __restrict__ g,
                                  const uint16_t* __restrict__ u, uint16_t* __restrict__ dg,
                                  uint16_t* __restrict__ du, int64_t M, int F, int64_t ld) {
  pdl_trigger();
  pdl_wait();
  const int64_t n8 = M * F / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    const int64_t row = t * 8 / F, off = row * ld + t * 8 % F;
    float fdm[8], fg[8], fu[8], odg[8], odu[8];
    load8_bf16(dm + t * 8, fdm);
    load8_bf16(g + off, fg);
    load8_bf16(u + off, fu);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float s = sigmoidf_(fg[e]);
      odg[e] = fdm[e] * fu[e] * s * (1.0f + fg[e] * (1.0f - s));
      odu[e] = fdm[e] * fg[e] * s;
    }
    store8_bf16(dg + off, odg);
    store8_bf16(du + off, odu);
  }
}

// Backward of hs -> RMS(hs) * w with a residual pass-through:
//   dx = w * (the fp32 dxf, or the sum of up to three bf16 GEMM outputs);
//   y = h * rstd;  dh_out = dh_in + rstd * (dx - y * sum(dx * y) / D);
//   dh_in and w nullable (no residual, no weight); optional bf16 copy.
__global__ void __launch_bounds__(kRowThreads) rms_bwd_kernel(
    const float* __restrict__ dh_in, const uint16_t* __restrict__ dx0, const uint16_t* __restrict__ dx1,
    const uint16_t* __restrict__ dx2, const float* __restrict__ dxf, const float* __restrict__ h,
    const float* __restrict__ rstd, const float* __restrict__ w, float* __restrict__ dh_out,
    uint16_t* __restrict__ dh_bf16, int D) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kRowThreads / 32];
  const int64_t row = blockIdx.x;
  const float r = rstd[row];
  auto dx_at = [&](int i, float (&f)[8]) {
    if (dxf) {
      load8_f32(dxf + row * D + i, f);
    } else {
      load8_bf16(dx0 + row * D + i, f);
    }
    if (dx1) {
      float t[8];
      load8_bf16(dx1 + row * D + i, t);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] += t[e];
    }
    if (dx2) {
      float t[8];
      load8_bf16(dx2 + row * D + i, t);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] += t[e];
    }
    if (w) {
      float fw[8];
      load8_f32(w + i, fw);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] *= fw[e];
    }
  };
  float dot = 0.0f;
  for (int i = threadIdx.x * 8; i < D; i += kRowThreads * 8) {
    float fx[8], fh[8];
    dx_at(i, fx);
    load8_f32(h + row * D + i, fh);
#pragma unroll
    for (int e = 0; e < 8; ++e) dot = fmaf(fx[e], fh[e] * r, dot);
  }
  const float c = block_sum(dot, red) / static_cast<float>(D);
  for (int i = threadIdx.x * 8; i < D; i += kRowThreads * 8) {
    float fx[8], fh[8], fd[8];
    dx_at(i, fx);
    load8_f32(h + row * D + i, fh);
    if (dh_in) {
      load8_f32(dh_in + row * D + i, fd);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) fd[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) fd[e] += r * (fx[e] - fh[e] * r * c);
    store8_f32(dh_out + row * D + i, fd);
    if (dh_bf16) store8_bf16(dh_bf16 + row * D + i, fd);
  }
}

// dq = bf16(da * rep(k)); dk = bf16(sum over the g heads of da * q); dv = bf16(sum of da)
// da dense [M, D]; q, dq at row stride ldq; k, dk, dv at row stride ldkv.
__global__ void mix_bwd_kernel(const uint16_t* __restrict__ da, const uint16_t* __restrict__ q,
                               const uint16_t* __restrict__ k, uint16_t* __restrict__ dq,
                               uint16_t* __restrict__ dk, uint16_t* __restrict__ dv, int64_t M, int D, int Dkv,
                               int64_t ldq, int64_t ldkv) {
  pdl_trigger();
  pdl_wait();
  const int g = D / Dkv;
  const int64_t n8 = M * Dkv / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    const int64_t e0 = t * 8;
    const int64_t m = e0 / Dkv;
    const int c = static_cast<int>(e0 % Dkv);
    const int kvh = c / 128, e = c % 128;
    float fk[8], sk[8], sv[8];
    load8_bf16(k + m * ldkv + c, fk);
#pragma unroll
    for (int i = 0; i < 8; ++i) sk[i] = sv[i] = 0.0f;
    for (int hh = 0; hh < g; ++hh) {
      const int col = (kvh * g + hh) * 128 + e;
      float fa[8], fq[8], fdq[8];
      load8_bf16(da + m * D + col, fa);
      load8_bf16(q + m * ldq + col, fq);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sk[i] = fmaf(fa[i], fq[i], sk[i]);
        sv[i] += fa[i];
        fdq[i] = fa[i] * fk[i];
      }
      store8_bf16(dq + m * ldq + col, fdq);
    }
    store8_bf16(dk + m * ldkv + c, sk);
    store8_bf16(dv + m * ldkv + c, sv);
  }
}

// h0[m] = fp32(embed[tokens[m]]) (8 elements per thread); a token outside
// [0, V) gives a zero row and SL_ERR_INVALID in the device error word.
__global__ void embed_kernel(const int32_t* __restrict__ tokens, const uint16_t* __restrict__ embed, int64_t V,
                             float* __restrict__ h0, int64_t M, int D, int* err) {
  pdl_trigger();
  pdl_wait();
  const int64_t n8 = M * D / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n8; t += stride) {
    const int64_t m = t * 8 / D;
    const int j = static_cast<int>(t * 8 % D);
    const int64_t tok = tokens[m];
    float f[8];
    if (tok >= 0 && tok < V) {
      load8_bf16(embed + tok * D + j, f);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = 0.0f;
      if (j == 0) report_device_error(err, SL_ERR_INVALID);
    }
    store8_f32(h0 + m * D + j, f);
  }
}

static int ew_grid(int64_t n8) {
  int64_t g = ceil_div(n8, 256);
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  return static_cast<int>(g < 1 ? 1 : (g > cap ? cap : g));
}

sl_status glue_rms_fwd(const float* h, const uint16_t* add, float* h_out, uint16_t* x, float* rstd,
                       const float* w, int64_t M, int D, cudaStream_t s) {
  return launch_pdl("rms_fwd_kernel", rms_fwd_kernel, dim3(static_cast<unsigned>(M)), dim3(kRowThreads), 0, s, h,
                    add, h_out, x, rstd, w, D);
}
sl_status glue_mix_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* a, int64_t M, int D,
                       int Dkv, int64_t ldq, int64_t ldkv, cudaStream_t s) {
  return launch_pdl("mix_fwd_kernel", mix_fwd_kernel, dim3(ew_grid(M * D / 8)), dim3(256), 0, s, q, k, v, a, M, D,
                    Dkv, ldq, ldkv);
}
sl_status glue_swiglu_fwd(const uint16_t* g, const uint16_t* u, uint16_t* m, int64_t M, int F, int64_t ld,
                          cudaStream_t s) {
  return launch_pdl("swiglu_fwd_kernel", swiglu_fwd_kernel, dim3(ew_grid(M * F / 8)), dim3(256), 0, s, g, u, m, M, F,
                    ld);
}
sl_status glue_resid_add(const float* h, const uint16_t* add, float* out, int64_t n, cudaStream_t s) {
  return launch_pdl("resid_add_kernel", resid_add_kernel, dim3(ew_grid(n / 8)), dim3(256), 0, s, h, add, out, n);
}
sl_status glue_to_bf16(const float* x, uint16_t* y, int64_t n, cudaStream_t s) {
  return launch_pdl("f32_to_bf16_kernel", f32_to_bf16_kernel, dim3(ew_grid(n / 8)), dim3(256), 0, s, x, y, n);
}
sl_status glue_swiglu_bwd(const uint16_t* dm, const uint16_t* g, const uint16_t* u, uint16_t* dg, uint16_t* du,
                          int64_t M, int F, int64_t ld, cudaStream_t s) {
  return launch_pdl("swiglu_bwd_kernel", swiglu_bwd_kernel, dim3(ew_grid(M * F / 8)), dim3(256), 0, s, dm, g, u, dg,
                    du, M, F, ld);
}
sl_status glue_rms_bwd(const float* dh_in, const uint16_t* dx0, const uint16_t* dx1, const uint16_t* dx2,
                       const float* dxf, const float* h, const float* rstd, const float* w, float* dh_out,
                       uint16_t* dh_bf16, int64_t M, int D, cudaStream_t s) {
  return launch_pdl("rms_bwd_kernel", rms_bwd_kernel, dim3(static_cast<unsigned>(M)), dim3(kRowThreads), 0, s, dh_in,
                    dx0, dx1, dx2, dxf, h, rstd, w, dh_out, dh_bf16, D);
}
sl_status glue_mix_bwd(const uint16_t* da, const uint16_t* q, const uint16_t* k, uint16_t* dq, uint16_t* dk,
                       uint16_t* dv, int64_t M, int D, int Dkv, int64_t ldq, int64_t ldkv, cudaStream_t s) {
  return launch_pdl("mix_bwd_kernel", mix_bwd_kernel, dim3(ew_grid(M * Dkv / 8)), dim3(256), 0, s, da, q, k, dq, dk,
                    dv, M, D, Dkv, ldq, ldkv);
}

}  // namespace sl

namespace sl {
sl_status glue_embed(const int32_t* tokens, const uint16_t* embed, int64_t V, float* h0, int64_t M, int D, int* err,
                     cudaStream_t s) {
  return launch_pdl("embed_kernel", embed_kernel, dim3(ew_grid(M * D / 8)), dim3(256), 0, s, tokens, embed, V, h0, M,
                    D, err);
}
}  // namespace sl
