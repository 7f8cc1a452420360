// Step a8: cross-entropy over the LM head, loss and dH, without the logits.
//
// "Exact Layer Streaming ..." (abstract) measures the cross-entropy logits
// term at 14 bytes per logit element; here no [M, V] tensor exists, and the
// logits are computed once (online softmax over vocab chunks):
//   per chunk c of chunk_V rows of W
//     logits  one tcgen05 GEMM Z_c = H W_c^T whose epilogue writes, per row
//             and 128-column half tile h, its max m_h, P = bf16(exp(z - m_h))
//             into a [M, chunk_V] scratch and s_h = sum exp(z - m_h), and
//             gathers the label's logit;
//     rows    per row: the chunk's max and sum from its half tiles (fixed
//             order), the running max m and sum S updated, P rescaled in
//             place to exp(z - m_new), and alpha = exp(m_old - m_new);
//     dH      acc = alpha * acc + P W_c (fp32, tcgen05 with an MN-major W);
//   last      lse = m + log S, loss = mean over valid rows of lse - z_label
//             (fixed order), dH = acc / (S N_valid) - W[label] / N_valid
//             (the one-hot part exact in fp32, ignored rows 0).
// Two passes over the head instead of three; extra device bytes: the chunk
// scratch plus O(M * chunk_V / 128) partials.
#include "common.cuh"
#include "gemm.cuh"

namespace sl {

namespace {

struct CEPlan {
  size_t part_max, part_sum, label_logit, run_max, run_sum, alpha, lse, term, scale, P, split, split_bytes, total;
  int halves;  // 128-column half tiles of a chunk
};

CEPlan ce_plan(int64_t M, int64_t D, int64_t V, int64_t chunk_V) {
  (void)D;
  (void)V;
  CEPlan p{};
  size_t off = 0;
  auto take = [&](size_t b) {
    const size_t o = off;
    off = align_up(off + b, 256);
    return o;
  };
  p.halves = static_cast<int>(ceil_div(chunk_V, kBN)) * 2;
  p.part_max = take(static_cast<size_t>(M) * p.halves * 4);
  p.part_sum = take(static_cast<size_t>(M) * p.halves * 4);
  p.label_logit = take(M * 4);
  p.run_max = take(M * 4);
  p.run_sum = take(M * 4);
  p.alpha = take(M * 4);
  p.lse = take(M * 4);
  p.term = take(M * 4);
  p.scale = take(M * 4);
  p.P = take(static_cast<size_t>(M) * chunk_V * 2);
  // the pair GEMMs (M > 128) split a last partial wave along K in this scratch
  p.split_bytes = M > 128 ? split_scratch_bytes() : 0;
  p.split = take(p.split_bytes);
  p.total = off;
  return p;
}

// One warp per row, after a chunk's logits GEMM: the chunk's max and sum from
// its half-tile partials (fixed order), the running (max, sum) updated, the
// row's P rescaled in place from exp(z - m_h) to exp(z - m_new), and
// alpha = exp(m_old - m_new) for the dH accumulator.  first: no earlier chunk.
// halves: this chunk's half tiles; part_ld: the partials' row stride.
__global__ void ce_chunk_kernel(const float* __restrict__ pmax, const float* __restrict__ psum, int halves,
                                int part_ld, int ncols, int64_t M, uint16_t* __restrict__ P, int ldp,
                                float* __restrict__ run_max, float* __restrict__ run_sum, float* __restrict__ alpha,
                                int first) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const float* pm = pmax + row * part_ld;
  const float* ps = psum + row * part_ld;
  // chunk max, then chunk sum in half-tile order (lane 0 sums: fixed order)
  float cm = -INFINITY;
  for (int h = lane; h < halves; h += 32) cm = fmaxf(cm, pm[h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
  const float m_old = first ? -INFINITY : run_max[row];
  const float m_new = fmaxf(m_old, cm);
  if (lane == 0) {
    float cs = 0.0f;
    for (int h = 0; h < halves; ++h)
      if (pm[h] != -INFINITY) cs += ps[h] * __expf(pm[h] - m_new);
    const float a = (m_old == -INFINITY) ? 0.0f : __expf(m_old - m_new);
    run_sum[row] = (first ? 0.0f : run_sum[row] * a) + cs;
    run_max[row] = m_new;
    alpha[row] = a;
  }
  // P[row, h * 128 .. +128) *= exp(m_h - m_new): lanes take 8-element chunks
  uint16_t* pr = P + row * static_cast<int64_t>(ldp);
  for (int c = lane * 8; c < ncols; c += 32 * 8) {
    const float f = (pm[c / 128] == -INFINITY) ? 0.0f : __expf(pm[c / 128] - m_new);
    uint4 v = *reinterpret_cast<const uint4*>(pr + c);
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = pack_bf16x2(bf16_lo(w[k]) * f, bf16_hi(w[k]) * f);
    *reinterpret_cast<uint4*>(pr + c) = v;
  }
}

// One warp per row: lse = m + log S and the row's loss term lse - z_label
// (0 for ignored rows).  Out-of-range labels are reported through the error
// word and treated as ignored.
__global__ void ce_row_kernel(const float* __restrict__ run_max, const float* __restrict__ run_sum,
                              const float* __restrict__ zlab, const int32_t* __restrict__ labels, int ignore, int V,
                              int64_t M, float* __restrict__ lse, float* __restrict__ term, int* err) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= M) return;
  const float l = run_max[row] + logf(run_sum[row]);
  lse[row] = l;
  const int lab = labels[row];
  const bool valid = lab != ignore && lab >= 0 && lab < V;
  if (lab != ignore && !valid) report_device_error(err, SL_ERR_INVALID);
  term[row] = valid ? (l - zlab[row]) : 0.0f;
}

// Single block: N_valid, loss = sum(term) / N_valid (fixed order), per-row scale.
__global__ void __launch_bounds__(1024) ce_finalize_kernel(const int32_t* __restrict__ labels, int ignore, int V,
                                                           const float* __restrict__ term, int64_t M,
                                                           float* __restrict__ loss, float* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
  __shared__ float s_sum[32];
  __shared__ int s_cnt[32];
  float acc = 0.0f;
  int cnt = 0;
  for (int64_t i = threadIdx.x; i < M; i += blockDim.x) {
    const int lab = labels[i];
    if (lab != ignore && lab >= 0 && lab < V) {
      ++cnt;
      acc += term[i];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc += __shfl_xor_sync(0xffffffffu, acc, o);
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  if ((threadIdx.x & 31) == 0) {
    s_sum[threadIdx.x >> 5] = acc;
    s_cnt[threadIdx.x >> 5] = cnt;
  }
  __syncthreads();
  __shared__ float s_inv;
  if (threadIdx.x == 0) {
    float t = 0.0f;
    int n = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
      t += s_sum[w];
      n += s_cnt[w];
    }
    *loss = n > 0 ? t / static_cast<float>(n) : 0.0f;
    s_inv = n > 0 ? 1.0f / static_cast<float>(n) : 0.0f;
  }
  __syncthreads();
  for (int64_t i = threadIdx.x; i < M; i += blockDim.x) {
    const int lab = labels[i];
    scale[i] = (lab != ignore && lab >= 0 && lab < V) ? s_inv : 0.0f;
  }
}

// dH[i, :] = acc[i, :] * scale_i / S_i - W[label_i, :] * scale_i (valid rows; 0 otherwise)
__global__ void ce_final_kernel(float* __restrict__ dH, const uint16_t* __restrict__ W,
                                const int32_t* __restrict__ labels, const float* __restrict__ scale,
                                const float* __restrict__ run_sum, int ignore, int V, int D) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int lab = labels[row];
  const bool valid = lab != ignore && lab >= 0 && lab < V;
  const float sc = valid ? scale[row] : 0.0f;
  const float f = valid ? sc / run_sum[row] : 0.0f;
  for (int j = threadIdx.x * 8; j < D; j += blockDim.x * 8) {
    float4* o = reinterpret_cast<float4*>(dH + row * D + j);
    float4 a = o[0], b = o[1];
    a.x *= f; a.y *= f; a.z *= f; a.w *= f;
    b.x *= f; b.y *= f; b.z *= f; b.w *= f;
    if (valid) {
      const uint4 w = *reinterpret_cast<const uint4*>(W + static_cast<int64_t>(lab) * D + j);
      const uint32_t p[4] = {w.x, w.y, w.z, w.w};
      a.x -= bf16_lo(p[0]) * sc;
      a.y -= bf16_hi(p[0]) * sc;
      a.z -= bf16_lo(p[1]) * sc;
      a.w -= bf16_hi(p[1]) * sc;
      b.x -= bf16_lo(p[2]) * sc;
      b.y -= bf16_hi(p[2]) * sc;
      b.z -= bf16_lo(p[3]) * sc;
      b.w -= bf16_hi(p[3]) * sc;
    }
    o[0] = a;
    o[1] = b;
  }
}

}  // namespace

sl_status ce_fwd_bwd(const void* H, int64_t M, int64_t D, const void* W, int64_t V, const int32_t* labels,
                     int32_t ignore, int64_t chunk_V, float* loss, float* dH, void* ws, size_t ws_bytes,
                     cudaStream_t stream) {
  SL_REQUIRE(H && W && labels && loss && dH && ws, "sl_ce_fwd_bwd: null argument");
  SL_REQUIRE(M > 0 && M < (1LL << 31) && D > 0 && V > 0 && V < (1LL << 31), "sl_ce_fwd_bwd: bad sizes");
  SL_REQUIRE(D % 256 == 0, "sl_ce_fwd_bwd: D must be a multiple of 256");
  SL_REQUIRE(V % 32 == 0, "sl_ce_fwd_bwd: V must be a multiple of 32");
  SL_REQUIRE(chunk_V > 0 && chunk_V % 256 == 0, "sl_ce_fwd_bwd: chunk_V must be a positive multiple of 256");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255) == 0, "sl_ce_fwd_bwd: workspace must be 256-byte aligned");
  const CEPlan P = ce_plan(M, D, V, chunk_V);
  SL_REQUIRE(ws_bytes >= P.total, "sl_ce_fwd_bwd: workspace too small (need " + std::to_string(P.total) + ")");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* pmax = reinterpret_cast<float*>(base + P.part_max);
  float* psum = reinterpret_cast<float*>(base + P.part_sum);
  float* zlab = reinterpret_cast<float*>(base + P.label_logit);
  float* run_max = reinterpret_cast<float*>(base + P.run_max);
  float* run_sum = reinterpret_cast<float*>(base + P.run_sum);
  float* alpha = reinterpret_cast<float*>(base + P.alpha);
  float* lse = reinterpret_cast<float*>(base + P.lse);
  float* term = reinterpret_cast<float*>(base + P.term);
  float* scale = reinterpret_cast<float*>(base + P.scale);
  uint16_t* Pc = reinterpret_cast<uint16_t*>(base + P.P);
  const uint16_t* Wh = static_cast<const uint16_t*>(W);
  sl_status st = SL_OK;
  for (int64_t v0 = 0; v0 < V; v0 += chunk_V) {
    const int64_t vc = (V - v0 < chunk_V) ? (V - v0) : chunk_V;
    // logits of the chunk: exp against the half-tile max, partials, label logit
    GemmLaunch g{};
    g.bsrc = kBSrcBF16;
    g.bmn = 0;
    g.epi = kEpiCEExp;
    g.A = H;
    g.lda = D;
    g.w = Wh + v0 * D;
    g.ldw = D;
    g.args.M = static_cast<int>(M);
    g.args.N = static_cast<int>(vc);
    g.args.K = static_cast<int>(D);
    g.args.out = Pc;
    g.args.ld_out = chunk_V;
    g.args.labels = labels;
    g.args.ignore_index = ignore;
    g.args.vocab_base = static_cast<int>(v0);
    g.args.part_max = pmax;
    g.args.part_sum = psum;
    g.args.label_logit = zlab;
    g.args.part_ld = P.halves;
    g.args.err = err;
    g.split_ws = P.split_bytes ? base + P.split : nullptr;
    g.split_ws_bytes = P.split_bytes;
    st = launch_gemm(g, stream);
    if (st != SL_OK) return st;
    // running (max, sum); P rescaled to the running max; alpha for dH
    const int halves_c = static_cast<int>(ceil_div(vc, kBN)) * 2;
    st = launch_pdl("ce_chunk_kernel", ce_chunk_kernel, dim3(static_cast<unsigned>(ceil_div(M * 32, 256))), dim3(256),
                    0, stream, pmax, psum, halves_c, P.halves, static_cast<int>(vc), M, Pc, static_cast<int>(chunk_V),
                    run_max, run_sum, alpha, v0 == 0 ? 1 : 0);
    if (st != SL_OK) return st;
    // dH accumulator = alpha * dH accumulator + P W_c
    GemmLaunch h{};
    h.bsrc = kBSrcBF16;
    h.bmn = 1;
    h.epi = kEpiAddF32;
    h.A = Pc;
    h.lda = chunk_V;
    h.w = Wh + v0 * D;
    h.ldw = D;
    h.args.M = static_cast<int>(M);
    h.args.N = static_cast<int>(D);
    h.args.K = static_cast<int>(vc);
    h.args.out = dH;
    h.args.ld_out = D;
    h.args.accumulate = v0 > 0 ? 1 : 0;
    h.args.row_alpha = alpha;
    h.args.err = err;
    h.split_ws = P.split_bytes ? base + P.split : nullptr;
    h.split_ws_bytes = P.split_bytes;
    st = launch_gemm(h, stream);
    if (st != SL_OK) return st;
  }
  st = launch_pdl("ce_row_kernel", ce_row_kernel, dim3(static_cast<unsigned>(ceil_div(M, 256))), dim3(256), 0, stream,
                  run_max, run_sum, zlab, labels, ignore, static_cast<int>(V), M, lse, term, err);
  if (st != SL_OK) return st;
  st = launch_pdl("ce_finalize_kernel", ce_finalize_kernel, dim3(1), dim3(1024), 0, stream, labels, ignore,
                  static_cast<int>(V), term, M, loss, scale);
  if (st != SL_OK) return st;
  return launch_pdl("ce_final_kernel", ce_final_kernel, dim3(static_cast<unsigned>(M)), dim3(256), 0, stream, dH, Wh,
                    labels, scale, run_sum, ignore, static_cast<int>(V), static_cast<int>(D));
}

}  // namespace sl

using namespace sl;

extern "C" sl_status sl_ce_fwd_bwd(const void* H, int64_t M, int64_t D, const void* W_head, int64_t V,
                                   const int32_t* labels, int32_t ignore_index, int64_t chunk_V, float* loss,
                                   float* dH, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return ce_fwd_bwd(H, M, D, W_head, V, labels, ignore_index, chunk_V, loss, dH, ws, ws_bytes, stream);
}

extern "C" size_t sl_ce_workspace_size(int64_t M, int64_t D, int64_t V, int64_t chunk_V) {
  if (M <= 0 || D <= 0 || V <= 0 || chunk_V <= 0) return 0;
  return ce_plan(M, D, V, chunk_V).total;
}
