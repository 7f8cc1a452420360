// Step a8: cross-entropy over the LM head, loss and dH, without the logits.
//
// "Exact Layer Streaming ..." (abstract) measures the cross-entropy logits
// term at 14 bytes per logit element; here no [M, V] tensor exists at all:
//   pass 1  one tcgen05 GEMM Z = H W^T whose epilogue keeps, per row and per
//           256-wide vocab tile, only (max, sum exp) and the label's logit;
//   rows    lse_i = log sum exp(z_i) from the tile partials (fixed order),
//           loss = mean over valid rows of lse_i - z_i,label (fixed order);
//   pass 2  per vocab chunk of chunk_V rows of W: recompute Z_c, write
//           G_c = softmax(Z_c) / N_valid (bf16, [M, chunk_V] scratch), then
//           dH += G_c W_c (fp32, tcgen05 with an MN-major W operand);
//   last    dH_i -= W[label_i] / N_valid (fp32 gather; the one-hot part is
//           kept out of the bf16 chunk so that it is exact).
// Extra device bytes: the chunk scratch plus O(M * V / 256) partials.
#include "common.cuh"
#include "gemm.cuh"

namespace sl {

namespace {

struct CEPlan {
  size_t part_max, part_sum, label_logit, lse, term, scale, G, total;
  int ntiles;
};

CEPlan ce_plan(int64_t M, int64_t D, int64_t V, int64_t chunk_V) {
  (void)D;
  CEPlan p{};
  size_t off = 0;
  auto take = [&](size_t b) {
    const size_t o = off;
    off = align_up(off + b, 256);
    return o;
  };
  p.ntiles = static_cast<int>(ceil_div(V, kBN)) * 2;   // two column halves per 256-wide tile
  p.part_max = take(static_cast<size_t>(M) * p.ntiles * 4);
  p.part_sum = take(static_cast<size_t>(M) * p.ntiles * 4);
  p.label_logit = take(M * 4);
  p.lse = take(M * 4);
  p.term = take(M * 4);
  p.scale = take(M * 4);
  p.G = take(static_cast<size_t>(M) * chunk_V * 2);
  p.total = off;
  return p;
}

// One warp per row: lse from the per-half-tile (max, sum exp) partials; the row's
// loss term lse - z_label (0 for ignored rows).  Out-of-range labels are
// reported through the error word and treated as ignored.
__global__ void ce_row_kernel(const float* __restrict__ pmax, const float* __restrict__ psum, int ntiles,
                              const float* __restrict__ zlab, const int32_t* __restrict__ labels, int ignore, int V,
                              int64_t M, float* __restrict__ lse, float* __restrict__ term, int* err) {
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  float mx = -INFINITY, sm = 0.0f;
  for (int t = lane; t < ntiles; t += 32) {
    const float m2 = pmax[row * ntiles + t], s2 = psum[row * ntiles + t];
    const float nm = fmaxf(mx, m2);
    if (nm == -INFINITY) continue;
    sm = sm * __expf(mx - nm) + s2 * __expf(m2 - nm);
    mx = nm;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mx, o), s2 = __shfl_xor_sync(0xffffffffu, sm, o);
    const float nm = fmaxf(mx, m2);
    if (nm != -INFINITY) {
      sm = sm * __expf(mx - nm) + s2 * __expf(m2 - nm);
      mx = nm;
    }
  }
  if (lane == 0) {
    const float l = mx + logf(sm);
    lse[row] = l;
    const int lab = labels[row];
    const bool valid = lab != ignore && lab >= 0 && lab < V;
    if (lab != ignore && !valid) report_device_error(err, SL_ERR_INVALID);
    term[row] = valid ? (l - zlab[row]) : 0.0f;
  }
}

// Single block: N_valid, loss = sum(term) / N_valid (fixed order), per-row scale.
__global__ void __launch_bounds__(1024) ce_finalize_kernel(const int32_t* __restrict__ labels, int ignore, int V,
                                                           const float* __restrict__ term, int64_t M,
                                                           float* __restrict__ loss, float* __restrict__ scale) {
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

// dH[i, :] -= W[label_i, :] * scale_i   (valid rows)
__global__ void ce_label_kernel(float* __restrict__ dH, const uint16_t* __restrict__ W,
                                const int32_t* __restrict__ labels, const float* __restrict__ scale, int ignore,
                                int V, int D) {
  const int64_t row = blockIdx.x;
  const int lab = labels[row];
  if (lab == ignore || lab < 0 || lab >= V) return;
  const float sc = scale[row];
  for (int j = threadIdx.x * 8; j < D; j += blockDim.x * 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(W + static_cast<int64_t>(lab) * D + j);
    const uint32_t p[4] = {w.x, w.y, w.z, w.w};
    float4* o = reinterpret_cast<float4*>(dH + row * D + j);
    float4 a = o[0], b = o[1];
    a.x -= bf16_lo(p[0]) * sc;
    a.y -= bf16_hi(p[0]) * sc;
    a.z -= bf16_lo(p[1]) * sc;
    a.w -= bf16_hi(p[1]) * sc;
    b.x -= bf16_lo(p[2]) * sc;
    b.y -= bf16_hi(p[2]) * sc;
    b.z -= bf16_lo(p[3]) * sc;
    b.w -= bf16_hi(p[3]) * sc;
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
  float* lse = reinterpret_cast<float*>(base + P.lse);
  float* term = reinterpret_cast<float*>(base + P.term);
  float* scale = reinterpret_cast<float*>(base + P.scale);
  uint16_t* G = reinterpret_cast<uint16_t*>(base + P.G);
  const uint16_t* Wh = static_cast<const uint16_t*>(W);

  // pass 1: row (max, sum exp) partials and label logits over the whole vocab
  {
    GemmLaunch g{};
    g.bsrc = kBSrcBF16;
    g.bmn = 0;
    g.epi = kEpiCELse;
    g.A = H;
    g.lda = D;
    g.w = W;
    g.ldw = D;
    g.args.M = static_cast<int>(M);
    g.args.N = static_cast<int>(V);
    g.args.K = static_cast<int>(D);
    g.args.labels = labels;
    g.args.ignore_index = ignore;
    g.args.vocab_base = 0;
    g.args.part_max = pmax;
    g.args.part_sum = psum;
    g.args.label_logit = zlab;
    g.args.part_ld = P.ntiles;
    g.args.tile_base = 0;
    g.args.err = err;
    sl_status st = launch_gemm(g, stream);
    if (st != SL_OK) return st;
  }
  ce_row_kernel<<<static_cast<unsigned>(ceil_div(M * 32, 256)), 256, 0, stream>>>(
      pmax, psum, P.ntiles, zlab, labels, ignore, static_cast<int>(V), M, lse, term, err);
  sl_status st = check_launch("ce_row_kernel");
  if (st != SL_OK) return st;
  ce_finalize_kernel<<<1, 1024, 0, stream>>>(labels, ignore, static_cast<int>(V), term, M, loss, scale);
  st = check_launch("ce_finalize_kernel");
  if (st != SL_OK) return st;

  // pass 2: chunked softmax gradient and dH accumulation
  for (int64_t v0 = 0; v0 < V; v0 += chunk_V) {
    const int64_t vc = (V - v0 < chunk_V) ? (V - v0) : chunk_V;
    GemmLaunch g{};
    g.bsrc = kBSrcBF16;
    g.bmn = 0;
    g.epi = kEpiCEGrad;
    g.A = H;
    g.lda = D;
    g.w = Wh + v0 * D;
    g.ldw = D;
    g.args.M = static_cast<int>(M);
    g.args.N = static_cast<int>(vc);
    g.args.K = static_cast<int>(D);
    g.args.out = G;
    g.args.ld_out = chunk_V;
    g.args.labels = labels;
    g.args.ignore_index = ignore;
    g.args.vocab_base = static_cast<int>(v0);
    g.args.row_lse = lse;
    g.args.row_scale = scale;
    g.args.err = err;
    st = launch_gemm(g, stream);
    if (st != SL_OK) return st;

    GemmLaunch h{};
    h.bsrc = kBSrcBF16;
    h.bmn = 1;
    h.epi = kEpiAddF32;
    h.A = G;
    h.lda = chunk_V;
    h.w = Wh + v0 * D;
    h.ldw = D;
    h.args.M = static_cast<int>(M);
    h.args.N = static_cast<int>(D);
    h.args.K = static_cast<int>(vc);
    h.args.out = dH;
    h.args.ld_out = D;
    h.args.accumulate = v0 > 0 ? 1 : 0;
    h.args.err = err;
    st = launch_gemm(h, stream);
    if (st != SL_OK) return st;
  }
  ce_label_kernel<<<static_cast<unsigned>(M), 256, 0, stream>>>(dH, Wh, labels, scale, ignore, static_cast<int>(V),
                                                               static_cast<int>(D));
  return check_launch("ce_label_kernel");
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
