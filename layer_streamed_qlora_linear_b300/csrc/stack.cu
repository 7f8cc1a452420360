// The layer-streamed stack step (steps a2, a5, a7 plus the seven linears of
// every layer).
//
// "Soup CLI Lets You Fine-Tune an 8B LLM on a 4 GB Laptop GPU", "How Layer
// Streaming Works": the frozen base stays in system RAM and decoder layers
// are brought to the GPU for the forward and backward passes.  "Soup:
// Fine-Tuning an 8B LLM ... with One YAML File", "Layer Streaming: The
// Mechanism Behind the 4 GB Claim": a pinned base store and two device
// buffers.  "Exact Layer Streaming ..." (abstract): the streamed run is
// bit-exact against a resident run of the same numerics.
//
// Design: one pinned host blob per layer (sl_stack_blob_layout); two device
// buffers; layer l lives in buffer l % 2.  A non-blocking copy stream does
// one cudaMemcpyAsync per layer; event ready[b] (recorded after the copy)
// gates the compute stream, event free[b] (recorded after the last kernel
// that read buffer b) gates the next copy into b.  The forward walks layers
// 0..L-1 prefetching l+2, the backward walks L-1..0 prefetching l-2; the two
// layers resident at the turn are not copied again, and neither are layers
// 0 and 1 at the start of the next step when the buffers still hold them
// (the base is frozen).  RESIDENT mode runs the same kernels in the same
// order on device copies of the blobs, so both modes give identical bits.
#include <algorithm>
#include <cstring>
#include <vector>

#include "attn.cuh"
#include "common.cuh"
#include "glue.cuh"
#include "gemm.cuh"
#include "linear.cuh"
#include "skinny.cuh"

using namespace sl;

struct sl_stack {
  int L = 0;
  int kind = 0;
  int64_t D = 0, Dkv = 0, F = 0;
  int mixer = SL_MIX_TOKEN_LOCAL;
  int64_t seq_len = 0;
  double rope_theta = 0.0;
  std::vector<const void*> host;
  std::vector<const void*> dev;
  size_t offs[16] = {0};
  // NF4_DQ: per projection its group's qabsmax / absmax2 arrays, their row
  // lengths and the projection's first column in them
  size_t dq_q[7] = {0}, dq_a2[7] = {0};
  int64_t dq_qld[7] = {0}, dq_a2ld[7] = {0}, dq_col0[7] = {0};
  size_t blob_bytes = 0;
  void* buf[2] = {nullptr, nullptr};
  int buf_layer[2] = {-1, -1};
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ready[2] = {nullptr, nullptr};
  cudaEvent_t freed[2] = {nullptr, nullptr};
  // The step runs on main_stream (highest priority); each projection unit's
  // adapter-gradient passes (dA, dB) run on the caller's stream once its U
  // is written (fork[u]) and mark done[u]; main_stream waits on done[u]
  // only before it overwrites what those passes read.  step_in / step_out
  // join the caller's stream at the start and end of a step.
  cudaStream_t main_stream = nullptr;
  cudaEvent_t step_in = nullptr, step_out = nullptr;
  cudaEvent_t fork[4] = {nullptr, nullptr, nullptr, nullptr};
  cudaEvent_t done[4] = {nullptr, nullptr, nullptr, nullptr};
  int device = 0;
  uint64_t last_h2d = 0;
  uint64_t last_kernels = 0;
};

namespace {

struct Proj {
  int64_t N, K;
};

void proj_shapes(int64_t D, int64_t Dkv, int64_t F, Proj p[7]) {
  p[0] = {D, D};    // q
  p[1] = {Dkv, D};  // k
  p[2] = {Dkv, D};  // v
  p[3] = {D, D};    // o
  p[4] = {F, D};    // gate
  p[5] = {F, D};    // up
  p[6] = {D, F};    // down
}

struct DqLayout {
  size_t q[7], a2[7];
  int64_t q_ld[7], a2_ld[7], col0[7];
};

// Absmax groups of a double-quantised blob: q/k/v, o, gate/up, down (the
// projections of one group read one input, so their absmax share one
// transposed 8-bit array and the projection group reads it as one weight).
constexpr int kDqFirst[4] = {0, 3, 4, 6};
constexpr int kDqCount[4] = {3, 1, 2, 1};

sl_status layout(int kind, int64_t D, int64_t Dkv, int64_t F, size_t offs[16], size_t* total, DqLayout* dq) {
  Proj p[7];
  proj_shapes(D, Dkv, F, p);
  // NF4: all codes, then all absmax, so that the q, k, v and the gate, up
  // codes (and absmax) are contiguous: with D, F multiples of 256 and Dkv a
  // multiple of 128 every region is a multiple of 256 bytes (no padding).
  size_t off = 0;
  for (int i = 0; i < 7; ++i) {
    const size_t n = static_cast<size_t>(p[i].N) * static_cast<size_t>(p[i].K);
    offs[2 * i] = off;
    off = align_up(off + (kind == SL_WEIGHT_BF16 ? n * 2 : n / 2), 256);
    offs[2 * i + 1] = 0;
  }
  if (kind == SL_WEIGHT_NF4)
    for (int i = 0; i < 7; ++i) {
      const size_t n = static_cast<size_t>(p[i].N) * static_cast<size_t>(p[i].K);
      offs[2 * i + 1] = off;
      off = align_up(off + n / 64 * 4, 256);
    }
  if (kind == SL_WEIGHT_NF4_DQ)
    for (int g = 0; g < 4; ++g) {
      const int p0 = kDqFirst[g];
      int64_t N = 0;
      for (int i = 0; i < kDqCount[g]; ++i) N += p[p0 + i].N;
      const int64_t rows = p[p0].K / 64, q_ld = N, a2_ld = (2 * (N / 256) + 3) / 4 * 4;
      const size_t q_off = off;
      off = align_up(off + static_cast<size_t>(rows * q_ld), 256);
      const size_t a2_off = off;
      off = align_up(off + static_cast<size_t>(rows * a2_ld) * 4, 256);
      int64_t col = 0;
      for (int i = 0; i < kDqCount[g]; ++i) {
        const int pi = p0 + i;
        offs[2 * pi + 1] = q_off;
        if (dq) {
          dq->q[pi] = q_off;
          dq->a2[pi] = a2_off;
          dq->q_ld[pi] = q_ld;
          dq->a2_ld[pi] = a2_ld;
          dq->col0[pi] = col;
        }
        col += p[pi].N;
      }
    }
  // the two RMS-norm weights (fp32 [D]: before attention, before the MLP)
  for (int i = 0; i < 2; ++i) {
    offs[14 + i] = off;
    off = align_up(off + static_cast<size_t>(D) * 4, 256);
  }
  *total = off;
  return SL_OK;
}

// Workspace plan: per-layer saved activations plus shared scratch.  The
// q/k/v outputs live in one region of M x (D + 2 Dkv) and the gate/up
// outputs in one of M x 2 F: as column blocks (row stride D + 2 Dkv, 2 F)
// when a projection group produced them, as dense arrays one after the
// other otherwise; the same holds for their gradients and side products T.
struct Plan {
  size_t total = 0;
  // per layer
  std::vector<size_t> hin, h1, rstd1, rstd2, x1, qkv, a, x2, gu, m;
  std::vector<size_t> Tqkv, To, Tgu, Td, lse;
  // shared
  size_t o, d, dhA, dhB, dd, dm, dgu, dx2a, dx2b, dh1, do_, da, dqkv, dx1q, dx1k, dx1v, lin_ws;
  // U of each projection unit's backward (down, gate/up, o, q/k/v), kept
  // until that unit's dA pass has read it: [M, G r] fp32 each
  size_t U[4] = {0, 0, 0, 0};
  size_t U_bytes[4] = {0, 0, 0, 0};
  // scratch that lets the persistent GEMMs split their last partial wave
  // along K (the GEMMs run one after another on the main stream)
  size_t split = 0, split_bytes = 0;
  size_t att_ws = 0, rope = 0;  // attention: Di [H, M] and the rotary table [S, 128]
  size_t lin_ws_bytes = 0;
};

Plan make_plan(const sl_stack* s, int64_t M, int r) {
  Plan P;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t MD = static_cast<size_t>(M) * s->D, MF = static_cast<size_t>(M) * s->F;
  const size_t MQKV = static_cast<size_t>(M) * (s->D + 2 * s->Dkv);
  const int L = s->L;
  const int rr = r > 0 ? r : 0;
  const size_t Tr = static_cast<size_t>(M) * (rr ? rr : 1) * 4;
  for (int l = 0; l < L; ++l) {
    P.hin.push_back(l == 0 ? 0 : take(MD * 4));
    P.h1.push_back(take(MD * 4));
    P.rstd1.push_back(take(M * 4));
    P.rstd2.push_back(take(M * 4));
    P.x1.push_back(take(MD * 2));
    P.qkv.push_back(take(MQKV * 2));
    P.a.push_back(take(MD * 2));
    P.x2.push_back(take(MD * 2));
    P.gu.push_back(take(2 * MF * 2));
    P.m.push_back(take(MF * 2));
    P.Tqkv.push_back(take(3 * Tr));
    P.To.push_back(take(Tr));
    P.Tgu.push_back(take(2 * Tr));
    P.Td.push_back(take(Tr));
    P.lse.push_back(s->mixer == SL_MIX_ATTENTION ? take(static_cast<size_t>(M) * (s->D / 128) * 4) : 0);
  }
  P.o = take(MD * 2);
  P.d = take(MD * 2);
  P.dhA = take(MD * 4);
  P.dhB = take(MD * 4);
  P.dd = take(MD * 2);
  P.dm = take(MF * 2);
  P.dgu = take(2 * MF * 2);
  P.dx2a = take(MD * 2);
  P.dx2b = take(MD * 2);
  P.dh1 = take(MD * 4);
  P.do_ = take(MD * 2);
  P.da = take(MD * 2);
  P.dqkv = take(MQKV * 2);
  P.dx1q = take(MD * 2);
  P.dx1k = take(MD * 2);
  P.dx1v = take(MD * 2);
  Proj pr[7];
  proj_shapes(s->D, s->Dkv, s->F, pr);
  size_t lw = 0;
  for (int p = 0; p < 7; ++p) lw = std::max(lw, linear_ws_bytes(M, pr[p].N, pr[p].K, rr));
  if (rr) lw = std::max(lw, group_ws_bytes(M, 3, rr));
  P.lin_ws_bytes = lw;
  P.lin_ws = take(lw ? lw : 256);
  const int unit_G[4] = {1, 2, 1, 3};  // down, gate/up, o, q/k/v
  for (int u = 0; u < 4; ++u) {  // G regions of [M, r] (a group's [M, G r] fits in them)
    P.U_bytes[u] = unit_G[u] * align_up(static_cast<size_t>(M) * (rr ? rr : 1) * 4, 256);
    P.U[u] = take(P.U_bytes[u]);
  }
  if (M > 128 && s->kind != SL_WEIGHT_BF16) {
    P.split_bytes = split_scratch_bytes();
    P.split = take(P.split_bytes);
  }
  if (s->mixer == SL_MIX_ATTENTION) {
    P.att_ws = take(attention_ws_bytes(M, static_cast<int>(s->D / 128)));
    P.rope = take(static_cast<size_t>(s->seq_len) * 128 * 4);
  }
  P.total = off;
  return P;
}

struct StepCtx {
  sl_stack* s;
  const Plan* P;
  uint8_t* ws;
  int64_t M;
  int r;
  float alpha;
  const void* const* A;
  const void* const* B;
  float* const* dA;
  float* const* dB;
  cudaStream_t stream;   // the step's main stream (the handle's high-priority stream)
  cudaStream_t side;     // the caller's stream: adapter-gradient passes
  int accumulate = 0;
  bool group_qkv = false;  // q, k, v as one projection group
  bool group_gu = false;   // gate, up as one projection group
  uint64_t kernels = 0;

  template <typename T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(ws + off);
  }
};

void weights_of(const sl_stack* s, const void* base, sl_weight w[7], const float* norms[2]) {
  Proj p[7];
  proj_shapes(s->D, s->Dkv, s->F, p);
  const uint8_t* b = static_cast<const uint8_t*>(base);
  norms[0] = reinterpret_cast<const float*>(b + s->offs[14]);
  norms[1] = reinterpret_cast<const float*>(b + s->offs[15]);
  for (int i = 0; i < 7; ++i) {
    w[i].kind = s->kind;
    w[i].N = p[i].N;
    w[i].K = p[i].K;
    w[i].qabsmax = nullptr;
    w[i].qabsmax_ld = 0;
    w[i].absmax2 = nullptr;
    w[i].absmax2_ld = 0;
    w[i].dq_col0 = 0;
    if (s->kind == SL_WEIGHT_NF4) {
      w[i].codes = b + s->offs[2 * i];
      w[i].absmax = reinterpret_cast<const float*>(b + s->offs[2 * i + 1]);
      w[i].w = nullptr;
    } else if (s->kind == SL_WEIGHT_NF4_DQ) {
      w[i].codes = b + s->offs[2 * i];
      w[i].absmax = nullptr;
      w[i].w = nullptr;
      w[i].qabsmax = reinterpret_cast<const int8_t*>(b + s->dq_q[i]);
      w[i].qabsmax_ld = s->dq_qld[i];
      w[i].absmax2 = reinterpret_cast<const float*>(b + s->dq_a2[i]);
      w[i].absmax2_ld = s->dq_a2ld[i];
      w[i].dq_col0 = s->dq_col0[i];
    } else {
      w[i].codes = nullptr;
      w[i].absmax = nullptr;
      w[i].w = b + s->offs[2 * i];
    }
  }
}

#define SL_TRY(expr)                  \
  do {                                \
    sl_status _st = (expr);           \
    if (_st != SL_OK) return _st;     \
  } while (0)

// The q/k/v (p0 = 0, G = 3) or gate/up (p0 = 4, G = 2) weights as one NF4
// weight: the blob keeps them back to back (and a double-quantised blob
// their absmax in one array, from the first projection's column on).
sl_weight group_weight(const sl_weight w[7], int p0, int G) {
  sl_weight g = w[p0];
  for (int i = 1; i < G; ++i) g.N += w[p0 + i].N;
  return g;
}

sl_status layer_fwd(StepCtx& c, int l, const sl_weight w[7], const float* const norms[2], const float* h_in,
                    float* h_out) {
  const Plan& P = *c.P;
  const sl_stack* s = c.s;
  const int64_t M = c.M;
  const int D = static_cast<int>(s->D), Dkv = static_cast<int>(s->Dkv), F = static_cast<int>(s->F);
  const int r = c.r;
  const int64_t rr = r > 0 ? r : 1;
  auto A = [&](int p) { return r > 0 ? c.A[7 * l + p] : nullptr; };
  auto B = [&](int p) { return r > 0 ? c.B[7 * l + p] : nullptr; };
  void* spl = P.split_bytes ? c.at<uint8_t>(P.split) : nullptr;
  const size_t spb = P.split_bytes;
  uint16_t* x1 = c.at<uint16_t>(P.x1[l]);
  uint16_t* qkv = c.at<uint16_t>(P.qkv[l]);
  uint16_t* a = c.at<uint16_t>(P.a[l]);
  uint16_t* x2 = c.at<uint16_t>(P.x2[l]);
  uint16_t* gu = c.at<uint16_t>(P.gu[l]);
  uint16_t* m = c.at<uint16_t>(P.m[l]);
  float* Tqkv = c.at<float>(P.Tqkv[l]);
  float* Tgu = c.at<float>(P.Tgu[l]);
  float* h1 = c.at<float>(P.h1[l]);
  uint16_t* o = c.at<uint16_t>(P.o);
  uint16_t* d = c.at<uint16_t>(P.d);
  SL_TRY(glue_rms_fwd(h_in, nullptr, nullptr, x1, c.at<float>(P.rstd1[l]), norms[0], M, D, c.stream));
  // q, k, v
  uint16_t *q, *k, *v;
  int64_t ldq, ldkv;
  if (c.group_qkv) {
    const sl_weight wg = group_weight(w, 0, 3);
    const int64_t Ng[3] = {D, Dkv, Dkv};
    SL_TRY(group_fwd_x(&wg, 3, Ng, x1, M, A(0), B(0), r, c.alpha, qkv, Tqkv, spl, spb, c.stream));
    q = qkv;
    k = qkv + D;
    v = qkv + D + Dkv;
    ldq = ldkv = D + 2 * Dkv;
  } else {
    uint16_t* yq = qkv;
    uint16_t* yk = qkv + M * D;
    uint16_t* yv = yk + M * Dkv;
    SL_TRY(linear_fwd_x(&w[0], x1, M, A(0), B(0), r, c.alpha, yq, Tqkv, spl, spb, c.stream));
    SL_TRY(linear_fwd_x(&w[1], x1, M, A(1), B(1), r, c.alpha, yk, Tqkv + M * rr, spl, spb, c.stream));
    SL_TRY(linear_fwd_x(&w[2], x1, M, A(2), B(2), r, c.alpha, yv, Tqkv + 2 * M * rr, spl, spb, c.stream));
    q = yq;
    k = yk;
    v = yv;
    ldq = D;
    ldkv = Dkv;
  }
  if (s->mixer == SL_MIX_ATTENTION) {
    // rotate q and k in place (the saved q/k are the rotated ones), then attention
    const float* rope = c.at<float>(P.rope);
    if (c.group_qkv) {
      SL_TRY(rope_apply(q, ldq, M, (D + Dkv) / 128, s->seq_len, rope, 0, c.stream));  // q | k columns
    } else {
      SL_TRY(rope_apply(q, ldq, M, D / 128, s->seq_len, rope, 0, c.stream));
      SL_TRY(rope_apply(k, ldkv, M, Dkv / 128, s->seq_len, rope, 0, c.stream));
    }
    const AttnShape sh{M, s->seq_len, D / 128, Dkv / 128};
    SL_TRY(attention_fwd(sh, q, ldq, k, ldkv, v, ldkv, a, D, c.at<float>(P.lse[l]), c.stream));
  } else {
    SL_TRY(glue_mix_fwd(q, k, v, a, M, D, Dkv, ldq, ldkv, c.stream));
  }
  SL_TRY(linear_fwd_x(&w[3], a, M, A(3), B(3), r, c.alpha, o, c.at<float>(P.To[l]), spl, spb, c.stream));
  SL_TRY(glue_rms_fwd(h_in, o, h1, x2, c.at<float>(P.rstd2[l]), norms[1], M, D, c.stream));
  // gate, up
  if (c.group_gu) {
    const sl_weight wg = group_weight(w, 4, 2);
    const int64_t Ng[2] = {F, F};
    SL_TRY(group_fwd_x(&wg, 2, Ng, x2, M, A(4), B(4), r, c.alpha, gu, Tgu, spl, spb, c.stream));
    SL_TRY(glue_swiglu_fwd(gu, gu + F, m, M, F, 2 * F, c.stream));
  } else {
    SL_TRY(linear_fwd_x(&w[4], x2, M, A(4), B(4), r, c.alpha, gu, Tgu, spl, spb, c.stream));
    SL_TRY(linear_fwd_x(&w[5], x2, M, A(5), B(5), r, c.alpha, gu + M * F, Tgu + M * rr, spl, spb, c.stream));
    SL_TRY(glue_swiglu_fwd(gu, gu + M * F, m, M, F, F, c.stream));
  }
  SL_TRY(linear_fwd_x(&w[6], m, M, A(6), B(6), r, c.alpha, d, c.at<float>(P.Td[l]), spl, spb, c.stream));
  SL_TRY(glue_resid_add(h1, d, h_out, M * s->D, c.stream));
  return SL_OK;
}

// dh2: gradient w.r.t. this layer's output (fp32) and its bf16 copy dd;
// writes dh (w.r.t. the layer input) and, if dh_bf16, its bf16 copy.
sl_status layer_bwd(StepCtx& c, int l, const sl_weight w[7], const float* const norms[2], const float* h_in,
                    const float* dh2, const uint16_t* dd, float* dh, uint16_t* dh_bf16) {
  const Plan& P = *c.P;
  const sl_stack* s = c.s;
  const int64_t M = c.M;
  const int D = static_cast<int>(s->D), Dkv = static_cast<int>(s->Dkv), F = static_cast<int>(s->F);
  const int r = c.r;
  const int64_t rr = r > 0 ? r : 1;
  auto A = [&](int p) { return r > 0 ? c.A[7 * l + p] : nullptr; };
  auto B = [&](int p) { return r > 0 ? c.B[7 * l + p] : nullptr; };
  auto dA = [&](int p) { return r > 0 ? c.dA[7 * l + p] : nullptr; };
  auto dB = [&](int p) { return r > 0 ? c.dB[7 * l + p] : nullptr; };
  void* spl = P.split_bytes ? c.at<uint8_t>(P.split) : nullptr;
  const size_t spb = P.split_bytes;
  uint16_t* dm = c.at<uint16_t>(P.dm);
  uint16_t* dgu = c.at<uint16_t>(P.dgu);
  uint16_t* dx2a = c.at<uint16_t>(P.dx2a);
  uint16_t* dx2b = c.at<uint16_t>(P.dx2b);
  float* dh1 = c.at<float>(P.dh1);
  uint16_t* do_ = c.at<uint16_t>(P.do_);
  uint16_t* da = c.at<uint16_t>(P.da);
  uint16_t* dqkv = c.at<uint16_t>(P.dqkv);
  uint16_t* dx1q = c.at<uint16_t>(P.dx1q);
  uint16_t* dx1k = c.at<uint16_t>(P.dx1k);
  uint16_t* dx1v = c.at<uint16_t>(P.dx1v);
  const uint16_t* x1 = c.at<uint16_t>(P.x1[l]);
  const uint16_t* x2 = c.at<uint16_t>(P.x2[l]);
  const uint16_t* qkv = c.at<uint16_t>(P.qkv[l]);
  const uint16_t* gu = c.at<uint16_t>(P.gu[l]);
  const float* Tqkv = c.at<float>(P.Tqkv[l]);
  const float* Tgu = c.at<float>(P.Tgu[l]);
  // Unit u's dA / dB run on the side stream (the caller's); before this
  // layer overwrites what the previous layer's passes of unit u read (its U
  // region, its dY region), the main stream waits for them (done[u]).
  enum { kDown = 0, kGU = 1, kO = 2, kQKV = 3 };
  auto side = [&](int u) {
    return GradSide{c.side, s->fork[u], s->done[u]};
  };
  auto wait_unit = [&](int u) -> sl_status {
    SL_CHECK_CUDA(cudaStreamWaitEvent(c.stream, s->done[u], 0));
    return SL_OK;
  };
  const size_t U1 = align_up(static_cast<size_t>(M) * rr * 4, 256);
  auto U_of = [&](int u, int i) { return c.ws + P.U[u] + static_cast<size_t>(i) * U1; };
  {
    SL_TRY(wait_unit(kDown));
    const GradSide sd = side(kDown);
    SL_TRY(linear_bwd_split(&w[6], c.at<uint16_t>(P.m[l]), dd, M, A(6), B(6), r, c.alpha, c.at<float>(P.Td[l]), dm,
                            dA(6), dB(6), c.accumulate, U_of(kDown, 0), P.U_bytes[kDown], c.stream, &sd, spl, spb));
  }
  // gate, up
  SL_TRY(wait_unit(kGU));
  if (c.group_gu) {
    // dg, du fused with the group's U_cat = [dg | du] blockdiag(B_g, B_u) when it has adapters
    const bool fuse_u = A(4) && B(4) && F % 128 == 0;
    if (fuse_u)
      SL_TRY(skinny_swiglu_u(dm, gu, gu + F, 2 * F, dgu, dgu + F, 2 * F, M, F, static_cast<const uint16_t*>(B(4)), r,
                             reinterpret_cast<float*>(U_of(kGU, 0)), c.stream));
    else
      SL_TRY(glue_swiglu_bwd(dm, gu, gu + F, dgu, dgu + F, M, F, 2 * F, c.stream));
    const sl_weight wg = group_weight(w, 4, 2);
    const int64_t Ng[2] = {F, F};
    const GradSide sd = side(kGU);
    SL_TRY(group_bwd_split(&wg, 2, Ng, x2, dgu, M, A(4), B(4), r, c.alpha, Tgu, dx2a, dA(4), dB(4), c.accumulate,
                           U_of(kGU, 0), P.U_bytes[kGU], c.stream, &sd, spl, spb, fuse_u));
    SL_TRY(wait_unit(kO));
    SL_TRY(glue_rms_bwd(dh2, dx2a, nullptr, nullptr, nullptr, c.at<float>(P.h1[l]), c.at<float>(P.rstd2[l]),
                        norms[1], dh1, do_, M, D, c.stream));
  } else {
    SL_TRY(glue_swiglu_bwd(dm, gu, gu + M * F, dgu, dgu + M * F, M, F, F, c.stream));
    const GradSide s0{c.side, s->fork[kGU], nullptr};
    const GradSide s1 = side(kGU);
    SL_TRY(linear_bwd_split(&w[4], x2, dgu, M, A(4), B(4), r, c.alpha, Tgu, dx2a, dA(4), dB(4), c.accumulate,
                            U_of(kGU, 0), U1, c.stream, &s0, spl, spb));
    SL_TRY(linear_bwd_split(&w[5], x2, dgu + M * F, M, A(5), B(5), r, c.alpha, Tgu + M * rr, dx2b, dA(5), dB(5),
                            c.accumulate, U_of(kGU, 1), U1, c.stream, &s1, spl, spb));
    SL_TRY(wait_unit(kO));
    SL_TRY(glue_rms_bwd(dh2, dx2a, dx2b, nullptr, nullptr, c.at<float>(P.h1[l]), c.at<float>(P.rstd2[l]),
                        norms[1], dh1, do_, M, D, c.stream));
  }
  {
    const GradSide sd = side(kO);
    SL_TRY(linear_bwd_split(&w[3], c.at<uint16_t>(P.a[l]), do_, M, A(3), B(3), r, c.alpha, c.at<float>(P.To[l]), da,
                            dA(3), dB(3), c.accumulate, U_of(kO, 0), P.U_bytes[kO], c.stream, &sd, spl, spb));
  }
  // q, k, v: the mixing step's backward into the dq/dk/dv region
  auto mix_bwd = [&](const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t ldq, int64_t ldkv,
                     uint16_t* dq, uint16_t* dk, uint16_t* dv) -> sl_status {
    if (s->mixer != SL_MIX_ATTENTION) return glue_mix_bwd(da, q, k, dq, dk, dv, M, D, Dkv, ldq, ldkv, c.stream);
    const AttnShape sh{M, s->seq_len, D / 128, Dkv / 128};
    return attention_bwd(sh, q, ldq, k, ldkv, v, ldkv, c.at<uint16_t>(P.a[l]), D, da, D, c.at<float>(P.lse[l]), dq,
                         ldq, dk, ldkv, dv, ldkv, c.at<float>(P.rope), c.at<uint8_t>(P.att_ws), c.stream);
  };
  SL_TRY(wait_unit(kQKV));
  if (c.group_qkv) {
    const int64_t ld = D + 2 * Dkv;
    SL_TRY(mix_bwd(qkv, qkv + D, qkv + D + Dkv, ld, ld, dqkv, dqkv + D, dqkv + D + Dkv));
    const sl_weight wg = group_weight(w, 0, 3);
    const int64_t Ng[3] = {D, Dkv, Dkv};
    const GradSide sd = side(kQKV);
    SL_TRY(group_bwd_split(&wg, 3, Ng, x1, dqkv, M, A(0), B(0), r, c.alpha, Tqkv, dx1q, dA(0), dB(0), c.accumulate,
                           U_of(kQKV, 0), P.U_bytes[kQKV], c.stream, &sd, spl, spb));
    SL_TRY(wait_unit(kDown));  // dd (this layer's down dY) is overwritten next
    SL_TRY(glue_rms_bwd(dh1, dx1q, nullptr, nullptr, nullptr, h_in, c.at<float>(P.rstd1[l]), norms[0], dh, dh_bf16, M,
                        D, c.stream));
  } else {
    uint16_t* dq = dqkv;
    uint16_t* dk = dqkv + M * D;
    uint16_t* dv = dk + M * Dkv;
    SL_TRY(mix_bwd(qkv, qkv + M * D, qkv + M * D + M * Dkv, D, Dkv, dq, dk, dv));
    const GradSide s0{c.side, s->fork[kQKV], nullptr};
    const GradSide s2 = side(kQKV);
    SL_TRY(linear_bwd_split(&w[0], x1, dq, M, A(0), B(0), r, c.alpha, Tqkv, dx1q, dA(0), dB(0), c.accumulate,
                            U_of(kQKV, 0), U1, c.stream, &s0, spl, spb));
    SL_TRY(linear_bwd_split(&w[1], x1, dk, M, A(1), B(1), r, c.alpha, Tqkv + M * rr, dx1k, dA(1), dB(1),
                            c.accumulate, U_of(kQKV, 1), U1, c.stream, &s0, spl, spb));
    SL_TRY(linear_bwd_split(&w[2], x1, dv, M, A(2), B(2), r, c.alpha, Tqkv + 2 * M * rr, dx1v, dA(2), dB(2),
                            c.accumulate, U_of(kQKV, 2), U1, c.stream, &s2, spl, spb));
    SL_TRY(wait_unit(kDown));  // dd (this layer's down dY) is overwritten next
    SL_TRY(glue_rms_bwd(dh1, dx1q, dx1k, dx1v, nullptr, h_in, c.at<float>(P.rstd1[l]), norms[0], dh, dh_bf16, M, D,
                        c.stream));
  }
  return SL_OK;
}

// Projections p0 .. p0+G-1 run as one group when the weights are NF4, M
// allows the CTA-pair GEMM, every projection is a whole number of 256-column
// tiles, the folded rank fits, and every layer stores the group's adapters
// and their gradients back to back.
bool can_group(const sl_stack* s, int64_t M, int r, int p0, int G, const void* const* A, const void* const* B,
               float* const* dA, float* const* dB) {
  if (s->kind == SL_WEIGHT_BF16 || M <= 128 || M >= (1LL << 31)) return false;
  if (r > 0 && G * r > 64) return false;
  Proj p[7];
  proj_shapes(s->D, s->Dkv, s->F, p);
  for (int i = 0; i < G; ++i)
    if (p[p0 + i].N % 256) return false;  // a GEMM tile must not straddle two projections
  if (r == 0) return true;
  for (int l = 0; l < s->L; ++l)
    for (int i = 1; i < G; ++i) {
      const int cur = 7 * l + p0 + i, prev = cur - 1;
      const size_t a_prev = static_cast<size_t>(r) * p[p0 + i - 1].K, b_prev = static_cast<size_t>(p[p0 + i - 1].N) * r;
      if (static_cast<const uint8_t*>(A[cur]) != static_cast<const uint8_t*>(A[prev]) + a_prev * 2) return false;
      if (static_cast<const uint8_t*>(B[cur]) != static_cast<const uint8_t*>(B[prev]) + b_prev * 2) return false;
      if (dA[cur] != dA[prev] + a_prev) return false;
      if (dB[cur] != dB[prev] + b_prev) return false;
    }
  return true;
}

// Make sure buffer l % 2 holds layer l (copy only if it does not already).
sl_status ensure_layer(sl_stack* s, int l, uint64_t* h2d) {
  const int b = l % 2;
  if (s->buf_layer[b] == l) return SL_OK;
  SL_CHECK_CUDA(cudaStreamWaitEvent(s->copy_stream, s->freed[b], 0));
  SL_CHECK_CUDA(cudaMemcpyAsync(s->buf[b], s->host[l], s->blob_bytes, cudaMemcpyHostToDevice, s->copy_stream));
  SL_CHECK_CUDA(cudaEventRecord(s->ready[b], s->copy_stream));
  s->buf_layer[b] = l;
  *h2d += s->blob_bytes;
  return SL_OK;
}

}  // namespace

extern "C" sl_status sl_stack_blob_layout(int32_t kind, int64_t D, int64_t Dkv, int64_t F, size_t offsets[16],
                                          size_t* blob_bytes) {
  SL_REQUIRE(offsets && blob_bytes, "sl_stack_blob_layout: null output");
  SL_REQUIRE(kind == SL_WEIGHT_NF4 || kind == SL_WEIGHT_BF16 || kind == SL_WEIGHT_NF4_DQ,
             "sl_stack_blob_layout: unknown kind");
  SL_REQUIRE(D > 0 && Dkv > 0 && F > 0 && D % 256 == 0 && F % 256 == 0 && Dkv % 128 == 0 && D % Dkv == 0,
             "sl_stack_blob_layout: need D, F multiples of 256, Dkv a multiple of 128 dividing D");
  SL_REQUIRE(kind != SL_WEIGHT_NF4_DQ || Dkv % 256 == 0,
             "sl_stack_blob_layout: the double-quantised absmax needs Dkv a multiple of 256");
  return layout(kind, D, Dkv, F, offsets, blob_bytes, nullptr);
}

extern "C" sl_status sl_stack_dq_layout(int64_t D, int64_t Dkv, int64_t F, size_t q_off[7], int64_t q_ld[7],
                                        size_t a2_off[7], int64_t a2_ld[7], int64_t col0[7]) {
  SL_REQUIRE(q_off && q_ld && a2_off && a2_ld && col0, "sl_stack_dq_layout: null output");
  size_t offs[16], bytes = 0;
  sl_status st = sl_stack_blob_layout(SL_WEIGHT_NF4_DQ, D, Dkv, F, offs, &bytes);
  if (st != SL_OK) return st;
  DqLayout dq{};
  layout(SL_WEIGHT_NF4_DQ, D, Dkv, F, offs, &bytes, &dq);
  for (int i = 0; i < 7; ++i) {
    q_off[i] = dq.q[i];
    q_ld[i] = dq.q_ld[i];
    a2_off[i] = dq.a2[i];
    a2_ld[i] = dq.a2_ld[i];
    col0[i] = dq.col0[i];
  }
  return SL_OK;
}

extern "C" sl_status sl_stack_create(const sl_stack_desc* desc, sl_stack** out, size_t* host_bytes,
                                     size_t* buffer_bytes) {
  SL_REQUIRE(desc && out, "sl_stack_create: null argument");
  SL_REQUIRE(desc->L > 0 && desc->host_blobs, "sl_stack_create: need L > 0 and host_blobs");
  size_t offs[16], bytes = 0;
  sl_status st = sl_stack_blob_layout(desc->kind, desc->D, desc->Dkv, desc->F, offs, &bytes);
  if (st != SL_OK) return st;
  SL_REQUIRE(desc->mixer == SL_MIX_TOKEN_LOCAL || desc->mixer == SL_MIX_ATTENTION, "sl_stack_create: unknown mixer");
  SL_REQUIRE(desc->mixer != SL_MIX_ATTENTION ||
                 (desc->seq_len > 0 && desc->seq_len % 128 == 0 && desc->rope_theta > 1.0),
             "sl_stack_create: attention needs seq_len a positive multiple of 128 and rope_theta > 1");
  for (int l = 0; l < desc->L; ++l) {
    const void* p = desc->host_blobs[l];
    SL_REQUIRE(p, "sl_stack_create: null host blob");
    for (const void* q : {p, static_cast<const void*>(static_cast<const uint8_t*>(p) + bytes - 1)}) {
      cudaPointerAttributes at{};
      cudaError_t e = cudaPointerGetAttributes(&at, q);
      if (e != cudaSuccess || at.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return set_error(SL_ERR_INVALID, "sl_stack_create: host blob " + std::to_string(l) +
                                             " is not page-locked (pinned) host memory");
      }
    }
    if (desc->device_blobs) {
      cudaPointerAttributes at{};
      cudaError_t e = cudaPointerGetAttributes(&at, desc->device_blobs[l]);
      if (e != cudaSuccess || at.type != cudaMemoryTypeDevice) {
        cudaGetLastError();
        return set_error(SL_ERR_INVALID, "sl_stack_create: device blob " + std::to_string(l) +
                                             " is not device memory");
      }
    }
  }
  sl_stack* s = new sl_stack();
  s->L = desc->L;
  s->kind = desc->kind;
  s->D = desc->D;
  s->Dkv = desc->Dkv;
  s->F = desc->F;
  s->mixer = desc->mixer;
  s->seq_len = desc->seq_len;
  s->rope_theta = desc->rope_theta;
  s->host.assign(desc->host_blobs, desc->host_blobs + desc->L);
  if (desc->device_blobs) s->dev.assign(desc->device_blobs, desc->device_blobs + desc->L);
  std::memcpy(s->offs, offs, sizeof(offs));
  if (s->kind == SL_WEIGHT_NF4_DQ) {
    DqLayout dq{};
    layout(s->kind, s->D, s->Dkv, s->F, offs, &bytes, &dq);
    for (int i = 0; i < 7; ++i) {
      s->dq_q[i] = dq.q[i];
      s->dq_a2[i] = dq.a2[i];
      s->dq_qld[i] = dq.q_ld[i];
      s->dq_a2ld[i] = dq.a2_ld[i];
      s->dq_col0[i] = dq.col0[i];
    }
  }
  s->blob_bytes = bytes;
  cudaGetDevice(&s->device);
  auto fail = [&](cudaError_t e, const char* what) {
    sl_status r = cuda_error(e, what);
    sl_stack_destroy(s);
    return r;
  };
  cudaError_t e;
  for (int b = 0; b < 2; ++b) {
    if ((e = cudaMalloc(&s->buf[b], bytes)) != cudaSuccess) return fail(e, "sl_stack_create: cudaMalloc buffer");
    if ((e = cudaEventCreateWithFlags(&s->ready[b], cudaEventDisableTiming)) != cudaSuccess)
      return fail(e, "sl_stack_create: event");
    if ((e = cudaEventCreateWithFlags(&s->freed[b], cudaEventDisableTiming)) != cudaSuccess)
      return fail(e, "sl_stack_create: event");
  }
  if ((e = cudaStreamCreateWithFlags(&s->copy_stream, cudaStreamNonBlocking)) != cudaSuccess)
    return fail(e, "sl_stack_create: copy stream");
  int least = 0, greatest = 0;
  if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess)
    return fail(e, "sl_stack_create: stream priorities");
  if ((e = cudaStreamCreateWithPriority(&s->main_stream, cudaStreamNonBlocking, greatest)) != cudaSuccess)
    return fail(e, "sl_stack_create: main stream");
  cudaEvent_t* evs[10] = {&s->step_in, &s->step_out, &s->fork[0], &s->fork[1], &s->fork[2], &s->fork[3],
                          &s->done[0], &s->done[1], &s->done[2], &s->done[3]};
  for (cudaEvent_t* ev : evs)
    if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess)
      return fail(e, "sl_stack_create: event");
  if (host_bytes) *host_bytes = bytes * static_cast<size_t>(desc->L);
  if (buffer_bytes) *buffer_bytes = 2 * bytes;
  *out = s;
  return SL_OK;
}

extern "C" sl_status sl_stack_destroy(sl_stack* s) {
  if (!s) return SL_OK;
  if (s->copy_stream) cudaStreamSynchronize(s->copy_stream);
  for (int b = 0; b < 2; ++b) {
    if (s->freed[b]) cudaEventSynchronize(s->freed[b]);
    if (s->buf[b]) cudaFree(s->buf[b]);
    if (s->ready[b]) cudaEventDestroy(s->ready[b]);
    if (s->freed[b]) cudaEventDestroy(s->freed[b]);
  }
  if (s->copy_stream) cudaStreamDestroy(s->copy_stream);
  if (s->main_stream) {
    cudaStreamSynchronize(s->main_stream);
    cudaStreamDestroy(s->main_stream);
  }
  cudaEvent_t evs[10] = {s->step_in, s->step_out, s->fork[0], s->fork[1], s->fork[2], s->fork[3],
                         s->done[0], s->done[1], s->done[2], s->done[3]};
  for (cudaEvent_t ev : evs)
    if (ev) cudaEventDestroy(ev);
  delete s;
  return SL_OK;
}

extern "C" size_t sl_stack_workspace_size(const sl_stack* s, int64_t M, int32_t r) {
  if (!s || M <= 0) return 0;
  return make_plan(s, M, r).total;
}

namespace {

// Checks shared by the stack step and the SFT step.
sl_status check_step(const sl_stack* s, int32_t mode, int64_t M, int32_t r, const void* const* A,
                     const void* const* B, float* const* dA, float* const* dB, const void* ws) {
  SL_REQUIRE(s, "stack step: null stack");
  SL_REQUIRE(mode == SL_MODE_STREAMED || mode == SL_MODE_RESIDENT, "stack step: bad mode");
  SL_REQUIRE(mode == SL_MODE_STREAMED || !s->dev.empty(), "stack step: RESIDENT needs device_blobs");
  SL_REQUIRE(ws && M > 0, "stack step: null workspace or M <= 0");
  SL_REQUIRE(r == 0 || (A && B && dA && dB), "stack step: adapters and gradients required for r > 0");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255) == 0, "stack step: workspace must be 256-byte aligned");
  if (s->kind == SL_WEIGHT_NF4_DQ && M <= 128)
    return set_error(SL_ERR_UNSUPPORTED, "stack step: double-quantised stacks need M > 128");
  SL_REQUIRE(s->mixer != SL_MIX_ATTENTION || M % s->seq_len == 0,
             "stack step: attention needs M a multiple of the sequence length");
  int dev = 0;
  SL_CHECK_CUDA(cudaGetDevice(&dev));
  SL_REQUIRE(dev == s->device, "stack step: current device differs from the handle's");
  return SL_OK;
}

// The forward over layers 0..L-1 and the backward over L-1..0 of one step;
// the two layers resident at the turn are not copied again.
struct Runner {
  sl_stack* s;
  StepCtx& c;
  const Plan& P;
  bool streamed;
  uint64_t h2d = 0;

  const void* base_of(int l) const { return streamed ? s->buf[l % 2] : s->dev[l]; }
  const float* h_in(int l, const float* h0) const { return l == 0 ? h0 : c.at<float>(P.hin[l]); }

  sl_status forward(const float* h0, float* hL) {
    const int L = s->L;
    if (s->mixer == SL_MIX_ATTENTION)
      SL_TRY(rope_table(s->seq_len, s->rope_theta, c.at<float>(P.rope), c.stream));
    if (streamed) {
      SL_TRY(ensure_layer(s, 0, &h2d));
      if (L > 1) SL_TRY(ensure_layer(s, 1, &h2d));
    }
    sl_weight w[7];
    const float* norms[2];
    for (int l = 0; l < L; ++l) {
      if (streamed) SL_CHECK_CUDA(cudaStreamWaitEvent(c.stream, s->ready[l % 2], 0));
      weights_of(s, base_of(l), w, norms);
      float* out = (l == L - 1) ? hL : c.at<float>(P.hin[l + 1]);
      SL_TRY(layer_fwd(c, l, w, norms, h_in(l, h0), out));
      if (streamed) {
        SL_CHECK_CUDA(cudaEventRecord(s->freed[l % 2], c.stream));
        if (l + 2 < L) SL_TRY(ensure_layer(s, l + 2, &h2d));
      }
    }
    return SL_OK;
  }

  sl_status backward(const float* h0, const float* dh_top, float* dh0) {
    const int L = s->L;
    float* dhA = c.at<float>(P.dhA);
    float* dhB = c.at<float>(P.dhB);
    uint16_t* dd = c.at<uint16_t>(P.dd);
    SL_TRY(glue_to_bf16(dh_top, dd, c.M * s->D, c.stream));
    const float* dh_cur = dh_top;
    sl_weight w[7];
    const float* norms[2];
    for (int l = L - 1; l >= 0; --l) {
      if (streamed) {
        SL_TRY(ensure_layer(s, l, &h2d));
        SL_CHECK_CUDA(cudaStreamWaitEvent(c.stream, s->ready[l % 2], 0));
      }
      weights_of(s, base_of(l), w, norms);
      float* dh_next = (l == 0) ? dh0 : ((dh_cur == dhA) ? dhB : dhA);
      SL_TRY(layer_bwd(c, l, w, norms, h_in(l, h0), dh_cur, dd, dh_next, l == 0 ? nullptr : dd));
      dh_cur = dh_next;
      if (streamed) {
        SL_CHECK_CUDA(cudaEventRecord(s->freed[l % 2], c.stream));
        if (l - 2 >= 0) SL_TRY(ensure_layer(s, l - 2, &h2d));
      }
    }
    return SL_OK;
  }
};

// Regions of the SFT step's workspace after the stack plan.
struct SftPlan {
  size_t h0, hL, xf, rstd, dX, dh_top, dh0, ce_ws, total;
  size_t ce_bytes;
};

SftPlan make_sft_plan(const Plan& P, int64_t M, int64_t D, int64_t V, int64_t chunk_V) {
  SftPlan S{};
  size_t off = P.total;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t MD = static_cast<size_t>(M) * D;
  S.h0 = take(MD * 4);
  S.hL = take(MD * 4);
  S.xf = take(MD * 2);
  S.rstd = take(M * 4);
  S.dX = take(MD * 4);
  S.dh_top = take(MD * 4);
  S.dh0 = take(MD * 4);
  S.ce_bytes = sl_ce_workspace_size(M, D, V, chunk_V);
  S.ce_ws = take(S.ce_bytes ? S.ce_bytes : 256);
  S.total = off;
  return S;
}

// The step's main stream starts after the caller's stream has reached the
// call, and the caller's stream continues after the main stream's last
// kernel (its own queue already holds every adapter-gradient pass).
sl_status join_in(sl_stack* s, cudaStream_t caller) {
  SL_CHECK_CUDA(cudaEventRecord(s->step_in, caller));
  SL_CHECK_CUDA(cudaStreamWaitEvent(s->main_stream, s->step_in, 0));
  return SL_OK;
}
sl_status join_out(sl_stack* s, cudaStream_t caller) {
  SL_CHECK_CUDA(cudaEventRecord(s->step_out, s->main_stream));
  SL_CHECK_CUDA(cudaStreamWaitEvent(caller, s->step_out, 0));
  return SL_OK;
}

sl_status sft_body(StepCtx& c, Runner& run, const SftPlan& S, const int32_t* tokens, const int32_t* labels,
                          int64_t M, const void* embed, int64_t V, const float* norm_final, const void* W_head,
                          int64_t chunk_V, float* loss, int* err) {
  const sl_stack* s = c.s;
  const int D = static_cast<int>(s->D);
  cudaStream_t stream = c.stream;
  float* h0 = c.at<float>(S.h0);
  float* hL = c.at<float>(S.hL);
  uint16_t* xf = c.at<uint16_t>(S.xf);
  float* rstd = c.at<float>(S.rstd);
  float* dX = c.at<float>(S.dX);
  float* dh_top = c.at<float>(S.dh_top);
  SL_TRY(glue_embed(tokens, static_cast<const uint16_t*>(embed), V, h0, M, D, err, stream));
  SL_TRY(run.forward(h0, hL));
  SL_TRY(glue_rms_fwd(hL, nullptr, nullptr, xf, rstd, norm_final, M, D, stream));
  SL_TRY(sl_ce_fwd_bwd(xf, M, D, W_head, V, labels, -100, chunk_V, loss, dX, c.at<uint8_t>(S.ce_ws), S.ce_bytes,
                       stream));
  SL_TRY(glue_rms_bwd(nullptr, nullptr, nullptr, nullptr, dX, hL, rstd, norm_final, dh_top, nullptr, M, D, stream));
  return run.backward(h0, dh_top, c.at<float>(S.dh0));
}

}  // namespace

extern "C" sl_status sl_stream_stack_step(sl_stack* s, int32_t mode, const float* h0, int64_t M,
                                          const float* dh_top, const void* const* A, const void* const* B,
                                          int32_t r, float alpha, float* hL, float* dh0, float* const* dA,
                                          float* const* dB, int32_t accumulate, void* ws, size_t ws_bytes,
                                          cudaStream_t stream) {
  sl_status st = check_step(s, mode, M, r, A, B, dA, dB, ws);
  if (st != SL_OK) return st;
  SL_REQUIRE(h0 && dh_top && hL && dh0, "sl_stream_stack_step: null argument");
  const Plan P = make_plan(s, M, r);
  SL_REQUIRE(ws_bytes >= P.total, "sl_stream_stack_step: workspace too small (need " + std::to_string(P.total) +
                                      " bytes)");
  StepCtx c{s, &P, static_cast<uint8_t*>(ws), M, r, alpha, A, B, dA, dB, s->main_stream, stream};
  c.accumulate = accumulate ? 1 : 0;
  c.group_qkv = can_group(s, M, r, 0, 3, A, B, dA, dB);
  c.group_gu = can_group(s, M, r, 4, 2, A, B, dA, dB);
  const uint64_t launches0 = launch_count();
  Runner run{s, c, P, mode == SL_MODE_STREAMED};
  SL_TRY(join_in(s, stream));
  const sl_status st1 = run.forward(h0, hL);
  const sl_status st2 = st1 == SL_OK ? run.backward(h0, dh_top, dh0) : st1;
  SL_TRY(join_out(s, stream));
  SL_TRY(st2);
  s->last_h2d = run.h2d;
  s->last_kernels = launch_count() - launches0;
  return SL_OK;
}

extern "C" size_t sl_sft_workspace_size(const sl_stack* s, int64_t M, int32_t r, int64_t V, int64_t chunk_V) {
  if (!s || M <= 0 || V <= 0 || chunk_V <= 0) return 0;
  return make_sft_plan(make_plan(s, M, r), M, s->D, V, chunk_V).total;
}

extern "C" sl_status sl_sft_step(sl_stack* s, int32_t mode, const int32_t* tokens, const int32_t* labels, int64_t M,
                                 const void* embed, int64_t V, const float* norm_final, const void* W_head,
                                 int64_t chunk_V, const void* const* A, const void* const* B, int32_t r, float alpha,
                                 float* loss, float* const* dA, float* const* dB, int32_t accumulate, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  sl_status st = check_step(s, mode, M, r, A, B, dA, dB, ws);
  if (st != SL_OK) return st;
  SL_REQUIRE(tokens && labels && embed && W_head && loss && V > 0, "sl_sft_step: null argument");
  const Plan P = make_plan(s, M, r);
  const SftPlan S = make_sft_plan(P, M, s->D, V, chunk_V);
  SL_REQUIRE(ws_bytes >= S.total, "sl_sft_step: workspace too small (need " + std::to_string(S.total) + " bytes)");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  StepCtx c{s, &P, static_cast<uint8_t*>(ws), M, r, alpha, A, B, dA, dB, s->main_stream, stream};
  c.accumulate = accumulate ? 1 : 0;
  c.group_qkv = can_group(s, M, r, 0, 3, A, B, dA, dB);
  c.group_gu = can_group(s, M, r, 4, 2, A, B, dA, dB);
  const uint64_t launches0 = launch_count();
  Runner run{s, c, P, mode == SL_MODE_STREAMED};
  SL_TRY(join_in(s, stream));
  const sl_status st1 = sft_body(c, run, S, tokens, labels, M, embed, V, norm_final, W_head, chunk_V, loss, err);
  SL_TRY(join_out(s, stream));
  SL_TRY(st1);
  s->last_h2d = run.h2d;
  s->last_kernels = launch_count() - launches0;
  return SL_OK;
}

extern "C" sl_status sl_stack_last_step_stats(const sl_stack* s, uint64_t* h2d_bytes, uint64_t* kernels) {
  SL_REQUIRE(s, "sl_stack_last_step_stats: null stack");
  if (h2d_bytes) *h2d_bytes = s->last_h2d;
  if (kernels) *kernels = s->last_kernels;
  return SL_OK;
}
