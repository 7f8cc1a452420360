// The rank-r side products of the LoRA linear on the tensor cores.
//
// "Exact Layer Streaming ..." (abstract) trains only A [r, K] and B [N, r]
// beside a frozen base; around the fused base GEMM four skinny products
// remain, each one pass over a large bf16 operand Q:
//   forward   T  = X A^T          [M, r]   reduce over K     (mode kSkKA)
//   backward  U  = dY B           [M, r]   reduce over N     (mode kSkKB)
//             dA = s U^T X        [r, K]   reduce over M     (mode kSkM)
//             dB = s dY^T T       [N, r]   reduce over M     (mode kSkM)
// A group of G adapters whose projections read the same input (q, k, v or
// gate, up of a decoder layer) is done in the same four passes, with the
// adapters stored back to back (A_cat [G r, K], B_cat [sum N_g, r], output
// columns concatenated): T_cat = X A_cat^T, U_cat = dY_cat blockdiag(B_g),
// dA_cat = s U_cat^T X, and dB_cat, whose rows in projection g use the
// columns g r .. g r + r - 1 of T_cat.
// These are HBM-bound streams (2r FLOP per element of Q); on the CUDA cores
// the FMAs alone would outlast the read, so each pass runs tcgen05 MMAs with
// a narrow N over TMA-staged steps of Q:
//   * mode K: D[128 rows of Q, n] += Q[128 x step] * W[n x step]^T; W = A_cat
//     is TMA-loaded directly (K-major), W = blockdiag(B_g)^T is transposed
//     from a raw TMA tile of B_cat by four converter warps;
//   * mode M: D[128 columns of Q, n] += Q^T[128 x step] * P'[n x step]^T, Q^T
//     read MN-major straight from the TMA tile and P' = [P_hi ; P_lo] the
//     two-term bf16 split of the fp32 operand (U or T) written by the
//     converter warps (hi in D columns 0.., lo from the next multiple of 32), so
//     D = Q^T P to fp32 accuracy.
// One variant fuses the SwiGLU backward into the U pass that reads its
// output, so dY of the gate/up group is written once and never read back
// (GLUE = 2, mode K with blockdiag(B)^T): dg = dm u s (1 + g (1 - s)) and
// du = dm g s (s = sigmoid(g)) from dm, g, u tiles, each step 64 columns of
// dg followed by the same 64 columns of du, and U = [dg | du]
// blockdiag(B_g, B_u).  Sixteen converter warps compute the glue from the
// TMA-staged inputs in the same 128-byte-swizzled positions, write it over
// the u and g tiles (which become the MMA operand) and store it to global
// memory; the arithmetic is glue.cu's, expression for expression, so dg and
// du are bitwise the elementwise kernel's.  (The same fusion of the forward,
// m = SiLU(g) u with the down adapter's T = m A^T, measured slower than the
// two separate kernels: 28.9 against 12.1 + 11.4 us at M = 1024, F = 14336,
// and is not built.)
// The long reduction is split over the CTAs of a thread-block cluster (up to
// 16, sized so that the grid is one wave); their fp32 partials are summed
// through distributed shared memory in rank order, so one launch writes the
// final result with no partial buffers in global memory and bitwise
// reproducible sums.  Every wait is bounded.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "skinny.cuh"
#include "timing.cuh"
#include "tmap.cuh"

namespace sl {

enum SkMode { kSkKA = 0, kSkKB = 1, kSkM = 2 };

// warp 0 TMA, warp 1 MMA, warps 2..5 converters + epilogue; the fused
// SwiGLU backward adds twelve converter warps for the glue arithmetic
constexpr int kSkThreads = 192;
__host__ __device__ constexpr int sk_threads(int glue) { return glue == 2 ? 64 + 512 : kSkThreads; }
constexpr int kSkMaxStages = 8;
constexpr int kSkTmemCols = 128;
constexpr int kSkBarBytes = 1024; // barriers + misc, ahead of the 1024-aligned data
constexpr int kSkSmemBudget = 227 * 1024 - 1024 - kSkBarBytes;
constexpr int kSkRedLd = 68;      // fp32 partial row stride (64 columns + pad)

struct SkArgs {
  int M;           // rows of Q
  int C;           // columns of Q
  int r;           // adapter rank (multiple of 8, <= 32)
  int R;           // G r: mode K output columns; mode M row stride of P
  int rout;        // mode M: result columns per column of Q (R for dA, r for dB)
  int select;      // mode M: use P columns [g r, g r + r) of the column block's group g
  int G;           // adapters in the group (<= kSkMaxGroups)
  int bounds[kSkMaxGroups + 1];  // group g covers columns [bounds[g], bounds[g+1]) of Q (multiples of 128)
  int step;        // reduced elements per pipeline step: 64 or 128
  int nsteps;      // steps of the reduced extent (C in mode K, M in mode M)
  int stages;      // pipeline depth (<= kSkMaxStages), sized to the shared memory
  float s;         // output scale (mode M)
  int transpose;   // mode M: out[i * C + c] (dA) instead of out[c * rout + i] (dB)
  int accumulate;  // mode M: out += result
  float* out;
  int* err;
  uint16_t* glue0;  // GLUE 2: dg
  uint16_t* glue1;  // GLUE 2: du
  int64_t glue_ld;  // row stride of glue0 / glue1 (elements)
  int F;            // GLUE 2: columns of dg (= of du); C = 2 F
  int nb0;          // GLUE 3: blocks of the first pass (the rest run the second)
};

// Mode M: first D column of the lo half (32-aligned, so TMEM loads of
// result columns c .. c+31 and lo_col + c .. stay aligned).
__host__ __device__ inline int sk_lo_col(int rout) { return (rout + 31) / 32 * 32; }
// MMA N and the per-stage bytes of the three shared-memory regions.
__host__ __device__ inline int sk_n_mma(int mode, int R, int rout) {
  return mode == kSkM ? sk_lo_col(rout) + (rout + 15) / 16 * 16 : (R + 15) / 16 * 16;
}
__host__ __device__ inline int sk_q_bytes(int step) { return 128 * step * 2; }
__host__ __device__ inline int sk_op_bytes(int mode, int R, int rout, int step) {
  return sk_n_mma(mode, R, rout) * step * 2;
}
__host__ __device__ inline int sk_raw_bytes(int mode, int r, int rout, int step, int glue = 0) {
  if (glue == 2) return sk_q_bytes(64) + step * r * 2;     // the dm tile + B_g, B_u rows of the step
  return mode == kSkKA ? 0 : (mode == kSkKB ? step * r * 2 : step * rout * 4);
}
__host__ __device__ inline int sk_stage_bytes(int mode, int r, int R, int rout, int step, int glue = 0) {
  return sk_q_bytes(step) + sk_op_bytes(mode, R, rout, step) + sk_raw_bytes(mode, r, rout, step, glue);
}

__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr));
  return v;
}

__device__ __forceinline__ uint4* sw128_chunk(uint8_t* tile, int row, int chunk) {
  return reinterpret_cast<uint4*>(tile + row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Adapter of column `col` of Q (constant indices: the bounds stay in registers).
__device__ __forceinline__ int group_of(const SkArgs& a, int col) {
  int g = 0;
  if (a.G > 1 && col >= a.bounds[1]) g = 1;
  if (a.G > 2 && col >= a.bounds[2]) g = 2;
  if (a.G > 3 && col >= a.bounds[3]) g = 3;
  return g;
}

// The logistic function as glue.cu computes it (fast exponential and
// division: the IEEE division dominated the fused kernels' time).
__device__ __forceinline__ float sk_sigmoid(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = bf16_lo(w[e]);
    f[2 * e + 1] = bf16_hi(w[e]);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// GLUE: 0 plain pass over a TMA-loaded Q; 2 the fused SwiGLU backward
// (map_q: dm, map_x1: g, map_x2: u); 3 two mode-M passes in one launch (dA
// and dB of one backward): the blocks from a0.nb0 on run the second with
// map_x1, map_x2 and a1.
template <int MODE, int GLUE>
__global__ void __launch_bounds__(sk_threads(GLUE), 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_w,
                  const __grid_constant__ CUtensorMap map_x1, const __grid_constant__ CUtensorMap map_x2,
                  const SkArgs a0, const SkArgs a1) {
  static_assert(GLUE == 0 || (GLUE == 2 && MODE == kSkKB) || (GLUE == 3 && MODE == kSkM),
                "skinny_kernel glue");
  const bool second = GLUE == 3 && static_cast<int>(blockIdx.x) >= a0.nb0;
  const SkArgs& a = second ? a1 : a0;
  const CUtensorMap* mq = second ? &map_x1 : &map_q;
  const CUtensorMap* mw = second ? &map_x2 : &map_w;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = ptx::align1024(smem_raw);
  const int r = a.r;
  const int S = a.stages;
  const int step = a.step;
  const int nh = step / 64;  // 64-wide halves of a step
  const int n_mma = sk_n_mma(MODE, a.R, a.rout);
  const int op_half = n_mma * 128;  // one 64-wide K chunk of the skinny operand
  const int q_bytes = sk_q_bytes(step);
  const int op_bytes = sk_op_bytes(MODE, a.R, a.rout, step);
  const int raw_bytes = sk_raw_bytes(MODE, r, a.rout, step, GLUE);
  const int ncols = MODE == kSkM ? a.rout : a.R;  // result columns per row of the accumulator
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* full = bars;                      // TMA bytes of the stage landed
  uint64_t* conv = bars + kSkMaxStages;       // converter warps wrote the stage's skinny operand
  uint64_t* empty = bars + 2 * kSkMaxStages;  // MMAs of the stage completed
  uint64_t* acc_full = bars + 3 * kSkMaxStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 516);
  uint8_t* sQ = smem + kSkBarBytes;
  uint8_t* sOp = sQ + S * q_bytes;
  uint8_t* sRaw = sOp + S * op_bytes;
  float* red = reinterpret_cast<float*>(sQ);  // fp32 partial [128][kSkRedLd] after the main loop

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int cs = static_cast<int>(gridDim.y);  // cluster = the CTAs of one blockIdx.x
  const int rank = static_cast<int>(blockIdx.y);
  const int s0 = static_cast<int>(static_cast<int64_t>(a.nsteps) * rank / cs);
  const int s1 = static_cast<int>(static_cast<int64_t>(a.nsteps) * (rank + 1) / cs);
  const int nloc = s1 - s0;
  // rows of Q (mode K) or columns of Q (mode M)
  const int base = (static_cast<int>(blockIdx.x) - (second ? a0.nb0 : 0)) * 128;
  // mode M with select: this column block's adapter g reads P columns g r ..
  const int p_col0 = (MODE == kSkM && a.select) ? group_of(a, base) * r : 0;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&conv[i], (sk_threads(GLUE) - 64) / 32);
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(acc_full, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(mq);
    ptx::tma_prefetch_desc(mw);
    if (GLUE == 2) {
      ptx::tma_prefetch_desc(&map_x1);
      ptx::tma_prefetch_desc(&map_x2);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, kSkTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();  // the next kernel may start its prologue
  pdl_wait();     // the previous kernel's writes are visible from here on

  auto give_up = [&]() {
    *abort_flag = 1;
    report_device_error(a.err, SL_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t tx = q_bytes + (MODE == kSkKA ? nh * op_half : 0) + raw_bytes;
      int j = 0;
      for (; j < nloc; ++j) {
        const int st = j % S;
        if (!ptx::mbar_wait(&empty[st], ((j / S) & 1) ^ 1, abort_flag)) {
          give_up();
          break;
        }
        const int k0 = (s0 + j) * step;
        uint8_t* q = sQ + st * q_bytes;
        ptx::mbar_arrive_expect_tx(&full[st], tx);
        if (GLUE == 2) {  // step j: columns c .. c+63 of dg then du; u / g tiles become dg / du
          const int c = (s0 + j) * 64;
          uint8_t* raw = sRaw + st * raw_bytes;
          ptx::tma_load_2d(q, &map_x2, &full[st], c, base);
          ptx::tma_load_2d(q + 16384, &map_x1, &full[st], c, base);
          ptx::tma_load_2d(raw, &map_q, &full[st], c, base);
          ptx::tma_load_2d(raw + 16384, &map_w, &full[st], 0, c);
          ptx::tma_load_2d(raw + 16384 + 64 * r * 2, &map_w, &full[st], 0, a.F + c);
        } else if (MODE != kSkM) {  // Q [128 rows x step], 64-wide halves 16 KB apart
          for (int h = 0; h < nh; ++h) ptx::tma_load_2d(q + h * 16384, mq, &full[st], k0 + 64 * h, base);
          if (MODE == kSkKA)
            for (int h = 0; h < nh; ++h)
              ptx::tma_load_2d(sOp + st * op_bytes + h * op_half, mw, &full[st], k0 + 64 * h, 0);
          else
            ptx::tma_load_2d(sRaw + st * raw_bytes, mw, &full[st], 0, k0);
        } else {  // Q rows k0 .. k0+step-1, columns base .. base+127 (two 64-column atoms); raw P rows
          ptx::tma_load_2d(q, mq, &full[st], base, k0);
          ptx::tma_load_2d(q + step * 128, mq, &full[st], base + 64, k0);
          ptx::tma_load_2d(sRaw + st * raw_bytes, mw, &full[st], p_col0, k0);
        }
      }
      if (*abort_flag)
        for (int k = (j > S ? j - S : 0); k < j; ++k) ptx::mbar_wait(&full[k % S], (k / S) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16(128, static_cast<uint32_t>(n_mma), MODE == kSkM ? 1 : 0, 0);
      const uint32_t q_base = ptx::smem_addr(sQ);
      const uint32_t op_base = ptx::smem_addr(sOp);
      for (int j = 0; j < nloc; ++j) {
        const int st = j % S;
        const uint32_t ph = (j / S) & 1;
        if (!ptx::mbar_wait(&full[st], ph, abort_flag) ||
            (MODE != kSkKA && !ptx::mbar_wait(&conv[st], ph, abort_flag))) {
          give_up();
          break;
        }
        ptx::tc_fence_after();
        const uint32_t qs = q_base + st * q_bytes;
        const uint32_t os = op_base + st * op_bytes;
        for (int kk = 0; kk < step / 16; ++kk) {
          const int h = kk >> 2, k4 = kk & 3;
          // mode K: A = Q K-major, half h at +16 KB; mode M: A = Q^T MN-major,
          // 16 reduced rows (2 KB) per k16 step, the two 64-column atoms step * 128 B apart
          const uint64_t ad = MODE == kSkM ? ptx::smem_desc(qs + kk * 2048, step * 128, 1024, 2)
                                           : ptx::smem_desc(qs + h * 16384 + k4 * 32, 16, 1024, 2);
          const uint64_t bd = ptx::smem_desc(os + h * op_half + k4 * 32, 16, 1024, 2);
          ptx::mma_bf16(tmem, ad, bd, idesc, (j | kk) ? 1u : 0u);
        }
        ptx::mma_commit(&empty[st]);
      }
      ptx::mma_commit(acc_full);
    }
  } else {
    // ------------------------------------ converters (modes KB, M), then epilogue
    const int e = tid - 64;  // 0 .. NT-1
    constexpr int NT = sk_threads(GLUE) - 64;
    if (MODE != kSkKA) {
      for (int j = 0; j < nloc; ++j) {
        const int st = j % S;
        if (!ptx::mbar_wait(&full[st], (j / S) & 1, abort_flag)) {
          give_up();
          break;
        }
        uint8_t* op = sOp + st * op_bytes;
        uint8_t* raw = sRaw + st * raw_bytes;
        uint8_t* q = sQ + st * q_bytes;
        const int nch = step / 8;  // 8-element chunks of the step
        if (GLUE == 2) {
          // dg over the u tile (K half 0), du over the g tile (K half 1)
          const int c = (s0 + j) * 64;
          for (int task = e; task < 128 * 8; task += NT) {
            const int row = task >> 3, c8 = task & 7;
            const int off = row * 128 + ((c8 ^ (row & 7)) << 4);
            float fdm[8], fg[8], fu[8], odg[8], odu[8];
            unpack8(*reinterpret_cast<const uint4*>(raw + off), fdm);
            unpack8(*reinterpret_cast<const uint4*>(q + 16384 + off), fg);
            unpack8(*reinterpret_cast<const uint4*>(q + off), fu);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float sg = sk_sigmoid(fg[i]);
              odg[i] = fdm[i] * fu[i] * sg * (1.0f + fg[i] * (1.0f - sg));
              odu[i] = fdm[i] * fg[i] * sg;
            }
            const uint4 vg = pack8(odg), vu = pack8(odu);
            *reinterpret_cast<uint4*>(q + off) = vg;
            *reinterpret_cast<uint4*>(q + 16384 + off) = vu;
            const int64_t gm = base + row;
            const int col = c + c8 * 8;
            if (gm < a.M && col < a.F) {
              *reinterpret_cast<uint4*>(a.glue0 + gm * a.glue_ld + col) = vg;
              *reinterpret_cast<uint4*>(a.glue1 + gm * a.glue_ld + col) = vu;
            }
          }
          // operand rows i (K half 0) = B_g[c + k][i], rows r + i (K half 1) = B_u[c + k][i]; zero elsewhere
          const uint16_t* rb = reinterpret_cast<const uint16_t*>(raw + 16384);
          for (int task = e; task < n_mma * 16; task += NT) {
            const int row = task % n_mma, ch = task / n_mma, h = ch >> 3;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            const int i = row - h * r;
            if (i >= 0 && i < r) {
              const uint16_t* pb = rb + h * 64 * r + ((ch & 7) * 8) * r + i;
#pragma unroll
              for (int qq = 0; qq < 4; ++qq)
                w[qq] = static_cast<uint32_t>(pb[(2 * qq) * r]) | (static_cast<uint32_t>(pb[(2 * qq + 1) * r]) << 16);
            }
            *sw128_chunk(op + h * op_half, row, ch & 7) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else if (MODE == kSkKB) {
          // raw: B_cat rows k0 .. k0+step-1 (r bf16 each), all of group g;
          // operand rows g r + i = B[k][i], every other row zero
          const int g0 = group_of(a, (s0 + j) * step) * r;
          const uint16_t* rb = reinterpret_cast<const uint16_t*>(raw);
          for (int task = e; task < n_mma * nch; task += 128) {
            const int row = task % n_mma, ch = task / n_mma;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            const int i = row - g0;
            if (i >= 0 && i < r) {
              const uint16_t* p = rb + (ch * 8) * r + i;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                w[q] = static_cast<uint32_t>(p[(2 * q) * r]) | (static_cast<uint32_t>(p[(2 * q + 1) * r]) << 16);
            }
            *sw128_chunk(op + (ch >> 3) * op_half, row, ch & 7) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          // raw: P rows k0 .. k0+step-1, rout fp32 each -> rows i (hi) and lo_col + i (lo)
          const int ro = a.rout;
          const int lo_col = sk_lo_col(ro);
          const float* rf = reinterpret_cast<const float*>(raw);
          for (int task = e; task < ro * nch; task += 128) {
            const int i = task % ro, ch = task / ro;  // i fastest: a warp reads consecutive words
            const float* p = rf + (ch * 8) * ro + i;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float v0 = p[(2 * q) * ro], v1 = p[(2 * q + 1) * ro];
              hi[q] = pack_bf16x2(v0, v1);
              lo[q] = pack_bf16x2(v0 - bf16_lo(hi[q]), v1 - bf16_hi(hi[q]));
            }
            uint8_t* oh = op + (ch >> 3) * op_half;
            *sw128_chunk(oh, i, ch & 7) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *sw128_chunk(oh, lo_col + i, ch & 7) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&conv[st]);
      }
    }
    // epilogue (warps 2..5): TMEM lane `row` holds this CTA's partial for
    // row `row` of the 128 block; result columns are read 32 at a time
    // (mode M adds the lo half from column lo_col + c)
    if (warp < 6) {
    bool ready = ptx::mbar_wait(acc_full, 0, abort_flag) && !*abort_flag;
    ready = __all_sync(0xffffffffu, ready);
    if (!ready && !*abort_flag) give_up();
    ptx::tc_fence_after();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const bool keep = ready && nloc > 0;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    for (int c0 = 0; c0 < ncols; c0 += 32) {
      float v[32];
      {
        uint32_t u[32];
        ptx::tmem_ld_32x32b_x32(lane_addr + c0, u);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = keep ? __uint_as_float(u[c]) : 0.0f;
        if (MODE == kSkM) {
          ptx::tmem_ld_32x32b_x32(lane_addr + sk_lo_col(a.rout) + c0, u);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] += keep ? __uint_as_float(u[c]) : 0.0f;
        }
      }
      const int nc = ncols - c0 < 32 ? ncols - c0 : 32;  // a multiple of 8
      if (cs == 1) {
        // the whole reduction ran here: write straight from registers
        if (MODE != kSkM) {
          const int gm = base + row;
          if (gm < a.M)
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4)
              if (i4 * 4 < nc)
                *reinterpret_cast<float4*>(a.out + static_cast<int64_t>(gm) * a.R + c0 + i4 * 4) =
                    make_float4(v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2], v[4 * i4 + 3]);
        } else {
          const int gc = base + row;
          if (gc < a.C) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (i >= nc) break;
              float* o = a.transpose ? a.out + static_cast<int64_t>(c0 + i) * a.C + gc
                                     : a.out + static_cast<int64_t>(gc) * a.rout + c0 + i;
              const float x = v[i] * a.s;
              *o = a.accumulate ? *o + x : x;
            }
          }
        }
      } else {
        float* dst = red + row * kSkRedLd + c0;
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4)
          if (i4 * 4 < nc)
            *reinterpret_cast<float4*>(dst + i4 * 4) = make_float4(v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2], v[4 * i4 + 3]);
      }
    }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (cs > 1) {
    ptx::cluster_sync();  // every CTA's partial is in its shared memory
    // This CTA writes rows [rank * 128 / cs, (rank + 1) * 128 / cs) of the
    // 128-row block: partials summed over the cluster in rank order, four
    // result columns per task, all ranks' loads in flight at once.
    const int r0 = rank * 128 / cs, nrows = (rank + 1) * 128 / cs - r0;
    const int nq = ncols / 4;
    const bool by_col = MODE == kSkM && a.transpose;  // dA: rows vary fastest for coalesced stores
    for (int task = tid; task < nrows * nq; task += sk_threads(GLUE)) {
      const int rl = by_col ? task % nrows : task / nq;
      const int i4 = by_col ? task / nrows : task % nq;
      const int row = r0 + rl;
      const uint32_t own = ptx::smem_addr(red + row * kSkRedLd + i4 * 4);
      float4 h[16];
#pragma unroll
      for (int p = 0; p < 16; ++p) {
        if (p < cs) {
          uint32_t src;
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(src) : "r"(own), "r"(p));
          h[p] = ld_dsmem_f32x4(src);
        }
      }
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int p = 0; p < 16; ++p) {
        if (p < cs) {
          acc.x += h[p].x; acc.y += h[p].y; acc.z += h[p].z; acc.w += h[p].w;
        }
      }
      if (MODE != kSkM) {
        const int gm = base + row;
        if (gm < a.M) *reinterpret_cast<float4*>(a.out + static_cast<int64_t>(gm) * a.R + i4 * 4) = acc;
      } else {
        const int gc = base + row;
        if (gc < a.C) {
          const float x[4] = {acc.x * a.s, acc.y * a.s, acc.z * a.s, acc.w * a.s};
          if (!a.transpose) {
            float4* o = reinterpret_cast<float4*>(a.out + static_cast<int64_t>(gc) * a.rout + i4 * 4);
            float4 v4 = make_float4(x[0], x[1], x[2], x[3]);
            if (a.accumulate) {
              const float4 old = *o;
              v4.x += old.x; v4.y += old.y; v4.z += old.z; v4.w += old.w;
            }
            *o = v4;
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float* o = a.out + static_cast<int64_t>(i4 * 4 + k) * a.C + gc;
              *o = a.accumulate ? *o + x[k] : x[k];
            }
          }
        }
      }
    }
    ptx::cluster_sync();  // no CTA leaves while a peer may still read its partial
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kSkTmemCols);
  }
}

// ------------------------------------------------------------------ host side
namespace {

// Step width and pipeline depth: the pair with the most Q bytes in flight
// (the fused SwiGLU backward's paired steps are 128 wide).
void choose_pipeline(int mode, int r, int R, int rout, SkArgs& a, int glue = 0) {
  int best = -1;
  for (int step : {128, 64}) {
    if (glue == 2 && step != 128) continue;
    const int s = std::min(kSkMaxStages, kSkSmemBudget / sk_stage_bytes(mode, r, R, rout, step, glue));
    if (s >= 2 && s * sk_q_bytes(step) > best) {
      best = s * sk_q_bytes(step);
      a.step = step;
      a.stages = s;
    }
  }
}

template <int MODE, int GLUE>
sl_status set_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(skinny_kernel<MODE, GLUE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(skinny_kernel<MODE, GLUE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  return err == cudaSuccess ? SL_OK : cuda_error(err, "skinny_kernel attributes");
}

template <int MODE, int GLUE>
cudaLaunchConfig_t make_config(int64_t blocks, int cs, const SkArgs& a, cudaStream_t stream,
                               cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(cs), 1);
  cfg.blockDim = dim3(sk_threads(GLUE), 1, 1);
  cfg.dynamicSmemBytes =
      static_cast<size_t>(1024 + kSkBarBytes + a.stages * sk_stage_bytes(MODE, a.r, a.R, a.rout, a.step, GLUE));
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of `cs` CTAs that the device can hold at once for this shared-
// memory size (driver query, cached per device, size and cluster size).
template <int MODE, int GLUE>
int max_active_clusters(int cs, const SkArgs& a) {
  static std::mutex mu;
  static int cache[64][64][17];  // [device][smem / 4 KB][cs], 0 = not yet asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_config<MODE, GLUE>(1, cs, a, nullptr, attr);
  const int key = static_cast<int>(cfg.dynamicSmemBytes / 4096) & 63;
  std::lock_guard<std::mutex> lk(mu);
  int& slot = cache[dev][key][cs];
  if (slot == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, skinny_kernel<MODE, GLUE>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    slot = n > 0 ? n : -1;
  }
  return slot;
}

// Cluster size: the largest split of the reduction (at least two steps per
// CTA) whose clusters all fit on the device at once, so that the launch is
// one wave of at most one CTA per SM.
template <int MODE, int GLUE>
int choose_split(int64_t blocks, const SkArgs& a) {
  for (int cs = 16; cs > 1; --cs) {
    if (blocks * cs > num_sms() || a.nsteps < 2 * cs) continue;
    if (max_active_clusters<MODE, GLUE>(cs, a) >= blocks) return cs;
  }
  return 1;
}

// Algorithmic bytes of one pass: Q once, the skinny operand once, the output
// written (and read too when accumulating).
double pass_bytes(int mode, const SkArgs& a) {
  const double q = 2.0 * a.M * static_cast<double>(a.C);
  if (mode != kSkM) return q + (mode == kSkKA ? 2.0 * a.R * a.C : 2.0 * a.r * a.C) + 4.0 * a.M * a.R;
  return q + 4.0 * a.M * a.rout + 4.0 * a.C * a.rout * (a.accumulate ? 2 : 1);
}

template <int MODE, int GLUE = 0>
sl_status launch(const CUtensorMap& mq, const CUtensorMap& mw, const SkArgs& a, int64_t blocks,
                 cudaStream_t stream, const CUtensorMap* mx1 = nullptr, const CUtensorMap* mx2 = nullptr,
                 double bytes = 0.0, const SkArgs* a2 = nullptr) {
  sl_status st = set_attributes<MODE, GLUE>();
  if (st != SL_OK) return st;
  const int cs = choose_split<MODE, GLUE>(blocks, a);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_config<MODE, GLUE>(blocks, cs, a, stream, attr);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_trigger / pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  const TimingToken tt =
      timing_begin(MODE == kSkKA ? 6 : (MODE == kSkKB ? 7 : 8), GLUE ? bytes : pass_bytes(MODE, a), stream);
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, skinny_kernel<MODE, GLUE>, mq, mw, mx1 ? *mx1 : mq, mx2 ? *mx2 : mq, a, a2 ? *a2 : a);
  timing_end(tt, stream);
  if (e != cudaSuccess) return cuda_error(e, "skinny_kernel launch");
  return check_launch("skinny_kernel");
}

// Two mode-M passes in one launch: `q` sizes the launch (shared memory,
// cluster split); each block runs its own pass's arguments.
sl_status launch_pair(const CUtensorMap& mq0, const CUtensorMap& mw0, const CUtensorMap& mq1, const CUtensorMap& mw1,
                      const SkArgs& a0, const SkArgs& a1, const SkArgs& q, int64_t blocks, double bytes,
                      cudaStream_t stream) {
  sl_status st = set_attributes<kSkM, 3>();
  if (st != SL_OK) return st;
  const int cs = choose_split<kSkM, 3>(blocks, q);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_config<kSkM, 3>(blocks, cs, q, stream, attr);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_trigger / pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  const TimingToken tt = timing_begin(8, bytes, stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, skinny_kernel<kSkM, 3>, mq0, mw0, mq1, mw1, a0, a1);
  timing_end(tt, stream);
  if (e != cudaSuccess) return cuda_error(e, "skinny_kernel launch");
  return check_launch("skinny_kernel");
}

// bounds == nullptr: the pass does not split Q's columns by adapter (T_cat,
// dA_cat); otherwise G + 1 increasing offsets, multiples of 128, ending at C.
sl_status check_groups(int G, const int* bounds, int C, int r, SkArgs& a) {
  SL_REQUIRE(r >= 8 && r <= 32 && r % 8 == 0, "rank-r product: r must be 8, 16, 24 or 32");
  SL_REQUIRE(G >= 1 && G <= kSkMaxGroups && G * r <= 64, "rank-r product: need 1 <= G <= 4 and G r <= 64");
  a.G = G;
  a.r = r;
  a.R = G * r;
  a.bounds[0] = 0;
  for (int g = 0; g < G; ++g) {
    if (!bounds) {
      a.bounds[g + 1] = C;
      continue;
    }
    const int b = bounds[g + 1];
    SL_REQUIRE(b > a.bounds[g] && (g + 1 == G ? b == C : b % 128 == 0),
               "rank-r product: group bounds must increase in multiples of 128 and end at C");
    a.bounds[g + 1] = b;
  }
  return SL_OK;
}

}  // namespace

sl_status skinny_down(const uint16_t* Q, int64_t M, int C, const uint16_t* W, int wt, int r, int G, const int* bounds,
                      float* out, cudaStream_t stream) {
  SL_REQUIRE(C % 8 == 0 && M > 0 && M < (1LL << 31), "rank-r product: need C % 8 == 0 and 0 < M < 2^31");
  SkArgs a{};
  sl_status st = check_groups(G, bounds, C, r, a);
  if (st != SL_OK) return st;
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  const int mode = wt == 0 ? kSkKA : kSkKB;
  SL_REQUIRE(mode == kSkKA || G == 1 || bounds, "rank-r product: a grouped U pass needs the group bounds");
  a.M = static_cast<int>(M);
  a.C = C;
  a.rout = a.R;
  choose_pipeline(mode, r, a.R, a.rout, a);
  a.nsteps = static_cast<int>(ceil_div(C, a.step));
  a.s = 1.0f;
  a.out = out;
  a.err = err;
  CUtensorMap mq, mw;
  st = make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, C, M, static_cast<uint64_t>(C) * 2, 64, 128,
                CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  if (wt == 0)  // A_cat [G r, C]: operand rows straight from TMA (rows past G r read as zero)
    st = make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, C, a.R, static_cast<uint64_t>(C) * 2, 64,
                  sk_n_mma(mode, a.R, a.rout), CU_TENSOR_MAP_SWIZZLE_128B);
  else  // B_cat [C, r]: raw step x r tiles, transposed by the converter warps
    st = make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, r, C, static_cast<uint64_t>(r) * 2, r, a.step,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != SL_OK) return st;
  const int64_t blocks = ceil_div(M, 128);
  return wt == 0 ? launch<kSkKA>(mq, mw, a, blocks, stream) : launch<kSkKB>(mq, mw, a, blocks, stream);
}

namespace {

// Arguments and tensor maps of one mode-M pass (dA or dB).
sl_status prep_grad(const float* P, const uint16_t* Q, int64_t M, int C, int r, int G, const int* bounds, int select,
                    float s, float* out, int transpose, int accumulate, SkArgs& a, CUtensorMap& mq, CUtensorMap& mw) {
  SL_REQUIRE(C % 8 == 0 && M > 0 && M < (1LL << 31), "rank-r product: need C % 8 == 0 and 0 < M < 2^31");
  a = SkArgs{};
  sl_status st = check_groups(G, bounds, C, r, a);
  if (st != SL_OK) return st;
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  SL_REQUIRE(!select || G == 1 || bounds, "rank-r product: a grouped dB pass needs the group bounds");
  a.M = static_cast<int>(M);
  a.C = C;
  a.select = select;
  a.rout = select ? r : a.R;
  choose_pipeline(kSkM, r, a.R, a.rout, a);
  a.nsteps = static_cast<int>(ceil_div(M, a.step));
  a.s = s;
  a.transpose = transpose;
  a.accumulate = accumulate;
  a.out = out;
  a.err = err;
  st = make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, C, M, static_cast<uint64_t>(C) * 2, 64, a.step,
                CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  return make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, P, a.R, M, static_cast<uint64_t>(a.R) * 4, a.rout, a.step,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

sl_status skinny_grad(const float* P, const uint16_t* Q, int64_t M, int C, int r, int G, const int* bounds, int select,
                      float s, float* out, int transpose, int accumulate, cudaStream_t stream) {
  SkArgs a;
  CUtensorMap mq, mw;
  const sl_status st = prep_grad(P, Q, M, C, r, G, bounds, select, s, out, transpose, accumulate, a, mq, mw);
  if (st != SL_OK) return st;
  return launch<kSkM>(mq, mw, a, ceil_div(C, 128), stream);
}

sl_status skinny_grad_pair(const GradPass& p0, const GradPass& p1, int64_t M, int r, int G, float s, int accumulate,
                           cudaStream_t stream) {
  SkArgs a0, a1;
  CUtensorMap mq0, mw0, mq1, mw1;
  sl_status st = prep_grad(p0.P, p0.Q, M, p0.C, r, G, p0.bounds, p0.select, s, p0.out, p0.transpose, accumulate, a0,
                           mq0, mw0);
  if (st != SL_OK) return st;
  st = prep_grad(p1.P, p1.Q, M, p1.C, r, G, p1.bounds, p1.select, s, p1.out, p1.transpose, accumulate, a1, mq1, mw1);
  if (st != SL_OK) return st;
  const int64_t b0 = ceil_div(p0.C, 128), b1 = ceil_div(p1.C, 128);
  a0.nb0 = static_cast<int>(b0);
  // one launch, one cluster size and the larger of the two shared-memory footprints: the cluster
  // split and the occupancy query read the pass with the larger stages and the fewer steps
  SkArgs q = a0;
  if (sk_stage_bytes(kSkM, a1.r, a1.R, a1.rout, a1.step) * a1.stages >
      sk_stage_bytes(kSkM, a0.r, a0.R, a0.rout, a0.step) * a0.stages) {
    q = a1;
    q.nb0 = a0.nb0;
  }
  q.nsteps = std::min(a0.nsteps, a1.nsteps);
  return launch_pair(mq0, mw0, mq1, mw1, a0, a1, q, b0 + b1, pass_bytes(kSkM, a0) + pass_bytes(kSkM, a1), stream);
}

sl_status skinny_swiglu_u(const uint16_t* dm, const uint16_t* g, const uint16_t* u, int64_t ld_in, uint16_t* dg,
                          uint16_t* du, int64_t ld_out, int64_t M, int F, const uint16_t* B_cat, int r, float* U,
                          cudaStream_t stream) {
  SL_REQUIRE(dm && g && u && dg && du && B_cat && U && M > 0 && M < (1LL << 31),
             "fused SwiGLU backward: null pointer or bad M");
  SL_REQUIRE(F % 128 == 0 && ld_in % 8 == 0 && ld_out % 8 == 0 && ld_in >= F && ld_out >= F,
             "fused SwiGLU backward: need F % 128 == 0 and row strides % 8 == 0");
  SL_REQUIRE(((reinterpret_cast<uintptr_t>(dg) | reinterpret_cast<uintptr_t>(du)) & 15) == 0,
             "fused SwiGLU backward: dg and du must be 16-byte aligned");
  SkArgs a{};
  const int bounds[3] = {0, F, 2 * F};
  sl_status st = check_groups(2, bounds, 2 * F, r, a);
  if (st != SL_OK) return st;
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  a.M = static_cast<int>(M);
  a.C = 2 * F;
  a.F = F;
  a.rout = a.R;
  choose_pipeline(kSkKB, r, a.R, a.rout, a, 2);
  a.nsteps = F / 64;
  a.s = 1.0f;
  a.out = U;
  a.err = err;
  a.glue0 = dg;
  a.glue1 = du;
  a.glue_ld = ld_out;
  CUtensorMap mdm, mg, mu, mw;
  st = make_map(&mdm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dm, F, M, static_cast<uint64_t>(F) * 2, 64, 128,
                CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  st = make_map(&mg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g, F, M, static_cast<uint64_t>(ld_in) * 2, 64, 128,
                CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  st = make_map(&mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u, F, M, static_cast<uint64_t>(ld_in) * 2, 64, 128,
                CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  // B_cat [2F, r]: raw 64 x r tiles of B_g (rows c ..) and B_u (rows F + c ..)
  st = make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B_cat, r, 2 * F, static_cast<uint64_t>(r) * 2, r, 64,
                CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != SL_OK) return st;
  // dm, g, u read, dg and du written, B read, U written
  const double bytes = 10.0 * static_cast<double>(M) * F + 4.0 * r * F + 8.0 * static_cast<double>(M) * r;
  return launch<kSkKB, 2>(mdm, mw, a, ceil_div(M, 128), stream, &mg, &mu, bytes);
}

}  // namespace sl
