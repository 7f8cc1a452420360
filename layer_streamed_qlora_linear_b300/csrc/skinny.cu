// The rank-r side products of the LoRA linear on the tensor cores.
//
// "Exact Layer Streaming ..." (abstract) trains only A [r, K] and B [N, r]
// beside a frozen base; around the fused base GEMM four skinny products
// remain, each one pass over a large bf16 operand Q:
//   forward   T  = X A^T          [M, r]   reduce over K     (mode kSkKA)
//   backward  U  = dY B           [M, r]   reduce over N     (mode kSkKB)
//             dA = s U^T X        [r, K]   reduce over M     (mode kSkM)
//             dB = s dY^T T       [N, r]   reduce over M     (mode kSkM)
// These are HBM-bound streams (2r FLOP per element of Q); on the CUDA cores
// the FMAs alone would outlast the read, so each pass runs tcgen05 MMAs with
// a narrow N (r .. 2r columns) over TMA-staged tiles of Q:
//   * mode K: D[128 rows of Q, r16] += Q[128 x 64] * W[r16 x 64]^T per step;
//     W = A is TMA-loaded directly (K-major), W = B^T is transposed from a
//     raw TMA tile by four converter warps;
//   * mode M: D[128 columns of Q, 2r] += Q^T[128 x 64] * P'[2r x 64]^T per
//     step, Q^T read MN-major straight from the TMA tile and P' = [P_hi ;
//     P_lo] the two-term bf16 split of the fp32 operand (U or T), written by
//     the converter warps, so D = Q^T P to fp32 accuracy.
// The long reduction is split over the CTAs of a thread-block cluster (up to
// 16); their fp32 partials are summed through distributed shared memory in
// rank order, so one launch writes the final result with no partial buffers
// in global memory and bitwise reproducible sums.  Every wait is bounded.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"
#include "skinny.cuh"
#include "timing.cuh"
#include "tmap.cuh"

namespace sl {

enum SkMode { kSkKA = 0, kSkKB = 1, kSkM = 2 };

constexpr int kSkThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2..5 converters + epilogue
constexpr int kSkMaxStages = 8;
constexpr int kSkStep = 128;      // reduced elements per pipeline step
constexpr int kSkQBytes = 128 * kSkStep * 2;  // Q tile of a step: two 16 KB TMA boxes (64 x 128)
constexpr int kSkTmemCols = 64;
constexpr int kSkBarBytes = 1024; // barriers + misc, ahead of the 1024-aligned data
constexpr int kSkSmemBudget = 227 * 1024 - 1024 - kSkBarBytes;

struct SkArgs {
  int M;          // rows of Q
  int C;          // columns of Q
  int r;          // rank (multiple of 8, <= 32)
  int nsteps;     // 128-wide steps of the reduced extent (C in mode K, M in mode M)
  int stages;     // pipeline depth (<= kSkMaxStages), sized to the shared memory
  float s;        // output scale (mode M)
  int transpose;  // mode M: out[i * C + c] (dA) instead of out[c * r + i] (dB)
  int accumulate; // mode M: out += result
  float* out;
  int* err;
};

// Per-stage byte counts of the three regions (Q, skinny operand, raw tile).
__host__ __device__ inline int sk_n_mma(int mode, int r) { return mode == kSkM ? 2 * r : (r + 15) / 16 * 16; }
__host__ __device__ inline int sk_op_bytes(int mode, int r) { return 2 * sk_n_mma(mode, r) * 128; }
__host__ __device__ inline int sk_raw_bytes(int mode, int r) {
  return mode == kSkKA ? 0 : (mode == kSkKB ? kSkStep * r * 2 : kSkStep * r * 4);
}
__host__ __device__ inline int sk_stage_bytes(int mode, int r) {
  return kSkQBytes + sk_op_bytes(mode, r) + sk_raw_bytes(mode, r);
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

template <int MODE>
__global__ void __launch_bounds__(kSkThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_w,
                  const SkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int r = a.r;
  const int S = a.stages;
  const int n_mma = sk_n_mma(MODE, r);
  const int op_half = n_mma * 128;  // one 64-wide K chunk of the skinny operand
  const int op_bytes = sk_op_bytes(MODE, r);
  const int raw_bytes = sk_raw_bytes(MODE, r);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* full = bars;                      // TMA bytes of the stage landed
  uint64_t* conv = bars + kSkMaxStages;       // converter warps wrote the stage's skinny operand
  uint64_t* empty = bars + 2 * kSkMaxStages;  // MMAs of the stage completed
  uint64_t* acc_full = bars + 3 * kSkMaxStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 516);
  uint8_t* sQ = smem + kSkBarBytes;
  uint8_t* sOp = sQ + S * kSkQBytes;
  uint8_t* sRaw = sOp + S * op_bytes;
  const int red_ld = 36;                      // fp32 partial [128][36] (r <= 32 columns) in the Q region
  float* red = reinterpret_cast<float*>(sQ);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int cs = static_cast<int>(gridDim.y);  // cluster = the CTAs of one blockIdx.x
  const int rank = static_cast<int>(blockIdx.y);
  const int s0 = static_cast<int>(static_cast<int64_t>(a.nsteps) * rank / cs);
  const int s1 = static_cast<int>(static_cast<int64_t>(a.nsteps) * (rank + 1) / cs);
  const int nloc = s1 - s0;
  const int base = static_cast<int>(blockIdx.x) * 128;  // rows of Q (mode K) or columns of Q (mode M)

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&conv[i], 4);
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(acc_full, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&map_q);
    ptx::tma_prefetch_desc(&map_w);
  }
  if (MODE == kSkKB && n_mma > r) {
    // rows r .. n_mma-1 of the transposed B operand stay zero for the whole kernel
    const int pad = n_mma - r;
    for (int i = tid; i < S * 2 * pad * 8; i += kSkThreads) {
      const int st = i / (2 * pad * 8), h = (i / (pad * 8)) & 1, row = r + (i / 8) % pad, c = i % 8;
      *sw128_chunk(sOp + st * op_bytes + h * op_half, row, c) = make_uint4(0, 0, 0, 0);
    }
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, kSkTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  auto give_up = [&]() {
    *abort_flag = 1;
    report_device_error(a.err, SL_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t tx = kSkQBytes + (MODE == kSkKA ? 2 * n_mma * 128 : raw_bytes);
      int j = 0;
      for (; j < nloc; ++j) {
        const int st = j % S;
        if (!ptx::mbar_wait(&empty[st], ((j / S) & 1) ^ 1, abort_flag)) {
          give_up();
          break;
        }
        const int k0 = (s0 + j) * kSkStep;
        uint8_t* q = sQ + st * kSkQBytes;
        ptx::mbar_arrive_expect_tx(&full[st], tx);
        if (MODE == kSkKA) {  // Q [128 rows x 128 reduced], A [n_mma x 128 reduced], 64-wide halves
          ptx::tma_load_2d(q, &map_q, &full[st], k0, base);
          ptx::tma_load_2d(q + kSkQBytes / 2, &map_q, &full[st], k0 + 64, base);
          ptx::tma_load_2d(sOp + st * op_bytes, &map_w, &full[st], k0, 0);
          ptx::tma_load_2d(sOp + st * op_bytes + op_half, &map_w, &full[st], k0 + 64, 0);
        } else if (MODE == kSkKB) {  // Q as above; raw B rows k0 .. k0+127
          ptx::tma_load_2d(q, &map_q, &full[st], k0, base);
          ptx::tma_load_2d(q + kSkQBytes / 2, &map_q, &full[st], k0 + 64, base);
          ptx::tma_load_2d(sRaw + st * raw_bytes, &map_w, &full[st], 0, k0);
        } else {  // Q rows k0 .. k0+127, columns base .. base+127 (two 64-column atoms); raw P rows
          ptx::tma_load_2d(q, &map_q, &full[st], base, k0);
          ptx::tma_load_2d(q + kSkQBytes / 2, &map_q, &full[st], base + 64, k0);
          ptx::tma_load_2d(sRaw + st * raw_bytes, &map_w, &full[st], 0, k0);
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
        const uint32_t qs = q_base + st * kSkQBytes;
        const uint32_t os = op_base + st * op_bytes;
#pragma unroll
        for (int kk = 0; kk < kSkStep / 16; ++kk) {
          const int h = kk >> 2, k4 = kk & 3;
          // mode K: A = Q K-major, half h at +16 KB; mode M: A = Q^T MN-major,
          // 16 reduced rows (2 KB) per k16 step, the two 64-column atoms 16 KB apart
          const uint64_t ad = MODE == kSkM ? ptx::smem_desc(qs + kk * 2048, kSkQBytes / 2, 1024, 2)
                                           : ptx::smem_desc(qs + h * (kSkQBytes / 2) + k4 * 32, 16, 1024, 2);
          const uint64_t bd = ptx::smem_desc(os + h * op_half + k4 * 32, 16, 1024, 2);
          ptx::mma_bf16(tmem, ad, bd, idesc, (j | kk) ? 1u : 0u);
        }
        ptx::mma_commit(&empty[st]);
      }
      ptx::mma_commit(acc_full);
    }
  } else {
    // ------------------------------------ converters (modes KB, M), then epilogue
    const int e = tid - 64;  // 0..127
    if (MODE != kSkKA) {
      for (int j = 0; j < nloc; ++j) {
        const int st = j % S;
        if (!ptx::mbar_wait(&full[st], (j / S) & 1, abort_flag)) {
          give_up();
          break;
        }
        uint8_t* op = sOp + st * op_bytes;
        const uint8_t* raw = sRaw + st * raw_bytes;
        // task = (8-wide chunk ch of the 128 reduced elements, rank index i),
        // i fastest so that a warp reads consecutive words of the raw rows
        for (int task = e; task < r * 16; task += 128) {
          const int i = task % r, ch = task / r;
          uint8_t* oh = op + (ch >> 3) * op_half;
          const int c8 = ch & 7;
          if (MODE == kSkKB) {
            // raw: B rows k0 .. k0+127, r bf16 each -> operand row i = B[k][i]
            const uint16_t* rb = reinterpret_cast<const uint16_t*>(raw) + (ch * 8) * r + i;
            uint32_t w[4];
#pragma unroll
            for (int p = 0; p < 4; ++p)
              w[p] = static_cast<uint32_t>(rb[(2 * p) * r]) | (static_cast<uint32_t>(rb[(2 * p + 1) * r]) << 16);
            *sw128_chunk(oh, i, c8) = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            // raw: P rows k0 .. k0+127, r fp32 each -> rows i (hi) and r + i (lo)
            const float* rf = reinterpret_cast<const float*>(raw) + (ch * 8) * r + i;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const float v0 = rf[(2 * p) * r], v1 = rf[(2 * p + 1) * r];
              hi[p] = pack_bf16x2(v0, v1);
              lo[p] = pack_bf16x2(v0 - bf16_lo(hi[p]), v1 - bf16_hi(hi[p]));
            }
            *sw128_chunk(oh, i, c8) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *sw128_chunk(oh, r + i, c8) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&conv[st]);
      }
    }
    // epilogue: TMEM lane `row` of the accumulator holds this CTA's partial
    // for row `row` of the block (mode M: hi and lo halves, added here)
    bool ready = ptx::mbar_wait(acc_full, 0, abort_flag) && !*abort_flag;
    ready = __all_sync(0xffffffffu, ready);
    if (!ready && !*abort_flag) give_up();
    ptx::tc_fence_after();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const bool keep = ready && nloc > 0;
    float v[32];  // the r (<= 32) result columns of this row
    {
      uint32_t u[32];
      ptx::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16), u);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] = keep ? __uint_as_float(u[c]) : 0.0f;
      if (MODE == kSkM) {
        // D columns: [0, r) from P_hi, [r, 2r) from P_lo (r in {8, 16, 24, 32});
        // the lo term of result column c sits at column c + r
        uint32_t w[32];
        ptx::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + 32, w);
        ptx::tmem_wait_ld();
        auto add_lo = [&](auto rc) {
          constexpr int R = decltype(rc)::value;
#pragma unroll
          for (int c = 0; c < R; ++c) v[c] += keep ? __uint_as_float(c + R < 32 ? u[(c + R) & 31] : w[(c + R) & 31]) : 0.0f;
        };
        switch (r) {
          case 8: add_lo(std::integral_constant<int, 8>{}); break;
          case 16: add_lo(std::integral_constant<int, 16>{}); break;
          case 24: add_lo(std::integral_constant<int, 24>{}); break;
          default: add_lo(std::integral_constant<int, 32>{}); break;
        }
      }
    }
    if (cs == 1) {
      // the whole reduction ran here: write straight from registers
      if (MODE != kSkM) {
        const int gm = base + row;
        if (gm < a.M)
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4)
            if (i4 * 4 < r)
              *reinterpret_cast<float4*>(a.out + static_cast<int64_t>(gm) * r + i4 * 4) =
                  make_float4(v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2], v[4 * i4 + 3]);
      } else {
        const int gc = base + row;
        if (gc < a.C) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i >= r) break;
            float* o = a.transpose ? a.out + static_cast<int64_t>(i) * a.C + gc : a.out + static_cast<int64_t>(gc) * r + i;
            const float x = v[i] * a.s;
            *o = a.accumulate ? *o + x : x;
          }
        }
      }
    } else {
      float* dst = red + row * red_ld;
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4)
        if (i4 * 4 < r)
          *reinterpret_cast<float4*>(dst + i4 * 4) = make_float4(v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2], v[4 * i4 + 3]);
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
    const int nq = r / 4;
    const bool by_col = MODE == kSkM && a.transpose;  // dA: rows vary fastest for coalesced stores
    for (int task = tid; task < nrows * nq; task += kSkThreads) {
      const int rl = by_col ? task % nrows : task / nq;
      const int i4 = by_col ? task / nrows : task % nq;
      const int row = r0 + rl;
      const uint32_t own = ptx::smem_addr(red + row * red_ld + i4 * 4);
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
        if (gm < a.M) *reinterpret_cast<float4*>(a.out + static_cast<int64_t>(gm) * r + i4 * 4) = acc;
      } else {
        const int gc = base + row;
        if (gc < a.C) {
          const float x[4] = {acc.x * a.s, acc.y * a.s, acc.z * a.s, acc.w * a.s};
          if (!a.transpose) {
            float4* o = reinterpret_cast<float4*>(a.out + static_cast<int64_t>(gc) * r + i4 * 4);
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

int stages_for(int mode, int r) {
  const int s = kSkSmemBudget / sk_stage_bytes(mode, r);
  return s < kSkMaxStages ? s : kSkMaxStages;
}

template <int MODE>
sl_status set_attributes() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(skinny_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(skinny_kernel<MODE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  return err == cudaSuccess ? SL_OK : cuda_error(err, "skinny_kernel attributes");
}

template <int MODE>
cudaLaunchConfig_t make_config(int64_t blocks, int cs, int stages, int r, cudaStream_t stream,
                               cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(cs), 1);
  cfg.blockDim = dim3(kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(1024 + kSkBarBytes + stages * sk_stage_bytes(MODE, r));
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Clusters of `cs` CTAs that the device can hold at once (driver query,
// cached per device, mode, rank and cluster size).
template <int MODE>
int max_active_clusters(int cs, int stages, int r) {
  static std::mutex mu;
  static int cache[64][5][17];  // [device][r / 8][cs], 0 = not yet asked
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  int& slot = cache[dev][r / 8][cs];
  if (slot == 0) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_config<MODE>(1, cs, stages, r, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, skinny_kernel<MODE>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    slot = n > 0 ? n : -1;
  }
  return slot;
}

// Cluster size: the largest split of the reduction (at least two 128-wide
// steps per CTA) whose clusters all fit on the device at once, so that the
// launch is one wave of at most one CTA per SM.
template <int MODE>
int choose_split(int64_t blocks, int64_t nsteps, int stages, int r) {
  for (int cs = 16; cs > 1; --cs) {
    if (blocks * cs > num_sms() || nsteps < 2 * cs) continue;
    if (max_active_clusters<MODE>(cs, stages, r) >= blocks) return cs;
  }
  return 1;
}

// Algorithmic bytes of one pass: Q once, the skinny operand once, the output
// written (and read too when accumulating).
double pass_bytes(int mode, const SkArgs& a) {
  const double q = 2.0 * a.M * static_cast<double>(a.C);
  if (mode != kSkM) return q + 2.0 * a.r * a.C + 4.0 * a.M * a.r;
  return q + 4.0 * a.M * a.r + 4.0 * a.C * a.r * (a.accumulate ? 2 : 1);
}

template <int MODE>
sl_status launch(const CUtensorMap& mq, const CUtensorMap& mw, const SkArgs& a, int64_t blocks,
                 cudaStream_t stream) {
  sl_status st = set_attributes<MODE>();
  if (st != SL_OK) return st;
  const int cs = choose_split<MODE>(blocks, a.nsteps, a.stages, a.r);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_config<MODE>(blocks, cs, a.stages, a.r, stream, attr);
  const TimingToken tt = timing_begin(MODE == kSkKA ? 7 : (MODE == kSkKB ? 8 : 9), pass_bytes(MODE, a), stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, skinny_kernel<MODE>, mq, mw, a);
  timing_end(tt, stream);
  if (e != cudaSuccess) return cuda_error(e, "skinny_kernel launch");
  return check_launch("skinny_kernel");
}

}  // namespace

sl_status skinny_down(const uint16_t* Q, int64_t M, int C, const uint16_t* W, int wt, int r, float* out,
                      cudaStream_t stream) {
  SL_REQUIRE(r >= 8 && r <= 32 && r % 8 == 0, "rank-r product: r must be 8, 16, 24 or 32");
  SL_REQUIRE(C % 8 == 0 && M > 0 && M < (1LL << 31), "rank-r product: need C % 8 == 0 and 0 < M < 2^31");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  CUtensorMap mq, mw;
  sl_status st = make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, C, M, static_cast<uint64_t>(C) * 2, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  if (wt == 0)  // A [r, C]: operand rows straight from TMA (rows past r read as zero)
    st = make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, C, r, static_cast<uint64_t>(C) * 2, 64,
                  (r + 15) / 16 * 16, CU_TENSOR_MAP_SWIZZLE_128B);
  else  // B [C, r]: raw 64 x r tiles, transposed by the converter warps
    st = make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, r, C, static_cast<uint64_t>(r) * 2, r, kSkStep,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != SL_OK) return st;
  SkArgs a{};
  a.M = static_cast<int>(M);
  a.C = C;
  a.r = r;
  a.nsteps = static_cast<int>(ceil_div(C, kSkStep));
  a.stages = stages_for(wt == 0 ? kSkKA : kSkKB, r);
  a.s = 1.0f;
  a.out = out;
  a.err = err;
  const int64_t blocks = ceil_div(M, 128);
  return wt == 0 ? launch<kSkKA>(mq, mw, a, blocks, stream) : launch<kSkKB>(mq, mw, a, blocks, stream);
}

sl_status skinny_grad(const float* P, const uint16_t* Q, int64_t M, int C, int r, float s, float* out, int transpose,
                      int accumulate, cudaStream_t stream) {
  SL_REQUIRE(r >= 8 && r <= 32 && r % 8 == 0, "rank-r product: r must be 8, 16, 24 or 32");
  SL_REQUIRE(C % 8 == 0 && M > 0 && M < (1LL << 31), "rank-r product: need C % 8 == 0 and 0 < M < 2^31");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  CUtensorMap mq, mw;
  sl_status st = make_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, C, M, static_cast<uint64_t>(C) * 2, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  st = make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, P, r, M, static_cast<uint64_t>(r) * 4, r, kSkStep,
                CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st != SL_OK) return st;
  SkArgs a{};
  a.M = static_cast<int>(M);
  a.C = C;
  a.r = r;
  a.nsteps = static_cast<int>(ceil_div(M, kSkStep));
  a.stages = stages_for(kSkM, r);
  a.s = s;
  a.transpose = transpose;
  a.accumulate = accumulate;
  a.out = out;
  a.err = err;
  const int64_t blocks = ceil_div(C, 128);
  return launch<kSkM>(mq, mw, a, blocks, stream);
}

}  // namespace sl
