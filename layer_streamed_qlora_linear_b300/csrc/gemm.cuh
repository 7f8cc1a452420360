// The tensor-core GEMM of libsl (sm_103a, tcgen05 + TMEM + TMA).
//
//   C[m, j] = sum_k A[m, k] * Bop[j, k]  (+ sum_i Xe[m, i] * Be[j, i])
//
// A    : activations [M, K] bf16, K contiguous, brought in by TMA (128-byte
//        swizzle, 128 x 64 tiles).
// Bop  : the frozen weight.  Two layouts:
//        K-major  (forward, CE logits): W [N, K] (Linear.weight),
//        MN-major (dX, CE dH):          W [K, N] read as rows of the reduction.
//        Two sources: bf16 via TMA, or NF4 -- TMA brings the packed codes and
//        the fp32 absmax into shared memory and four dequant warps expand them
//        to bf16(T[code] * absmax) directly in the 128-byte-swizzled layout
//        the tensor core reads; both layouts share one dequant routine
//        because a row of 64 elements with one absmax is the unit of both.
// Xe/Be: the rank-r LoRA side product, folded into the same TMEM
//        accumulator after the main loop: s*Xe (fp32) is split into bf16
//        hi + lo and multiplied by [Be | Be] over K = 2r (r <= 32, padded to
//        16): forward Xe = T = X A^T, Be = B;  dX Xe = U = dY B, Be = A
//        (MN-major).
//
// Tile: 128 (M) x 256 (N) x 64 (K), fp32 accumulator in 256 TMEM columns,
// one tcgen05.mma.cta_group::1.kind::f16 128x256x16 per 16 of K.
// Warp roles (192 threads):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator + MMA issuer (one lane)
//   warps 2..5  NF4 dequant during the main loop, LoRA staging, epilogue
//               (warp w reads TMEM lanes 32*(w%4) .. +31).
// Pipeline: S stages, mbarriers tma_full / b_full / empty, one acc_full.
// Every wait is bounded (two seconds); a wait that gives up records
// SL_ERR_TIMEOUT in the device error word and the CTA winds down cleanly.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "nf4.cuh"
#include "ptx.cuh"

namespace sl {

enum GemmBSrc { kBSrcBF16 = 0, kBSrcNF4 = 1 };
enum GemmEpi {
  kEpiStoreBF16 = 0,   // out[m, j] = bf16(acc)
  kEpiCELse = 1,       // per-row (max, sum exp) over the tile + label logit gather
  kEpiCEGrad = 2,      // out[m, j] = bf16(exp(acc - lse[m]) * scale[m])  (softmax / N_valid)
  kEpiAddF32 = 3,      // outf[m, j] (+)= acc (fp32), "beta" = 0 on the first call
};

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kATileBytes = kBM * kBK * 2;  // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;  // 32 KB
constexpr int kCodesBytes = kBN * kBK / 2;  // 8 KB (both layouts)
constexpr int kAbsmaxBytes = kBN * 16;      // 4 KB (K-major box 4 x 256; MN-major uses 1 KB)
constexpr int kGemmThreads = 192;

template <int BSRC>
struct GemmCfg {
  static constexpr int S = (BSRC == kBSrcNF4) ? 3 : 4;
  static constexpr int kRawBytes = (BSRC == kBSrcNF4) ? (kCodesBytes + kAbsmaxBytes) : 0;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + S * kATileBytes;
  static constexpr int kOffRaw = kOffB + S * kBTileBytes;
  static constexpr int kOffTab = kOffRaw + S * kRawBytes;
  static constexpr int kOffBar = kOffTab + 128;
  static constexpr int kNumBars = 3 * S + 3;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kSmem = kBytes + 1024;  // slack for 1024-byte alignment
};

struct GemmArgs {
  int M, N, K;                 // rows, output columns, reduction length
  const float* lora_x;         // [M, r] fp32 (T or U) or nullptr
  const uint16_t* lora_w;      // K-major: [N, r]; MN-major: [r, N] (ld N); bf16
  int r;
  float s;                     // LoRA scale alpha / r
  void* out;                   // epilogue output
  int64_t ld_out;              // elements
  // cross-entropy epilogues
  const int32_t* labels;       // [M]
  int32_t ignore_index;
  int vocab_base;              // first vocab id of this chunk
  float* part_max;             // [M, ntiles] (kEpiCELse)
  float* part_sum;             // [M, ntiles]
  float* label_logit;          // [M] written by the tile that holds the label
  int part_ld;                 // ntiles of the whole vocab
  int tile_base;               // tile index of this launch's first column tile
  const float* row_lse;        // [M] (kEpiCEGrad)
  const float* row_scale;      // [M] 1/N_valid or 0 (kEpiCEGrad)
  int accumulate;              // kEpiAddF32: add into out (1) or overwrite (0)
  int* err;                    // device error word
};

// One row segment: 16 packed code bytes (32 elements) with one absmax ->
// four 16-byte chunks (logical chunk index chunk0 + j) of a 128-byte
// swizzled smem row.  tab: 16 fp32 levels (per-half-warp copy).
__device__ __forceinline__ void dequant_half_row(const uint4 q, float amax, const float* tab, uint8_t* row,
                                                 int chunk0, int rsw) {
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w = words[j];
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t byte = (w >> (8 * b)) & 0xFFu;
      const float v0 = __fmul_rn(tab[byte >> 4], amax);
      const float v1 = __fmul_rn(tab[byte & 15u], amax);
      op[b] = pack_bf16x2(v0, v1);
    }
    *reinterpret_cast<uint4*>(row + (((chunk0 + j) ^ rsw) << 4)) = o;
  }
}

template <int BSRC, int BMN, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_s, const GemmArgs args) {
  using Cfg = GemmCfg<BSRC>;
  constexpr int S = Cfg::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + Cfg::kOffA;
  uint8_t* sB = smem + Cfg::kOffB;
  uint8_t* sRaw = smem + Cfg::kOffRaw;
  float* sTab = reinterpret_cast<float*>(smem + Cfg::kOffTab);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* tma_full = bars;
  uint64_t* b_full = bars + S;
  uint64_t* empty = bars + 2 * S;
  uint64_t* lora_full = bars + 3 * S;
  uint64_t* acc_full = bars + 3 * S + 1;
  uint64_t* main_done = bars + 3 * S + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n0 = blockIdx.x * kBN;
  const int m0 = blockIdx.y * kBM;
  const int KB = (args.K + kBK - 1) / kBK;
  const bool has_lora = args.lora_x != nullptr && args.r > 0;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(&tma_full[i], 1);
      ptx::mbar_init(&b_full[i], 128);
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(lora_full, 128);
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(main_done, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&map_a);
    ptx::tma_prefetch_desc(&map_b);
    if (BSRC == kBSrcNF4) ptx::tma_prefetch_desc(&map_s);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, 256);
    ptx::tmem_relinquish();
  }
  if (tid >= 64 && tid < 96) sTab[tid - 64] = __uint_as_float(d_nf4_level_bits[(tid - 64) & 15]);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  auto give_up = [&]() {
    *abort_flag = 1;
    report_device_error(args.err, SL_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t tx = kATileBytes;
      if (BSRC == kBSrcBF16) tx += kBTileBytes;
      else tx += kCodesBytes + (BMN ? kBK * 16 : kAbsmaxBytes);
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % S;
        const uint32_t round = kb / S;
        if (!ptx::mbar_wait(&empty[s], (round & 1) ^ 1, abort_flag)) {
          give_up();
          break;
        }
        ptx::mbar_arrive_expect_tx(&tma_full[s], tx);
        ptx::tma_load_2d(sA + s * kATileBytes, &map_a, &tma_full[s], kb * kBK, m0);
        uint8_t* b_dst = sB + s * kBTileBytes;
        uint8_t* raw = sRaw + s * Cfg::kRawBytes;
        if (BSRC == kBSrcBF16) {
          if (!BMN) {
            ptx::tma_load_2d(b_dst, &map_b, &tma_full[s], kb * kBK, n0);
          } else {
#pragma unroll
            for (int a = 0; a < kBN / 64; ++a)
              ptx::tma_load_2d(b_dst + a * (64 * 128), &map_b, &tma_full[s], n0 + a * 64, kb * kBK);
          }
        } else {
          if (!BMN) {
            ptx::tma_load_2d(raw, &map_b, &tma_full[s], kb * (kBK / 2), n0);
            ptx::tma_load_2d(raw + kCodesBytes, &map_s, &tma_full[s], kb & ~3, n0);
          } else {
            ptx::tma_load_2d(raw, &map_b, &tma_full[s], n0 / 2, kb * kBK);
            ptx::tma_load_2d(raw + kCodesBytes, &map_s, &tma_full[s], n0 / 64, kb * kBK);
          }
        }
        ++issued;
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's smem is released.
        for (int kb = (issued > S ? issued - S : 0); kb < issued; ++kb)
          ptx::mbar_wait(&tma_full[kb % S], (kb / S) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16(kBM, kBN, 0, BMN);
      const uint32_t a_base = ptx::smem_addr(sA);
      const uint32_t b_base = ptx::smem_addr(sB);
      bool ok = true;
      for (int kb = 0; kb < KB && ok; ++kb) {
        const int s = kb % S;
        const uint32_t ph = (kb / S) & 1;
        if (!ptx::mbar_wait(&tma_full[s], ph, abort_flag) ||
            (BSRC == kBSrcNF4 && !ptx::mbar_wait(&b_full[s], ph, abort_flag))) {
          give_up();
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc(a_base + s * kATileBytes + kk * 32, 16, 1024, 2);
          const uint64_t bd = BMN ? ptx::smem_desc(b_base + s * kBTileBytes + kk * 2048, 64 * 128, 1024, 2)
                                  : ptx::smem_desc(b_base + s * kBTileBytes + kk * 32, 16, 1024, 2);
          ptx::mma_bf16(tmem, ad, bd, idesc, (kb | kk) ? 1u : 0u);
        }
        ptx::mma_commit(&empty[s]);
      }
      if (ok && has_lora) {
        // Every main-loop MMA done (and hence every TMA load consumed): the
        // staging warps may now overwrite stage KB % S with the LoRA operands.
        ptx::mma_commit(main_done);
        if (!ptx::mbar_wait(lora_full, 0, abort_flag)) {
          give_up();
          ok = false;
        } else {
          ptx::tc_fence_after();
          const int s = KB % S;
          const int ksteps = (2 * args.r + 15) / 16;
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint64_t ad = ptx::smem_desc(a_base + s * kATileBytes + kk * 32, 16, 1024, 2);
            const uint64_t bd = BMN ? ptx::smem_desc(b_base + s * kBTileBytes + kk * 2048, 64 * 128, 1024, 2)
                                    : ptx::smem_desc(b_base + s * kBTileBytes + kk * 32, 16, 1024, 2);
            ptx::mma_bf16(tmem, ad, bd, idesc, 1u);
          }
        }
      }
      ptx::mma_commit(acc_full);
      if (!ok) ptx::mbar_wait(acc_full, 0, nullptr);  // drain issued MMAs before TMEM is freed
    }
  } else {
    // ------------------------------------------- dequant / LoRA staging / epilogue
    const int dq = tid - 64;  // 0..127
    const float* tab = sTab + ((lane >> 4) << 4);
    bool ok = true;
    // LoRA side operands.  s * Xe (fp32; Xe = T or U) is split into bf16
    // hi + lo halves and folded over K = 2r columns [hi | lo] against
    // [Be | Be], so the side product keeps fp32 accuracy; Be (B_lora for the
    // forward, A_lora for dX) is used as stored.  The folded K is zero-padded
    // to a multiple of 16.  Thread dq owns row dq of Xe; Be is handled in
    // 2 * r/8 sixteen-byte tasks per thread (K-major: rows dq and dq + 128 x
    // rank groups; MN-major: rank rows x 32 column chunks).
    const int r = args.r;
    const int nr = r / 8;
    const int kpad = ((2 * r + 15) / 16) * 16;
    const int nchunk = kpad / 8;
    const int nbe = 2 * nr;
    auto load_xe = [&](int g, float (&v)[8]) {
      const int gm = m0 + dq;
      if (gm < args.M) {
        const float4* p = reinterpret_cast<const float4*>(args.lora_x + static_cast<int64_t>(gm) * r + g * 8);
        const float4 a = p[0], b = p[1];
        v[0] = a.x * args.s; v[1] = a.y * args.s; v[2] = a.z * args.s; v[3] = a.w * args.s;
        v[4] = b.x * args.s; v[5] = b.y * args.s; v[6] = b.z * args.s; v[7] = b.w * args.s;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.0f;
      }
    };
    auto chunk_at = [&](uint8_t* base, int row, int c) {
      return reinterpret_cast<uint4*>(base + row * 128 + ((c ^ (row & 7)) << 4));
    };
    auto store_xe = [&](uint8_t* at, int g, const float (&v)[8]) {
      uint4 hi, lo;
      uint32_t* ph = reinterpret_cast<uint32_t*>(&hi);
      uint32_t* pl = reinterpret_cast<uint32_t*>(&lo);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        ph[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
        pl[e] = pack_bf16x2(v[2 * e] - bf16_lo(ph[e]), v[2 * e + 1] - bf16_hi(ph[e]));
      }
      *chunk_at(at, dq, g) = hi;
      *chunk_at(at, dq, nr + g) = lo;
    };
    auto load_be = [&](int t) -> uint4 {
      if (!BMN) {
        const int j = dq + 128 * (t / nr), g = t % nr;
        const int gn = n0 + j;
        if (gn < args.N) return *reinterpret_cast<const uint4*>(args.lora_w + static_cast<int64_t>(gn) * r + g * 8);
      } else {
        const int task = dq + 128 * t;
        const int i = task >> 5, gcol = n0 + (task & 31) * 8;
        if (gcol < args.N) return *reinterpret_cast<const uint4*>(args.lora_w + static_cast<int64_t>(i) * args.N + gcol);
      }
      return make_uint4(0, 0, 0, 0);
    };
    auto mn_chunk = [&](uint8_t* bt, int i, int cc) {
      return reinterpret_cast<uint4*>(bt + (cc >> 3) * (64 * 128) + i * 128 + (((cc & 7) ^ (i & 7)) << 4));
    };
    auto store_be = [&](uint8_t* bt, int t, uint4 v) {
      if (!BMN) {
        const int j = dq + 128 * (t / nr), g = t % nr;
        *chunk_at(bt, j, g) = v;
        *chunk_at(bt, j, nr + g) = v;
      } else {
        const int task = dq + 128 * t;
        const int i = task >> 5, cc = task & 31;
        *mn_chunk(bt, i, cc) = v;
        *mn_chunk(bt, r + i, cc) = v;
      }
    };
    auto store_pad = [&](uint8_t* at, uint8_t* bt) {  // zero the K columns 2r .. kpad-1
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int c = 2 * nr; c < nchunk; ++c) {
        *chunk_at(at, dq, c) = z;
        if (!BMN) {
          *chunk_at(bt, dq, c) = z;
          *chunk_at(bt, dq + 128, c) = z;
        }
      }
      if (BMN)
        for (int task = dq; task < (kpad - 2 * r) * 32; task += 128) *mn_chunk(bt, 2 * r + (task >> 5), task & 31) = z;
    };
    // Rank <= 16: fetch the operands now, while the main loop runs.
    const bool lora_pref = has_lora && r <= 16;
    float pre_x[2][8];
    uint4 pre_b[4];
    if (lora_pref) {
      for (int g = 0; g < nr; ++g) load_xe(g, pre_x[g]);
      for (int t = 0; t < nbe; ++t) pre_b[t] = load_be(t);
    }
    if (BSRC == kBSrcNF4) {
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % S;
        if (!ptx::mbar_wait(&tma_full[s], (kb / S) & 1, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        const uint8_t* codes = sRaw + s * Cfg::kRawBytes;
        const float* amax = reinterpret_cast<const float*>(codes + kCodesBytes);
        uint8_t* bt = sB + s * kBTileBytes;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = i * 128 + dq;
          if (!BMN) {
            const int row = h >> 1, half = h & 1;
            const uint4 q = *reinterpret_cast<const uint4*>(codes + row * 32 + half * 16);
            dequant_half_row(q, amax[row * 4 + (kb & 3)], tab, bt + row * 128, half * 4, row & 7);
          } else {
            const int n = h >> 3, a = (h >> 1) & 3, half = h & 1;
            const uint4 q = *reinterpret_cast<const uint4*>(codes + n * 128 + a * 32 + half * 16);
            dequant_half_row(q, amax[n * 4 + a], tab, bt + a * (64 * 128) + n * 128, half * 4, n & 7);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&b_full[s]);
      }
    }
    if (ok && has_lora) {
      const int s = KB % S;
      if (!ptx::mbar_wait(main_done, 0, abort_flag)) {
        give_up();
        ok = false;
      } else {
        uint8_t* at = sA + s * kATileBytes;
        uint8_t* bt = sB + s * kBTileBytes;
        if (lora_pref) {
          for (int g = 0; g < nr; ++g) store_xe(at, g, pre_x[g]);
          for (int t = 0; t < nbe; ++t) store_be(bt, t, pre_b[t]);
        } else {
          for (int g = 0; g < nr; ++g) {
            float v[8];
            load_xe(g, v);
            store_xe(at, g, v);
          }
          for (int t = 0; t < nbe; ++t) store_be(bt, t, load_be(t));
        }
        store_pad(at, bt);
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(lora_full);
      }
    }
    // ------------------------------------------------------------ epilogue
    bool acc_ready = ptx::mbar_wait(acc_full, 0, abort_flag) && !*abort_flag;
    acc_ready = __all_sync(0xffffffffu, acc_ready);  // tcgen05.ld below is warp-collective
    if (acc_ready) {
      ptx::tc_fence_after();
      const int q = warp & 3;
      const int row = q * 32 + lane;
      const int gm = m0 + row;
      const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
      if (EPI == kEpiStoreBF16) {
        uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, v);
          ptx::tmem_wait_ld();
          if (gm < args.M && n0 + c0 < args.N) {
            uint4* dst = reinterpret_cast<uint4*>(out + static_cast<int64_t>(gm) * args.ld_out + n0 + c0);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]));
              o.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
              o.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]));
              o.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
              dst[g] = o;
            }
          }
        }
      } else if (EPI == kEpiAddF32) {
        float* out = reinterpret_cast<float*>(args.out);
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, v);
          ptx::tmem_wait_ld();
          if (gm < args.M && n0 + c0 < args.N) {
            float4* dst = reinterpret_cast<float4*>(out + static_cast<int64_t>(gm) * args.ld_out + n0 + c0);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              float4 o = make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                     __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
              if (args.accumulate) {
                const float4 p = dst[g];
                o.x += p.x;
                o.y += p.y;
                o.z += p.z;
                o.w += p.w;
              }
              dst[g] = o;
            }
          }
        }
      } else if (EPI == kEpiCELse) {
        // Online (max, sum exp) over this tile's 256 vocab columns, in a
        // fixed left-to-right order; the label's logit is gathered here too.
        const int lab = (gm < args.M) ? args.labels[gm] : args.ignore_index;
        float mx = -INFINITY, sm = 0.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, v);
          ptx::tmem_wait_ld();
          if (n0 + c0 < args.N) {
            float cm = -INFINITY;
#pragma unroll
            for (int e = 0; e < 32; ++e) cm = fmaxf(cm, __uint_as_float(v[e]));
            const float nm = fmaxf(mx, cm);
            float acc = 0.0f;
#pragma unroll
            for (int e = 0; e < 32; ++e) acc += __expf(__uint_as_float(v[e]) - nm);
            sm = sm * __expf(mx - nm) + acc;
            mx = nm;
            const int vid = args.vocab_base + n0 + c0;
            if (lab >= vid && lab < vid + 32 && gm < args.M) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (lab == vid + e) args.label_logit[gm] = __uint_as_float(v[e]);
            }
          }
        }
        if (gm < args.M) {
          const int64_t p = static_cast<int64_t>(gm) * args.part_ld + args.tile_base + blockIdx.x;
          args.part_max[p] = mx;
          args.part_sum[p] = sm;
        }
      } else if (EPI == kEpiCEGrad) {
        uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
        const float lse = (gm < args.M) ? args.row_lse[gm] : 0.0f;
        const float sc = (gm < args.M) ? args.row_scale[gm] : 0.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, v);
          ptx::tmem_wait_ld();
          if (gm < args.M && n0 + c0 < args.N) {
            uint4* dst = reinterpret_cast<uint4*>(out + static_cast<int64_t>(gm) * args.ld_out + n0 + c0);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __expf(__uint_as_float(v[8 * g + e]) - lse) * sc;
              uint4 o;
              o.x = pack_bf16x2(f[0], f[1]);
              o.y = pack_bf16x2(f[2], f[3]);
              o.z = pack_bf16x2(f[4], f[5]);
              o.w = pack_bf16x2(f[6], f[7]);
              dst[g] = o;
            }
          }
        }
      }
    } else if (!*abort_flag) {
      give_up();
    }
  }
  __syncwarp();

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 256);
  }
}

// Host side: build tensor maps and launch.  Defined in gemm.cu.
struct GemmLaunch {
  int bsrc;              // kBSrcBF16 / kBSrcNF4
  int bmn;               // 0: W [N, K]; 1: W [K, N]
  int epi;               // GemmEpi
  const void* A;         // [M, K] bf16
  int64_t lda;           // elements (>= K)
  const void* w;         // bf16 weight (kBSrcBF16)
  const uint8_t* codes;  // NF4 codes (kBSrcNF4)
  const float* absmax;   // NF4 absmax
  int64_t ldw;           // weight row length in elements (K for K-major, N for MN-major)
  GemmArgs args;
};

sl_status launch_gemm(const GemmLaunch& g, cudaStream_t stream);

}  // namespace sl
