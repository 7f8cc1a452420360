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
// Warp roles (320 threads):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator + MMA issuer (one lane)
//   warps 2..9  NF4 dequant during the main loop (one 64-element row per
//               thread per k-block), LoRA staging, epilogue (warp w reads
//               TMEM lanes 32*(w%4) .. +31, columns of its half).
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
  kEpiCEExp = 1,       // per row and 128-column half tile: m = max, out = bf16(exp(acc - m)), sum, label logit
  kEpiAddF32 = 3,      // outf[m, j] = (accumulate ? outf[m, j] * alpha[m] : 0) + acc (fp32; alpha 1 if absent)
};

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kATileBytes = kBM * kBK * 2;  // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;  // 32 KB
constexpr int kCodesBytes = kBN * kBK / 2;  // 8 KB (both layouts)
constexpr int kAbsmaxBytes = kBN * 16;      // 4 KB (K-major box 4 x 256; MN-major uses 1 KB)
constexpr int kNumDq = 256;                 // dequant / staging / epilogue threads (warps 2..9)
constexpr int kGemmThreads = 64 + kNumDq;

template <int BSRC>
struct GemmCfg {
  static constexpr int S = (BSRC == kBSrcNF4) ? 3 : 4;
  static constexpr int kRawBytes = (BSRC == kBSrcNF4) ? (kCodesBytes + kAbsmaxBytes) : 0;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + S * kATileBytes;
  static constexpr int kOffRaw = kOffB + S * kBTileBytes;
  static constexpr int kOffTab = kOffRaw + S * kRawBytes;
  static constexpr int kOffBar = kOffTab + 128;
  static constexpr int kNumBars = 3 * S + 3 + 8;  // + one epilogue barrier per epilogue warp
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kSmem = kBytes + 1024;  // slack for 1024-byte alignment
};

struct GemmArgs {
  int M, N, K;                 // rows, output columns, reduction length
  const float* lora_x;         // [M, r] fp32 (T or U) or nullptr
  const uint16_t* lora_w;      // K-major: [N, r]; MN-major: [r, N] (ld N); bf16
  int r;                       // rank of the folded side product (a group's G r in the grouped dX)
  int lora_ld;                 // row stride of lora_x in floats (0: r)
  int lora_G;                  // grouped forward: projections sharing the GEMM (0 or 1: none)
  int lora_bounds[5];          // grouped forward: first output column of projection g (multiples of 256), [G] = N
  float s;                     // LoRA scale alpha / r
  int dq;                      // NF4 with the double-quantised absmax (persistent pair GEMM)
  int dq_col0;                 // the weight's first column in the qabsmax / absmax2 arrays
  void* out;                   // epilogue output
  int64_t ld_out;              // elements
  // cross-entropy epilogues
  const int32_t* labels;       // [M]
  int32_t ignore_index;
  int vocab_base;              // first vocab id of this chunk
  float* part_max;             // [M, part_ld] per 128-column half tile of the chunk (kEpiCEExp)
  float* part_sum;             // [M, part_ld]
  float* label_logit;          // [M] written by the tile that holds the label
  int part_ld;                 // half tiles of a chunk
  const float* row_alpha;      // [M] kEpiAddF32: factor on the accumulated output, or nullptr
  int accumulate;              // kEpiAddF32: add into out (1) or overwrite (0)
  int tma_out;                 // gemm_tc_kernel: the output moves by TMA through map_o (else direct stores)
  int* err;                    // device error word
  // persistent pair GEMM, last partial wave split along K: every cluster
  // takes split_rounds full tiles, then the split_R tail tiles go in
  // split_P pieces of contiguous k-blocks to clusters 0 .. split_R*split_P-1;
  // piece p > 0 leaves its fp32 accumulator in split_part (slot
  // j*(split_P-1)+p-1 of tail tile j: [2 CTAs][256 columns][128 rows]) and
  // raises split_flag[slot * 2 + CTA] to split_tag; piece 0 adds them in
  // piece order.  split_P < 2: no split.
  int split_P, split_R, split_rounds;
  float* split_part;
  unsigned long long* split_flag;
  unsigned long long split_tag;
  // launch timing on the device clock (nullptr: off): clk[0] = min over CTAs
  // of %globaltimer once past the dependency wait, clk[1] = max once done
  unsigned long long* clk;
};

__device__ __forceinline__ void clk_start(const GemmArgs& a) {
  if (a.clk && threadIdx.x == 0) atomicMin(a.clk, globaltimer_ns());
}
__device__ __forceinline__ void clk_end(const GemmArgs& a) {
  if (a.clk && threadIdx.x == 0) atomicMax(a.clk + 1, globaltimer_ns());
}

// One row segment of 64 NF4 elements (32 packed code bytes, one absmax) ->
// 64 bf16 = bf16(T[code] * absmax), written as eight 16-byte chunks of a
// 128-byte-swizzled smem row (logical chunk j at physical j ^ rsw).
//
// The 16 products bf16(T[i] * absmax) are formed once per segment (fp32
// multiply, one rounding) and split into byte planes L (low bytes) and H
// (high bytes), four registers each.  A code then costs a few byte
// permutes: prmt selects from entries 0-7 and 8-15 by the code's low 3 bits,
// and a lop3 picks between the two by the code's bit 3 (a byte mask made by
// prmt's sign-replicate mode from the packed codes themselves).  No shared
// memory table, no per-element multiply.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t select_bytes(uint32_t lo8, uint32_t hi8, uint32_t mask) {
  uint32_t d;  // (lo8 & ~mask) | (hi8 & mask)
  asm("lop3.b32 %0, %1, %2, %3, 0xD8;" : "=r"(d) : "r"(lo8), "r"(hi8), "r"(mask));
  return d;
}

__device__ __forceinline__ void nf4_row_bf16(const uint8_t* codes, float amax, uint8_t* row, int rsw) {
  uint32_t P[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    P[i] = pack_bf16x2(__fmul_rn(__uint_as_float(d_nf4_level_bits[2 * i]), amax),
                       __fmul_rn(__uint_as_float(d_nf4_level_bits[2 * i + 1]), amax));
  const uint32_t L0 = prmt(P[0], P[1], 0x6420), H0 = prmt(P[0], P[1], 0x7531);
  const uint32_t L1 = prmt(P[2], P[3], 0x6420), H1 = prmt(P[2], P[3], 0x7531);
  const uint32_t L2 = prmt(P[4], P[5], 0x6420), H2 = prmt(P[4], P[5], 0x7531);
  const uint32_t L3 = prmt(P[6], P[7], 0x6420), H3 = prmt(P[6], P[7], 0x7531);
  const uint4 q0 = *reinterpret_cast<const uint4*>(codes);
  const uint4 q1 = *reinterpret_cast<const uint4*>(codes + 16);
  const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t w = words[j];         // byte i = (e_{2i} << 4) | e_{2i+1}
    const uint32_t w4 = w << 4;          // bit 7 of byte i = bit 3 of e_{2i+1}
    const uint32_t s7 = w & 0x77777777u; // code bits 0-2
    const uint32_t sA = s7, sB = s7 >> 16;
    // nibbles of sA: (e1, e0, e3, e2); of sB: (e5, e4, e7, e6)
    const uint32_t mA = prmt(w4, w, 0xD9C8), mB = prmt(w4, w, 0xFBEA);  // 0xFF where bit 3 set
    const uint32_t loA = select_bytes(prmt(L0, L1, sA), prmt(L2, L3, sA), mA);
    const uint32_t hiA = select_bytes(prmt(H0, H1, sA), prmt(H2, H3, sA), mA);
    const uint32_t loB = select_bytes(prmt(L0, L1, sB), prmt(L2, L3, sB), mB);
    const uint32_t hiB = select_bytes(prmt(H0, H1, sB), prmt(H2, H3, sB), mB);
    uint4 o;
    o.x = prmt(loA, hiA, 0x4051);  // (e0, e1)
    o.y = prmt(loA, hiA, 0x6273);  // (e2, e3)
    o.z = prmt(loB, hiB, 0x4051);  // (e4, e5)
    o.w = prmt(loB, hiB, 0x6273);  // (e6, e7)
    *reinterpret_cast<uint4*>(row + ((j ^ rsw) << 4)) = o;
  }
}

template <int BSRC, int BMN, int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_o,
                   const GemmArgs args) {
  using Cfg = GemmCfg<BSRC>;
  constexpr int S = Cfg::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = ptx::align1024(smem_raw);
  uint8_t* sA = smem + Cfg::kOffA;
  uint8_t* sB = smem + Cfg::kOffB;
  uint8_t* sRaw = smem + Cfg::kOffRaw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* tma_full = bars;
  uint64_t* b_full = bars + S;
  uint64_t* empty = bars + 2 * S;
  uint64_t* lora_full = bars + 3 * S;
  uint64_t* acc_full = bars + 3 * S + 1;
  uint64_t* main_done = bars + 3 * S + 2;
  uint64_t* epi_bar = bars + 3 * S + 3;  // [8] kEpiAddF32 with TMA: the epilogue warp's old output landed
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
      ptx::mbar_init(&b_full[i], kNumDq);
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(lora_full, kNumDq);
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(main_done, 1);
    for (int i = 0; i < 8; ++i) ptx::mbar_init(&epi_bar[i], 1);
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
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // No early pdl_trigger: this grid is one CTA per tile, often several waves;
  // dependents launch as its CTAs exit (an early trigger let small follow-up
  // kernels wait beside the last wave and slowed it).
  pdl_wait();  // the previous kernel's writes are visible from here on
  clk_start(args);

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
    const int dq = tid - 64;  // 0..255
    bool ok = true;
    // LoRA side operands.  s * Xe (fp32; Xe = T or U) is split into bf16
    // hi + lo halves and folded over K = 2r columns [hi | lo] against
    // [Be | Be], so the side product keeps fp32 accuracy; Be (B_lora for the
    // forward, A_lora for dX) is used as stored.  The folded K is zero-padded
    // to a multiple of 16.  Threads dq < 128 own row dq of Xe; Be is handled
    // in r/8 sixteen-byte tasks per thread (K-major: row dq x rank groups;
    // MN-major: rank rows x 32 column chunks, task dq + 256 t).
    const int r = args.r;
    const int nr = r / 8;
    const int kpad = ((2 * r + 15) / 16) * 16;
    const int nchunk = kpad / 8;
    const int nbe = nr;
    const bool xe_row = dq < kBM;
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
        const int j = dq, g = t;
        const int gn = n0 + j;
        if (gn < args.N) return *reinterpret_cast<const uint4*>(args.lora_w + static_cast<int64_t>(gn) * r + g * 8);
      } else {
        const int task = dq + kNumDq * t;
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
        const int j = dq, g = t;
        *chunk_at(bt, j, g) = v;
        *chunk_at(bt, j, nr + g) = v;
      } else {
        const int task = dq + kNumDq * t;
        const int i = task >> 5, cc = task & 31;
        *mn_chunk(bt, i, cc) = v;
        *mn_chunk(bt, r + i, cc) = v;
      }
    };
    auto store_pad = [&](uint8_t* at, uint8_t* bt) {  // zero the K columns 2r .. kpad-1
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int c = 2 * nr; c < nchunk; ++c) {
        if (xe_row) *chunk_at(at, dq, c) = z;
        if (!BMN) *chunk_at(bt, dq, c) = z;
      }
      if (BMN)
        for (int task = dq; task < (kpad - 2 * r) * 32; task += kNumDq)
          *mn_chunk(bt, 2 * r + (task >> 5), task & 31) = z;
    };
    // Rank <= 16: fetch the operands now, while the main loop runs.
    const bool lora_pref = has_lora && r <= 16;
    float pre_x[2][8];
    uint4 pre_b[2];
    if (lora_pref) {
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (xe_row && g < nr) load_xe(g, pre_x[g]);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (t < nbe) pre_b[t] = load_be(t);
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
        if (!BMN) {  // row dq of the [256 x 64] tile
          nf4_row_bf16(codes + dq * 32, amax[dq * 4 + (kb & 3)], bt + dq * 128, dq & 7);
        } else {     // reduction row n, 64-column atom a of the [64 x 256] tile
          const int n = dq >> 2, a = dq & 3;
          nf4_row_bf16(codes + n * 128 + a * 32, amax[n * 4 + a], bt + a * (64 * 128) + n * 128, n & 7);
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
#pragma unroll
          for (int g = 0; g < 2; ++g)
            if (xe_row && g < nr) store_xe(at, g, pre_x[g]);
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (t < nbe) store_be(bt, t, pre_b[t]);
        } else {
          for (int g = 0; g < nr && xe_row; ++g) {
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
      const int q = warp & 3;                 // TMEM lane quadrant of this warp
      const int ch = (warp - 2) >> 2;         // column half: warps 2-5 -> 0..127, 6-9 -> 128..255
      const int cbeg = ch * (kBN / 2), cend = cbeg + kBN / 2;
      const int row = q * 32 + lane;
      const int gm = m0 + row;
      const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
      // TMA-store path: the main loop is over and every stage consumed, so the
      // stage buffers serve as staging.  This warp's 32 rows x 128 columns
      // leave as 64-column bf16 boxes (2 x 4 KB) or 32-column fp32 boxes
      // (4 x 4 KB) in the 128-byte-swizzled layout; rows and columns past the
      // output are clipped by the tensor map.
      uint8_t* stg = smem + (warp - 2) * (EPI == kEpiAddF32 ? 16384 : 8192);
      const uint32_t stg_a = ptx::smem_addr(stg);
      auto stg_chunk = [&](int lc, int j) {  // 16-byte chunk j of local column block lc / (box width)
        constexpr int kBoxCols = EPI == kEpiAddF32 ? 32 : 64;
        return stg_a + (lc / kBoxCols) * 4096 + lane * 128 + ((j ^ (lane & 7)) << 4);
      };
      auto tma_store_boxes = [&]() {
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          constexpr int kBoxes = EPI == kEpiAddF32 ? 4 : 2, kBoxCols = 128 / kBoxes;
          for (int b = 0; b < kBoxes; ++b)
            ptx::tma_store_2d(&map_o, stg + b * 4096, n0 + cbeg + b * kBoxCols, m0 + q * 32);
          ptx::bulk_commit();
          ptx::bulk_wait_read0();  // the staging is read before the CTA's shared memory goes
        }
        __syncwarp();
      };
      if (args.tma_out && EPI == kEpiStoreBF16) {
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, v);
          ptx::tmem_wait_ld();
          const int lc = c0 - cbeg;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg_chunk(lc, (lc % 64) / 8 + g)),
                         "r"(pack_bf16x2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]))),
                         "r"(pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]))),
                         "r"(pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]))),
                         "r"(pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7])))
                         : "memory");
        }
        tma_store_boxes();
      } else if (args.tma_out && EPI == kEpiAddF32) {
        const float alpha = (args.row_alpha && gm < args.M) ? args.row_alpha[gm] : 1.0f;
        bool got = true;
        if (args.accumulate) {  // the old output of these rows and columns, by TMA
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(&epi_bar[warp - 2], 4 * 4096);
            for (int b = 0; b < 4; ++b)
              ptx::tma_load_2d(stg + b * 4096, &map_o, &epi_bar[warp - 2], n0 + cbeg + b * 32, m0 + q * 32);
          }
          got = ptx::mbar_wait(&epi_bar[warp - 2], 0, abort_flag);
          got = __all_sync(0xffffffffu, got);
          if (!got && lane == 0) {
            give_up();
            ptx::mbar_wait(&epi_bar[warp - 2], 0, nullptr);  // the copy lands before the smem goes
          }
        }
        if (got) {
#pragma unroll 1
          for (int c0 = cbeg; c0 < cend; c0 += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(t_row + c0, v);
            ptx::tmem_wait_ld();
            const int lc = c0 - cbeg;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const uint32_t at = stg_chunk(lc, g);
              float4 o = make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                     __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
              if (args.accumulate) {
                float4 p;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(p.x), "=f"(p.y), "=f"(p.z), "=f"(p.w)
                             : "r"(at));
                o.x = fmaf(p.x, alpha, o.x);
                o.y = fmaf(p.y, alpha, o.y);
                o.z = fmaf(p.z, alpha, o.z);
                o.w = fmaf(p.w, alpha, o.w);
              }
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(at), "f"(o.x), "f"(o.y), "f"(o.z),
                           "f"(o.w)
                           : "memory");
            }
          }
          tma_store_boxes();
        }
      } else if (EPI == kEpiStoreBF16) {
        uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
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
      } else if (EPI == kEpiAddF32) {  // direct stores
        float* out = reinterpret_cast<float*>(args.out);
        const float alpha = (args.row_alpha && gm < args.M) ? args.row_alpha[gm] : 1.0f;
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
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
                o.x = fmaf(p.x, alpha, o.x);
                o.y = fmaf(p.y, alpha, o.y);
                o.z = fmaf(p.z, alpha, o.z);
                o.w = fmaf(p.w, alpha, o.w);
              }
              dst[g] = o;
            }
          }
        }
      } else if (EPI == kEpiCEExp) {
        // This thread's row over its 128-column half tile: the max m (one
        // read of the accumulator), then P = bf16(exp(z - m)) to the chunk
        // scratch and the fp32 sum of exp(z - m) (a second read), both in a
        // fixed left-to-right order; the label's logit is gathered here too.
        uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
        const int lab = (gm < args.M) ? args.labels[gm] : args.ignore_index;
        float mx = -INFINITY;
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, v);
          ptx::tmem_wait_ld();
          if (n0 + c0 < args.N)
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(v[e]));
        }
        float sm = 0.0f;
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, v);
          ptx::tmem_wait_ld();
          if (n0 + c0 < args.N) {
            float f[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              f[e] = __expf(__uint_as_float(v[e]) - mx);
              sm += f[e];
            }
            if (args.tma_out) {
              const int lc = c0 - cbeg;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stg_chunk(lc, (lc % 64) / 8 + g)),
                             "r"(pack_bf16x2(f[8 * g + 0], f[8 * g + 1])), "r"(pack_bf16x2(f[8 * g + 2], f[8 * g + 3])),
                             "r"(pack_bf16x2(f[8 * g + 4], f[8 * g + 5])), "r"(pack_bf16x2(f[8 * g + 6], f[8 * g + 7]))
                             : "memory");
            } else if (gm < args.M) {
              uint4* dst = reinterpret_cast<uint4*>(out + static_cast<int64_t>(gm) * args.ld_out + n0 + c0);
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                uint4 o;
                o.x = pack_bf16x2(f[8 * g + 0], f[8 * g + 1]);
                o.y = pack_bf16x2(f[8 * g + 2], f[8 * g + 3]);
                o.z = pack_bf16x2(f[8 * g + 4], f[8 * g + 5]);
                o.w = pack_bf16x2(f[8 * g + 6], f[8 * g + 7]);
                dst[g] = o;
              }
            }
            const int vid = args.vocab_base + n0 + c0;
            if (lab >= vid && lab < vid + 32 && gm < args.M) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (lab == vid + e) args.label_logit[gm] = __uint_as_float(v[e]);
            }
          }
        }
        if (args.tma_out) tma_store_boxes();
        if (gm < args.M) {
          const int64_t p = static_cast<int64_t>(gm) * args.part_ld + 2 * blockIdx.x + ch;
          args.part_max[p] = mx;
          args.part_sum[p] = sm;
        }
      }
    } else if (!*abort_flag) {
      give_up();
    }
  }
  __syncwarp();
  if (args.clk) ptx::bulk_wait0();  // this thread's output stores complete before the end stamp

  ptx::tc_fence_before();
  __syncthreads();
  clk_end(args);
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
  int grouped;           // a projection group: persistent CTA-pair kernel (NF4, M > 128) required
  // double-quantised absmax (args.dq): int8 [weight K / 64][q_ld], (c, s) pairs [weight K / 64][a2_ld]
  const int8_t* qabsmax;
  int64_t q_ld;
  const float* absmax2;
  int64_t a2_ld;
  // scratch for splitting the persistent kernel's last partial wave along K
  // (split_scratch_bytes(); 256-byte aligned); nullptr: no split
  void* split_ws;
  size_t split_ws_bytes;
};

sl_status launch_gemm(const GemmLaunch& g, cudaStream_t stream);
// Scratch that lets a persistent pair GEMM split its last partial wave
// along K: a flag and a [2][256][128] fp32 partial tile per piece, for up to
// one piece per resident cluster.
size_t split_scratch_bytes();

}  // namespace sl
