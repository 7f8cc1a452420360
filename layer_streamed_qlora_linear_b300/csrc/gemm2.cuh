// The fused NF4 GEMM on a CTA pair (tcgen05.mma.cta_group::2), M = 256 per pair.
//
// Same computation as gemm_tc_kernel<kBSrcNF4, ...> (see gemm.cuh), laid
// out across the two CTAs of a cluster:
//   * each CTA brings in (TMA) its own 128 rows of A and the packed NF4
//     codes + absmax of its own 128-row half of the 256-row B tile, and its
//     8 dequant warps expand only that half;
//   * the leader CTA (rank 0) issues tcgen05.mma.cta_group::2 (M = 256,
//     N = 256); the tensor core reads A and B halves from both CTAs' shared
//     memory at the same offsets and writes each CTA's 128 accumulator rows
//     into that CTA's TMEM;
//   * A tiles of both CTAs complete on the leader's `full` barrier (TMA
//     .cta_group::2); the leader's dequant warps arrive on `full` too, the
//     peer's on their local `b_local`, and one thread of the peer forwards
//     that to the leader's `full` as a 16-byte async-proxy copy
//     (complete_tx): the MMA issuer waits once per k-block; MMA
//     completion is multicast to both CTAs' `empty` / `main_done` /
//     `acc_full` barriers.
// Per SM this halves the dequant work of every k-block while keeping one
// 128-row accumulator per SM, so small-M problems keep their parallelism.
// Every wait is bounded like in gemm.cuh.
#pragma once
#include "gemm.cuh"

namespace sl {

constexpr int kHalfBTileBytes = 128 * kBK * 2;   // 16 KB: this CTA's half of the B tile
constexpr int kHalfCodesBytes = 128 * kBK / 2;   // 4 KB of packed codes
constexpr int kPairAbsBytes = 128 * 16;          // 2 KB: K-major box 4 x 128 (MN-major uses 1 KB)
constexpr int kNumDq2 = 256;
constexpr int kGemm2Threads = 64 + kNumDq2;

struct Gemm2Cfg {
  static constexpr int S = 5;
  static constexpr int kRawBytes = kHalfCodesBytes + kPairAbsBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + S * kATileBytes;
  static constexpr int kOffRaw = kOffB + S * kHalfBTileBytes;
  static constexpr int kOffBar = kOffRaw + S * kRawBytes;
  static constexpr int kNumBars = 4 * S + 3;
  static constexpr int kOffSink = (kOffBar + kNumBars * 8 + 15) / 16 * 16;  // 16-byte signal landing pad
  static constexpr int kOffMisc = kOffSink + 16;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kSmem = kBytes + 1024;
};

// NW words (8 NF4 codes each) with one absmax -> NW sixteen-byte chunks of a
// 128-byte swizzled row, logical chunks chunk0 .. chunk0 + NW - 1.
template <int NW>
__device__ __forceinline__ void nf4_words_bf16(const uint32_t (&words)[NW], float amax, uint8_t* row, int chunk0,
                                               int rsw) {
  uint32_t P[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    P[i] = pack_bf16x2(__fmul_rn(__uint_as_float(d_nf4_level_bits[2 * i]), amax),
                       __fmul_rn(__uint_as_float(d_nf4_level_bits[2 * i + 1]), amax));
  const uint32_t L0 = prmt(P[0], P[1], 0x6420), H0 = prmt(P[0], P[1], 0x7531);
  const uint32_t L1 = prmt(P[2], P[3], 0x6420), H1 = prmt(P[2], P[3], 0x7531);
  const uint32_t L2 = prmt(P[4], P[5], 0x6420), H2 = prmt(P[4], P[5], 0x7531);
  const uint32_t L3 = prmt(P[6], P[7], 0x6420), H3 = prmt(P[6], P[7], 0x7531);
#pragma unroll
  for (int j = 0; j < NW; ++j) {
    const uint32_t w = words[j];
    const uint32_t w4 = w << 4;
    const uint32_t s7 = w & 0x77777777u;
    const uint32_t sA = s7, sB = s7 >> 16;
    const uint32_t mA = prmt(w4, w, 0xD9C8), mB = prmt(w4, w, 0xFBEA);
    const uint32_t loA = select_bytes(prmt(L0, L1, sA), prmt(L2, L3, sA), mA);
    const uint32_t hiA = select_bytes(prmt(H0, H1, sA), prmt(H2, H3, sA), mA);
    const uint32_t loB = select_bytes(prmt(L0, L1, sB), prmt(L2, L3, sB), mB);
    const uint32_t hiB = select_bytes(prmt(H0, H1, sB), prmt(H2, H3, sB), mB);
    uint4 o;
    o.x = prmt(loA, hiA, 0x4051);
    o.y = prmt(loA, hiA, 0x6273);
    o.z = prmt(loB, hiB, 0x4051);
    o.w = prmt(loB, hiB, 0x6273);
    *reinterpret_cast<uint4*>(row + (((chunk0 + j) ^ rsw) << 4)) = o;
  }
}

template <int BMN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemm2Threads, 1)
    gemm_nf4_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_c,
                         const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_o,
                         const GemmArgs args) {
  using Cfg = Gemm2Cfg;
  constexpr int S = Cfg::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = ptx::align1024(smem_raw);
  uint8_t* sA = smem + Cfg::kOffA;
  uint8_t* sB = smem + Cfg::kOffB;
  uint8_t* sRaw = smem + Cfg::kOffRaw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  uint64_t* full = bars;               // leader: stage ready (A of both CTAs, both B halves)
  uint64_t* raw_full = bars + S;       // each CTA: its codes + absmax landed
  uint64_t* b_local = bars + 2 * S;    // peer: its own B half dequantised (4 warps of one group)
  uint64_t* empty = bars + 3 * S;      // each CTA: stage consumed by the MMAs
  uint64_t* lora_full = bars + 4 * S;  // leader: both CTAs staged the LoRA operands
  uint64_t* acc_full = bars + 4 * S + 1;
  uint64_t* main_done = bars + 4 * S + 2;
  uint8_t* sink = smem + Cfg::kOffSink;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int m0 = (blockIdx.x >> 1) * 256 + static_cast<int>(rank) * 128;  // this CTA's A rows
  const int n0 = blockIdx.y * kBN;                                          // the pair's 256 columns
  const int nh = n0 + static_cast<int>(rank) * 128;                         // this CTA's half of B
  const int KB = (args.K + kBK - 1) / kBK;
  const bool has_lora = args.lora_x != nullptr && args.r > 0;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(&full[i], 1 + kNumDq2 / 64);  // producer + the 4 warps of the owning dequant group
      ptx::mbar_init(&raw_full[i], 1);
      ptx::mbar_init(&b_local[i], kNumDq2 / 64);  // the 4 warps of the group that owns this k-block
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(lora_full, 2 * (kNumDq2 / 32));
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(main_done, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&map_a);
    ptx::tma_prefetch_desc(&map_c);
    ptx::tma_prefetch_desc(&map_s);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, 256);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  pdl_trigger();  // the next kernel may start its prologue
  pdl_wait();     // the previous kernel's writes are visible from here on
  clk_start(args);

  auto give_up = [&]() {
    *abort_flag = 1;
    report_device_error(args.err, SL_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t rawtx = kHalfCodesBytes + (BMN ? kBK * 16 : 128 * 16);
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % S;
        if (!ptx::mbar_wait_cluster(&empty[s], ((kb / S) & 1) ^ 1, abort_flag)) {
          give_up();
          break;
        }
        if (leader) ptx::mbar_arrive_expect_tx(&full[s], 2 * kATileBytes + 16);  // + the peer's signal
        ptx::tma_load_2d_pair(sA + s * kATileBytes, &map_a, ptx::map_to_rank(&full[s], 0), kb * kBK, m0);
        uint8_t* raw = sRaw + s * Cfg::kRawBytes;
        ptx::mbar_arrive_expect_tx(&raw_full[s], rawtx);
        if (!BMN) {
          ptx::tma_load_2d(raw, &map_c, &raw_full[s], kb * (kBK / 2), nh);
          ptx::tma_load_2d(raw + kHalfCodesBytes, &map_s, &raw_full[s], kb & ~3, nh);
        } else {
          ptx::tma_load_2d(raw, &map_c, &raw_full[s], nh / 2, kb * kBK);
          ptx::tma_load_2d(raw + kHalfCodesBytes, &map_s, &raw_full[s], n0 / 64, kb * kBK);
        }
        ++issued;
      }
      if (*abort_flag) {
        for (int kb = (issued > S ? issued - S : 0); kb < issued; ++kb)
          ptx::mbar_wait_cluster(&raw_full[kb % S], (kb / S) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = ptx::idesc_bf16(256, kBN, 0, BMN);
      const uint32_t a_base = ptx::smem_addr(sA);
      const uint32_t b_base = ptx::smem_addr(sB);
      // descriptors of stage 0, k-step 0; the start-address field sits in the
      // low word below 2^14, so a stage / k-step offset is a 32-bit add
      const uint64_t a_desc0 = ptx::smem_desc(a_base, 16, 1024, 2);
      const uint64_t b_desc0 = BMN ? ptx::smem_desc(b_base, 64 * 128, 1024, 2) : ptx::smem_desc(b_base, 16, 1024, 2);
      const uint32_t a_lo0 = static_cast<uint32_t>(a_desc0), a_hi = static_cast<uint32_t>(a_desc0 >> 32);
      const uint32_t b_lo0 = static_cast<uint32_t>(b_desc0), b_hi = static_cast<uint32_t>(b_desc0 >> 32);
      constexpr uint32_t kBStep = BMN ? 2048 : 32;
      bool ok = true;
      int s = 0;
      uint32_t ph = 0;
      for (int kb = 0; kb < KB && ok; ++kb) {
        if (!ptx::mbar_wait_cluster(&full[s], ph, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(s) * (kATileBytes >> 4);
        const uint32_t b_lo = b_lo0 + static_cast<uint32_t>(s) * (kHalfBTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          ptx::mma_bf16_pair_lohi(tmem, a_lo + kk * (32 >> 4), a_hi, b_lo + kk * (kBStep >> 4), b_hi, idesc,
                                  (kb | kk) ? 1u : 0u);
        ptx::mma_commit_pair(&empty[s], 0x3);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok && has_lora) {
        ptx::mma_commit_pair(main_done, 0x3);
        if (!ptx::mbar_wait_cluster(lora_full, 0, abort_flag)) {
          give_up();
          ok = false;
        } else {
          ptx::tc_fence_after();
          const int s = KB % S;
          const int ksteps = (2 * args.r + 15) / 16;
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint64_t ad = ptx::smem_desc(a_base + s * kATileBytes + kk * 32, 16, 1024, 2);
            const uint64_t bd = BMN ? ptx::smem_desc(b_base + s * kHalfBTileBytes + kk * 2048, 64 * 128, 1024, 2)
                                    : ptx::smem_desc(b_base + s * kHalfBTileBytes + kk * 32, 16, 1024, 2);
            ptx::mma_bf16_pair(tmem, ad, bd, idesc, 1u);
          }
        }
      }
      ptx::mma_commit_pair(acc_full, 0x3);
      if (!ok) ptx::mbar_wait_cluster(acc_full, 0, nullptr);
    } else if (lane == 0) {
      // Peer CTA: tell the leader "my B half of stage s is ready" once the
      // local dequant warps have arrived (their smem writes were fenced for
      // the async proxy), with a 16-byte async-proxy copy that completes on
      // the leader's full[s] -- no memory fence on this path.
      const uint32_t leader_full = ptx::map_to_rank(&full[0], 0);
      const uint32_t leader_sink = ptx::map_to_rank(sink, 0);
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % S;
        if (!ptx::mbar_wait(&b_local[s], (kb / S) & 1, abort_flag)) {
          give_up();
          break;
        }
        ptx::bulk_signal_16(leader_sink, sink, leader_full + s * 8);
      }
    }
  } else {
    // -------------------------------- dequant / LoRA staging / epilogue (each CTA)
    const int dq = tid - 64;  // 0..255
    bool ok = true;
    const int r = args.r;
    const int nr = r / 8;
    const int kpad = ((2 * r + 15) / 16) * 16;
    const int nchunk = kpad / 8;
    const bool xe_row = dq < 128;  // this CTA's 128 rows of Xe
    auto chunk_at = [&](uint8_t* base, int row, int c) {
      return reinterpret_cast<uint4*>(base + row * 128 + ((c ^ (row & 7)) << 4));
    };
    auto mn_chunk = [&](uint8_t* bt, int i, int cc) {  // cc: 0..15 (two 64-column atoms)
      return reinterpret_cast<uint4*>(bt + (cc >> 3) * (64 * 128) + i * 128 + (((cc & 7) ^ (i & 7)) << 4));
    };
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
    // Be tasks.  K-major: rows j = dq < 128 of this CTA's half, rank groups
    // t < nr.  MN-major: task dq + 256 t over (rank row i, chunk cc of 16).
    const int nbe = BMN ? (r * 16 + kNumDq2 - 1) / kNumDq2 : nr;
    auto be_valid = [&](int t) { return BMN ? (dq + kNumDq2 * t < r * 16) : (dq < 128 && t < nr); };
    auto load_be = [&](int t) -> uint4 {
      if (!BMN) {
        const int gn = nh + dq;
        if (gn < args.N) return *reinterpret_cast<const uint4*>(args.lora_w + static_cast<int64_t>(gn) * r + t * 8);
      } else {
        const int task = dq + kNumDq2 * t;
        const int i = task >> 4, gcol = nh + (task & 15) * 8;
        if (gcol < args.N) return *reinterpret_cast<const uint4*>(args.lora_w + static_cast<int64_t>(i) * args.N + gcol);
      }
      return make_uint4(0, 0, 0, 0);
    };
    auto store_be = [&](uint8_t* bt, int t, uint4 v) {
      if (!BMN) {
        *chunk_at(bt, dq, t) = v;
        *chunk_at(bt, dq, nr + t) = v;
      } else {
        const int task = dq + kNumDq2 * t;
        const int i = task >> 4, cc = task & 15;
        *mn_chunk(bt, i, cc) = v;
        *mn_chunk(bt, r + i, cc) = v;
      }
    };
    auto store_pad = [&](uint8_t* at, uint8_t* bt) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int c = 2 * nr; c < nchunk; ++c) {
        if (xe_row) *chunk_at(at, dq, c) = z;
        if (!BMN && dq < 128) *chunk_at(bt, dq, c) = z;
      }
      if (BMN)
        for (int task = dq; task < (kpad - 2 * r) * 16; task += kNumDq2)
          *mn_chunk(bt, 2 * r + (task >> 4), task & 15) = z;
    };
    const bool lora_pref = has_lora && r <= 16;
    float pre_x[2][8];
    uint4 pre_b[2];
    if (lora_pref) {
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (xe_row && g < nr) load_xe(g, pre_x[g]);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (t < nbe && be_valid(t)) pre_b[t] = load_be(t);
    }

    // Two groups of four warps take alternate k-blocks; each thread expands
    // one full 64-element row (one 16-entry table per row and k-block).
    const int grp = (warp - 2) >> 2;  // 0: even k-blocks, 1: odd
    const int t = dq & 127;
    for (int kb = grp; kb < KB; kb += 2) {
      const int s = kb % S;
      if (!ptx::mbar_wait_cluster(&raw_full[s], (kb / S) & 1, abort_flag)) {
        give_up();
        ok = false;
        break;
      }
      const uint8_t* codes = sRaw + s * Cfg::kRawBytes;
      const float* amax = reinterpret_cast<const float*>(codes + kHalfCodesBytes);
      uint8_t* bt = sB + s * kHalfBTileBytes;
      if (!BMN) {  // row t of the [128 x 64] half tile
        const uint4 q0 = *reinterpret_cast<const uint4*>(codes + t * 32);
        const uint4 q1 = *reinterpret_cast<const uint4*>(codes + t * 32 + 16);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        nf4_words_bf16<8>(w, amax[t * 4 + (kb & 3)], bt + t * 128, 0, t & 7);
      } else {     // reduction row n, 64-column atom a (of 2)
        // eight consecutive lanes (one 128-byte store phase) take eight rows
        // n with distinct n % 8, so their swizzled chunks fall in different banks
        const int n = ((t >> 5) << 4) | (t & 7) | ((t >> 1) & 8);
        const int a = ((t >> 1) ^ (t >> 3)) & 1;
        const uint4 q0 = *reinterpret_cast<const uint4*>(codes + n * 64 + a * 32);
        const uint4 q1 = *reinterpret_cast<const uint4*>(codes + n * 64 + a * 32 + 16);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        nf4_words_bf16<8>(w, amax[n * 4 + 2 * static_cast<int>(rank) + a], bt + a * (64 * 128) + n * 128, 0,
                          n & 7);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(leader ? &full[s] : &b_local[s]);
    }
    if (ok && has_lora) {
      const int s = KB % S;
      if (!ptx::mbar_wait_cluster(main_done, 0, abort_flag)) {
        give_up();
        ok = false;
      } else {
        uint8_t* at = sA + s * kATileBytes;
        uint8_t* bt = sB + s * kHalfBTileBytes;
        if (lora_pref) {
#pragma unroll
          for (int g = 0; g < 2; ++g)
            if (xe_row && g < nr) store_xe(at, g, pre_x[g]);
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (t < nbe && be_valid(t)) store_be(bt, t, pre_b[t]);
        } else {
          for (int g = 0; g < nr && xe_row; ++g) {
            float v[8];
            load_xe(g, v);
            store_xe(at, g, v);
          }
          for (int t = 0; t < nbe; ++t)
            if (be_valid(t)) store_be(bt, t, load_be(t));
        }
        store_pad(at, bt);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ptx::map_to_rank(lora_full, 0));
      }
    }
    // ---------------------------------------------------------------- epilogue
    bool acc_ready = ptx::mbar_wait_cluster(acc_full, 0, abort_flag) && !*abort_flag;
    acc_ready = __all_sync(0xffffffffu, acc_ready);
    if (acc_ready) {
      ptx::tc_fence_after();
      const int q = warp & 3;
      const int ch = (warp - 2) >> 2;
      const int cbeg = ch * (kBN / 2), cend = cbeg + kBN / 2;
      const int row = q * 32 + lane;
      const int gm = m0 + row;
      const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16);
      uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
      if (args.tma_out) {
        // Every MMA of the pair has completed, so the stage buffers are free:
        // this warp's 32 rows x 128 columns leave as two 64-column bf16 TMA
        // boxes (128-byte swizzle); the tensor map clips rows and columns past
        // the output.
        uint8_t* stg = smem + (warp - 2) * 8192;
        const uint32_t stg_a = ptx::smem_addr(stg);
#pragma unroll 1
        for (int c0 = cbeg; c0 < cend; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, v);
          ptx::tmem_wait_ld();
          const int lc = c0 - cbeg;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             stg_a + (lc / 64) * 4096 + lane * 128 + ((((lc % 64) / 8 + g) ^ (lane & 7)) << 4)),
                         "r"(pack_bf16x2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]))),
                         "r"(pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]))),
                         "r"(pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]))),
                         "r"(pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7])))
                         : "memory");
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(&map_o, stg, n0 + cbeg, m0 + q * 32);
          ptx::tma_store_2d(&map_o, stg + 4096, n0 + cbeg + 64, m0 + q * 32);
          ptx::bulk_commit();
          ptx::bulk_wait_read0();  // the staging is read before the CTA's shared memory goes
        }
        __syncwarp();
      } else {
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
  ptx::cluster_sync();  // neither CTA leaves while the pair's MMAs may still read its smem
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 256);
  }
}

}  // namespace sl
