// Persistent fused NF4 GEMM on CTA pairs (tcgen05.mma.cta_group::2).
//
// The computation and the per-k-block pipeline are those of
// gemm_nf4_pair_kernel (gemm2.cuh); this kernel adds:
//   * persistence: one cluster (two SMs) per SM pair walks its share of the
//     256 x 256 pair tiles; the stage ring runs on across tiles;
//   * two TMEM accumulators (2 x 256 columns): four epilogue warps drain one
//     while the MMAs of the next tile fill the other (acc_full / acc_empty);
//   * the LoRA side product is folded after the last k-block of a tile from
//     a dedicated shared-memory region that the epilogue warps fill while
//     the tile's main loop runs (lora_full / lora_empty): no pipeline drain,
//     and the dequant warps carry no LoRA state;
//   * projection groups (q, k, v or gate, up stored back to back along N):
//     in the forward each tile folds the side product of the projection it
//     lies in (T_cat columns g r .., row stride G r); the grouped dX is the
//     plain fold at rank G r (s U_cat A_cat), up to 64;
// The MMA issuer waits once per k-block: the leader's full[s] counts the A
// tiles of both CTAs, the leader's own dequant warps and the peer's
// forwarded "B half ready" signal.
// Warps: 0 A/code TMA producer, 1 MMA issuer (leader) or peer forwarder,
// 2..9 NF4 dequant (two groups on alternate k-blocks), 10..13 LoRA staging +
// epilogue.  Every wait is bounded.
// gemm_bf16_pair_persistent_kernel is the same kernel for a bf16 (unquantised)
// weight: each CTA's producer loads its B half by TMA next to its A tile, both
// counted on the leader's full[s], and warps 2..9 have no work.
#pragma once
#include "gemm2.cuh"

namespace sl {

constexpr int kNumEpi3 = 128;
constexpr int kGemm3Threads = 64 + kNumDq2 + kNumEpi3;

constexpr int kLoraMaxR = 64;               // folded rank: K of the fold up to 2 * 64
constexpr int kLoraAtom = 128 * 128;         // one 128-row x 128-byte SW128 atom

// SMALL = 1: folded rank at most 32 (2R <= 64 K columns): the LoRA operands
// take one atom each (32 KB), which leaves room for a fifth pipeline stage;
// SMALL = 0: folded rank up to 64 (a projection group's dX), four stages.
template <int SMALL>
struct Gemm3Cfg {
  static constexpr int S = SMALL ? 5 : 4;
  static constexpr int kLA = SMALL ? 1 : 2;                       // Xe atoms (64 K columns each)
  static constexpr int kLBAtomMN = SMALL ? 64 * 128 : kLoraAtom;  // MN-major Be atom: 2R rows of 128 bytes
  static constexpr int kLBBytes = SMALL ? kLoraAtom : 2 * kLoraAtom;
  static constexpr int kRawBytes = kHalfCodesBytes + kPairAbsBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + S * kATileBytes;
  static constexpr int kOffLA = kOffB + S * kHalfBTileBytes;     // LoRA Xe: K-major [128 rows x 2R], kLA atoms
  static constexpr int kOffLB = kOffLA + kLA * kLoraAtom;        // LoRA Be: K-major [128 x 2r] / MN-major 2 atoms of [2R x 64]
  static constexpr int kOffRaw = kOffLB + kLBBytes;
  static constexpr int kOffBar = kOffRaw + S * kRawBytes;
  static constexpr int kNumBars = 4 * S + 7;
  static constexpr int kOffSink = (kOffBar + kNumBars * 8 + 15) / 16 * 16;
  static constexpr int kOffMisc = kOffSink + 16;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kSmem = kBytes + 1024;
};
static_assert(Gemm3Cfg<0>::kSmem <= 232448 && Gemm3Cfg<1>::kSmem <= 232448, "persistent GEMM shared memory");
// the epilogue's TMA staging (4 warps x 8 KB) lives in the LoRA region
static_assert(Gemm3Cfg<1>::kOffLA % 1024 == 0 && Gemm3Cfg<1>::kLA * kLoraAtom + Gemm3Cfg<1>::kLBBytes >= 4 * 8192 &&
                  Gemm3Cfg<0>::kOffLA % 1024 == 0 && Gemm3Cfg<0>::kLA * kLoraAtom + Gemm3Cfg<0>::kLBBytes >= 4 * 8192,
              "persistent GEMM epilogue staging");

// Barrier of the four epilogue warps only (named barrier 1).
__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kNumEpi3) : "memory"); }

// The kernel body, over the weight source: BF16 = 0 NF4 (codes + absmax by
// TMA, dequantised by warps 2..9 into the B halves), BF16 = 1 bf16 weights
// (each CTA's B half by TMA straight into the operand layout, counted on the
// leader's full[s] like the A tiles; warps 2..9 and the peer forwarder idle).
// map_c: NF4 codes / the bf16 weight; map_s, map_s2: absmax (NF4 only).
template <int BF16, int BMN, int SMALL, int EPI>
__device__ __forceinline__ void pair_persistent_body(const CUtensorMap& map_a, const CUtensorMap& map_c,
                                                     const CUtensorMap& map_s, const CUtensorMap& map_s2,
                                                     const CUtensorMap& map_o, const GemmArgs& args) {
  using Cfg = Gemm3Cfg<SMALL>;
  constexpr int S = Cfg::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = ptx::align1024(smem_raw);
  uint8_t* sA = smem + Cfg::kOffA;
  uint8_t* sB = smem + Cfg::kOffB;
  uint8_t* sLA = smem + Cfg::kOffLA;
  uint8_t* sLB = smem + Cfg::kOffLB;
  uint8_t* sRaw = smem + Cfg::kOffRaw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kOffBar);
  // full[s] (leader) completes when stage s is ready for the MMAs: the A
  // tiles of both CTAs landed (TMA bytes), the leader's B half is
  // dequantised (4 warp arrivals) and the peer's is (a 16-byte async-proxy
  // signal from the peer, counted as bytes) -- one wait per k-block.
  uint64_t* full = bars;                 // [S] leader: stage s ready for the MMAs
  uint64_t* raw_full = bars + S;         // [S] each CTA: codes + absmax landed
  uint64_t* b_local = bars + 2 * S;      // [S] peer: its B half dequantised (4 warps of one group)
  uint64_t* empty = bars + 3 * S;        // [S] each CTA: stage consumed by the MMAs
  uint64_t* lora_full = bars + 4 * S;    // leader: both CTAs staged this tile's LoRA operands
  uint64_t* lora_empty = lora_full + 1;  // each CTA: the fold MMAs of the previous tile are done with them
  uint64_t* acc_full = lora_full + 2;    // [2] each CTA: accumulator a holds a finished segment
  uint64_t* acc_empty = lora_full + 4;   // [2] leader: both CTAs' epilogues drained accumulator a
  uint64_t* drain = lora_full + 6;       // leader, failure path only: issued MMAs completed
  uint8_t* sink = smem + Cfg::kOffSink;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);
  volatile int* epi_stop = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 8);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int mpairs = (args.M + 255) / 256;
  const int ntiles_n = (args.N + kBN - 1) / kBN;
  const int ntiles = mpairs * ntiles_n;
  const int KB = (args.K + kBK - 1) / kBK;
  const bool has_lora = args.lora_x != nullptr && args.r > 0;
  // pair tile t -> (m pair, n tile); concurrent clusters share the n tile (weight reuse in L2)
  auto tile_m0 = [&](int t) { return (t % mpairs) * 256 + static_cast<int>(rank) * 128; };
  auto tile_n0 = [&](int t) { return (t / mpairs) * kBN; };
  // This cluster's work items, the same list for every role: its full tiles
  // (cluster, cluster + nclusters, ...) and, when the last partial wave is
  // split along K, one piece of a tail tile (piece 0 folds the side product
  // and adds the other pieces' partial sums in piece order).
  const int split_P = args.split_P;
  const bool split = split_P >= 2;
  const int rounds = split ? args.split_rounds : (ntiles - cluster + nclusters - 1) / nclusters;
  const int n_items = rounds + ((split && cluster < args.split_R * split_P) ? 1 : 0);
  struct Item {
    int t, kb0, kb1, piece, slot0;  // piece -1: a full tile
  };
  auto item = [&](int i) {
    Item x;
    if (i < rounds) {
      x.t = cluster + i * nclusters;
      x.kb0 = 0;
      x.kb1 = KB;
      x.piece = -1;
      x.slot0 = 0;
    } else {
      const int j = cluster / split_P, p = cluster % split_P;
      x.t = rounds * nclusters + j;
      x.kb0 = p * KB / split_P;
      x.kb1 = (p + 1) * KB / split_P;
      x.piece = p;
      x.slot0 = j * (split_P - 1);
    }
    return x;
  };

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      ptx::mbar_init(&full[i], BF16 ? 1 : 1 + kNumDq2 / 64);  // producer (+ the 4 warps of the owning dequant group)
      ptx::mbar_init(&raw_full[i], 1);
      ptx::mbar_init(&b_local[i], kNumDq2 / 64);
      ptx::mbar_init(&empty[i], 1);
    }
    ptx::mbar_init(lora_full, 2 * (kNumEpi3 / 32));
    ptx::mbar_init(lora_empty, 1);
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 2 * (kNumEpi3 / 32));
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    *epi_stop = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&map_a);
    ptx::tma_prefetch_desc(&map_c);
    if (!BF16) ptx::tma_prefetch_desc(&map_s);
    if (!BF16 && args.dq) ptx::tma_prefetch_desc(&map_s2);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, 512);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
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
      // absmax per stage: fp32 (K-major 4 x 128, MN-major 4 x 64) or, double
      // quantised, 128 int8 + 16 B (K-major) / 32 B (MN-major) of (c, s) pairs
      const uint32_t rawtx =
          kHalfCodesBytes + (args.dq ? (128 + (BMN ? 32 : 16)) : (BMN ? kBK * 16 : 128 * 16));
      int g = 0;  // k-blocks issued by this cluster
      bool ok = true;
      for (int i = 0; ok && i < n_items; ++i) {
        const Item x = item(i);
        const int t = x.t;
        const int m0 = tile_m0(t), n0 = tile_n0(t), nh = n0 + static_cast<int>(rank) * 128;
        for (int kb = x.kb0; kb < x.kb1; ++kb, ++g) {
          const int s = g % S;
          if (!ptx::mbar_wait_cluster(&empty[s], ((g / S) & 1) ^ 1, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          // A tiles of both CTAs and the peer's 16-byte "B half ready" signal
          // (bf16 weights: the B halves of both CTAs instead)
          if (leader) ptx::mbar_arrive_expect_tx(&full[s], BF16 ? 2 * (kATileBytes + kHalfBTileBytes) : 2 * kATileBytes + 16);
          ptx::tma_load_2d_pair(sA + s * kATileBytes, &map_a, ptx::map_to_rank(&full[s], 0), kb * kBK, m0);
          if (BF16) {  // this CTA's 128 weight rows (K-major) / columns (MN-major, two 64-column atoms)
            uint8_t* bt = sB + s * kHalfBTileBytes;
            if (!BMN) {
              ptx::tma_load_2d_pair(bt, &map_c, ptx::map_to_rank(&full[s], 0), kb * kBK, nh);
            } else {
              ptx::tma_load_2d_pair(bt, &map_c, ptx::map_to_rank(&full[s], 0), nh, kb * kBK);
              ptx::tma_load_2d_pair(bt + 64 * 128, &map_c, ptx::map_to_rank(&full[s], 0), nh + 64, kb * kBK);
            }
            continue;
          }
          uint8_t* raw = sRaw + s * Cfg::kRawBytes;
          ptx::mbar_arrive_expect_tx(&raw_full[s], rawtx);
          if (!BMN) {
            ptx::tma_load_2d(raw, &map_c, &raw_full[s], kb * (kBK / 2), nh);
            if (!args.dq) {
              ptx::tma_load_2d(raw + kHalfCodesBytes, &map_s, &raw_full[s], kb & ~3, nh);
            } else {  // int8 absmax of rows nh .. nh+127 at block kb; their (c, s) pair
              const int col = args.dq_col0 + nh;
              ptx::tma_load_2d(raw + kHalfCodesBytes, &map_s, &raw_full[s], col, kb);
              // the 16-byte box at x = 4 (col / 512) (TMA: x * 4 B on a 16-byte
              // boundary) holds the pairs of 256-blocks 2 (col / 512) and + 1
              ptx::tma_load_2d(raw + kHalfCodesBytes + 128, &map_s2, &raw_full[s], 4 * (col / 512), kb);
            }
          } else {
            ptx::tma_load_2d(raw, &map_c, &raw_full[s], nh / 2, kb * kBK);
            if (!args.dq) {
              ptx::tma_load_2d(raw + kHalfCodesBytes, &map_s, &raw_full[s], n0 / 64, kb * kBK);
            } else {  // int8 absmax of weight rows kb*64 .. +63 at blocks nh/64, +1; their (c, s) pairs
              const int col = args.dq_col0 + kb * kBK;
              ptx::tma_load_2d(raw + kHalfCodesBytes, &map_s, &raw_full[s], col, nh / 64);
              ptx::tma_load_2d(raw + kHalfCodesBytes + 128, &map_s2, &raw_full[s], 4 * (col / 512), nh / 64);
            }
          }
        }
      }
      if (!ok && !BF16) {
        for (int k = (g > S ? g - S : 0); k < g; ++k) ptx::mbar_wait_cluster(&raw_full[k % S], (k / S) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16(256, kBN, 0, BMN);
      const uint32_t a_base = ptx::smem_addr(sA);
      const uint32_t b_base = ptx::smem_addr(sB);
      const uint32_t la = ptx::smem_addr(sLA);
      const uint32_t lb = ptx::smem_addr(sLB);
      // descriptors of stage 0, k-step 0; a stage / k-step adds its byte
      // offset / 16 to the start-address field (bits 0..13)
      const uint64_t a_desc0 = ptx::smem_desc(a_base, 16, 1024, 2);
      const uint64_t b_desc0 = BMN ? ptx::smem_desc(b_base, 64 * 128, 1024, 2) : ptx::smem_desc(b_base, 16, 1024, 2);
      // the start-address field is in the low word and stays below 2^14
      // (shared memory < 256 KB): stepping it is a 32-bit add
      const uint32_t a_lo0 = static_cast<uint32_t>(a_desc0), a_hi = static_cast<uint32_t>(a_desc0 >> 32);
      const uint32_t b_lo0 = static_cast<uint32_t>(b_desc0), b_hi = static_cast<uint32_t>(b_desc0 >> 32);
      constexpr uint32_t kBStep = BMN ? 2048 : 32;  // bytes between k16 steps of the B half
      const int ksteps = has_lora ? (2 * args.r + 15) / 16 : 0;
      int g = 0, it = 0, lit = 0;  // k-blocks, items and folded items of this cluster
      bool ok = true;
      for (; ok && it < n_items; ++it) {
        const Item x = item(it);
        const bool fold = has_lora && x.piece <= 0;
        const int acc = it & 1;
        const uint32_t d = tmem + static_cast<uint32_t>(acc * kBN);
        if (!ptx::mbar_wait_cluster(&acc_empty[acc], ((it >> 1) & 1) ^ 1, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        int s = g % S;                       // stage and phase, stepped without division
        uint32_t ph = (g / S) & 1;
        for (int kb = x.kb0; kb < x.kb1; ++kb, ++g) {
          if (!ptx::mbar_wait_cluster(&full[s], ph, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(s) * (kATileBytes >> 4);
          const uint32_t b_lo = b_lo0 + static_cast<uint32_t>(s) * (kHalfBTileBytes >> 4);
          const uint32_t first = kb == x.kb0 ? 0u : 1u;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::mma_bf16_pair_lohi(d, a_lo + kk * (32 >> 4), a_hi, b_lo + kk * (kBStep >> 4), b_hi, idesc,
                                    (first | kk) ? 1u : 0u);
          ptx::mma_commit_pair(&empty[s], 0x3);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (fold) {  // fold the LoRA side product into this accumulator
          if (!ptx::mbar_wait_cluster(lora_full, lit & 1, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint64_t ad = ptx::smem_desc(la + (kk >> 2) * kLoraAtom + (kk & 3) * 32, 16, 1024, 2);
            const uint64_t bd = BMN ? ptx::smem_desc(lb + kk * 2048, Cfg::kLBAtomMN, 1024, 2)
                                    : ptx::smem_desc(lb + kk * 32, 16, 1024, 2);
            ptx::mma_bf16_pair(d, ad, bd, idesc, 1u);
          }
          ptx::mma_commit_pair(lora_empty, 0x3);
          ++lit;
        }
        ptx::mma_commit_pair(&acc_full[acc], 0x3);
      }
      if (!ok) {  // let the MMAs already issued finish before teardown
        ptx::mma_commit_pair(drain, 0x1);
        ptx::mbar_wait(drain, 0, nullptr);
      }
    } else if (lane == 0 && !BF16) {
      // -------------------------------------------------- peer: B-ready forwarder
      // (a 16-byte async-proxy copy whose bytes complete on the leader's full[s])
      const uint32_t leader_full = ptx::map_to_rank(&full[0], 0);
      const uint32_t leader_sink = ptx::map_to_rank(sink, 0);
      int g = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_items; ++i) {
        const Item x = item(i);
        for (int kb = x.kb0; kb < x.kb1; ++kb, ++g) {
          const int s = g % S;
          if (!ptx::mbar_wait(&b_local[s], (g / S) & 1, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          ptx::bulk_signal_16(leader_sink, sink, leader_full + s * 8);
        }
      }
    }
  } else if (warp < 10) {
    // ------------------------------------------- NF4 dequant (each CTA, 256 threads)
    if (!BF16) {
      const int dq = tid - 64;
      const int grp = (warp - 2) >> 2;
      const int tr = dq & 127;
      int g = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_items; ++i) {
        const Item x = item(i);
        const int t = x.t;
        // two groups of four warps take alternate k-blocks (cluster counter g)
        for (int kb = x.kb0; kb < x.kb1; ++kb, ++g) {
          if ((g & 1) != grp) continue;
          const int s = g % S;
          if (!ptx::mbar_wait_cluster(&raw_full[s], (g / S) & 1, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          const uint8_t* codes = sRaw + s * Cfg::kRawBytes;
          const float* amax = reinterpret_cast<const float*>(codes + kHalfCodesBytes);
          const int8_t* qam = reinterpret_cast<const int8_t*>(codes + kHalfCodesBytes);
          const float* cs = reinterpret_cast<const float*>(codes + kHalfCodesBytes + 128);
          uint8_t* bt = sB + s * kHalfBTileBytes;
          if (!BMN) {
            const uint4 q0 = *reinterpret_cast<const uint4*>(codes + tr * 32);
            const uint4 q1 = *reinterpret_cast<const uint4*>(codes + tr * 32 + 16);
            const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            const int p = ((args.dq_col0 + tile_n0(t) + static_cast<int>(rank) * 128) >> 8) & 1;
            const float am =
                args.dq ? fmaf(cs[2 * p + 1], static_cast<float>(qam[tr]), cs[2 * p]) : amax[tr * 4 + (kb & 3)];
            nf4_words_bf16<8>(w, am, bt + tr * 128, 0, tr & 7);
          } else {
            // eight consecutive lanes (one 128-byte store phase) take eight rows
            // n with distinct n % 8, so their swizzled chunks fall in different banks
            const int n = ((tr >> 5) << 4) | (tr & 7) | ((tr >> 1) & 8);
            const int a = ((tr >> 1) ^ (tr >> 3)) & 1;
            const uint4 q0 = *reinterpret_cast<const uint4*>(codes + n * 64 + a * 32);
            const uint4 q1 = *reinterpret_cast<const uint4*>(codes + n * 64 + a * 32 + 16);
            const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
            const int p = ((args.dq_col0 + kb * kBK) >> 8) & 1;
            const float am = args.dq ? fmaf(cs[a * 4 + 2 * p + 1], static_cast<float>(qam[a * 64 + n]), cs[a * 4 + 2 * p])
                                     : amax[n * 4 + 2 * static_cast<int>(rank) + a];
            nf4_words_bf16<8>(w, am, bt + a * (64 * 128) + n * 128, 0, n & 7);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(leader ? &full[s] : &b_local[s]);
        }
      }
    }
  } else {
    // ------------------------------------- LoRA staging + epilogue (each CTA, 128 threads)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int e = tid - (64 + kNumDq2);  // 0..127
    const uint32_t acc_empty_leader = ptx::map_to_rank(&acc_empty[0], 0);
    const uint32_t lora_full_leader = ptx::map_to_rank(lora_full, 0);
    uint16_t* out = reinterpret_cast<uint16_t*>(args.out);
    const int r = args.r;
    const int nr = r / 8;  // r % 8 == 0, so 2r is a whole number of k16 steps: no padding
    auto chunk_at = [&](uint8_t* base, int rw, int c) {
      return reinterpret_cast<uint4*>(base + rw * 128 + ((c ^ (rw & 7)) << 4));
    };
    auto mn_chunk = [&](uint8_t* bt, int i, int cc) {  // cc: 0..15 over two 64-column atoms of 128 rows
      return reinterpret_cast<uint4*>(bt + (cc >> 3) * Cfg::kLBAtomMN + i * 128 + (((cc & 7) ^ (i & 7)) << 4));
    };
    auto xe_chunk = [&](int rw, int c) {  // 16-byte chunk c (8 elements of K) of Xe row rw, two atoms
      return reinterpret_cast<uint4*>(sLA + (c >> 3) * kLoraAtom + rw * 128 + (((c & 7) ^ (rw & 7)) << 4));
    };
    const int lora_ld = args.lora_ld > 0 ? args.lora_ld : r;
    // Xe = [s T_hi | s T_lo] (row e of this CTA's 128 rows; in a grouped
    // forward the columns of tile t's projection), Be = [B | B] for this
    // CTA's 128 output columns, in the operand layouts of the main loop.
    auto stage_lora = [&](int t) {
      const int gm = tile_m0(t) + e;
      const int nh = tile_n0(t) + static_cast<int>(rank) * 128;
      int xcol = 0;
      if (!BMN && args.lora_G > 1) {
        const int n0 = tile_n0(t);
        int g = 0;
        if (args.lora_G > 1 && n0 >= args.lora_bounds[1]) g = 1;
        if (args.lora_G > 2 && n0 >= args.lora_bounds[2]) g = 2;
        if (args.lora_G > 3 && n0 >= args.lora_bounds[3]) g = 3;
        xcol = g * r;
      }
      for (int gi = 0; gi < nr; ++gi) {
        float v[8];
        if (gm < args.M) {
          const float4* p =
              reinterpret_cast<const float4*>(args.lora_x + static_cast<int64_t>(gm) * lora_ld + xcol + gi * 8);
          const float4 a0 = p[0], a1 = p[1];
          v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w; v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) v[k] = 0.0f;
        }
        uint4 hi, lo;
        uint32_t* ph = reinterpret_cast<uint32_t*>(&hi);
        uint32_t* pl = reinterpret_cast<uint32_t*>(&lo);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x0 = v[2 * k] * args.s, x1 = v[2 * k + 1] * args.s;
          ph[k] = pack_bf16x2(x0, x1);
          pl[k] = pack_bf16x2(x0 - bf16_lo(ph[k]), x1 - bf16_hi(ph[k]));
        }
        *xe_chunk(e, gi) = hi;
        *xe_chunk(e, nr + gi) = lo;
      }
      if (!BMN) {
        const int gn = nh + e;
        for (int gi = 0; gi < nr; ++gi) {
          uint4 b = make_uint4(0, 0, 0, 0);
          if (gn < args.N) b = *reinterpret_cast<const uint4*>(args.lora_w + static_cast<int64_t>(gn) * r + gi * 8);
          *chunk_at(sLB, e, gi) = b;
          *chunk_at(sLB, e, nr + gi) = b;
        }
      } else {
        for (int task = e; task < r * 16; task += kNumEpi3) {
          const int i = task >> 4, cc = task & 15, gcol = nh + cc * 8;
          uint4 b = make_uint4(0, 0, 0, 0);
          if (gcol < args.N) b = *reinterpret_cast<const uint4*>(args.lora_w + static_cast<int64_t>(i) * args.N + gcol);
          *mn_chunk(sLB, i, cc) = b;
          *mn_chunk(sLB, r + i, cc) = b;
        }
      }
    };
    // bf16 store of the finished columns c0 .. c0+31 of this thread's row
    auto store32 = [&](int gm, int n0, int c0, const float (&v)[32]) {
      if (gm < args.M && n0 + c0 < args.N) {
        uint4* dst = reinterpret_cast<uint4*>(out + static_cast<int64_t>(gm) * args.ld_out + n0 + c0);
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          uint4 o;
          o.x = pack_bf16x2(v[8 * g4 + 0], v[8 * g4 + 1]);
          o.y = pack_bf16x2(v[8 * g4 + 2], v[8 * g4 + 3]);
          o.z = pack_bf16x2(v[8 * g4 + 4], v[8 * g4 + 5]);
          o.w = pack_bf16x2(v[8 * g4 + 6], v[8 * g4 + 7]);
          dst[g4] = o;
        }
      }
    };
    // The four epilogue warps leave the loop together (they share named
    // barrier 1): a warp whose wait failed raises epi_stop before the first
    // barrier; every warp reads it between the two.
    auto agree = [&](bool ok_w) {
      if (!ok_w && lane == 0) *epi_stop = 1;
      epi_bar_sync();
      const bool go = *epi_stop == 0;
      epi_bar_sync();
      return go;
    };
    // Split tail tiles: this CTA's slot of a piece's partial sums, column-major
    // over its 128 rows ([256 columns][128 rows] fp32), and its flag.
    auto part_of = [&](int slot) {
      return args.split_part + (static_cast<size_t>(slot) * 2 + rank) * (static_cast<size_t>(kBN) * 128);
    };
    auto flag_of = [&](int slot) { return args.split_flag + static_cast<size_t>(slot) * 2 + rank; };
    int it = 0, lit = 0;  // items and folded items of this cluster
    for (; it < n_items; ++it) {
      const Item x = item(it);
      const int t = x.t;
      const int acc = it & 1;
      if (has_lora && x.piece <= 0) {
        // the region is free once the previous tile's fold MMAs completed
        bool free_ = ptx::mbar_wait_cluster_backoff(lora_empty, (lit & 1) ^ 1, abort_flag) && !*abort_flag;
        free_ = __all_sync(0xffffffffu, free_);
        if (!free_ && !*abort_flag) give_up();
        if (!agree(free_)) break;
        stage_lora(t);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(lora_full_leader);
        ++lit;
      }
      bool ready = ptx::mbar_wait_cluster_backoff(&acc_full[acc], (it >> 1) & 1, abort_flag) && !*abort_flag;
      ready = __all_sync(0xffffffffu, ready);
      if (!ready && !*abort_flag) give_up();
      if (!agree(ready)) break;
      ptx::tc_fence_after();
      const int gm = tile_m0(t) + row;
      const int n0 = tile_n0(t);
      const uint32_t t_row = tmem + static_cast<uint32_t>(acc * kBN) + (static_cast<uint32_t>(q * 32) << 16);
      if (x.piece > 0) {
        // a later piece of a split tile: its partial sums go to its slot, then the flag
        float* part = part_of(x.slot0 + x.piece - 1);
#pragma unroll 1
        for (int c0 = 0; c0 < kBN; c0 += 32) {
          uint32_t u[32];
          ptx::tmem_ld_32x32b_x32(t_row + c0, u);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) part[(c0 + j) * 128 + row] = __uint_as_float(u[j]);
        }
        epi_bar_sync();  // every row of this CTA is stored
        if (e == 0) {
          __threadfence();
          ptx::st_release_gpu_u64(flag_of(x.slot0 + x.piece - 1), args.split_tag);
        }
      } else {
        // piece 0 of a split tile adds the later pieces' partial sums, in piece order
        int nparts = x.piece == 0 ? split_P - 1 : 0;
        if (nparts > 0) {
          bool got = true;
          if (lane == 0)
            for (int p = 0; p < nparts && got; ++p) got = ptx::wait_flag_u64(flag_of(x.slot0 + p), args.split_tag, abort_flag);
          got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
          if (!got) {  // a piece never arrived: the error is recorded and the tile left incomplete
            if (!*abort_flag) give_up();
            nparts = 0;
          }
          for (int p = 0; p < nparts; ++p) ptx::wait_flag_u64(flag_of(x.slot0 + p), args.split_tag, nullptr);
        }
        auto add_parts = [&](float (&v)[32], int c0) {
          for (int p = 0; p < nparts; ++p) {
            const float* part = part_of(x.slot0 + p);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += __ldcg(part + (c0 + j) * 128 + row);
          }
        };
        if (EPI == kEpiCEExp) {
          // This thread's row over each 128-column half of the tile: the max
          // (one read of the accumulator), then bf16(exp(z - max)) to the
          // chunk scratch and the fp32 sum of exp(z - max) (a second read),
          // both left to right, and the label's logit; half h's partials go
          // to column 2 (n0 / 256) + h.  The exp values leave as 64-column
          // TMA boxes staged like the bf16 store below.
          const int lab = gm < args.M ? args.labels[gm] : args.ignore_index;
          uint8_t* stg = sLA + (warp - 10) * 8192;
          const uint32_t stg_a = ptx::smem_addr(stg);
#pragma unroll 1
          for (int h2 = 0; h2 < 2; ++h2) {
            float mx = -INFINITY;
#pragma unroll 1
            for (int c0 = h2 * 128; c0 < h2 * 128 + 128; c0 += 32) {
              uint32_t u[32];
              ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c0), u);
              ptx::tmem_wait_ld();
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
              add_parts(v, c0);
              if (n0 + c0 < args.N)
#pragma unroll
                for (int j = 0; j < 32; ++j) mx = fmaxf(mx, v[j]);
            }
            float sm = 0.0f;
#pragma unroll 1
            for (int pp = 0; pp < 2; ++pp) {
              const int p = h2 * 2 + pp, b = p & 1;
              if (args.tma_out && p >= 2) {  // buffer b's previous box has been read out
                if (lane == 0) ptx::bulk_wait_read1();
                __syncwarp();
              }
#pragma unroll 1
              for (int hh = 0; hh < 2; ++hh) {
                const int c0 = p * 64 + hh * 32;
                uint32_t u[32];
                ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c0), u);
                ptx::tmem_wait_ld();
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
                add_parts(v, c0);
                const bool in = n0 + c0 < args.N;
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  f[j] = in ? __expf(v[j] - mx) : 0.0f;
                  sm += f[j];
                }
                if (args.tma_out) {
#pragma unroll
                  for (int g4 = 0; g4 < 4; ++g4)
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                     stg_a + b * 4096 + lane * 128 + (((hh * 4 + g4) ^ (lane & 7)) << 4)),
                                 "r"(pack_bf16x2(f[8 * g4 + 0], f[8 * g4 + 1])),
                                 "r"(pack_bf16x2(f[8 * g4 + 2], f[8 * g4 + 3])),
                                 "r"(pack_bf16x2(f[8 * g4 + 4], f[8 * g4 + 5])),
                                 "r"(pack_bf16x2(f[8 * g4 + 6], f[8 * g4 + 7]))
                                 : "memory");
                } else {
                  store32(gm, n0, c0, f);
                }
                const int vid = args.vocab_base + n0 + c0;
                if (in && gm < args.M && lab >= vid && lab < vid + 32) {
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    if (lab == vid + j) args.label_logit[gm] = v[j];
                }
              }
              if (args.tma_out) {
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  ptx::tma_store_2d(&map_o, stg + b * 4096, n0 + p * 64, tile_m0(t) + q * 32);
                  ptx::bulk_commit();
                }
              }
            }
            if (gm < args.M) {
              const int64_t pi = static_cast<int64_t>(gm) * args.part_ld + 2 * (n0 / kBN) + h2;
              args.part_max[pi] = mx;
              args.part_sum[pi] = sm;
            }
          }
          if (args.tma_out) {
            if (lane == 0) ptx::bulk_wait_read0();  // the region is free again before the next barrier
            __syncwarp();
          }
        } else if (EPI == kEpiAddF32) {
          // fp32 out[m, j] = (accumulate ? out[m, j] * alpha[m] : 0) + acc,
          // each thread its row's 32 columns at a time (128 contiguous bytes)
          float* outf = reinterpret_cast<float*>(args.out);
          const float ra = (args.row_alpha && gm < args.M) ? args.row_alpha[gm] : 1.0f;
#pragma unroll 1
          for (int c0 = 0; c0 < kBN; c0 += 32) {
            uint32_t u[32];
            ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c0), u);
            const bool in = gm < args.M && n0 + c0 < args.N;
            float4* dst = reinterpret_cast<float4*>(outf + static_cast<int64_t>(in ? gm : 0) * args.ld_out + (in ? n0 + c0 : 0));
            float4 old[8];
            if (in && args.accumulate) {  // loads in flight beside the accumulator read
#pragma unroll
              for (int g8 = 0; g8 < 8; ++g8) old[g8] = dst[g8];
            }
            ptx::tmem_wait_ld();
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
            add_parts(v, c0);
            if (in) {
#pragma unroll
              for (int g8 = 0; g8 < 8; ++g8) {
                float4 o = make_float4(v[4 * g8], v[4 * g8 + 1], v[4 * g8 + 2], v[4 * g8 + 3]);
                if (args.accumulate) {
                  o.x = fmaf(old[g8].x, ra, o.x);
                  o.y = fmaf(old[g8].y, ra, o.y);
                  o.z = fmaf(old[g8].z, ra, o.z);
                  o.w = fmaf(old[g8].w, ra, o.w);
                }
                dst[g8] = o;
              }
            }
          }
        } else if (args.tma_out) {
          // The LoRA region is free from the fold's completion (acc_full) until
          // the next stage_lora, which follows the epilogue warps' barrier:
          // this warp stages its 32 rows there as 64-column bf16 boxes (two
          // 4 KB buffers in turn) and stores them by TMA.
          uint8_t* stg = sLA + (warp - 10) * 8192;
          const uint32_t stg_a = ptx::smem_addr(stg);
#pragma unroll 1
          for (int p = 0; p < kBN / 64; ++p) {
            const int b = p & 1;
            if (p >= 2) {  // buffer b's previous box has been read out
              if (lane == 0) ptx::bulk_wait_read1();
              __syncwarp();
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t u[32];
              ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(p * 64 + h * 32), u);
              ptx::tmem_wait_ld();
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
              add_parts(v, p * 64 + h * 32);
#pragma unroll
              for (int g4 = 0; g4 < 4; ++g4)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 stg_a + b * 4096 + lane * 128 + (((h * 4 + g4) ^ (lane & 7)) << 4)),
                             "r"(pack_bf16x2(v[8 * g4 + 0], v[8 * g4 + 1])),
                             "r"(pack_bf16x2(v[8 * g4 + 2], v[8 * g4 + 3])),
                             "r"(pack_bf16x2(v[8 * g4 + 4], v[8 * g4 + 5])),
                             "r"(pack_bf16x2(v[8 * g4 + 6], v[8 * g4 + 7]))
                             : "memory");
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(&map_o, stg + b * 4096, n0 + p * 64, tile_m0(t) + q * 32);
              ptx::bulk_commit();
            }
          }
          if (lane == 0) ptx::bulk_wait_read0();  // the region is free again before any warp passes the next barrier
          __syncwarp();
        } else {
#pragma unroll 1
          for (int c0 = 0; c0 < kBN; c0 += 32) {
            uint32_t u[32];
            ptx::tmem_ld_32x32b_x32(t_row + c0, u);
            ptx::tmem_wait_ld();
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
            add_parts(v, c0);
            store32(gm, n0, c0, v);
          }
        }
      }
      // accumulator drained: let the leader reuse it
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(acc_empty_leader + acc * 8);
    }
  }
  __syncwarp();
  if (args.clk) ptx::bulk_wait0();  // this thread's output stores complete before the end stamp
  ptx::tc_fence_before();
  __syncthreads();
  clk_end(args);
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

template <int BMN, int SMALL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemm3Threads, 1)
    gemm_nf4_pair_persistent_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_c,
                                    const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_s2,
                                    const __grid_constant__ CUtensorMap map_o,
                                    const GemmArgs args) {
  pair_persistent_body<0, BMN, SMALL, kEpiStoreBF16>(map_a, map_c, map_s, map_s2, map_o, args);
}

// bf16 weights (unquantised base, K-major W [N, K] or MN-major W [K, N] by
// TMA boxes of 64 x 128 / 64 x 64); map_s, map_s2 are not read.  EPI: the
// bf16 store (with the LoRA fold), or the cross-entropy epilogues of
// gemm.cuh (the logits chunk's exp values and half-tile partials; the fp32
// dH accumulation), which fold no side product.
template <int BMN, int SMALL, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemm3Threads, 1)
    gemm_bf16_pair_persistent_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
                                     const __grid_constant__ CUtensorMap map_s, const __grid_constant__ CUtensorMap map_s2,
                                     const __grid_constant__ CUtensorMap map_o,
                                     const GemmArgs args) {
  pair_persistent_body<1, BMN, SMALL, EPI>(map_a, map_w, map_s, map_s2, map_o, args);
}

}  // namespace sl
