// Causal grouped-query attention with rotary positions on tcgen05.
//
// All three tensor-core kernels are persistent: one CTA per SM walks work
// items (numbered heaviest first) in a serpentine order; barriers, TMEM and
// the operand rings run on across items, and the per-item operand (Q, or K
// and V) of the next item loads as soon as the current item's last MMA that
// reads it has completed.
//
// Forward (items: 128-query tile, head, sequence): Q stays in shared
// memory; K and V tiles of 128 keys stream through a two-stage TMA ring
// (K released once S is computed, V once P V is).  The MMA warp computes
// S = Q K^T into one of two TMEM buffers one tile ahead.  Eight row workers
// (TMEM lane quarter x column half; 64 scores per thread) exchange their
// row maxima through shared memory and write P = exp2(S c - m) as bf16
// pairs back into TMEM over the scores; the MMA warp accumulates O += P V
// in TMEM with P as a TMEM operand and V as an MN-major shared operand.  A
// row's reference maximum moves only when a tile's maximum exceeds it by
// more than 8 (log2 units); only then is the row's O rescaled in TMEM (after
// the previous P V has completed), so most tiles hand P over without
// waiting for the tensor pipe.
//
// Backward (no atomics: every output element is summed in one CTA in a
// fixed order, so results are bitwise reproducible):
//   dq kernel  (items: 128-query tile and head): over the key blocks of 64
//              (a three-stage ring), S = Q K^T and dP = dO V^T into TMEM,
//              dS = P (dP - Di) written back over S, dQ += dS K with dS as
//              a TMEM operand;
//   dkdv kernel (items: 128-key tile and kv head, or query head when the
//              kv heads alone leave SMs idle): over the query blocks of 64
//              that see the key tile (a three-stage ring), S^T = K Q^T and
//              dP^T = V dO^T into TMEM, P^T and dS^T written back over
//              them, dV += P^T dO and dK += dS^T Q with TMEM operands;
//              per-query-head results leave as fp32 partials that
//              attn_kv_reduce_kernel sums over the heads of each kv head in
//              head order.
// A TMEM buffer is rewritten by the MMA two blocks later, which the tensor
// pipe runs after the MMA that read it (tcgen05.mma ops of one thread run in
// issue order).
// Di = rowsum(dO * O) is computed by the dq kernel's row workers from the
// O and dO tiles it loads, and stored for the dkdv kernel.  The epilogues scale dQ
// and dK by 1/sqrt(128) and rotate them back by the inverse rotary angle.
// Every wait is bounded; a timeout raises SL_ERR_TIMEOUT through the
// library's device error word.
#include <algorithm>
#include <cmath>
#include <type_traits>
#include <utility>

#include "attn.cuh"
#include "ptx.cuh"
#include "timing.cuh"
#include "tmap.cuh"

namespace sl {
namespace {

constexpr int kAtAtom128 = 128 * 128;   // 128 rows x 128 B (one SW128 atom of 128 rows)
constexpr int kAtAtom64 = 64 * 128;     // 64 rows x 128 B
constexpr int kAtTile = 2 * kAtAtom128; // [128 rows][128] bf16
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
  const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
  return lo | (hi << 16);
}
// 2^x by the hardware approximation (ex2.approx, relative error ~2^-22; -inf -> +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Store 16 bytes at chunk c (0..7) of row `row` of a 128-byte-swizzled atom
// at shared address `atom` (st.shared: the address space is explicit).
__device__ __forceinline__ void sts_swz(uint32_t atom, int row, int c, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(atom + row * 128 + ((c ^ (row & 7)) << 4)), "r"(x),
               "r"(y), "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ float4 lds128(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// The k-th work item of this CTA in a persistent grid: rounds of gridDim.x
// consecutive items (ordered heaviest first), walked forwards and backwards in
// turn so that every CTA gets a similar mix of heavy and light items.  The
// sequence increases with k, so the first index past the end ends the walk.
__device__ __forceinline__ int nth_item(int k) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return k * G + ((k & 1) ? G - 1 - c : c);
}

// Shared-memory descriptors of SW128 operands, built once per buffer and
// advanced by constant adds: the address field counts 16-byte units and no
// offset inside the CTA's shared memory (< 228 KB) carries out of it.
__device__ __forceinline__ uint64_t kdesc0(uint32_t base) { return ptx::smem_desc(base, 16, 1024, 2); }
// MN-major, N = 128 as two atoms of `atom` bytes along N
__device__ __forceinline__ uint64_t mndesc0(uint32_t base, int atom) { return ptx::smem_desc(base, atom, 1024, 2); }
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }
// k16 step kk of a K-major operand whose K extent spans atoms of `atom` bytes
__device__ __forceinline__ uint64_t kstep(uint64_t d0, int kk, int atom) {
  return dadd(d0, static_cast<uint32_t>((kk >> 2) * atom + (kk & 3) * 32));
}
// k16 step kk of an MN-major operand (16 rows of 128 bytes)
__device__ __forceinline__ uint64_t mnstep(uint64_t d0, int kk) { return dadd(d0, static_cast<uint32_t>(kk * 2048)); }

// ------------------------------------------------------------------- rope
__global__ void rope_table_kernel(int64_t S, double theta, float* __restrict__ table) {
  pdl_trigger();
  pdl_wait();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= S * 64) return;
  const int64_t p = t / 64;
  const int i = static_cast<int>(t % 64);
  const double ang = static_cast<double>(p) * pow(theta, -static_cast<double>(i) / 64.0);
  table[p * 128 + i] = static_cast<float>(cos(ang));
  table[p * 128 + 64 + i] = static_cast<float>(sin(ang));
}

// One thread per (row, head, 8 pairs).
__global__ void rope_apply_kernel(uint16_t* __restrict__ x, int64_t ld, int64_t M, int nheads, int64_t S,
                                  const float* __restrict__ table, float sgn) {
  pdl_trigger();
  pdl_wait();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= M * nheads * 8) return;
  const int64_t row = t / (nheads * 8);
  const int hc = static_cast<int>(t % (nheads * 8));
  const int h = hc / 8, c = hc % 8;
  uint16_t* p = x + row * ld + h * 128 + c * 8;
  const float* cs = table + (row % S) * 128 + c * 8;
  uint4 a = *reinterpret_cast<const uint4*>(p);
  uint4 b = *reinterpret_cast<const uint4*>(p + 64);
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
  uint32_t ao[4], bo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float x1[2] = {bf_lo(aw[e]), bf_hi(aw[e])}, x2[2] = {bf_lo(bw[e]), bf_hi(bw[e])}, y1[2], y2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float cv = cs[2 * e + u], sv = sgn * cs[64 + 2 * e + u];
      y1[u] = x1[u] * cv - x2[u] * sv;
      y2[u] = x2[u] * cv + x1[u] * sv;
    }
    ao[e] = pack2(y1[0], y1[1]);
    bo[e] = pack2(y2[0], y2[1]);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(ao[0], ao[1], ao[2], ao[3]);
  *reinterpret_cast<uint4*>(p + 64) = make_uint4(bo[0], bo[1], bo[2], bo[3]);
}

// ------------------------------------------------------------ shared args
struct AttnArgs {
  int S, H, Hkv, nseq;
  float c;        // log2(e) / sqrt(128)
  uint16_t* out0; // fwd: o;  dq kernel: dq;  dkdv kernel: dk (in-CTA head sum only)
  int64_t ld0;
  uint16_t* out1; // dkdv kernel: dv (in-CTA head sum only)
  int64_t ld1;
  float* lse;     // fwd output [H][M] (natural log); bwd input
  float* Di;       // bwd: [H][M], written by the dq kernel, read by the dkdv kernel
  const float* rope;  // bwd: table [S][128] or nullptr
  int heads_per_cta;  // dK dV kernel: query heads summed inside one CTA (1, or H / Hkv: direct bf16 output)
  int* err;
};

// Roles of the 320-thread CTAs: warp 0 TMA producer, warp 1 MMA issuer (and
// TMEM owner), warps 2..9 row workers: worker w = warp - 2 reads TMEM lane
// quarter warp % 4 (rows 32 (warp % 4) ..) and column half w / 4.
constexpr int kAtThreads = 320;
constexpr int kAtWorkers = 8;

// Barrier of the eight worker warps only (named barrier 1).
__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

struct FwdCfg {
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kAtTile;        // 2 stages
  static constexpr int kOffV = kOffK + 2 * kAtTile;    // 2 stages
  static constexpr int kOffO = kOffV + 2 * kAtTile;    // O staging for its TMA store: 2 atoms of [128][64]
  static constexpr int kOffRed = kOffO + kAtTile;       // row maxima [2][2][128], row sums [2][128], stop flags
  static constexpr int kOffBar = kOffRed + 6 * 128 * 4 + 16;
  static constexpr int kNumBars = 20;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffMisc + 16 + 1024;
};

// Persistent: one CTA per SM walks the (query tile, head, sequence) items,
// numbered heaviest first (the last query tiles see the most keys), in the
// order nth_item gives.  Barriers, TMEM and the K/V ring run on across
// items (tile parities count tiles over all of the CTA's items); Q of the
// next item loads as soon as the current item's last S = Q K^T has
// completed, while the row workers finish the item.
__global__ void __launch_bounds__(kAtThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                    const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = ptx::align1024(smem_raw);
  uint8_t* sQ = smem + FwdCfg::kOffQ;
  uint8_t* sK = smem + FwdCfg::kOffK;
  uint8_t* sV = smem + FwdCfg::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + FwdCfg::kOffBar);
  uint64_t* q_full = bars;        // Q of the item landed
  uint64_t* k_full = bars + 1;    // [2] K tile of the stage landed
  uint64_t* k_empty = bars + 3;   // [2] its S MMA done
  uint64_t* v_full = bars + 5;    // [2] V tile landed
  uint64_t* v_empty = bars + 7;   // [2] its PV MMA done
  uint64_t* s_full = bars + 9;    // [2] S tile in TMEM buffer b
  uint64_t* p_full = bars + 11;   // P written (8 warp arrivals); S buffer read
  uint64_t* o_full = bars + 12;   // [2] the P V of a tile of parity b completed
  uint64_t* drain = bars + 16;    // failure path: every issued MMA completed
  uint64_t* q_empty = bars + 17;  // the item's last S MMA done: Q may be replaced
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + FwdCfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + FwdCfg::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntq = a.S / 128;
  const int per = a.H * a.nseq;
  const int nitems = ntq * per;
  struct Item {
    int qt, h, g, row0, kv0, n;
  };
  auto item_of = [&](int item) {
    Item t;
    t.qt = ntq - 1 - item / per;  // heaviest tiles first
    const int hb = item % per;
    t.h = hb % a.H;
    const int b = hb / a.H;
    t.g = t.h / (a.H / a.Hkv);
    t.row0 = b * a.S + t.qt * 128;
    t.kv0 = b * a.S;
    t.n = t.qt + 1;  // key tiles 0..qt
    return t;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&k_full[i], 1);
      ptx::mbar_init(&k_empty[i], 1);
      ptx::mbar_init(&v_full[i], 1);
      ptx::mbar_init(&v_empty[i], 1);
      ptx::mbar_init(&s_full[i], 1);
      ptx::mbar_init(&o_full[i], 1);
    }
    ptx::mbar_init(p_full, kAtWorkers);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    reinterpret_cast<volatile int*>(smem + FwdCfg::kOffRed + 6 * 128 * 4)[0] = 0;
    reinterpret_cast<volatile int*>(smem + FwdCfg::kOffRed + 6 * 128 * 4)[1] = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&map_q);
    ptx::tma_prefetch_desc(&map_k);
    ptx::tma_prefetch_desc(&map_v);
    ptx::tma_prefetch_desc(&map_o);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // No early pdl_trigger: the grid keeps every SM busy until its end; the
  // next kernel launches as its CTAs exit.
  pdl_wait();  // the previous kernel's writes are visible from here on
  auto give_up = [&]() {
    *abort_flag = 1;
    report_device_error(a.err, SL_ERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      // K of tile t + 2 loads once S of tile t is done, V once P V of tile t is
      int issued_k = 0, issued_v = 0, issued_q = 0, it = 0, gt = 0;
      bool ok = true;
      for (int k = 0, item = nth_item(0); ok && item < nitems; item = nth_item(++k), ++it) {
        const Item t = item_of(item);
        if (!ptx::mbar_wait(q_empty, (it & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(q_full, kAtTile);
        ptx::tma_load_2d(sQ, &map_q, q_full, t.h * 128, t.row0);
        ptx::tma_load_2d(sQ + kAtAtom128, &map_q, q_full, t.h * 128 + 64, t.row0);
        ++issued_q;
        for (int j = 0; j < t.n; ++j, ++gt) {
          const int s = gt & 1;
          const uint32_t par = ((gt >> 1) & 1) ^ 1;
          const int y = t.kv0 + j * 128;
          if (!ptx::mbar_wait(&k_empty[s], par, abort_flag)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&k_full[s], kAtTile);
          ptx::tma_load_2d(sK + s * kAtTile, &map_k, &k_full[s], t.g * 128, y);
          ptx::tma_load_2d(sK + s * kAtTile + kAtAtom128, &map_k, &k_full[s], t.g * 128 + 64, y);
          ++issued_k;
          if (!ptx::mbar_wait(&v_empty[s], par, abort_flag)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&v_full[s], kAtTile);
          ptx::tma_load_2d(sV + s * kAtTile, &map_v, &v_full[s], t.g * 128, y);
          ptx::tma_load_2d(sV + s * kAtTile + kAtAtom128, &map_v, &v_full[s], t.g * 128 + 64, y);
          ++issued_v;
        }
      }
      if (!ok) {  // before the CTA exits every issued copy must have landed
        give_up();
        if (issued_q > 0) ptx::mbar_wait(q_full, (issued_q - 1) & 1, nullptr);
        for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; ++j)
          ptx::mbar_wait(&k_full[j & 1], (j >> 1) & 1, nullptr);
        for (int j = (issued_v > 2 ? issued_v - 2 : 0); j < issued_v; ++j)
          ptx::mbar_wait(&v_full[j & 1], (j >> 1) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = ptx::idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t id_o = ptx::idesc_bf16(128, 128, 0, 1);
      const uint64_t dq0 = kdesc0(ptx::smem_addr(sQ)), dk0 = kdesc0(ptx::smem_addr(sK)),
                     dv0 = mndesc0(ptx::smem_addr(sV), kAtAtom128);
      auto issue_s = [&](int gt) {  // S of the CTA's tile gt into TMEM buffer gt & 1
        const int s = gt & 1;
        if (!ptx::mbar_wait(&k_full[s], (gt >> 1) & 1, abort_flag)) return false;
        ptx::tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(s * 128);
        const uint64_t dk = dadd(dk0, s * kAtTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(d, kstep(dq0, kk, kAtAtom128), kstep(dk, kk, kAtAtom128), id_s, kk ? 1u : 0u);
        ptx::mma_commit(&s_full[s]);
        ptx::mma_commit(&k_empty[s]);
        return true;
      };
      bool ok = true;
      int it = 0, gt = 0;
      for (int k = 0, item = nth_item(0); ok && item < nitems; item = nth_item(++k), ++it) {
        const int n = item_of(item).n;
        if (!ptx::mbar_wait(q_full, it & 1, abort_flag) || !issue_s(gt)) {
          ok = false;
          break;
        }
        if (n == 1) ptx::mma_commit(q_empty);
        for (int j = 0; j < n; ++j) {
          const int cur = gt + j;
          if (j + 1 < n) {
            if (!issue_s(cur + 1)) {
              ok = false;
              break;
            }
            if (j + 2 == n) ptx::mma_commit(q_empty);  // the item's last S has been issued
          }
          const int s = cur & 1;
          // P written (and O rescaled where a row's maximum moved)
          if (!ptx::mbar_wait(p_full, cur & 1, abort_flag) ||
              !ptx::mbar_wait(&v_full[s], (cur >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t dv = dadd(dv0, s * kAtTile);
          // O += P V; P of keys 16 kk ..: the column half kk / 4 wrote it over its first 32 S columns
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            ptx::mma_bf16_ts(tmem + 256u, tmem + static_cast<uint32_t>(s * 128 + (kk >> 2) * 64 + (kk & 3) * 8),
                             mnstep(dv, kk), id_o, (j | kk) ? 1u : 0u);
          ptx::mma_commit(&o_full[s]);
          ptx::mma_commit(&v_empty[s]);
        }
        gt += n;
      }
      if (!ok) {
        give_up();
        // let every issued MMA finish before TMEM is released
        ptx::mma_commit(drain);
        ptx::mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    // Worker (quarter, half): row r, S / P / O columns 64 half .. 64 half + 63.
    // The two halves of a row exchange their maxima through red_max (double-
    // buffered by tile parity) at one worker barrier per tile; the barrier
    // also carries stop flags (per parity, only ever set) so that a timed-out
    // wait ends every worker at the same barrier.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;  // query row in the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(half * 64);
    float* red = reinterpret_cast<float*>(smem + FwdCfg::kOffRed);  // maxima [2 parity][2 half][128], sums [2][128]
    const uint32_t o_atom = ptx::smem_addr(smem + FwdCfg::kOffO) + half * kAtAtom128;
    volatile int* stop = reinterpret_cast<volatile int*>(red + 6 * 128);  // [2 parity]
    auto wait_all = [&](uint64_t* bar, uint32_t par) {
      bool w = ptx::mbar_wait(bar, par, abort_flag);
      w = __all_sync(0xffffffffu, w);
      if (!w && lane == 0 && !*abort_flag) give_up();
      return w;
    };
    // O accumulates in TMEM (P V MMAs with accumulate); a row's reference
    // maximum m only moves when the tile maximum exceeds it by more than
    // kRescale (log2 units), and only then is the row's O rescaled in TMEM.
    // P = exp2(S c - m) stays below 2^kRescale.
    constexpr float kRescale = 8.0f;
    bool bad = false, stopped = false;
    int gt = 0;
    for (int k = 0, item = nth_item(0); !stopped && item < nitems; item = nth_item(++k)) {
      const int n = ntq - item / per;  // key tiles of the item (its query tile + 1)
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < n; ++j) {
        const int cur = gt + j;
        const int s = cur & 1;
        const bool diag = (j == n - 1);
        uint32_t u[2][32];
        float mt = -INFINITY;
        if (!bad) bad = !wait_all(&s_full[s], (cur >> 1) & 1);
        if (!bad) {
          ptx::tc_fence_after();
          const uint32_t s_addr = lane_base + static_cast<uint32_t>(s * 128);
          ptx::tmem_ld_32x32b_x32(s_addr, u[0]);
          ptx::tmem_ld_32x32b_x32(s_addr + 32, u[1]);
          ptx::tmem_wait_ld();
          if (diag) {  // keys above the diagonal do not exist
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (half * 64 + c * 32 + e > r) u[c][e] = __float_as_uint(-INFINITY);
          }
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) mx[e & 3] = fmaxf(mx[e & 3], __uint_as_float(u[c][e]));
          mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        }
        red[(s * 2 + half) * 128 + r] = mt;
        if (bad && lane == 0) stop[s] = 1;
        workers_sync();
        if (stop[s]) {
          stopped = true;
          break;
        }
        const float m_tile = fmaxf(mt, red[(s * 2 + (half ^ 1)) * 128 + r]) * a.c;
        const bool move = m_tile > m + kRescale;  // always on the item's first tile
        const float alpha = move ? ex2(m - m_tile) : 1.0f;
        if (move) m = m_tile;
        if (j > 0 && __any_sync(0xffffffffu, move)) {
          // O through the previous tile: wait for its P V (this tile's S has
          // completed, so every earlier P V but that one has), then O *= alpha
          if (!wait_all(&o_full[(cur - 1) & 1], ((cur - 1) >> 1) & 1)) {
            bad = true;
            continue;  // raise the stop flag at the next barrier
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t ov[32];
            ptx::tmem_ld_32x32b_x32(lane_base + 256u + static_cast<uint32_t>(c * 32), ov);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            ptx::tmem_st_32x32b_x32(lane_base + 256u + static_cast<uint32_t>(c * 32), ov);
          }
        }
        // P = exp2(S c - m) as bf16 pairs over the first 32 of the 64 S
        // columns this thread has read (every worker has read its S: the
        // barrier above), the P V MMA's A operand
        float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = ex2(fmaf(__uint_as_float(u[c][e]), a.c, -m));
            const float p1 = ex2(fmaf(__uint_as_float(u[c][e + 1]), a.c, -m));
            ls[e & 3] += p0;
            ls[(e + 1) & 3] += p1;
            w[e / 2] = pack2(p0, p1);
          }
          ptx::tmem_st_32x32b_x16(lane_base + static_cast<uint32_t>(s * 128 + c * 16), w);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full);
        l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      }
      if (stopped) break;
      // the final O once the last P V has completed, then the two halves'
      // row sums (the barrier of the CTA's next tile parity)
      const int nxt = gt + n;
      if (!bad) bad = !wait_all(&o_full[(nxt - 1) & 1], ((nxt - 1) >> 1) & 1);
      red[(2 * 2 + half) * 128 + r] = l;
      if (bad && lane == 0) stop[nxt & 1] = 1;
      workers_sync();
      if (stop[nxt & 1]) {
        stopped = true;
        break;
      }
      const Item t = item_of(item);
      const float lrow = red[(4 + 0) * 128 + r] + red[(4 + 1) * 128 + r];
      const float inv = 1.0f / lrow;
      // O leaves through shared memory: this warp's 32 rows x 64 columns are
      // one TMA box (its previous box has been read out before it is reused)
      if (lane == 0) ptx::bulk_wait_read0();
      __syncwarp();
      ptx::tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t ov[32];
        ptx::tmem_ld_32x32b_x32(lane_base + 256u + static_cast<uint32_t>(c * 32), ov);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float* f = reinterpret_cast<const float*>(ov + 8 * q4);
          sts_swz(o_atom, r, c * 4 + q4, pack2(f[0] * inv, f[1] * inv), pack2(f[2] * inv, f[3] * inv),
                  pack2(f[4] * inv, f[5] * inv), pack2(f[6] * inv, f[7] * inv));
        }
      }
      // O has left TMEM before this warp's next P arrival, after which the
      // next item's first P V overwrites it
      ptx::tc_fence_before();
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(&map_o, smem + FwdCfg::kOffO + half * kAtAtom128 + quarter * 32 * 128, t.h * 128 + half * 64,
                          t.row0 + quarter * 32);
        ptx::bulk_commit();
      }
      if (half == 0) {
        const int64_t M = static_cast<int64_t>(a.nseq) * a.S;
        a.lse[static_cast<int64_t>(t.h) * M + t.row0 + r] = (m + log2f(lrow)) * 0.69314718055994531f;
      }
      gt = nxt;
    }
    if (lane == 0) ptx::bulk_wait0();  // this warp's O stores are complete
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}


// cos and sin of the rotation pairs 32 half .. 32 half + 31 at one position
// (the table row holds cos at 0..63 and sin at 64..127), loaded ahead of use.
struct RotRow {
  float4 c[8], s[8];
};
__device__ __forceinline__ void load_rot(const float* table, int pos, int half, RotRow& t) {
  const float4* cs = reinterpret_cast<const float4*>(table + static_cast<int64_t>(pos) * 128 + half * 32);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    t.c[i] = __ldg(cs + i);
    t.s[i] = __ldg(cs + 16 + i);
  }
}

// Rotation pairs 32 half .. 32 half + 31 of one 128-wide gradient row: lo
// holds columns 32 half .., hi columns 64 + 32 half ..; scale by 1/sqrt(128),
// rotate back by the inverse angle of the row's position (rot may be null:
// no rotation) and round to bf16 pairs: o1 the columns 32 half .., o2
// 64 + 32 half ...
__device__ __forceinline__ void grad_pairs(const uint32_t (&lo)[32], const uint32_t (&hi)[32], float scale,
                                           const RotRow* rot, uint32_t (&o1)[16], uint32_t (&o2)[16]) {
#pragma unroll
  for (int e4 = 0; e4 < 32; e4 += 4) {
    float cv[4] = {1.0f, 1.0f, 1.0f, 1.0f}, sv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (rot) {
      const float4 c = rot->c[e4 / 4], sn = rot->s[e4 / 4];
      cv[0] = c.x, cv[1] = c.y, cv[2] = c.z, cv[3] = c.w;
      sv[0] = sn.x, sv[1] = sn.y, sv[2] = sn.z, sv[3] = sn.w;
    }
    float y1[4], y2[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x1 = __uint_as_float(lo[e4 + u]) * scale, x2 = __uint_as_float(hi[e4 + u]) * scale;
      if (rot) {
        y1[u] = x1 * cv[u] + x2 * sv[u];
        y2[u] = x2 * cv[u] - x1 * sv[u];
      } else {
        y1[u] = x1;
        y2[u] = x2;
      }
    }
    o1[e4 / 2] = pack2(y1[0], y1[1]);
    o1[e4 / 2 + 1] = pack2(y1[2], y1[3]);
    o2[e4 / 2] = pack2(y2[0], y2[1]);
    o2[e4 / 2 + 1] = pack2(y2[2], y2[3]);
  }
}
// ... stored straight into the gradient row
__device__ __forceinline__ void store_grad_pairs(const uint32_t (&lo)[32], const uint32_t (&hi)[32], float scale,
                                                 const RotRow* rot, int half, uint16_t* row) {
  uint32_t o1[16], o2[16];
  grad_pairs(lo, hi, scale, rot, o1, o2);
  uint4* d1 = reinterpret_cast<uint4*>(row + half * 32);
  uint4* d2 = reinterpret_cast<uint4*>(row + 64 + half * 32);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    d1[c] = make_uint4(o1[4 * c], o1[4 * c + 1], o1[4 * c + 2], o1[4 * c + 3]);
    d2[c] = make_uint4(o2[4 * c], o2[4 * c + 1], o2[4 * c + 2], o2[4 * c + 3]);
  }
}
// ... or into row r of a [128][128] staging tile of two 128-byte-swizzled
// atoms (columns 0..63 at atom0, 64..127 at atom1) for a TMA store
__device__ __forceinline__ void stage_grad_pairs(const uint32_t (&lo)[32], const uint32_t (&hi)[32], float scale,
                                                 const RotRow* rot, int half, uint32_t atom0, int r) {
  uint32_t o1[16], o2[16];
  grad_pairs(lo, hi, scale, rot, o1, o2);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    sts_swz(atom0, r, half * 4 + c, o1[4 * c], o1[4 * c + 1], o1[4 * c + 2], o1[4 * c + 3]);
    sts_swz(atom0 + kAtAtom128, r, half * 4 + c, o2[4 * c], o2[4 * c + 1], o2[4 * c + 2], o2[4 * c + 3]);
  }
}
// ------------------------------------------------------------ dQ
// TMEM column of k16 step kk (keys 16 kk ..) of a 64-key block's bf16 dS or
// P^T / dS^T stored over fp32 buffer b (64 columns at 64 b): each half of the
// block (32 keys) sits in the first 16 columns of its own 32.
__device__ __forceinline__ uint32_t ds_col(int b, int kk) {
  return static_cast<uint32_t>(b * 64 + (kk >> 1) * 32 + (kk & 1) * 8);
}

constexpr int kAtStages = 3;  // key/value ring of the dQ kernel
constexpr int kKvStages = 3;  // query/dO ring of the dK dV kernel

struct DqCfg {
  static constexpr int kOffQ = 0;                      // [128][128]
  static constexpr int kOffDO = kOffQ + kAtTile;       // [128][128]
  static constexpr int kOffO = kOffDO + kAtTile;       // [128][128]: O, for Di = rowsum(dO * O)
  static constexpr int kOffK = kOffO + kAtTile;        // kAtStages stages of [64][128]
  static constexpr int kOffV = kOffK + kAtStages * 2 * kAtAtom64;
  static constexpr int kOffOut = kOffV + kAtStages * 2 * kAtAtom64;  // dQ staging: 2 atoms of [128][64]
  static constexpr int kOffBar = kOffOut + kAtTile;
  static constexpr int kNumBars = 24;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffMisc + 16 + 1024;
};

// Persistent: one CTA per SM walks the (query tile, head, sequence) items,
// numbered heaviest first, in the order nth_item gives.  The key/value ring and
// the S / dP / dS buffers run on across items (block parities count the
// CTA's 64-key blocks over all of its items); Q and dO of the next item load
// as soon as the current item's last S / dP MMAs have completed.
__global__ void __launch_bounds__(kAtThreads, 1)
    attn_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                   const __grid_constant__ CUtensorMap map_o, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_dq,
                   const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = ptx::align1024(smem_raw);
  uint8_t* sQ = smem + DqCfg::kOffQ;
  uint8_t* sDO = smem + DqCfg::kOffDO;
  uint8_t* sK = smem + DqCfg::kOffK;
  uint8_t* sV = smem + DqCfg::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DqCfg::kOffBar);
  uint64_t* q_full = bars;         // Q, dO and O of the item landed
  uint64_t* kv_full = bars + 1;                  // [kAtStages]
  uint64_t* kv_empty = bars + 1 + kAtStages;     // [kAtStages]
  uint64_t* sp_full = bars + 1 + 2 * kAtStages;  // [2] S and dP in TMEM buffer b
  uint64_t* ds_full = sp_full + 2;               // [2] dS written over S in buffer b (8 warp arrivals)
  uint64_t* acc_full = sp_full + 4;              // dQ of the item complete
  uint64_t* drain = sp_full + 5;                 // failure path: every issued MMA completed
  uint64_t* q_empty = sp_full + 6;               // the item's last S / dP MMAs done and Di read out of dO, O
                                                 // (1 commit + 8 warp arrivals): they may be replaced
  uint64_t* stage_full = sp_full + 7;            // [4] quarter q's staging rows written (2 warp arrivals)
  uint64_t* stage_free = sp_full + 11;           // [4] quarter q's previous TMA stores have read them
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + DqCfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + DqCfg::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntq = a.S / 128;
  const int per = a.H * a.nseq;
  const int nitems = ntq * per;
  const int64_t M = static_cast<int64_t>(a.nseq) * a.S;
  struct Item {
    int qt, h, g, row0, kv0, n;
  };
  auto item_of = [&](int item) {
    Item t;
    t.qt = ntq - 1 - item / per;  // heaviest tiles first
    const int hb = item % per;
    t.h = hb % a.H;
    const int b = hb / a.H;
    t.g = t.h / (a.H / a.Hkv);
    t.row0 = b * a.S + t.qt * 128;
    t.kv0 = b * a.S;
    t.n = 2 * (t.qt + 1);  // key blocks of 64
    return t;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(q_full, 1);
    ptx::mbar_init(q_empty, 1 + kAtWorkers);
    for (int i = 0; i < kAtStages; ++i) {
      ptx::mbar_init(&kv_full[i], 1);
      ptx::mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&sp_full[i], 1);
      ptx::mbar_init(&ds_full[i], kAtWorkers);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(&stage_full[i], 2);
      ptx::mbar_init(&stage_free[i], 1);
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&map_q);
    ptx::tma_prefetch_desc(&map_do);
    ptx::tma_prefetch_desc(&map_k);
    ptx::tma_prefetch_desc(&map_v);
    ptx::tma_prefetch_desc(&map_dq);
    ptx::tma_prefetch_desc(&map_o);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // No early pdl_trigger: the grid keeps every SM busy until its end; the
  // next kernel launches as its CTAs exit.
  pdl_wait();  // the previous kernel's writes are visible from here on
  // TMEM: S buffers at 0 / 64 (dS over them as bf16 pairs), dP at 128 / 192,
  // dQ at 256, each worker's rotary row at 384 + 64 half.  A buffer is
  // rewritten by the S MMA two blocks later, which the tensor pipe runs after
  // the dQ MMA that reads its dS (issue order).
  auto give_up = [&]() {
    *abort_flag = 1;
    report_device_error(a.err, SL_ERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0, issued_q = 0, it = 0, gb = 0;
      bool ok = true;
      for (int k = 0, item = nth_item(0); ok && item < nitems; item = nth_item(++k), ++it) {
        const Item t = item_of(item);
        if (!ptx::mbar_wait(q_empty, (it & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(q_full, 3 * kAtTile);
        ptx::tma_load_2d(sQ, &map_q, q_full, t.h * 128, t.row0);
        ptx::tma_load_2d(sQ + kAtAtom128, &map_q, q_full, t.h * 128 + 64, t.row0);
        ptx::tma_load_2d(sDO, &map_do, q_full, t.h * 128, t.row0);
        ptx::tma_load_2d(sDO + kAtAtom128, &map_do, q_full, t.h * 128 + 64, t.row0);
        ptx::tma_load_2d(smem + DqCfg::kOffO, &map_o, q_full, t.h * 128, t.row0);
        ptx::tma_load_2d(smem + DqCfg::kOffO + kAtAtom128, &map_o, q_full, t.h * 128 + 64, t.row0);
        ++issued_q;
        for (int j = 0; j < t.n; ++j, ++gb) {
          const int s = gb % kAtStages;
          if (!ptx::mbar_wait(&kv_empty[s], ((gb / kAtStages) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&kv_full[s], 4 * kAtAtom64);
          uint8_t* k_dst = sK + s * 2 * kAtAtom64;
          uint8_t* v_dst = sV + s * 2 * kAtAtom64;
          const int y = t.kv0 + j * 64;
          ptx::tma_load_2d(k_dst, &map_k, &kv_full[s], t.g * 128, y);
          ptx::tma_load_2d(k_dst + kAtAtom64, &map_k, &kv_full[s], t.g * 128 + 64, y);
          ptx::tma_load_2d(v_dst, &map_v, &kv_full[s], t.g * 128, y);
          ptx::tma_load_2d(v_dst + kAtAtom64, &map_v, &kv_full[s], t.g * 128 + 64, y);
          ++issued;
        }
      }
      if (!ok) {  // before the CTA exits every issued copy must have landed
        give_up();
        if (issued_q > 0) ptx::mbar_wait(q_full, (issued_q - 1) & 1, nullptr);
        for (int j = (issued > kAtStages ? issued - kAtStages : 0); j < issued; ++j)
          ptx::mbar_wait(&kv_full[j % kAtStages], (j / kAtStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = ptx::idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t id_q = ptx::idesc_bf16(128, 128, 0, 1);
      const uint64_t dq0 = kdesc0(ptx::smem_addr(sQ)), ddo0 = kdesc0(ptx::smem_addr(sDO)),
                     dk0 = kdesc0(ptx::smem_addr(sK)), dv0 = kdesc0(ptx::smem_addr(sV)),
                     dkmn0 = mndesc0(ptx::smem_addr(sK), kAtAtom64);
      auto issue_sp = [&](int gb) {  // S and dP of the CTA's block gb into TMEM buffer gb & 1
        const int s = gb % kAtStages, b2 = gb & 1;
        if (!ptx::mbar_wait(&kv_full[s], (gb / kAtStages) & 1, abort_flag)) return false;
        ptx::tc_fence_after();
        const uint64_t dk = dadd(dk0, s * 2 * kAtAtom64), dv = dadd(dv0, s * 2 * kAtAtom64);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + static_cast<uint32_t>(b2 * 64), kstep(dq0, kk, kAtAtom128), kstep(dk, kk, kAtAtom64),
                        id_s, kk ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + 128u + static_cast<uint32_t>(b2 * 64), kstep(ddo0, kk, kAtAtom128),
                        kstep(dv, kk, kAtAtom64), id_s, kk ? 1u : 0u);
        ptx::mma_commit(&sp_full[b2]);
        return true;
      };
      bool ok = true;
      int it = 0, gb = 0;
      for (int k = 0, item = nth_item(0); ok && item < nitems; item = nth_item(++k), ++it) {
        const int n = item_of(item).n;  // >= 2
        if (!ptx::mbar_wait(q_full, it & 1, abort_flag) || !issue_sp(gb)) {
          ok = false;
          break;
        }
        for (int j = 0; j < n; ++j) {
          const int cur = gb + j;
          if (j + 1 < n) {
            if (!issue_sp(cur + 1)) {
              ok = false;
              break;
            }
            if (j + 2 == n) ptx::mma_commit(q_empty);  // the item's last S / dP have been issued
          }
          if (!ptx::mbar_wait(&ds_full[cur & 1], (cur >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t dkmn = dadd(dkmn0, (cur % kAtStages) * 2 * kAtAtom64);
          // dS of keys 16 kk .. in the columns the two halves wrote (see the workers)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_bf16_ts(tmem + 256u, tmem + ds_col(cur & 1, kk), mnstep(dkmn, kk), id_q, (j | kk) ? 1u : 0u);
          ptx::mma_commit(&kv_empty[cur % kAtStages]);
        }
        if (!ok) break;
        ptx::mma_commit(acc_full);
        gb += n;
      }
      if (!ok) {
        give_up();
        ptx::mma_commit(drain);
        ptx::mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // Worker (quarter, half): query row r, key columns 32 half .. 32 half + 31
    // of each 64-key block; in the epilogue the rotation pairs 32 half ..
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    auto wait_all = [&](uint64_t* bar, uint32_t par) {
      bool w = ptx::mbar_wait(bar, par, abort_flag);
      w = __all_sync(0xffffffffu, w);
      if (!w && lane == 0 && !*abort_flag) give_up();
      return w;
    };
    // The epilogue rotates dQ back with the row's 32 cos and 32 sin of this
    // warp's half.  Read from global in one burst at the item's end, those
    // loads held up the issue of the item's last dQ MMAs by ~3 us per item
    // (the row's 16-byte pieces sit 512 bytes apart from the next row's);
    // the first four 64-key blocks now bring four pieces each into TMEM
    // columns 384 + 64 half .. (cos at +0, sin at +32), read back in the
    // epilogue (an item of two blocks loads its last eight pieces there).
    const bool rotate = a.rope != nullptr;
    const uint32_t rope_col = lane_base + 384u + static_cast<uint32_t>(half * 64);
    bool ok = true;
    int it = 0, gb = 0;
    for (int k = 0, item = nth_item(0); ok && item < nitems; item = nth_item(++k), ++it) {
      const Item t = item_of(item);
      const int qrow = t.qt * 128 + r;  // position in the sequence
      const float lse2 = a.lse[static_cast<int64_t>(t.h) * M + t.row0 + r] * kLog2e;
      // 16-byte piece p of the row: cos p (p < 8) or sin p - 8, TMEM column rope_col + 4 p
      const float4* rope_row =
          rotate ? reinterpret_cast<const float4*>(a.rope + static_cast<int64_t>(qrow) * 128 + half * 32) : nullptr;
      // Di = rowsum(dO * O) of row r over all 128 columns (both warps of the
      // row compute it), from the item's shared tiles; half 0 stores it for
      // the dK dV kernel
      if (!wait_all(q_full, it & 1)) {
        ok = false;
        break;
      }
      float di;
      {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint32_t sdo = ptx::smem_addr(sDO), so = ptx::smem_addr(smem + DqCfg::kOffO);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t off = (c >> 3) * kAtAtom128 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
          const float4 x = lds128(sdo + off), y = lds128(so + off);
          const uint32_t xa[4] = {__float_as_uint(x.x), __float_as_uint(x.y), __float_as_uint(x.z), __float_as_uint(x.w)};
          const uint32_t ya[4] = {__float_as_uint(y.x), __float_as_uint(y.y), __float_as_uint(y.z), __float_as_uint(y.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] += bf_lo(xa[e]) * bf_lo(ya[e]) + bf_hi(xa[e]) * bf_hi(ya[e]);
        }
        di = (acc[0] + acc[1]) + (acc[2] + acc[3]);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(q_empty);
      if (half == 0) a.Di[static_cast<int64_t>(t.h) * M + t.row0 + r] = di;
      for (int j = 0; j < t.n; ++j) {
        const int cur = gb + j;
        const int s = cur & 1;
        if (!wait_all(&sp_full[s], (cur >> 1) & 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // pieces 4 j .. 4 j + 3 of the rotary row in the first four blocks
        const bool rope_here = rotate && j < 4;
        float4 rv[4];
        if (rope_here) {
#pragma unroll
          for (int i = 0; i < 4; ++i) rv[i] = __ldg(rope_row + (j < 2 ? 4 * j + i : 8 + 4 * j + i));
        }
        uint32_t w[16];
        {
          uint32_t us[32], up[32];
          ptx::tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(s * 64 + half * 32), us);
          ptx::tmem_ld_32x32b_x32(lane_base + 128u + static_cast<uint32_t>(s * 64 + half * 32), up);
          ptx::tmem_wait_ld();
          const int key0 = j * 64 + half * 32;
          auto dS = [&](auto masked) {  // only the item's last two blocks reach the diagonal
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float ds2[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                float p = ex2(fmaf(__uint_as_float(us[e + u]), a.c, -lse2));
                if (decltype(masked)::value && key0 + e + u > qrow) p = 0.0f;
                ds2[u] = p * (__uint_as_float(up[e + u]) - di);
              }
              w[e / 2] = pack2(ds2[0], ds2[1]);
            }
          };
          if (j + 2 >= t.n)
            dS(std::true_type{});
          else
            dS(std::false_type{});
        }
        // dS of this half's 32 keys over the first 16 columns of the S columns
        // this thread has just read (no other warp reads them)
        ptx::tmem_st_32x32b_x16(lane_base + static_cast<uint32_t>(s * 64 + half * 32), w);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ds_full[s]);
        if (rope_here) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            ptx::tmem_st_32x32b_x4(rope_col + 4u * static_cast<uint32_t>(4 * j + i), __float_as_uint(rv[i].x),
                                   __float_as_uint(rv[i].y), __float_as_uint(rv[i].z), __float_as_uint(rv[i].w));
        }
      }
      RotRow rot;
      if (ok && rotate) {
        ptx::tmem_wait_st();  // this thread's rotary pieces have landed
        uint32_t u[32];
        ptx::tmem_ld_32x32b_x32(rope_col, u);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          rot.c[i] = make_float4(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]), __uint_as_float(u[4 * i + 2]),
                                 __uint_as_float(u[4 * i + 3]));
        if (t.n >= 4) {
          ptx::tmem_ld_32x32b_x32(rope_col + 32u, u);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            rot.s[i] = make_float4(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                                   __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3]));
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) rot.s[i] = __ldg(rope_row + 16 + i);
        }
      }
      if (!ok || !wait_all(acc_full, it & 1)) {
        ok = false;
        break;
      }
      // dQ leaves TMEM before this warp's next dS arrival, after which the
      // next item's first dQ MMA overwrites it
      ptx::tc_fence_after();
      uint32_t lo[32], hi[32];
      ptx::tmem_ld_32x32b_x32(lane_base + 256u + static_cast<uint32_t>(half * 32), lo);
      ptx::tmem_ld_32x32b_x32(lane_base + 256u + static_cast<uint32_t>(64 + half * 32), hi);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      // dQ leaves through shared memory: the quarter's two warps fill its 32
      // rows of both atoms, then the half-0 warp issues one TMA store per
      // atom.  The rows are rewritten only after the previous item's stores
      // have read them (stage_free, raised by the issuing lane).
      if (half == 0 && it > 0) {
        if (lane == 0) {
          ptx::bulk_wait_read0();
          ptx::mbar_arrive(&stage_free[quarter]);
        }
        __syncwarp();
      }
      if (!wait_all(&stage_free[quarter], (it & 1) ^ 1)) {
        ok = false;
        break;
      }
      if (rotate)
        stage_grad_pairs(lo, hi, 0.08838834764831845f, &rot, half, ptx::smem_addr(smem + DqCfg::kOffOut), r);
      else
        stage_grad_pairs(lo, hi, 0.08838834764831845f, nullptr, half, ptx::smem_addr(smem + DqCfg::kOffOut), r);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&stage_full[quarter]);
      if (half == 0) {
        if (!wait_all(&stage_full[quarter], it & 1)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* box = smem + DqCfg::kOffOut + quarter * 32 * 128;
          ptx::tma_store_2d(&map_dq, box, t.h * 128, t.row0 + quarter * 32);
          ptx::tma_store_2d(&map_dq, box + kAtAtom128, t.h * 128 + 64, t.row0 + quarter * 32);
          ptx::bulk_commit();
        }
      }
      gb += t.n;
    }
    if (half == 0 && lane == 0) ptx::bulk_wait0();  // this quarter's dQ stores are complete
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------ dK, dV
// One work item per (128-key tile, group of heads_per_cta query heads,
// sequence): dK and dV of the key tile accumulate in TMEM over those heads'
// query blocks that see it.  heads_per_cta = H / Hkv (enough items to fill the
// GPU): the item covers its kv head's query heads in head order and writes
// bf16 dk (scaled, rotated back) and dv itself; heads_per_cta = 1: fp32
// per-head partials [H][M][128] that attn_kv_reduce_kernel sums in head order.
struct DkvCfg {
  static constexpr int kOffK = 0;                    // [128][128]
  static constexpr int kOffV = kOffK + kAtTile;      // [128][128]
  static constexpr int kStage = 4 * kAtAtom64;              // Q [64][128], dO [64][128] (1024-aligned tiles)
  static constexpr int kStageBytes = kStage + 512;           // + lse and Di of the 64 rows
  static constexpr int kOffStage = kOffV + kAtTile;          // kKvStages stages
  // the item's 128 rotary rows (direct dK only): four 128-byte-swizzled
  // boxes [128 rows][32 fp32]: cos of pairs 0.., 32.., sin of pairs 0.., 32..
  static constexpr int kOffRope = kOffStage + kKvStages * kStage;
  static constexpr int kRopeBytes = 4 * 128 * 128;
  static constexpr int kOffLD = kOffRope + kRopeBytes;       // kKvStages x (lse [64], Di [64]) fp32
  static constexpr int kOffBar = kOffLD + kKvStages * 512;
  static constexpr int kNumBars = 18;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffMisc + 16 + 1024;
};
static_assert(DkvCfg::kSmem <= 232448, "dK/dV shared memory exceeds the per-CTA limit");
static_assert(DqCfg::kSmem <= 232448, "dQ shared memory exceeds the per-CTA limit");
static_assert(FwdCfg::kSmem <= 232448, "forward shared memory exceeds the per-CTA limit");
static_assert(1 + 2 * kAtStages + 15 <= DqCfg::kNumBars, "dQ barrier count");
static_assert(1 + 2 * kKvStages + 11 <= DkvCfg::kNumBars, "dK/dV barrier count");
static_assert(DkvCfg::kOffRope % 1024 == 0, "dK/dV rotary boxes must be 1024-byte aligned");

// Persistent: one CTA per SM walks the (key tile, head group, sequence)
// items, numbered heaviest first (the first key tiles are seen by the most
// query blocks), in the order nth_item gives.  The query/dO ring and the
// S^T / dP^T / P^T / dS^T buffers run on across items; K and V of the next
// item load once the current item's last S^T / dP^T MMAs have completed.
__global__ void __launch_bounds__(kAtThreads, 1)
    attn_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                     const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                     const __grid_constant__ CUtensorMap map_lse, const __grid_constant__ CUtensorMap map_di,
                     const __grid_constant__ CUtensorMap map_rope, const AttnArgs a, float* __restrict__ part_dk,
                     float* __restrict__ part_dv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = ptx::align1024(smem_raw);
  uint8_t* sK = smem + DkvCfg::kOffK;
  uint8_t* sV = smem + DkvCfg::kOffV;
  uint8_t* sStage = smem + DkvCfg::kOffStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DkvCfg::kOffBar);
  uint64_t* kv_full = bars;                      // K and V of the item landed
  uint64_t* st_full = bars + 1;                  // [kKvStages]
  uint64_t* st_empty = bars + 1 + kKvStages;     // [kKvStages]
  uint64_t* sp_full = bars + 1 + 2 * kKvStages;  // [2] S^T and dP^T in TMEM buffer b
  uint64_t* ds_full = sp_full + 2;               // [2] P^T, dS^T written over buffer b (8 warp arrivals)
  uint64_t* acc_full = sp_full + 6;              // dK, dV of the item complete
  uint64_t* drain = sp_full + 7;                 // failure path: every issued MMA completed
  uint64_t* kv_empty = sp_full + 8;              // the item's last S^T / dP^T MMAs done: K, V may be replaced
  uint64_t* rope_full = sp_full + 9;             // the item's rotary rows landed (direct dK with rotation)
  uint64_t* rope_empty = sp_full + 10;           // the epilogue has read them (8 warp arrivals)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + DkvCfg::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + DkvCfg::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hpc = a.heads_per_cta;
  // The direct epilogue rotates dK back with each key row's 64 cos and sin.
  // Read from global at the item's end (each thread its own row, 512 bytes
  // from the next), those loads held up the MMA issue and the workers; the
  // producer now brings the item's rows into shared memory by TMA while the
  // item's last query blocks stream in.
  const bool rope_smem = a.rope != nullptr && hpc == a.H / a.Hkv;
  const int ngrp = a.H / hpc;
  const int per = ngrp * a.nseq;
  const int ntk = a.S / 128;
  const int nitems = ntk * per;
  const int64_t M = static_cast<int64_t>(a.nseq) * a.S;
  struct Item {
    int kt, h0, g, b, key0, nqb, n;
  };
  auto item_of = [&](int item) {
    Item t;
    t.kt = item / per;  // key tile; heaviest (kt = 0) first
    const int hb = item % per;
    t.h0 = (hb % ngrp) * hpc;
    t.b = hb / ngrp;
    t.g = t.h0 / (a.H / a.Hkv);
    t.key0 = t.b * a.S + t.kt * 128;
    t.nqb = a.S / 64 - 2 * t.kt;  // query blocks of 64 that see this key tile
    t.n = hpc * t.nqb;            // iterations: (query head, query block)
    return t;
  };

  if (threadIdx.x == 0) {
    ptx::mbar_init(kv_full, 1);
    ptx::mbar_init(kv_empty, 1);
    for (int i = 0; i < kKvStages; ++i) {
      ptx::mbar_init(&st_full[i], 1);
      ptx::mbar_init(&st_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&sp_full[i], 1);
      ptx::mbar_init(&ds_full[i], kAtWorkers);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(rope_full, 1);
    ptx::mbar_init(rope_empty, kAtWorkers);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::tma_prefetch_desc(&map_q);
    ptx::tma_prefetch_desc(&map_do);
    ptx::tma_prefetch_desc(&map_k);
    ptx::tma_prefetch_desc(&map_v);
    if (rope_smem) ptx::tma_prefetch_desc(&map_rope);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // No early pdl_trigger: the grid keeps every SM busy until its end; the
  // next kernel launches as its CTAs exit.
  pdl_wait();  // the previous kernel's writes are visible from here on
  // TMEM: S^T buffers at 0 / 64 (P^T over them as bf16 pairs), dP^T at
  // 128 / 192 (dS^T over them), dV at 256, dK at 384.  A buffer is rewritten
  // by the S^T / dP^T MMAs two iterations later, which the tensor pipe runs
  // after the dV / dK MMAs that read it (issue order).
  auto give_up = [&]() {
    *abort_flag = 1;
    report_device_error(a.err, SL_ERR_TIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0, issued_kv = 0, issued_rope = 0, it = 0, gs = 0;
      bool ok = true;
      for (int k = 0, item = nth_item(0); ok && item < nitems; item = nth_item(++k), ++it) {
        const Item t = item_of(item);
        if (!ptx::mbar_wait(kv_empty, (it & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        ptx::mbar_arrive_expect_tx(kv_full, 2 * kAtTile);
        ptx::tma_load_2d(sK, &map_k, kv_full, t.g * 128, t.key0);
        ptx::tma_load_2d(sK + kAtAtom128, &map_k, kv_full, t.g * 128 + 64, t.key0);
        ptx::tma_load_2d(sV, &map_v, kv_full, t.g * 128, t.key0);
        ptx::tma_load_2d(sV + kAtAtom128, &map_v, kv_full, t.g * 128 + 64, t.key0);
        ++issued_kv;
        for (int u = 0; u < t.n; ++u, ++gs) {
          const int s = gs % kKvStages;
          if (!ptx::mbar_wait(&st_empty[s], ((gs / kKvStages) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const int h = t.h0 + u / t.nqb, qrow = t.b * a.S + (2 * t.kt + u % t.nqb) * 64;
          uint8_t* st = sStage + s * DkvCfg::kStage;
          ptx::mbar_arrive_expect_tx(&st_full[s], DkvCfg::kStageBytes);
          ptx::tma_load_2d(st, &map_q, &st_full[s], h * 128, qrow);
          ptx::tma_load_2d(st + kAtAtom64, &map_q, &st_full[s], h * 128 + 64, qrow);
          ptx::tma_load_2d(st + 2 * kAtAtom64, &map_do, &st_full[s], h * 128, qrow);
          ptx::tma_load_2d(st + 3 * kAtAtom64, &map_do, &st_full[s], h * 128 + 64, qrow);
          uint8_t* ld = smem + DkvCfg::kOffLD + s * 512;
          ptx::tma_load_2d(ld, &map_lse, &st_full[s], qrow, h);
          ptx::tma_load_2d(ld + 256, &map_di, &st_full[s], qrow, h);
          ++issued;
          if (rope_smem && u + 1 == t.n) {
            // the item's rotary rows (positions kt 128 ..), once the previous
            // item's epilogue has read its own
            if (!ptx::mbar_wait(rope_empty, (it & 1) ^ 1, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* rb = smem + DkvCfg::kOffRope;
            ptx::mbar_arrive_expect_tx(rope_full, DkvCfg::kRopeBytes);
#pragma unroll
            for (int bx = 0; bx < 4; ++bx) ptx::tma_load_2d(rb + bx * 16384, &map_rope, rope_full, bx * 32, t.kt * 128);
            ++issued_rope;
          }
        }
      }
      if (!ok) {  // before the CTA exits every issued copy must have landed
        give_up();
        if (issued_kv > 0) ptx::mbar_wait(kv_full, (issued_kv - 1) & 1, nullptr);
        if (issued_rope > 0) ptx::mbar_wait(rope_full, (issued_rope - 1) & 1, nullptr);
        for (int u = (issued > kKvStages ? issued - kKvStages : 0); u < issued; ++u)
          ptx::mbar_wait(&st_full[u % kKvStages], (u / kKvStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_s = ptx::idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t id_g = ptx::idesc_bf16(128, 128, 0, 1);
      const uint64_t dk0 = kdesc0(ptx::smem_addr(sK)), dv0 = kdesc0(ptx::smem_addr(sV)),
                     dst0 = kdesc0(ptx::smem_addr(sStage)), dstmn0 = mndesc0(ptx::smem_addr(sStage), kAtAtom64);
      auto issue_sp = [&](int gs) {  // S^T and dP^T of the CTA's iteration gs into TMEM buffer gs & 1
        const int s = gs % kKvStages, b2 = gs & 1;
        if (!ptx::mbar_wait(&st_full[s], (gs / kKvStages) & 1, abort_flag)) return false;
        ptx::tc_fence_after();
        const uint64_t dq = dadd(dst0, s * DkvCfg::kStage), ddo = dadd(dq, 2 * kAtAtom64);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + static_cast<uint32_t>(b2 * 64), kstep(dk0, kk, kAtAtom128), kstep(dq, kk, kAtAtom64),
                        id_s, kk ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_bf16(tmem + 128u + static_cast<uint32_t>(b2 * 64), kstep(dv0, kk, kAtAtom128),
                        kstep(ddo, kk, kAtAtom64), id_s, kk ? 1u : 0u);
        ptx::mma_commit(&sp_full[b2]);
        return true;
      };
      bool ok = true;
      int it = 0, gs = 0;
      for (int k = 0, item = nth_item(0); ok && item < nitems; item = nth_item(++k), ++it) {
        const int n = item_of(item).n;  // >= hpc * 2
        if (!ptx::mbar_wait(kv_full, it & 1, abort_flag) || !issue_sp(gs)) {
          ok = false;
          break;
        }
        for (int u = 0; u < n; ++u) {
          const int cur = gs + u;
          if (u + 1 < n) {
            if (!issue_sp(cur + 1)) {
              ok = false;
              break;
            }
            if (u + 2 == n) ptx::mma_commit(kv_empty);  // the item's last S^T / dP^T have been issued
          }
          if (!ptx::mbar_wait(&ds_full[cur & 1], (cur >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t qmn = dadd(dstmn0, (cur % kKvStages) * DkvCfg::kStage), domn = dadd(qmn, 2 * kAtAtom64);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_bf16_ts(tmem + 256u, tmem + ds_col(cur & 1, kk), mnstep(domn, kk), id_g, (u | kk) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_bf16_ts(tmem + 384u, tmem + 128u + ds_col(cur & 1, kk), mnstep(qmn, kk), id_g,
                             (u | kk) ? 1u : 0u);
          ptx::mma_commit(&st_empty[cur % kKvStages]);
        }
        if (!ok) break;
        ptx::mma_commit(acc_full);
        gs += n;
      }
      if (!ok) {
        give_up();
        ptx::mma_commit(drain);
        ptx::mbar_wait(drain, 0, nullptr);
      }
    }
  } else {
    // Worker (quarter, half): key row r, query columns 32 half .. 32 half + 31
    // of each 64-query block; in the epilogue dV / dK columns 64 half ..
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;  // key row in the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    auto wait_all = [&](uint64_t* bar, uint32_t par) {
      bool w = ptx::mbar_wait(bar, par, abort_flag);
      w = __all_sync(0xffffffffu, w);
      if (!w && lane == 0 && !*abort_flag) give_up();
      return w;
    };
    bool ok = true;
    int it = 0, gs = 0;
    for (int k = 0, item = nth_item(0); ok && item < nitems; item = nth_item(++k), ++it) {
      const Item t = item_of(item);
      const int kpos = t.kt * 128 + r;  // key position in the sequence
      for (int u = 0; u < t.n; ++u) {
        const int cur = gs + u;
        const int b2 = cur & 1;
        if (!wait_all(&sp_full[b2], (cur >> 1) & 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // this half's 32 query rows: lse (scaled to log2) and Di, from the stage's shared copy
        const uint32_t ls_addr = ptx::smem_addr(smem + DkvCfg::kOffLD) + (cur % kKvStages) * 512 + half * 128;
        float lse2[32], dis[32];
#pragma unroll
        for (int v4 = 0; v4 < 8; ++v4) {
          const float4 lv = lds128(ls_addr + v4 * 16), dv4 = lds128(ls_addr + 256 + v4 * 16);
          lse2[4 * v4] = lv.x * kLog2e;
          lse2[4 * v4 + 1] = lv.y * kLog2e;
          lse2[4 * v4 + 2] = lv.z * kLog2e;
          lse2[4 * v4 + 3] = lv.w * kLog2e;
          dis[4 * v4] = dv4.x;
          dis[4 * v4 + 1] = dv4.y;
          dis[4 * v4 + 2] = dv4.z;
          dis[4 * v4 + 3] = dv4.w;
        }
        const int q0 = (2 * t.kt + u % t.nqb) * 64 + half * 32;
        uint32_t wp[16], wd[16];
        {
          uint32_t us[32], up[32];
          ptx::tmem_ld_32x32b_x32(lane_base + static_cast<uint32_t>(b2 * 64 + half * 32), us);
          ptx::tmem_ld_32x32b_x32(lane_base + 128u + static_cast<uint32_t>(b2 * 64 + half * 32), up);
          ptx::tmem_wait_ld();
          auto pds = [&](auto masked) {  // only the two query blocks of the key tile's own rows reach the diagonal
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float p2[2], d2[2];
#pragma unroll
              for (int v = 0; v < 2; ++v) {
                const int qi = e + v;
                float p = ex2(fmaf(__uint_as_float(us[qi]), a.c, -lse2[qi]));
                if (decltype(masked)::value && q0 + qi < kpos) p = 0.0f;
                p2[v] = p;
                d2[v] = p * (__uint_as_float(up[qi]) - dis[qi]);
              }
              wp[e / 2] = pack2(p2[0], p2[1]);
              wd[e / 2] = pack2(d2[0], d2[1]);
            }
          };
          if (u % t.nqb < 2)
            pds(std::true_type{});
          else
            pds(std::false_type{});
        }
        // P^T and dS^T of this half's 32 queries over the first 16 columns of
        // the S^T and dP^T columns this thread has just read
        ptx::tmem_st_32x32b_x16(lane_base + static_cast<uint32_t>(b2 * 64 + half * 32), wp);
        ptx::tmem_st_32x32b_x16(lane_base + 128u + static_cast<uint32_t>(b2 * 64 + half * 32), wd);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ds_full[b2]);
      }
      if (!ok || !wait_all(acc_full, it & 1)) {
        ok = false;
        break;
      }
      // dV and dK leave TMEM before this warp's next arrival, after which the
      // next item's first MMAs overwrite them
      ptx::tc_fence_after();
      if (hpc == a.H / a.Hkv) {
        // every query head of the kv head is in: dV and dK of rotation pairs 32 half ..
        uint32_t lo[32], hi[32];
        ptx::tmem_ld_32x32b_x32(lane_base + 256u + static_cast<uint32_t>(half * 32), lo);
        ptx::tmem_ld_32x32b_x32(lane_base + 256u + static_cast<uint32_t>(64 + half * 32), hi);
        ptx::tmem_wait_ld();
        store_grad_pairs(lo, hi, 1.0f, nullptr, half, a.out1 + static_cast<int64_t>(t.key0 + r) * a.ld1 + t.g * 128);
        uint16_t* dk_row = a.out0 + static_cast<int64_t>(t.key0 + r) * a.ld0 + t.g * 128;
        if (a.rope) {
          RotRow rot;
          if (!wait_all(rope_full, it & 1)) {
            ok = false;
            break;
          }
          {
            // row r of the cos box of this half and of the sin box, 16 bytes at a time
            const uint32_t rb = ptx::smem_addr(smem + DkvCfg::kOffRope);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t off = static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
              rot.c[c] = lds128(rb + static_cast<uint32_t>(half * 16384) + off);
              rot.s[c] = lds128(rb + static_cast<uint32_t>((2 + half) * 16384) + off);
            }
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(rope_empty);
          ptx::tmem_ld_32x32b_x32(lane_base + 384u + static_cast<uint32_t>(half * 32), lo);
          ptx::tmem_ld_32x32b_x32(lane_base + 384u + static_cast<uint32_t>(64 + half * 32), hi);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          store_grad_pairs(lo, hi, 0.08838834764831845f, &rot, half, dk_row);
        } else {
          ptx::tmem_ld_32x32b_x32(lane_base + 384u + static_cast<uint32_t>(half * 32), lo);
          ptx::tmem_ld_32x32b_x32(lane_base + 384u + static_cast<uint32_t>(64 + half * 32), hi);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          store_grad_pairs(lo, hi, 0.08838834764831845f, nullptr, half, dk_row);
        }
      } else {
        // fp32 partials of this query head, row key0 + r, columns 64 half ..
        const int64_t row = static_cast<int64_t>(t.h0) * M + t.key0 + r;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float* dst = (part ? part_dk : part_dv) + row * 128 + half * 64;
          uint32_t u0[32], u1[32];
          const uint32_t base = lane_base + (part ? 384u : 256u) + static_cast<uint32_t>(half * 64);
          ptx::tmem_ld_32x32b_x32(base, u0);
          ptx::tmem_ld_32x32b_x32(base + 32, u1);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            reinterpret_cast<float4*>(dst)[e / 4] = make_float4(__uint_as_float(u0[e]), __uint_as_float(u0[e + 1]),
                                                                __uint_as_float(u0[e + 2]), __uint_as_float(u0[e + 3]));
            reinterpret_cast<float4*>(dst + 32)[e / 4] =
                make_float4(__uint_as_float(u1[e]), __uint_as_float(u1[e + 1]), __uint_as_float(u1[e + 2]),
                            __uint_as_float(u1[e + 3]));
          }
        }
        ptx::tc_fence_before();
      }
      gs += t.n;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// dk[row, g*128 + i] = rot^-1(scale * sum_{h of g} part_dk[h][row]) and
// dv = sum_{h of g} part_dv[h][row] in head order, bf16.  One thread per
// (row, kv head, 8 rotation pairs): columns i .. i+7 and 64 + i .. 64 + i + 7.
__global__ void attn_kv_reduce_kernel(const float* __restrict__ part_dk, const float* __restrict__ part_dv, int64_t M,
                                      int S, int H, int Hkv, const float* __restrict__ rope, float scale,
                                      uint16_t* __restrict__ dk, int64_t lddk, uint16_t* __restrict__ dv,
                                      int64_t lddv) {
  pdl_trigger();
  pdl_wait();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= M * Hkv * 8) return;
  const int64_t row = t / (Hkv * 8);
  const int gc = static_cast<int>(t % (Hkv * 8));
  const int g = gc / 8, c = gc % 8;
  const int rep = H / Hkv;
  float k1[8] = {}, k2[8] = {}, v1[8] = {}, v2[8] = {};
  for (int i = 0; i < rep; ++i) {
    const int64_t base = (static_cast<int64_t>(g * rep + i) * M + row) * 128 + c * 8;
    const float4* pk = reinterpret_cast<const float4*>(part_dk + base);
    const float4* pv = reinterpret_cast<const float4*>(part_dv + base);
    const float4 a0 = pk[0], a1 = pk[1], b0 = pk[16], b1 = pk[17];
    const float4 c0 = pv[0], c1 = pv[1], d0 = pv[16], d1 = pv[17];
    const float ka[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float kb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const float va[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float vb[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      k1[e] += ka[e];
      k2[e] += kb[e];
      v1[e] += va[e];
      v2[e] += vb[e];
    }
  }
  uint32_t o1[4], o2[4], w1[4], w2[4];
  const float* cs = rope ? rope + (row % S) * 128 + c * 8 : nullptr;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float y1[2], y2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float x1 = k1[e + u] * scale, x2 = k2[e + u] * scale;
      if (cs) {
        const float cv = cs[e + u], sv = cs[64 + e + u];
        y1[u] = x1 * cv + x2 * sv;
        y2[u] = x2 * cv - x1 * sv;
      } else {
        y1[u] = x1;
        y2[u] = x2;
      }
    }
    o1[e / 2] = pack2(y1[0], y1[1]);
    o2[e / 2] = pack2(y2[0], y2[1]);
    w1[e / 2] = pack2(v1[e], v1[e + 1]);
    w2[e / 2] = pack2(v2[e], v2[e + 1]);
  }
  uint16_t* pk = dk + row * lddk + g * 128 + c * 8;
  uint16_t* pv = dv + row * lddv + g * 128 + c * 8;
  *reinterpret_cast<uint4*>(pk) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
  *reinterpret_cast<uint4*>(pk + 64) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
  *reinterpret_cast<uint4*>(pv) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  *reinterpret_cast<uint4*>(pv + 64) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
}

// ------------------------------------------------------------ host side
// Algorithmic FLOPs: 2 d per product per visible (query, key) pair; the
// forward has 2 products (Q K^T, P V), the backward 5 (S recomputed once, dP,
// dV, dQ, dK).
double causal_pairs(const AttnShape& sh) {
  return static_cast<double>(sh.M / sh.S) * sh.H * static_cast<double>(sh.S) * (sh.S + 1) / 2.0;
}

sl_status check_shape(const AttnShape& sh) {
  SL_REQUIRE(sh.M > 0 && sh.S > 0 && sh.S % 128 == 0 && sh.M % sh.S == 0,
             "attention: need S a positive multiple of 128 and M a multiple of S");
  SL_REQUIRE(sh.H > 0 && sh.Hkv > 0 && sh.H % sh.Hkv == 0, "attention: need H a multiple of Hkv");
  SL_REQUIRE(sh.M < (1LL << 31) && static_cast<int64_t>(sh.H) * sh.M < (1LL << 31), "attention: M too large");
  return SL_OK;
}

sl_status map_rows(CUtensorMap* m, const uint16_t* base, int64_t cols, int64_t rows, int64_t ld, int box_rows) {
  SL_REQUIRE(base, "attention: null operand");
  SL_REQUIRE(ld >= cols && (ld * 2) % 16 == 0, "attention: row stride must cover the row and be a multiple of 8");
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                  static_cast<uint64_t>(ld) * 2, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename K>
sl_status set_smem(K kern, int bytes) {
  static bool done[64] = {false};
  int dev = 0;
  SL_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64 || !done[dev]) {
    SL_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
    if (dev >= 0 && dev < 64) done[dev] = true;
  }
  return SL_OK;
}

}  // namespace

sl_status rope_table(int64_t S, double theta, float* table, cudaStream_t stream) {
  SL_REQUIRE(S > 0 && table && theta > 1.0, "rope table: need S > 0, theta > 1 and a table");
  const int64_t n = S * 64;
  return launch_pdl("rope_table_kernel", rope_table_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                    stream, S, theta, table);
}

sl_status rope_apply(uint16_t* x, int64_t ld, int64_t M, int nheads, int64_t S, const float* table, int inverse,
                     cudaStream_t stream) {
  SL_REQUIRE(x && table && M > 0 && nheads > 0 && S > 0 && ld >= nheads * 128 && ld % 8 == 0,
             "rope: bad arguments");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(x) & 15) == 0, "rope: x must be 16-byte aligned");
  const int64_t n = M * nheads * 8;
  return launch_pdl("rope_apply_kernel", rope_apply_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0,
                    stream, x, ld, M, nheads, S, table, inverse ? -1.0f : 1.0f);
}

sl_status attention_fwd(const AttnShape& sh, const uint16_t* q, int64_t ldq, const uint16_t* k, int64_t ldk,
                        const uint16_t* v, int64_t ldv, uint16_t* o, int64_t ldo, float* lse, cudaStream_t stream) {
  sl_status st = check_shape(sh);
  if (st != SL_OK) return st;
  SL_REQUIRE(o && lse && ldo >= sh.H * 128 && ldo % 8 == 0 && (reinterpret_cast<uintptr_t>(o) & 15) == 0,
             "attention_fwd: bad output");
  CUtensorMap mq, mk, mv, mo;
  if ((st = map_rows(&mq, q, sh.H * 128, sh.M, ldq, 128)) != SL_OK) return st;
  if ((st = map_rows(&mk, k, sh.Hkv * 128, sh.M, ldk, 128)) != SL_OK) return st;
  if ((st = map_rows(&mv, v, sh.Hkv * 128, sh.M, ldv, 128)) != SL_OK) return st;
  if ((st = map_rows(&mo, o, sh.H * 128, sh.M, ldo, 32)) != SL_OK) return st;
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  AttnArgs a{};
  a.S = static_cast<int>(sh.S);
  a.H = sh.H;
  a.Hkv = sh.Hkv;
  a.nseq = static_cast<int>(sh.M / sh.S);
  a.c = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));
  a.out0 = o;
  a.ld0 = ldo;
  a.lse = lse;
  a.err = err;
  if ((st = set_smem(attn_fwd_kernel, FwdCfg::kSmem)) != SL_OK) return st;
  const int64_t items = (sh.S / 128) * sh.H * a.nseq;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(items, num_sms()));
  const TimingToken tt = timing_begin(9, 2.0 * 2.0 * kAtD * causal_pairs(sh), stream);
  st = launch_pdl("attn_fwd_kernel", attn_fwd_kernel, dim3(grid), dim3(kAtThreads), FwdCfg::kSmem, stream, mq, mk, mv,
                  mo, a);
  timing_end(tt, stream);
  return st;
}

// Backward workspace: Di [H, M], then the fp32 partials of dK and dV [H, M, 128] each.
static size_t di_bytes(int64_t M, int H) { return (static_cast<size_t>(M) * H * 4 + 255) / 256 * 256; }
size_t attention_ws_bytes(int64_t M, int H) { return di_bytes(M, H) + 2 * static_cast<size_t>(M) * H * 128 * 4; }

static sl_status attention_bwd_launch(const AttnShape& sh, const uint16_t* q, int64_t ldq, const uint16_t* k,
                                      int64_t ldk, const uint16_t* v, int64_t ldv, const uint16_t* o, int64_t ldo,
                                      const uint16_t* dout, int64_t lddo, const float* lse, uint16_t* dq,
                                      int64_t lddq, uint16_t* dk, int64_t lddk, uint16_t* dv, int64_t lddv,
                                      const float* rope, float* Di, int* err, cudaStream_t stream);

sl_status attention_bwd(const AttnShape& sh, const uint16_t* q, int64_t ldq, const uint16_t* k, int64_t ldk,
                        const uint16_t* v, int64_t ldv, const uint16_t* o, int64_t ldo, const uint16_t* dout,
                        int64_t lddo, const float* lse, uint16_t* dq, int64_t lddq, uint16_t* dk, int64_t lddk,
                        uint16_t* dv, int64_t lddv, const float* rope, void* ws, cudaStream_t stream) {
  sl_status st = check_shape(sh);
  if (st != SL_OK) return st;
  SL_REQUIRE(o && dout && lse && ws && dq && dk && dv, "attention_bwd: null argument");
  SL_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 15) == 0 && (reinterpret_cast<uintptr_t>(lse) & 15) == 0,
             "attention_bwd: lse and workspace must be 16-byte aligned");
  SL_REQUIRE(ldo % 8 == 0 && lddo % 8 == 0 && (reinterpret_cast<uintptr_t>(o) & 15) == 0 &&
                 (reinterpret_cast<uintptr_t>(dout) & 15) == 0,
             "attention_bwd: o and do rows must be 16-byte aligned");
  for (auto pr : {std::make_pair(static_cast<const void*>(dq), lddq), std::make_pair(static_cast<const void*>(dk), lddk),
                  std::make_pair(static_cast<const void*>(dv), lddv)})
    SL_REQUIRE((reinterpret_cast<uintptr_t>(pr.first) & 15) == 0 && pr.second % 8 == 0,
               "attention_bwd: gradient outputs must be 16-byte aligned with row strides a multiple of 8");
  SL_REQUIRE(lddq >= sh.H * 128 && lddk >= sh.Hkv * 128 && lddv >= sh.Hkv * 128, "attention_bwd: row strides");
  int* err = device_error_word();
  if (!err) return SL_ERR_CUDA;
  float* Di = static_cast<float*>(ws);
  const TimingToken tt = timing_begin(10, 5.0 * 2.0 * kAtD * causal_pairs(sh), stream);
  st = attention_bwd_launch(sh, q, ldq, k, ldk, v, ldv, o, ldo, dout, lddo, lse, dq, lddq, dk, lddk, dv, lddv, rope,
                            Di, err, stream);
  timing_end(tt, stream);
  return st;
}

static sl_status attention_bwd_launch(const AttnShape& sh, const uint16_t* q, int64_t ldq, const uint16_t* k,
                                      int64_t ldk, const uint16_t* v, int64_t ldv, const uint16_t* o, int64_t ldo,
                                      const uint16_t* dout, int64_t lddo, const float* lse, uint16_t* dq,
                                      int64_t lddq, uint16_t* dk, int64_t lddk, uint16_t* dv, int64_t lddv,
                                      const float* rope, float* Di, int* err, cudaStream_t stream) {
  sl_status st;
  AttnArgs a{};
  a.S = static_cast<int>(sh.S);
  a.H = sh.H;
  a.Hkv = sh.Hkv;
  a.nseq = static_cast<int>(sh.M / sh.S);
  a.c = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));
  a.lse = const_cast<float*>(lse);
  a.Di = Di;
  a.rope = rope;
  a.err = err;
  // dQ
  {
    CUtensorMap mq, mdo, mo, mk, mv, mdq;
    if ((st = map_rows(&mq, q, sh.H * 128, sh.M, ldq, 128)) != SL_OK) return st;
    if ((st = map_rows(&mdo, dout, sh.H * 128, sh.M, lddo, 128)) != SL_OK) return st;
    if ((st = map_rows(&mo, o, sh.H * 128, sh.M, ldo, 128)) != SL_OK) return st;
    if ((st = map_rows(&mdq, dq, sh.H * 128, sh.M, lddq, 32)) != SL_OK) return st;
    if ((st = map_rows(&mk, k, sh.Hkv * 128, sh.M, ldk, 64)) != SL_OK) return st;
    if ((st = map_rows(&mv, v, sh.Hkv * 128, sh.M, ldv, 64)) != SL_OK) return st;
    AttnArgs ad = a;
    ad.out0 = dq;
    ad.ld0 = lddq;
    if ((st = set_smem(attn_dq_kernel, DqCfg::kSmem)) != SL_OK) return st;
    const int64_t items = (sh.S / 128) * sh.H * a.nseq;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(items, num_sms()));
    if ((st = launch_pdl("attn_dq_kernel", attn_dq_kernel, dim3(grid), dim3(kAtThreads), DqCfg::kSmem, stream, mq, mdo,
                         mo, mk, mv, mdq, ad)) != SL_OK)
      return st;
  }
  // dK, dV
  {
    CUtensorMap mq, mdo, mk, mv, ml, md;
    if ((st = map_rows(&mq, q, sh.H * 128, sh.M, ldq, 64)) != SL_OK) return st;
    if ((st = map_rows(&mdo, dout, sh.H * 128, sh.M, lddo, 64)) != SL_OK) return st;
    if ((st = map_rows(&mk, k, sh.Hkv * 128, sh.M, ldk, 128)) != SL_OK) return st;
    if ((st = map_rows(&mv, v, sh.Hkv * 128, sh.M, ldv, 128)) != SL_OK) return st;
    if ((st = make_map(&ml, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, lse, static_cast<uint64_t>(sh.M),
                       static_cast<uint64_t>(sh.H), static_cast<uint64_t>(sh.M) * 4, 64, 1,
                       CU_TENSOR_MAP_SWIZZLE_NONE)) != SL_OK)
      return st;
    if ((st = make_map(&md, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, Di, static_cast<uint64_t>(sh.M),
                       static_cast<uint64_t>(sh.H), static_cast<uint64_t>(sh.M) * 4, 64, 1,
                       CU_TENSOR_MAP_SWIZZLE_NONE)) != SL_OK)
      return st;
    float* part_dk = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(Di) + di_bytes(sh.M, sh.H));
    float* part_dv = part_dk + static_cast<size_t>(sh.M) * sh.H * 128;
    if ((st = set_smem(attn_dkdv_kernel, DkvCfg::kSmem)) != SL_OK) return st;
    // an item per kv head when that alone fills the GPU or a kv head has one
    // query head (no partials), else per query head
    const bool direct = sh.H == sh.Hkv || (sh.S / 128) * sh.Hkv * a.nseq >= num_sms();
    AttnArgs ak = a;
    ak.heads_per_cta = direct ? sh.H / sh.Hkv : 1;
    ak.out0 = dk;
    ak.ld0 = lddk;
    ak.out1 = dv;
    ak.ld1 = lddv;
    const int64_t items = (sh.S / 128) * (sh.H / ak.heads_per_cta) * a.nseq;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(items, num_sms()));
    // the rotary table [S, 128] fp32 as 128-row boxes of 32 columns (the direct epilogue's rows)
    CUtensorMap mr = ml;
    if (rope && direct &&
        (st = make_map(&mr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rope, 128, static_cast<uint64_t>(sh.S), 128 * 4, 32, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B)) != SL_OK)
      return st;
    if ((st = launch_pdl("attn_dkdv_kernel", attn_dkdv_kernel, dim3(grid), dim3(kAtThreads), DkvCfg::kSmem, stream, mq,
                         mdo, mk, mv, ml, md, mr, ak, part_dk, part_dv)) != SL_OK)
      return st;
    if (direct) return SL_OK;
    const int64_t nt = sh.M * sh.Hkv * 8;
    if ((st = launch_pdl("attn_kv_reduce_kernel", attn_kv_reduce_kernel, dim3(static_cast<unsigned>((nt + 255) / 256)),
                         dim3(256), 0, stream, static_cast<const float*>(part_dk), static_cast<const float*>(part_dv),
                         sh.M, static_cast<int>(sh.S), sh.H, sh.Hkv, rope, 0.08838834764831845f, dk, lddk, dv,
                         lddv)) != SL_OK)
      return st;
  }
  return SL_OK;
}

}  // namespace sl

// ------------------------------------------------------------------ C ABI
using namespace sl;

extern "C" sl_status sl_rope_table(int64_t S, double theta, float* table, cudaStream_t stream) {
  return rope_table(S, theta, table, stream);
}

extern "C" sl_status sl_rope_apply(void* x, int64_t ld, int64_t M, int32_t nheads, int64_t S, const float* table,
                                   int32_t inverse, cudaStream_t stream) {
  return rope_apply(static_cast<uint16_t*>(x), ld, M, nheads, S, table, inverse, stream);
}

extern "C" sl_status sl_attention_fwd(const void* q, int64_t ldq, const void* k, int64_t ldk, const void* v,
                                      int64_t ldv, int64_t M, int64_t S, int32_t H, int32_t Hkv, void* o,
                                      int64_t ldo, float* lse, cudaStream_t stream) {
  const AttnShape sh{M, S, H, Hkv};
  return attention_fwd(sh, static_cast<const uint16_t*>(q), ldq, static_cast<const uint16_t*>(k), ldk,
                       static_cast<const uint16_t*>(v), ldv, static_cast<uint16_t*>(o), ldo, lse, stream);
}

extern "C" size_t sl_attention_workspace_size(int64_t M, int32_t H) {
  return M > 0 && H > 0 ? attention_ws_bytes(M, H) : 0;
}

extern "C" sl_status sl_attention_bwd(const void* q, int64_t ldq, const void* k, int64_t ldk, const void* v,
                                      int64_t ldv, const void* o, int64_t ldo, const void* dO, int64_t lddo,
                                      const float* lse, int64_t M, int64_t S, int32_t H, int32_t Hkv, void* dq,
                                      int64_t lddq, void* dk, int64_t lddk, void* dv, int64_t lddv,
                                      const float* rope_table_or_null, void* ws, size_t ws_bytes,
                                      cudaStream_t stream) {
  const AttnShape sh{M, S, H, Hkv};
  SL_REQUIRE(M > 0 && H > 0 && ws_bytes >= attention_ws_bytes(M, H), "sl_attention_bwd: workspace too small");
  return attention_bwd(sh, static_cast<const uint16_t*>(q), ldq, static_cast<const uint16_t*>(k), ldk,
                       static_cast<const uint16_t*>(v), ldv, static_cast<const uint16_t*>(o), ldo,
                       static_cast<const uint16_t*>(dO), lddo, lse, static_cast<uint16_t*>(dq), lddq,
                       static_cast<uint16_t*>(dk), lddk, static_cast<uint16_t*>(dv), lddv, rope_table_or_null, ws,
                       stream);
}
