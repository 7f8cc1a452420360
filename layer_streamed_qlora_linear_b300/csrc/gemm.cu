// Host side of the tcgen05 GEMM: TMA tensor maps and launch dispatch.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "gemm.cuh"
#include "gemm2.cuh"
#include "gemm3.cuh"
#include "timing.cuh"
#include "tmap.cuh"

namespace sl {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

sl_status make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                          uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return set_error(SL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (pitch_bytes & 15))
    return set_error(SL_ERR_INVALID, "TMA operand: base and row pitch must be 16-byte aligned");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(SL_ERR_INVALID, "cuTensorMapEncodeTiled failed (code " + std::to_string((int)r) + ")");
  return SL_OK;
}

// ------------------------------------------------------------ launch timing
namespace {
struct TimedLaunch {
  cudaEvent_t start, stop;
  int variant;
  double flops;
};
std::mutex g_time_mu;
bool g_time_on = false;
std::vector<TimedLaunch> g_timed;
std::vector<cudaEvent_t> g_event_pool;
// Device-clock slots of the timed GEMM launches ({first start, last end}
// per launch, %globaltimer ns), allocated on the first timing enable.
constexpr int kClkSlots = 16384;
unsigned long long* g_clk = nullptr;
int g_clk_dev = -1;
int g_clk_used = 0;
std::vector<int> g_clk_slot;  // slot of g_timed[i], or -1

__global__ void clk_init_kernel(unsigned long long* c, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    c[2 * i] = ~0ull;
    c[2 * i + 1] = 0ull;
  }
}

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

int variant_of(const GemmLaunch& g) {
  if (g.epi == kEpiCEExp) return 4;
  if (g.epi == kEpiAddF32) return 5;
  return (g.bsrc == kBSrcNF4 ? 0 : 2) + (g.bmn ? 1 : 0);
}
}  // namespace

TimingToken timing_begin(int variant, double work, cudaStream_t stream) {
  TimingToken t;
  std::lock_guard<std::mutex> lk(g_time_mu);
  if (!g_time_on) return t;
  t.start = pool_event();
  t.stop = pool_event();
  t.variant = variant;
  t.work = work;
  int dev = -1;
  if (variant <= 5 && g_clk && cudaGetDevice(&dev) == cudaSuccess && dev == g_clk_dev && g_clk_used < kClkSlots)
    t.clk = g_clk + 2 * g_clk_used++;
  if (t.start) cudaEventRecord(t.start, stream);
  return t;
}

void timing_end(const TimingToken& t, cudaStream_t stream) {
  if (!t.start || !t.stop) return;
  cudaEventRecord(t.stop, stream);
  std::lock_guard<std::mutex> lk(g_time_mu);
  g_timed.push_back(TimedLaunch{t.start, t.stop, t.variant, t.work});
  g_clk_slot.push_back(t.clk ? static_cast<int>((t.clk - g_clk) / 2) : -1);
}

// NF4 GEMM on CTA pairs (M = 256 per pair); used when M > 128.
template <int BMN>
static sl_status run_pair(const CUtensorMap& ma, const CUtensorMap& mc, const CUtensorMap& ms, const GemmArgs& a,
                          cudaStream_t stream) {
  auto kern = gemm_nf4_pair_kernel<BMN>;
  static bool attr_set[64] = {false};
  int dev = 0;
  SL_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    SL_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gemm2Cfg::kSmem));
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // bf16 output by TMA boxes of 64 columns x 32 rows when a tensor map can
  // describe it (16-byte aligned base and row stride); else direct stores
  GemmArgs ao = a;
  CUtensorMap mo = ma;
  ao.tma_out = (reinterpret_cast<uintptr_t>(a.out) % 16 == 0) && (a.ld_out * 2) % 16 == 0 &&
               make_map(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.out, a.N, a.M, static_cast<uint64_t>(a.ld_out) * 2, 64,
                        32, CU_TENSOR_MAP_SWIZZLE_128B) == SL_OK;
  dim3 grid(static_cast<unsigned>(2 * ceil_div(a.M, 256)), static_cast<unsigned>(ceil_div(a.N, kBN)));
  return launch_pdl("gemm_nf4_pair_kernel", kern, grid, dim3(kGemm2Threads), Gemm2Cfg::kSmem, stream, ma, mc, ms, mo,
                    ao);
}

// The persistent pair kernel for a weight source (BF16 = 1: bf16 weights by
// TMA) and epilogue (NF4: the bf16 store only).
template <int BF16, int BMN, int SMALL, int EPI>
static auto pair_persistent_kernel() {
  static_assert(BF16 || EPI == kEpiStoreBF16, "NF4 pair GEMM: bf16 store epilogue only");
  if constexpr (BF16) return gemm_bf16_pair_persistent_kernel<BMN, SMALL, EPI>;
  else return gemm_nf4_pair_persistent_kernel<BMN, SMALL>;
}

// CTA pairs of the persistent kernel that the device holds at once (driver
// query, once per device); the grid never exceeds it, so all clusters run
// together and none waits for a second wave.
template <int BF16, int BMN, int SMALL, int EPI = kEpiStoreBF16>
static int pair_clusters_resident() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms() / 2;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    cudaFuncSetAttribute(pair_persistent_kernel<BF16, BMN, SMALL, EPI>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Gemm3Cfg<SMALL>::kSmem);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kGemm3Threads, 1, 1);
    cfg.dynamicSmemBytes = Gemm3Cfg<SMALL>::kSmem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, pair_persistent_kernel<BF16, BMN, SMALL, EPI>(), &cfg) != cudaSuccess ||
        n <= 0) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    cached[dev] = std::min(n, num_sms() / 2);
  }
  return cached[dev];
}

// Persistent NF4 GEMM on CTA pairs: one cluster per SM pair walks its share
// of the pair tiles.
// Most pieces a split tail tile is cut into: the owning piece reads every
// other piece's 128 KB partial per CTA, so pieces pay only while a piece's
// k-loop outlasts those reads (about KB / 4 pieces squared).
static int split_pieces(int KB) {
  int p = 1;
  while ((p + 1) * (p + 1) * 4 <= KB) ++p;
  return p;
}

static int max_split_slots() { return num_sms() / 2; }
static size_t split_flag_bytes() { return align_up(static_cast<size_t>(max_split_slots()) * 2 * 8, 256); }
size_t split_scratch_bytes() {
  return split_flag_bytes() + static_cast<size_t>(max_split_slots()) * 2 * kBN * 128 * 4;
}

// Splits the last partial wave along K when the tail tiles are few enough
// for two or more pieces each and scratch is given.
static void set_split(GemmArgs& a, int ntiles, int nclusters, void* ws, size_t bytes) {
  static std::atomic<unsigned long long> tag{0x5EEDull << 48};
  a.split_P = 0;
  const int R = ntiles % nclusters;
  if (!ws || bytes < split_scratch_bytes() || R == 0 || ntiles < nclusters) return;
  const int KB = static_cast<int>(ceil_div(a.K, kBK));
  const int P = std::min(nclusters / R, split_pieces(KB));
  if (P < 2 || R * (P - 1) > max_split_slots()) return;
  a.split_P = P;
  a.split_R = R;
  a.split_rounds = ntiles / nclusters;
  uint8_t* p = static_cast<uint8_t*>(ws);
  a.split_flag = reinterpret_cast<unsigned long long*>(p);
  a.split_part = reinterpret_cast<float*>(p + split_flag_bytes());
  a.split_tag = tag.fetch_add(1) + 1;
}

template <int BF16, int BMN, int SMALL, int EPI = kEpiStoreBF16>
static sl_status run_persistent(const CUtensorMap& ma, const CUtensorMap& mc, const CUtensorMap& ms,
                                const CUtensorMap& ms2, const GemmArgs& a, void* split_ws, size_t split_bytes,
                                cudaStream_t stream) {
  auto kern = pair_persistent_kernel<BF16, BMN, SMALL, EPI>();
  static bool attr_set[64] = {false};
  int dev = 0;
  SL_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    SL_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Gemm3Cfg<SMALL>::kSmem));
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int ntiles = ceil_div(a.M, 256) * ceil_div(a.N, kBN);
  const int nclusters = std::min(ntiles, pair_clusters_resident<BF16, BMN, SMALL, EPI>());
  GemmArgs ao = a;
  set_split(ao, ntiles, nclusters, split_ws, split_bytes);
  // bf16 output by TMA boxes of 64 columns x 32 rows when a tensor map can
  // describe it (16-byte aligned base and row stride); else direct stores
  // (always for the fp32 accumulation)
  CUtensorMap mo = ma;
  ao.tma_out = EPI != kEpiAddF32 && (reinterpret_cast<uintptr_t>(a.out) % 16 == 0) && (a.ld_out * 2) % 16 == 0 &&
               make_map(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.out, a.N, a.M, static_cast<uint64_t>(a.ld_out) * 2, 64,
                        32, CU_TENSOR_MAP_SWIZZLE_128B) == SL_OK;
  return launch_pdl(BF16 ? "gemm_bf16_pair_persistent_kernel" : "gemm_nf4_pair_persistent_kernel", kern,
                    dim3(static_cast<unsigned>(2 * nclusters)),
                    dim3(kGemm3Threads), Gemm3Cfg<SMALL>::kSmem, stream, ma, mc, ms, ms2, mo, ao);
}

template <int BSRC, int BMN, int EPI>
static sl_status run(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ms, const GemmArgs& a,
                     cudaStream_t stream) {
  using Cfg = GemmCfg<BSRC>;
  auto kern = gemm_tc_kernel<BSRC, BMN, EPI>;
  static bool attr_set[64] = {false};
  int dev = 0;
  SL_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    SL_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem));
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // The output moves by TMA when a tensor map can describe it (16-byte
  // aligned base and row stride); otherwise the epilogue stores directly.
  GemmArgs ao = a;
  CUtensorMap mo = ma;
  {
    const bool f32 = EPI == kEpiAddF32;
    const int esz = f32 ? 4 : 2;
    ao.tma_out = a.M >= 32 && a.N >= 128 && (reinterpret_cast<uintptr_t>(a.out) % 16 == 0) &&
                 (a.ld_out * esz) % 16 == 0 &&
                 make_map(&mo, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.out, a.N,
                          a.M, static_cast<uint64_t>(a.ld_out) * esz, f32 ? 32 : 64, 32,
                          CU_TENSOR_MAP_SWIZZLE_128B) == SL_OK;
  }
  dim3 grid(static_cast<unsigned>(ceil_div(a.N, kBN)), static_cast<unsigned>(ceil_div(a.M, kBM)));
  return launch_pdl("gemm_tc_kernel", kern, grid, dim3(kGemmThreads), Cfg::kSmem, stream, ma, mb, ms, mo, ao);
}

sl_status dispatch(const GemmLaunch& g, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ms,
                   cudaStream_t stream);
static sl_status launch_timed(const GemmLaunch& g, bool pair, const CUtensorMap& ma, const CUtensorMap& mb,
                              const CUtensorMap& ms, const CUtensorMap& ms2, const TimingToken& tl,
                              cudaStream_t stream);

sl_status launch_gemm(const GemmLaunch& g, cudaStream_t stream) {
  const GemmArgs& a = g.args;
  if (a.M <= 0 || a.N <= 0 || a.K <= 0) return set_error(SL_ERR_INVALID, "gemm: empty problem");
  if (a.N % 32) return set_error(SL_ERR_INVALID, "gemm: output columns must be a multiple of 32");
  if (a.r < 0 || a.r > (g.grouped ? kLoraMaxR : 32) || (a.r % 8))
    return set_error(SL_ERR_INVALID, "gemm: LoRA rank must be 0..32 (a group's 0..64), multiple of 8");
  if (g.grouped && (g.bsrc != kBSrcNF4 || g.epi != kEpiStoreBF16 || a.M <= kBM))
    return set_error(SL_ERR_UNSUPPORTED, "gemm: projection groups need NF4 weights and M > 128");
  if (a.dq && (g.bsrc != kBSrcNF4 || g.epi != kEpiStoreBF16 || a.M <= kBM))
    return set_error(SL_ERR_UNSUPPORTED, "gemm: the double-quantised absmax needs M > 128 (persistent pair GEMM)");
  CUtensorMap ma, mb, ms, ms2;
  bool pair = false;
  sl_status st = make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.A, a.K, a.M, g.lda * 2, kBK, kBM,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  if (g.bsrc == kBSrcBF16) {
    // CTA pairs (the persistent kernel) at M > 128 for the bf16 store and the
    // CE epilogues: each CTA loads its own 128 weight rows (K-major) or two
    // 64-column boxes (MN-major)
    pair = a.M > kBM && (g.epi == kEpiStoreBF16 || (g.epi == kEpiCEExp && !g.bmn) || (g.epi == kEpiAddF32 && g.bmn));
    if (!g.bmn)
      st = make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.w, a.K, a.N, g.ldw * 2, kBK, pair ? 128 : kBN,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    else
      st = make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.w, a.N, a.K, g.ldw * 2, 64, kBK,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != SL_OK) return st;
    ms = mb;
    ms2 = mb;
  } else {
    // NF4: codes are bytes (two elements each), absmax one fp32 per 64 elements of a row.
    const int64_t rows = g.bmn ? a.K : a.N;   // weight rows
    const int64_t cols = g.ldw;               // weight row length in elements
    if (cols % 256) return set_error(SL_ERR_INVALID, "gemm: NF4 weight rows must be a multiple of 256 elements");
    if (g.epi == kEpiStoreBF16 && a.M > kBM) {
      // CTA-pair kernel: each CTA maps its own half of the B tile.
      if (!g.bmn) {
        st = make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, cols / 2, rows, cols / 2, kBK / 2, 128,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st == SL_OK)
          st = make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.absmax, cols / 64, rows, cols / 64 * 4, 4, 128,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
      } else {
        st = make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, cols / 2, rows, cols / 2, 64, kBK,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st == SL_OK)
          st = make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.absmax, cols / 64, rows, cols / 64 * 4, 4, kBK,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
      }
      if (st == SL_OK && a.dq) {
        // int8 absmax, transposed: [cols / 64][dq_col0 + rows]; (c, s) pairs fp32
        // [cols / 64][2 per 256 of dq_col0 + rows], read as aligned 16-byte boxes
        const int64_t qcols = a.dq_col0 + rows, pcols = 2 * (qcols / 256);
        if (a.dq_col0 < 0 || a.dq_col0 % 256 || rows % 256 || g.q_ld < qcols || g.a2_ld < pcols)
          return set_error(SL_ERR_INVALID, "gemm: double-quantised absmax layout (column offset, row lengths)");
        st = make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.qabsmax, qcols, cols / 64, g.q_ld, g.bmn ? 64 : 128,
                      g.bmn ? 2 : 1, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st == SL_OK)
          st = make_map(&ms2, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.absmax2, pcols, cols / 64, g.a2_ld * 4, 4,
                        g.bmn ? 2 : 1, CU_TENSOR_MAP_SWIZZLE_NONE);
      } else {
        ms2 = ms;
      }
      if (st != SL_OK) return st;
      pair = true;
    } else if (!g.bmn) {
      st = make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, cols / 2, rows, cols / 2, kBK / 2, kBN,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
      if (st == SL_OK)
        st = make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.absmax, cols / 64, rows, cols / 64 * 4, 4, kBN,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
      st = make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.codes, cols / 2, rows, cols / 2, kBN / 2, kBK,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
      if (st == SL_OK)
        st = make_map(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.absmax, cols / 64, rows, cols / 64 * 4, 4, kBK,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (st != SL_OK) return st;
  }
  const TimingToken tl = timing_begin(
      variant_of(g), 2.0 * a.M * static_cast<double>(a.N) * a.K + 2.0 * a.M * static_cast<double>(a.N) * a.r, stream);
  GemmLaunch gc = g;  // with the launch's device-clock slot, if timed
  gc.args.clk = tl.clk;
  return launch_timed(gc, pair, ma, mb, ms, ms2, tl, stream);
}

static sl_status launch_timed(const GemmLaunch& g, bool pair, const CUtensorMap& ma, const CUtensorMap& mb,
                              const CUtensorMap& ms, const CUtensorMap& ms2, const TimingToken& tl,
                              cudaStream_t stream) {
  const GemmArgs& a = g.args;
  sl_status st = SL_OK;
  // More pair tiles than resident clusters: the persistent kernel (its
  // epilogue overlaps the next tile); one wave or less: one cluster per tile
  // with the epilogue spread over all eight dequant warps.
  // bf16 weights on CTA pairs: always the persistent kernel (the one-tile
  // pair kernel dequantises NF4 only); folded rank <= 32 there.
  const bool bf16_pair = pair && g.bsrc == kBSrcBF16;
  const bool persistent =
      pair && (bf16_pair || g.grouped || a.dq ||
               ceil_div(a.M, 256) * ceil_div(a.N, kBN) >
                   (g.bmn ? pair_clusters_resident<0, 1, 1>() : pair_clusters_resident<0, 0, 1>()));
  // folded rank <= 32: the five-stage variant; above (a group's dX): four stages
  if (bf16_pair && g.epi == kEpiCEExp)
    st = run_persistent<1, 0, 1, kEpiCEExp>(ma, mb, ms, ms2, a, g.split_ws, g.split_ws_bytes, stream);
  else if (bf16_pair && g.epi == kEpiAddF32)
    st = run_persistent<1, 1, 1, kEpiAddF32>(ma, mb, ms, ms2, a, g.split_ws, g.split_ws_bytes, stream);
  else if (bf16_pair)
    st = g.bmn ? run_persistent<1, 1, 1>(ma, mb, ms, ms2, a, g.split_ws, g.split_ws_bytes, stream)
               : run_persistent<1, 0, 1>(ma, mb, ms, ms2, a, g.split_ws, g.split_ws_bytes, stream);
  else if (persistent && a.r <= 32)
    st = g.bmn ? run_persistent<0, 1, 1>(ma, mb, ms, ms2, a, g.split_ws, g.split_ws_bytes, stream)
               : run_persistent<0, 0, 1>(ma, mb, ms, ms2, a, g.split_ws, g.split_ws_bytes, stream);
  else if (persistent)
    st = g.bmn ? run_persistent<0, 1, 0>(ma, mb, ms, ms2, a, g.split_ws, g.split_ws_bytes, stream)
               : run_persistent<0, 0, 0>(ma, mb, ms, ms2, a, g.split_ws, g.split_ws_bytes, stream);
  else
    st = pair ? (g.bmn ? run_pair<1>(ma, mb, ms, a, stream) : run_pair<0>(ma, mb, ms, a, stream))
              : dispatch(g, ma, mb, ms, stream);
  timing_end(tl, stream);
  return st;
}

sl_status dispatch(const GemmLaunch& g, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ms,
                   cudaStream_t stream) {
  const GemmArgs& a = g.args;
#define SL_GEMM_CASE(B, MN, E) \
  if (g.bsrc == B && g.bmn == MN && g.epi == E) return run<B, MN, E>(ma, mb, ms, a, stream);
  SL_GEMM_CASE(kBSrcNF4, 0, kEpiStoreBF16)
  SL_GEMM_CASE(kBSrcNF4, 1, kEpiStoreBF16)
  SL_GEMM_CASE(kBSrcBF16, 0, kEpiStoreBF16)
  SL_GEMM_CASE(kBSrcBF16, 1, kEpiStoreBF16)
  SL_GEMM_CASE(kBSrcBF16, 0, kEpiCEExp)
  SL_GEMM_CASE(kBSrcBF16, 1, kEpiAddF32)
#undef SL_GEMM_CASE
  return set_error(SL_ERR_UNSUPPORTED, "gemm: unsupported (source, layout, epilogue) combination");
}

}  // namespace sl

using namespace sl;

extern "C" sl_status sl_kernel_timing(int32_t enable) {
  std::lock_guard<std::mutex> lk(g_time_mu);
  if (enable) {
    // the previous region's records stay readable until timing is enabled
    // again; only then do their events go back to the pool (once each)
    for (auto& t : g_timed) {
      cudaEventSynchronize(t.stop);
      g_event_pool.push_back(t.start);
      g_event_pool.push_back(t.stop);
    }
    g_timed.clear();
    g_clk_slot.clear();
    // device-clock slots on the current device (outside any timed region: this synchronises)
    int dev = -1;
    SL_CHECK_CUDA(cudaGetDevice(&dev));
    if (g_clk && g_clk_dev != dev) {
      cudaFree(g_clk);
      g_clk = nullptr;
    }
    if (!g_clk) {
      SL_CHECK_CUDA(cudaMalloc(&g_clk, sizeof(unsigned long long) * 2 * kClkSlots));
      g_clk_dev = dev;
    }
    clk_init_kernel<<<64, 256>>>(g_clk, kClkSlots);
    SL_CHECK_CUDA(cudaGetLastError());
    SL_CHECK_CUDA(cudaDeviceSynchronize());
    g_clk_used = 0;
  }
  g_time_on = enable != 0;
  return SL_OK;
}

extern "C" sl_status sl_kernel_timing_read_clock(int32_t variant, uint64_t* launches, double* ms) {
  SL_REQUIRE(variant >= 0 && variant <= 5, "sl_kernel_timing_read_clock: variant must be a GEMM variant 0..5");
  std::lock_guard<std::mutex> lk(g_time_mu);
  uint64_t n = 0;
  double t = 0.0;
  if (g_clk && g_clk_used > 0) {
    for (auto& tl : g_timed) SL_CHECK_CUDA(cudaEventSynchronize(tl.stop));
    std::vector<unsigned long long> h(2 * static_cast<size_t>(g_clk_used));
    SL_CHECK_CUDA(cudaMemcpy(h.data(), g_clk, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < g_timed.size(); ++i) {
      const int sl_ = g_clk_slot[i];
      if (g_timed[i].variant != variant || sl_ < 0) continue;
      const unsigned long long a = h[2 * sl_], b = h[2 * sl_ + 1];
      if (a == ~0ull || b < a) continue;  // a launch that never stamped
      ++n;
      t += static_cast<double>(b - a) * 1e-6;
    }
  }
  if (launches) *launches = n;
  if (ms) *ms = t;
  return SL_OK;
}

extern "C" sl_status sl_kernel_timing_read(int32_t variant, uint64_t* launches, double* ms, double* flops) {
  SL_REQUIRE(variant >= 0 && variant < kNumTimedVariants, "sl_kernel_timing_read: variant must be 0..8");
  std::lock_guard<std::mutex> lk(g_time_mu);
  uint64_t n = 0;
  double t = 0.0, f = 0.0;
  for (auto& tl : g_timed) {
    if (tl.variant != variant) continue;
    SL_CHECK_CUDA(cudaEventSynchronize(tl.stop));
    float e = 0.0f;
    SL_CHECK_CUDA(cudaEventElapsedTime(&e, tl.start, tl.stop));
    ++n;
    t += e;
    f += tl.flops;
  }
  if (launches) *launches = n;
  if (ms) *ms = t;
  if (flops) *flops = f;
  return SL_OK;
}
