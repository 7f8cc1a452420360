// Host side of the tcgen05 GEMM: TMA tensor maps and launch dispatch.
#include <cudaTypedefs.h>

#include <mutex>
#include <vector>

#include "gemm.cuh"
#include "gemm2.cuh"

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

// 2-D map over a row-major matrix: inner extent `cols`, outer `rows`, row
// pitch `pitch_bytes`; box (box_cols x box_rows).
static sl_status make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
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
  if (g.epi == kEpiCELse) return 4;
  if (g.epi == kEpiCEGrad) return 5;
  if (g.epi == kEpiAddF32) return 6;
  return (g.bsrc == kBSrcNF4 ? 0 : 2) + (g.bmn ? 1 : 0);
}
}  // namespace

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
  dim3 grid(static_cast<unsigned>(2 * ceil_div(a.M, 256)), static_cast<unsigned>(ceil_div(a.N, kBN)));
  kern<<<grid, kGemm2Threads, Gemm2Cfg::kSmem, stream>>>(ma, mc, ms, a);
  return check_launch("gemm_nf4_pair_kernel");
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
  dim3 grid(static_cast<unsigned>(ceil_div(a.N, kBN)), static_cast<unsigned>(ceil_div(a.M, kBM)));
  kern<<<grid, kGemmThreads, Cfg::kSmem, stream>>>(ma, mb, ms, a);
  return check_launch("gemm_tc_kernel");
}

sl_status dispatch(const GemmLaunch& g, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& ms,
                   cudaStream_t stream);

sl_status launch_gemm(const GemmLaunch& g, cudaStream_t stream) {
  const GemmArgs& a = g.args;
  if (a.M <= 0 || a.N <= 0 || a.K <= 0) return set_error(SL_ERR_INVALID, "gemm: empty problem");
  if (a.N % 32) return set_error(SL_ERR_INVALID, "gemm: output columns must be a multiple of 32");
  if (a.r < 0 || a.r > 32 || (a.r % 8)) return set_error(SL_ERR_INVALID, "gemm: LoRA rank must be 0..32, multiple of 8");
  CUtensorMap ma, mb, ms;
  bool pair = false;
  sl_status st = make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.A, a.K, a.M, g.lda * 2, kBK, kBM,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != SL_OK) return st;
  if (g.bsrc == kBSrcBF16) {
    if (!g.bmn)
      st = make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.w, a.K, a.N, g.ldw * 2, kBK, kBN,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    else
      st = make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.w, a.N, a.K, g.ldw * 2, 64, kBK,
                    CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != SL_OK) return st;
    ms = mb;
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
  TimedLaunch tl{nullptr, nullptr, 0, 0.0};
  {
    std::lock_guard<std::mutex> lk(g_time_mu);
    if (g_time_on) {
      tl.start = pool_event();
      tl.stop = pool_event();
      tl.variant = variant_of(g);
      tl.flops = 2.0 * a.M * static_cast<double>(a.N) * a.K + 2.0 * a.M * static_cast<double>(a.N) * a.r;
      if (tl.start) cudaEventRecord(tl.start, stream);
    }
  }
  st = pair ? (g.bmn ? run_pair<1>(ma, mb, ms, a, stream) : run_pair<0>(ma, mb, ms, a, stream))
            : dispatch(g, ma, mb, ms, stream);
  if (tl.start && tl.stop) {
    cudaEventRecord(tl.stop, stream);
    std::lock_guard<std::mutex> lk(g_time_mu);
    g_timed.push_back(tl);
  }
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
  SL_GEMM_CASE(kBSrcBF16, 0, kEpiCELse)
  SL_GEMM_CASE(kBSrcBF16, 0, kEpiCEGrad)
  SL_GEMM_CASE(kBSrcBF16, 1, kEpiAddF32)
#undef SL_GEMM_CASE
  return set_error(SL_ERR_UNSUPPORTED, "gemm: unsupported (source, layout, epilogue) combination");
}

}  // namespace sl

using namespace sl;

extern "C" sl_status sl_kernel_timing(int32_t enable) {
  std::lock_guard<std::mutex> lk(g_time_mu);
  for (auto& t : g_timed) {
    cudaEventSynchronize(t.stop);
    g_event_pool.push_back(t.start);
    g_event_pool.push_back(t.stop);
  }
  if (enable) g_timed.clear();
  g_time_on = enable != 0;
  return SL_OK;
}

extern "C" sl_status sl_kernel_timing_read(int32_t variant, uint64_t* launches, double* ms, double* flops) {
  SL_REQUIRE(variant >= 0 && variant <= 6, "sl_kernel_timing_read: variant must be 0..6");
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
