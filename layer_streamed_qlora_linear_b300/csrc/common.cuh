// Shared host/device helpers of libsl: status plumbing, the device error word,
// bf16 packing and small math.  No tensor-framework types anywhere in libsl.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>
#include <string>

#include "../../include/sl.h"

namespace sl {

// ---------------------------------------------------------------- errors (host)
// Records a message for sl_last_error() (thread-local) and returns the status.
sl_status set_error(sl_status st, const std::string& msg);
sl_status cuda_error(cudaError_t e, const char* what);

#define SL_CHECK_CUDA(expr)                                        \
  do {                                                             \
    cudaError_t _e = (expr);                                       \
    if (_e != cudaSuccess) return ::sl::cuda_error(_e, #expr);     \
  } while (0)

#define SL_REQUIRE(cond, msg)                                                  \
  do {                                                                         \
    if (!(cond)) return ::sl::set_error(SL_ERR_INVALID, std::string(msg));     \
  } while (0)

// After a launch: map a launch error to SL_ERR_CUDA; counts successful launches.
sl_status check_launch(const char* what);
uint64_t launch_count();  // libsl kernel launches so far (all threads)

// Programmatic dependent launch.  The training step's kernels are launched
// with programmatic stream serialisation: the next kernel in the stream may
// start while this one runs.  Every such kernel calls pdl_trigger() (its
// dependents may launch once every CTA of it has started, so waiting CTAs
// never hold resources its own CTAs need) and then pdl_wait() before its
// first global-memory access (returns once the previous kernel has completed
// and its writes are visible).  Both are no-ops under a normal launch.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch with programmatic stream serialisation (see above), then check_launch.
template <typename... KArgs, typename... Args>
sl_status launch_pdl(const char* what, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) return cuda_error(e, what);
  return check_launch(what);
}

// ------------------------------------------------------ device error word
// One int per device in a file-scope device array (zero at module load; no
// allocation), read and cleared by sl_check_device_errors().  Kernels whose
// bounded waits give up write a nonzero sl_status code here instead of
// trapping.
int* device_error_word();   // nullptr (and sl_last_error set) if its address cannot be found

// Bounded-wait limit used by every spin in libsl kernels (nanoseconds of
// %globaltimer).  A healthy wait in these kernels lasts microseconds; two
// seconds only expires when the producer side is gone.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// -------------------------------------------------------- device helpers
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report_device_error(int* word, int code) {
  if (word) atomicCAS(word, 0, code);
}

// Two floats -> packed bf16x2 (round to nearest even); lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int num_sms();

// A library-owned stream per device at the highest stream priority, created
// on first use (nullptr if that fails).  The LoRA backward runs its U pass
// and dX GEMM there while the adapter-gradient passes run on the caller's
// stream; blocks of the high-priority stream are dispatched first, so the
// gradient passes fill the SMs the GEMM leaves idle.
cudaStream_t hi_stream();
// Thread-local events for fork/join between a caller's stream and
// hi_stream() (per device; `i` < 4).
cudaEvent_t fork_event(int i);

}  // namespace sl
