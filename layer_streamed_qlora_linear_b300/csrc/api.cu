// Library-wide entry points: error reporting, version, the NF4 table export,
// the per-device error word and the bounded-wait probe.
#include <atomic>
#include <mutex>
#include <string>
#include <cstring>

#include "common.cuh"
#include "nf4.cuh"
#include "ptx.cuh"

namespace sl {

static thread_local std::string g_last_error;

sl_status set_error(sl_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

sl_status cuda_error(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return e == cudaErrorMemoryAllocation ? SL_ERR_OOM : SL_ERR_CUDA;
}

static std::atomic<uint64_t> g_launches{0};

sl_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, what);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SL_OK;
}

uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

// words[0]: error word; words[1]: a flag that nothing ever sets (timeout probe).
// A file-scope device array, zero when the module loads, so that no call of
// libsl allocates (or synchronises) to get it; its device address is looked
// up once per device with that device current.
static __device__ int g_device_words[2];
static std::mutex g_word_mu;
static int* g_words[64] = {nullptr};

static int* device_words() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    set_error(SL_ERR_CUDA, "device_error_word: no current device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_word_mu);
  if (!g_words[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_device_words);
    if (e != cudaSuccess || !p) {
      cuda_error(e, "device_error_word: cudaGetSymbolAddress");
      return nullptr;
    }
    g_words[dev] = static_cast<int*>(p);
  }
  return g_words[dev];
}

int* device_error_word() { return device_words(); }

cudaStream_t hi_stream() {
  static std::mutex mu;
  static cudaStream_t streams[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!streams[dev]) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&streams[dev], cudaStreamNonBlocking, greatest) != cudaSuccess) {
      cudaGetLastError();
      streams[dev] = nullptr;
    }
  }
  return streams[dev];
}

cudaEvent_t fork_event(int i) {
  thread_local cudaEvent_t events[64][4] = {};
  int dev = 0;
  if (i < 0 || i >= 4 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!events[dev][i] && cudaEventCreateWithFlags(&events[dev][i], cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    events[dev][i] = nullptr;
  }
  return events[dev][i];
}

int num_sms() {
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 148;
  }
  return sms[dev];
}

// Polls a flag nobody sets, or waits on an mbarrier nobody arrives on, until
// limit_ns elapses; then records SL_ERR_TIMEOUT and returns.
__global__ void timeout_probe_kernel(const volatile int* never, int* err, long long limit_ns, int use_mbar) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const unsigned long long t0 = globaltimer_ns();
  if (use_mbar) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
    for (uint32_t i = 0;; ++i) {
      if (ptx::mbar_try_wait(&bar, 0)) return;  // never completes: nobody arrives
      if ((i & 63u) == 0 && globaltimer_ns() - t0 > (unsigned long long)limit_ns) break;
    }
  } else {
    while (*never == 0) {
      if (globaltimer_ns() - t0 > (unsigned long long)limit_ns) break;
      __nanosleep(1000);
    }
    if (*never != 0) return;
  }
  report_device_error(err, SL_ERR_TIMEOUT);
}

}  // namespace sl

using namespace sl;

extern "C" {

const char* sl_last_error(void) { return g_last_error.c_str(); }

int32_t sl_version(void) { return 1 * 10000 + 0 * 100 + 0; }

uint64_t sl_launch_count(void) { return sl::launch_count(); }

void sl_nf4_code_table(float out[16]) {
  if (!out) return;
  for (int i = 0; i < 16; ++i) {
    uint32_t b = kNF4LevelBits[i];
    std::memcpy(&out[i], &b, 4);
  }
}

sl_status sl_check_device_errors(cudaStream_t stream) {
  int* w = device_words();
  if (!w) return SL_ERR_CUDA;
  SL_CHECK_CUDA(cudaStreamSynchronize(stream));
  int h = 0;
  SL_CHECK_CUDA(cudaMemcpy(&h, w, sizeof(int), cudaMemcpyDeviceToHost));
  if (h != 0) {
    SL_CHECK_CUDA(cudaMemset(w, 0, sizeof(int)));
    SL_CHECK_CUDA(cudaDeviceSynchronize());
    return set_error(static_cast<sl_status>(h), "a kernel recorded an error on the device (code " +
                                                    std::to_string(h) + ")");
  }
  return SL_OK;
}

sl_status sl_debug_timeout_probe(int64_t limit_ns, int32_t mbarrier, cudaStream_t stream) {
  int* w = device_words();
  if (!w) return SL_ERR_CUDA;
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 2000000000LL) limit_ns = 2000000000LL;
  timeout_probe_kernel<<<1, 32, 0, stream>>>(w + 1, w, (long long)limit_ns, mbarrier ? 1 : 0);
  return check_launch("timeout_probe_kernel");
}

}  // extern "C"
