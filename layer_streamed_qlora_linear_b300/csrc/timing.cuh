// Optional CUDA-event timing of libsl's launches (sl_kernel_timing).
#pragma once
#include "common.cuh"

namespace sl {

// Variants: 0..5 tensor-core GEMMs (see sl_kernel_timing), 6 rank-r T = X A^T,
// 7 rank-r U = dY B, 8 rank-r dA / dB, 9 attention forward, 10 attention
// backward (all of its kernels).
constexpr int kNumTimedVariants = 11;

struct TimingToken {
  cudaEvent_t start = nullptr, stop = nullptr;
  int variant = 0;
  double work = 0.0;  // algorithmic FLOPs (GEMMs) or bytes (rank-r passes)
  // GEMMs: the launch's device-clock slot {first start, last end} in %globaltimer
  // ns, which the kernel fills itself (nullptr when not timing)
  unsigned long long* clk = nullptr;
};

// No-ops (null events) unless timing is enabled.
TimingToken timing_begin(int variant, double work, cudaStream_t stream);
void timing_end(const TimingToken& t, cudaStream_t stream);

}  // namespace sl
