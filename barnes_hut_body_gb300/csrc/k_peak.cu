// fp32 throughput probe: the denominator of the roofline of the walk and
// direct-sum kernels, which are bound by fp32 arithmetic, not by memory.
//
// Every thread runs 8 independent chains x <- x*b + c (b, c kernel
// arguments, so nothing folds) with no memory access inside the loop; 8
// chains per thread and 64 warps per SM hide the FMA latency many times
// over, so the launch measures the issue rate of the FMA pipe alone.  Two
// forms: scalar fma.rn.f32 (one lane-FMA per thread and instruction) and
// Blackwell's packed fma.rn.f32x2 (two per instruction), the form the
// interaction loops use.  The chains' sum is stored only when the runtime
// flag `write` is set, which the host never sets: the compiler must keep
// every FMA, and the launch writes no memory.
#include <cuda_runtime.h>

#include "bh_internal.h"

namespace bh {

namespace {

constexpr int kPeakThreads = 256;
constexpr int kPeakChains = 8;

template <bool kPacked>
__global__ void __launch_bounds__(kPeakThreads)
fma_peak_kernel(int iters, float b, float c, int write, float *sink, int nsink) {
  const int tid = blockIdx.x * kPeakThreads + threadIdx.x;
  float s = 0.f;
  if constexpr (kPacked) {
    f2 x[kPeakChains];
    const f2 b2 = pk(b, b), c2 = pk(c, c);
#pragma unroll
    for (int k = 0; k < kPeakChains; ++k)
      x[k] = pk(1e-3f * (float)(threadIdx.x + k), 2e-3f * (float)(threadIdx.x + k));
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < kPeakChains; ++k) x[k] = fma2(x[k], b2, c2);
    }
#pragma unroll
    for (int k = 0; k < kPeakChains; ++k) {
      float lo, hi;
      upk(x[k], lo, hi);
      s += lo + hi;
    }
  } else {
    float x[kPeakChains];
#pragma unroll
    for (int k = 0; k < kPeakChains; ++k) x[k] = 1e-3f * (float)(threadIdx.x + k);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int k = 0; k < kPeakChains; ++k) x[k] = __fmaf_rn(x[k], b, c);
    }
#pragma unroll
    for (int k = 0; k < kPeakChains; ++k) s += x[k];
  }
  if (write) sink[tid % nsink] = s;
}

}  // namespace

long long fma_probe_flops(bool packed, int iters, int num_sms) {
  const long long blocks = (long long)num_sms * (2048 / kPeakThreads);
  return blocks * kPeakThreads * (long long)iters * kPeakChains * (packed ? 2 : 1) * 2;
}

cudaError_t launch_fma_probe(bool packed, int iters, int num_sms, float *sink,
                             int nsink, cudaStream_t s) {
  // 8 blocks of 256 threads per SM: 2048 resident threads, a full SM
  const int blocks = num_sms * (2048 / kPeakThreads);
  // b < 1 keeps every chain bounded (it converges to c / (1 - b))
  const float b = 0.999f, c = 1e-4f;
  if (packed)
    fma_peak_kernel<true><<<blocks, kPeakThreads, 0, s>>>(iters, b, c, 0, sink, nsink);
  else
    fma_peak_kernel<false><<<blocks, kPeakThreads, 0, s>>>(iters, b, c, 0, sink, nsink);
  return cudaGetLastError();
}

}  // namespace bh
