// Throughput probes for the units the scan leans on: the special-function unit (ex2.approx, the
// exponential of every state step), scalar FP32 fused multiply-add, and the packed f32x2 form.
// One CTA of 512 threads per SM runs a fixed number of iterations of independent dependency
// chains (enough in flight to cover each unit's latency); thread 0 of each CTA records the clock
// cycles between two CTA barriers around the loop.  operations / cycles is the per-SM rate, which
// the benchmark uses as the peak of its special-function roofline instead of a datasheet figure.
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kChains = 8;  // independent chains per thread
constexpr int kIters = 4096;

enum ProbeKind { kMufuEx2 = 0, kFfma = 1, kFfma2 = 2 };

template <int KIND>
__global__ void __launch_bounds__(kProbeThreads) probe_kernel(long long* cycles) {
  float x[kChains];
  float2 x2[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) {
    x[c] = 0.25f + 0.01f * float(threadIdx.x % 7 + c);
    x2[c] = make_float2(x[c], x[c] + 0.5f);
  }
  __syncthreads();
  const long long t0 = clock64();
#pragma unroll 4
  for (int i = 0; i < kIters; ++i) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      if constexpr (KIND == kMufuEx2) {
        x[c] = ex2_approx(-x[c]);  // converges to a fixed point in (0, 1)
      } else if constexpr (KIND == kFfma) {
        x[c] = fmaf(x[c], 0.999f, 0.0005f);
      } else {
        x2[c] = __ffma2_rn(x2[c], make_float2(0.999f, 0.999f), make_float2(0.0005f, 0.0005f));
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float acc = 0.0f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) acc += x[c] + x2[c].x + x2[c].y;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
  if (acc == 1234.5f) cycles[blockIdx.x] = -1;  // never true; keeps the chains alive
}

}  // namespace

cudaError_t launch_probe(int kind, int nblocks, long long* cycles, cudaStream_t stream) {
  void* params[] = {&cycles};
  const void* fn = kind == kMufuEx2 ? reinterpret_cast<const void*>(probe_kernel<kMufuEx2>)
                   : kind == kFfma  ? reinterpret_cast<const void*>(probe_kernel<kFfma>)
                                    : reinterpret_cast<const void*>(probe_kernel<kFfma2>);
  return cudaLaunchKernel(fn, dim3(unsigned(nblocks)), dim3(kProbeThreads), params, 0, stream);
}

// Lane-operations one CTA issues in one probe launch (an f32x2 operation counts as two).
double probe_ops_per_cta(int kind) {
  return double(kProbeThreads) * kIters * kChains * (kind == kFfma2 ? 2.0 : 1.0);
}

}  // namespace ssm
