// Throughput probes for the units the scan leans on: the special-function unit (ex2.approx, the
// exponential of every state step), scalar FP32 fused multiply-add, the packed f32x2 form, and two
// mixes that show how the special-function and FP32 pipes share one SM when both are busy.
// One CTA of 512 threads per SM runs a fixed number of iterations of independent dependency
// chains (enough in flight to cover each unit's latency); thread 0 of each CTA records the clock
// cycles between two CTA barriers around the loop.  operations / cycles is the per-SM rate, which
// the benchmark uses as the peak of its special-function roofline instead of a datasheet figure.
//
// The mixes:
//  * kEx2Ffma2: per chain and iteration one ex2 and one independent packed f32x2 FMA (2 FP32
//    lane-operations), i.e. the special-function unit and the FP32 pipe loaded at their nominal
//    1 : 4 rate ratio.  Counted in ex2 operations; if the two pipes overlap fully it runs at the
//    ex2-alone rate.
//  * kRecurrence: the scan's own per-state work on a pair of states, as the forward kernel issues
//    it: x = Delta*A (f32x2 multiply), two ex2, b = (Delta*u)*B (f32x2 multiply),
//    h = Abar*h + b (f32x2 FMA), y += C*h (f32x2 FMA).  Counted in state-steps (two per pair and
//    iteration), so cycles / state-step is the recurrence's arithmetic floor on this SM.
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kChains = 8;  // independent chains per thread
constexpr int kIters = 4096;

enum ProbeKind { kMufuEx2 = 0, kFfma = 1, kFfma2 = 2, kEx2Ffma2 = 3, kRecurrence = 4, kWaitTimeout = 5 };

// The forward kernels' bounded barrier wait (mbar_wait) on a barrier that nothing arrives on: one
// warp per CTA waits with a limit of 2^20 cycles and must give up; thread 0 writes the cycles the
// wait took, or -1 if it completed.
constexpr long long kProbeWaitLimit = 1LL << 20;
__global__ void __launch_bounds__(32) probe_wait_kernel(long long* cycles) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  __shared__ unsigned long long gave_up;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    gave_up = 0;
  }
  __syncthreads();
  const long long t0 = clock64();
  const bool done = mbar_wait(&bar, 0, &abort_flag, kProbeWaitLimit, &gave_up, 256);
  const long long t1 = clock64();
  __syncthreads();
  if (threadIdx.x == 0) cycles[blockIdx.x] = (done || gave_up == 0) ? -1 : t1 - t0;
}

template <int KIND>
__global__ void __launch_bounds__(kProbeThreads) probe_kernel(long long* cycles) {
  float x[kChains];
  float2 x2[kChains];
  float2 acc[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) {
    x[c] = 0.25f + 0.01f * float(threadIdx.x % 7 + c);
    x2[c] = make_float2(x[c], x[c] + 0.5f);
    acc[c] = make_float2(0.0f, 0.0f);
  }
  // Per-chain operands of the recurrence mix, kept in registers as the scan keeps A, B and C; they
  // differ per chain so that no two chains compute the same values.
  float2 dA[kChains], uB[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) {
    dA[c] = make_float2(-0.03f - 0.001f * float(c + (threadIdx.x & 3)), -0.05f - 0.002f * float(c));
    uB[c] = make_float2(0.002f + 0.0001f * float(c), 0.003f + 0.0001f * float(threadIdx.x & 1));
  }
  const float2 Cv = make_float2(0.5f, -0.25f);
  const int dbits = __float_as_int(0.02f) + int(threadIdx.x & 7);
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
      } else if constexpr (KIND == kFfma2) {
        x2[c] = __ffma2_rn(x2[c], make_float2(0.999f, 0.999f), make_float2(0.0005f, 0.0005f));
      } else if constexpr (KIND == kEx2Ffma2) {
        x[c] = ex2_approx(-x[c]);
        x2[c] = __ffma2_rn(x2[c], make_float2(0.999f, 0.999f), make_float2(0.0005f, 0.0005f));
      } else {
        // Delta (duplicated in both halves, as the kernel reads it from its step table) changes
        // every step by integer arithmetic only, so the FP32 pipe carries just the recurrence
        const int di = dbits + (i & 255);
        const float2 d = make_float2(__int_as_float(di), __int_as_float(di));
        const float2 g = __fmul2_rn(d, dA[c]);
        const float2 a = make_float2(ex2_approx(g.x), ex2_approx(g.y));
        const float2 b = __fmul2_rn(d, uB[c]);
        x2[c] = __ffma2_rn(a, x2[c], b);
        acc[c] = __ffma2_rn(Cv, x2[c], acc[c]);
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += x[c] + x2[c].x + x2[c].y + acc[c].x + acc[c].y;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
  if (s == 1234.5f) cycles[blockIdx.x] = -1;  // never true; keeps the chains alive
}

template <int KIND>
const void* probe_fn() {
  return reinterpret_cast<const void*>(probe_kernel<KIND>);
}

}  // namespace

cudaError_t launch_probe(int kind, int nblocks, long long* cycles, cudaStream_t stream) {
  void* params[] = {&cycles};
  if (kind == kWaitTimeout)
    return cudaLaunchKernel(reinterpret_cast<const void*>(probe_wait_kernel), dim3(unsigned(nblocks)), dim3(32),
                            params, 0, stream);
  const void* fn = kind == kMufuEx2    ? probe_fn<kMufuEx2>()
                   : kind == kFfma     ? probe_fn<kFfma>()
                   : kind == kFfma2    ? probe_fn<kFfma2>()
                   : kind == kEx2Ffma2 ? probe_fn<kEx2Ffma2>()
                                       : probe_fn<kRecurrence>();
  return cudaLaunchKernel(fn, dim3(unsigned(nblocks)), dim3(kProbeThreads), params, 0, stream);
}

// Operations one CTA performs in one probe launch: lane-operations for the single-unit kinds (an
// f32x2 operation counts as two), ex2 operations for the ex2 + f32x2 mix, state-steps for the
// recurrence mix; 0 for the bounded-wait probe.
double probe_ops_per_cta(int kind) {
  if (kind == kWaitTimeout) return 0.0;
  const double per = kind == kFfma2 ? 2.0 : kind == kRecurrence ? 2.0 : 1.0;
  return double(kProbeThreads) * kIters * kChains * per;
}

}  // namespace ssm
