// Single-token decode step (selective_state_update) for sm_103a.
//
// One step of the recurrence on a stored float32 state, in place:
//   Delta = softplus(dt + dt_bias[d]);  s[n] <- exp(Delta A[d,n]) s[n] + Delta B[n] x
//   y = sum_n C[n] s[n] + D[d] x;  out = y * silu(z)
// (constant-memory inference from the previous state and the current input only).
//
// The step is bound by HBM: the state is read and written once (8 bytes per state element),
// everything else is small.  A channel's dstate floats are contiguous, so lanes are laid out
// four states each along the state row: a warp streams 32 x 16 contiguous bytes per access,
// and the readout sum over n is a butterfly over the R = NPAD/4 lanes of a channel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kBlock = 256;

template <typename T, int NPAD, bool VEC>
__global__ void __launch_bounds__(kBlock) state_update_kernel(const UpdateArgs a) {
  constexpr int R = NPAD / 4;
  const long long gid = (long long)blockIdx.x * kBlock + threadIdx.x;
  const long long nch = (long long)a.batch * a.dim;
  const long long ch = gid / R;
  const int g = int(gid % R);
  const bool ok = ch < nch;  // out-of-range lanes still take part in the shuffles below
  const long long chc = ok ? ch : 0;
  const int b = int(chc / a.dim), d = int(chc % a.dim);
  const int N = a.dstate;

  const T* __restrict__ gx = static_cast<const T*>(a.x);
  const T* __restrict__ gdt = static_cast<const T*>(a.dt);
  const T* __restrict__ gB = static_cast<const T*>(a.B);
  const T* __restrict__ gC = static_cast<const T*>(a.C);

  float s[4] = {0.f, 0.f, 0.f, 0.f};
  float* srow = a.state + chc * N + 4 * g;
  if (ok) {
    if constexpr (VEC) {
      const float4 v = *reinterpret_cast<const float4*>(srow);
      s[0] = v.x, s[1] = v.y, s[2] = v.z, s[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * g + i < N) s[i] = srow[i];
    }
  }
  float x = 0.f, step = 0.f;
  if (ok) {
    x = to_f32<T>(gx[chc]);
    float r = to_f32<T>(gdt[chc]);
    if (a.dt_bias) r += a.dt_bias[d];
    step = a.softplus ? softplus_f32(r) : r;
  }
  const float dx = step * x;
  float part = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = 4 * g + i;
    if (ok && n < N) {
      const float abar = ex2_approx(step * (a.A[size_t(d) * N + n] * kLog2e));
      s[i] = fmaf(abar, s[i], dx * to_f32<T>(gB[size_t(b) * N + n]));
      part = fmaf(to_f32<T>(gC[size_t(b) * N + n]), s[i], part);
    }
  }
#pragma unroll
  for (int off = R / 2; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
  if (ok) {
    if constexpr (VEC) {
      *reinterpret_cast<float4*>(srow) = make_float4(s[0], s[1], s[2], s[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * g + i < N) srow[i] = s[i];
    }
    if (g == 0) {
      float y = part;
      if (a.D) y = fmaf(a.D[d], x, y);
      if (a.z) y *= silu_f32(to_f32<T>(static_cast<const T*>(a.z)[chc]));
      static_cast<T*>(a.out)[chc] = from_f32<T>(y);
    }
  }
}

template <typename T, int NPAD>
cudaError_t launch_npad(const UpdateArgs& a, cudaStream_t stream) {
  constexpr int R = NPAD / 4;
  const long long threads = (long long)a.batch * a.dim * R;
  const long long nblk = (threads + kBlock - 1) / kBlock;
  if (nblk <= 0) return cudaSuccess;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const bool vec = a.dstate == NPAD && (reinterpret_cast<uintptr_t>(a.state) & 15u) == 0;
  UpdateArgs args = a;
  void* params[] = {&args};
  const void* fn = vec ? reinterpret_cast<const void*>(state_update_kernel<T, NPAD, true>)
                       : reinterpret_cast<const void*>(state_update_kernel<T, NPAD, false>);
  return cudaLaunchKernel(fn, dim3(unsigned(nblk)), dim3(kBlock), params, 0, stream);
}

template <typename T>
cudaError_t dispatch(const UpdateArgs& a, cudaStream_t stream) {
  if (a.dstate <= 4) return launch_npad<T, 4>(a, stream);
  if (a.dstate <= 8) return launch_npad<T, 8>(a, stream);
  return launch_npad<T, 16>(a, stream);
}

}  // namespace

cudaError_t launch_state_update(const UpdateArgs& a, cudaStream_t stream) {
  return a.io == kF32 ? dispatch<float>(a, stream) : dispatch<__nv_bfloat16>(a, stream);
}

}  // namespace ssm
