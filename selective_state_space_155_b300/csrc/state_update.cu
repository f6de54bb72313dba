// Single-token decode step (selective_state_update) for sm_103a.
//
// One step of the recurrence on a stored float32 state, in place:
//   Delta = softplus(dt + dt_bias[d]);  s[n] <- exp(Delta A[d,n]) s[n] + Delta B[n] x
//   y = sum_n C[n] s[n] + D[d] x;  out = y * silu(z)
// (constant-memory inference from the previous state and the current input only).
//
// The step is bound by HBM: the state is read and written once (8 bytes per state element),
// everything else is small.  A channel's dstate floats are contiguous, so lanes take four states
// each along the state row (a warp moves 32 x 16 contiguous bytes per access) and the readout sum
// over n is a butterfly over the R = NPAD/4 lanes of a channel.  Each thread handles two such
// units, issuing all of their loads before any arithmetic, so that enough bytes are in flight to
// cover HBM latency at full bandwidth.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kBlock = 256;
constexpr int kItems = 2;

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 q = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
  v[0] = lo.x, v[1] = lo.y, v[2] = hi.x, v[3] = hi.y;
}

template <typename T, int NPAD, bool VEC>
__global__ void __launch_bounds__(kBlock) state_update_kernel(const UpdateArgs a) {
  constexpr int R = NPAD / 4;
  const long long nch = (long long)a.batch * a.dim;
  const long long lanes = nch * R;
  const long long stride = (long long)gridDim.x * kBlock;  // a multiple of 32: a channel's R lanes share a warp
  const int N = a.dstate;
  const T* __restrict__ gx = static_cast<const T*>(a.x);
  const T* __restrict__ gdt = static_cast<const T*>(a.dt);
  const T* __restrict__ gz = static_cast<const T*>(a.z);
  const T* __restrict__ gB = static_cast<const T*>(a.B);
  const T* __restrict__ gC = static_cast<const T*>(a.C);

  float s[kItems][4], Av[kItems][4], Bv[kItems][4], Cv[kItems][4], x[kItems], r[kItems], zz[kItems];
  bool ok[kItems];
  long long chs[kItems];
  int gs[kItems], ds[kItems];

  // all loads first
#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const long long unit = (long long)blockIdx.x * kBlock + threadIdx.x + it * stride;
    ok[it] = unit < lanes;
    const long long ch = ok[it] ? unit / R : 0;
    const int g = int(unit % R);
    const int b = int(ch / a.dim), d = int(ch % a.dim);
    chs[it] = ch, gs[it] = g, ds[it] = d;
    float* srow = a.state + ch * N + 4 * g;
#pragma unroll
    for (int i = 0; i < 4; ++i) s[it][i] = Av[it][i] = Bv[it][i] = Cv[it][i] = 0.0f;
    x[it] = r[it] = 0.0f;
    zz[it] = 0.0f;
    if (ok[it]) {
      if constexpr (VEC) {
        const float4 v = *reinterpret_cast<const float4*>(srow);
        s[it][0] = v.x, s[it][1] = v.y, s[it][2] = v.z, s[it][3] = v.w;
        const float4 q = __ldg(reinterpret_cast<const float4*>(a.A + size_t(d) * N + 4 * g));
        Av[it][0] = q.x, Av[it][1] = q.y, Av[it][2] = q.z, Av[it][3] = q.w;
        load4<T>(gB + size_t(b) * N + 4 * g, Bv[it]);
        load4<T>(gC + size_t(b) * N + 4 * g, Cv[it]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = 4 * g + i;
          if (n < N) {
            s[it][i] = srow[i];
            Av[it][i] = __ldg(a.A + size_t(d) * N + n);
            Bv[it][i] = to_f32<T>(gB[size_t(b) * N + n]);
            Cv[it][i] = to_f32<T>(gC[size_t(b) * N + n]);
          }
        }
      }
      x[it] = to_f32<T>(gx[ch]);
      r[it] = to_f32<T>(gdt[ch]);
      if (a.dt_bias) r[it] += __ldg(a.dt_bias + d);
      if (gz) zz[it] = to_f32<T>(gz[ch]);
    }
  }

#pragma unroll
  for (int it = 0; it < kItems; ++it) {
    const float step = a.softplus ? softplus_f32(r[it]) : r[it];
    const float dx = step * x[it];
    float part = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float abar = ex2_approx(step * (Av[it][i] * kLog2e));
      s[it][i] = fmaf(abar, s[it][i], dx * Bv[it][i]);
      part = fmaf(Cv[it][i], s[it][i], part);
    }
#pragma unroll
    for (int off = R / 2; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (ok[it]) {
      float* srow = a.state + chs[it] * N + 4 * gs[it];
      if constexpr (VEC) {
        *reinterpret_cast<float4*>(srow) = make_float4(s[it][0], s[it][1], s[it][2], s[it][3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (4 * gs[it] + i < N) srow[i] = s[it][i];
      }
      if (gs[it] == 0) {
        float y = part;
        if (a.D) y = fmaf(__ldg(a.D + ds[it]), x[it], y);
        if (gz) y *= silu_f32(zz[it]);
        static_cast<T*>(a.out)[chs[it]] = from_f32<T>(y);
      }
    }
  }
}

template <typename T, int NPAD>
cudaError_t launch_npad(const UpdateArgs& a, cudaStream_t stream) {
  constexpr int R = NPAD / 4;
  const long long lanes = (long long)a.batch * a.dim * R;
  const long long nblk = (lanes + kBlock * kItems - 1) / (kBlock * kItems);
  if (nblk <= 0) return cudaSuccess;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto al = [](const void* p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; };
  const uintptr_t bc_align = a.io == kF32 ? 16 : 8;
  const bool vec = a.dstate == NPAD && al(a.state, 16) && al(a.A, 16) && al(a.B, bc_align) && al(a.C, bc_align);
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
