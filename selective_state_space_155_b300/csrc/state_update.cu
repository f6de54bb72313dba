// Single-token decode step (selective_state_update) for sm_103a.
//
// One step of the recurrence on a stored float32 state, in place:
//   Delta = softplus(dt + dt_bias[d]);  s[n] <- exp(Delta A[d,n]) s[n] + Delta B[n] x
//   (or, with the exact zero-order hold, (exp(Delta A[d,n]) - 1) / A[d,n] B[n] x in place of Delta B[n] x)
//   y = sum_n C[n] s[n] + D[d] x;  out = y * silu(z)
// (constant-memory inference from the previous state and the current input only).
//
// The step is bound by HBM: the float32 state is read and written once (8 bytes per state
// element), everything else is small.  One thread owns one (batch, channel) and all NPAD of its
// states, so the per-channel work (softplus, silu, the readout sum) is done once, with no
// cross-lane traffic, and each thread keeps NPAD*4 bytes of state in flight (four 16-byte loads
// issued back to back for dstate 16).  A, B and C rows are small and shared (A by every batch row,
// B and C by every channel of a batch row), so they come from L1/L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kBlock = 128;

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

// NPAD consecutive io values (16-byte aligned) as float32
template <typename T, int NPAD>
__device__ __forceinline__ void load_row(const T* p, float (&v)[NPAD]) {
  if constexpr (std::is_same<T, float>::value) {
#pragma unroll
    for (int i = 0; i < NPAD; i += 4) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p + i));
      v[i] = q.x, v[i + 1] = q.y, v[i + 2] = q.z, v[i + 3] = q.w;
    }
  } else if constexpr (NPAD >= 8) {
#pragma unroll
    for (int i = 0; i < NPAD; i += 8) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(p + i));
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        v[i + 2 * k] = f.x, v[i + 2 * k + 1] = f.y;
      }
    }
  } else {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
    v[0] = lo.x, v[1] = lo.y, v[2] = hi.x, v[3] = hi.y;
  }
}

template <typename T, int NPAD, bool VEC>
__global__ void __launch_bounds__(kBlock) state_update_kernel(const UpdateArgs a) {
  const long long ch = (long long)blockIdx.x * kBlock + threadIdx.x;
  if (ch >= (long long)a.batch * a.dim) return;
  // (b, d) = divmod(ch, dim): the multiply-shift division below 2^32 channels
  const long long bq = ch < (1LL << 32) ? (long long)fast_div(uint32_t(ch), a.div_dim) : ch / a.dim;
  const int b = int(bq), d = int(ch - bq * a.dim);
  const int N = a.dstate;
  float* srow = a.state + ch * N;
  const float* Arow = a.A + size_t(d) * N;
  const T* Brow = static_cast<const T*>(a.B) + size_t(b) * N;
  const T* Crow = static_cast<const T*>(a.C) + size_t(b) * N;

  // loads first: the state (the HBM stream), then the small operands
  float s[NPAD], Av[NPAD], Bv[NPAD], Cv[NPAD];
  if constexpr (VEC) {
#pragma unroll
    for (int i = 0; i < NPAD; i += 4) {
      const float4 q = *reinterpret_cast<const float4*>(srow + i);
      s[i] = q.x, s[i + 1] = q.y, s[i + 2] = q.z, s[i + 3] = q.w;
    }
    load_row<float, NPAD>(Arow, Av);
    load_row<T, NPAD>(Brow, Bv);
    load_row<T, NPAD>(Crow, Cv);
  } else {
#pragma unroll
    for (int i = 0; i < NPAD; ++i) {
      const bool ok = i < N;
      s[i] = ok ? srow[i] : 0.0f;
      Av[i] = ok ? __ldg(Arow + i) : 0.0f;
      Bv[i] = ok ? to_f32<T>(Brow[i]) : 0.0f;
      Cv[i] = ok ? to_f32<T>(Crow[i]) : 0.0f;
    }
  }
  const float x = to_f32<T>(static_cast<const T*>(a.x)[ch]);
  float r = to_f32<T>(static_cast<const T*>(a.dt)[ch]);
  if (a.dt_bias) r += __ldg(a.dt_bias + d);
  const float zz = a.z ? to_f32<T>(static_cast<const T*>(a.z)[ch]) : 0.0f;
  const float Dd = a.D ? __ldg(a.D + d) : 0.0f;

  const float step = a.softplus ? softplus_f32(r) : r;
  const float2 dd = f2(step * kLog2e, step * kLog2e), dx = f2(step * x, step * x);
  float2 acc = f2(0.0f, 0.0f);
  if (a.zoh) {
    const float2 sd = f2(step, step), xx = f2(x, x);
#pragma unroll
    for (int i = 0; i < NPAD; i += 2) {
      const float2 Ai = f2(Av[i], Av[i + 1]);
      const float2 g = __fmul2_rn(dd, Ai);
      const float2 ab = f2(ex2_approx(g.x), ex2_approx(g.y));
      const float2 c = zoh_factor2(__fmul2_rn(sd, Ai), ab, sd, f2(zoh_inv(Ai.x), zoh_inv(Ai.y)));
      const float2 sn = __ffma2_rn(ab, f2(s[i], s[i + 1]), __fmul2_rn(c, __fmul2_rn(xx, f2(Bv[i], Bv[i + 1]))));
      s[i] = sn.x, s[i + 1] = sn.y;
      acc = __ffma2_rn(f2(Cv[i], Cv[i + 1]), sn, acc);
    }
  } else {
#pragma unroll
    for (int i = 0; i < NPAD; i += 2) {
      const float2 g = __fmul2_rn(dd, f2(Av[i], Av[i + 1]));
      const float2 ab = f2(ex2_approx(g.x), ex2_approx(g.y));
      const float2 sn = __ffma2_rn(ab, f2(s[i], s[i + 1]), __fmul2_rn(dx, f2(Bv[i], Bv[i + 1])));
      s[i] = sn.x, s[i + 1] = sn.y;
      acc = __ffma2_rn(f2(Cv[i], Cv[i + 1]), sn, acc);
    }
  }
  float y = fmaf(Dd, x, acc.x + acc.y);
  if (a.z) y *= silu_f32(zz);
  static_cast<T*>(a.out)[ch] = from_f32<T>(y);

  if constexpr (VEC) {
#pragma unroll
    for (int i = 0; i < NPAD; i += 4)
      *reinterpret_cast<float4*>(srow + i) = make_float4(s[i], s[i + 1], s[i + 2], s[i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < NPAD; ++i)
      if (i < N) srow[i] = s[i];
  }
}

template <typename T, int NPAD>
cudaError_t launch_npad(const UpdateArgs& a, cudaStream_t stream) {
  const long long nch = (long long)a.batch * a.dim;
  const long long nblk = (nch + kBlock - 1) / kBlock;
  if (nblk <= 0) return cudaSuccess;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  // vector rows: every row starts 16-byte aligned (dstate == NPAD) and the bf16 B/C rows are whole
  // 16-byte (NPAD >= 8) or 8-byte (NPAD == 4) pieces
  const bool bc_ok = a.io == kF32 ? (al(a.B) && al(a.C))
                                  : (NPAD >= 8 ? (al(a.B) && al(a.C))
                                               : ((reinterpret_cast<uintptr_t>(a.B) & 7u) == 0 &&
                                                  (reinterpret_cast<uintptr_t>(a.C) & 7u) == 0));
  const bool vec = a.dstate == NPAD && al(a.state) && al(a.A) && bc_ok;
  UpdateArgs args = a;
  args.div_dim = make_fastdiv(uint32_t(a.dim));
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
