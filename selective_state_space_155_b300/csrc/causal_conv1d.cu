// Causal depthwise conv1d (width W <= 4) with bias and optional silu: the step of the Mamba block
// that produces the scan's input u.  For every (batch b, channel d, step t):
//   out_t = act(bias[d] + sum_k w[d,k] * x_{t-(W-1)+k}),   x_{-1}, x_{-2}, ... from state_in
// and state_out = the W-1 last inputs of concat(state_in, x), so that a long row can be streamed
// in pieces.  The decode form applies the same filter to one new input and shifts the state.
//
// The op moves 2 x io bytes per element and does W multiply-adds: it is bound by HBM.  The
// sequence layout is [batch][dim][seqlen] (time innermost), so one thread takes 16 contiguous
// bytes of one row (8 bf16 or 4 float32 steps) at a time, loads them with one 16-byte load, gets
// the W-1 inputs before them from the previous lane by a shuffle (the first vector of a row takes
// them from state_in, the first lane of a warp from global memory, where its neighbour's load has
// just put them in L1), and writes its 16 bytes of output with one store; two such vectors per
// thread, loads first.  Rows whose length or base is not 16-byte aligned take a
// one-element-per-thread form of the same arithmetic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kThreads = 256;

template <typename T>
struct Vec16;  // 16 bytes of io elements as float32
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      v[2 * k] = f.x, v[2 * k + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
      w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

__device__ __forceinline__ float act(float v, bool silu) { return silu ? silu_f32(v) : v; }

// q = n / f.d and r = n % f.d: the multiply-shift division while n fits in 32 bits (every tensor
// below 2^32 work items), a 64-bit division beyond.
__device__ __forceinline__ void divmod(long long n, const FastDiv& f, long long& q, long long& r) {
  if (n < (1LL << 32)) {
    q = fast_div(uint32_t(n), f);
  } else {
    q = n / (long long)f.d;
  }
  r = n - q * (long long)f.d;
}

// Each thread takes K vectors of 16 bytes, kThreads apart, so that consecutive lanes hold
// consecutive vectors; all K loads are issued before any arithmetic to keep enough bytes in
// flight.  Every row is 16-byte aligned and a whole number of vectors, so vector v starts at
// element v*E of the flattened [batch*dim][seqlen] tensor.
constexpr int kVecPerThread = 2;

template <typename T, int W>
__global__ void __launch_bounds__(kThreads) conv_vec_kernel(const ConvArgs a) {
  constexpr int E = Vec16<T>::N, H = W - 1, K = kVecPerThread;
  const long long vpr = a.seqlen / E;
  const long long nvec = (long long)a.batch * a.dim * vpr;
  const long long base = (long long)blockIdx.x * kThreads * K + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const T* x = static_cast<const T*>(a.x);

  float xv[K][E];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const long long v = base + (long long)i * kThreads;
#pragma unroll
    for (int e = 0; e < E; ++e) xv[i][e] = 0.0f;
    if (v < nvec) Vec16<T>::load(x + v * E, xv[i]);
  }
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const long long v = base + (long long)i * kThreads;
    const bool active = v < nvec;
    // the H inputs before xv[i][0]: the previous lane's last ones, unless this vector starts a
    // row (state_in) or a warp (global memory)
    float hl[H > 0 ? H : 1];
#pragma unroll
    for (int h = 0; h < H; ++h) hl[h] = __shfl_up_sync(0xffffffffu, xv[i][E - H + h], 1);
    if (!active) continue;
    long long row, j, dq, dr;
    divmod(v, a.div_row, row, j);
    if (j == 0) {
      const T* si = static_cast<const T*>(a.state_in);
#pragma unroll
      for (int h = 0; h < H; ++h) hl[h] = si ? to_f32<T>(si[row * H + h]) : 0.0f;
    } else if (lane == 0) {
#pragma unroll
      for (int h = 0; h < H; ++h) hl[h] = to_f32<T>(x[v * E - H + h]);
    }
    divmod(row, a.div_dim, dq, dr);
    const int d = int(dr);
    float w[W];
#pragma unroll
    for (int k = 0; k < W; ++k) w[k] = __ldg(a.weight + (size_t)d * W + k);
    const float bias = a.bias ? __ldg(a.bias + d) : 0.0f;
    float ov[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float acc = bias;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const int s = e - H + k;  // position relative to xv[i][0]
        acc = fmaf(w[k], s >= 0 ? xv[i][s] : hl[H + s], acc);
      }
      ov[e] = act(acc, a.silu != 0);
    }
    Vec16<T>::store(static_cast<T*>(a.out) + v * E, ov);
    if (a.state_out && j == vpr - 1) {
      T* so = static_cast<T*>(a.state_out);
#pragma unroll
      for (int h = 0; h < H; ++h) so[row * H + h] = from_f32<T>(xv[i][E - H + h]);
    }
  }
}

// Rows of an even number of vectors: each thread takes two consecutive vectors of one row (32
// contiguous bytes), so the channel's filter is loaded once and the second vector's W-1 earlier
// inputs are the first vector's last ones; only the first vector needs the previous lane.
template <typename T, int W>
__global__ void __launch_bounds__(kThreads) conv_pair_kernel(const ConvArgs a) {
  constexpr int E = Vec16<T>::N, H = W - 1;
  const long long vpr = a.seqlen / E;  // even
  const long long npair = (long long)a.batch * a.dim * (vpr / 2);
  const long long pidx = (long long)blockIdx.x * kThreads + threadIdx.x;
  const bool active = pidx < npair;
  const long long v = 2 * pidx;  // first vector; v + 1 is in the same row
  const int lane = threadIdx.x & 31;
  const T* x = static_cast<const T*>(a.x);

  float xv[2][E];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) xv[i][e] = 0.0f;
  if (active) {
    Vec16<T>::load(x + v * E, xv[0]);
    Vec16<T>::load(x + (v + 1) * E, xv[1]);
  }
  float hl[H > 0 ? H : 1];
#pragma unroll
  for (int h = 0; h < H; ++h) hl[h] = __shfl_up_sync(0xffffffffu, xv[1][E - H + h], 1);
  if (!active) return;
  long long row, j, dq, dr;
  divmod(v, a.div_row, row, j);  // div_row divides by vpr here
  if (j == 0) {
    const T* si = static_cast<const T*>(a.state_in);
#pragma unroll
    for (int h = 0; h < H; ++h) hl[h] = si ? to_f32<T>(si[row * H + h]) : 0.0f;
  } else if (lane == 0) {
#pragma unroll
    for (int h = 0; h < H; ++h) hl[h] = to_f32<T>(x[v * E - H + h]);
  }
  divmod(row, a.div_dim, dq, dr);
  const int d = int(dr);
  float w[W];
#pragma unroll
  for (int k = 0; k < W; ++k) w[k] = __ldg(a.weight + (size_t)d * W + k);
  const float bias = a.bias ? __ldg(a.bias + d) : 0.0f;
  const bool silu = a.silu != 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float ov[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      float acc = bias;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const int s = e - H + k;  // position relative to xv[i][0]
        const float in = s >= 0 ? xv[i][s] : (i == 0 ? hl[H + s] : xv[0][E + s]);
        acc = fmaf(w[k], in, acc);
      }
      ov[e] = act(acc, silu);
    }
    Vec16<T>::store(static_cast<T*>(a.out) + (v + i) * E, ov);
  }
  if (a.state_out && j + 2 == vpr) {
    T* so = static_cast<T*>(a.state_out);
#pragma unroll
    for (int h = 0; h < H; ++h) so[row * H + h] = from_f32<T>(xv[1][E - H + h]);
  }
}

// One thread per output element, then one per state slot (rows x H items after the outputs).
template <typename T, int W>
__global__ void __launch_bounds__(kThreads) conv_scalar_kernel(const ConvArgs a) {
  constexpr int H = W - 1;
  const long long rows = (long long)a.batch * a.dim;
  const long long nout = rows * a.seqlen;
  const long long e = (long long)blockIdx.x * kThreads + threadIdx.x;
  const T* x = static_cast<const T*>(a.x);
  const T* si = static_cast<const T*>(a.state_in);
  // input at time s (< seqlen) of row r: the row itself, or the carried state before t = 0
  auto in = [&](long long r, long long s) -> float {
    if (s >= 0) return to_f32<T>(x[r * a.seqlen + s]);
    return si ? to_f32<T>(si[r * H + H + s]) : 0.0f;
  };
  if (e < nout) {
    long long r, t, dq, dr;
    divmod(e, a.div_row, r, t);
    divmod(r, a.div_dim, dq, dr);
    const int d = int(dr);
    float acc = a.bias ? __ldg(a.bias + d) : 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k) acc = fmaf(__ldg(a.weight + (size_t)d * W + k), in(r, t - H + k), acc);
    static_cast<T*>(a.out)[e] = from_f32<T>(act(acc, a.silu != 0));
  } else if (H > 0 && a.state_out && e < nout + rows * H) {
    const long long q = e - nout, r = q / (H > 0 ? H : 1), i = q % (H > 0 ? H : 1);
    static_cast<T*>(a.state_out)[r * H + i] = from_f32<T>(in(r, a.seqlen - H + i));
  }
}

// Decode step: out = act(bias + sum_{k<H} w[k] state[k] + w[H] x); state <- (state[1..], x).
template <typename T, int W>
__global__ void __launch_bounds__(kThreads) conv_update_kernel(const ConvUpdateArgs a) {
  constexpr int H = W - 1;
  const long long ch = (long long)blockIdx.x * kThreads + threadIdx.x;
  if (ch >= (long long)a.batch * a.dim) return;
  long long bq, dr;
  divmod(ch, a.div_dim, bq, dr);
  const int d = int(dr);
  T* st = static_cast<T*>(a.state);
  float s[H > 0 ? H : 1];
#pragma unroll
  for (int i = 0; i < H; ++i) s[i] = to_f32<T>(st[ch * H + i]);
  const float xv = to_f32<T>(static_cast<const T*>(a.x)[ch]);
  float acc = a.bias ? __ldg(a.bias + d) : 0.0f;
#pragma unroll
  for (int k = 0; k < H; ++k) acc = fmaf(__ldg(a.weight + (size_t)d * W + k), s[k], acc);
  acc = fmaf(__ldg(a.weight + (size_t)d * W + H), xv, acc);
  static_cast<T*>(a.out)[ch] = from_f32<T>(act(acc, a.silu != 0));
#pragma unroll
  for (int i = 0; i < H; ++i) st[ch * H + i] = from_f32<T>(i + 1 < H ? s[i + 1] : xv);
}

template <typename T, int W>
cudaError_t launch_fwd(const ConvArgs& a, bool vec, cudaStream_t stream) {
  const long long rows = (long long)a.batch * a.dim;
  constexpr int E = 16 / sizeof(T);
  const long long vpr = a.seqlen / E;
  const bool pair = vec && vpr % 2 == 0;
  const long long items = vec ? rows * vpr : rows * a.seqlen + (a.state_out ? rows * (W - 1) : 0);
  if (items <= 0) return cudaSuccess;
  const long long per_block = pair ? 2LL * kThreads : (vec ? (long long)kThreads * kVecPerThread : kThreads);
  const long long nblk = (items + per_block - 1) / per_block;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ConvArgs args = a;
  args.div_row = make_fastdiv(uint32_t(vec ? a.seqlen / E : (a.seqlen > 0 ? a.seqlen : 1)));
  args.div_dim = make_fastdiv(uint32_t(a.dim));
  void* params[] = {&args};
  const void* fn = pair  ? reinterpret_cast<const void*>(conv_pair_kernel<T, W>)
                   : vec ? reinterpret_cast<const void*>(conv_vec_kernel<T, W>)
                         : reinterpret_cast<const void*>(conv_scalar_kernel<T, W>);
  return cudaLaunchKernel(fn, dim3(unsigned(nblk)), dim3(kThreads), params, 0, stream);
}

template <typename T>
cudaError_t dispatch_fwd(const ConvArgs& a, cudaStream_t stream) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec = a.seqlen > 0 && (size_t(a.seqlen) * sizeof(T)) % 16 == 0 && al(a.x) && al(a.out);
  switch (a.width) {
    case 1: return launch_fwd<T, 1>(a, vec, stream);
    case 2: return launch_fwd<T, 2>(a, vec, stream);
    case 3: return launch_fwd<T, 3>(a, vec, stream);
    default: return launch_fwd<T, 4>(a, vec, stream);
  }
}

template <typename T, int W>
cudaError_t launch_update(const ConvUpdateArgs& a, cudaStream_t stream) {
  const long long nblk = ((long long)a.batch * a.dim + kThreads - 1) / kThreads;
  if (nblk <= 0) return cudaSuccess;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ConvUpdateArgs args = a;
  args.div_dim = make_fastdiv(uint32_t(a.dim));
  void* params[] = {&args};
  return cudaLaunchKernel(reinterpret_cast<const void*>(conv_update_kernel<T, W>), dim3(unsigned(nblk)),
                          dim3(kThreads), params, 0, stream);
}

template <typename T>
cudaError_t dispatch_update(const ConvUpdateArgs& a, cudaStream_t stream) {
  switch (a.width) {
    case 1: return launch_update<T, 1>(a, stream);
    case 2: return launch_update<T, 2>(a, stream);
    case 3: return launch_update<T, 3>(a, stream);
    default: return launch_update<T, 4>(a, stream);
  }
}

}  // namespace

cudaError_t launch_causal_conv1d(const ConvArgs& a, cudaStream_t stream) {
  return a.io == kF32 ? dispatch_fwd<float>(a, stream) : dispatch_fwd<__nv_bfloat16>(a, stream);
}

cudaError_t launch_causal_conv1d_update(const ConvUpdateArgs& a, cudaStream_t stream) {
  return a.io == kF32 ? dispatch_update<float>(a, stream) : dispatch_update<__nv_bfloat16>(a, stream);
}

}  // namespace ssm
