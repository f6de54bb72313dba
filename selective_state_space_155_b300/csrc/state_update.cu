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
//
// For dstate 16 on large batches a persistent, tiled form runs instead (SSM_DECODE_VARIANT=thread
// forces the form above): each CTA walks tiles of 128 channels, copying a tile's states, A rows
// and x, dt, z into shared memory with coalesced 16-byte cp.async two tiles ahead, so that the
// bytes in flight do not wait on registers; it computes one channel per thread from shared
// memory and writes the new states back with coalesced stores.  A thread reads its 64-byte rows
// in a rotated order of 16-byte quarters, quarter (k + t/2) mod 4 at its k-th access, which keeps
// the eight threads of every quarter-warp on distinct banks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {

// Stage waits of the bulk-copy decode kernel that gave up, since the library was loaded.
__device__ unsigned long long g_decode_wait_timeouts;

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

// ---- the tiled form (dstate 16) ----
constexpr int kTile = 128;   // channels per tile = threads per CTA
constexpr int kStages = 3;   // tiles resident per CTA: the current one and two in flight
constexpr int kTiledCtasPerSm = 4;

template <typename T>
struct TiledSmem {
  float st[kStages][kTile * 16];  // states of the tile's channels, [channel][16]
  float A[kStages][kTile * 16];   // their A rows
  T x[kStages][kTile], dt[kStages][kTile], z[kStages][kTile];
  float bias[kStages][kTile], Dv[kStages][kTile];  // dt_bias, D of the tile's channels (row tiles)
  T bc[kStages][2][16];                              // B, C rows of the tile's batch row (row tiles)
};

// The 16-byte quarter (four states) a thread touches at its k-th access of a 64-byte row.
__device__ __forceinline__ int rot_quarter(int k, int t) { return (k + (t >> 1)) & 3; }

// Four io values (states 4q .. 4q+3 of a B or C row, in global or shared memory) as float32.
template <typename T>
__device__ __forceinline__ float4 load_quarter(const T* row, int q) {
  if constexpr (std::is_same<T, float>::value) {
    return *reinterpret_cast<const float4*>(row + 4 * q);
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(row + 4 * q);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  }
}

// One channel's step on a staged tile: thread tid of the tile updates channel ch (= tile start +
// tid) from the tile's states and A rows (rows of 16 floats at tid * 16) and its x, dt, z (and,
// with row_tiles, dt_bias, D and the batch row's B, C) in shared memory; the new states go back
// to the same shared rows, the output to global memory.
template <typename T>
__device__ __forceinline__ void update_staged_channel(const UpdateArgs& a, float* st_s, const float* A_s,
                                                      const T* x_s, const T* dt_s, const T* z_s,
                                                      const float* bias_s, const float* D_s, const T* B_s,
                                                      const T* C_s, long long ch, int row_tiles) {
  const int tid = threadIdx.x;
  const T* gz = static_cast<const T*>(a.z);
  const uint32_t bq = fast_div(uint32_t(ch), a.div_dim);
  const int b = int(bq), d = int(ch - (long long)bq * a.dim);
  const T* Brow = row_tiles ? B_s : static_cast<const T*>(a.B) + size_t(b) * 16;
  const T* Crow = row_tiles ? C_s : static_cast<const T*>(a.C) + size_t(b) * 16;
  // registers hold the row quarters in this thread's rotated order (k-th = quarter rot_quarter(k))
  float s[16], Av[16], Bv[16], Cv[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int q = rot_quarter(k, tid);
    const float4 sv = *reinterpret_cast<const float4*>(&st_s[tid * 16 + 4 * q]);
    const float4 av = *reinterpret_cast<const float4*>(&A_s[tid * 16 + 4 * q]);
    const float4 bv = load_quarter<T>(Brow, q), cv = load_quarter<T>(Crow, q);
    s[4 * k] = sv.x, s[4 * k + 1] = sv.y, s[4 * k + 2] = sv.z, s[4 * k + 3] = sv.w;
    Av[4 * k] = av.x, Av[4 * k + 1] = av.y, Av[4 * k + 2] = av.z, Av[4 * k + 3] = av.w;
    Bv[4 * k] = bv.x, Bv[4 * k + 1] = bv.y, Bv[4 * k + 2] = bv.z, Bv[4 * k + 3] = bv.w;
    Cv[4 * k] = cv.x, Cv[4 * k + 1] = cv.y, Cv[4 * k + 2] = cv.z, Cv[4 * k + 3] = cv.w;
  }
  const float x = to_f32<T>(x_s[tid]);
  float r = to_f32<T>(dt_s[tid]);
  if (a.dt_bias) r += row_tiles ? bias_s[tid] : __ldg(a.dt_bias + d);
  const float zz = gz ? to_f32<T>(z_s[tid]) : 0.0f;
  const float Dd = a.D ? (row_tiles ? D_s[tid] : __ldg(a.D + d)) : 0.0f;
  const float step = a.softplus ? softplus_f32(r) : r;
  const float2 dd = f2(step * kLog2e, step * kLog2e), dx = f2(step * x, step * x);
  float2 acc = f2(0.0f, 0.0f);
  if (a.zoh) {
    const float2 sd = f2(step, step), xx = f2(x, x);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
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
    for (int i = 0; i < 16; i += 2) {
      const float2 g = __fmul2_rn(dd, f2(Av[i], Av[i + 1]));
      const float2 ab = f2(ex2_approx(g.x), ex2_approx(g.y));
      const float2 sn = __ffma2_rn(ab, f2(s[i], s[i + 1]), __fmul2_rn(dx, f2(Bv[i], Bv[i + 1])));
      s[i] = sn.x, s[i + 1] = sn.y;
      acc = __ffma2_rn(f2(Cv[i], Cv[i + 1]), sn, acc);
    }
  }
  float y = fmaf(Dd, x, acc.x + acc.y);
  if (gz) y *= silu_f32(zz);
  static_cast<T*>(a.out)[ch] = from_f32<T>(y);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<float4*>(&st_s[tid * 16 + 4 * rot_quarter(k, tid)]) =
        make_float4(s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3]);
}

// row_tiles: dim is a multiple of the tile, so a tile lies in one batch row and covers 128
// consecutive channels; their dt_bias, D and the row's B, C then ride the same copies.
template <typename T>
__global__ void __launch_bounds__(kTile)
    state_update_tiled_kernel(const UpdateArgs a, long long nch, int ntiles, int row_tiles) {
  extern __shared__ __align__(16) unsigned char smem_bytes[];
  TiledSmem<T>& sm = *reinterpret_cast<TiledSmem<T>*>(smem_bytes);
  constexpr int EPV = 16 / int(sizeof(T));  // io elements per 16-byte copy
  const int tid = threadIdx.x;
  const T* gx = static_cast<const T*>(a.x);
  const T* gdt = static_cast<const T*>(a.dt);
  const T* gz = static_cast<const T*>(a.z);

  // copies of tile `tile` into stage `st`: the state and A rows (512 16-byte pieces each, four per
  // thread, consecutive threads on consecutive pieces) and x, dt, z (one piece per thread)
  auto issue = [&](int tile, int st) {
    if (tile < ntiles) {
      const long long bd0 = (long long)tile * kTile;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = tid + kTile * k;  // piece c = quarter c % 4 of channel c / 4
        const long long ch = bd0 + (c >> 2);
        if (ch < nch) {
          cp_async_16(&sm.st[st][4 * c], a.state + bd0 * 16 + 4 * c, 16);
          const uint32_t d = uint32_t(ch - (long long)fast_div(uint32_t(ch), a.div_dim) * a.dim);
          cp_async_16(&sm.A[st][4 * c], a.A + size_t(d) * 16 + 4 * (c & 3), 16);
        }
      }
      if (tid < kTile / EPV) {
        const long long e0 = bd0 + tid * EPV;
        if (e0 < nch) {
          cp_async_16(&sm.x[st][tid * EPV], gx + e0, 16);
          cp_async_16(&sm.dt[st][tid * EPV], gdt + e0, 16);
          if (gz) cp_async_16(&sm.z[st][tid * EPV], gz + e0, 16);
        }
      }
      if (row_tiles) {
        const uint32_t b0 = fast_div(uint32_t(bd0), a.div_dim);
        const int d0 = int(bd0 - (long long)b0 * a.dim);
        constexpr int kFP = kTile / 4;  // 16-byte pieces of a float row slice
        constexpr int kBP = 16 / EPV;   // 16-byte pieces of a B or C row
        if (tid < kFP) {
          if (a.dt_bias) cp_async_16(&sm.bias[st][4 * tid], a.dt_bias + d0 + 4 * tid, 16);
        } else if (tid < 2 * kFP) {
          if (a.D) cp_async_16(&sm.Dv[st][4 * (tid - kFP)], a.D + d0 + 4 * (tid - kFP), 16);
        } else if (tid < 2 * kFP + 2 * kBP) {
          const int j = tid - 2 * kFP, which = j / kBP, p = j % kBP;
          const T* row = static_cast<const T*>(which ? a.C : a.B) + size_t(b0) * 16;
          cp_async_16(&sm.bc[st][which][p * EPV], row + p * EPV, 16);
        }
      }
    }
    cp_async_commit();
  };

  const int stride = gridDim.x;
#pragma unroll
  for (int s0 = 0; s0 < kStages - 1; ++s0) issue(blockIdx.x + s0 * stride, s0);
  int it = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += stride, ++it) {
    const int st = it % kStages;
    issue(tile + (kStages - 1) * stride, (it + kStages - 1) % kStages);
    cp_async_wait<kStages - 1>();  // this thread's copies of the current tile have landed
    __syncthreads();               // and everyone's
    const long long bd0 = (long long)tile * kTile, ch = bd0 + tid;
    if (ch < nch) update_staged_channel<T>(a, sm.st[st], sm.A[st], sm.x[st], sm.dt[st], sm.z[st], sm.bias[st],
                                           sm.Dv[st], sm.bc[st][0], sm.bc[st][1], ch, row_tiles);
    __syncthreads();  // the tile's new states are in shared memory
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = tid + kTile * k;
      if (bd0 + (c >> 2) < nch)
        *reinterpret_cast<float4*>(a.state + bd0 * 16 + 4 * c) = *reinterpret_cast<const float4*>(&sm.st[st][4 * c]);
    }
    __syncthreads();  // the stage is free for the copies issued at the next tile
  }
  cp_async_wait<0>();
}

// ---- the bulk-copy form (dstate 16, tiles inside one batch row) ----
// Same tiles, stages and per-channel step as the tiled form, but a tile's operands are contiguous
// ranges (the tile's 128 state rows, their 128 A rows, x, dt, z, dt_bias, D slices, the row's B and
// C), so thread 0 moves each with one bulk copy completing on the stage's mbarrier, and writes the
// tile's new states back with one bulk store: no per-thread copy issue or address arithmetic.
template <typename T>
struct __align__(16) BulkSmem {
  float st[kStages][kTile * 16];
  float A[kStages][kTile * 16];
  T x[kStages][kTile], dt[kStages][kTile], z[kStages][kTile];
  float bias[kStages][kTile], Dv[kStages][kTile];
  T bc[kStages][2][16];
  uint64_t bar[kStages];
};

// longest a stage wait may take before the kernel gives up on it, in SM clock cycles (~1 s)
constexpr long long kDecodeWaitLimit = 1LL << 31;

template <typename T>
__global__ void __launch_bounds__(kTile) state_update_bulk_kernel(const UpdateArgs a, int ntiles) {
  extern __shared__ __align__(128) unsigned char smem_bytes[];
  BulkSmem<T>& sm = *reinterpret_cast<BulkSmem<T>*>(smem_bytes);
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  const T* gx = static_cast<const T*>(a.x);
  const T* gdt = static_cast<const T*>(a.dt);
  const T* gz = static_cast<const T*>(a.z);
  const uint32_t xb = kTile * sizeof(T), fb = kTile * sizeof(float), bcb = 16 * sizeof(T);
  const uint32_t bytes = 2u * kTile * 16 * sizeof(float) + (gz ? 3u : 2u) * xb + (a.dt_bias ? fb : 0u) +
                         (a.D ? fb : 0u) + 2u * bcb;
  if (tid == 0) {
    abort_flag = 0;
#pragma unroll
    for (int i = 0; i < kStages; ++i) mbar_init(&sm.bar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // thread 0: the copies of tile `tile` into stage `stg`; pend[stg] = the iteration whose copies
  // into that stage were issued and not yet seen complete by thread 0 (-1: none)
  int pend[kStages];
#pragma unroll
  for (int i = 0; i < kStages; ++i) pend[i] = -1;
  auto issue = [&](int tile, int stg) {
    const long long bd0 = (long long)tile * kTile;
    const uint32_t b0 = fast_div(uint32_t(bd0), a.div_dim);
    const int d0 = int(bd0 - (long long)b0 * a.dim);
    uint64_t* bar = &sm.bar[stg];
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(sm.st[stg], a.state + bd0 * 16, kTile * 16 * sizeof(float), bar);
    bulk_load(sm.A[stg], a.A + size_t(d0) * 16, kTile * 16 * sizeof(float), bar);
    bulk_load(sm.x[stg], gx + bd0, xb, bar);
    bulk_load(sm.dt[stg], gdt + bd0, xb, bar);
    if (gz) bulk_load(sm.z[stg], gz + bd0, xb, bar);
    if (a.dt_bias) bulk_load(sm.bias[stg], a.dt_bias + d0, fb, bar);
    if (a.D) bulk_load(sm.Dv[stg], a.D + d0, fb, bar);
    bulk_load(sm.bc[stg][0], static_cast<const T*>(a.B) + size_t(b0) * 16, bcb, bar);
    bulk_load(sm.bc[stg][1], static_cast<const T*>(a.C) + size_t(b0) * 16, bcb, bar);
  };
  auto set_pend = [&](int stg, int v) {
#pragma unroll
    for (int i = 0; i < kStages; ++i)
      if (i == stg) pend[i] = v;
  };

  const int stride = gridDim.x;
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i)
      if (blockIdx.x + i * stride < ntiles) issue(blockIdx.x + i * stride, i), set_pend(i, i);
  }
  int it = 0;
  for (int tile = blockIdx.x; tile < ntiles; tile += stride, ++it) {
    const int stg = it % kStages;
    const int nxt = tile + (kStages - 1) * stride, nstg = (it + kStages - 1) % kStages;
    if (tid == 0 && nxt < ntiles && !abort_flag) {
      // the stage's previous tile (iteration it - 1) was stored from it: its bulk store must have
      // read the stage before new copies land there
      bulk_wait_read();
      issue(nxt, nstg), set_pend(nstg, it + kStages - 1);
    }
    const bool ok = mbar_wait(&sm.bar[stg], uint32_t(it / kStages) & 1u, &abort_flag, kDecodeWaitLimit,
                              &g_decode_wait_timeouts, 32);
    if (tid == 0 && ok) set_pend(stg, -1);
    const long long bd0 = (long long)tile * kTile, ch = bd0 + tid;
    update_staged_channel<T>(a, sm.st[stg], sm.A[stg], sm.x[stg], sm.dt[stg], sm.z[stg], sm.bias[stg], sm.Dv[stg],
                             sm.bc[stg][0], sm.bc[stg][1], ch, 1);
    fence_proxy_async_smem();  // this thread's new states, before the bulk store reads them
    __syncthreads();
    if (tid == 0) {
      bulk_store(a.state + bd0 * 16, sm.st[stg], kTile * 16 * sizeof(float));
      bulk_commit();
    }
  }
  if (tid == 0) {
    // copies that a given-up wait left in flight (bounded, ignoring the flag), then the stores
#pragma unroll
    for (int i = 0; i < kStages; ++i)
      if (pend[i] >= 0)
        mbar_wait(&sm.bar[i], uint32_t(pend[i] / kStages) & 1u, nullptr, kDecodeWaitLimit, &g_decode_wait_timeouts, 32);
    bulk_wait_done();
  }
}

// The tiled form applies to dstate 16 when every row it copies is whole 16-byte pieces and the
// batch is large enough to keep a persistent grid busy.
template <typename T>
bool tiled_applies(const UpdateArgs& a) {
  auto al = [](const void* p, uintptr_t m) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & m) == 0; };
  const long long nch = (long long)a.batch * a.dim;
  const uintptr_t bc_mask = sizeof(T) == 4 ? 15u : 7u;  // quarter loads of B and C rows
  return a.dstate == 16 && nch % 8 == 0 && nch >= (1LL << 16) && nch < (1LL << 32) && al(a.state, 15) &&
         al(a.A, 15) && al(a.x, 15) && al(a.dt, 15) && al(a.z, 15) && al(a.B, bc_mask) && al(a.C, bc_mask);
}

// Tiles lie in one batch row, and the per-channel and per-row operands copy as 16-byte pieces.
template <typename T>
bool row_tiles_apply(const UpdateArgs& a) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return a.dim % kTile == 0 && al(a.dt_bias) && al(a.D) && al(a.B) && al(a.C);
}

template <typename T>
cudaError_t launch_tiled(const UpdateArgs& a, cudaStream_t stream) {
  auto kernel = state_update_tiled_kernel<T>;
  constexpr size_t kSmem = sizeof(TiledSmem<T>);
  static std::atomic<uint64_t> configured{0};  // the dynamic shared-memory opt-in, once per device
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const long long nch = (long long)a.batch * a.dim;
  const int ntiles = int((nch + kTile - 1) / kTile);
  const int grid = std::min(ntiles, sms * kTiledCtasPerSm);
  UpdateArgs args = a;
  args.div_dim = make_fastdiv(uint32_t(a.dim));
  long long n = nch;
  int nt = ntiles;
  int rt = row_tiles_apply<T>(a) ? 1 : 0;
  void* params[] = {&args, &n, &nt, &rt};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kernel), dim3(unsigned(grid)), dim3(kTile), params, kSmem,
                          stream);
}

// The bulk form: the tiled form's conditions, tiles inside one batch row, and every range it
// copies 16-byte aligned in whole 16-byte pieces.
template <typename T>
bool bulk_applies(const UpdateArgs& a) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return tiled_applies<T>(a) && a.dim % kTile == 0 && al(a.dt_bias) && al(a.D) && al(a.B) && al(a.C) &&
         al(a.x) && al(a.dt) && al(a.z);
}

template <typename T>
cudaError_t launch_bulk(const UpdateArgs& a, cudaStream_t stream) {
  auto kernel = state_update_bulk_kernel<T>;
  constexpr size_t kSmem = sizeof(BulkSmem<T>);
  static std::atomic<uint64_t> configured{0};  // the dynamic shared-memory opt-in, once per device
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const long long nch = (long long)a.batch * a.dim;
  const int ntiles = int(nch / kTile);
  const int grid = std::min(ntiles, sms * kTiledCtasPerSm);
  UpdateArgs args = a;
  args.div_dim = make_fastdiv(uint32_t(a.dim));
  int nt = ntiles;
  void* params[] = {&args, &nt};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kernel), dim3(unsigned(grid)), dim3(kTile), params, kSmem,
                          stream);
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
  const char* force = std::getenv("SSM_DECODE_VARIANT");
  const bool plain = force && std::strcmp(force, "thread") == 0;
  const bool tiled_only = force && std::strcmp(force, "tiled") == 0;
  if (!plain && !tiled_only && bulk_applies<T>(a)) return launch_bulk<T>(a, stream);
  if (!plain && tiled_applies<T>(a)) return launch_tiled<T>(a, stream);
  if (a.dstate <= 4) return launch_npad<T, 4>(a, stream);
  if (a.dstate <= 8) return launch_npad<T, 8>(a, stream);
  return launch_npad<T, 16>(a, stream);
}

}  // namespace

cudaError_t launch_state_update(const UpdateArgs& a, cudaStream_t stream) {
  return a.io == kF32 ? dispatch<float>(a, stream) : dispatch<__nv_bfloat16>(a, stream);
}

cudaError_t decode_wait_timeouts(unsigned long long& count) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  return cudaMemcpyFromSymbol(&count, g_decode_wait_timeouts, sizeof(count));
}

}  // namespace ssm
