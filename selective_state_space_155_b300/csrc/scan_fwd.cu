// Selective scan forward for sm_103a.
//
// What it computes (per batch row b, channel d, state n; see ssm_scan.h for the sources):
//   Delta_t = softplus(delta_t + dt_bias[d]);  Abar = exp(Delta_t A[d,n]);  h_t = Abar h_{t-1} + Delta_t B_t[n] u_t
//   y_t = sum_n C_t[n] h_t[n] + D[d] u_t;  out_t = y_t * silu(z_t);  last_state = h_{L-1}
//
// Design (B300: 148 SMs, MUFU ex2 32/clk/SM, FP32 FMA 128/clk/SM, packed f32x2 FMA at the same
// lane rate).  The path is a scan, not a contraction, so it runs on the SIMT pipes:
//  * A CTA owns CPB channels of one batch row and walks L in chunks of CHUNK steps.  Chunk k+1
//    is fetched with 16-byte cp.async (zero-filled past the sequence end) while chunk k is
//    computed, so HBM sees u, delta, z, B, C once and y once; the expanded (L, D, N) tensors
//    Abar and Bbar never exist outside registers.
//  * Four states per lane: a channel spans R = NPAD/4 lanes.  The float32 state lives in
//    registers for the whole sequence and is the carried prefix between chunks.
//  * Per chunk, a prologue turns (delta, u) into (Delta, Delta*u) once per (channel, t) and
//    parks them in shared memory, so softplus is not repeated by the R lanes of a channel.
//  * The readout sum over n spans the R lanes of a channel: each group of R consecutive steps
//    is reduced with a transpose-reduce (R-1 shuffles per R outputs per lane), after which lane
//    g owns step g of the group and runs the D skip, the gate and the output rounding for it.
//  * Padded states (n >= dstate) get A = 0 and B = C = 0; padded steps (t >= seqlen) get
//    Delta = 0.  Both leave the state unchanged, so one code path serves every size.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kChunk = 64;

template <typename T, int NPAD>
struct ScanCfg {
  static constexpr int R = NPAD / 4;             // lanes per channel
  static constexpr int WARPS = R;                // so that every CTA holds 32 channels
  static constexpr int NT = 32 * WARPS;          // threads per CTA
  static constexpr int CPW = 32 / R;             // channels per warp
  static constexpr int CPB = CPW * WARPS;        // channels per CTA (32)
  static constexpr int EPV = 16 / sizeof(T);     // elements per 16-byte vector
  static constexpr int RS = kChunk + EPV;        // padded row stride (elements) of staged rows
  static constexpr int VPR = kChunk / EPV;       // vectors per staged row
  static constexpr int ROWS = 3 * CPB + 2 * NPAD;  // u, delta, z rows, then B rows, then C rows
  static constexpr int PS = CPB + 4;             // padded row stride (float2) of the (Delta, Delta*u) table
  // shared memory map (bytes)
  static constexpr size_t kRawStage = size_t(ROWS) * RS * sizeof(T);
  static constexpr size_t kRaw = 2 * kRawStage;
  static constexpr size_t kBC = size_t(2) * kChunk * NPAD * sizeof(float);
  static constexpr size_t kP = size_t(kChunk) * PS * sizeof(float2);
  static constexpr size_t kY = size_t(CPB) * RS * sizeof(T);
  static constexpr size_t kSmem = kRaw + kBC + kP + kY;
};

template <typename T, int NPAD, bool VEC>
__global__ void __launch_bounds__(ScanCfg<T, NPAD>::NT) scan_fwd_kernel(const ScanArgs a) {
  using Cfg = ScanCfg<T, NPAD>;
  constexpr int R = Cfg::R, CPW = Cfg::CPW, CPB = Cfg::CPB, EPV = Cfg::EPV, RS = Cfg::RS, VPR = Cfg::VPR;
  constexpr int kThreads = Cfg::NT;
  constexpr int ROWS = Cfg::ROWS, PS = Cfg::PS;

  extern __shared__ __align__(16) unsigned char smem[];
  T* raw = reinterpret_cast<T*>(smem);  // [2][ROWS][RS]
  float* Bs = reinterpret_cast<float*>(smem + Cfg::kRaw);  // [CHUNK][NPAD]
  float* Cs = Bs + kChunk * NPAD;                          // [CHUNK][NPAD]
  float2* Ps = reinterpret_cast<float2*>(smem + Cfg::kRaw + Cfg::kBC);  // [CHUNK][PS]
  T* Ys = reinterpret_cast<T*>(smem + Cfg::kRaw + Cfg::kBC + Cfg::kP);   // [CPB][RS]

  const int tid = threadIdx.x;
  const int nblk_d = (a.dim + CPB - 1) / CPB;
  const int b = blockIdx.x / nblk_d;
  const int d0 = (blockIdx.x % nblk_d) * CPB;
  const int warp = tid >> 5, lane = tid & 31;
  const int cw = lane / R, g = lane % R;
  const int cl = warp * CPW + cw;  // channel within the CTA
  const int d = d0 + cl;
  const bool ch_ok = d < a.dim;
  const int L = a.seqlen, N = a.dstate;
  const bool has_z = a.z != nullptr;

  const T* __restrict__ gu = static_cast<const T*>(a.u);
  const T* __restrict__ gd = static_cast<const T*>(a.delta);
  const T* __restrict__ gz = static_cast<const T*>(a.z);
  const T* __restrict__ gB = static_cast<const T*>(a.B);
  const T* __restrict__ gC = static_cast<const T*>(a.C);
  T* __restrict__ gy = static_cast<T*>(a.y);

  // Per-lane constants and state: states n = 4g .. 4g+3 of channel d.
  float A2[4], h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = 4 * g + i;
    const bool ok = ch_ok && n < N;
    A2[i] = ok ? a.A[size_t(d) * N + n] * kLog2e : 0.0f;
    h[i] = (ok && a.h0) ? a.h0[(size_t(b) * a.dim + d) * N + n] : 0.0f;
  }
  const float Dd = (ch_ok && a.D) ? a.D[d] : 0.0f;

  // Source row of staged row r (u, delta, z rows of the CTA's channels, then B and C rows).
  auto row_src = [&](int r, bool& ok) -> const T* {
    if (r < 3 * CPB) {
      const int which = r / CPB, c = r % CPB;
      const T* base = which == 0 ? gu : (which == 1 ? gd : gz);
      ok = (d0 + c < a.dim) && (which < 2 || has_z);
      return base + (size_t(b) * a.dim + (d0 + c)) * L;
    }
    const int rr = r - 3 * CPB;
    const int which = rr / NPAD, n = rr % NPAD;
    ok = n < N;
    return (which == 0 ? gB : gC) + (size_t(b) * N + n) * L;
  };

  auto stage_load = [&](int stage, int t0) {
    T* dst = raw + size_t(stage) * ROWS * RS;
    if constexpr (VEC) {
      for (int v = tid; v < ROWS * VPR; v += kThreads) {
        const int r = v / VPR, j = v % VPR;
        if (!has_z && r >= 2 * CPB && r < 3 * CPB) continue;  // z rows are never read without a gate
        bool ok;
        const T* src = row_src(r, ok);
        const int t = t0 + j * EPV;
        int bytes = ok ? min(EPV, L - t) * int(sizeof(T)) : 0;
        bytes = max(bytes, 0);
        // a zero-byte copy only zero-fills, but its source must still be a valid aligned address
        cp_async_16(dst + r * RS + j * EPV, bytes > 0 ? static_cast<const void*>(src + t) : gu, bytes);
      }
    } else {
      for (int e = tid; e < ROWS * kChunk; e += kThreads) {
        const int r = e / kChunk, j = e % kChunk;
        if (!has_z && r >= 2 * CPB && r < 3 * CPB) continue;
        bool ok;
        const T* src = row_src(r, ok);
        const int t = t0 + j;
        dst[r * RS + j] = (ok && t < L) ? src[t] : from_f32<T>(0.0f);
      }
    }
  };

  const int nchunks = (L + kChunk - 1) / kChunk;
  if (nchunks > 0) stage_load(0, 0);
  cp_async_commit();

  for (int k = 0; k < nchunks; ++k) {
    const int t0 = k * kChunk;
    if (k + 1 < nchunks) stage_load((k + 1) & 1, t0 + kChunk);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const T* st = raw + size_t(k & 1) * ROWS * RS;
    const T* su = st;
    const T* sd = st + CPB * RS;
    const T* sz = st + 2 * CPB * RS;
    const T* sB = st + 3 * CPB * RS;
    const T* sC = sB + NPAD * RS;

    // (a) B, C rows -> float32 [t][n] tables.
    for (int e = tid; e < 2 * kChunk * NPAD; e += kThreads) {
      const int which = e / (kChunk * NPAD), rem = e % (kChunk * NPAD);
      const int t = rem / NPAD, n = rem % NPAD;
      const T* srow = (which == 0 ? sB : sC) + n * RS;
      (which == 0 ? Bs : Cs)[t * NPAD + n] = to_f32<T>(srow[t]);
    }
    // (b) (Delta, Delta*u) for this warp's channels; zero past the sequence end.
    {
      for (int e = lane; e < CPW * kChunk; e += 32) {
        const int c = e % CPW, t = e / CPW;
        const int clc = warp * CPW + c, dc = d0 + clc;
        float dl = 0.0f, du = 0.0f;
        if (t0 + t < L && dc < a.dim) {
          float x = to_f32<T>(sd[clc * RS + t]);
          if (a.dt_bias) x += a.dt_bias[dc];
          dl = a.softplus ? softplus_f32(x) : x;
          du = dl * to_f32<T>(su[clc * RS + t]);
        }
        Ps[t * PS + clc] = make_float2(dl, du);
      }
    }
    __syncthreads();

    // (c) the recurrence, R steps per group; lane g finishes step g of each group.
#pragma unroll 1
    for (int tt = 0; tt < kChunk; tt += R) {
      float yp[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int t = tt + j;
        const float2 p = Ps[t * PS + cl];
        const float4 bb = *reinterpret_cast<const float4*>(Bs + t * NPAD + 4 * g);
        const float4 cc = *reinterpret_cast<const float4*>(Cs + t * NPAD + 4 * g);
        const float a0 = ex2_approx(p.x * A2[0]);
        const float a1 = ex2_approx(p.x * A2[1]);
        const float a2 = ex2_approx(p.x * A2[2]);
        const float a3 = ex2_approx(p.x * A2[3]);
        h[0] = fmaf(a0, h[0], p.y * bb.x);
        h[1] = fmaf(a1, h[1], p.y * bb.y);
        h[2] = fmaf(a2, h[2], p.y * bb.z);
        h[3] = fmaf(a3, h[3], p.y * bb.w);
        yp[j] = fmaf(cc.w, h[3], fmaf(cc.z, h[2], fmaf(cc.y, h[1], cc.x * h[0])));
      }
      float yv;
      if constexpr (R == 1) {
        yv = yp[0];
      } else if constexpr (R == 2) {
        const bool hi = g & 1;
        const float send = hi ? yp[0] : yp[1];
        yv = (hi ? yp[1] : yp[0]) + __shfl_xor_sync(0xffffffffu, send, 1);
      } else {
        const bool hi2 = g & 2;
        const float s0 = hi2 ? yp[0] : yp[2];
        const float s1 = hi2 ? yp[1] : yp[3];
        float k0 = hi2 ? yp[2] : yp[0];
        float k1 = hi2 ? yp[3] : yp[1];
        k0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        k1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        const bool hi1 = g & 1;
        const float s = hi1 ? k0 : k1;
        yv = (hi1 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, s, 1);
      }
      // epilogue for step tt + g of channel cl
      const int t = tt + g;
      float out = fmaf(Dd, to_f32<T>(su[cl * RS + t]), yv);
      if (has_z) out *= silu_f32(to_f32<T>(sz[cl * RS + t]));
      Ys[cl * RS + t] = from_f32<T>(out);
    }
    __syncthreads();

    // (d) the chunk of y -> global.
    if constexpr (VEC) {
      for (int v = tid; v < CPB * VPR; v += kThreads) {
        const int c = v / VPR, j = v % VPR;
        const int t = t0 + j * EPV;
        if (d0 + c < a.dim && t < L)
          *reinterpret_cast<uint4*>(gy + (size_t(b) * a.dim + d0 + c) * L + t) =
              *reinterpret_cast<const uint4*>(Ys + c * RS + j * EPV);
      }
    } else {
      for (int e = tid; e < CPB * kChunk; e += kThreads) {
        const int c = e / kChunk, j = e % kChunk;
        const int t = t0 + j;
        if (d0 + c < a.dim && t < L) gy[(size_t(b) * a.dim + d0 + c) * L + t] = Ys[c * RS + j];
      }
    }
  }
  cp_async_wait<0>();

  if (a.last_state && ch_ok) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * g + i;
      if (n < N) a.last_state[(size_t(b) * a.dim + d) * N + n] = h[i];
    }
  }
}

template <typename T, int NPAD, bool VEC>
cudaError_t launch_cfg(const ScanArgs& a, cudaStream_t stream) {
  using Cfg = ScanCfg<T, NPAD>;
  auto kernel = scan_fwd_kernel<T, NPAD, VEC>;
  // The dynamic shared-memory opt-in is a per-device function attribute; set it once per device.
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmem));
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const long long nblk = (long long)((a.dim + Cfg::CPB - 1) / Cfg::CPB) * a.batch;
  if (nblk <= 0) return cudaSuccess;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ScanArgs args = a;
  void* params[] = {&args};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kernel), dim3(unsigned(nblk)), dim3(Cfg::NT), params,
                          Cfg::kSmem, stream);
}

template <typename T, bool VEC>
cudaError_t dispatch_npad(const ScanArgs& a, cudaStream_t stream) {
  if (a.dstate <= 4) return launch_cfg<T, 4, VEC>(a, stream);
  if (a.dstate <= 8) return launch_cfg<T, 8, VEC>(a, stream);
  return launch_cfg<T, 16, VEC>(a, stream);
}

template <typename T>
bool rows_vectorisable(const ScanArgs& a) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return (size_t(a.seqlen) * sizeof(T)) % 16 == 0 && al(a.u) && al(a.delta) && al(a.z) && al(a.B) && al(a.C) &&
         al(a.y);
}

}  // namespace

cudaError_t launch_scan_fwd(const ScanArgs& a, cudaStream_t stream) {
  if (a.io == kF32)
    return rows_vectorisable<float>(a) ? dispatch_npad<float, true>(a, stream)
                                       : dispatch_npad<float, false>(a, stream);
  return rows_vectorisable<__nv_bfloat16>(a) ? dispatch_npad<__nv_bfloat16, true>(a, stream)
                                             : dispatch_npad<__nv_bfloat16, false>(a, stream);
}

}  // namespace ssm
