// Selective scan forward, lane-per-channel form, for sm_103a.
//
// Same operation as scan_fwd.cu (see ssm_scan.h for the definition and its sources), laid out so
// that one lane owns one (batch, channel) and all NPAD of its states:
//  * B_t and C_t are the same for every channel of a batch row, so the loads of them are
//    warp-uniform (shared-memory broadcast) and no lane ever needs another lane's data: there
//    is no cross-lane readout reduction at all.
//  * The per-element work (softplus of delta + dt_bias, Delta*u, D*u, silu(z)) is done by the
//    owning lane, in registers, from the staged rows of its own channel; nothing per element
//    goes back through shared memory.
//  * Each lane finishes 8 consecutive steps of its channel and stores them as one 16-byte (bf16)
//    or two 16-byte (float32) vectors.
//  * CTAs hold two warps (64 channels).  Chunks of 32 steps of u, delta, z, B, C are fetched with
//    16-byte cp.async into a three-stage ring, so a chunk's rows stay valid while every lane reads
//    them and the next chunk is already in flight; B and C are converted once per CTA into
//    float32 [t][n] tables.
// Each warp carries NPAD independent state chains per lane.  Measured on B300 this form is slower
// than the four-lanes-per-channel form at every size tried (1.45x with 27-69 channel warps per
// SM), so it runs only when SSM_SCAN_VARIANT=lane selects it; it is kept, and parity-tested, as
// the other point of the lanes-per-channel trade-off.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

constexpr int kLChunk = 32;  // steps per staged chunk
constexpr int kLSub = 8;     // steps per register window
constexpr int kLWarps = 2;
constexpr int kLThreads = 32 * kLWarps;
constexpr int kLStages = 3;

template <typename T, int NPAD>
struct LaneCfg {
  static constexpr int CPB = kLThreads;               // channels per CTA
  static constexpr int EPV = 16 / sizeof(T);          // io elements per 16-byte vector
  static constexpr int RS = kLChunk + EPV;            // padded row stride (elements): 5 vectors (bf16) / 9 (f32)
  static constexpr int VPR = kLChunk / EPV;           // vectors per staged row
  static constexpr int ROWS = 3 * CPB + 2 * NPAD;     // u, delta, z rows, then B rows, then C rows
  static constexpr size_t kStage = size_t(ROWS) * RS * sizeof(T);
  static constexpr size_t kRaw = kLStages * kStage;
  static constexpr size_t kBC = size_t(2) * kLChunk * NPAD * sizeof(float);
  static constexpr size_t kSmem = kRaw + kBC;
};

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

template <typename T>
__device__ __forceinline__ void unpack8(const uint4 v, float (&o)[8]);
template <>
__device__ __forceinline__ void unpack8<__nv_bfloat16>(const uint4 v, float (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    o[2 * i] = p.x, o[2 * i + 1] = p.y;
  }
}

// 8 consecutive io elements of a staged row (16-byte aligned) as float32
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&o)[8]) {
  if constexpr (std::is_same<T, float>::value) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    o[0] = a.x, o[1] = a.y, o[2] = a.z, o[3] = a.w, o[4] = b.x, o[5] = b.y, o[6] = b.z, o[7] = b.w;
  } else {
    unpack8<T>(*reinterpret_cast<const uint4*>(p), o);
  }
}

template <typename T, int NPAD, bool VEC>
__global__ void __launch_bounds__(kLThreads) scan_fwd_lane_kernel(const ScanArgs a) {
  using Cfg = LaneCfg<T, NPAD>;
  constexpr int CPB = Cfg::CPB, EPV = Cfg::EPV, RS = Cfg::RS, VPR = Cfg::VPR, ROWS = Cfg::ROWS;
  constexpr int NP = NPAD / 2;  // state pairs per lane

  extern __shared__ __align__(16) unsigned char smem[];
  T* raw = reinterpret_cast<T*>(smem);
  float* Bs = reinterpret_cast<float*>(smem + Cfg::kRaw);
  float* Cs = Bs + kLChunk * NPAD;

  const int tid = threadIdx.x;
  const int nblk_d = (a.dim + CPB - 1) / CPB;
  const int b = blockIdx.x / nblk_d;
  const int d0 = (blockIdx.x % nblk_d) * CPB;
  const int d = d0 + tid;
  const bool ch_ok = d < a.dim;
  const int L = a.seqlen, N = a.dstate;
  const bool has_z = a.z != nullptr;

  const T* __restrict__ gu = static_cast<const T*>(a.u);
  const T* __restrict__ gd = static_cast<const T*>(a.delta);
  const T* __restrict__ gz = static_cast<const T*>(a.z);
  const T* __restrict__ gB = static_cast<const T*>(a.B);
  const T* __restrict__ gC = static_cast<const T*>(a.C);

  float2 A2[NP], h[NP];
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    float av[2], hv[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int n = 2 * i + k;
      const bool ok = ch_ok && n < N;
      av[k] = ok ? a.A[size_t(d) * N + n] * kLog2e : 0.0f;
      hv[k] = (ok && a.h0) ? a.h0[(size_t(b) * a.dim + d) * N + n] : 0.0f;
    }
    A2[i] = f2(av[0], av[1]);
    h[i] = f2(hv[0], hv[1]);
  }
  const float bias = (ch_ok && a.dt_bias) ? a.dt_bias[d] : 0.0f;
  const float Dd = (ch_ok && a.D) ? a.D[d] : 0.0f;
  T* yrow = static_cast<T*>(a.y) + (size_t(b) * a.dim + (ch_ok ? d : 0)) * L;

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
      for (int v = tid; v < ROWS * VPR; v += kLThreads) {
        const int r = v / VPR, j = v % VPR;
        if (!has_z && r >= 2 * CPB && r < 3 * CPB) continue;
        bool ok;
        const T* src = row_src(r, ok);
        const int t = t0 + j * EPV;
        int bytes = ok ? min(EPV, L - t) * int(sizeof(T)) : 0;
        bytes = max(bytes, 0);
        // a zero-byte copy only zero-fills, but its source must still be a valid aligned address
        cp_async_16(dst + r * RS + j * EPV, bytes > 0 ? static_cast<const void*>(src + t) : gu, bytes);
      }
    } else {
      for (int e = tid; e < ROWS * kLChunk; e += kLThreads) {
        const int r = e / kLChunk, j = e % kLChunk;
        if (!has_z && r >= 2 * CPB && r < 3 * CPB) continue;
        bool ok;
        const T* src = row_src(r, ok);
        const int t = t0 + j;
        dst[r * RS + j] = (ok && t < L) ? src[t] : from_f32<T>(0.0f);
      }
    }
  };

  const int nchunks = (L + kLChunk - 1) / kLChunk;
  if (nchunks > 0) stage_load(0, 0);
  cp_async_commit();

  for (int k = 0; k < nchunks; ++k) {
    const int t0 = k * kLChunk;
    // stage (k+1)%3 was last read in chunk k-2, before this thread's previous barrier pair
    if (k + 1 < nchunks) stage_load((k + 1) % kLStages, t0 + kLChunk);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const T* st = raw + size_t(k % kLStages) * ROWS * RS;
    const T* sB = st + 3 * CPB * RS;
    const T* sC = sB + NPAD * RS;
    // B, C rows -> float32 [t][n] tables (all lanes of the CTA read every entry)
    for (int e = tid; e < 2 * NPAD * kLChunk; e += kLThreads) {
      const int which = e / (NPAD * kLChunk), rem = e % (NPAD * kLChunk);
      const int t = rem / NPAD, n = rem % NPAD;
      (which == 0 ? Bs : Cs)[t * NPAD + n] = to_f32<T>((which == 0 ? sB : sC)[n * RS + t]);
    }
    __syncthreads();

    const T* su = st + tid * RS;
    const T* sd = st + (CPB + tid) * RS;
    const T* sz = st + (2 * CPB + tid) * RS;
#pragma unroll 1
    for (int w = 0; w < kLChunk; w += kLSub) {
      // per-element prologue for 8 steps of this lane's channel
      float dv[8], uv[8], zv[8];
      load8<T>(sd + w, dv);
      load8<T>(su + w, uv);
      if (has_z) load8<T>(sz + w, zv);
      float dl[8], du[8], Du[8], sg[8];
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        float2 x = __fadd2_rn(f2(dv[j], dv[j + 1]), f2(bias, bias));
        if (a.softplus) x = f2(softplus_f32(x.x), softplus_f32(x.y));
        const bool in0 = t0 + w + j < L, in1 = t0 + w + j + 1 < L;
        dl[j] = in0 ? x.x : 0.0f;
        dl[j + 1] = in1 ? x.y : 0.0f;
        const float2 dd = __fmul2_rn(f2(dl[j], dl[j + 1]), f2(uv[j], uv[j + 1]));
        du[j] = dd.x, du[j + 1] = dd.y;
        const float2 dD = __fmul2_rn(f2(Dd, Dd), f2(uv[j], uv[j + 1]));
        Du[j] = dD.x, Du[j + 1] = dD.y;
        sg[j] = has_z ? silu_f32(zv[j]) : 1.0f;
        sg[j + 1] = has_z ? silu_f32(zv[j + 1]) : 1.0f;
      }
      // the recurrence: all NPAD states of this channel, 8 steps
      float yv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float* Bt = Bs + (w + j) * NPAD;
        const float* Ct = Cs + (w + j) * NPAD;
        const float2 dd = f2(dl[j], dl[j]), uu = f2(du[j], du[j]);
        float2 acc = f2(0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < NPAD / 4; ++q) {
          const float4 bb = *reinterpret_cast<const float4*>(Bt + 4 * q);
          const float4 cc = *reinterpret_cast<const float4*>(Ct + 4 * q);
          const float2 g0 = __fmul2_rn(dd, A2[2 * q]), g1 = __fmul2_rn(dd, A2[2 * q + 1]);
          const float2 a0 = f2(ex2_approx(g0.x), ex2_approx(g0.y));
          const float2 a1 = f2(ex2_approx(g1.x), ex2_approx(g1.y));
          h[2 * q] = __ffma2_rn(a0, h[2 * q], __fmul2_rn(uu, f2(bb.x, bb.y)));
          h[2 * q + 1] = __ffma2_rn(a1, h[2 * q + 1], __fmul2_rn(uu, f2(bb.z, bb.w)));
          acc = __ffma2_rn(f2(cc.x, cc.y), h[2 * q], acc);
          acc = __ffma2_rn(f2(cc.z, cc.w), h[2 * q + 1], acc);
        }
        yv[j] = acc.x + acc.y;
      }
      // epilogue: (y + D u) * silu(z) -> io type, 8 consecutive steps
      float ov[8];
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const float2 o = __fmul2_rn(__fadd2_rn(f2(yv[j], yv[j + 1]), f2(Du[j], Du[j + 1])), f2(sg[j], sg[j + 1]));
        ov[j] = o.x, ov[j + 1] = o.y;
      }
      const int tg = t0 + w;
      if (ch_ok) {
        const int n = L - tg;
        if constexpr (VEC && std::is_same<T, __nv_bfloat16>::value) {
          if (n >= 8) {
            uint32_t wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const __nv_bfloat162 p = __floats2bfloat162_rn(ov[2 * j], ov[2 * j + 1]);
              wv[j] = *reinterpret_cast<const uint32_t*>(&p);
            }
            *reinterpret_cast<uint4*>(yrow + tg) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        } else if constexpr (VEC) {
          if (n >= 4) *reinterpret_cast<float4*>(yrow + tg) = make_float4(ov[0], ov[1], ov[2], ov[3]);
          if (n >= 8) *reinterpret_cast<float4*>(yrow + tg + 4) = make_float4(ov[4], ov[5], ov[6], ov[7]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < n) yrow[tg + j] = from_f32<T>(ov[j]);
        }
      }
    }
  }
  cp_async_wait<0>();

  if (a.last_state && ch_ok) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int n = 2 * i + k;
        if (n < N) a.last_state[(size_t(b) * a.dim + d) * N + n] = k == 0 ? h[i].x : h[i].y;
      }
    }
  }
}

template <typename T, int NPAD, bool VEC>
cudaError_t launch_lane_cfg(const ScanArgs& a, cudaStream_t stream) {
  using Cfg = LaneCfg<T, NPAD>;
  auto kernel = scan_fwd_lane_kernel<T, NPAD, VEC>;
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
  return cudaLaunchKernel(reinterpret_cast<const void*>(kernel), dim3(unsigned(nblk)), dim3(kLThreads), params,
                          Cfg::kSmem, stream);
}

template <typename T, bool VEC>
cudaError_t lane_dispatch_npad(const ScanArgs& a, cudaStream_t stream) {
  if (a.dstate <= 4) return launch_lane_cfg<T, 4, VEC>(a, stream);
  if (a.dstate <= 8) return launch_lane_cfg<T, 8, VEC>(a, stream);
  return launch_lane_cfg<T, 16, VEC>(a, stream);
}

}  // namespace

cudaError_t launch_scan_fwd_lane(const ScanArgs& a, bool vec, cudaStream_t stream) {
  if (a.io == kF32)
    return vec ? lane_dispatch_npad<float, true>(a, stream) : lane_dispatch_npad<float, false>(a, stream);
  return vec ? lane_dispatch_npad<__nv_bfloat16, true>(a, stream) : lane_dispatch_npad<__nv_bfloat16, false>(a, stream);
}

}  // namespace ssm
