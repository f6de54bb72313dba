// Device helpers for the scan kernels: MUFU approximations, softplus, silu, io conversions,
// mbarriers with bounded waits.
//
// Accuracy (float32 arithmetic throughout):
//  * ex2.approx.ftz.f32 / lg2.approx.ftz.f32 / rcp.approx.ftz.f32 / tanh.approx.f32 are the PTX
//    special-function approximations (a few ulp for ex2, lg2, rcp; about 2^-11 relative for tanh;
//    subnormal results flush to zero).
//  * softplus_f32 (decode step, backward): max(x, 0) + log1p(e), e = exp(-|x|) in (0, 1]; log1p(e)
//    is the alternating Taylor series e - e^2/2 + ... - e^6/6 when e < 1/16 (truncation below
//    e^7/7 < 5e-10 relative) and lg2(1 + e) * ln 2 otherwise (1 + e >= 17/16 there, so lg2's
//    absolute error stays small next to the result).
//  * softplus2 (forward scan): the same max(x, 0) + log1p(e) with log1p(e) = e P(e), P a degree-7
//    polynomial (below): one MUFU op per value and no branch.
//  * silu(z) = z / (1 + 2^(-z log2 e)), or h + h tanh(h) with h = z / 2 where the output is bf16.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float softplus_f32(float x) {
  const float e = ex2_approx(-fabsf(x) * kLog2e);
  // Horner form of e - e^2/2 + e^3/3 - e^4/4 + e^5/5 - e^6/6
  float s = fmaf(e, -1.0f / 6.0f, 1.0f / 5.0f);
  s = fmaf(e, -s, 1.0f / 4.0f);
  s = fmaf(e, -s, 1.0f / 3.0f);
  s = fmaf(e, -s, 1.0f / 2.0f);
  s = fmaf(e, -s, 1.0f);
  s *= e;
  const float viaLog = lg2_approx(1.0f + e) * kLn2;
  return fmaxf(x, 0.0f) + (e < 0.0625f ? s : viaLog);
}

__device__ __forceinline__ float silu_f32(float z) { return z * rcp_approx(1.0f + ex2_approx(-z * kLog2e)); }

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus of two values: max(x, 0) + log1p(e), e = exp(-|x|) in (0, 1], with log1p(e) = e P(e)
// and P a degree-7 polynomial for log1p(e) / e on [0, 1] (Chebyshev interpolation of that function,
// coefficients rounded to float32; relative error of e P(e) below 3.3e-7 evaluated in float32, so
// softplus stays within 6e-7 relative over |x| <= 10).  One MUFU op per value, no branch, and no
// loss of relative precision for small e.
__device__ __forceinline__ float2 softplus2(float2 x) {
  const float2 e = make_float2(ex2_approx(-fabsf(x.x) * kLog2e), ex2_approx(-fabsf(x.y) * kLog2e));
  auto c = [](float v) { return make_float2(v, v); };
  float2 p = __ffma2_rn(e, c(-0.00837115291506052f), c(0.04349390044808388f));
  p = __ffma2_rn(e, p, c(-0.1068500280380249f));
  p = __ffma2_rn(e, p, c(0.1768747717142105f));
  p = __ffma2_rn(e, p, c(-0.24474774301052094f));
  p = __ffma2_rn(e, p, c(0.3327192962169647f));
  p = __ffma2_rn(e, p, c(-0.49997174739837646f));
  p = __ffma2_rn(e, p, c(0.9999997615814209f));
  return __ffma2_rn(p, e, make_float2(fmaxf(x.x, 0.0f), fmaxf(x.y, 0.0f)));
}

// silu of two values, z sigmoid(z).  BF16 selects h + h tanh(h), h = z / 2: one MUFU op, whose
// relative error (about 2^-11) stays far below bf16 output rounding.  Otherwise z / (1 + 2^(-z
// log2 e)) with ex2 and rcp (a few ulp), for float outputs.
template <bool BF16>
__device__ __forceinline__ float2 silu2(float2 z) {
  if constexpr (BF16) {
    const float2 h = __fmul2_rn(z, make_float2(0.5f, 0.5f));
    return __ffma2_rn(h, make_float2(tanh_approx(h.x), tanh_approx(h.y)), h);
  } else {
    return make_float2(silu_f32(z.x), silu_f32(z.y));
  }
}

// ---- mbarriers with bounded waits ----
// A CTA-scope shared-memory mbarrier.  Arrivals release the arriving thread's prior shared-memory
// accesses; a completed wait acquires them.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Arrive on `bar` and add `bytes` to the transaction count its current phase waits for (the bytes a
// tensor copy issued next will deliver).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Make the mbarrier initialisations visible to the tensor-copy unit before its first completion.
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// Tensor copy (TMA) of the 2-D box at (x = column, y = row) of the tensor map into shared memory
// at dst (128-byte aligned), completing `bytes` of the transaction count of `bar`.  Columns past the
// tensor's extent and rows past its end are filled with zeros.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// The same for a 3-D box at (x, y, z).
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Bulk (non-tensor) copies: `bytes` (a multiple of 16, both addresses 16-byte aligned) from global
// to shared memory, completing on `bar`'s transaction count; and from shared to global memory in
// the issuing thread's bulk group, which bulk_commit closes and bulk_wait_read / bulk_wait_done
// wait for (until the source was read / the writes were performed).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(reinterpret_cast<uint64_t>(dst)), "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's earlier shared-memory writes before later bulk copies that read them.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Wait until `bar` completes the phase of the given parity.  The wait is bounded: it gives up after
// `limit` clock cycles, or at once when *abort (a CTA-wide flag in shared memory) is set; giving up
// sets *abort, adds one to *timeouts for the wait that ran out, and returns false, so that a broken
// hand-off ends the kernel (with garbage outputs and a counted timeout) instead of hanging it.
// Between tests the warp sleeps for `backoff_ns` nanoseconds, so that a waiting warp takes almost
// no issue slots from the warps doing the work.  With abort == nullptr the wait runs to its limit
// regardless of any flag (used to drain copies still in flight before a CTA exits).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, long long limit,
                                          unsigned long long* timeouts, unsigned backoff_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    __nanosleep(backoff_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if (clock64() - t0 > limit) {
      if (abort) *abort = 1;
      atomicAdd(timeouts, 1ull);
      return false;
    }
  }
}

// Exact zero-order hold: Bbar = (exp(Delta a) - 1) / a * B for a diagonal A.  This returns the
// factor Bbar / B from x = Delta*a, abar = exp(x) (already computed by the caller), Delta and
// inv_a = 1/a.  For |x| >= 1/16 it is (abar - 1) * inv_a: abar carries a relative error of a few
// 2^-23, which against |abar - 1| >= 1 - e^(-1/16) = 0.06 costs at most a few units in the
// sixth digit.  Below that, abar - 1 would cancel, so it is Delta * (e^x - 1)/x from the Taylor
// series 1 + x/2 + x^2/6 + x^3/24, whose first omitted term x^4/120 is under 1.3e-7 relative
// there; this branch also covers a = 0, where the factor is its limit Delta and inv_a is never
// used.
__device__ __forceinline__ float zoh_factor(float x, float abar, float delta, float inv_a) {
  float p = fmaf(x, 1.0f / 24.0f, 1.0f / 6.0f);
  p = fmaf(x, p, 0.5f);
  p = fmaf(x, p, 1.0f);
  return fabsf(x) < 0.0625f ? delta * p : (abar - 1.0f) * inv_a;
}
// zoh_factor on a pair of states with packed arithmetic.
__device__ __forceinline__ float2 zoh_factor2(float2 x, float2 abar, float2 delta, float2 inv_a) {
  float2 p = __ffma2_rn(x, make_float2(1.0f / 24.0f, 1.0f / 24.0f), make_float2(1.0f / 6.0f, 1.0f / 6.0f));
  p = __ffma2_rn(x, p, make_float2(0.5f, 0.5f));
  p = __ffma2_rn(x, p, make_float2(1.0f, 1.0f));
  p = __fmul2_rn(p, delta);
  const float2 q = __fmul2_rn(__fadd2_rn(abar, make_float2(-1.0f, -1.0f)), inv_a);
  return make_float2(fabsf(x.x) < 0.0625f ? p.x : q.x, fabsf(x.y) < 0.0625f ? p.y : q.y);
}
// zoh_factor2 from the base-2 exponent g = x / ln 2 that the recurrence already has (abar =
// 2^g): the same series and switch point, with the powers of ln 2 folded into the coefficients.
__device__ __forceinline__ float2 zoh_factor2_log2(float2 g, float2 abar, float2 delta, float2 inv_a) {
  constexpr double ln2 = 0.6931471805599453;
  constexpr float c1 = float(ln2 / 2), c2 = float(ln2 * ln2 / 6), c3 = float(ln2 * ln2 * ln2 / 24);
  constexpr float gmax = float(0.0625 / ln2);
  float2 p = __ffma2_rn(g, make_float2(c3, c3), make_float2(c2, c2));
  p = __ffma2_rn(g, p, make_float2(c1, c1));
  p = __ffma2_rn(g, p, make_float2(1.0f, 1.0f));
  p = __fmul2_rn(p, delta);
  const float2 q = __fmul2_rn(__fadd2_rn(abar, make_float2(-1.0f, -1.0f)), inv_a);
  return make_float2(fabsf(g.x) < gmax ? p.x : q.x, fabsf(g.y) < gmax ? p.y : q.y);
}

// d(Bbar/B)/da of the zero-order hold, for the backward pass: with c = zoh_factor(...),
// dc/da = (Delta abar - c) / a = Delta^2 phi(x), phi(x) = (x e^x - e^x + 1) / x^2.  For |x| >= 1/2
// the first form cancels by at most a few bits.  Below that it is Delta^2 times phi's Taylor
// series, sum_k (k+1)/(k+2)! x^k through x^7, whose first omitted term is under 1e-7 relative
// there; that branch also covers a = 0 (limit Delta^2 / 2), where inv_a is never used.
__device__ __forceinline__ float2 zoh_factor_da2(float2 x, float2 abar, float2 delta, float2 c, float2 inv_a) {
  float2 p = __ffma2_rn(x, make_float2(1.0f / 45360.0f, 1.0f / 45360.0f), make_float2(1.0f / 5760.0f, 1.0f / 5760.0f));
  p = __ffma2_rn(x, p, make_float2(1.0f / 840.0f, 1.0f / 840.0f));
  p = __ffma2_rn(x, p, make_float2(1.0f / 144.0f, 1.0f / 144.0f));
  p = __ffma2_rn(x, p, make_float2(1.0f / 30.0f, 1.0f / 30.0f));
  p = __ffma2_rn(x, p, make_float2(1.0f / 8.0f, 1.0f / 8.0f));
  p = __ffma2_rn(x, p, make_float2(1.0f / 3.0f, 1.0f / 3.0f));
  p = __ffma2_rn(x, p, make_float2(0.5f, 0.5f));
  p = __fmul2_rn(p, __fmul2_rn(delta, delta));
  const float2 q = __fmul2_rn(__ffma2_rn(delta, abar, make_float2(-c.x, -c.y)), inv_a);
  return make_float2(fabsf(x.x) < 0.5f ? p.x : q.x, fabsf(x.y) < 0.5f ? p.y : q.y);
}

// 1/a for the zero-order-hold factor (0 where a = 0: that state always takes the series branch).
__device__ __forceinline__ float zoh_inv(float a) { return a != 0.0f ? 1.0f / a : 0.0f; }

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// 16-byte asynchronous global->shared copy; bytes in [0, 16] are read, the rest is zero-filled.
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src, int src_bytes) {
  const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(gmem_src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace ssm
