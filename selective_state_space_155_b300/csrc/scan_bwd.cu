// Backward pass of the selective scan for sm_103a, for either discretisation of B.
//
// Forward, per batch row b, channel d, state n (see scan_fwd.cu):
//   Delta_t = softplus(delta_t + dt_bias[d]),  a_t = exp(Delta_t A[d,n]),  h_t = a_t h_{t-1} + c_t B_t u_t
//   y_t = sum_n C_t h_t + D u_t,  out_t = y_t silu(z_t)
// with c_t = Delta_t (Delta*B form) or c_t = (a_t - 1) / A (exact zero-order hold, ZOH).
// Backward, for dout_t = dLoss/dout_t, with dy_t = dout_t silu(z_t) and the adjoint state
//   lambda_t = dy_t C_t + a_{t+1} lambda_{t+1}      (run from t = L-1 down to 0):
//   du_t     = dy_t D + sum_n lambda_t c_t B_t
//   dDelta_t = sum_n lambda_t (A a_t h_{t-1} + dc/dDelta B_t u_t),   ddelta_t = dDelta_t sigmoid(delta_t + dt_bias)
//   dA       = sum_{b,t} lambda_t (Delta_t a_t h_{t-1} + dc/dA B_t u_t),    dB_t = sum_d lambda_t c_t u_t
//   dC_t     = sum_d dy_t h_t,   dD = sum_{b,t} dy_t u_t,   dz_t = dout_t y_t silu'(z_t)
//   ddt_bias = sum_{b,t} ddelta_t,   dh0 = a_0 lambda_0
// where dc/dDelta = 1 and dc/dA = 0 in the Delta*B form, and dc/dDelta = a_t and
// dc/dA = (Delta_t a_t - c_t) / A under the hold (zoh_factor_da2 in device_math.cuh).
//
// Layout of the work.  A CTA owns 32 channels of one batch row; lane (g, cw) of warp w holds
// states 4g .. 4g+3 of channel 8w + cw (the forward's four-lanes-per-channel layout).  Chunks of
// 32 steps are processed last to first.  For each chunk all 128 threads stage the per-(channel,
// step) values (Delta, u, dy, the softplus and silu derivatives) and B, C into shared-memory
// tables from raw input rows that were copied into shared memory (16-byte cp.async when rows are
// 16-byte aligned) while the previous chunk was being computed, together with the four states the
// training forward checkpointed at the chunk's 8-step sub-chunk starts; then every lane walks the
// sub-chunks last to first: from the sub-chunk's checkpoint it recomputes the 8 states (and the
// readout y that dz needs) into registers, and runs the adjoint recurrence backwards over them.  Sums over a channel's 4 lanes take two
// shuffles (y) or two shuffles for the du and dDelta sums together (a reduce-scatter that leaves
// one of them on each lane); dB and dC, shared by all channels, are reduce-scattered over the 8
// channels of a warp by shuffles; a step's sums wait in registers until its sub-chunk ends, are
// then added across the warps in shared memory, and finally added to the float32 outputs with
// one atomic per (state, step) and CTA.  dA, dD and ddt_bias are added
// across CTAs the same way; the launcher zeroes these accumulated outputs first.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "device_math.cuh"
#include "internal.h"

namespace ssm {
namespace {

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

constexpr int kK = kScanChunk;  // steps per chunk
constexpr int kS = kCkptSteps;  // steps per register sub-chunk (the forward's checkpoint interval)
constexpr int kSub = kK / kS;
static_assert(kS == 8, "the adjoint's deferred sums are sized for 8-step sub-chunks");
constexpr int kCPB = 32;        // channels per CTA
constexpr int kThr = 128;       // four warps; four lanes per channel, four states per lane
constexpr int kTS = kK + 1;     // padded row stride of the per-(channel, step) tables
static_assert(kK % kS == 0 && kK == 32, "chunk layout");

struct __align__(16) BwdSmem {
  float Bs[kK][16];
  float Cs[kK][16];
  float acc[kK][2][16];  // dB, dC of the chunk, summed over the CTA's channels
  float dl[kCPB][kTS];   // Delta
  float uu[kCPB][kTS];   // u
  float dy[kCPB][kTS];   // dout * silu(z)  (dout without a gate)
  float sg[kCPB][kTS];   // dDelta/ddelta: sigmoid(delta + dt_bias) with softplus, else 1
  float qz[kCPB][kTS];   // dout * silu'(z)
  float yv[kCPB][kTS];   // y before the gate, recomputed
  float gu[kCPB][kTS];   // sum_n lambda B (Delta*B form) or sum_n lambda c B (hold)
  float pad[16];         // puts gd[c][t] 16 banks away from gu[c][t]: one store writes both
  float gd[kCPB][kTS];   // dDelta
};

// Raw input rows of one chunk, as copied from global memory.
template <typename T>
struct __align__(16) BwdRaw {
  static constexpr int kEPV = 16 / int(sizeof(T));  // elements per 16-byte copy
  static constexpr int kPPR = kK / kEPV;            // 16-byte copies per 32-step row
  static constexpr int kRSBC = kK + kEPV;           // B/C row stride, padded against bank conflicts
  T x[4][kCPB][kK];          // u, delta, z, dout
  T bc[2][16][kRSBC];        // B, C
  float ck[kSub][kCPB][16];  // the states at the chunk's sub-chunk starts
};

template <typename T>
constexpr size_t bwd_smem_bytes() {
  return sizeof(BwdSmem) + sizeof(BwdRaw<T>);
}

template <typename T, bool ZOH, bool VEC>
__global__ void __launch_bounds__(kThr, 3) scan_bwd_kernel(const ScanBwdArgs a) {
  extern __shared__ __align__(16) unsigned char smem_bytes[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(smem_bytes);
  using Raw = BwdRaw<T>;
  Raw& raw = *reinterpret_cast<Raw*>(smem_bytes + sizeof(BwdSmem));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int dim = a.dim, N = a.dstate, L = a.seqlen;
  const int nblk_d = (dim + kCPB - 1) / kCPB;
  const int b = blockIdx.x / nblk_d;
  const int d0 = (blockIdx.x % nblk_d) * kCPB;
  const int nchunks = (L + kK - 1) / kK;
  const int nck = (L + kS - 1) / kS;  // checkpoints per batch row
  const T* gu_ = static_cast<const T*>(a.u);
  const T* gdl = static_cast<const T*>(a.delta);
  const T* gz = static_cast<const T*>(a.z);
  const T* gdo = static_cast<const T*>(a.dout);
  const T* gB = static_cast<const T*>(a.B);
  const T* gC = static_cast<const T*>(a.C);

  // recurrence role
  const int cw = lane & 7, g = lane >> 3;
  const int cl = warp * 8 + cw, d = d0 + cl;
  const bool ch_ok = d < dim;
  float An[4], An2[4], iA[4], carry[4], dA[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = 4 * g + i;
    An[i] = (ch_ok && n < N) ? a.A[size_t(d) * N + n] : 0.0f;
    An2[i] = An[i] * kLog2e;
    iA[i] = ZOH ? zoh_inv(An[i]) : 0.0f;
    carry[i] = 0.0f;
    dA[i] = 0.0f;
  }
  const float2 ln2 = f2(kLn2, kLn2);
  // B's factor c_t (and a_t) of one state pair at step t: Bbar u = c (u B) as in the forward
  auto bbar_u = [&](float2 dl2, float2 gp, float2 ap, int p, float2 ub) {
    if constexpr (ZOH) {
      return __fmul2_rn(zoh_factor2(__fmul2_rn(gp, ln2), ap, dl2, f2(iA[2 * p], iA[2 * p + 1])), ub);
    } else {
      return ub;  // u already carries Delta
    }
  };
  // epilogue role: channel tid / 4, steps 8 (tid % 4) + j
  const int ec = tid >> 2, eq = tid & 3;
  const int ed = d0 + ec;
  const bool e_ok = ed < dim;
  const float eD = (e_ok && a.D) ? a.D[ed] : 0.0f;
  float accD = 0.0f, accBias = 0.0f;
  const bool has_z = gz != nullptr;

  // Copies of the raw inputs of chunk k (the next one to process, the previous one in time) into
  // the raw rows.  With VEC (every row 16-byte aligned) they are asynchronous 16-byte copies that
  // land while the current chunk is computed; otherwise plain loads and stores.  Copies past the
  // end of a row or of the channels are skipped: the staging never reads those elements.
  auto gx = [&](int x) { return x == 0 ? gu_ : x == 1 ? gdl : x == 2 ? gz : gdo; };  // x known at compile time
  const bool ck_vec = VEC && (N % 4) == 0 && (reinterpret_cast<uintptr_t>(a.ckpt) & 15u) == 0;
  auto issue = [&](int k) {
    const int t0 = k * kK;
    if constexpr (VEC) {
      constexpr int kXP = kCPB * Raw::kPPR;  // copies per input tensor
      static_assert(kXP % kThr == 0, "copy split");
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const T* src = gx(x);
        if (src == nullptr) continue;
#pragma unroll
        for (int i = 0; i < kXP / kThr; ++i) {
          const int p = tid + kThr * i;
          const int r = p / Raw::kPPR, j = p % Raw::kPPR;
          const int dd = d0 + r, t = t0 + j * Raw::kEPV;
          if (dd < dim && t < L) cp_async_16(&raw.x[x][r][j * Raw::kEPV], src + (size_t(b) * dim + dd) * L + t, 16);
        }
      }
      constexpr int kBP = 2 * 16 * Raw::kPPR;
      static_assert(kBP % kThr == 0, "copy split");
#pragma unroll
      for (int i = 0; i < kBP / kThr; ++i) {
        const int p = tid + kThr * i;
        const int which = p / (16 * Raw::kPPR), n = (p / Raw::kPPR) % 16, j = p % Raw::kPPR;
        const int t = t0 + j * Raw::kEPV;
        if (n < N && t < L)
          cp_async_16(&raw.bc[which][n][j * Raw::kEPV], (which ? gC : gB) + (size_t(b) * N + n) * L + t, 16);
      }
    } else {
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const T* src = gx(x);
        if (src == nullptr) continue;
        for (int e = tid; e < kCPB * kK; e += kThr) {
          const int r = e / kK, t = e % kK;
          const int dd = d0 + r, tg = t0 + t;
          if (dd < dim && tg < L) raw.x[x][r][t] = src[(size_t(b) * dim + dd) * L + tg];
        }
      }
      for (int e = tid; e < 2 * 16 * kK; e += kThr) {
        const int which = e / (16 * kK), n = (e / kK) % 16, t = e % kK;
        const int tg = t0 + t;
        if (n < N && tg < L) raw.bc[which][n][t] = (which ? gC : gB)[(size_t(b) * N + n) * L + tg];
      }
    }
#pragma unroll
    for (int sb = 0; sb < kSub; ++sb) {
      const int ci = k * kSub + sb;  // checkpoint index; sub-chunks past the sequence have none
      if (ci >= nck) continue;
      const float* ck = a.ckpt + (size_t(b) * nck + ci) * dim * size_t(N);
      if (ck_vec) {
        // one 16-byte copy per (channel, 4 states): 32 x 4 = kThr copies
        const int c = tid >> 2, q = tid & 3;
        if (d0 + c < dim && 4 * q < N) cp_async_16(&raw.ck[sb][c][4 * q], ck + size_t(d0 + c) * N + 4 * q, 16);
      } else {
        for (int e = tid; e < kCPB * 16; e += kThr) {
          const int c = e >> 4, n = e & 15;
          if (d0 + c < dim && n < N) raw.ck[sb][c][n] = ck[size_t(d0 + c) * N + n];
        }
      }
    }
    cp_async_commit();
  };
  issue(nchunks - 1);

  for (int k = nchunks - 1; k >= 0; --k) {
    const int t0 = k * kK;
    cp_async_wait<0>();  // this thread's copies of chunk k have landed
    __syncthreads();     // everyone's have, and the previous chunk is finished with every table
    // ---- stage the chunk's tables from the raw rows ----
    {
      const int t = tid & (kK - 1), tg = t0 + t;
#pragma unroll
      for (int j = 0; j < kCPB * kK / kThr; ++j) {
        const int c = (tid >> 5) + 4 * j, dd = d0 + c;
        float dl = 0.0f, u = 0.0f, dyv = 0.0f, sgv = 0.0f, qzv = 0.0f;
        if (dd < dim && tg < L) {
          u = to_f32<T>(raw.x[0][c][t]);
          const float raw_d = to_f32<T>(raw.x[1][c][t]) + (a.dt_bias ? a.dt_bias[dd] : 0.0f);
          if (a.softplus) {
            dl = softplus_f32(raw_d);
            sgv = rcp_approx(1.0f + ex2_approx(-raw_d * kLog2e));
          } else {
            dl = raw_d;
            sgv = 1.0f;
          }
          const float go = to_f32<T>(raw.x[3][c][t]);
          if (has_z) {
            const float zz = to_f32<T>(raw.x[2][c][t]);
            const float s = rcp_approx(1.0f + ex2_approx(-zz * kLog2e));
            dyv = go * (zz * s);
            qzv = go * (s * (1.0f + zz * (1.0f - s)));
          } else {
            dyv = go;
          }
        }
        sm.dl[c][t] = dl, sm.uu[c][t] = u, sm.dy[c][t] = dyv, sm.sg[c][t] = sgv, sm.qz[c][t] = qzv;
      }
      // consecutive threads take consecutive states of a step: conflict-free table stores
#pragma unroll
      for (int j = 0; j < 2 * 16 * kK / kThr; ++j) {
        const int e = tid + kThr * j;
        const int which = e / (16 * kK), r = e % (16 * kK), n = r % 16, tt = r / 16;
        (which ? sm.Cs : sm.Bs)[tt][n] = (n < N && t0 + tt < L) ? to_f32<T>(raw.bc[which][n][tt]) : 0.0f;
      }
    }
    for (int e = tid; e < kK * 2 * 16; e += kThr) (&sm.acc[0][0][0])[e] = 0.0f;
    // the sub-chunks' starting states, from the checkpoints (zero past the sequence's end)
    float hs[kSub][4];
#pragma unroll
    for (int sb = 0; sb < kSub; ++sb) {
      const float4 c4 = *reinterpret_cast<const float4*>(&raw.ck[sb][cl][4 * g]);  // conflict-free
      const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
      const bool in = ch_ok && t0 + sb * kS < L;
#pragma unroll
      for (int i = 0; i < 4; ++i) hs[sb][i] = (in && 4 * g + i < N) ? cv[i] : 0.0f;
    }
    __syncthreads();     // tables written; the raw rows are free
    if (k > 0) issue(k - 1);  // in flight while this chunk is computed

    // ---- recurrence role: sub-chunks last to first, adjoint recurrence backwards ----
    const int k1 = (cw >> 2) & 1, k2 = (cw >> 1) & 1, k3 = cw & 1;
#pragma unroll
    for (int sb = kSub - 1; sb >= 0; --sb) {
      float2 ht[kS][2];  // states after each step of the sub-chunk, as (0,1), (2,3) pairs
      {
        float2 h01 = f2(hs[sb][0], hs[sb][1]), h23 = f2(hs[sb][2], hs[sb][3]);
#pragma unroll
        for (int j = 0; j < kS; ++j) {
          const int t = sb * kS + j;
          const float dl = sm.dl[cl][t], du = ZOH ? sm.uu[cl][t] : dl * sm.uu[cl][t];
          const float4 bb = *reinterpret_cast<const float4*>(&sm.Bs[t][4 * g]);
          const float2 dl2 = f2(dl, dl), du2 = f2(du, du);
          const float2 g01 = __fmul2_rn(dl2, f2(An2[0], An2[1])), g23 = __fmul2_rn(dl2, f2(An2[2], An2[3]));
          const float2 a01 = f2(ex2_approx(g01.x), ex2_approx(g01.y)), a23 = f2(ex2_approx(g23.x), ex2_approx(g23.y));
          h01 = __ffma2_rn(a01, h01, bbar_u(dl2, g01, a01, 0, __fmul2_rn(du2, f2(bb.x, bb.y))));
          h23 = __ffma2_rn(a23, h23, bbar_u(dl2, g23, a23, 1, __fmul2_rn(du2, f2(bb.z, bb.w))));
          ht[j][0] = h01, ht[j][1] = h23;
          if (has_z) {  // y before the gate, for dz: the readout summed over the channel's 4 lanes
            const float4 cc = *reinterpret_cast<const float4*>(&sm.Cs[t][4 * g]);
            const float2 yp2 = __ffma2_rn(f2(cc.z, cc.w), h23, __fmul2_rn(f2(cc.x, cc.y), h01));
            float yp = yp2.x + yp2.y;
            yp += __shfl_xor_sync(0xffffffffu, yp, 8);
            yp += __shfl_xor_sync(0xffffffffu, yp, 16);
            if (g == 0) sm.yv[cl][t] = yp;
          }
        }
      }
      // Each step's dB/dC sum (and, in the Delta*B form, its du/dDelta sums) is kept in registers
      // and stored after the sub-chunk's steps, so that the stores and shared-memory atomics do
      // not hold back the loads of the next steps.  Under ZOH, whose arithmetic needs more live
      // registers, the du/dDelta sums are stored at once.
      constexpr bool kDeferG = !ZOH;
      float rr[kS], gg[kS];
#pragma unroll
      for (int j = kS - 1; j >= 0; --j) {
        const int t = sb * kS + j;
        const float dl = sm.dl[cl][t], u = sm.uu[cl][t], dyv = sm.dy[cl][t];
        const float4 bb = *reinterpret_cast<const float4*>(&sm.Bs[t][4 * g]);
        const float4 cc = *reinterpret_cast<const float4*>(&sm.Cs[t][4 * g]);
        const float2 dl2 = f2(dl, dl), du2 = f2(dl * u, dl * u), u2 = f2(u, u), dy2 = f2(dyv, dyv);
        const float2 bp[2] = {f2(bb.x, bb.y), f2(bb.z, bb.w)}, cp[2] = {f2(cc.x, cc.y), f2(cc.z, cc.w)};
        float2 gu2 = f2(0.0f, 0.0f), gd2 = f2(0.0f, 0.0f);
        float v[8];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          const float2 Ap = f2(An[2 * p], An[2 * p + 1]);
          const float2 gp = __fmul2_rn(dl2, f2(An2[2 * p], An2[2 * p + 1]));
          const float2 ap = f2(ex2_approx(gp.x), ex2_approx(gp.y));  // a_t, as in the recompute
          const float2 hp = j > 0 ? ht[j - 1][p] : f2(hs[sb][2 * p], hs[sb][2 * p + 1]);  // h_{t-1}
          const float2 lam = __ffma2_rn(dy2, cp[p], f2(carry[2 * p], carry[2 * p + 1]));
          const float2 ahp = __fmul2_rn(ap, hp);
          const float2 vc = __fmul2_rn(dy2, ht[j][p]);  // dC
          if constexpr (ZOH) {
            const float2 xp = __fmul2_rn(gp, ln2), ia = f2(iA[2 * p], iA[2 * p + 1]);
            const float2 cz = zoh_factor2(xp, ap, dl2, ia);
            const float2 lc = __fmul2_rn(lam, cz), bu = __fmul2_rn(bp[p], u2);
            const float2 vb = __fmul2_rn(lc, u2);  // dB = lambda c u
            v[2 * p] = vb.x, v[2 * p + 1] = vb.y, v[4 + 2 * p] = vc.x, v[4 + 2 * p + 1] = vc.y;
            gu2 = __ffma2_rn(lc, bp[p], gu2);
            // dc/dDelta = a: dDelta gets lambda a (A h_{t-1} + B u)
            gd2 = __ffma2_rn(lam, __fmul2_rn(ap, __ffma2_rn(Ap, hp, bu)), gd2);
            const float2 dcda = zoh_factor_da2(xp, ap, dl2, cz, ia);
            const float2 da = __ffma2_rn(lam, __ffma2_rn(dl2, ahp, __fmul2_rn(dcda, bu)), f2(dA[2 * p], dA[2 * p + 1]));
            dA[2 * p] = da.x, dA[2 * p + 1] = da.y;
          } else {
            const float2 vb = __fmul2_rn(lam, du2);  // dB
            v[2 * p] = vb.x, v[2 * p + 1] = vb.y, v[4 + 2 * p] = vc.x, v[4 + 2 * p + 1] = vc.y;
            gu2 = __ffma2_rn(lam, bp[p], gu2);
            gd2 = __ffma2_rn(lam, __ffma2_rn(Ap, ahp, __fmul2_rn(bp[p], u2)), gd2);
            const float2 da = __ffma2_rn(__fmul2_rn(lam, dl2), ahp, f2(dA[2 * p], dA[2 * p + 1]));
            dA[2 * p] = da.x, dA[2 * p + 1] = da.y;
          }
          const float2 cr = __fmul2_rn(lam, ap);
          carry[2 * p] = cr.x, carry[2 * p + 1] = cr.y;
        }
        const float gup = gu2.x + gu2.y, gdp = gd2.x + gd2.y;
        // sums over the channel's four lanes, reduce-scattered: lanes with even g end with the
        // du sum, lanes with odd g the dDelta sum
        const bool odd = g & 1;
        const float gs = (odd ? gdp : gup) + __shfl_xor_sync(0xffffffffu, odd ? gup : gdp, 8);
        gg[j] = gs + __shfl_xor_sync(0xffffffffu, gs, 16);
        if constexpr (!kDeferG) {
          if (g < 2) (odd ? sm.gd : sm.gu)[cl][t] = gg[j];
        }
        // dB, dC summed over the warp's 8 channels: reduce-scatter over cw, lane keeps value cw
        float w[4], x[2];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float send = k1 ? v[q] : v[4 + q], keep = k1 ? v[4 + q] : v[q];
          w[q] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float send = k2 ? w[q] : w[2 + q], keep = k2 ? w[2 + q] : w[q];
          x[q] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        const float send = k3 ? x[0] : x[1], keep = k3 ? x[1] : x[0];
        rr[j] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
      }
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        const int t = sb * kS + j;
        atomicAdd(&sm.acc[t][cw >> 2][4 * g + (cw & 3)], rr[j]);
        if constexpr (kDeferG) {
          if (g < 2) ((g & 1) ? sm.gd : sm.gu)[cl][t] = gg[j];
        }
      }
    }
    __syncthreads();

    // ---- epilogue: per-element gradients of the chunk, and its dB, dC ----
#pragma unroll
    for (int j = 0; j < kK / 4; ++j) {
      const int t = eq * (kK / 4) + j, tg = t0 + t;
      if (e_ok && tg < L) {
        const float dl = sm.dl[ec][t], u = sm.uu[ec][t], dyv = sm.dy[ec][t];
        // sum_n lambda c B: the Delta*B form leaves c = Delta out of the sum
        const float dut = fmaf(dyv, eD, ZOH ? sm.gu[ec][t] : dl * sm.gu[ec][t]);
        const float ddl = sm.gd[ec][t] * sm.sg[ec][t];
        const size_t off = (size_t(b) * dim + ed) * L + tg;
        static_cast<T*>(a.du)[off] = from_f32<T>(dut);
        static_cast<T*>(a.ddelta)[off] = from_f32<T>(ddl);
        // dz = dout silu'(z) y, with y = C.h + D u before the gate
        if (a.dz && has_z) static_cast<T*>(a.dz)[off] = from_f32<T>(sm.qz[ec][t] * fmaf(eD, u, sm.yv[ec][t]));
        accD = fmaf(dyv, u, accD);
        accBias += ddl;
      }
    }
    for (int e = tid; e < kK * 2 * 16; e += kThr) {
      const int t = e >> 5, which = (e >> 4) & 1, n = e & 15;
      const int tg = t0 + t;
      if (n < N && tg < L) atomicAdd((which ? a.dC : a.dB) + (size_t(b) * N + n) * L + tg, sm.acc[t][which][n]);
    }
  }

  if (ch_ok) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * g + i;
      if (n < N) {
        atomicAdd(a.dA + size_t(d) * N + n, dA[i]);
        if (a.dh0) a.dh0[(size_t(b) * dim + d) * N + n] = carry[i];
      }
    }
  }
  accD += __shfl_xor_sync(0xffffffffu, accD, 1);
  accD += __shfl_xor_sync(0xffffffffu, accD, 2);
  accBias += __shfl_xor_sync(0xffffffffu, accBias, 1);
  accBias += __shfl_xor_sync(0xffffffffu, accBias, 2);
  if (eq == 0 && e_ok) {
    if (a.dD && a.D) atomicAdd(a.dD + ed, accD);
    if (a.ddt_bias && a.dt_bias) atomicAdd(a.ddt_bias + ed, accBias);
  }
}

// Zero up to four float32 buffers (the gradients the backward accumulates with atomics).
struct ZeroSpans {
  float* p[4];
  long long n[4];
};

__global__ void __launch_bounds__(256) zero_kernel(const ZeroSpans z) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (int s = 0; s < 4; ++s)
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < z.n[s]; i += stride) z.p[s][i] = 0.0f;
}

// Rows of every per-(batch, channel) and per-(batch, state) input are 16-byte aligned.
template <typename T>
bool rows_vectorisable(const ScanBwdArgs& a) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return (size_t(a.seqlen) * sizeof(T)) % 16 == 0 && al(a.u) && al(a.delta) && al(a.z) && al(a.dout) && al(a.B) &&
         al(a.C);
}

template <typename T, bool ZOH, bool VEC>
cudaError_t launch_bwd(const ScanBwdArgs& a, long long nblk, cudaStream_t stream) {
  auto kernel = scan_bwd_kernel<T, ZOH, VEC>;
  constexpr size_t kSmem = bwd_smem_bytes<T>();
  // the dynamic shared-memory opt-in is a per-device function attribute; set it once per device
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem));
    if (err != cudaSuccess) return err;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  ScanBwdArgs args = a;
  void* params[] = {&args};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kernel), dim3(unsigned(nblk)), dim3(kThr), params, kSmem,
                          stream);
}

}  // namespace

cudaError_t launch_scan_bwd(const ScanBwdArgs& a, cudaStream_t stream) {
  ZeroSpans zs{};
  zs.p[0] = a.dA, zs.n[0] = (long long)a.dim * a.dstate;
  zs.p[1] = a.dB, zs.n[1] = (long long)a.batch * a.dstate * a.seqlen;
  zs.p[2] = a.dC, zs.n[2] = (long long)a.batch * a.dstate * a.seqlen;
  // dD and ddt_bias are zeroed only when they are accumulated
  float* small = (a.dD && a.D) ? a.dD : nullptr;
  zs.p[3] = small, zs.n[3] = small ? a.dim : 0;
  {
    void* params[] = {&zs};
    cudaError_t err = cudaLaunchKernel(reinterpret_cast<const void*>(zero_kernel), dim3(592), dim3(256), params, 0,
                                       stream);
    if (err != cudaSuccess) return err;
  }
  if (a.ddt_bias && a.dt_bias) {
    ZeroSpans zb{};
    zb.p[0] = a.ddt_bias, zb.n[0] = a.dim;
    void* params[] = {&zb};
    cudaError_t err = cudaLaunchKernel(reinterpret_cast<const void*>(zero_kernel), dim3(8), dim3(256), params, 0,
                                       stream);
    if (err != cudaSuccess) return err;
  }
  if (a.seqlen <= 0) {
    // no steps: the initial state's gradient is zero
    if (!a.dh0) return cudaSuccess;
    ZeroSpans zh{};
    zh.p[0] = a.dh0, zh.n[0] = (long long)a.batch * a.dim * a.dstate;
    void* params[] = {&zh};
    return cudaLaunchKernel(reinterpret_cast<const void*>(zero_kernel), dim3(592), dim3(256), params, 0, stream);
  }
  const long long nblk = (long long)((a.dim + kCPB - 1) / kCPB) * a.batch;
  if (nblk <= 0) return cudaSuccess;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (a.io == kF32) {
    const bool vec = rows_vectorisable<float>(a);
    if (a.zoh) return vec ? launch_bwd<float, true, true>(a, nblk, stream) : launch_bwd<float, true, false>(a, nblk, stream);
    return vec ? launch_bwd<float, false, true>(a, nblk, stream) : launch_bwd<float, false, false>(a, nblk, stream);
  }
  using bf = __nv_bfloat16;
  const bool vec = rows_vectorisable<bf>(a);
  if (a.zoh) return vec ? launch_bwd<bf, true, true>(a, nblk, stream) : launch_bwd<bf, true, false>(a, nblk, stream);
  return vec ? launch_bwd<bf, false, true>(a, nblk, stream) : launch_bwd<bf, false, false>(a, nblk, stream);
}

}  // namespace ssm
