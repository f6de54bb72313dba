// Selective scan forward for sm_103a: warp-specialised, four lanes per channel.
//
// What it computes (per batch row b, channel d, state n; sources cited in ssm_scan.h):
//   Delta_t = softplus(delta_t + dt_bias[d]);  Abar = exp(Delta_t A[d,n]);  h_t = Abar h_{t-1} + Delta_t B_t[n] u_t
//   y_t = sum_n C_t[n] h_t[n] + D[d] u_t;  out_t = y_t * silu(z_t);  last_state = h_{L-1}
// or, with the exact zero-order hold (ZOH), Delta_t B_t[n] replaced by (Abar - 1) / A[d,n] B_t[n].
//
// Why it looks like this.  On B300 the scan is not HBM-bound in practice: per element it needs 16
// MUFU ex2, ~64 FP32 lane-operations and a cross-lane readout, and a straightforward kernel spends
// its time in a chain of latency-bound phases (wait for the chunk, convert, per-element prologue,
// barrier, recurrence, readout reduction, epilogue) that one set of warps walks in turn.  This
// kernel gives the phases to different warps so that they overlap:
//  * PREP warps (4) own the HBM traffic and all per-element work.  They stream chunks of 32 steps
//    of u, delta, z, B, C with 16-byte cp.async into a two-stage raw ring (zero-filled past the
//    sequence end), convert B and C into float32 [t][n] tables, and compute, once per element,
//    Delta = softplus(delta + dt_bias), Delta*u, D*u and silu(z) into a two-stage table ring.
//  * RECURRENCE warps (R = NPAD/4) each own 32/R channels, four states per lane (lanes of a
//    quarter-warp share one n-group, so their B/C loads hit one address).  The float32 state lives
//    in registers for the whole sequence.  Per 16-step window the recurrence runs on float2 pairs
//    (mul/fma.f32x2) keeping the readout partials C.h in registers; the sum over the R lanes of a
//    channel is a reduce-scatter of warp shuffles (no shared-memory traffic: the kernel is bound by
//    the shared-memory data path, which its B, C and step-table loads already fill); lane (g, c)
//    then finishes 16/R consecutive steps of channel c, (y + D u) * silu(z), stored straight to HBM.
//  * Hand-off is by mbarriers in shared memory: table stage s is FULL once every prep thread has
//    arrived on it, EMPTY once every lane of the group's recurrence warps has.  Each recurrence
//    warp waits for FULL on its own, so the warps of a group are not re-aligned at every chunk
//    (aligned warps reach their window-end readouts together and leave the schedulers idle).  The
//    prep, which runs ahead and waits at almost every chunk, waits for EMPTY in one warp while the
//    other prep warps block on their own named barrier, and the waiting warp sleeps between tests,
//    so waiting costs the recurrence warps almost no issue slots.  Every wait is bounded (about a
//    second): one that gives up sets a CTA-wide abort flag that ends every other wait at once and
//    is counted in g_scan_wait_timeouts (ssm_wait_timeouts), so the kernel always ends.  The only
//    named barriers left are among the prep threads, which all run the same control flow.
//  * For dstate 9..16 (four recurrence warps, one warpgroup each) setmaxnreg moves registers from
//    the prep warpgroup (48) to the recurrence warpgroup (112), whose unrolled window is the long
//    pole; the kernel is launched at 80 registers per thread and the shares add up to that.
//  * Padded states (n >= dstate) have A = 0 and B = C = 0; padded steps (t >= seqlen) have
//    Delta = 0.  Both leave the state unchanged, so one code path serves every size.
//  * With a checkpoint buffer (the training forward), the recurrence lanes also store the state
//    at the start of every chunk, which is what the backward pass restarts from.
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
namespace {

constexpr int kChunk = kScanChunk;  // steps per chunk (the checkpoint interval)
constexpr int kWin = 16;    // steps per recurrence window (readout partials held in registers)
constexpr int kPrepWarps = 4;

// Register split of the four-recurrence-warp layout (dstate 9..16): the kernel is launched with
// kLaunchRegs per thread; the prep warpgroup gives registers back and the recurrence warpgroup,
// whose unrolled window is the long pole, takes them.  The shares add up to the launch total.
constexpr int kLaunchRegs = 80, kPrepRegs = 48, kRecRegs = 112;
static_assert(4 * kPrepRegs + 4 * kRecRegs == 8 * kLaunchRegs && kPrepWarps == 4,
              "setmaxnreg shares (one warpgroup each) must add up to the launch total");

// named barrier ids within a group's block of five (0 is __syncthreads): the one-time sync after
// the mbarriers are initialised, and the prep threads' own syncs
constexpr int kBarInit = 1, kBarPrep = 5;
// sleep between two tests of a hand-off barrier: the prep (ahead, waiting long) and the recurrence
// warps (rarely waiting, and then only briefly), in nanoseconds
constexpr unsigned kPrepBackoff = 256, kRecBackoff = 32;
// longest a hand-off wait may take before the kernel gives up on it, in SM clock cycles (~1 s)
constexpr long long kWaitLimit = 1LL << 31;

}  // namespace

// Hand-off waits of the forward kernels that gave up, since the library was loaded.
__device__ unsigned long long g_scan_wait_timeouts;

namespace {

template <typename T, int NPAD>
struct ScanCfg {
  static constexpr int R = NPAD / 4;                  // lanes per channel
  static constexpr int CWARPS = R;                    // recurrence warps: 32 channels per CTA
  static constexpr int NT = 32 * (CWARPS + kPrepWarps);
  static constexpr int PT = 32 * kPrepWarps;          // prep threads
  static constexpr int CPW = 32 / R;                  // channels per recurrence warp
  static constexpr int CPB = CPW * CWARPS;            // channels per CTA (32)
  static constexpr int EPV = 16 / sizeof(T);          // elements per 16-byte vector
  static constexpr int RS = kChunk + EPV;             // padded row stride (elements) of staged rows
  static constexpr int VPR = kChunk / EPV;            // 16-byte vectors per staged row
  static constexpr int ROWS = 3 * CPB + 2 * NPAD;     // u, delta, z rows, then B rows, then C rows
  static constexpr int PSS = CPB + 4;                 // row stride (float2) of the (Delta, Delta*u) table
  static constexpr int DSS = kChunk + 2;              // row stride (float2) of the (D*u, silu z) table
  static constexpr int OPL = kWin / R;                // outputs each lane finishes per window
  // shared memory map (bytes)
  static constexpr size_t kRawStage = size_t(ROWS) * RS * sizeof(T);
  static constexpr int kCOfs = kChunk * NPAD + 16;    // float offset of the C table after the B table
  static constexpr size_t kBCStage = size_t(kCOfs + kChunk * NPAD) * sizeof(float);  // Bs, Cs [CHUNK][NPAD]
  static constexpr size_t kPStage = size_t(kChunk) * PSS * sizeof(float2);      // Ps [CHUNK][PSS]
  static constexpr size_t kDSStage = size_t(CPB) * DSS * sizeof(float2);        // DS [CPB][DSS]
  static constexpr size_t kTabStage = kBCStage + kPStage + kDSStage;
  static constexpr size_t kRaw = 2 * kRawStage;
  static constexpr size_t kTab = 2 * kTabStage;
  static constexpr size_t kBarOfs = kRaw + kTab;                 // FULL0, FULL1, EMPTY0, EMPTY1 mbarriers
  static constexpr size_t kSmem = kBarOfs + 4 * sizeof(uint64_t);
  static_assert(kRawStage % 16 == 0 && kBCStage % 16 == 0 && kPStage % 16 == 0 && kDSStage % 16 == 0, "align");
  static_assert(OPL % 4 == 0 && kChunk % kWin == 0, "each lane finishes whole 16-byte units of the window");
  static_assert((RS * sizeof(T)) % 16 == 0 && kChunk % 8 == 0, "staged rows hold whole 16-byte vectors");
};

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <typename T>
__device__ __forceinline__ float2 load2(const T* p);  // two consecutive io elements as float32
template <>
__device__ __forceinline__ float2 load2<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 load2<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// Eight consecutive staged io elements (16-byte aligned) as float32, with 16-byte loads.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  const float4 lo = *reinterpret_cast<const float4*>(p), hi = *reinterpret_cast<const float4*>(p + 4);
  v[0] = lo.x, v[1] = lo.y, v[2] = lo.z, v[3] = lo.w, v[4] = hi.x, v[5] = hi.y, v[6] = hi.z, v[7] = hi.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    v[2 * k] = f.x, v[2 * k + 1] = f.y;
  }
}

// Store n consecutive outputs (n <= OPL valid ones of the OPL given) as io type.  With VEC the
// row is 16-byte aligned and its length a multiple of 16 bytes, so every 16-byte (or, for 8-byte
// groups, 8-byte) piece is either wholly inside the row or wholly past its end.
template <typename T, int OPL, bool VEC>
__device__ __forceinline__ void store_out(T* dst, const float (&v)[OPL], int n) {
  if constexpr (VEC && std::is_same<T, __nv_bfloat16>::value) {
    uint32_t w[OPL / 2];
#pragma unroll
    for (int j = 0; j < OPL / 2; ++j) {
      const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&p);
    }
    if constexpr (OPL == 4) {
      if (n >= 4) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else {
#pragma unroll
      for (int q = 0; q < OPL / 8; ++q)
        if (n >= 8 * q + 8)
          *reinterpret_cast<uint4*>(dst + 8 * q) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
  } else if constexpr (VEC) {
#pragma unroll
    for (int q = 0; q < OPL / 4; ++q)
      if (n >= 4 * q + 4)
        *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < OPL; ++j)
      if (j < n) dst[j] = from_f32<T>(v[j]);
  }
}

// One group of warps (4 prep + R recurrence) scanning the channels [d0, dlim) of batch row b, at
// most CPB of them, with its own shared-memory block `smem` (mbarriers included) and the named
// barriers bar0 + 1 .. bar0 + 5; tid is the thread's index within the group, abort the CTA's
// give-up flag.  A CTA of the plain kernel is one group.
template <typename T, int NPAD, bool VEC, bool ZOH>
__device__ __forceinline__ void scan_group(const ScanArgs& a, unsigned char* smem, const int tid, const int b,
                                           const int d0, const int dlim, const int bar0, volatile int* abort) {
  using Cfg = ScanCfg<T, NPAD>;
  constexpr int R = Cfg::R, CPW = Cfg::CPW, CPB = Cfg::CPB, EPV = Cfg::EPV, RS = Cfg::RS, VPR = Cfg::VPR;
  constexpr int NT = Cfg::NT, PT = Cfg::PT, ROWS = Cfg::ROWS, PSS = Cfg::PSS, DSS = Cfg::DSS, OPL = Cfg::OPL;
  constexpr int CWARPS = Cfg::CWARPS;

  T* raw = reinterpret_cast<T*>(smem);
  unsigned char* tab = smem + Cfg::kRaw;
  auto tabBs = [&](int s) { return reinterpret_cast<float*>(tab + s * Cfg::kTabStage); };
  auto tabCs = [&](int s) { return reinterpret_cast<float*>(tab + s * Cfg::kTabStage) + Cfg::kCOfs; };
  auto tabPs = [&](int s) { return reinterpret_cast<float2*>(tab + s * Cfg::kTabStage + Cfg::kBCStage); };
  auto tabDS = [&](int s) {
    return reinterpret_cast<float2*>(tab + s * Cfg::kTabStage + Cfg::kBCStage + Cfg::kPStage);
  };

  const int bPrep = kBarPrep + bar0;
  const int warp = tid >> 5, lane = tid & 31;
  const int L = a.seqlen, N = a.dstate;
  const bool has_z = a.z != nullptr;
  const int nchunks = (L + kChunk - 1) / kChunk;

  // mbarriers: FULL[s] completes when all PT prep threads have written table stage s, EMPTY[s]
  // when every lane of the recurrence warps holding a channel of the group is done reading it
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOfs);
  const int rec_warps = min(CWARPS, (dlim - d0 + CPW - 1) / CPW);
  if (tid == 0) {
    mbar_init(&mb[0], PT), mbar_init(&mb[1], PT);
    mbar_init(&mb[2], 32 * rec_warps), mbar_init(&mb[3], 32 * rec_warps);
  }
  bar_sync(kBarInit + bar0, NT);  // the group's mbarriers are initialised before anyone uses them

  if (warp >= CWARPS) {
    // ================================ prep warps ================================
    if constexpr (CWARPS == 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPrepRegs));
    const int ptid = tid - 32 * CWARPS;
    const int pw = warp - CWARPS;
    const int dim = a.dim;
    const bool softplus = a.softplus != 0;
    const T* __restrict__ gu = static_cast<const T*>(a.u);
    const T* __restrict__ gd = static_cast<const T*>(a.delta);
    const T* __restrict__ gz = static_cast<const T*>(a.z);
    const T* __restrict__ gB = static_cast<const T*>(a.B);
    const T* __restrict__ gC = static_cast<const T*>(a.C);

    // Global start of staged row r (u, delta, z rows by channel, then B and C rows by state);
    // ok = the row exists.  Rows of channels past dim and z rows without a gate are never used
    // by another channel, so they are not copied; B and C rows past dstate are zero-filled
    // (every channel reads them).
    auto row_src = [&](int r, bool& ok, bool& fill) -> const T* {
      if (r < 3 * CPB) {
        const int which = r / CPB, c = r % CPB;
        const T* base = which == 0 ? gu : (which == 1 ? gd : gz);
        ok = (d0 + c < dlim) && (which < 2 || has_z);
        fill = false;
        return ok ? base + (size_t(b) * dim + (d0 + c)) * L : gu;
      }
      const int rr = r - 3 * CPB;
      const int which = rr / NPAD, n = rr % NPAD;
      ok = n < N;
      fill = true;
      return ok ? (which == 0 ? gB : gC) + (size_t(b) * N + n) * L : gu;
    };

    // Each prep thread owns the same SLOTS 16-byte copy slots (row, column) in every chunk, so
    // their addresses are worked out once.
    constexpr int NV = ROWS * VPR;
    constexpr int SLOTS = (NV + PT - 1) / PT;
    const T* s_src[SLOTS];  // global address of the slot's first element in chunk 0
    int s_dst[SLOTS];       // element offset within a raw stage, -1 = nothing to copy
    int s_col[SLOTS];       // first step of the slot within a chunk
    bool s_ok[SLOTS];
    if constexpr (VEC) {
#pragma unroll
      for (int i = 0; i < SLOTS; ++i) {
        const int v = ptid + i * PT;
        const int r = v / VPR, j = v % VPR;
        bool ok = false, fill = false;
        const T* src = v < NV ? row_src(r, ok, fill) : gu;
        s_src[i] = ok ? src + j * EPV : gu;
        s_dst[i] = (v < NV && (ok || fill)) ? r * RS + j * EPV : -1;
        s_col[i] = j * EPV;
        s_ok[i] = ok;
      }
    }
    auto stage_load = [&](int stage, int t0) {
      T* dst = raw + size_t(stage) * ROWS * RS;
      if constexpr (VEC) {
#pragma unroll
        for (int i = 0; i < SLOTS; ++i) {
          if (s_dst[i] < 0) continue;
          // rows are 16-byte multiples, so a vector is wholly inside or wholly past the end;
          // a zero-byte copy only zero-fills, but its source must still be a valid address
          const bool in = s_ok[i] && t0 + s_col[i] < L;
          cp_async_16(dst + s_dst[i], in ? static_cast<const void*>(s_src[i] + t0) : gu, in ? 16 : 0);
        }
      } else {
        for (int e = ptid; e < ROWS * kChunk; e += PT) {
          const int r = e / kChunk, j = e % kChunk;
          bool ok, fill;
          const T* src = row_src(r, ok, fill);
          if (!ok && !fill) continue;
          const int t = t0 + j;
          dst[r * RS + j] = (ok && t < L) ? src[t] : from_f32<T>(0.0f);
        }
      }
    };

    // B, C conversion items: one item = 8 steps of one row.  Lanes 0..NPAD-1 of a group take the
    // B rows and the next NPAD lanes the C rows of the same steps; the C table is offset by 16
    // words so that both halves land in different banks.
    constexpr int SPI = 8;
    constexpr int NITEM = 2 * NPAD * (kChunk / SPI);
    constexpr int IPT = (NITEM + PT - 1) / PT;
    int c_src[IPT], c_dst[IPT];
#pragma unroll
    for (int m = 0; m < IPT; ++m) {
      const int e = ptid + m * PT;
      const int n = e % NPAD, which = (e / NPAD) % 2, q = e / (2 * NPAD);
      c_src[m] = e < NITEM ? (3 * CPB + which * NPAD + n) * RS + q * SPI : -1;
      c_dst[m] = which * Cfg::kCOfs + (q * SPI) * NPAD + n;
    }

    // prologue mapping: prep warp pw handles channels PCW*pw + (lane % PCW); the lanes lane/PCW +
    // PPL*i walk the step pairs of the chunk (conflict-free reads of the staged rows)
    constexpr int PCW = CPB / kPrepWarps;  // channels per prep warp (8)
    constexpr int PPL = 32 / PCW;          // step-pair lanes per channel (4)
    const int pcl = pw * PCW + (lane % PCW);
    const int tq = lane / PCW;
    const bool pch_ok = d0 + pcl < dlim;
    const float p_bias = (pch_ok && a.dt_bias) ? a.dt_bias[d0 + pcl] : 0.0f;
    const float p_D = (pch_ok && a.D) ? a.D[d0 + pcl] : 0.0f;
    const int r_ofs = pcl * RS + 2 * tq;     // element offset of this lane's first step pair in a row
    const int ps_ofs = 2 * tq * PSS + pcl;   // float2 offset of its first (Delta, Delta*u) entry
    const int ds_ofs = pcl * DSS + 2 * tq;   // float2 offset of its first (D*u, silu z) entry

    if (nchunks > 0) stage_load(0, 0);
    cp_async_commit();
    if (nchunks > 1) stage_load(1, kChunk);
    cp_async_commit();

    for (int k = 0; k < nchunks; ++k) {
      const int s = k & 1;
      const int t0 = k * kChunk;
      cp_async_wait<1>();           // this thread's copies of chunk k have landed
      // the recurrence warps are done with table stage s (their reads of chunk k - 2): one prep warp
      // waits, the others learn it from the named barrier below
      if (k >= 2 && pw == 0)
        mbar_wait(&mb[2 + s], ((k - 2) >> 1) & 1, abort, kWaitLimit, &g_scan_wait_timeouts, kPrepBackoff);
      bar_sync(bPrep, PT);          // every prep thread's copies have landed, and stage s is free

      const T* st = raw + size_t(s) * ROWS * RS;
      float* BCs = tabBs(s);
      float2* Ps = tabPs(s);
      float2* DS = tabDS(s);

#pragma unroll
      for (int m = 0; m < IPT; ++m) {
        if (c_src[m] < 0) continue;
        float v[SPI];
        load8<T>(st + c_src[m], v);
        float* dst = BCs + c_dst[m];
#pragma unroll
        for (int j = 0; j < SPI; ++j) dst[j * NPAD] = v[j];
      }

      // per-element work: Delta, Delta*u, D*u, silu(z), two steps per item.  Steps past the end
      // (and channels past dim) get Delta = 0, which leaves the state unchanged.
      const int lim = pch_ok ? L - t0 : 0;
      auto items = [&](auto masked) {
#pragma unroll
        for (int i = 0; i < kChunk / 2 / PPL; ++i) {
          const int o = 2 * PPL * i;
          const float2 uu = load2<T>(st + r_ofs + o);
          const float2 dr = load2<T>(st + CPB * RS + r_ofs + o);
          const float2 zz = load2<T>(st + 2 * CPB * RS + r_ofs + o);
          const float2 dx = __fadd2_rn(dr, f2(p_bias, p_bias));
          const float2 sp = softplus2(dx);
          float2 dl = softplus ? sp : dx;
          if constexpr (decltype(masked)::value) {
            const int t = 2 * tq + o;
            dl.x = t < lim ? dl.x : 0.0f;
            dl.y = t + 1 < lim ? dl.y : 0.0f;
          }
          // the recurrence's input factor: Delta*u, or u alone for the zero-order hold (whose
          // Bbar factor needs Delta and A together and is formed in the recurrence)
          const float2 du = ZOH ? uu : __fmul2_rn(dl, uu);
          const float2 Du = __fmul2_rn(f2(p_D, p_D), uu);
          const float2 sg = has_z ? silu2<std::is_same<T, __nv_bfloat16>::value>(zz) : f2(1.0f, 1.0f);
          Ps[ps_ofs + o * PSS] = f2(dl.x, du.x);
          Ps[ps_ofs + (o + 1) * PSS] = f2(dl.y, du.y);
          *reinterpret_cast<float4*>(DS + ds_ofs + o) = make_float4(Du.x, sg.x, Du.y, sg.y);
        }
      };
      if (lim >= kChunk)
        items(std::false_type{});
      else
        items(std::true_type{});

      bar_sync(bPrep, PT);               // every prep thread is done reading raw stage s
      mbar_arrive(&mb[s]);               // this thread's part of table stage s is written
      if (k + 2 < nchunks) stage_load(s, t0 + 2 * kChunk);
      cp_async_commit();
    }
    cp_async_wait<0>();
    return;
  }

  // ============================== recurrence warps ==============================
  if constexpr (CWARPS == 4) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRecRegs));
  // n-group major: the lanes of a quarter-warp (R = 4) share one n-group, so their B and C loads
  // hit one address; the R lanes of channel cw are cw, cw + CPW, ...
  const int cw = lane % CPW, g = lane / CPW;
  const int cl = warp * CPW + cw;  // this lane's channel within the CTA
  const int d = d0 + cl;
  const bool ch_ok = d < dlim;
  if (warp >= rec_warps) return;  // none of this warp's channels is in the group (not counted in EMPTY)

  float2 A01, A23, h01, h23, iA01, iA23;
  {
    float Av[4], hv[4], iv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * g + i;
      const bool ok = ch_ok && n < N;
      const float av = ok ? a.A[size_t(d) * N + n] : 0.0f;
      Av[i] = av * kLog2e;
      iv[i] = zoh_inv(av);
      hv[i] = (ok && a.h0) ? a.h0[(size_t(b) * a.dim + d) * N + n] : 0.0f;
    }
    A01 = f2(Av[0], Av[1]), A23 = f2(Av[2], Av[3]);
    iA01 = f2(iv[0], iv[1]), iA23 = f2(iv[2], iv[3]);
    h01 = f2(hv[0], hv[1]), h23 = f2(hv[2], hv[3]);
  }
  T* yrow = static_cast<T*>(a.y) + (size_t(b) * a.dim + (ch_ok ? d : 0)) * L;

  for (int k = 0; k < nchunks; ++k) {
    const int s = k & 1;
    const int t0 = k * kChunk;
    if (a.ckpt && ch_ok) {
      // the state at the start of chunk k, for the backward pass: [batch][chunk][dim][dstate]
      float* cp = a.ckpt + ((size_t(b) * nchunks + k) * a.dim + d) * N;
      const float hv[4] = {h01.x, h01.y, h23.x, h23.y};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * g + i < N) cp[4 * g + i] = hv[i];
    }
    mbar_wait(&mb[s], (k >> 1) & 1, abort, kWaitLimit, &g_scan_wait_timeouts, kRecBackoff);
    const float* Bs = tabBs(s);
    const float* Cs = tabCs(s);
    const float2* Ps = tabPs(s);
    const float2* DS = tabDS(s);

#pragma unroll 1
    for (int w = 0; w < kChunk; w += kWin) {
      float2 acc[kWin];
#pragma unroll
      for (int j = 0; j < kWin; ++j) {
        const int t = w + j;
        const float2 p = Ps[t * PSS + cl];
        const float4 bb = *reinterpret_cast<const float4*>(Bs + t * NPAD + 4 * g);
        const float4 cc = *reinterpret_cast<const float4*>(Cs + t * NPAD + 4 * g);
        const float2 dd = f2(p.x, p.x), uu = f2(p.y, p.y);
        const float2 g01 = __fmul2_rn(dd, A01), g23 = __fmul2_rn(dd, A23);
        const float2 a01 = f2(ex2_approx(g01.x), ex2_approx(g01.y));
        const float2 a23 = f2(ex2_approx(g23.x), ex2_approx(g23.y));
        if constexpr (ZOH) {
          // p.y is u here; Bbar*u = zoh_factor(Delta*A) * u * B
          const float2 ln2 = f2(kLn2, kLn2);
          const float2 c01 = zoh_factor2(__fmul2_rn(g01, ln2), a01, dd, iA01);
          const float2 c23 = zoh_factor2(__fmul2_rn(g23, ln2), a23, dd, iA23);
          h01 = __ffma2_rn(a01, h01, __fmul2_rn(c01, __fmul2_rn(uu, f2(bb.x, bb.y))));
          h23 = __ffma2_rn(a23, h23, __fmul2_rn(c23, __fmul2_rn(uu, f2(bb.z, bb.w))));
        } else {
          h01 = __ffma2_rn(a01, h01, __fmul2_rn(uu, f2(bb.x, bb.y)));
          h23 = __ffma2_rn(a23, h23, __fmul2_rn(uu, f2(bb.z, bb.w)));
        }
        acc[j] = __ffma2_rn(f2(cc.z, cc.w), h23, __fmul2_rn(f2(cc.x, cc.y), h01));
      }
      // sums over the R lanes of the channel (lanes cw, cw + CPW, ...) and the pair halves, by a
      // reduce-scatter of warp shuffles (which take no shared-memory bandwidth, the kernel's
      // tightest resource): in each round the lanes whose state-group bit is set keep the later
      // half of their steps and send the earlier half, the others the reverse.  Lane (g, cw) ends
      // with OPL consecutive steps of channel cl, starting at window step tb - w.
      float pv[kWin];
#pragma unroll
      for (int j = 0; j < kWin; ++j) pv[j] = acc[j].x + acc[j].y;
      float yv[OPL];
      int tb = w;  // first step (within the chunk) this lane finishes
      if constexpr (R == 1) {
#pragma unroll
        for (int j = 0; j < kWin; ++j) yv[j] = pv[j];
      } else {
        const bool b0 = g & 1;
        float k8[kWin / 2];
#pragma unroll
        for (int i = 0; i < kWin / 2; ++i) {
          const float snd = b0 ? pv[i] : pv[i + kWin / 2];
          const float kp = b0 ? pv[i + kWin / 2] : pv[i];
          k8[i] = kp + __shfl_xor_sync(0xffffffffu, snd, CPW);
        }
        tb += b0 ? kWin / 2 : 0;
        if constexpr (R == 2) {
#pragma unroll
          for (int i = 0; i < OPL; ++i) yv[i] = k8[i];
        } else {
          const bool b1 = (g >> 1) & 1;
#pragma unroll
          for (int i = 0; i < OPL; ++i) {
            const float snd = b1 ? k8[i] : k8[i + OPL];
            const float kp = b1 ? k8[i + OPL] : k8[i];
            yv[i] = kp + __shfl_xor_sync(0xffffffffu, snd, 2 * CPW);
          }
          tb += b1 ? OPL : 0;
        }
      }
      // epilogue: (y + D u) * silu(z) -> io type, straight to HBM
      float ov[OPL];
#pragma unroll
      for (int j = 0; j < OPL; j += 2) {
        const float4 ds = *reinterpret_cast<const float4*>(DS + cl * DSS + tb + j);
        const float2 o = __fmul2_rn(__fadd2_rn(f2(yv[j], yv[j + 1]), f2(ds.x, ds.z)), f2(ds.y, ds.w));
        ov[j] = o.x, ov[j + 1] = o.y;
      }
      const int tg = t0 + tb;  // first global step
      if (ch_ok) store_out<T, OPL, VEC>(yrow + tg, ov, L - tg);
    }
    mbar_arrive(&mb[2 + s]);  // this lane is done reading table stage s
  }

  if (a.last_state && ch_ok) {
    const float hv[4] = {h01.x, h01.y, h23.x, h23.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * g + i;
      if (n < N) a.last_state[(size_t(b) * a.dim + d) * N + n] = hv[i];
    }
  }
}

// The plain kernel: CTA blockIdx.x scans 32-channel block (blockIdx.x % blocks per row) of batch
// row blockIdx.x / blocks per row.
template <typename T, int NPAD, bool VEC, bool ZOH>
__global__ void __launch_bounds__(ScanCfg<T, NPAD>::NT, 3) scan_fwd_kernel(const ScanArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int CPB = ScanCfg<T, NPAD>::CPB;
  const int nblk_d = (a.dim + CPB - 1) / CPB;
  const int b = blockIdx.x / nblk_d;
  const int d0 = (blockIdx.x % nblk_d) * CPB;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  scan_group<T, NPAD, VEC, ZOH>(a, smem, threadIdx.x, b, d0, a.dim, 0, &abort_flag);
}

// The balanced form: one CTA per SM holding kFusedGroups groups, each on a channel range (8 to 32
// channels of one batch row) from a host plan that evens out the channels per SM.  With 32-channel
// CTAs an SM carries 64 or 96 channels when the total is not a multiple of 96 per SM; the plan
// gives every SM within 8 channels of the mean.  Plan entry: b << 16 | (d0 / 8) << 4 | (channels / 8),
// 0 for an empty group.
constexpr int kFusedGroups = 3;
constexpr int kMaxFusedCtas = 160;
struct FusedPlan {
  uint32_t e[kFusedGroups * kMaxFusedCtas];
};

template <typename T, int NPAD, bool VEC, bool ZOH>
__global__ void __launch_bounds__(kFusedGroups * ScanCfg<T, NPAD>::NT, 1)
    scan_fwd_fused_kernel(const ScanArgs a, const FusedPlan plan) {
  extern __shared__ __align__(16) unsigned char smem[];
  using Cfg = ScanCfg<T, NPAD>;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  const int grp = threadIdx.x / Cfg::NT;
  const uint32_t e = plan.e[blockIdx.x * kFusedGroups + grp];
  const int nch = int(e & 15u) * 8;
  if (nch == 0) return;  // an empty group: its warps leave, the other groups do not wait on them
  const int b = int(e >> 16), d0 = int((e >> 4) & 0xfffu) * 8;
  scan_group<T, NPAD, VEC, ZOH>(a, smem + grp * Cfg::kSmem, threadIdx.x - grp * Cfg::NT, b, d0,
                                min(a.dim, d0 + nch), 5 * grp, &abort_flag);
}

// Host plan for the balanced form: units of 8 channels, groups of at most 4 units inside one batch
// row, at most kFusedGroups groups per CTA, CTA c taking ceil(units left / CTAs left) units.
// Returns the CTA count, or 0 when the plan does not apply or does not lower the busiest SM's load
// below that of the plain kernel (32-channel CTAs spread over the SMs).
int make_fused_plan(const ScanArgs& a, int sms, FusedPlan& plan) {
  if (a.dim % 8 != 0 || a.batch >= (1 << 16) || a.dim / 8 >= (1 << 12) || sms <= 0 || sms > kMaxFusedCtas) return 0;
  const long long ur = a.dim / 8, units = (long long)a.batch * ur;
  if (units == 0 || units > (long long)sms * kFusedGroups * 4) return 0;
  const long long blocks = (long long)a.batch * ((a.dim + 31) / 32);
  const long long plain_max = 4 * ((blocks + sms - 1) / sms);  // units on the busiest SM, plain kernel
  long long left = units, row = 0, pos = 0, worst = 0;
  int ctas = 0;
  for (int c = 0; c < sms && left > 0; ++c) {
    const long long target = (left + (sms - c) - 1) / (sms - c);
    long long load = 0;
    for (int g = 0; g < kFusedGroups; ++g) {
      uint32_t entry = 0;
      if (load < target && row < a.batch) {
        const long long take = std::min(std::min(4LL, target - load), ur - pos);
        entry = uint32_t(row) << 16 | uint32_t(pos) << 4 | uint32_t(take);
        load += take, pos += take, left -= take;
        if (pos == ur) ++row, pos = 0;
      }
      plan.e[c * kFusedGroups + g] = entry;
    }
    worst = std::max(worst, load);
    ctas = c + 1;
  }
  return (left == 0 && worst < plain_max) ? ctas : 0;
}

// Once per device: the balanced kernel's shared-memory opt-in, and whether the build has the
// register count its setmaxnreg split was sized for (if not, the plain kernel runs).  Returns
// whether the balanced kernel may launch; err reports a failing CUDA call.
template <typename T, int NPAD, bool VEC, bool ZOH>
bool fused_ready(int dev, cudaError_t& err) {
  using Cfg = ScanCfg<T, NPAD>;
  auto kernel = scan_fwd_fused_kernel<T, NPAD, VEC, ZOH>;
  constexpr size_t kSmem = kFusedGroups * Cfg::kSmem;
  static std::atomic<uint64_t> configured{0}, usable{0};
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    if ((err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmem))) != cudaSuccess)
      return false;
    cudaFuncAttributes fa{};
    if ((err = cudaFuncGetAttributes(&fa, kernel)) != cudaSuccess) return false;
    if (fa.numRegs == kLaunchRegs) usable.fetch_or(bit, std::memory_order_acq_rel);
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  return (usable.load(std::memory_order_acquire) & bit) != 0;
}

// CTAs of the balanced form for `a` (bf16, dstate 9..16: three groups' shared memory fit one CTA),
// or 0 when the plain kernel runs instead (no plan, SSM_SCAN_VARIANT=quad_plain, or a build
// whose register count does not match the split).
template <typename T, int NPAD, bool VEC, bool ZOH>
int fused_ctas(const ScanArgs& a, FusedPlan& plan, int& dev, cudaError_t& err) {
  if constexpr (NPAD != 16 || !std::is_same<T, __nv_bfloat16>::value) {
    return 0;
  } else {
    const char* force = std::getenv("SSM_SCAN_VARIANT");
    if (force && std::strcmp(force, "quad_plain") == 0) return 0;
    int sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return 0;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return 0;
    const int ctas = make_fused_plan(a, sms, plan);
    if (ctas == 0) return 0;
    return fused_ready<T, NPAD, VEC, ZOH>(dev, err) ? ctas : 0;
  }
}

// Launches the balanced form when its plan applies; returns false when the plain kernel should run.
template <typename T, int NPAD, bool VEC, bool ZOH>
bool launch_fused(const ScanArgs& a, cudaStream_t stream, cudaError_t& err) {
  using Cfg = ScanCfg<T, NPAD>;
  FusedPlan plan;
  int dev = 0;
  const int ctas = fused_ctas<T, NPAD, VEC, ZOH>(a, plan, dev, err);
  if (err != cudaSuccess) return true;
  if (ctas == 0) return false;
  ScanArgs args = a;
  void* params[] = {&args, &plan};
  err = cudaLaunchKernel(reinterpret_cast<const void*>(scan_fwd_fused_kernel<T, NPAD, VEC, ZOH>), dim3(unsigned(ctas)),
                         dim3(kFusedGroups * Cfg::NT), params, kFusedGroups * Cfg::kSmem, stream);
  return true;
}

template <typename T, int NPAD, bool VEC, bool ZOH>
cudaError_t launch_cfg(const ScanArgs& a, cudaStream_t stream) {
  using Cfg = ScanCfg<T, NPAD>;
  {
    cudaError_t err = cudaSuccess;
    if (launch_fused<T, NPAD, VEC, ZOH>(a, stream, err)) return err;
  }
  auto kernel = scan_fwd_kernel<T, NPAD, VEC, ZOH>;
  // The dynamic shared-memory opt-in is a per-device function attribute; set it once per device.
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmem));
    if (err != cudaSuccess) return err;
    if constexpr (Cfg::CWARPS == 4) {
      // the setmaxnreg split assumes the launch allocation it was sized for; a build whose
      // register count differs would make the recurrence warps wait for registers forever
      cudaFuncAttributes fa{};
      err = cudaFuncGetAttributes(&fa, kernel);
      if (err != cudaSuccess) return err;
      if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidDeviceFunction;
    }
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

template <typename T, bool VEC, bool ZOH>
cudaError_t dispatch_npad(const ScanArgs& a, cudaStream_t stream) {
  if (a.dstate <= 4) return launch_cfg<T, 4, VEC, ZOH>(a, stream);
  if (a.dstate <= 8) return launch_cfg<T, 8, VEC, ZOH>(a, stream);
  return launch_cfg<T, 16, VEC, ZOH>(a, stream);
}

template <typename T, bool VEC>
cudaError_t dispatch_disc(const ScanArgs& a, cudaStream_t stream) {
  return a.zoh ? dispatch_npad<T, VEC, true>(a, stream) : dispatch_npad<T, VEC, false>(a, stream);
}

template <typename T>
bool rows_vectorisable(const ScanArgs& a) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return (size_t(a.seqlen) * sizeof(T)) % 16 == 0 && al(a.u) && al(a.delta) && al(a.z) && al(a.B) && al(a.C) &&
         al(a.y);
}


}  // namespace

cudaError_t launch_scan_fwd_quad(const ScanArgs& a, bool vec, cudaStream_t stream) {
  if (a.io == kF32)
    return vec ? dispatch_disc<float, true>(a, stream) : dispatch_disc<float, false>(a, stream);
  return vec ? dispatch_disc<__nv_bfloat16, true>(a, stream) : dispatch_disc<__nv_bfloat16, false>(a, stream);
}

cudaError_t scan_fwd_form(const ScanArgs& a, bool vec, int& form, int& ctas) {
  cudaError_t err = cudaSuccess;
  int c = 0, dev = 0;
  if (a.io == kBF16 && a.dstate > 8) {
    FusedPlan plan;
    c = vec ? (a.zoh ? fused_ctas<__nv_bfloat16, 16, true, true>(a, plan, dev, err)
                     : fused_ctas<__nv_bfloat16, 16, true, false>(a, plan, dev, err))
            : (a.zoh ? fused_ctas<__nv_bfloat16, 16, false, true>(a, plan, dev, err)
                     : fused_ctas<__nv_bfloat16, 16, false, false>(a, plan, dev, err));
    if (err != cudaSuccess) return err;
  }
  form = c > 0 ? kFormBalanced : kFormPlain;
  ctas = c > 0 ? c : int(std::min<long long>(0x7fffffffLL, (long long)((a.dim + 31) / 32) * a.batch));
  return cudaSuccess;
}

cudaError_t scan_wait_timeouts(unsigned long long& count) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  return cudaMemcpyFromSymbol(&count, g_scan_wait_timeouts, sizeof(count));
}

cudaError_t launch_scan_fwd(const ScanArgs& a, cudaStream_t stream) {
  const bool vec = a.io == kF32 ? rows_vectorisable<float>(a) : rows_vectorisable<__nv_bfloat16>(a);
  return launch_scan_fwd_quad(a, vec, stream);
}

}  // namespace ssm
