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
//  * PREP warps (4) own the HBM traffic and all per-element work.  Tensor copies (TMA) bring u,
//    delta, z, B, C into a two-stage raw ring, two 32-step chunks per copy when the sequence is a
//    whole number of chunks (zero-filled past the sequence end); the prep converts B and C into
//    float32 [t][n] tables and computes, once per element, Delta = softplus(delta + dt_bias),
//    Delta*u, D*u and silu(z) into a two-stage table ring.
//  * RECURRENCE warps (R = NPAD/4) each own 32/R channels, four states per lane (lanes of a
//    quarter-warp share one n-group, so their B/C loads hit one address).  The float32 state lives
//    in registers for the whole sequence.  Per 16-step window the recurrence runs on float2 pairs
//    (mul/fma.f32x2) keeping the readout partials C.h in registers; the sum over the R lanes of a
//    channel is a reduce-scatter of warp shuffles (no shared-memory traffic: the shared-memory data
//    path is the recurrence's busiest, its B, C and step-table loads already fill most of it);
//    lane (g, c) then finishes 16/R consecutive steps of channel c, (y + D u) * silu(z), stored
//    straight to HBM.
//  * Hand-off is by mbarriers in shared memory: table stage s is FULL once the prep has written it
//    (one arrival after the prep threads' closing barrier), EMPTY once every recurrence warp of the
//    group has read it (one arrival per warp, after the warp's lanes have synchronised).  Each recurrence
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
//  * With a checkpoint buffer (the training forward, its own instantiation), the recurrence lanes
//    also store the state before every 8th step, which is what the backward pass restarts from.
//  * Few channels and a long sequence leave an SM one warp group, which is latency-bound.  The
//    split form then scans segments of the sequence side by side: a carry pass (the same groups
//    without C, z or output) gives each carry segment's end state from zero and its sum of Delta, a
//    small kernel folds them with the associative pair operator (a1, b1) o (a2, b2) =
//    (a1 a2, a2 b1 + b2) into the state entering each segment (the parallel associative scan of the
//    53ai.com Mamba article, section 3.3, applied once per segment), and the segment pass scans
//    every segment from it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "device_math.cuh"
#include "internal.h"
#include "scan_plan.h"

namespace ssm {
namespace {

constexpr int kChunk = kScanChunk;  // steps per chunk (the checkpoint interval)
constexpr int kWin = 16;    // steps per recurrence window (readout partials held in registers)
constexpr int kPrepWarps = 4;
constexpr int kUnitRows = 8;  // channels per balanced-plan unit (and per small tensor-copy box)

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

// Tensor maps (TMA descriptors) of the five streamed inputs: u, delta, z with rows batch*dim in
// boxes of 32 channels, B and C with rows batch*dstate in boxes of NPAD states.  With `pair` set
// (the sequence a whole number of chunks), each is a 3-D view [chunk][row][step of the chunk]
// and one copy brings two chunks, landing chunk-major ([chunk][row][step]); otherwise a 2-D view
// [row][step] with one chunk per copy (steps past the end read as zeros).  Passed by value as a
// kernel parameter; the z map is unused (zero) when there is no gate.
struct alignas(64) TmaMaps {
  CUtensorMap u, delta, z, B, C;
  int pair;
};

template <typename T, int NPAD>
struct ScanCfg {
  static constexpr int R = NPAD / 4;                  // lanes per channel
  static constexpr int CWARPS = R;                    // recurrence warps: 32 channels per CTA
  static constexpr int NT = 32 * (CWARPS + kPrepWarps);
  static constexpr int PT = 32 * kPrepWarps;          // prep threads
  static constexpr int CPW = 32 / R;                  // channels per recurrence warp
  static constexpr int CPB = CPW * CWARPS;            // channels per CTA (32)
  static constexpr int EPV = 16 / sizeof(T);          // elements per 16-byte vector
  static constexpr int VPR = kChunk / EPV;            // 16-byte vectors per staged row
  static constexpr int ROWS = 3 * CPB + 2 * NPAD;     // u, delta, z rows, then B rows, then C rows
  static constexpr int PSS = kChunk + 2;              // row stride (float2) of the (Delta, Delta*u) table
  static constexpr int DSS = kChunk + 2;              // row stride (float2) of the (D*u, silu z) table
  static constexpr int OPL = kWin / R;                // outputs each lane finishes per window
  // raw stage: room for SLOTS chunks as five tiles [slot][rows][kChunk] (u, delta, z, B, C); the
  // element offsets of the tiles and of one chunk slot within a tile
  static constexpr int SLOTS = sizeof(T) == 2 ? 2 : 1;
  static constexpr int kUTile = 0, kDTile = SLOTS * CPB * kChunk, kZTile = 2 * SLOTS * CPB * kChunk,
                       kBTile = 3 * SLOTS * CPB * kChunk, kCTile = kBTile + SLOTS * NPAD * kChunk;
  static constexpr int kXSlot = CPB * kChunk, kBCSlot = NPAD * kChunk;
  static constexpr uint32_t kXBytes = CPB * kChunk * sizeof(T), kBBytes = NPAD * kChunk * sizeof(T);
  // shared memory map (bytes)
  static constexpr size_t kRawStage = size_t(SLOTS) * ROWS * kChunk * sizeof(T);
  static constexpr int kCOfs = kChunk * NPAD + 16;    // float offset of the C table after the B table
  static constexpr size_t kBCStage = size_t(kCOfs + kChunk * NPAD) * sizeof(float);  // Bs, Cs [CHUNK][NPAD]
  static constexpr size_t kPStage = size_t(CPB) * PSS * sizeof(float2);         // Ps [CPB][PSS]
  static constexpr size_t kDSStage = size_t(CPB) * DSS * sizeof(float2);        // DS [CPB][DSS]
  static constexpr size_t kTabStage = kBCStage + kPStage + kDSStage;
  static constexpr size_t kRaw = 2 * kRawStage;
  static constexpr size_t kTab = 2 * kTabStage;
  // mbarriers: FULL0, FULL1 (tables written), EMPTY0, EMPTY1 (tables read), RAW0, RAW1 (raw chunk
  // landed); then the prep's copy decision word
  static constexpr size_t kBarOfs = kRaw + kTab;
  static constexpr size_t kSmem = (kBarOfs + 6 * sizeof(uint64_t) + 16 + 127) / 128 * 128;
  static_assert(kRawStage % 128 == 0 && kXBytes % 128 == 0 && kBBytes % 128 == 0,
                "tensor-copy destinations are 128-byte aligned");
  static_assert(kRawStage % 16 == 0 && kBCStage % 16 == 0 && kPStage % 16 == 0 && kDSStage % 16 == 0, "align");
  static_assert(OPL % 4 == 0 && kChunk % kWin == 0, "each lane finishes whole 16-byte units of the window");
  static_assert((kChunk * sizeof(T)) % 16 == 0, "staged rows hold whole 16-byte vectors");
};

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }

__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

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
// most CPB of them, over the chunks [kc0, kc1) of segment seg, with its own shared-memory block
// `smem` (mbarriers included) and the named barriers bar0 + 1 .. bar0 + 5; tid is the thread's index
// within the group, abort the CTA's give-up flag.  A CTA of the plain kernel is one group over the
// whole sequence.  SEGS: the group's range is a segment of a split sequence ([kc0, kc1), seg);
// otherwise the whole row (seg 0).  CARRY: the carry pass of a split sequence (state and
// step-size sum only: no C, z, readout or output).
template <typename T, int NPAD, bool VEC, bool ZOH, bool CK, bool SEGS = false, bool CARRY = false>
__device__ __forceinline__ void scan_group(const ScanArgs& a, const TmaMaps& maps, unsigned char* smem, const int tid,
                                           const int b, const int d0, const int dlim, const int seg, const int kc0,
                                           const int kc1, const int bar0, volatile int* abort) {
  using Cfg = ScanCfg<T, NPAD>;
  constexpr int R = Cfg::R, CPW = Cfg::CPW, CPB = Cfg::CPB, EPV = Cfg::EPV, VPR = Cfg::VPR;
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
  const bool has_z = !CARRY && a.z != nullptr;
  // The group's chunk count and first step.  For a segment they are kept in the group's shared
  // words and read where used (a few loads per chunk), not held in registers across the loops: both
  // warp roles are at their register limits, and for whole rows they are constants or
  // kernel-parameter expressions the compiler recomputes for free.
  volatile int* gvals = reinterpret_cast<volatile int*>(smem + Cfg::kBarOfs + 6 * sizeof(uint64_t)) + 1;
  if (SEGS && tid == 0) gvals[0] = kc1 - kc0, gvals[1] = kc0 * kChunk;  // read after the init barrier
  auto n_chunks = [&]() -> int { return SEGS ? gvals[0] : (L + kChunk - 1) / kChunk; };
  auto t_first = [&]() -> int { return SEGS ? gvals[1] : 0; };

  // mbarriers: FULL[s] completes when the prep threads have written table stage s (one arrival
  // after their closing barrier), EMPTY[s] when every recurrence warp holding a channel of the
  // group is done reading it
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOfs);
  const int rec_warps = min(CWARPS, (dlim - d0 + CPW - 1) / CPW);
  if (tid == 0) {
    mbar_init(&mb[0], 1), mbar_init(&mb[1], 1);  // FULL: one arrival after the prep's closing barrier
    mbar_init(&mb[2], rec_warps), mbar_init(&mb[3], rec_warps);  // EMPTY: one arrival per recurrence warp
    mbar_init(&mb[4], 1), mbar_init(&mb[5], 1);  // RAW: one expect-tx arrival each
    fence_mbar_init();
  }
  bar_sync(kBarInit + bar0, NT);  // the group's mbarriers are initialised before anyone uses them

  if (warp >= CWARPS) {
    // ================================ prep warps ================================
    if constexpr (CWARPS == 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPrepRegs));
    const int ptid = tid - 32 * CWARPS;
    const int pw = warp - CWARPS;
    const int dim = a.dim;
    const bool softplus = a.softplus != 0;

    // A raw stage holds G chunks (G = 2 with paired copies, else 1) as five dense tiles: u, delta,
    // z rows of the group's 32 channel slots, then the NPAD B and C rows of batch row b.  On the
    // 16-byte path they arrive by tensor copies (TMA), whose completion the stage's RAW mbarrier
    // counts; rows past a tensor's end and steps past the sequence end arrive as zeros.  Channel
    // slots past the group's range hold other channels' rows and are ignored (their Delta and D
    // are 0 and their lanes store nothing); B and C rows past dstate are set to 0 in the
    // conversion.  A copy takes its issuing thread a few hundred cycles (the SM's copy unit takes
    // instructions one at a time), so the five copies of a stage are spread over the prep warps'
    // lane 0: warp 0 copies B and C, warps 1, 2, 3 copy u, delta and z.  Before any of them is
    // issued, ptid 0 has arrived on the stage's RAW barrier with the stage's byte count, so the
    // barrier's transaction count never runs ahead of its arrival.
    const bool pair = VEC && Cfg::SLOTS == 2 && maps.pair != 0;
    const int lg = pair ? 1 : 0;  // log2 of the chunks per raw stage
    const uint32_t stage_bytes = uint32_t((has_z ? 3 : 2) * Cfg::kXBytes + (CARRY ? 1 : 2) * Cfg::kBBytes) << lg;
    auto issue_copies = [&](int stage, int t0) {  // lane 0 of every prep warp
      T* dst = raw + size_t(stage) * Cfg::SLOTS * ROWS * kChunk;
      uint64_t* rb = &mb[4 + stage];
      const int c0 = t0 / kChunk;
      if (pw == 0) {
        if (pair) {
          tma_load_3d(dst + Cfg::kBTile, &maps.B, 0, b * N, c0, rb);
          if (!CARRY) tma_load_3d(dst + Cfg::kCTile, &maps.C, 0, b * N, c0, rb);
        } else {
          tma_load_2d(dst + Cfg::kBTile, &maps.B, t0, b * N, rb);
          if (!CARRY) tma_load_2d(dst + Cfg::kCTile, &maps.C, t0, b * N, rb);
        }
      } else if (pw < 3 || has_z) {
        const CUtensorMap* m = pw == 1 ? &maps.u : (pw == 2 ? &maps.delta : &maps.z);
        T* tile = dst + (pw - 1) * Cfg::SLOTS * CPB * kChunk;
        if (pair)
          tma_load_3d(tile, m, 0, b * dim + d0, c0, rb);
        else
          tma_load_2d(tile, m, t0, b * dim + d0, rb);
      }
    };
    // element-wise copy of one chunk into slot 0 of a stage by every prep thread (rows not 16-byte
    // aligned)
    auto stage_copy = [&](int stage, int t0) {
      T* dst = raw + size_t(stage) * Cfg::SLOTS * ROWS * kChunk;
      const T* gu = static_cast<const T*>(a.u);
      const T* gd = static_cast<const T*>(a.delta);
      const T* gz = static_cast<const T*>(a.z);
      const T* gB = static_cast<const T*>(a.B);
      const T* gC = static_cast<const T*>(a.C);
      for (int e = ptid; e < ROWS * kChunk; e += PT) {
        const int r = e / kChunk, j = e % kChunk, t = t0 + j;
        T v = from_f32<T>(0.0f);
        int o;
        if (r < 3 * CPB) {
          const int which = r / CPB, c = r % CPB;
          const T* base = which == 0 ? gu : (which == 1 ? gd : gz);
          if (d0 + c < dlim && (which < 2 || has_z) && t < L) v = base[(size_t(b) * dim + d0 + c) * L + t];
          o = which * Cfg::SLOTS * CPB * kChunk + c * kChunk + j;
        } else {
          const int rr = r - 3 * CPB, which = rr / NPAD, n = rr % NPAD;
          if (n < N && t < L) v = (which == 0 ? gB : gC)[(size_t(b) * N + n) * L + t];
          o = (which == 0 ? Cfg::kBTile : Cfg::kCTile) + n * kChunk + j;
        }
        dst[o] = v;
      }
    };

    // B, C conversion items: one 16-byte vector (EPV steps) of one row.  Lanes 0..NPAD-1 take the B
    // rows and the next NPAD lanes the C rows; each lane reads vector (q + rotation) of its row, a
    // rotation by row that puts the eight rows of a quarter-warp on different banks of the dense
    // stage (bf16 rows are 64 bytes, two to a bank line).
    constexpr int NITEM = 2 * NPAD * VPR;
    constexpr int IPT = (NITEM + PT - 1) / PT;
    int c_src[IPT], c_dst[IPT];
    bool c_ok[IPT];
#pragma unroll
    for (int m = 0; m < IPT; ++m) {
      const int e = ptid + m * PT;
      const int n = e % NPAD, which = (e / NPAD) % 2, q = e / (2 * NPAD);
      const int qr = (q + (sizeof(T) == 2 ? (n >> 1) : n)) & (VPR - 1);
      c_src[m] = e < NITEM && (!CARRY || which == 0) ? (which == 0 ? Cfg::kBTile : Cfg::kCTile) + n * kChunk + qr * EPV
                                                     : -1;
      c_dst[m] = which * Cfg::kCOfs + (qr * EPV) * NPAD + n;
      c_ok[m] = n < N;
    }

    // Element items: (channel, step pair), item e = ptid + PT i covering channel e / 16 and steps
    // 2 (e % 16), 2 (e % 16) + 1, so that a warp reads two channels' rows of one chunk: 32 lanes on 32
    // different banks.  Each thread keeps the same step pair and IPE channels.
    constexpr int IPE = CPB * (kChunk / 2) / PT;
    static_assert(IPE * PT == CPB * (kChunk / 2), "whole element items per prep thread");
    const int ep = ptid % (kChunk / 2);  // step pair
    const int ech0 = ptid / (kChunk / 2);  // first channel; item i takes channel ech0 + i * PT / 16
    constexpr int ECH = PT / (kChunk / 2);
    float e_bias[IPE], e_D[IPE];
#pragma unroll
    for (int i = 0; i < IPE; ++i) {
      const int c = d0 + ech0 + i * ECH;
      e_bias[i] = (c < dlim && a.dt_bias) ? a.dt_bias[c] : 0.0f;
      e_D[i] = (!CARRY && c < dlim && a.D) ? a.D[c] : 0.0f;
    }

    // Copies in flight, tracked by ptid 0: the raw-stage use (chunk >> lg) whose copies into raw
    // stage 0 / 1 have been issued but not yet seen complete, or -1.  Whether a stage is refilled
    // is decided once, by ptid 0 before the closing barrier of the stage's last chunk, and read by
    // every issuing lane after it: only after the stage's last copies were seen complete and
    // while no wait has given up, so that no copy lands on one still in flight and every issued
    // copy belongs to a counted phase.  Before the CTA exits, ptid 0 waits once more for copies
    // still in flight.
    volatile int* decide = reinterpret_cast<volatile int*>(smem + Cfg::kBarOfs + 6 * sizeof(uint64_t));
    const bool tma_ok = (smem_u32(raw) & 127u) == 0;  // tensor copies need a 128-byte aligned destination
    auto n_stages = [&]() { return (n_chunks() + (1 << lg) - 1) >> lg; };  // raw-stage uses
    int pend0 = -1, pend1 = -1;
    if (VEC && !tma_ok && ptid == 0) {
      *abort = 1;  // give up at once rather than copy
      atomicAdd(&g_scan_wait_timeouts, 1ull);
    }
    if (VEC && tma_ok) {
      if (ptid == 0) {
        if (n_stages() > 0) mbar_arrive_expect_tx(&mb[4], stage_bytes), pend0 = 0;
        if (n_stages() > 1) mbar_arrive_expect_tx(&mb[5], stage_bytes), pend1 = 1;
      }
      bar_sync(bPrep, PT);
      if (lane == 0) {
        if (n_stages() > 0) issue_copies(0, t_first());
        if (n_stages() > 1) issue_copies(1, t_first() + (kChunk << lg));
      }
    }

    for (int k = 0; k < n_chunks(); ++k) {
      const int s = k & 1;
      const int t0 = t_first() + k * kChunk;
      const int su = k >> lg, rs = su & 1;   // raw-stage use and raw stage of chunk k
      const int slot = k & ((1 << lg) - 1);  // its slot within the stage
      if (VEC) {
        // one prep warp waits for the raw chunk and for a free table stage; the others learn both
        // from the named barrier below (waiting warps there take no issue slots)
        if (pw == 0) {
          if (slot == 0 && mbar_wait(&mb[4 + rs], (su >> 1) & 1, abort, kWaitLimit, &g_scan_wait_timeouts, kPrepBackoff))
            (rs ? pend1 : pend0) = -1;
          if (k >= 2)
            mbar_wait(&mb[2 + s], ((k - 2) >> 1) & 1, abort, kWaitLimit, &g_scan_wait_timeouts, kPrepBackoff);
        }
      } else {
        stage_copy(rs, t0);
        if (pw == 0 && k >= 2)
          mbar_wait(&mb[2 + s], ((k - 2) >> 1) & 1, abort, kWaitLimit, &g_scan_wait_timeouts, kPrepBackoff);
      }
      bar_sync(bPrep, PT);  // raw chunk k is in its stage for every prep thread, and table stage s is free

      const T* st = raw + size_t(rs) * Cfg::SLOTS * ROWS * kChunk;
      const int xo = slot * Cfg::kXSlot, bo = slot * Cfg::kBCSlot;  // this chunk's slot in the tiles
      float* BCs = tabBs(s);
      float2* Ps = tabPs(s);
      float2* DS = tabDS(s);

#pragma unroll
      for (int m = 0; m < IPT; ++m) {
        if (c_src[m] < 0) continue;
        float v[EPV];
        if constexpr (sizeof(T) == 2) {
          float w8[8];
          load8<T>(st + bo + c_src[m], w8);
#pragma unroll
          for (int j = 0; j < EPV; ++j) v[j] = w8[j];
        } else {
          const float4 w4 = *reinterpret_cast<const float4*>(st + bo + c_src[m]);
          v[0] = w4.x, v[1] = w4.y, v[2] = w4.z, v[3] = w4.w;
        }
        float* dst = BCs + c_dst[m];
#pragma unroll
        for (int j = 0; j < EPV; ++j) dst[j * NPAD] = c_ok[m] ? v[j] : 0.0f;
      }

      // per-element work: Delta, Delta*u (u alone for the zero-order hold, whose Bbar factor needs
      // Delta and A together and is formed in the recurrence), D*u, silu(z).  Steps past the end
      // and channels past the group's range get Delta = 0, which leaves the state unchanged.
      const int lim = L - t0;
#pragma unroll
      for (int i = 0; i < IPE; ++i) {
        const int ch = ech0 + i * ECH;
        const int o = ch * kChunk + 2 * ep;
        const float2 uu = load2<T>(st + Cfg::kUTile + xo + o);
        const float2 dr = load2<T>(st + Cfg::kDTile + xo + o);
        const float2 dx = __fadd2_rn(dr, f2(e_bias[i], e_bias[i]));
        float2 dl = softplus ? softplus2(dx) : dx;
        const int lim_c = d0 + ch < dlim ? lim : 0;
        dl.x = 2 * ep < lim_c ? dl.x : 0.0f;
        dl.y = 2 * ep + 1 < lim_c ? dl.y : 0.0f;
        const float2 du = ZOH ? uu : __fmul2_rn(dl, uu);
        *reinterpret_cast<float4*>(Ps + ch * PSS + 2 * ep) = make_float4(dl.x, du.x, dl.y, du.y);
        if constexpr (!CARRY) {
          const float2 Du = __fmul2_rn(f2(e_D[i], e_D[i]), uu);
          const float2 sg = has_z ? silu2<std::is_same<T, __nv_bfloat16>::value>(load2<T>(st + Cfg::kZTile + xo + o))
                                  : f2(1.0f, 1.0f);
          *reinterpret_cast<float4*>(DS + ch * DSS + 2 * ep) = make_float4(Du.x, sg.x, Du.y, sg.y);
        }
      }

      const bool last_of_stage = slot == (1 << lg) - 1 || k == n_chunks() - 1;
      if (VEC && ptid == 0 && last_of_stage) {
        const bool refill = su + 2 < n_stages() && (rs ? pend1 : pend0) < 0 && !*abort;
        if (refill) mbar_arrive_expect_tx(&mb[4 + rs], stage_bytes), (rs ? pend1 : pend0) = su + 2;
        *decide = refill ? 1 : 0;
      }
      bar_sync(bPrep, PT);  // every prep thread is done reading chunk k; the decision is visible
      if (ptid == 0) mbar_arrive(&mb[s]);  // table stage s is written (the barrier above ordered every prep write)
      if (VEC && lane == 0 && last_of_stage && *decide) issue_copies(rs, t_first() + (su + 2) * (kChunk << lg));
    }
    if (VEC && ptid == 0) {  // these last waits ignore the CTA's give-up flag
      if (pend0 >= 0) mbar_wait(&mb[4], (pend0 >> 1) & 1, nullptr, kWaitLimit, &g_scan_wait_timeouts, kPrepBackoff);
      if (pend1 >= 0) mbar_wait(&mb[5], (pend1 >> 1) & 1, nullptr, kWaitLimit, &g_scan_wait_timeouts, kPrepBackoff);
    }
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
      // the state the group starts from: h0 for the first segment; for a later one of a split
      // sequence, zero in the carry pass and in the full pass the state its carries combined to
      // (the combine kernel left it in the last carry slot before the segment)
      float hs = 0.0f;
      if (ok && seg == 0 && a.h0) hs = a.h0[(size_t(b) * a.dim + d) * N + n];
      if (!CARRY && ok && seg > 0)
        hs = a.carry_h[((size_t(seg * a.seg_carries - 1) * a.batch + b) * a.dim + d) * N + n];
      hv[i] = hs;
    }
    A01 = f2(Av[0], Av[1]), A23 = f2(Av[2], Av[3]);
    iA01 = f2(iv[0], iv[1]), iA23 = f2(iv[2], iv[3]);
    h01 = f2(hv[0], hv[1]), h23 = f2(hv[2], hv[3]);
  }
  float dsum = 0.0f;  // the carry pass: sum of this channel's Delta over the segment
  // the output row from the group's first step on, and the steps left in the row from there
  T* yrow = static_cast<T*>(a.y) + (size_t(b) * a.dim + (ch_ok ? d : 0)) * L + t_first();

  // two chunks per iteration: more independent work for the scheduler around the hand-offs (not
  // with the zero-order hold, whose longer step body would then outgrow the instruction cache)
  constexpr int kChunkUnroll = ZOH ? 1 : 2;
  // checkpoints for the backward pass, [batch][ceil(L / kCkptSteps)][dim][dstate]: the state
  // before every kCkptSteps-th step (null when not requested, or for a lane without a channel)
  const int nck = (L + kCkptSteps - 1) / kCkptSteps;
  float* const ckrow = (CK && ch_ok) ? a.ckpt + (size_t(b) * nck * a.dim + d) * N + 4 * g : nullptr;
  const size_t ckstride = size_t(a.dim) * N;  // between consecutive checkpoints of this channel
  const int nst = min(4, N - 4 * g);          // this lane's real states
  // one 16-byte store per lane when its four states are real and the rows 16-byte aligned
  const bool ck16 = CK && nst == 4 && N % 4 == 0 && (reinterpret_cast<uintptr_t>(a.ckpt) & 15u) == 0;
  auto checkpoint = [&](int tg) {
    if (ckrow != nullptr && tg < L) {
      float* cp = ckrow + size_t(tg / kCkptSteps) * ckstride;
      if (ck16) {
        *reinterpret_cast<float4*>(cp) = make_float4(h01.x, h01.y, h23.x, h23.y);
      } else {
        const float hv[4] = {h01.x, h01.y, h23.x, h23.y};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (i < nst) cp[i] = hv[i];
      }
    }
  };

#pragma unroll kChunkUnroll
  for (int k = 0; k < n_chunks(); ++k) {
    const int s = k & 1;
    const int t0 = k * kChunk;  // from the group's first step
    mbar_wait(&mb[s], (k >> 1) & 1, abort, kWaitLimit, &g_scan_wait_timeouts, kRecBackoff);
    const float* Bs = tabBs(s);
    const float* Cs = tabCs(s);
    const float2* Ps = tabPs(s);
    const float2* DS = tabDS(s);

    if constexpr (CARRY) {
      // state and step-size sum only
#pragma unroll
      for (int t = 0; t < kChunk; ++t) {
        const float2 p = Ps[cl * PSS + t];
        const float4 bb = *reinterpret_cast<const float4*>(Bs + t * NPAD + 4 * g);
        const float2 dd = f2(p.x, p.x), uu = f2(p.y, p.y);
        const float2 g01 = __fmul2_rn(dd, A01), g23 = __fmul2_rn(dd, A23);
        const float2 a01 = f2(ex2_approx(g01.x), ex2_approx(g01.y));
        const float2 a23 = f2(ex2_approx(g23.x), ex2_approx(g23.y));
        if constexpr (ZOH) {
          const float2 c01 = zoh_factor2_log2(g01, a01, dd, iA01);
          const float2 c23 = zoh_factor2_log2(g23, a23, dd, iA23);
          h01 = __ffma2_rn(a01, h01, __fmul2_rn(c01, __fmul2_rn(uu, f2(bb.x, bb.y))));
          h23 = __ffma2_rn(a23, h23, __fmul2_rn(c23, __fmul2_rn(uu, f2(bb.z, bb.w))));
        } else {
          h01 = __ffma2_rn(a01, h01, __fmul2_rn(uu, f2(bb.x, bb.y)));
          h23 = __ffma2_rn(a23, h23, __fmul2_rn(uu, f2(bb.z, bb.w)));
        }
        dsum += p.x;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&mb[2 + s]);
      continue;
    }

    // both windows of the chunk unrolled: the first window's readout reduction and epilogue (a
    // chain of dependent shuffles) then overlap the second window's loads and exponentials
#pragma unroll
    for (int w = 0; w < kChunk; w += kWin) {
      float2 acc[kWin];
#pragma unroll
      for (int j = 0; j < kWin; ++j) {
        const int t = w + j;
        if constexpr (CK) {
          if (j % kCkptSteps == 0) checkpoint(t_first() + t0 + t);
        }
        const float2 p = Ps[cl * PSS + t];
        const float4 bb = *reinterpret_cast<const float4*>(Bs + t * NPAD + 4 * g);
        const float4 cc = *reinterpret_cast<const float4*>(Cs + t * NPAD + 4 * g);
        const float2 dd = f2(p.x, p.x), uu = f2(p.y, p.y);
        const float2 g01 = __fmul2_rn(dd, A01), g23 = __fmul2_rn(dd, A23);
        const float2 a01 = f2(ex2_approx(g01.x), ex2_approx(g01.y));
        const float2 a23 = f2(ex2_approx(g23.x), ex2_approx(g23.y));
        if constexpr (ZOH) {
          // p.y is u here; Bbar*u = zoh_factor(Delta*A) * u * B, from the base-2 exponent g
          const float2 c01 = zoh_factor2_log2(g01, a01, dd, iA01);
          const float2 c23 = zoh_factor2_log2(g23, a23, dd, iA23);
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
      const int tg = t0 + tb;  // first step, from the group's first
      if (ch_ok) store_out<T, OPL, VEC>(yrow + tg, ov, L - t_first() - tg);
    }
    __syncwarp();  // every lane of the warp is done reading table stage s ...
    if (lane == 0) mbar_arrive(&mb[2 + s]);  // ... which one arrival (release) then reports
  }

  const float hv[4] = {h01.x, h01.y, h23.x, h23.y};
  if constexpr (CARRY) {
    if (ch_ok) {
      const size_t row = (size_t(seg) * a.batch + b) * a.dim + d;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = 4 * g + i;
        if (n < N) a.carry_h[row * N + n] = hv[i];
      }
      if (g == 0) a.carry_d[row] = dsum;
    }
  } else if (a.last_state && ch_ok && n_chunks() * kChunk >= L - t_first()) {  // the last segment ends the row
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * g + i;
      if (n < N) a.last_state[(size_t(b) * a.dim + d) * N + n] = hv[i];
    }
  }
}

// The plain kernel: CTA blockIdx.x scans 32-channel block (blockIdx.x % blocks per row) of batch
// row blockIdx.x / blocks per row.
template <typename T, int NPAD, bool VEC, bool ZOH, bool CK>
__global__ void __launch_bounds__(ScanCfg<T, NPAD>::NT, 3)
    scan_fwd_kernel(const ScanArgs a, const __grid_constant__ TmaMaps maps) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int CPB = ScanCfg<T, NPAD>::CPB;
  const int nblk_d = (a.dim + CPB - 1) / CPB;
  const int b = blockIdx.x / nblk_d;
  const int d0 = (blockIdx.x % nblk_d) * CPB;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  scan_group<T, NPAD, VEC, ZOH, CK>(a, maps, smem, threadIdx.x, b, d0, a.dim, 0, 0, 0, 0, &abort_flag);
}

// The carry combine of a split sequence, one thread per (batch row, channel, state): carry slot j
// holds (S_j, h_j), the step-size sum and the end state (from zero; slot 0 from h0) of carry segment
// j, and the segment's decay is the product of its Abar, exp(A S_j).  Folding the slots left to right
// with the associative pair operator (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2) leaves in slot j the
// state after carry segment j, from which the next segment starts; only the running state is kept.
__global__ void __launch_bounds__(256) scan_carry_combine_kernel(const ScanArgs a, int ncarry, long long first) {
  const long long i = first + (long long)blockIdx.x * blockDim.x + threadIdx.x;  // from the split channels on
  const long long per = (long long)a.batch * a.dim * a.dstate;
  if (i >= per) return;
  const long long row = i / a.dstate;  // b * dim + d
  const int d = int(row % a.dim), n = int(i - row * a.dstate);
  const float al = a.A[size_t(d) * a.dstate + n] * kLog2e;
  float h = a.carry_h[i];
  const long long rows = (long long)a.batch * a.dim;
  // the slots' loads, eight at a time, ahead of the dependent chain and its stores
  constexpr int kBatch = 8;
  for (int j0 = 1; j0 < ncarry; j0 += kBatch) {
    float sd[kBatch], he[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int j = j0 + k;
      sd[k] = j < ncarry ? a.carry_d[j * rows + row] : 0.0f;
      he[k] = j < ncarry ? a.carry_h[j * per + i] : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int j = j0 + k;
      if (j < ncarry) {
        h = __fmaf_rn(ex2_approx(al * sd[k]), h, he[k]);
        a.carry_h[j * per + i] = h;
      }
    }
  }
}

// What one launch of the balanced form scans: whole rows, the segments of a split sequence (full
// pass), or its carry segments (carry pass).  Whole rows are their own instantiation, without the
// segment decode, which costs the unsplit kernel registers.
enum PassMode { kWhole = 0, kSegments = 1, kCarries = 2 };

template <typename T, int NPAD, bool VEC, bool ZOH, bool CK, int MODE>
__global__ void __launch_bounds__(kFusedGroups * ScanCfg<T, NPAD>::NT, 1)
    scan_fwd_fused_kernel(const ScanArgs a, const __grid_constant__ TmaMaps maps, const FusedPlan plan) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Cfg = ScanCfg<T, NPAD>;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  const int grp = threadIdx.x / Cfg::NT;
  const uint32_t e = plan.e[blockIdx.x * kFusedGroups + grp];
  const int nch = int(e & 15u) * 8;
  if (nch == 0) return;  // an empty group: its warps leave, the other groups do not wait on them
  const int d0 = int((e >> 4) & 0xfffu) * 8;
  int b = int(e >> 16), seg = 0, kc0 = 0, kc1 = 0;
  if (MODE != kWhole) {
    const int nck = (a.seqlen + kChunk - 1) / kChunk;
    seg = int(e >> kSegShift), b &= kMaxSplitBatch - 1;
    kc0 = seg * (a.seg_len / kChunk), kc1 = min(nck, kc0 + a.seg_len / kChunk);
  }
  scan_group<T, NPAD, VEC, ZOH, CK, MODE != kWhole, MODE == kCarries>(
      a, maps, smem + grp * Cfg::kSmem, threadIdx.x - grp * Cfg::NT, b, d0, min(a.dim, d0 + nch), seg, kc0, kc1,
      5 * grp, &abort_flag);
}

// The driver's tensor-map encoder, looked up once through the runtime (no link against the
// driver library); null if the driver does not offer it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// One map of io type T over a tensor [rows][L] with boxes of box_rows rows.  pair == false: a 2-D
// view [rows][L] with boxes of kChunk steps (steps and rows outside the tensor read as zeros).
// pair == true (L a multiple of kChunk): a 3-D view [L / kChunk][rows][kChunk] (the chunk axis
// strides kChunk elements, the row axis L), so that one box of two chunks lands chunk-major.
// The 128-byte L2 promotion brings in whole lines of which a chunk reads part, so the next chunk
// of the same rows finds them in L2.
template <typename T>
cudaError_t encode_map(CUtensorMap& m, const void* base, long long rows, int L, int box_rows, bool pair) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint32_t elem[3] = {1, 1, 1};
  CUresult r;
  if (pair) {
    const cuuint64_t dims[3] = {cuuint64_t(kChunk), cuuint64_t(rows), cuuint64_t(L / kChunk)};
    const cuuint64_t strides[2] = {cuuint64_t(L) * sizeof(T), cuuint64_t(kChunk) * sizeof(T)};
    const cuuint32_t box[3] = {cuuint32_t(kChunk), cuuint32_t(box_rows), 2};
    r = enc(&m, dt, 3, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[2] = {cuuint64_t(L), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(L) * sizeof(T)};
    const cuuint32_t box[2] = {cuuint32_t(kChunk), cuuint32_t(box_rows)};
    r = enc(&m, dt, 2, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The five maps of a call on the 16-byte path (rows 16-byte aligned, row counts below 2^31):
// paired two-chunk copies when the io type is bf16 and the sequence a whole number of chunks,
// else one chunk per copy.
template <typename T, int NPAD>
cudaError_t encode_maps(const ScanArgs& a, TmaMaps& m) {
  const long long rows = (long long)a.batch * a.dim, brows = (long long)a.batch * a.dstate;
  const int xr = ScanCfg<T, NPAD>::CPB;
  for (int pair = ScanCfg<T, NPAD>::SLOTS == 2 && a.seqlen % kChunk == 0 ? 1 : 0; pair >= 0; --pair) {
    const bool p = pair != 0;
    m.pair = pair;
    if (encode_map<T>(m.u, a.u, rows, a.seqlen, xr, p) == cudaSuccess &&
        encode_map<T>(m.delta, a.delta, rows, a.seqlen, xr, p) == cudaSuccess &&
        (!a.z || encode_map<T>(m.z, a.z, rows, a.seqlen, xr, p) == cudaSuccess) &&
        encode_map<T>(m.B, a.B, brows, a.seqlen, NPAD, p) == cudaSuccess &&
        encode_map<T>(m.C, a.C, brows, a.seqlen, NPAD, p) == cudaSuccess)
      return cudaSuccess;
  }
  return cudaErrorInvalidValue;
}

// Once per device: the balanced kernel's shared-memory opt-in, and whether the build has the
// register count its setmaxnreg split was sized for (if not, the plain kernel runs).  Returns
// whether the balanced kernel may launch; err reports a failing CUDA call.
template <typename T, int NPAD, bool VEC, bool ZOH, bool CK, int MODE>
bool fused_ready(int dev, cudaError_t& err) {
  using Cfg = ScanCfg<T, NPAD>;
  auto kernel = scan_fwd_fused_kernel<T, NPAD, VEC, ZOH, CK, MODE>;
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

// The current device and its SM count.
cudaError_t device_sms(int& dev, int& sms) {
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  return cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
}

bool balanced_allowed() {
  const char* force = std::getenv("SSM_SCAN_VARIANT");
  return !(force && std::strcmp(force, "quad_plain") == 0);
}

// CTAs of the balanced form for `a` over `rows` plan rows (bf16, dstate 9..16: three groups'
// shared memory fit one CTA), or 0 when it does not run (no plan, SSM_SCAN_VARIANT=quad_plain, or
// a build whose register count does not match the setmaxnreg split).
template <typename T, int NPAD, bool VEC, bool ZOH, bool CK, int MODE = kWhole>
int fused_ctas(const ScanArgs& a, long long rows, FusedPlan& plan, int& dev, cudaError_t& err) {
  static_assert(MODE == kWhole || (VEC && !CK), "the split runs on the 16-byte path without checkpoints");
  if constexpr (NPAD != 16 || !std::is_same<T, __nv_bfloat16>::value) {
    return 0;
  } else {
    if (!balanced_allowed()) return 0;
    int sms = 0;
    if ((err = device_sms(dev, sms)) != cudaSuccess) return 0;
    const int ctas = make_fused_plan(a, rows, sms, plan, MODE == kWhole);
    if (ctas == 0) return 0;
    return fused_ready<T, NPAD, VEC, ZOH, CK, MODE>(dev, err) ? ctas : 0;
  }
}

template <typename T, int NPAD, bool VEC, bool ZOH, bool CK, int MODE>
cudaError_t launch_fused_plan(const ScanArgs& a, const TmaMaps& maps, FusedPlan& plan, int ctas,
                              cudaStream_t stream) {
  using Cfg = ScanCfg<T, NPAD>;
  ScanArgs args = a;
  TmaMaps m = maps;
  void* params[] = {&args, &m, &plan};
  return cudaLaunchKernel(reinterpret_cast<const void*>(scan_fwd_fused_kernel<T, NPAD, VEC, ZOH, CK, MODE>),
                          dim3(unsigned(ctas)), dim3(kFusedGroups * Cfg::NT), params, kFusedGroups * Cfg::kSmem,
                          stream);
}

// Launches the balanced form when its plan applies; returns false when the plain kernel should run.
template <typename T, int NPAD, bool VEC, bool ZOH, bool CK>
bool launch_fused(const ScanArgs& a, const TmaMaps& maps, cudaStream_t stream, cudaError_t& err) {
  if constexpr (NPAD != 16 || !std::is_same<T, __nv_bfloat16>::value) {
    return false;  // the balanced form is built for bf16 with dstate 9..16 only
  } else {
    FusedPlan plan;
    int dev = 0;
    const int ctas = fused_ctas<T, NPAD, VEC, ZOH, CK>(a, a.batch, plan, dev, err);
    if (err != cudaSuccess) return true;
    if (ctas == 0) return false;
    err = launch_fused_plan<T, NPAD, VEC, ZOH, CK, kWhole>(a, maps, plan, ctas, stream);
    return true;
  }
}

// The split for `a` on the current device, with both passes' plans; false when the scan runs
// unsplit.
template <typename T, int NPAD, bool ZOH>
bool split_plans(const ScanArgs& a, SplitPlan& sp, FusedPlan& pw, int& cw, FusedPlan& p1, int& c1, FusedPlan& p2,
                 int& c2, cudaError_t& err) {
  if constexpr (NPAD != 16 || !std::is_same<T, __nv_bfloat16>::value) {
    return false;
  } else {
    int dev = 0, sms = 0;
    if (!balanced_allowed() || (err = device_sms(dev, sms)) != cudaSuccess) return false;
    if (!make_split_plans(a, sms, sp, pw, cw, p1, c1, p2, c2)) return false;
    return fused_ready<T, NPAD, true, ZOH, false, kCarries>(dev, err) &&
           fused_ready<T, NPAD, true, ZOH, false, kSegments>(dev, err);
  }
}

// The plain kernel over its first nblk CTAs (32-channel blocks in batch-row order).
template <typename T, int NPAD, bool VEC, bool ZOH, bool CK>
cudaError_t launch_plain(const ScanArgs& a, const TmaMaps& maps, long long nblk, cudaStream_t stream) {
  using Cfg = ScanCfg<T, NPAD>;
  auto kernel = scan_fwd_kernel<T, NPAD, VEC, ZOH, CK>;
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
  if (nblk <= 0) return cudaSuccess;
  if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ScanArgs args = a;
  TmaMaps m = maps;
  void* params[] = {&args, &m};
  return cudaLaunchKernel(reinterpret_cast<const void*>(kernel), dim3(unsigned(nblk)), dim3(Cfg::NT), params,
                          Cfg::kSmem, stream);
}

// Runs the split scan when it applies (the 16-byte path, no checkpoints), with its carry buffers
// in the caller's workspace (a.ws_given: the split runs only if a.ws holds SplitPlan's
// workspace_bytes) or else in a stream-ordered allocation freed after the launches.  Returns false
// when the scan should run unsplit.
template <typename T, int NPAD, bool ZOH>
bool launch_split(const ScanArgs& a, const TmaMaps& maps, cudaStream_t stream, cudaError_t& err) {
  if constexpr (NPAD != 16 || !std::is_same<T, __nv_bfloat16>::value) {
    return false;
  } else {
    SplitPlan sp;
    FusedPlan pw, p1, p2;
    int cw = 0, c1 = 0, c2 = 0;
    if (!split_plans<T, NPAD, ZOH>(a, sp, pw, cw, p1, c1, p2, c2, err)) return err != cudaSuccess;
    void* buf = nullptr;
    if (a.ws_given) {
      if (!a.ws || a.ws_bytes < sp.workspace_bytes) return false;  // no room: unsplit
      buf = a.ws;
    } else if (cudaMallocAsync(&buf, sp.workspace_bytes, stream) != cudaSuccess) {
      (void)cudaGetLastError();  // the unsplit scan runs instead
      return false;
    }
    ScanArgs c = a;
    c.carry_h = static_cast<float*>(buf);
    c.carry_d = c.carry_h + size_t(sp.ncarry) * a.batch * a.dim * a.dstate;
    c.seg_len = sp.carry_len, c.seg_carries = 0;
    // a tail split first scans the whole rows, one full group per SM: the plain kernel's first cw
    // 32-channel blocks are exactly the whole-row plan's groups (one per SM; a lone group runs ~3 %
    // faster in the plain kernel's CTA than in the balanced kernel's)
    if (cw > 0) err = launch_plain<T, NPAD, true, ZOH, false>(a, maps, cw, stream);
    if (err == cudaSuccess) err = launch_fused_plan<T, NPAD, true, ZOH, false, kCarries>(c, maps, p1, c1, stream);
    if (err == cudaSuccess) {
      // the carried states: every channel, or those of the tail of the last batch row
      long long first = ((long long)(a.batch - 1) * a.dim + 8LL * sp.tail_p0) * a.dstate;
      if (sp.whole_groups == 0) first = 0;
      const long long n = (long long)a.batch * a.dim * a.dstate - first;
      int ncarry = sp.ncarry;
      void* params[] = {&c, &ncarry, &first};
      err = cudaLaunchKernel(reinterpret_cast<const void*>(scan_carry_combine_kernel), dim3(unsigned((n + 255) / 256)),
                             dim3(256), params, 0, stream);
    }
    if (err == cudaSuccess) {
      c.seg_len = sp.seg_len, c.seg_carries = sp.carries_per_seg;
      err = launch_fused_plan<T, NPAD, true, ZOH, false, kSegments>(c, maps, p2, c2, stream);
    }
    if (!a.ws_given) {
      const cudaError_t ferr = cudaFreeAsync(buf, stream);
      if (err == cudaSuccess) err = ferr;
    }
    return true;
  }
}

template <typename T, int NPAD, bool VEC, bool ZOH, bool CK>
cudaError_t launch_cfg(const ScanArgs& a, cudaStream_t stream) {
  using Cfg = ScanCfg<T, NPAD>;
  TmaMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if constexpr (VEC) {
    // a shape the tensor-map encoder rejects runs the element-wise staging instead
    if (encode_maps<T, NPAD>(a, maps) != cudaSuccess) return launch_cfg<T, NPAD, false, ZOH, CK>(a, stream);
  }
  {
    cudaError_t err = cudaSuccess;
    if constexpr (VEC && !CK) {
      if (launch_split<T, NPAD, ZOH>(a, maps, stream, err)) return err;
    }
    if (launch_fused<T, NPAD, VEC, ZOH, CK>(a, maps, stream, err)) return err;
  }
  return launch_plain<T, NPAD, VEC, ZOH, CK>(a, maps, (long long)((a.dim + Cfg::CPB - 1) / Cfg::CPB) * a.batch,
                                             stream);
}

template <typename T, bool VEC, bool ZOH, bool CK>
cudaError_t dispatch_npad(const ScanArgs& a, cudaStream_t stream) {
  if (a.dstate <= 4) return launch_cfg<T, 4, VEC, ZOH, CK>(a, stream);
  if (a.dstate <= 8) return launch_cfg<T, 8, VEC, ZOH, CK>(a, stream);
  return launch_cfg<T, 16, VEC, ZOH, CK>(a, stream);
}

// The training forward (checkpoints requested) is its own instantiation, so that the inference
// kernels carry no checkpoint code in their unrolled windows.
template <typename T, bool VEC>
cudaError_t dispatch_disc(const ScanArgs& a, cudaStream_t stream) {
  if (a.ckpt) return a.zoh ? dispatch_npad<T, VEC, true, true>(a, stream) : dispatch_npad<T, VEC, false, true>(a, stream);
  return a.zoh ? dispatch_npad<T, VEC, true, false>(a, stream) : dispatch_npad<T, VEC, false, false>(a, stream);
}

// The 16-byte path: a non-empty sequence, every row 16-byte aligned (tensor copies in, vector
// stores out), and row indices that fit the copies' signed 32-bit coordinates.
template <typename T>
bool rows_vectorisable(const ScanArgs& a) {
  auto al = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  return a.seqlen > 0 && (size_t(a.seqlen) * sizeof(T)) % 16 == 0 && al(a.u) && al(a.delta) && al(a.z) && al(a.B) && al(a.C) &&
         al(a.y) && (long long)a.batch * a.dim < (1LL << 31) && (long long)a.batch * a.dstate < (1LL << 31);
}

// The split for `a` and the grid of its full pass, or segs = 0.
cudaError_t split_form(const ScanArgs& a, bool vec, SplitPlan& p, int& ctas) {
  cudaError_t err = cudaSuccess;
  p = SplitPlan{};
  ctas = 0;
  if (vec && a.io == kBF16 && a.dstate > 8 && !a.ckpt) {
    FusedPlan pw, p1, p2;
    int cw = 0, c1 = 0;
    const bool split = a.zoh ? split_plans<__nv_bfloat16, 16, true>(a, p, pw, cw, p1, c1, p2, ctas, err)
                             : split_plans<__nv_bfloat16, 16, false>(a, p, pw, cw, p1, c1, p2, ctas, err);
    if (!split) p = SplitPlan{}, ctas = 0;
  }
  return err;
}

}  // namespace

cudaError_t launch_scan_fwd_quad(const ScanArgs& a, bool vec, cudaStream_t stream) {
  if (a.io == kF32)
    return vec ? dispatch_disc<float, true>(a, stream) : dispatch_disc<float, false>(a, stream);
  return vec ? dispatch_disc<__nv_bfloat16, true>(a, stream) : dispatch_disc<__nv_bfloat16, false>(a, stream);
}

cudaError_t scan_fwd_split(const ScanArgs& a, bool vec, SplitPlan& p) {
  int ctas = 0;
  return split_form(a, vec, p, ctas);
}

cudaError_t scan_fwd_form(const ScanArgs& a, bool vec, int& form, int& ctas) {
  cudaError_t err = cudaSuccess;
  int c = 0, dev = 0;
  if (a.io == kBF16 && a.dstate > 8) {
    SplitPlan sp;
    if ((err = split_form(a, vec, sp, c)) != cudaSuccess) return err;
    if (sp.segs > 0) {
      form = kFormSplit, ctas = c;
      return cudaSuccess;
    }
    FusedPlan plan;
    c = vec ? (a.zoh ? fused_ctas<__nv_bfloat16, 16, true, true, false>(a, a.batch, plan, dev, err)
                     : fused_ctas<__nv_bfloat16, 16, true, false, false>(a, a.batch, plan, dev, err))
            : (a.zoh ? fused_ctas<__nv_bfloat16, 16, false, true, false>(a, a.batch, plan, dev, err)
                     : fused_ctas<__nv_bfloat16, 16, false, false, false>(a, a.batch, plan, dev, err));
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
