// Internal declarations shared by the library's translation units (not part of the C-ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

// Unsigned 32-bit division by a run-time constant d >= 1 with one multiply-high, an add and a
// shift (the round-up multiply-shift method of Granlund and Montgomery, "Division by invariant
// integers using multiplication"): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(n, m) + n) >> l for every 32-bit n (the sum is formed in 64 bits).
struct FastDiv {
  uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while (l < 32 && (uint64_t(1) << l) < d) ++l;
  const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
  return FastDiv{d, uint32_t(m), l};
}

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  return uint32_t((uint64_t(__umulhi(n, f.m)) + n) >> f.l);
}
#endif

enum Io { kF32 = 0, kBF16 = 1 };

// Arguments of one selective-scan launch; pointer and layout meaning as in ssm_scan.h.
struct ScanArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* dt_bias;
  const float* h0;
  void* y;
  float* last_state;
  int batch, dim, dstate, seqlen;
  int softplus;
  int io;
  int zoh;      // exact zero-order-hold Bbar instead of Delta * B
  float* ckpt;  // nullable: the state at the start of every kCkptSteps steps, for the backward
  // Sequence split (set by the launcher, zero otherwise): the steps of a row are cut into segments
  // of seg_len steps (a multiple of 2 * kScanChunk).  The carry pass scans every carry segment but
  // the last scan segment's from a zero state (the first from h0) and stores its end state and its
  // step-size sum; the full pass scans every segment from the state its carries combine to,
  // seg_carries carry segments per segment.
  int seg_len;
  int seg_carries;
  float* carry_h;  // [carry segment][batch][dim][dstate]
  float* carry_d;  // [carry segment][batch][dim]
  // Caller-owned scratch for the split (ws_given: never allocate; the split runs only when ws holds
  // its carry buffers).  Without it the launcher takes them from a stream-ordered allocation.
  void* ws;
  size_t ws_bytes;
  int ws_given;
};

// Steps per chunk of the scan kernels, and the interval of the training forward's checkpoints
// (the backward's register sub-chunk: it restarts each sub-chunk from its checkpoint).
constexpr int kScanChunk = 32;
constexpr int kCkptSteps = 8;
static_assert(kScanChunk % kCkptSteps == 0 && kCkptSteps % 8 == 0, "checkpoints at sub-window boundaries");

// Arguments of one backward pass of the scan; meaning as in ssm_scan.h.
struct ScanBwdArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* dt_bias;
  const float* ckpt;
  const void* dout;
  void* du;
  void* ddelta;
  float* dA;
  float* dB;
  float* dC;
  float* dD;
  void* dz;
  float* ddt_bias;
  float* dh0;
  int batch, dim, dstate, seqlen;
  int softplus;
  int io;
  int zoh;  // 1: exact zero-order hold for B, 0: Delta*B
};

// Arguments of one decode step; pointer and layout meaning as in ssm_scan.h.
struct UpdateArgs {
  float* state;
  const void* x;
  const void* dt;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* dt_bias;
  void* out;
  int batch, dim, dstate;
  int softplus;
  int io;
  int zoh;          // exact zero-order-hold Bbar instead of Delta * B
  FastDiv div_dim;  // filled at launch
};

// Arguments of one causal conv1d over whole rows; meaning as in ssm_scan.h.
struct ConvArgs {
  const void* x;
  const float* weight;
  const float* bias;
  const void* state_in;
  void* out;
  void* state_out;
  int batch, dim, seqlen, width;
  int silu;
  int io;
  FastDiv div_row;  // by the work items of one row (vectors or elements), filled at launch
  FastDiv div_dim;  // by dim, filled at launch
};

// Arguments of one causal conv1d decode step; meaning as in ssm_scan.h.
struct ConvUpdateArgs {
  void* state;
  const void* x;
  const float* weight;
  const float* bias;
  void* out;
  int batch, dim, width;
  int silu;
  int io;
  FastDiv div_dim;  // filled at launch
};

// Enqueue the scan on `stream`.  Arguments are already validated.
cudaError_t launch_scan_fwd(const ScanArgs& a, cudaStream_t stream);

// The four-lanes-per-channel scan (scan_fwd.cu): balanced layout where its plan applies (bf16,
// dstate 9..16; SSM_SCAN_VARIANT=quad_plain in the environment forces the 32-channel CTAs).
cudaError_t launch_scan_fwd_quad(const ScanArgs& a, bool vec, cudaStream_t stream);

// The form launch_scan_fwd runs for `a` (vec: rows take the 16-byte copy path) and its grid size.
enum ScanForm { kFormPlain = 0, kFormBalanced = 1, kFormSplit = 2 };
cudaError_t scan_fwd_form(const ScanArgs& a, bool vec, int& form, int& ctas);

// The sequence split the balanced form uses for `a` on the current device: segments, carry
// segments per segment, their lengths in steps, and the carry buffers' size in bytes; segs = 0
// when the scan is not split.
struct SplitPlan {
  int segs, carries_per_seg, seg_len, carry_len, ncarry;
  // whole_groups > 0: only the tail of the last batch row (8-channel units from tail_p0 on) is
  // split; the other units run whole rows, whole_groups 4-unit groups per SM, in the segment pass
  int whole_groups, tail_p0;
  size_t workspace_bytes;
};
cudaError_t scan_fwd_split(const ScanArgs& a, bool vec, SplitPlan& p);

// Hand-off waits of the forward kernels that gave up since the library was loaded (synchronises
// the device first).
cudaError_t scan_wait_timeouts(unsigned long long& count);

// Enqueue one decode step on `stream`.  Arguments are already validated.
cudaError_t launch_state_update(const UpdateArgs& a, cudaStream_t stream);

// Stage waits of the bulk-copy decode kernel that gave up since the library was loaded
// (synchronises the device first).
cudaError_t decode_wait_timeouts(unsigned long long& count);

// Enqueue the backward pass of the scan on `stream` (scan_bwd.cu): zero the accumulated
// gradients, then one launch.  Arguments are already validated.
cudaError_t launch_scan_bwd(const ScanBwdArgs& a, cudaStream_t stream);

// Unit-throughput probes (probe.cu): kind 0 = ex2.approx, 1 = FP32 FMA, 2 = packed f32x2 FMA,
// 3 = ex2 + packed f32x2 FMA interleaved, 4 = the recurrence's per-state-pair mix, 5 = a bounded
// mbarrier wait that nothing completes (it must give up).
cudaError_t launch_probe(int kind, int nblocks, long long* cycles, cudaStream_t stream);
double probe_ops_per_cta(int kind);

// Enqueue the causal conv1d / its decode step on `stream` (causal_conv1d.cu).  Arguments are
// already validated (width 1..4).
cudaError_t launch_causal_conv1d(const ConvArgs& a, cudaStream_t stream);
cudaError_t launch_causal_conv1d_update(const ConvUpdateArgs& a, cudaStream_t stream);

}  // namespace ssm
