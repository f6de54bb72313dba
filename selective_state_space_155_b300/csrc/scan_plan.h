// Host plans of the balanced forward scan and of its split form (scan_fwd.cu): which warp group of
// which CTA scans which channels and steps.  Plain host code, also compiled on its own by the
// host-side plan checks in tests/.
#pragma once

#include <stdint.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "internal.h"

namespace ssm {

// The balanced form: one CTA per SM holding kFusedGroups groups, each on a channel range (8 to 32
// channels of one batch row) from a host plan that evens out the channels per SM.  With 32-channel
// CTAs an SM carries 64 or 96 channels when the total is not a multiple of 96 per SM; the plan
// gives every SM within 8 channels of the mean.  Plan entry: b << 16 | (d0 / 8) << 4 | (channels / 8),
// 0 for an empty group; for the passes of a split sequence b takes 11 bits and the group's segment
// (it then scans that segment's steps only) the top 5.
constexpr int kFusedGroups = 3;
constexpr int kMaxFusedCtas = 160;
constexpr int kSegShift = 27, kMaxPlanSegs = 32, kMaxSplitBatch = 1 << 11;
struct FusedPlan {
  uint32_t e[kFusedGroups * kMaxFusedCtas];
};

// Fills group slots [slot0, kFusedGroups) of CTAs 0.. with the units at positions [p0, units per
// row) of `rows` plan rows, CTA c taking ceil(units left / CTAs left).  Plan row r is batch row
// r % batch of segment r / batch, or, with tail_b >= 0, batch row tail_b of segment r.  Returns the
// CTA count (0 if the units do not fit) and the busiest CTA's units in `worst`.
inline int fill_plan(const ScanArgs& a, long long rows, long long p0, int tail_b, int sms, int slot0, FusedPlan& plan,
              long long& worst) {
  worst = 0;
  if (a.dim % 8 != 0 || rows >= (1 << 16) || a.dim / 8 >= (1 << 12) || sms <= 0 || sms > kMaxFusedCtas) return 0;
  const long long ur = a.dim / 8, units = rows * (ur - p0);
  if (units <= 0 || units > (long long)sms * (kFusedGroups - slot0) * 4) return 0;
  long long left = units, row = 0, pos = p0;
  int ctas = 0;
  for (int c = 0; c < sms && left > 0; ++c) {
    const long long target = (left + (sms - c) - 1) / (sms - c);
    long long load = 0;
    for (int g = slot0; g < kFusedGroups; ++g) {
      uint32_t entry = 0;
      if (load < target && row < rows) {
        const long long take = std::min(std::min(4LL, target - load), ur - pos);
        // whole rows: row = b; split passes: segment < 32 in the top bits, batch < 2048
        const long long b = tail_b >= 0 ? tail_b : row % a.batch, sg = tail_b >= 0 ? row : row / a.batch;
        entry = uint32_t(b) << 16 | uint32_t(sg) << kSegShift | uint32_t(pos) << 4 | uint32_t(take);
        load += take, pos += take, left -= take;
        if (pos == ur) ++row, pos = p0;
      }
      plan.e[c * kFusedGroups + g] = entry;
    }
    worst = std::max(worst, load);
    ctas = c + 1;
  }
  return left == 0 ? ctas : 0;
}

// Host plan for the balanced form over `rows` rows of a.dim channels (the batch rows, or for a
// split sequence its (segment, batch row) pairs): units of 8 channels, groups of at most 4 units
// inside one row, at most kFusedGroups groups per CTA, CTA c taking ceil(units left / CTAs left)
// units.  Returns the CTA count, or 0 when the plan does not apply or (with `against_plain`) does
// not lower the busiest SM's load below that of the plain kernel (32-channel CTAs spread over the
// SMs; the passes of a split sequence have no plain alternative).
inline int make_fused_plan(const ScanArgs& a, long long rows, int sms, FusedPlan& plan, bool against_plain = true) {
  long long worst = 0;
  const int ctas = fill_plan(a, rows, 0, -1, sms, 0, plan, worst);
  const long long blocks = rows * ((a.dim + 31) / 32);
  const long long plain_max = 4 * ((blocks + sms - 1) / sms);  // units on the busiest SM, plain kernel
  return (ctas > 0 && (worst < plain_max || !against_plain)) ? ctas : 0;
}

// Sequence split for few channels and long sequences.  With few 8-channel units per SM the
// balanced form leaves each SM one warp group, which is latency-bound, and the split multiplies the
// groups by scanning segments of the sequence side by side: a carry pass (the recurrence without
// C, z or output) over the carry segments gives each one's end state from a zero state and its
// step-size sum, a combine folds them into the state entering each segment, and the full pass
// scans every segment from it.  The carry pass costs about 0.7 of the full scan per element over
// (segments - 1) / segments of the sequence, so the split is taken only where at least
// kMinSegs segments fit the SMs' groups at once (at most 3 units per SM); then as many segments
// as fit (up to kMaxPlanSegs, each at least kMinSegLen steps), and as many carry segments per
// segment as the groups hold (up to kMaxCarries, at most kMaxPlanSegs in all).  Both lengths are
// multiples of two chunks.
constexpr int kSplitMinLen = 8192;  // the shortest sequence split (the extra launches must pay)
constexpr int kMinSegs = 4, kMaxCarries = 4;
constexpr int kMinSegLen = 1024;

inline bool make_split(const ScanArgs& a, int sms, SplitPlan& p) {
  p = SplitPlan{};
  if (a.ckpt || a.dim % 8 != 0 || a.seqlen < kSplitMinLen || sms <= 0) return false;
  // the full pass reads h0 in one segment while another writes last_state
  const size_t nst = size_t(a.batch) * a.dim * a.dstate * sizeof(float);
  const uintptr_t h0 = reinterpret_cast<uintptr_t>(a.h0), ls = reinterpret_cast<uintptr_t>(a.last_state);
  if (h0 && ls && h0 < ls + nst && ls < h0 + nst) return false;
  const long long units = (long long)a.batch * (a.dim / 8), cap = (long long)sms * kFusedGroups * 4;
  if (units == 0) return false;
  // the plan entry's 5-bit segment field, and segments of at least kMinSegLen steps (shorter ones
  // spend more of their time filling the copy and table pipelines)
  const long long maxsegs = std::min<long long>(kMaxPlanSegs, std::max<long long>(kMinSegs, a.seqlen / kMinSegLen));
  long long segs = std::min<long long>(maxsegs, cap / units), per = 0;
  long long whole = 0, p0 = 0;  // the split of the tail only (below)
  const char* force = std::getenv("SSM_SCAN_SPLIT");
  if (force && std::strcmp(force, "off") == 0) return false;
  int fs = 0, fr = 0;
  if (force && std::sscanf(force, "%d,%d", &fs, &fr) == 2 && fs >= 2 && fr >= 1) {
    segs = fs, per = fr;  // forced (for measurements and tests)
    if (units * segs > cap || units * (segs - 1) * per > cap) return false;
  } else if (segs >= kMinSegs) {
    per = std::min<long long>(std::min<long long>(kMaxCarries, cap / (units * (segs - 1))), maxsegs / (segs - 1));
  } else {
    // Too many units to split them all, but whole rows would give every SM one full 4-unit group
    // and some SMs a second, smaller group whose per-chunk costs slow the SM down by a third: run
    // the full groups on whole rows (one group per SM) and then the tail of the last batch row as
    // a split of its own.  (With two full groups per SM the balanced plan already keeps the SMs
    // busy.)
    const long long ur = a.dim / 8;
    whole = units / (4LL * sms);
    const long long tail = units - 4LL * sms * whole;
    p0 = 4LL * sms * whole - (long long)(a.batch - 1) * ur;  // first tail unit within the last row
    if (whole != 1 || tail <= 0 || ur % 4 != 0 || p0 < 0) return false;
    segs = std::min<long long>(maxsegs, cap / tail);
    if (segs < kMinSegs) return false;
    per = std::min<long long>(std::min<long long>(kMaxCarries, cap / (tail * (segs - 1))), maxsegs / (segs - 1));
  }
  const long long step = 2 * kScanChunk;
  const long long clen = ((a.seqlen + segs * per - 1) / (segs * per) + step - 1) / step * step;
  const long long slen = clen * per;
  const long long nseg = (a.seqlen + slen - 1) / slen;
  if (nseg < 2 || a.batch >= kMaxSplitBatch || (nseg - 1) * per > kMaxPlanSegs || nseg > kMaxPlanSegs) return false;
  p.segs = int(nseg), p.carries_per_seg = int(per), p.seg_len = int(slen), p.carry_len = int(clen);
  p.ncarry = int((nseg - 1) * per);
  p.whole_groups = int(whole), p.tail_p0 = int(p0);
  p.workspace_bytes = size_t(p.ncarry) * a.batch * a.dim * (size_t(a.dstate) + 1) * sizeof(float);
  return true;
}

// The plans of the split for `a` on `sms` SMs (no device calls): for a tail split the whole-row
// launch's in pw over cw CTAs (cw = 0 otherwise; its group c is the plain kernel's 32-channel block
// c, which is what runs it), then the carry pass's in p1 over c1 CTAs and the segment pass's in p2
// over c2 CTAs.  False when the scan runs unsplit.
inline bool make_split_plans(const ScanArgs& a, int sms, SplitPlan& sp, FusedPlan& pw, int& cw, FusedPlan& p1,
                             int& c1, FusedPlan& p2, int& c2) {
  pw = FusedPlan{}, p1 = FusedPlan{}, p2 = FusedPlan{};
  cw = c1 = c2 = 0;
  if (!make_split(a, sms, sp)) return false;
  if (sp.whole_groups == 0) {
    c1 = make_fused_plan(a, (long long)sp.ncarry * a.batch, sms, p1, false);
    c2 = make_fused_plan(a, (long long)sp.segs * a.batch, sms, p2, false);
    return c1 > 0 && c2 > 0;
  }
  // the tail split: whole_groups whole-row groups of 4 units per CTA in their own launch, then the
  // carry pass and the segment pass over the tail of the last batch row
  const long long ur = a.dim / 8;
  long long worst = 0;
  for (int c = 0; c < sms; ++c)
    for (int g = 0; g < sp.whole_groups; ++g) {
      const long long u = (long long)(c * sp.whole_groups + g) * 4;
      pw.e[c * kFusedGroups + g] = uint32_t(u / ur) << 16 | uint32_t(u % ur) << 4 | 4u;
    }
  cw = sms;
  c1 = fill_plan(a, sp.ncarry, sp.tail_p0, a.batch - 1, sms, 0, p1, worst);
  c2 = fill_plan(a, sp.segs, sp.tail_p0, a.batch - 1, sms, 0, p2, worst);
  return c1 > 0 && c2 > 0;
}

}  // namespace ssm
