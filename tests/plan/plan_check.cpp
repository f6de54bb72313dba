// Host check of the forward scan's plans (scan_plan.h), built with the host compiler by
// tests/test_split_plan_host.py.  For each shape it builds the plans the library would launch on
// an SM count and checks, by walking the plan entries exactly as the kernel decodes them:
//  * balanced form: every (batch row, channel) in exactly one group, at most 4 units per group and
//    3 groups per CTA;
//  * split form: every (batch row, channel, chunk) scanned exactly once by the segment pass, or, for
//    a tail split, by the whole-row launch (all chunks of the rows it holds) and the segment pass
//    over the tail;
//  * split form, carry pass: every carry segment of every split channel scanned exactly once, none
//    reaching into the last segment;
//  * the workspace size: 4 (dstate + 1) bytes per batch row, channel and carry segment.
// Prints one line per shape and "all ok" or "FAILED".
#include <cstdio>
#include <vector>

#include "scan_plan.h"

using namespace ssm;

static int fails = 0;
#define EXPECT(c, ...)                       \
  do {                                       \
    if (!(c)) {                              \
      std::printf("  FAIL: " __VA_ARGS__);   \
      std::printf("\n");                     \
      ++fails;                               \
    }                                        \
  } while (0)

struct Entry {
  int b, d0, nch, seg;
};
static Entry decode(uint32_t e, bool split) {
  Entry x{int(e >> 16), int((e >> 4) & 0xfffu) * 8, int(e & 15u) * 8, 0};
  if (split) x.seg = int(e >> kSegShift), x.b &= kMaxSplitBatch - 1;
  return x;
}

static void check_balanced(int batch, int dim, int sms) {
  ScanArgs a{};
  a.batch = batch, a.dim = dim, a.dstate = 16, a.seqlen = 2048, a.io = kBF16;
  FusedPlan p{};
  const int ctas = make_fused_plan(a, batch, sms, p);
  std::printf("balanced b%d d%d on %d SMs: %d CTAs\n", batch, dim, sms, ctas);
  if (ctas == 0) return;
  std::vector<int> cov(size_t(batch) * dim, 0);
  for (int c = 0; c < ctas; ++c)
    for (int g = 0; g < kFusedGroups; ++g) {
      const uint32_t e = p.e[c * kFusedGroups + g];
      if (!e) continue;
      const Entry x = decode(e, false);
      EXPECT(x.nch >= 8 && x.nch <= 32, "group of %d channels", x.nch);
      for (int d = x.d0; d < x.d0 + x.nch && d < dim; ++d) cov[size_t(x.b) * dim + d]++;
    }
  for (size_t i = 0; i < cov.size(); ++i) EXPECT(cov[i] == 1, "channel %zu covered %d times", i, cov[i]);
}

static void check_split(int batch, int dim, int L, int sms, const char* expect) {
  ScanArgs a{};
  a.batch = batch, a.dim = dim, a.dstate = 16, a.seqlen = L, a.io = kBF16;
  SplitPlan sp{};
  FusedPlan pw, p1, p2;
  int cw = 0, c1 = 0, c2 = 0;
  const bool split = make_split_plans(a, sms, sp, pw, cw, p1, c1, p2, c2);
  std::printf("split b%d d%d L%d on %d SMs: %s", batch, dim, L, sms, split ? "" : "unsplit\n");
  if (split)
    std::printf("%d segments of %d, %d carry segments of %d, whole groups %d, tail from unit %d; CTAs %d + %d + %d\n",
                sp.segs, sp.seg_len, sp.ncarry, sp.carry_len, sp.whole_groups, sp.tail_p0, cw, c1, c2);
  EXPECT(split == (expect[0] != 'u'), "expected %s", expect);
  if (!split) return;
  EXPECT(sp.seg_len % 64 == 0 && sp.carry_len % 64 == 0 && sp.seg_len == sp.carry_len * sp.carries_per_seg,
         "segment lengths");
  EXPECT(sp.ncarry == (sp.segs - 1) * sp.carries_per_seg && sp.segs <= kMaxPlanSegs && sp.ncarry <= kMaxPlanSegs,
         "segment counts");
  EXPECT((cw > 0) == (sp.whole_groups > 0), "whole-row launch only for a tail split");
  EXPECT((long long)(sp.segs - 1) * sp.seg_len < L && (long long)sp.segs * sp.seg_len >= L, "segments cover L");
  EXPECT(sp.workspace_bytes == size_t(sp.ncarry) * batch * dim * 17 * 4, "workspace bytes");
  EXPECT(c1 <= sms && c2 <= sms && cw <= sms, "at most one CTA per SM");
  const int nck = (L + kScanChunk - 1) / kScanChunk;
  std::vector<int> cov(size_t(batch) * dim * nck, 0);
  for (int c = 0; c < cw; ++c)  // the whole-row launch of a tail split: every chunk of its rows
    for (int g = 0; g < kFusedGroups; ++g) {
      const uint32_t e = pw.e[c * kFusedGroups + g];
      if (!e) continue;
      const Entry x = decode(e, false);
      for (int d = x.d0; d < x.d0 + x.nch && d < dim; ++d)
        for (int k = 0; k < nck; ++k) cov[(size_t(x.b) * dim + d) * nck + k]++;
    }
  for (int c = 0; c < c2; ++c)
    for (int g = 0; g < kFusedGroups; ++g) {
      const uint32_t e = p2.e[c * kFusedGroups + g];
      if (!e) continue;
      const Entry x = decode(e, true);
      EXPECT(x.seg < sp.segs, "segment %d of %d", x.seg, sp.segs);
      const int k0 = x.seg * (sp.seg_len / kScanChunk), k1 = std::min(nck, k0 + sp.seg_len / kScanChunk);
      for (int d = x.d0; d < x.d0 + x.nch && d < dim; ++d)
        for (int k = k0; k < k1; ++k) cov[(size_t(x.b) * dim + d) * nck + k]++;
    }
  long long bad = 0;
  for (int v : cov) bad += v != 1;
  EXPECT(bad == 0, "%lld (channel, chunk) pairs not scanned exactly once", bad);
  // carry pass: the split channels (all, or the last row's tail), carry segments 0..ncarry-1
  const long long first = sp.whole_groups ? (long long)(batch - 1) * dim + 8LL * sp.tail_p0 : 0;
  std::vector<int> ccov(size_t(sp.ncarry) * batch * dim, 0);
  for (int c = 0; c < c1; ++c)
    for (int g = 0; g < kFusedGroups; ++g) {
      const uint32_t e = p1.e[c * kFusedGroups + g];
      if (!e) continue;
      const Entry x = decode(e, true);
      EXPECT(x.seg < sp.ncarry, "carry segment %d of %d", x.seg, sp.ncarry);
      if (x.seg >= sp.ncarry) continue;
      const long long end = (long long)(x.seg + 1) * sp.carry_len;
      EXPECT(end <= (long long)(sp.segs - 1) * sp.seg_len, "carry segment %d reaches the last segment", x.seg);
      for (int d = x.d0; d < x.d0 + x.nch && d < dim; ++d) ccov[(size_t(x.seg) * batch + x.b) * dim + d]++;
    }
  long long cbad = 0;
  for (int j = 0; j < sp.ncarry; ++j)
    for (long long r = 0; r < (long long)batch * dim; ++r)
      cbad += ccov[size_t(j) * batch * dim + r] != (r >= first ? 1 : 0);
  EXPECT(cbad == 0, "%lld carry slots not scanned exactly once", cbad);
}

int main() {
  for (int sms : {148, 132, 160}) {
    check_balanced(8, 1536, sms);
    check_balanced(1, 5120, sms);
    check_balanced(2, 1032, sms);
    check_balanced(7, 1544, sms);
  }
  check_split(1, 64, 8192, 148, "split");
  check_split(2, 64, 8232, 148, "split");
  check_split(1, 128, 9000, 148, "split");
  check_split(3, 40, 8256, 148, "split");
  check_split(1, 1536, 65536, 148, "split");
  check_split(1, 2048, 32768, 148, "split");
  check_split(1, 5120, 65536, 148, "split (tail)");
  check_split(1, 4800, 8192, 148, "split (tail)");
  check_split(2, 2400, 8192, 148, "split (tail)");
  check_split(1, 4768, 65536, 148, "split (tail)");
  check_split(1, 4736, 65536, 148, "unsplit");  // one full group per SM, no tail
  check_split(1, 4744, 65536, 148, "unsplit");  // a tail, but 593 units per row: groups would straddle
  check_split(8, 1536, 2048, 148, "unsplit");   // too short
  check_split(8, 1536, 8192, 148, "unsplit");   // many channels
  check_split(1, 64, 4096, 148, "unsplit");     // too short
  check_split(3000, 8, 8192, 148, "unsplit");   // batch beyond the split's 11 bits
  check_split(1, 1536, 65536, 132, "split");
  check_split(1, 5120, 65536, 132, "split (tail)");
  std::printf(fails ? "FAILED (%d)\n" : "all ok\n", fails);
  return fails ? 1 : 0;
}
