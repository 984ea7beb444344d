// Order of the work items of the stream MHLA kernel (tc_stream.cu).
//
// For H heads of C chunks each, the items are SUM(h, j) (chunk summaries),
// MIX(h, r) (I mixing items a head) and OUT(h, j) (chunk outputs).  They form
// one list of steps: step t holds SUM(t, 0..C-1), then MIX(t - Dx, 0..I-1),
// then OUT(t - Do, 0..C-1), each where that head exists (0 <= head < H), for
// t = 0 .. H + Do - 1, with 0 <= Dx <= Do <= H.  So MIX(h) follows every SUM(h)
// and OUT(h) every MIX(h) in the list.  Plain host/device functions with no
// CUDA dependency: the kernel and a host-only check compile the same code.
#pragma once

#include <algorithm>
#include <utility>

#ifdef __CUDACC__
#define SCHED_HD __host__ __device__ __forceinline__
#else
#define SCHED_HD inline
#endif

namespace mhla {
namespace sched {

enum : int { kSum = 0, kMix = 1, kOut = 2 };

struct Item {
  int kind, h, j;
};

struct Sched {
  int heads, C, I, Dx, Do;
};

SCHED_HD int clampi(int x, int hi) { return x < 0 ? 0 : (x > hi ? hi : x); }

// List position of the first item of step t.
SCHED_HD int step_start(const Sched& s, int t) {
  return s.C * clampi(t, s.heads) + s.I * clampi(t - s.Dx, s.heads) + s.C * clampi(t - s.Do, s.heads);
}

SCHED_HD int n_items(const Sched& s) { return step_start(s, s.heads + s.Do); }

// Item at list position pos (0 <= pos < n_items): the last step t with
// step_start(t) <= pos (steps without items are skipped), then the offset.
SCHED_HD Item item_at(const Sched& s, int pos) {
  int lo = 0, hi = s.heads + s.Do - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (step_start(s, mid) <= pos) lo = mid;
    else hi = mid - 1;
  }
  int r = pos - step_start(s, lo);
  if (lo < s.heads) {
    if (r < s.C) return {kSum, lo, r};
    r -= s.C;
  }
  const int hx = lo - s.Dx;
  if (hx >= 0 && hx < s.heads) {
    if (r < s.I) return {kMix, hx, r};
    r -= s.I;
  }
  return {kOut, lo - s.Do, r};
}

// Distance in list positions from head h's last SUM item to its first MIX
// item, and from its last MIX item to its first OUT item; the smaller one.
inline long long head_gap(const Sched& s, int h) {
  const long long sum_last = step_start(s, h) + s.C - 1;
  const long long mix_first = step_start(s, h + s.Dx) + (h + s.Dx < s.heads ? s.C : 0);
  const long long out_first =
      step_start(s, h + s.Do) + (h + s.Do < s.heads ? s.C : 0) + (h + s.Do - s.Dx < s.heads ? s.I : 0);
  return std::min(mix_first - sum_last, out_first - (mix_first + s.I - 1));
}

// The lags (Dx, Do): the smallest Do (the fewest heads between a head's SUM
// and OUT items, i.e. the least L2 held by partials and mixed summaries) whose
// worst head_gap reaches `target`; failing that, the largest worst gap.
inline std::pair<int, int> choose_lags(int heads, int C, int I, long long target) {
  if (heads <= 0) return {0, 0};
  long long best = -1;
  std::pair<int, int> arg{heads / 2, heads};
  const int do_max = std::min(heads, 256);
  const int hstep = heads > 1024 ? heads / 1024 : 1;
  for (int Do = 1; Do <= do_max; ++Do) {
    const int dx_lo = heads <= 64 ? 0 : std::max(0, Do / 2 - 3);
    const int dx_hi = heads <= 64 ? Do : std::min(Do, Do / 2 + 3);
    for (int Dx = dx_lo; Dx <= dx_hi; ++Dx) {
      const Sched s{heads, C, I, Dx, Do};
      long long worst = head_gap(s, heads - 1);
      for (int h = 0; h < heads; h += hstep) worst = std::min(worst, head_gap(s, h));
      const long long score = std::min(worst, target);
      if (score > best) {
        best = score;
        arg = {Dx, Do};
      }
    }
    if (best >= target) break;
  }
  return arg;
}

}  // namespace sched
}  // namespace mhla

#undef SCHED_HD
