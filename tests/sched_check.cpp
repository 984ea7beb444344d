// Host-only check of the stream kernel's item order (stream_sched.h): for each
// case given on the command line (heads C I target), every item appears once,
// every MIX item of a head comes after all of its SUM items and every OUT item
// after all of its MIX items, and item_at inverts step_start.  Prints
// "heads C I Dx Do items worst_gap" per case; exits non-zero on a violation.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "stream_sched.h"

using namespace mhla::sched;

static int check(int heads, int C, int I, long long target) {
  const auto lags = choose_lags(heads, C, I, target);
  const Sched s{heads, C, I, lags.first, lags.second};
  if (!(0 <= s.Dx && s.Dx <= s.Do && s.Do <= heads)) return 1;
  const int E = n_items(s);
  if (E != heads * (2 * C + I)) return 2;
  std::vector<int> seen((size_t)heads * (2 * C + I), 0);
  std::vector<int> sum_last(heads, -1), mix_first(heads, 1 << 30), mix_last(heads, -1), out_first(heads, 1 << 30);
  for (int pos = 0; pos < E; ++pos) {
    const Item it = item_at(s, pos);
    if (it.h < 0 || it.h >= heads) return 3;
    const int n = it.kind == kMix ? I : C;
    if (it.j < 0 || it.j >= n) return 4;
    const size_t id = (size_t)it.h * (2 * C + I) + (it.kind == kSum ? 0 : it.kind == kMix ? C : C + I) + it.j;
    if (seen[id]++) return 5;
    if (it.kind == kSum) sum_last[it.h] = pos;
    if (it.kind == kMix) {
      mix_first[it.h] = pos < mix_first[it.h] ? pos : mix_first[it.h];
      mix_last[it.h] = pos;
    }
    if (it.kind == kOut) out_first[it.h] = pos < out_first[it.h] ? pos : out_first[it.h];
  }
  long long worst = 1ll << 40;
  for (int h = 0; h < heads; ++h) {
    if (!(sum_last[h] < mix_first[h] && mix_last[h] < out_first[h])) return 6;
    const long long g1 = mix_first[h] - sum_last[h], g2 = out_first[h] - mix_last[h];
    const long long g = g1 < g2 ? g1 : g2;
    if (g != head_gap(s, h)) return 7;
    worst = g < worst ? g : worst;
  }
  std::printf("%d %d %d %d %d %d %lld\n", heads, C, I, s.Dx, s.Do, E, worst);
  return 0;
}

int main(int argc, char** argv) {
  for (int a = 1; a + 3 < argc; a += 4) {
    const int rc = check(std::atoi(argv[a]), std::atoi(argv[a + 1]), std::atoi(argv[a + 2]), std::atoll(argv[a + 3]));
    if (rc != 0) {
      std::printf("FAIL %s %s %s %s: %d\n", argv[a], argv[a + 1], argv[a + 2], argv[a + 3], rc);
      return rc;
    }
  }
  return 0;
}
