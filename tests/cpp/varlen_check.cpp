// Host check of the packed-response index math shared with the kernels: for random response
// lengths and tile sizes, every flat unit index of each kind maps back to the one response
// whose range holds it, and the per-response counts are the tile arithmetic's.
#include <cstdio>
#include <cstdlib>
#include <random>

#include "../../long_context_grpo_gb300/csrc/ls_internal.h"

static int fail(const char* what, int G, int b, int x) {
  std::printf("FAIL %s G=%d b=%d x=%d\n", what, G, b, x);
  return 1;
}

int main() {
  std::mt19937 rng(12345);
  const int qts[] = {128, 64, 42, 32, 25, 21, 18, 16, 14, 12, 11, 10, 9, 8};
  for (int trial = 0; trial < 2000; ++trial) {
    const int G = 1 + static_cast<int>(rng() % ls::kMaxPacked);
    const int qt = qts[rng() % (sizeof(qts) / sizeof(qts[0]))];
    int64_t cu[ls::kMaxPacked + 1];
    cu[0] = 0;
    for (int b = 0; b < G; ++b) cu[b + 1] = cu[b] + 1 + static_cast<int64_t>(rng() % 700);
    ls::Varlen v;
    ls::varlen_build(&v, G, cu, qt);
    if (v.G != G || v.row0[G] != cu[G]) return fail("totals", G, -1, -1);
    for (int b = 0; b < G; ++b) {
      const int R = static_cast<int>(cu[b + 1] - cu[b]);
      const int nq = (R + qt - 1) / qt;
      if (v.row0[b] != cu[b]) return fail("row0", G, b, -1);
      if (v.qt0[b + 1] - v.qt0[b] != nq) return fail("qt0", G, b, -1);
      if (v.pair0[b + 1] - v.pair0[b] != (nq + 1) / 2) return fail("pair0", G, b, -1);
      if (v.kt0[b + 1] - v.kt0[b] != (R + 127) / 128) return fail("kt0", G, b, -1);
    }
    const int* pres[3] = {v.pair0, v.qt0, v.kt0};
    const char* names[3] = {"pair", "qtile", "ktile"};
    for (int k = 0; k < 3; ++k) {
      const int* pre = pres[k];
      for (int x = 0; x < pre[G]; ++x) {
        const int b = ls::varlen_find(pre, G, x);
        if (b < 0 || b >= G || !(pre[b] <= x && x < pre[b + 1])) return fail(names[k], G, b, x);
      }
    }
  }
  std::printf("OK\n");
  return 0;
}
