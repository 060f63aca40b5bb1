// Host check of the member launch's carve (csrc/tb_layout.h, member_first):
// for random grid source offsets, capacities per source m, units d and extra
// units e, member g's range [member_first(off[g], m, d, e, g),
// member_first(off[g + 1], m, d, e, g + 1)) must hold ceil(n_g m / d) + e
// units, the ranges must be disjoint and in order, and the last one must end
// within member_first(total, m, d, e, B), the array size the host allocates.
#include <cstdint>
#include <cstdio>
#include <random>
#include <vector>

#include "tb_layout.h"

int main() {
  std::mt19937_64 rng(2024);
  long long cases = 0;
  const long long ds[] = {1, 1024, 2048};
  for (int trial = 0; trial < 20000; ++trial) {
    const int B = 1 + (int)(rng() % 64);
    std::vector<long long> off(B + 1, 0);
    for (int g = 0; g < B; ++g) {
      const int kind = (int)(rng() % 4);  // empty, tiny, medium, large grids
      const long long n = kind == 0 ? 0 : kind == 1 ? (long long)(rng() % 8) : kind == 2 ? (long long)(rng() % 5000)
                                                                                     : (long long)(rng() % 400000);
      off[g + 1] = off[g] + n;
    }
    const long long m = 1 + (long long)(rng() % 512);
    const long long d = ds[rng() % 3];
    const long long e = (long long)(rng() % 9);
    long long prev_end = 0;
    for (int g = 0; g < B; ++g) {
      const long long first = tb::member_first(off[g], m, d, e, g);
      const long long end = tb::member_first(off[g + 1], m, d, e, g + 1);
      const long long need = ((off[g + 1] - off[g]) * m + d - 1) / d + e;
      if (first < prev_end || end - first < need) {
        std::printf("FAIL B=%d g=%d m=%lld d=%lld e=%lld first=%lld end=%lld need=%lld prev_end=%lld\n", B, g, m, d,
                    e, first, end, need, prev_end);
        return 1;
      }
      prev_end = end;
      ++cases;
    }
    if (prev_end > tb::member_first(off[B], m, d, e, B)) {
      std::printf("FAIL: beyond the allocation\n");
      return 1;
    }
  }
  std::printf("OK %lld\n", cases);
  return 0;
}
