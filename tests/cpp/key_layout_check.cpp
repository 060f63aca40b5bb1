// Host check of the compressed canonical sort key (csrc/tb_layout.h,
// csrc/tb_common.cuh): for random batches and coordinate ranges -- tiny,
// tile-straddling, negative, wide -- the key must order leaves exactly as the
// canonical comparison does (grid, signed tile xyz, upper offset xyz, lower
// offset xyz), decode back to the same leaf, fit in W bits, and its
// lower_bits / node_bits prefixes must identify lower and upper nodes.
#include <algorithm>
#include <array>
#include <cstdint>
#include <cstdio>
#include <random>
#include <tuple>
#include <vector>

#include "tb_layout.h"

using namespace tb;

static int64_t cfloor(int64_t a, int64_t b) { return tb::floor_div(a, b); }
static int64_t cmod(int64_t a, int64_t b) { return a - b * cfloor(a, b); }

struct Leaf {
  uint32_t g;
  int32_t lc[3];
};

static std::array<int64_t, 10> canon(const Leaf& l) {
  std::array<int64_t, 10> k;
  k[0] = l.g;
  for (int a = 0; a < 3; ++a) {
    k[1 + a] = cfloor(l.lc[a], 512);
    k[4 + a] = cmod(cfloor(l.lc[a], 16), 32);
    k[7 + a] = cmod(l.lc[a], 16);
  }
  return k;
}

int main() {
  std::mt19937_64 rng(12345);
  int cases = 0;
  const int64_t spans[] = {1, 2, 7, 15, 16, 17, 40, 300, 511, 512, 513, 2000, 70000, 1 << 20};
  for (int trial = 0; trial < 3000; ++trial) {
    const int32_t B = 1 + (int32_t)(rng() % 70);
    int32_t bb[6];
    for (int a = 0; a < 3; ++a) {
      const int64_t span = spans[rng() % (sizeof spans / sizeof spans[0])] * 8;
      const int64_t lo_max = (int64_t)INT32_MAX - span;
      int64_t lo;
      switch (rng() % 4) {
        case 0: lo = -(int64_t)(rng() % 64) * 8 - 1 - (int64_t)(rng() % 8); break;  // just below 0
        case 1: lo = (int64_t)(rng() % 9000) - 4500; break;                           // around the origin
        case 2: lo = 4096 * ((int64_t)(rng() % 9) - 4) - (int64_t)(rng() % 300); break;  // around tile edges
        default: lo = (int64_t)(rng() % 4000000000ull) - 2000000000; break;
      }
      lo = std::max<int64_t>(std::min<int64_t>(lo, lo_max), INT32_MIN);
      bb[a] = (int32_t)lo;
      bb[3 + a] = (int32_t)(lo + span - 1 - (int64_t)(rng() % 8));
      if (bb[3 + a] < bb[a]) bb[3 + a] = bb[a];
    }
    KeyLayout K;
    if (!make_layout(B, bb, false, K)) continue;  // wider than 64 bits: reported as an error
    ++cases;
    std::vector<Leaf> leaves(200);
    for (auto& l : leaves) {
      l.g = (uint32_t)(rng() % B);
      for (int a = 0; a < 3; ++a) {
        const int64_t lo = cfloor(bb[a], 8), hi = cfloor(bb[3 + a], 8);
        int64_t v = lo + (int64_t)(rng() % (uint64_t)(hi - lo + 1));
        if (rng() % 5 == 0) v = (rng() & 1) ? lo : hi;
        l.lc[a] = (int32_t)v;
      }
    }
    for (size_t i = 0; i < leaves.size(); ++i) {
      const Leaf& x = leaves[i];
      const uint64_t kx = encode_key(K, x.g, x.lc[0], x.lc[1], x.lc[2]);
      if (K.W < 64 && (kx >> K.W) != 0) {
        std::printf("FAIL width W=%d\n", K.W);
        return 1;
      }
      uint32_t g;
      int32_t lc[3];
      decode_key(K, kx, g, lc);
      if (g != x.g || lc[0] != x.lc[0] || lc[1] != x.lc[1] || lc[2] != x.lc[2]) {
        std::printf("FAIL decode trial %d: (%u %d %d %d) -> (%u %d %d %d)\n", trial, x.g, x.lc[0], x.lc[1],
                    x.lc[2], g, lc[0], lc[1], lc[2]);
        return 1;
      }
      for (size_t j = 0; j < leaves.size(); j += 7) {
        const Leaf& y = leaves[j];
        const uint64_t ky = encode_key(K, y.g, y.lc[0], y.lc[1], y.lc[2]);
        const auto cx = canon(x), cy = canon(y);
        if ((kx < ky) != (cx < cy) || (kx == ky) != (cx == cy)) {
          std::printf("FAIL order trial %d W=%d\n", trial, K.W);
          return 1;
        }
        const bool same_lower = std::equal(cx.begin(), cx.begin() + 7, cy.begin());
        const bool same_upper = std::equal(cx.begin(), cx.begin() + 4, cy.begin());
        if ((shr64(kx, K.lower_bits) == shr64(ky, K.lower_bits)) != same_lower ||
            (shr64(kx, K.node_bits) == shr64(ky, K.node_bits)) != same_upper) {
          std::printf("FAIL node prefix trial %d\n", trial);
          return 1;
        }
      }
    }
  }
  std::printf("OK %d layouts\n", cases);
  return 0;
}
