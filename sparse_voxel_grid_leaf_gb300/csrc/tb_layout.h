// Host-side sort-key layout helpers shared by the pass drivers.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "tb_common.cuh"

namespace tb {

inline int bitwidth(uint64_t x) {
  int n = 0;
  while (x) {
    ++n;
    x >>= 1;
  }
  return n;
}

inline int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && (a < 0)) --q;
  return q;
}

// Key layout for B grids whose voxels lie in the bbox bb (min xyz, max xyz).
// Returns false if the key needs more than 64 bits.
inline bool make_layout(int32_t B, const int32_t bb[6], bool empty, KeyLayout& K) {
  std::memset(&K, 0, sizeof K);
  K.gw = B > 1 ? bitwidth((uint64_t)(B - 1)) : 0;
  for (int a = 0; a < 3; ++a) {
    int lw = 0;
    if (!empty) {
      const int64_t Lo = floor_div(bb[a], 8), Hi = floor_div(bb[3 + a], 8);
      const int64_t tlo = floor_div(Lo, 512), thi = floor_div(Hi, 512);
      K.tile_base[a] = (int32_t)tlo;
      K.tw[a] = bitwidth((uint64_t)(thi - tlo));
      lw = (thi > tlo) ? 9 : std::min(9, bitwidth((uint64_t)(Lo ^ Hi)));
      K.lc_const[a] = (int32_t)(Lo & 0x1FF & ~((1 << lw) - 1));
    }
    K.lwl[a] = std::min(lw, 4);
    K.uw[a] = std::max(lw - 4, 0);
  }
  K.lshift[2] = 0;
  K.lshift[1] = K.lwl[2];
  K.lshift[0] = K.lwl[2] + K.lwl[1];
  K.lower_bits = K.lwl[0] + K.lwl[1] + K.lwl[2];
  K.ushift[2] = K.lower_bits;
  K.ushift[1] = K.ushift[2] + K.uw[2];
  K.ushift[0] = K.ushift[1] + K.uw[1];
  K.node_bits = K.ushift[0] + K.uw[0];
  K.tshift[2] = K.node_bits;
  K.tshift[1] = K.tshift[2] + K.tw[2];
  K.tshift[0] = K.tshift[1] + K.tw[1];
  K.gshift = K.tshift[0] + K.tw[0];
  K.W = K.gshift + K.gw;
  return K.W <= 64;
}

}  // namespace tb
