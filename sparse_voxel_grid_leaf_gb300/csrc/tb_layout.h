// Sort-key layout helpers, on the host (pass planning) and on the device (the
// pass kernel plans a front end's key once it has read the input's bbox).
#pragma once

#include <cstdint>

#include "tb_common.cuh"

#ifdef __CUDACC__
#define TB_HD __host__ __device__
#else
#define TB_HD
#endif

namespace tb {

TB_HD inline int bitwidth(uint64_t x) {
  int n = 0;
  while (x) {
    ++n;
    x >>= 1;
  }
  return n;
}

TB_HD inline int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && (a < 0)) --q;
  return q;
}

TB_HD inline int64_t floor_mod(int64_t a, int64_t b) { return a - b * floor_div(a, b); }

TB_HD inline int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Target leaves per source leaf of a box dilation by [lo, hi] (|lo|, hi <= 7):
// offsets -1 (if lo < 0), 0, +1 (if hi > 0) per axis.
TB_HD inline int dilate_targets(const int32_t lo[3], const int32_t hi[3]) {
  int n = 1;
  for (int a = 0; a < 3; ++a) n *= 1 + (lo[a] < 0 ? 1 : 0) + (hi[a] > 0 ? 1 : 0);
  return n;
}

// Refine-then-dilate targets along one axis: fine leaf offsets (relative to
// the first child) from -1 (if lo < 0) to 2 (if hi > 0), else 0 .. 1.
TB_HD inline int refine_dilate_lo(int32_t lo) { return lo < 0 ? -1 : 0; }
TB_HD inline int refine_dilate_hi(int32_t hi) { return hi > 0 ? 2 : 1; }

TB_HD inline int log2_factor(int f) { return f == 8 ? 3 : (f == 4 ? 2 : 1); }

// Candidate target leaves per source leaf (or voxel) of a pass.
TB_HD inline int pass_targets(int op, int f, const int32_t lo[3], const int32_t hi[3]) {
  if (op == kRefine) return f * f * f;
  if (op == kDilate) return dilate_targets(lo, hi);
  if (op == kRefineDilate) {
    int n = 1;
    for (int a = 0; a < 3; ++a) n *= refine_dilate_hi(hi[a]) - refine_dilate_lo(lo[a]) + 1;
    return n;
  }
  return 1;
}

// Width of the target code in a slot value (see PassArgs::code_bits).
TB_HD inline int pass_code_bits(int op, int f) {
  if (op == kRefine || op == kCoarsen) return 3 * log2_factor(f);
  if (op == kDilate) return 5;
  if (op == kRefineDilate) return 6;
  return 0;
}

// Exact voxel bbox after a pass (refine by f: [f lo, f hi + f - 1]; coarsen by
// f: floor(lo / f), floor(hi / f); box dilation by [dlo, dhi]: [lo + dlo,
// hi + dhi]; refine-then-dilate: both; the front ends keep it).  Returns
// false if it leaves int32.
TB_HD inline bool propagate_bbox(int op, int f, const int32_t dlo[3], const int32_t dhi[3], const int32_t in[6],
                                 int32_t out[6]) {
  for (int a = 0; a < 3; ++a) {
    int64_t lo = in[a], hi = in[3 + a];
    if (op == kRefine) {
      lo = (int64_t)f * lo;
      hi = (int64_t)f * hi + f - 1;
    } else if (op == kCoarsen) {
      lo = floor_div(lo, f);
      hi = floor_div(hi, f);
    } else if (op == kDilate) {
      lo += dlo[a];
      hi += dhi[a];
    } else if (op == kRefineDilate) {
      lo = 2 * lo + dlo[a];
      hi = 2 * hi + 1 + dhi[a];
    }
    if (lo < INT32_MIN || hi > INT32_MAX) return false;
    out[a] = (int32_t)lo;
    out[3 + a] = (int32_t)hi;
  }
  return true;
}

// Key layout for B grids whose voxels lie in the bbox bb (min xyz, max xyz);
// see KeyLayout for the per-node shifted fields.  Returns false if the key
// needs more than 64 bits.
TB_HD inline bool make_layout(int32_t B, const int32_t bb[6], bool empty, KeyLayout& K) {
  K = KeyLayout{};
  K.gw = B > 1 ? bitwidth((uint64_t)(B - 1)) : 0;
  for (int a = 0; a < 3 && !empty; ++a) {
    const int64_t Lo = floor_div(bb[a], 8), Hi = floor_div(bb[3 + a], 8);  // leaf coordinates
    const int64_t Tlo = floor_div(Lo, 512), Thi = floor_div(Hi, 512);
    const int64_t Ulo = floor_mod(floor_div(Lo, 16), 32), Uhi = floor_mod(floor_div(Hi, 16), 32);
    const int64_t Blo = floor_div(Lo, 16), Bhi = floor_div(Hi, 16);     // lower-node blocks
    const int64_t Vlo = floor_mod(Lo, 16), Vhi = floor_mod(Hi, 16);
    K.t_lo[a] = (int32_t)Tlo;
    K.u_lo[a] = (int32_t)Ulo;
    K.v_lo[a] = (int32_t)Vlo;
    K.tw[a] = bitwidth((uint64_t)(Thi - Tlo));
    const int64_t umax = (Thi == Tlo) ? Uhi - Ulo : max64(31 - Ulo, Thi - Tlo >= 2 ? 31 : Uhi);
    const int64_t vmax = (Bhi == Blo) ? Vhi - Vlo : max64(15 - Vlo, Bhi - Blo >= 2 ? 15 : Vhi);
    K.uw[a] = bitwidth((uint64_t)umax);
    K.vw[a] = bitwidth((uint64_t)vmax);
  }
  K.vshift[2] = 0;
  K.vshift[1] = K.vw[2];
  K.vshift[0] = K.vw[2] + K.vw[1];
  K.lower_bits = K.vw[0] + K.vw[1] + K.vw[2];
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

// Member launches carve a chain's per-member arrays from the grids' stage-0
// source offsets: member g owns units [member_first(off[g], ...),
// member_first(off[g + 1], ...)) of an array where it needs
// ceil((off[g + 1] - off[g]) m / d) + e units.  The range always holds them:
// floor((x + y) / d) - floor(x / d) >= ceil(y / d) - 1, and each member adds
// e + 1 units.  member_first(total, m, d, e, B) is the array's size.
TB_HD inline long long member_first(long long off_g, long long m, long long d, long long e, long long g) {
  return (off_g * m) / d + g * (e + 1);
}

}  // namespace tb
