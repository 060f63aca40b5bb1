// Oracle for the batched generated-topology pass (TEST INFRASTRUCTURE ONLY).
//
// A plain, slow, single-threaded CPU statement of what the pass computes,
// written from the prose of fVDB issue #755 ("Generated-topology grid
// construction dominates per-iteration ConvolutionPlan cost") and fVDB PR #757
// ("Batched leaf-mask topology construction for generated conv grids").
// Only the tests, the smoke check and the benchmark's CPU-baseline leg may
// load it.  It shares no code, header or table with the CUDA library.
//
// Everything is done per voxel on std::set, as the definition reads:
//   1. expand the input into a set of voxels per grid (raw ijk, duplicates
//      collapse; or the set bits of each input leaf);
//   2. apply each op of the chain per voxel:
//        refine f   : v -> { f*v + d : d in [0,f)^3 }      (PR #757 summary 1:
//                      leaf-mask subdivision, every voxel becomes f^3 children)
//        coarsen f  : v -> floor(v / f)                    (PR #757 summary 1:
//                      a coarse voxel is active when any child is)
//        box dilate : v -> { v + d : d in [lo,hi]^3 }      (PR #757 summary 2:
//                      Minkowski sum with an axis-aligned unit box)
//   3. group voxels into 8^3 leaves: origin = 8*floor(v/8), local bit
//      n = 64*lx + 8*ly + lz, stored as eight 64-bit words (word lx,
//      bit 8*ly + lz); a leaf exists only if it holds a voxel;
//   4. order each grid's leaves canonically (PR #757 summary 1, second bullet:
//      root tiles by the tile coordinate floor(v/4096), then x-major upper
//      (32^3) child offsets, then x-major lower (16^3) child offsets); tile
//      coordinates compare as signed integers, x before y before z;
//   5. derive the per-leaf and per-grid arrays (leaf offsets, per-grid voxel
//      offsets, in-leaf word popcount prefixes, bounding boxes, node counts,
//      parent linkage), PR #757 summary 1, fourth bullet.
//
// Readings of points the pages leave open are listed in the design notes;
// the ones that shape the arithmetic here: floor (not truncation) for
// coarsening and grouping of negative coordinates, refine children at
// f*v + [0,f)^3, voxel offsets 0-based per grid, word prefix = seven 9-bit
// cumulative popcounts of words 0..k-1 (k = 1..7), empty grid bbox =
// (INT32_MAX x3, INT32_MIN x3).

#include <algorithm>
#include <array>
#include <climits>
#include <cstdint>
#include <cstring>
#include <map>
#include <set>
#include <tuple>
#include <vector>

namespace {

using Vox = std::array<int64_t, 3>;  // 64-bit so that overflow is visible

// Mathematical floor division and modulus for a positive divisor.
int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && (a < 0)) q -= 1;
  return q;
}
int64_t floor_mod(int64_t a, int64_t b) { return a - b * floor_div(a, b); }

enum { OP_REFINE = 0, OP_COARSEN = 1, OP_DILATE = 2 };

struct Op {
  int32_t kind;
  int32_t factor;
  int32_t lo[3];
  int32_t hi[3];
};

enum { ORACLE_OK = 0, ORACLE_OVERFLOW = 4, ORACLE_BAD_ARG = 1 };

bool in_int32(int64_t v) { return v >= INT32_MIN && v <= INT32_MAX; }

// Step 2: apply one op to every voxel of one grid.
int apply_op(const Op& op, const std::set<Vox>& in, std::set<Vox>& out) {
  out.clear();
  if (op.kind == OP_REFINE) {
    const int64_t f = op.factor;
    for (const Vox& v : in)
      for (int64_t dx = 0; dx < f; ++dx)
        for (int64_t dy = 0; dy < f; ++dy)
          for (int64_t dz = 0; dz < f; ++dz) {
            Vox w = {f * v[0] + dx, f * v[1] + dy, f * v[2] + dz};
            if (!in_int32(w[0]) || !in_int32(w[1]) || !in_int32(w[2])) return ORACLE_OVERFLOW;
            out.insert(w);
          }
  } else if (op.kind == OP_COARSEN) {
    const int64_t f = op.factor;
    for (const Vox& v : in) out.insert(Vox{floor_div(v[0], f), floor_div(v[1], f), floor_div(v[2], f)});
  } else if (op.kind == OP_DILATE) {
    for (const Vox& v : in)
      for (int64_t dx = op.lo[0]; dx <= op.hi[0]; ++dx)
        for (int64_t dy = op.lo[1]; dy <= op.hi[1]; ++dy)
          for (int64_t dz = op.lo[2]; dz <= op.hi[2]; ++dz) {
            Vox w = {v[0] + dx, v[1] + dy, v[2] + dz};
            if (!in_int32(w[0]) || !in_int32(w[1]) || !in_int32(w[2])) return ORACLE_OVERFLOW;
            out.insert(w);
          }
  } else {
    return ORACLE_BAD_ARG;
  }
  return ORACLE_OK;
}

// Canonical comparison tuple of a leaf origin: tile, then upper child
// offset, then lower child offset, each x-major (x, y, z).
using CanonKey = std::array<int64_t, 9>;
CanonKey canon_key(const Vox& o) {
  CanonKey k;
  for (int a = 0; a < 3; ++a) {
    k[a] = floor_div(o[a], 4096);                      // root tile coordinate
    k[3 + a] = floor_mod(floor_div(o[a], 128), 32);    // child of the upper node
    k[6 + a] = floor_mod(floor_div(o[a], 8), 16);      // child of the lower node
  }
  return k;
}

struct Leaf {
  Vox origin;
  std::array<uint64_t, 8> mask;
};

struct GridOut {
  std::vector<Leaf> leaves;        // canonical order
  std::vector<Vox> lowers;         // lower-node origins, canonical order
  std::vector<Vox> uppers;         // upper-node (root tile) origins
  std::vector<int32_t> leaf_parent;
  std::vector<int32_t> lower_parent;
};

int popcount64(uint64_t w) {
  int c = 0;
  while (w) {
    w &= w - 1;
    ++c;
  }
  return c;
}

// Steps 3-4 and the node lists of step 5 for one grid.
void group_and_order(const std::set<Vox>& vox, GridOut& g) {
  std::map<Vox, std::array<uint64_t, 8>> by_origin;
  for (const Vox& v : vox) {
    Vox o = {8 * floor_div(v[0], 8), 8 * floor_div(v[1], 8), 8 * floor_div(v[2], 8)};
    int64_t lx = v[0] - o[0], ly = v[1] - o[1], lz = v[2] - o[2];
    auto it = by_origin.find(o);
    if (it == by_origin.end()) it = by_origin.emplace(o, std::array<uint64_t, 8>{}).first;
    it->second[lx] |= (uint64_t(1) << (8 * ly + lz));
  }
  g.leaves.clear();
  for (auto& kv : by_origin) g.leaves.push_back(Leaf{kv.first, kv.second});
  std::sort(g.leaves.begin(), g.leaves.end(),
            [](const Leaf& a, const Leaf& b) { return canon_key(a.origin) < canon_key(b.origin); });

  // Internal nodes: the distinct lower (128^3) and upper (4096^3) blocks that
  // hold a leaf, each list in the same canonical order.
  std::set<Vox> lower_set, upper_set;
  for (const Leaf& l : g.leaves) {
    lower_set.insert(Vox{128 * floor_div(l.origin[0], 128), 128 * floor_div(l.origin[1], 128),
                         128 * floor_div(l.origin[2], 128)});
    upper_set.insert(Vox{4096 * floor_div(l.origin[0], 4096), 4096 * floor_div(l.origin[1], 4096),
                         4096 * floor_div(l.origin[2], 4096)});
  }
  g.lowers.assign(lower_set.begin(), lower_set.end());
  g.uppers.assign(upper_set.begin(), upper_set.end());
  auto by_canon = [](const Vox& a, const Vox& b) { return canon_key(a) < canon_key(b); };
  std::sort(g.lowers.begin(), g.lowers.end(), by_canon);
  std::sort(g.uppers.begin(), g.uppers.end(), by_canon);
  std::map<Vox, int32_t> lower_index, upper_index;
  for (size_t i = 0; i < g.lowers.size(); ++i) lower_index[g.lowers[i]] = int32_t(i);
  for (size_t i = 0; i < g.uppers.size(); ++i) upper_index[g.uppers[i]] = int32_t(i);
  g.leaf_parent.clear();
  for (const Leaf& l : g.leaves)
    g.leaf_parent.push_back(lower_index.at(Vox{128 * floor_div(l.origin[0], 128), 128 * floor_div(l.origin[1], 128),
                                               128 * floor_div(l.origin[2], 128)}));
  g.lower_parent.clear();
  for (const Vox& lo : g.lowers)
    g.lower_parent.push_back(upper_index.at(Vox{4096 * floor_div(lo[0], 4096), 4096 * floor_div(lo[1], 4096),
                                                4096 * floor_div(lo[2], 4096)}));
}

struct Result {
  int32_t B = 0;
  int32_t status = ORACLE_OK;
  std::vector<GridOut> grids;
};

int run_grid(std::set<Vox>& cur, const Op* ops, int32_t n_ops, GridOut& out) {
  std::set<Vox> next;
  for (int32_t k = 0; k < n_ops; ++k) {
    int st = apply_op(ops[k], cur, next);
    if (st != ORACLE_OK) return st;
    cur.swap(next);
  }
  group_and_order(cur, out);
  return ORACLE_OK;
}

bool ops_valid(const Op* ops, int32_t n_ops) {
  for (int32_t k = 0; k < n_ops; ++k) {
    const Op& op = ops[k];
    if (op.kind == OP_REFINE || op.kind == OP_COARSEN) {
      if (op.factor != 2 && op.factor != 4 && op.factor != 8) return false;
    } else if (op.kind == OP_DILATE) {
      for (int a = 0; a < 3; ++a)
        if (op.lo[a] > op.hi[a]) return false;
    } else {
      return false;
    }
  }
  return true;
}

}  // namespace

extern "C" {

// Runs the chain on a jagged voxel list (ijk [N,3] int32, offsets [B+1]).
void* oracle_run_voxels(const int32_t* ijk, const int64_t* offsets, int32_t B, const Op* ops, int32_t n_ops) {
  Result* r = new Result();
  r->B = B;
  r->grids.resize(B > 0 ? B : 0);
  if (!ops_valid(ops, n_ops)) {
    r->status = ORACLE_BAD_ARG;
    return r;
  }
  for (int32_t g = 0; g < B; ++g) {
    std::set<Vox> cur;
    for (int64_t i = offsets[g]; i < offsets[g + 1]; ++i) cur.insert(Vox{ijk[3 * i], ijk[3 * i + 1], ijk[3 * i + 2]});
    int st = run_grid(cur, ops, n_ops, r->grids[g]);
    if (st != ORACLE_OK) {
      r->status = st;
      return r;
    }
  }
  return r;
}

// Runs the chain on a jagged leaf list (origins [L,3], masks [L,8], offsets [B+1]).
void* oracle_run_leaves(const int32_t* origins, const uint64_t* masks, const int64_t* offsets, int32_t B,
                        const Op* ops, int32_t n_ops) {
  Result* r = new Result();
  r->B = B;
  r->grids.resize(B > 0 ? B : 0);
  if (!ops_valid(ops, n_ops)) {
    r->status = ORACLE_BAD_ARG;
    return r;
  }
  for (int32_t g = 0; g < B; ++g) {
    std::set<Vox> cur;
    for (int64_t i = offsets[g]; i < offsets[g + 1]; ++i)
      for (int lx = 0; lx < 8; ++lx)
        for (int ly = 0; ly < 8; ++ly)
          for (int lz = 0; lz < 8; ++lz)
            if ((masks[8 * i + lx] >> (8 * ly + lz)) & 1u)
              cur.insert(Vox{int64_t(origins[3 * i]) + lx, int64_t(origins[3 * i + 1]) + ly,
                             int64_t(origins[3 * i + 2]) + lz});
    int st = run_grid(cur, ops, n_ops, r->grids[g]);
    if (st != ORACLE_OK) {
      r->status = st;
      return r;
    }
  }
  return r;
}

int32_t oracle_status(const void* h) { return static_cast<const Result*>(h)->status; }

// sizes[0] = leaves, sizes[1] = lower nodes, sizes[2] = upper nodes (totals).
void oracle_sizes(const void* h, int64_t* sizes) {
  const Result* r = static_cast<const Result*>(h);
  sizes[0] = sizes[1] = sizes[2] = 0;
  for (const GridOut& g : r->grids) {
    sizes[0] += int64_t(g.leaves.size());
    sizes[1] += int64_t(g.lowers.size());
    sizes[2] += int64_t(g.uppers.size());
  }
}

// Step 5: writes every output array (caller-allocated, sized by oracle_sizes).
void oracle_fill(const void* h, int64_t* leaf_offsets, int32_t* origins, uint64_t* masks, int64_t* voxel_offset,
                 uint64_t* word_prefix, int32_t* leaf_bbox, int32_t* leaf_grid, int32_t* leaf_parent,
                 int64_t* voxel_counts, int32_t* grid_bbox, int32_t* node_counts, int64_t* lower_offsets,
                 int64_t* upper_offsets, int32_t* lower_origins, int32_t* lower_parent, int32_t* upper_origins) {
  const Result* r = static_cast<const Result*>(h);
  int64_t L = 0, NL = 0, NU = 0;
  for (int32_t g = 0; g < r->B; ++g) {
    const GridOut& G = r->grids[g];
    leaf_offsets[g] = L;
    lower_offsets[g] = NL;
    upper_offsets[g] = NU;
    int64_t vox_in_grid = 0;
    int64_t gmin[3] = {INT32_MAX, INT32_MAX, INT32_MAX};
    int64_t gmax[3] = {INT32_MIN, INT32_MIN, INT32_MIN};
    for (size_t i = 0; i < G.leaves.size(); ++i, ++L) {
      const Leaf& lf = G.leaves[i];
      for (int a = 0; a < 3; ++a) origins[3 * L + a] = int32_t(lf.origin[a]);
      for (int w = 0; w < 8; ++w) masks[8 * L + w] = lf.mask[w];
      voxel_offset[L] = vox_in_grid;
      // word prefix: field k-1 (bits 9(k-1) .. 9k-1) = voxels in words 0..k-1
      uint64_t wp = 0;
      int64_t run = 0;
      for (int k = 1; k <= 7; ++k) {
        run += popcount64(lf.mask[k - 1]);
        wp |= uint64_t(run) << (9 * (k - 1));
      }
      word_prefix[L] = wp;
      int64_t lmin[3] = {INT64_MAX, INT64_MAX, INT64_MAX};
      int64_t lmax[3] = {INT64_MIN, INT64_MIN, INT64_MIN};
      int64_t count = 0;
      for (int lx = 0; lx < 8; ++lx)
        for (int ly = 0; ly < 8; ++ly)
          for (int lz = 0; lz < 8; ++lz)
            if ((lf.mask[lx] >> (8 * ly + lz)) & 1u) {
              ++count;
              int64_t p[3] = {lf.origin[0] + lx, lf.origin[1] + ly, lf.origin[2] + lz};
              for (int a = 0; a < 3; ++a) {
                lmin[a] = std::min(lmin[a], p[a]);
                lmax[a] = std::max(lmax[a], p[a]);
              }
            }
      for (int a = 0; a < 3; ++a) {
        leaf_bbox[6 * L + a] = int32_t(lmin[a]);
        leaf_bbox[6 * L + 3 + a] = int32_t(lmax[a]);
        gmin[a] = std::min(gmin[a], lmin[a]);
        gmax[a] = std::max(gmax[a], lmax[a]);
      }
      vox_in_grid += count;
      leaf_grid[L] = g;
      leaf_parent[L] = G.leaf_parent[i];
    }
    for (size_t i = 0; i < G.lowers.size(); ++i, ++NL) {
      for (int a = 0; a < 3; ++a) lower_origins[3 * NL + a] = int32_t(G.lowers[i][a]);
      lower_parent[NL] = G.lower_parent[i];
    }
    for (size_t i = 0; i < G.uppers.size(); ++i, ++NU)
      for (int a = 0; a < 3; ++a) upper_origins[3 * NU + a] = int32_t(G.uppers[i][a]);
    voxel_counts[g] = vox_in_grid;
    for (int a = 0; a < 3; ++a) {
      grid_bbox[6 * g + a] = int32_t(gmin[a]);
      grid_bbox[6 * g + 3 + a] = int32_t(gmax[a]);
    }
    node_counts[3 * g + 0] = int32_t(G.uppers.size());
    node_counts[3 * g + 1] = int32_t(G.lowers.size());
    node_counts[3 * g + 2] = int32_t(G.leaves.size());
  }
  leaf_offsets[r->B] = L;
  lower_offsets[r->B] = NL;
  upper_offsets[r->B] = NU;
}

void oracle_free(void* h) { delete static_cast<Result*>(h); }

}  // extern "C"
