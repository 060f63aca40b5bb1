"""Mutation check of the oracle pins.

Each case plants one plausible mistake (a dropped term, a wrong sign, a
transposed index, truncation instead of floor, ...) in a private copy of
``oracle/oracle.cpp``, builds it, and requires that at least one pin of
``tests/test_oracle_pins.py``'s kind fails on it.  The real oracle is never
modified.
"""
import concurrent.futures as cf
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle
from sparse_voxel_grid_leaf_gb300 import synth
from tests import _helpers as H
from tests import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.cpp")

MUTANTS = {
    "coarsen_truncates": ("out.insert(Vox{floor_div(v[0], f), floor_div(v[1], f), floor_div(v[2], f)});",
                          "out.insert(Vox{v[0] / f, v[1] / f, v[2] / f});"),
    "refine_wrong_sign": ("Vox w = {f * v[0] + dx, f * v[1] + dy, f * v[2] + dz};",
                          "Vox w = {f * v[0] - dx, f * v[1] + dy, f * v[2] + dz};"),
    "dilate_drops_hi": ("for (int64_t dx = op.lo[0]; dx <= op.hi[0]; ++dx)",
                        "for (int64_t dx = op.lo[0]; dx < op.hi[0]; ++dx)"),
    "lower_offsets_z_major": ("k[6 + a] = floor_mod(floor_div(o[a], 8), 16);",
                              "k[8 - a] = floor_mod(floor_div(o[a], 8), 16);"),
    "upper_offsets_z_major": ("k[3 + a] = floor_mod(floor_div(o[a], 128), 32);",
                              "k[5 - a] = floor_mod(floor_div(o[a], 128), 32);"),
    "unsigned_tile_key": ("k[a] = floor_div(o[a], 4096);",
                          "k[a] = int64_t(uint32_t(floor_div(o[a], 4096)));"),
    "levels_swapped": ("k[6 + a] = floor_mod(floor_div(o[a], 8), 16);",
                       "k[6 + a] = k[3 + a]; k[3 + a] = floor_mod(floor_div(o[a], 8), 16);"),
    "bit_layout_transposed": ("it->second[lx] |= (uint64_t(1) << (8 * ly + lz));",
                              "it->second[lx] |= (uint64_t(1) << (8 * lz + ly));"),
    "word_prefix_shifted": ("run += popcount64(lf.mask[k - 1]);", "run += popcount64(lf.mask[k]);"),
    "leaf_bbox_max_is_min": ("leaf_bbox[6 * L + 3 + a] = int32_t(lmax[a]);",
                             "leaf_bbox[6 * L + 3 + a] = int32_t(lmin[a]);"),
    "voxel_offset_global": ("int64_t vox_in_grid = 0;\n", "static int64_t vox_in_grid = 0;\n"),
    "node_counts_swapped": ("node_counts[3 * g + 0] = int32_t(G.uppers.size());",
                            "node_counts[3 * g + 0] = int32_t(G.lowers.size());"),
    # lower-node list left in std::set's lexicographic order
    "lowers_unsorted": ("std::sort(g.lowers.begin(), g.lowers.end(), by_canon);", ""),
    # parent indices taken from the lexicographic order, the list itself sorted
    "leaf_parent_lexicographic": ("for (size_t i = 0; i < g.lowers.size(); ++i) lower_index[g.lowers[i]] = int32_t(i);",
                                  "{ int32_t i = 0; for (const Vox& v : lower_set) lower_index[v] = i++; }"),
}


def _pins(lib):
    """A compact run of the pin kinds; raises AssertionError on any mismatch."""
    sec = H.read_sections("canonical_order.txt")
    vox = np.array([[int(v) for v in r] for r in sec["voxels"]], np.int32)
    exp = np.array([[int(v) for v in r] for r in sec["expected_origins"]], np.int32)
    res = oracle.run_voxels(vox, np.array([0, len(vox)]), lib=lib)
    assert np.array_equal(res["origins"], exp)
    assert list(res["node_counts"][0]) == [int(v) for v in sec["expected_node_counts"][0]]

    res, sec = P.node_order_case(lib)
    P.check_node_order(res, sec)

    sec = H.read_sections("leaf_bits.txt")
    sets = [set(), set()]
    for g, x, y, z in ([int(v) for v in r] for r in sec["voxels"]):
        sets[g].add((x, y, z))
    ijk, off = H.pack_sets(sets)
    res = oracle.run_voxels(ijk, off, lib=lib)
    for i, r in enumerate(sec["expected_leaves"]):
        assert [int(w) for w in res["masks"][i]] == [int(v, 16) for v in r[3:11]]
        assert int(res["word_prefix"][i]) == int(r[12], 16)
        assert list(res["leaf_bbox"][i]) == [int(v) for v in r[13:19]]

    ijk, off = synth.random_voxels(3, 40, 24, seed=21, origin=(-12, 4084, -8))
    sets = H.jagged_sets(ijk, off)
    for ops, brute in ((("refine", 2),), lambda s: H.brute_refine(s, 2)), \
                      ((("coarsen", 2),), lambda s: H.brute_coarsen(s, 2)), \
                      ((("dilate", (-1,) * 3, (1,) * 3),), lambda s: H.brute_dilate(s, (-1,) * 3, (1,) * 3)):
        res = oracle.run_voxels(ijk, off, list(ops), lib=lib)
        for g in range(3):
            assert H.grid_voxels(res, g) == brute(sets[g])
        H.check_derived(res)


def test_real_oracle_passes_compact_pins():
    _pins(oracle._get())


@pytest.fixture(scope="module")
def mutant_libs():
    tmp = tempfile.mkdtemp(prefix="oracle_mutants_")
    base = open(SRC).read()

    def build_one(name):
        old, new = MUTANTS[name]
        assert base.count(old) >= 1, name
        src = os.path.join(tmp, name + ".cpp")
        with open(src, "w") as f:
            f.write(base.replace(old, new, 1))
        return name, oracle.build(force=True, out=os.path.join(tmp, name + ".so"), src=src,
                                  extra_flags=["-O1"])

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        libs = dict(ex.map(build_one, MUTANTS))
    yield libs
    shutil.rmtree(tmp, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, mutant_libs):
    lib = oracle.load(mutant_libs[name])
    with pytest.raises(AssertionError):
        _pins(lib)
