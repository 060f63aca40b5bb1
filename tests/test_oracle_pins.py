"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle (``oracle/``) against something other than its own
code: hand-worked fixtures under ``tests/golden/``, closed-form identities of
the ops (fVDB PR #757's test plan names the refine->coarsen round trip, the
k3s1 = [-1,1]^3 dilation alias and the +-4096 / negative-octant cases), brute
force on tiny inputs, and invariants such as V_out = 8 V_in for refinement.
"""
import itertools

import numpy as np
import pytest

import oracle
from sparse_voxel_grid_leaf_gb300 import synth
from tests import _helpers as H

FIELDS = ["leaf_offsets", "origins", "masks", "voxel_offset", "word_prefix", "leaf_bbox",
          "leaf_grid", "leaf_parent", "voxel_counts", "grid_bbox", "node_counts",
          "lower_offsets", "upper_offsets", "lower_origins", "lower_parent", "upper_origins"]


def same(a, b):
    for k in FIELDS:
        assert a[k].shape == b[k].shape, k
        assert np.array_equal(a[k], b[k]), k


def canon(o):
    o = [int(v) for v in o]
    return tuple(v // 4096 for v in o) + tuple((v // 128) % 32 for v in o) + tuple((v // 8) % 16 for v in o)


def strictly_canonical(res):
    B = len(res["leaf_offsets"]) - 1
    for g in range(B):
        lo, hi = int(res["leaf_offsets"][g]), int(res["leaf_offsets"][g + 1])
        keys = [canon(o) for o in res["origins"][lo:hi]]
        assert all(a < b for a, b in zip(keys, keys[1:]))


# ---------------------------------------------------------------- golden files

def test_golden_canonical_order():
    sec = H.read_sections("canonical_order.txt")
    vox = np.array([[int(v) for v in row] for row in sec["voxels"]], np.int32)
    exp = np.array([[int(v) for v in row] for row in sec["expected_origins"]], np.int32)
    res = oracle.run_voxels(vox, np.array([0, len(vox)], np.int64))
    assert np.array_equal(res["origins"], exp)
    assert list(res["node_counts"][0]) == [int(v) for v in sec["expected_node_counts"][0]]
    H.check_derived(res)


def node_order_case(lib=None):
    """The hand-worked node-order fixture through the oracle: (result, sections)."""
    sec = H.read_sections("node_order.txt")
    vox = np.array([[int(v) for v in row] for row in sec["voxels"]], np.int32)
    return oracle.run_voxels(vox, np.array([0, len(vox)], np.int64), lib=lib), sec


def check_node_order(res, sec):
    rows = lambda name: np.array([[int(v) for v in r] for r in sec[name]], np.int32)
    assert np.array_equal(res["origins"], rows("expected_origins"))
    assert np.array_equal(res["lower_origins"], rows("expected_lower_origins"))
    assert np.array_equal(res["upper_origins"], rows("expected_upper_origins"))
    assert res["leaf_parent"].tolist() == [int(v) for v in sec["expected_leaf_parent"][0]]
    assert res["lower_parent"].tolist() == [int(v) for v in sec["expected_lower_parent"][0]]
    assert list(res["node_counts"][0]) == [int(v) for v in sec["expected_node_counts"][0]]


def test_golden_node_order():
    # lower nodes in different root tiles: canonical order != lexicographic
    res, sec = node_order_case()
    check_node_order(res, sec)
    H.check_derived(res)


def test_golden_leaf_bits():
    sec = H.read_sections("leaf_bits.txt")
    B = int(sec["num_grids"][0][0])
    rows = [[int(v) for v in r] for r in sec["voxels"]]
    sets = [set() for _ in range(B)]
    for g, x, y, z in rows:
        sets[g].add((x, y, z))
    ijk, off = H.pack_sets(sets)
    res = oracle.run_voxels(ijk, off)
    exp = sec["expected_leaves"]
    assert res["origins"].shape[0] == len(exp)
    for i, r in enumerate(exp):
        assert list(res["origins"][i]) == [int(v) for v in r[0:3]]
        assert [int(w) for w in res["masks"][i]] == [int(v, 16) for v in r[3:11]]
        assert int(res["voxel_offset"][i]) == int(r[11])
        assert int(res["word_prefix"][i]) == int(r[12], 16)
        assert list(res["leaf_bbox"][i]) == [int(v) for v in r[13:19]]
    for g, r in enumerate(sec["expected_grids"]):
        r = [int(v) for v in r]
        assert int(res["voxel_counts"][g]) == r[0]
        assert list(res["grid_bbox"][g]) == r[1:7]
        assert list(res["node_counts"][g]) == r[7:10]


# ------------------------------------------------------------- from ijk (front end)

def test_from_ijk_dedups_and_matches_set():
    ijk, off = synth.random_voxels(3, 400, 40, seed=5, origin=(-20, -13, 4090), empty=(1,))
    res = oracle.run_voxels(ijk, off)
    sets = H.jagged_sets(ijk, off)
    for g in range(3):
        assert H.grid_voxels(res, g) == sets[g]
        assert res["voxel_counts"][g] == len(sets[g])
    strictly_canonical(res)
    H.check_derived(res)


# ------------------------------------------------------------------ refine

@pytest.mark.parametrize("f", [2, 4, 8])
def test_refine_brute_and_count(f):
    ijk, off = synth.random_voxels(2, 30, 20, seed=11, origin=(-10, -3, -4100))
    res = oracle.run_voxels(ijk, off, [("refine", f)])
    sets = H.jagged_sets(ijk, off)
    for g in range(2):
        got = H.grid_voxels(res, g)
        assert got == H.brute_refine(sets[g], f)
        assert len(got) == f ** 3 * len(sets[g])
    strictly_canonical(res)
    H.check_derived(res)


def test_refine_single_voxel_negative():
    # voxel (-1, 0, 5) -> children x in {-2,-1}, y in {0,1}, z in {10,11}
    res = oracle.run_voxels(np.array([[-1, 0, 5]], np.int32), np.array([0, 1]), [("refine", 2)])
    exp = {(x, y, z) for x in (-2, -1) for y in (0, 1) for z in (10, 11)}
    assert H.grid_voxels(res, 0) == exp
    assert res["origins"].tolist() == [[-8, 0, 8]]


def test_refine_coarsen_round_trip_stress_members():
    ijk, off = synth.make("stress_b64_res512")
    # a handful of members straddling +-4096 boundaries in different octants
    pick = [0, 3, 5, 10, 13]
    sub = [ijk[off[g]:off[g + 1]] for g in pick]
    ijk2, off2 = synth._pack(sub)
    base = oracle.run_voxels(ijk2, off2)
    back = oracle.run_voxels(ijk2, off2, [("refine", 2), ("coarsen", 2)])
    same(base, back)
    ref = oracle.run_voxels(ijk2, off2, [("refine", 2)])
    assert np.array_equal(ref["voxel_counts"], 8 * base["voxel_counts"])
    strictly_canonical(ref)


def test_refine_leaf_origins_equal_8_coarsen4():
    ijk, off = synth.make("pr1_b2_res32")
    ijk = ijk - np.array([16, 40, 3], np.int32)   # move into negative octants
    r2 = oracle.run_voxels(ijk, off, [("refine", 2)])
    c4 = oracle.run_voxels(ijk, off, [("coarsen", 4)])
    for g in range(2):
        lo, hi = r2["leaf_offsets"][g], r2["leaf_offsets"][g + 1]
        leaf_set = {tuple(o) for o in r2["origins"][lo:hi].tolist()}
        vox = {tuple(8 * v for v in t) for t in H.grid_voxels(c4, g)}
        assert leaf_set == vox


def test_refine_translation():
    ijk, off = synth.random_voxels(1, 60, 30, seed=3)
    t = np.array([8 * 37, -8 * 600, 8 * 5], np.int32)
    a = oracle.run_voxels(ijk, off, [("refine", 2)])
    b = oracle.run_voxels(ijk + t, off, [("refine", 2)])
    assert {tuple(v) for v in (a["origins"] + 2 * t).tolist()} == {tuple(v) for v in b["origins"].tolist()}


# ------------------------------------------------------------------ coarsen

def test_coarsen_floor_single_voxels():
    pts = [(-1, -1, -1), (-2, 3, -3), (3, -4, 0), (-9, 9, -17), (2 ** 31 - 1, -2 ** 31, 0)]
    for p in pts:
        res = oracle.run_voxels(np.array([p], np.int32), np.array([0, 1]), [("coarsen", 2)])
        assert H.grid_voxels(res, 0) == {tuple(v // 2 for v in p)}
    res = oracle.run_voxels(np.array([[-1, 0, 7]], np.int32), np.array([0, 1]), [("coarsen", 8)])
    assert H.grid_voxels(res, 0) == {(-1, 0, 0)}


@pytest.mark.parametrize("f", [2, 4, 8])
def test_coarsen_brute(f):
    ijk, off = synth.random_voxels(2, 300, 70, seed=9, origin=(-35, -4096 - 30, 20))
    res = oracle.run_voxels(ijk, off, [("coarsen", f)])
    sets = H.jagged_sets(ijk, off)
    for g in range(2):
        got = H.grid_voxels(res, g)
        assert got == H.brute_coarsen(sets[g], f)
        assert len(got) <= len(sets[g])
    H.check_derived(res)


def test_coarsen_chained_equals_direct():
    ijk, off = synth.make("pr1_b2_res32")
    ijk = ijk - np.array([20, 5, 31], np.int32)
    same(oracle.run_voxels(ijk, off, [("coarsen", 2), ("coarsen", 2)]),
         oracle.run_voxels(ijk, off, [("coarsen", 4)]))
    same(oracle.run_voxels(ijk, off, [("coarsen", 2)] * 3),
         oracle.run_voxels(ijk, off, [("coarsen", 8)]))
    same(oracle.run_voxels(ijk, off, [("refine", 2)] * 2),
         oracle.run_voxels(ijk, off, [("refine", 4)]))


# ------------------------------------------------------------------ dilate

BOXES = [((-1, -1, -1), (1, 1, 1)), ((-1, -1, -1), (0, 0, 0)), ((0, 0, 0), (1, 1, 1)),
         ((-1, 0, 0), (0, 1, 1)), ((0, -1, 0), (1, 0, 1))]


@pytest.mark.parametrize("box", BOXES)
def test_dilate_brute_minkowski(box):
    ijk, off = synth.random_voxels(2, 40, 24, seed=21, origin=(-12, 4084, -8))
    res = oracle.run_voxels(ijk, off, [("dilate", box[0], box[1])])
    sets = H.jagged_sets(ijk, off)
    for g in range(2):
        assert H.grid_voxels(res, g) == H.brute_dilate(sets[g], *box)
    strictly_canonical(res)
    H.check_derived(res)


def test_dilate_single_voxel_counts():
    one = (np.array([[7, -1, 8]], np.int32), np.array([0, 1]))
    n = [int(oracle.run_voxels(*one, [("dilate", lo, hi)])["voxel_counts"][0]) for lo, hi in BOXES[:3]]
    assert n == [27, 8, 8]


def test_dilate_pad_composition_and_reflection():
    ijk, off = synth.make("pr1_b2_res32")
    full = oracle.run_voxels(ijk, off, [("dilate", (-1,) * 3, (1,) * 3)])
    comp = oracle.run_voxels(ijk, off, [("dilate", (-1,) * 3, (0,) * 3), ("dilate", (0,) * 3, (1,) * 3)])
    same(full, comp)
    neg = -ijk
    a = oracle.run_voxels(neg, off, [("dilate", (0,) * 3, (1,) * 3)])
    b = oracle.run_voxels(ijk, off, [("dilate", (-1,) * 3, (0,) * 3)])
    for g in range(2):
        assert H.grid_voxels(a, g) == {(-x, -y, -z) for (x, y, z) in H.grid_voxels(b, g)}


# general boxes (stride-1 uniform-K topologies, integer-radius dilation):
# per axis lo in [-7, 0], hi in [0, 7]

GENERAL_BOXES = [((-2, -2, -2), (2, 2, 2)), ((-1, -1, -1), (2, 2, 2)), ((-7, 0, -3), (0, 5, 7)),
                 ((0, -4, -1), (6, 0, 1))]


@pytest.mark.parametrize("box", GENERAL_BOXES)
def test_general_box_single_voxel_closed_form(box):
    # one voxel v -> exactly the box v + [lo, hi]: (hi-lo+1) per axis, bbox v+lo .. v+hi
    lo, hi = box
    v = (-9, 4095, 16)
    res = oracle.run_voxels(np.array([v], np.int32), np.array([0, 1]), [("dilate", lo, hi)])
    n = 1
    for a in range(3):
        n *= hi[a] - lo[a] + 1
    assert int(res["voxel_counts"][0]) == n
    assert res["grid_bbox"][0].tolist() == [v[a] + lo[a] for a in range(3)] + [v[a] + hi[a] for a in range(3)]
    strictly_canonical(res)
    H.check_derived(res)


def test_general_box_is_a_sum_of_unit_boxes():
    # Minkowski sums of boxes add their bounds: [-2,2] = [-1,1] + [-1,1];
    # [-1,2] = [-1,1] + [0,1]; [-3,0]x[0,2]x[-1,1] = three unit steps
    ijk, off = synth.random_voxels(3, 60, 20, seed=5, origin=(-10, 4090, -3))
    unit = ("dilate", (-1,) * 3, (1,) * 3)
    same(oracle.run_voxels(ijk, off, [("dilate", (-2,) * 3, (2,) * 3)]), oracle.run_voxels(ijk, off, [unit, unit]))
    same(oracle.run_voxels(ijk, off, [("dilate", (-1,) * 3, (2,) * 3)]),
         oracle.run_voxels(ijk, off, [unit, ("dilate", (0,) * 3, (1,) * 3)]))
    steps = [("dilate", (-1, 0, -1), (0, 1, 0)), ("dilate", (-1, 0, 0), (0, 1, 1)), ("dilate", (-1, 0, 0), (0, 0, 0))]
    same(oracle.run_voxels(ijk, off, [("dilate", (-3, 0, -1), (0, 2, 1))]), oracle.run_voxels(ijk, off, steps))


def test_general_box_reflection():
    ijk, off = synth.random_voxels(2, 50, 30, seed=6, origin=(-4100, -20, 7))
    a = oracle.run_voxels(-ijk, off, [("dilate", (-5, 0, -2), (1, 7, 0))])
    b = oracle.run_voxels(ijk, off, [("dilate", (-1, -7, 0), (5, 0, 2))])
    for g in range(2):
        assert H.grid_voxels(a, g) == {(-x, -y, -z) for (x, y, z) in H.grid_voxels(b, g)}


# ------------------------------------------------------------------ batches

@pytest.mark.parametrize("empty", [(0,), (2,), (4,), (0, 1, 2, 3, 4)])
def test_empty_members(empty):
    ijk, off = synth.random_voxels(5, 50, 30, seed=2, empty=empty)
    for ops in ([], [("refine", 2)], [("coarsen", 2)], [("dilate", (-1,) * 3, (1,) * 3)]):
        res = oracle.run_voxels(ijk, off, ops)
        for g in empty:
            assert res["leaf_offsets"][g] == res["leaf_offsets"][g + 1]
            assert res["voxel_counts"][g] == 0
            assert list(res["grid_bbox"][g]) == [2 ** 31 - 1] * 3 + [-2 ** 31] * 3
            assert list(res["node_counts"][g]) == [0, 0, 0]
        H.check_derived(res)


def test_zero_grids():
    res = oracle.run_voxels(np.zeros((0, 3), np.int32), np.zeros(1, np.int64), [("refine", 2)])
    assert res["leaf_offsets"].tolist() == [0]
    assert res["origins"].shape == (0, 3)


def test_batch_members_independent():
    ijk, off = synth.make("pr1_b2_res32")
    both = oracle.run_voxels(ijk, off, [("refine", 2)])
    for g in range(2):
        alone = oracle.run_voxels(ijk[off[g]:off[g + 1]], np.array([0, off[g + 1] - off[g]]), [("refine", 2)])
        same(oracle.member(both, g), alone)


def test_run_leaves_equals_run_voxels():
    ijk, off = synth.random_voxels(3, 200, 50, seed=4, origin=(-25, -25, -25), empty=(1,))
    a = oracle.run_voxels(ijk, off)
    b = oracle.run_leaves(a["origins"], a["masks"], a["leaf_offsets"])
    same(a, b)
    c = oracle.run_leaves(a["origins"], a["masks"], a["leaf_offsets"], [("refine", 2)])
    same(oracle.run_voxels(ijk, off, [("refine", 2)]), c)


def test_overflow_is_reported():
    ijk = np.array([[2 ** 30, 0, 0]], np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.run_voxels(ijk, np.array([0, 1]), [("refine", 2)])
    assert e.value.status == oracle.STATUS_OVERFLOW
    with pytest.raises(oracle.OracleError):
        oracle.run_voxels(np.array([[2 ** 31 - 1, 0, 0]], np.int32), np.array([0, 1]),
                          [("dilate", (0, 0, 0), (1, 1, 1))])
    # the largest coordinate that still refines
    res = oracle.run_voxels(np.array([[2 ** 30 - 1, -2 ** 30, 0]], np.int32), np.array([0, 1]), [("refine", 2)])
    assert res["voxel_counts"][0] == 8


def test_workload_shells_structure():
    ijk, off = synth.make("shells_b16_res64")
    res = oracle.run_voxels(ijk, off)
    assert res["origins"].shape[0] > 0
    strictly_canonical(res)
    assert np.array_equal(res["voxel_counts"], np.array([len(s) for s in H.jagged_sets(ijk, off)]))


# ------------------------------------------------------------------ masked refine

def test_batch_voxel_order_matches_voxel_offsets():
    # the voxel order the masked refinement's flags follow: grid by grid, leaf by
    # leaf, ascending bit index; consistent with voxel_offset and voxel_counts
    ijk, off = synth.random_voxels(3, 120, 20, seed=41, origin=(-9, 4090, -4100), empty=(1,))
    res = oracle.run_voxels(ijk, off)
    vox, voffs = oracle.batch_voxels(res)
    assert voffs.tolist() == [0] + np.cumsum(res["voxel_counts"]).tolist()
    for g in range(3):
        part = [tuple(v) for v in vox[voffs[g]:voffs[g + 1]]]
        assert set(part) == H.grid_voxels(res, g)
        lo = int(res["leaf_offsets"][g])
        for i in range(lo, int(res["leaf_offsets"][g + 1])):
            first = int(voffs[g] + res["voxel_offset"][i])
            o = res["origins"][i]
            ns = [n for n in range(512) if (int(res["masks"][i][n >> 6]) >> (n & 63)) & 1]
            want = [(o[0] + (n >> 6), o[1] + ((n >> 3) & 7), o[2] + (n & 7)) for n in ns]
            assert part[first - voffs[g]:first - voffs[g] + len(ns)] == want


def test_masked_refine_all_none_and_brute():
    ijk, off = synth.random_voxels(3, 80, 16, seed=42, origin=(-20, 30, -4097))
    res = oracle.run_voxels(ijk, off)
    V = int(res["voxel_counts"].sum())
    same(oracle.run_masked_refine(res, np.ones(V, np.uint8), 2), oracle.run_voxels(ijk, off, [("refine", 2)]))
    empty = oracle.run_masked_refine(res, np.zeros(V, np.uint8), 2)
    assert int(empty["leaf_offsets"][-1]) == 0 and len(empty["leaf_offsets"]) == 4
    rng = np.random.default_rng(3)
    flags = (rng.random(V) < 0.3).astype(np.uint8)
    got = oracle.run_masked_refine(res, flags, 4)
    vox, voffs = oracle.batch_voxels(res)
    for g in range(3):
        sel = {tuple(int(c) for c in vox[j]) for j in range(voffs[g], voffs[g + 1]) if flags[j]}
        assert H.grid_voxels(got, g) == {(4 * x + a, 4 * y + b, 4 * z + c) for (x, y, z) in sel
                                         for a in range(4) for b in range(4) for c in range(4)}


def test_masked_refine_single_flag():
    # flag only the first voxel of the order: its 8 children at 2v + {0,1}^3
    one = (np.array([[5, -3, 9], [-8, 0, 1]], np.int32), np.array([0, 2]))
    res = oracle.run_voxels(*one)
    flags = np.zeros(2, np.uint8)
    flags[0] = 1
    got = oracle.run_masked_refine(res, flags, 2)
    first = min([(-8, 0, 1), (5, -3, 9)], key=lambda v: canon(v))  # canonical leaf order decides
    assert H.grid_voxels(got, 0) == {(2 * first[0] + a, 2 * first[1] + b, 2 * first[2] + c)
                                     for a in (0, 1) for b in (0, 1) for c in (0, 1)}


# ------------------------------------------------------------------ kernel maps

def _small():
    ijk, off = synth.random_voxels(3, 90, 14, seed=71, origin=(-7, 4088, -4100), empty=(1,))
    return oracle.run_voxels(ijk, off), ijk, off


def test_kernel_map_same_topology_identity_and_symmetry():
    res, _, _ = _small()
    m = oracle.run_kernel_map(res, res, (-1,) * 3, (1,) * 3)
    V = m.shape[0]
    assert m.shape == (V, 27)
    assert (m[:, 13] == np.arange(V)).all()          # d = 0 reads the voxel itself
    for j in range(V):                                # p reads q through d  <=>  q reads p through -d
        for k in range(27):
            if m[j, k] >= 0:
                assert m[m[j, k], 26 - k] == j


def test_kernel_map_k2s2_transpose_one_parent():
    res, ijk, off = _small()
    fine = oracle.run_voxels(ijk, off, [("refine", 2)])
    m = oracle.run_kernel_map(res, fine, (0,) * 3, (1,) * 3, stride=2, transposed=True)
    vin, _ = oracle.batch_voxels(res)
    vout, _ = oracle.batch_voxels(fine)
    for j, p in enumerate(vout):
        hits = np.nonzero(m[j] >= 0)[0]
        assert len(hits) == 1                          # exactly one parent, through d = p mod 2
        k = 4 * (p[0] & 1) + 2 * (p[1] & 1) + (p[2] & 1)
        assert hits[0] == k
        assert tuple(vin[m[j, k]]) == (p[0] >> 1, p[1] >> 1, p[2] >> 1)


def test_kernel_map_k2s2_forward_partitions_the_input():
    res, ijk, off = _small()
    coarse = oracle.run_voxels(ijk, off, [("coarsen", 2)])
    m = oracle.run_kernel_map(res, coarse, (0,) * 3, (1,) * 3, stride=2)
    hit = m[m >= 0]
    V = int(res["voxel_counts"].sum())
    assert sorted(hit.tolist()) == list(range(V))     # every input voxel feeds exactly one coarse voxel


def test_kernel_map_dilated_output_reads_each_input_27_times():
    res, ijk, off = _small()
    dil = oracle.run_voxels(ijk, off, [("dilate", (-1,) * 3, (1,) * 3)])
    m = oracle.run_kernel_map(res, dil, (-1,) * 3, (1,) * 3)
    counts = np.bincount(m[m >= 0], minlength=int(res["voxel_counts"].sum()))
    assert (counts == 27).all()
