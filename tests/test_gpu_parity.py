"""GPU parity: every output array of the CUDA path equals the oracle's, bit for
bit, on the same seeded inputs (fVDB PR #757's test plan compares topologies
element-wise; the result is a unique set in a total order, so any difference
is a bug).  Calls go through the C ABI via the Python binding."""
import ctypes

import numpy as np
import pytest

import oracle
from sparse_voxel_grid_leaf_gb300 import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_voxel_grid_leaf_gb300 as tb  # noqa: E402

DIL = ("dilate", (-1, -1, -1), (1, 1, 1))
PAD_N = ("dilate", (-1, -1, -1), (0, 0, 0))
PAD_P = ("dilate", (0, 0, 0), (1, 1, 1))


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def assert_same(got, exp, where=""):
    for k in tb.ARRAY_NAMES:
        g, e = got[k], exp[k]
        assert g.shape == e.shape, "%s %s shape %s vs %s" % (where, k, g.shape, e.shape)
        if not np.array_equal(g, e):
            bad = np.argwhere(g != e)[:5]
            raise AssertionError("%s %s differs at %s: got %s expected %s"
                                 % (where, k, bad.tolist(), g[tuple(bad[0])], e[tuple(bad[0])]))


def gpu_chain(ijk, off, ops):
    b = tb.from_ijk(dev(ijk), dev(off))
    if ops:
        b = tb.chain(b, ops)
    return b


def check(ijk, off, ops, where=""):
    b = gpu_chain(ijk, off, ops)
    got = b.to_numpy()
    exp = oracle.run_voxels(ijk, off, ops)
    assert_same(got, exp, where)
    b.validate()
    return b, got


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module", autouse=True, params=["grid", "grid-sort", "member"])
def launch_mode(request, _built):
    """Every test runs with both launch shapes of the pass kernel, forced for
    every input: the whole-grid cooperative kernel -- with the lower-node
    child masks ordering every pass whose lower nodes are few ("grid"), and
    with the radix sort for every pass ("grid-sort") -- and the member launch
    (one cluster per grid of every chain)."""
    shape = request.param.split("-")[0]
    prev = tb.set_launch_mode(shape)
    prev_node = tb.set_node_mode("sort" if request.param.endswith("-sort") else "auto")
    yield request.param
    tb.set_launch_mode(prev)
    tb.set_node_mode(prev_node)


# ------------------------------------------------------------- small exact cases

def test_pr1_from_ijk_then_refine():
    ijk, off = synth.make("pr1_b2_res32")
    check(ijk, off, [], "from_ijk")
    check(ijk, off, [("refine", 2)], "refine")


@pytest.mark.parametrize("ops", [
    [("refine", 2)], [("refine", 4)], [("refine", 8)],
    [("coarsen", 2)], [("coarsen", 4)], [("coarsen", 8)],
    [DIL], [PAD_N], [PAD_P], [("dilate", (-1, 0, -1), (0, 1, 1))], [("dilate", (0, -1, 0), (0, 0, 1))],
    [("refine", 2), PAD_N],                       # k3s2 transpose
    [("refine", 2), ("coarsen", 2)],               # round trip
    [("coarsen", 2), DIL, ("refine", 2), PAD_P],
], ids=lambda ops: "-".join(o[0] + str(o[1] if o[0] != "dilate" else "") for o in ops))
def test_ops_negative_and_tile_crossing(ops):
    # members straddle the +-4096 root-tile boundaries in negative octants
    ijk, off = synth.random_voxels(5, 300, 90, seed=13, origin=(-4140, -45, 4050), empty=(2,))
    check(ijk, off, ops)


def test_duplicates_and_unsorted_ijk():
    ijk, off = synth.random_voxels(3, 2000, 12, seed=1, origin=(-6, -6, -6))  # many duplicates
    rng = np.random.default_rng(0)
    perm = np.concatenate([off[g] + rng.permutation(off[g + 1] - off[g]) for g in range(3)])
    check(ijk[perm], off, [])


@pytest.mark.parametrize("empty", [(0,), (3,), (6,), tuple(range(7))])
def test_empty_members(empty):
    ijk, off = synth.random_voxels(7, 120, 40, seed=3, origin=(-20, 0, -20), empty=empty)
    for ops in ([], [("refine", 2)], [("coarsen", 2)], [DIL], [("refine", 2), PAD_N]):
        check(ijk, off, ops, "empty=%s ops=%s" % (empty, ops))


def test_zero_grids_and_zero_voxels():
    b = tb.from_ijk(dev(np.zeros((0, 3), np.int32)), dev(np.zeros(1, np.int64)))
    assert b.num_grids == 0 and b.num_leaves == 0
    r = tb.refine(b)
    assert r.num_leaves == 0 and r.leaf_offsets_host.tolist() == [0]
    b = tb.from_ijk(dev(np.zeros((0, 3), np.int32)), dev(np.zeros(4, np.int64)))
    got = tb.box_dilate(b).to_numpy()
    assert_same(got, oracle.run_voxels(np.zeros((0, 3), np.int32), np.zeros(4, np.int64), [DIL]))


def test_single_voxel_extremes():
    # coordinates at the int32 limits that each op can still represent
    for p, ops_list in (([2 ** 30 - 1, -2 ** 30, 0], ([], [("refine", 2)], [("coarsen", 8)], [DIL])),
                        ([-1, -1, -1], ([], [("refine", 8)], [("coarsen", 2)], [DIL])),
                        ([2 ** 31 - 2, -2 ** 31 + 1, 4095], ([], [("coarsen", 4)], [DIL], [PAD_N]))):
        for ops in ops_list:
            check(np.array([p], np.int32), np.array([0, 1]), ops, "%s %s" % (p, ops))


def test_key_wider_than_64_bits_is_reported():
    # one grid spanning most of the int32 range on two axes needs a >64-bit key
    pts = np.array([[-2 ** 31, -2 ** 31, -2 ** 31], [2 ** 31 - 1, 2 ** 31 - 1, 2 ** 31 - 1]], np.int32)
    with pytest.raises(tb.TBError) as e:
        tb.from_ijk(dev(pts), dev(np.array([0, 2])))
    assert e.value.status == 7


def test_from_leaves_merges_and_sorts():
    ijk, off = synth.random_voxels(4, 400, 30, seed=8, origin=(-15, 7, -4100))
    exp = oracle.run_voxels(ijk, off)
    # shuffle the leaves, split each into two half masks, add an all-zero leaf
    o, m, lo = exp["origins"], exp["masks"], exp["leaf_offsets"]
    rng = np.random.default_rng(1)
    origins, masks, offs = [], [], [0]
    for g in range(4):
        idx = rng.permutation(np.arange(lo[g], lo[g + 1]))
        for i in idx:
            half = m[i] & np.uint64(0x5555555555555555)
            origins += [o[i], o[i]]
            masks += [half, m[i] ^ half]
        origins.append(np.array([8, 8, 8], np.int32))
        masks.append(np.zeros(8, np.uint64))
        offs.append(len(origins))
    origins = np.array(origins, np.int32)
    masks = np.array(masks, np.uint64)
    offs = np.array(offs, np.int64)
    b = tb.from_leaves(dev(origins), dev(masks.view(np.int64)), dev(offs))
    assert_same(b.to_numpy(), exp, "from_leaves")


def test_host_inputs_match_device_inputs():
    ijk, off = synth.make("pr1_b2_res32")
    a = tb.from_ijk(ijk, off).to_numpy()          # numpy: staged by the library
    b = tb.from_ijk(dev(ijk), dev(off)).to_numpy()
    assert_same(a, b, "host vs device")


def test_errors_leave_the_device_usable():
    with pytest.raises(tb.TBError) as e:
        tb.refine(tb.from_ijk(dev(np.array([[2 ** 30, 0, 0]], np.int32)), dev(np.array([0, 1]))))
    assert e.value.status == 4
    with pytest.raises(tb.TBError) as e:
        tb.from_ijk(dev(np.zeros((3, 3), np.int32)), dev(np.array([0, 2, 1, 3])))
    assert e.value.status == 1
    with pytest.raises(tb.TBError) as e:
        tb.refine(tb.from_ijk(dev(np.zeros((1, 3), np.int32)), dev(np.array([0, 1]))), 3)
    assert e.value.status == 1
    with pytest.raises(tb.TBError) as e:
        tb.from_leaves(dev(np.array([[4, 0, 0]], np.int32)), dev(np.ones((1, 8), np.int64)), dev(np.array([0, 1])))
    assert e.value.status == 1
    check(*synth.make("pr1_b2_res32"), [("refine", 2)], "after errors")


@pytest.mark.parametrize("workload", ["shells_b16_res64", "mixed"])
def test_multi_equals_separate_chains(workload):
    if workload == "mixed":
        ijk, off = synth.random_voxels(5, 300, 90, seed=13, origin=(-4140, -45, 4050), empty=(2,))
    else:
        ijk, off = synth.make(workload)
    chains = [[("refine", 2)], [("coarsen", 2)], [DIL], [PAD_N], [PAD_P], [("refine", 2), PAD_N],
              [("coarsen", 4)], [], [("coarsen", 2), DIL, ("refine", 2)]]
    b0 = tb.from_ijk(dev(ijk), dev(off))
    outs = tb.multi(b0, chains)
    assert len(outs) == len(chains)
    for ops, b in zip(chains, outs):
        assert_same(b.to_numpy(), oracle.run_voxels(ijk, off, ops), "multi %s" % (ops,))
        b.validate()


@pytest.mark.parametrize("n", [270, 700])
def test_multi_many_chains(n):
    # more chains than one split scan holds (256), and more chains than the
    # pass kernel has blocks (every block then runs every chain in turn)
    ijk, off = synth.make("pr1_b2_res32")
    kinds = [[("refine", 2)], [("coarsen", 2)], [DIL], [PAD_P], [("coarsen", 2), DIL], []]
    chains = [kinds[i % len(kinds)] for i in range(n)]
    want = [oracle.run_voxels(ijk, off, ops) for ops in kinds]
    b0 = tb.from_ijk(dev(ijk), dev(off))
    outs = tb.multi(b0, chains)
    assert len(outs) == n
    for i, b in enumerate(outs):
        if i % 37 == 0 or i >= n - len(kinds):
            assert_same(b.to_numpy(), want[i % len(kinds)], "chain %d" % i)
        else:
            assert b.num_leaves == len(want[i % len(kinds)]["origins"])


GENERAL_BOXES = [((-2,) * 3, (2,) * 3), ((-1,) * 3, (2,) * 3), ((0,) * 3, (1,) * 3), ((-7,) * 3, (7,) * 3),
                 ((-7, 0, -3), (0, 5, 7)), ((0, -4, -1), (6, 0, 1)), ((-3, -3, 0), (0, 0, 3))]


@pytest.mark.parametrize("box", GENERAL_BOXES)
def test_general_box_dilation(box):
    # random voxels across the +-4096 tile boundaries and negative octants,
    # with an empty member; then the shell workload
    ijk, off = synth.random_voxels(5, 250, 60, seed=31, origin=(-4120, -30, 4070), empty=(3,))
    check(ijk, off, [("dilate", box[0], box[1])], "random %s" % (box,))
    volume = np.prod([h - l + 1 for l, h in zip(*box)])
    if volume <= 125:  # the oracle's cost grows with the box volume
        ijk, off = synth.make("shells_b16_res64")
        check(ijk, off, [("dilate", box[0], box[1])], "shells %s" % (box,))


@pytest.mark.parametrize("K", [2, 3, 4, 5])
def test_stride1_uniform_k(K):
    ijk, off = synth.make("pr1_b2_res32")
    b0 = tb.from_ijk(dev(ijk), dev(off))
    for transpose in (False, True):
        lo, hi = tb.stride1_box(K, transpose)
        got = (tb.conv_transpose_grid_stride1 if transpose else tb.conv_grid_stride1)(b0, K)
        assert_same(got.to_numpy(), oracle.run_voxels(ijk, off, [("dilate", lo, hi)]), "K=%d %s" % (K, transpose))
    for r in (0, 1, 2, 3):
        assert_same(tb.dilated_grid(b0, r).to_numpy(),
                    oracle.run_voxels(ijk, off, [("dilate", (-r,) * 3, (r,) * 3)]), "radius %d" % r)


def test_general_box_in_chains_and_multi():
    ijk, off = synth.random_voxels(4, 200, 50, seed=33, origin=(-60, 4000, -4100))
    chains = [[("refine", 2), ("dilate", (-2,) * 3, (1,) * 3)], [("dilate", (-7, 0, 0), (0, 0, 7)), ("coarsen", 2)],
              [("dilate", (-1,) * 3, (2,) * 3)]]
    b0 = tb.from_ijk(dev(ijk), dev(off))
    for ops, b in zip(chains, tb.multi(b0, chains)):
        assert_same(b.to_numpy(), oracle.run_voxels(ijk, off, ops), "multi %s" % (ops,))


def test_box_bounds_out_of_range_are_rejected():
    ijk, off = synth.make("pr1_b2_res32")
    b0 = tb.from_ijk(dev(ijk), dev(off))
    for lo, hi in (((-8, 0, 0), (0, 0, 0)), ((0, 0, 0), (0, 8, 0)), ((1, 0, 0), (1, 0, 0)), ((0, 0, 0), (0, 0, -1))):
        with pytest.raises(tb.TBError) as e:
            tb.box_dilate(b0, lo, hi)
        assert e.value.status == 1


def test_multi_single_launch():
    ijk, off = synth.make("pr1_b2_res32")
    b0 = tb.from_ijk(dev(ijk), dev(off))
    n0 = tb.kernel_launch_count()
    tb.multi(b0, [[("refine", 2)], [("coarsen", 2)], [DIL]])
    # one pass kernel and one writer for all chains
    assert tb.kernel_launch_count() - n0 == 2


def test_deterministic_repeat():
    ijk, off = synth.make("shells_b16_res64")
    b = tb.from_ijk(dev(ijk), dev(off))
    first = tb.box_dilate(b).to_numpy()
    for _ in range(3):
        assert_same(tb.box_dilate(b).to_numpy(), first, "repeat")


def test_auto_launch_shape():
    """The default picks a member launch for a batch of small grids; the
    outputs equal the whole-grid kernel's."""
    prev = tb.set_launch_mode("auto")
    try:
        ijk, off = synth.make("shells_b16_res64")
        tb.profile_read()
        tb.profile_enable(1)
        b = tb.from_ijk(dev(ijk), dev(off))
        small = tb.refine(b).to_numpy()
        names = tb.profile_read()
        assert "member" in names and "chain" not in names, names
        tb.set_launch_mode("grid")
        assert_same(small, tb.refine(b).to_numpy(), "auto vs grid")
        # grids of very unequal sizes (0.25x-4x): the whole-grid kernel
        tb.set_launch_mode("auto")
        ijk, off = synth.make("pyramid_b48_res64")
        b = tb.from_ijk(dev(ijk), dev(off))
        tb.profile_read()
        uneven = tb.refine(b).to_numpy()
        names = tb.profile_read()
        assert "chain" in names and "member" not in names, names
        tb.set_launch_mode("member")
        assert_same(uneven, tb.refine(b).to_numpy(), "auto vs member")
    finally:
        tb.profile_enable(0)
        tb.set_launch_mode(prev)


def test_outputs_sized_ahead_grow_and_shrink():
    """A call shape that repeats allocates its outputs before the count
    readback from the previous call's counts: when the new counts are larger
    the chain is written again at its exact size; when smaller the batch
    keeps spare room.  Either way every array equals the oracle's."""
    # same grid count and voxel count, very different leaf counts
    dense, off = synth.random_voxels(3, 400, 12, seed=91, origin=(-6, 5, -4100))
    sparse, off2 = synth.random_voxels(3, 400, 400, seed=92, origin=(-6, 5, -4100))
    assert np.array_equal(off, off2)
    for first, second in ((dense, sparse), (sparse, dense)):
        for ijk in (first, second):  # the second call reuses the first one's counts
            check(ijk, off, [("refine", 2)], "ahead %d" % len(ijk))
            b = tb.from_ijk(dev(ijk), dev(off))
            outs = tb.multi(b, [[("refine", 2)], [DIL]])
            for o, ops in zip(outs, ([("refine", 2)], [DIL])):
                assert_same(o.to_numpy(), oracle.run_voxels(ijk, off, ops), "ahead multi %s" % (ops,))


def _random_op(rng):
    k = int(rng.integers(0, 4))
    if k == 0:
        return ("refine", int(rng.choice([2, 4])))
    if k == 1:
        return ("coarsen", int(rng.choice([2, 4, 8])))
    lo = tuple(int(x) for x in rng.integers(-3, 1, 3))
    hi = tuple(int(x) for x in rng.integers(0, 4, 3))
    return ("dilate", lo, hi)


def _random_chain(rng, n_max, growth_max=128):
    """Up to n_max random ops whose voxel-count growth (refinement f^3, box
    volume) stays within growth_max, so the oracle's per-voxel sets stay small."""
    ops, growth = [], 1
    while len(ops) < n_max:
        op = _random_op(rng)
        g = op[1] ** 3 if op[0] == "refine" else (
            int(np.prod([h - l + 1 for l, h in zip(op[1], op[2])])) if op[0] == "dilate" else 1)
        if growth * g > growth_max:
            if ops:
                break
            continue
        ops.append(op)
        growth *= g
    return ops


def test_random_chains_fuzz():
    """Seeded random batches (grid counts, sizes, spans, origins across the
    tile boundaries, empty members) through random chains of up to three ops
    and a two-chain multi call, every array against the oracle."""
    rng = np.random.default_rng(1234)
    for trial in range(24):
        B = int(rng.integers(1, 7))
        n = int(rng.integers(1, 300))
        span = int(rng.integers(4, 120))
        origin = tuple(int(x) for x in rng.integers(-4200, 4200, 3))
        empty = tuple(int(g) for g in range(B) if rng.random() < 0.2)
        ijk, off = synth.random_voxels(B, n, span, seed=500 + trial, origin=origin, empty=empty)
        chain_a = _random_chain(rng, int(rng.integers(1, 4)))
        chain_b = _random_chain(rng, int(rng.integers(1, 3)))
        where = "trial %d B=%d n=%d span=%d %s / %s" % (trial, B, n, span, chain_a, chain_b)
        b = tb.from_ijk(dev(ijk), dev(off))
        assert_same(tb.chain(b, chain_a).to_numpy(), oracle.run_voxels(ijk, off, chain_a), where)
        outs = tb.multi(b, [chain_a, chain_b])
        assert_same(outs[0].to_numpy(), oracle.run_voxels(ijk, off, chain_a), where + " multi a")
        assert_same(outs[1].to_numpy(), oracle.run_voxels(ijk, off, chain_b), where + " multi b")


def test_launches_are_counted():
    n0 = tb.kernel_launch_count()
    ijk, off = synth.make("pr1_b2_res32")
    tb.refine(tb.from_ijk(dev(ijk), dev(off)))
    # front end: pass kernel (which reads the input's range itself), writer;
    # refine: pass kernel, writer
    assert tb.kernel_launch_count() - n0 == 4


# ---------------------------------------------------------- workload-sized cases

@pytest.mark.parametrize("ops", [[("coarsen", 2)], [("refine", 2)], [DIL], [PAD_N], [PAD_P],
                                 [("refine", 2), PAD_N]])
def test_shells_b16(ops):
    ijk, off = synth.make("shells_b16_res64")
    check(ijk, off, ops, "b16 %s" % (ops,))


@pytest.mark.parametrize("ops", [[("refine", 2)], [("coarsen", 2)], [DIL], [PAD_N], [PAD_P],
                                 [("refine", 2), PAD_N]])
def test_shells_b48(ops):
    ijk, off = synth.make("shells_b48_res64")
    check(ijk, off, ops, "b48 %s" % (ops,))


def test_pyramid_b48_schedule():
    """4-level pyramid: coarsen x2/x4/x8 from the finest grid, then refine back
    with a k3s1 dilation at each level (11 passes in 8 calls)."""
    ijk, off = synth.make("pyramid_b48_res64")
    L0 = tb.from_ijk(dev(ijk), dev(off))
    e1, e2, e3 = tb.coarsen(L0, 2), tb.coarsen(L0, 4), tb.coarsen(L0, 8)
    u2 = tb.refine(e3, 2)
    d2 = tb.box_dilate(u2)
    u1 = tb.refine(d2, 2)
    d1 = tb.box_dilate(u1)
    u0 = tb.refine(d1, 2)
    sched = {"e1": (e1, [("coarsen", 2)]), "e2": (e2, [("coarsen", 4)]), "e3": (e3, [("coarsen", 8)]),
             "u2": (u2, [("coarsen", 8), ("refine", 2)]),
             "d2": (d2, [("coarsen", 8), ("refine", 2), DIL]),
             "u1": (u1, [("coarsen", 8), ("refine", 2), DIL, ("refine", 2)]),
             "d1": (d1, [("coarsen", 8), ("refine", 2), DIL, ("refine", 2), DIL]),
             "u0": (u0, [("coarsen", 8), ("refine", 2), DIL, ("refine", 2), DIL, ("refine", 2)])}
    for name, (b, ops) in sched.items():
        assert_same(b.to_numpy(), oracle.run_voxels(ijk, off, ops), name)


K5S1 = ("dilate", (-2, -2, -2), (2, 2, 2))   # conv_grid k5s1
STRESS_OPS = {"from_ijk": [], "refine2": [("refine", 2)], "coarsen4": [("coarsen", 4)], "dilate_k3s1": [DIL],
              "pad_neg": [PAD_N], "k3s2": [("refine", 2), PAD_N], "conv_k5s1": [K5S1],
              "round_trip": [("refine", 2), ("coarsen", 2)]}
MULTI5 = [[("refine", 2)], [("coarsen", 2)], [DIL], [PAD_N], [("refine", 2), PAD_N]]
_STRESS_ORACLE = {}


def member_oracle(ijk, off, ops):
    """The oracle's result for every member run alone (members are
    independent), on a thread pool: {g: arrays}.  Cached per chain, so both
    launch shapes compare against one oracle run."""
    import concurrent.futures as cf
    import os
    key = repr(ops)
    if key not in _STRESS_ORACLE:
        def one(g):
            sub = ijk[off[g]:off[g + 1]]
            return oracle.run_voxels(sub, np.array([0, len(sub)]), ops)
        with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
            _STRESS_ORACLE[key] = dict(enumerate(ex.map(one, range(len(off) - 1))))
    return _STRESS_ORACLE[key]


def assert_members(got, ijk, off, ops, where):
    exp = member_oracle(ijk, off, ops)
    assert len(got["leaf_offsets"]) == len(off)
    for g in range(len(off) - 1):
        assert_same(oracle.member(got, g), exp[g], "%s member %d" % (where, g))


@pytest.fixture(scope="module")
def stress():
    ijk, off = synth.make("stress_b64_res512")
    return ijk, off, tb.from_ijk(dev(ijk), dev(off))


@pytest.mark.parametrize("name", sorted(STRESS_OPS))
def test_stress_full_size_all_members(stress, name):
    """Full B=64 res-512 batch (shells and blobs straddling the +-4096 tiles in
    all eight octants) in the launch configuration the benchmark times; every
    member's arrays equal the oracle's run of that member alone."""
    ijk, off, b0 = stress
    ops = STRESS_OPS[name]
    b = tb.chain(b0, ops) if ops else b0
    got = b.to_numpy()
    b.validate()
    assert_members(got, ijk, off, ops, name)
    if name == "k3s2":
        # above the fused refine-then-pad bound this chain runs as two passes
        assert b.build_source_leaves != b0.num_leaves
    if name == "refine2":
        assert np.array_equal(got["voxel_counts"], 8 * b0.to_numpy(["voxel_counts"])["voxel_counts"])
    if name == "round_trip":
        assert_same(got, b0.to_numpy(), "refine->coarsen")


def test_stress_multi5_all_members(stress):
    """The five conv-grid chains in one tb_multi call at stress size."""
    ijk, off, b0 = stress
    for ops, b in zip(MULTI5, tb.multi(b0, MULTI5)):
        assert_members(b.to_numpy(), ijk, off, ops, "multi %s" % (ops,))
        b.validate()


def test_stress_masked_refine_half(stress):
    """Masked refinement with half of the stress batch's voxels flagged."""
    ijk, off, b0 = stress
    base = b0.to_numpy()
    V = int(base["voxel_counts"].sum())
    flags = (np.random.default_rng(0).random(V) < 0.5).astype(np.uint8)
    key = "masked-half"
    if key not in _STRESS_ORACLE:
        _STRESS_ORACLE[key] = oracle.run_masked_refine(base, flags, 2)
    got = tb.refine_masked(b0, torch.from_numpy(flags).cuda(), 2)
    assert_same(got.to_numpy(), _STRESS_ORACLE[key], "masked half")
    got.validate()


# ---------------------------------------------------------- masked refinement

@pytest.mark.parametrize("factor", [2, 4])
def test_masked_refine(factor):
    import torch
    for ijk, off in (synth.random_voxels(6, 300, 50, seed=51, origin=(-4110, 20, 4080), empty=(0, 4)),
                     synth.make("shells_b16_res64")):
        b0 = tb.from_ijk(dev(ijk), dev(off))
        base = b0.to_numpy()
        V = int(base["voxel_counts"].sum())
        rng = np.random.default_rng(factor)
        flags = (rng.random(V) < 0.35).astype(np.uint8)
        exp = oracle.run_masked_refine(base, flags, factor)
        got = tb.refine_masked(b0, torch.from_numpy(flags).cuda(), factor)
        assert_same(got.to_numpy(), exp, "masked x%d" % factor)
        got.validate()
        # flags from host memory and as bools
        assert_same(tb.refine_masked(b0, flags.astype(bool), factor).to_numpy(), exp, "host flags")


def test_masked_refine_all_and_none():
    import torch
    ijk, off = synth.make("pr1_b2_res32")
    b0 = tb.from_ijk(dev(ijk), dev(off))
    V = int(b0.to_numpy(["voxel_counts"])["voxel_counts"].sum())
    assert_same(tb.refine_masked(b0, torch.ones(V, dtype=torch.bool, device="cuda")).to_numpy(),
                oracle.run_voxels(ijk, off, [("refine", 2)]), "all flags")
    none = tb.refine_masked(b0, torch.zeros(V, dtype=torch.bool, device="cuda"))
    assert none.num_leaves == 0 and none.num_grids == 2
    none.validate()


# ---------------------------------------------------------- fused chains

FUSED = [
    [("refine", 2), ("dilate", (-1, -1, -1), (1, 1, 1))],      # refine then k3s1: one fused pass
    [("refine", 2), ("dilate", (-1, 0, 0), (0, 1, 1))],
    [("refine", 2), ("dilate", (0, -1, 0), (1, 0, 0))],
    [("refine", 2), ("refine", 2)],                            # refine x4 in one pass
    [("refine", 2), ("refine", 4)],                            # refine x8
    [("coarsen", 2), ("coarsen", 2), ("coarsen", 2)],          # coarsen x8
    [("dilate", (-1,) * 3, (1,) * 3), ("dilate", (-1,) * 3, (0,) * 3)],  # boxes add up
    [("refine", 2), PAD_N, ("coarsen", 4)],
]


@pytest.mark.parametrize("ops", FUSED)
def test_fused_chains(ops):
    ijk, off = synth.random_voxels(5, 220, 45, seed=61, origin=(-4105, 4090, -20), empty=(2,))
    check(ijk, off, ops, "fused random %s" % (ops,))
    ijk, off = synth.make("shells_b16_res64")
    check(ijk, off, ops, "fused shells %s" % (ops,))


def test_node_path_is_taken(launch_mode):
    """The whole-grid kernel orders by lower-node child masks where the
    output's lower nodes are few (no digit passes), by radix sort where told
    to; the member launch always sorts."""
    ijk, off = synth.make("shells_b16_res64")
    b0 = tb.from_ijk(dev(ijk), dev(off))
    for ops in ([("refine", 2)], [DIL], [("coarsen", 2)], [("refine", 2), PAD_N]):
        b = tb.chain(b0, ops)
        if launch_mode == "grid":
            assert b.build_digit_passes == 0, ops
        else:
            assert b.build_digit_passes > 0, ops


def test_fused_chains_are_one_pass():
    ijk, off = synth.make("pr1_b2_res32")
    b0 = tb.from_ijk(dev(ijk), dev(off))
    for ops in ([("refine", 2), PAD_N], [("coarsen", 4)], [("refine", 8)], [DIL, DIL]):
        b = tb.chain(b0, ops)
        # one pass: its source leaves are the input's
        assert b.build_source_leaves == b0.num_leaves, ops


# ---------------------------------------------------------- kernel maps

KMAP_CASES = [
    # (ops producing the output from the input, box lo, box hi, stride, transposed)
    ([], (-1,) * 3, (1,) * 3, 1, False),                       # k3s1 same topology
    ([("dilate", (-1,) * 3, (1,) * 3)], (-1,) * 3, (1,) * 3, 1, False),  # conv_grid k3s1
    ([("refine", 2)], (0,) * 3, (1,) * 3, 2, True),            # conv_transpose_grid k2s2
    ([("coarsen", 2)], (0,) * 3, (1,) * 3, 2, False),          # conv_grid k2s2
    ([("refine", 2), PAD_N], (-1,) * 3, (1,) * 3, 2, True),     # k3s2 transpose
    ([("coarsen", 2)], (-2, -1, 0), (3, 1, 2), 2, False),       # uneven box, forward stride 2
    ([], (-7, 0, -2), (0, 7, 2), 1, False),                    # large box
    ([PAD_P], (-1,) * 3, (1,) * 3, 1, True),                   # transposed stride 1
    ([("refine", 2)], (-2,) * 3, (2,) * 3, 2, True),           # k5s2 transpose
    ([("refine", 2)], (0, 0, 0), (3, 0, 0), 2, True),          # 4 columns, two per parity class
    ([("refine", 2)], (-7, -7, 0), (-7, -6, 1), 2, True),      # a reach past the output leaf's own
]


KMAP_FORMS = ["auto", "staged", "staged_prepass", "tabulated", "per_entry"]


@pytest.fixture(params=KMAP_FORMS)
def kmap_form(request):
    prev = tb.set_kmap_mode(request.param)
    yield request.param
    tb.set_kmap_mode(prev)


@pytest.mark.parametrize("case", range(len(KMAP_CASES)))
def test_kernel_map(case, kmap_form):
    ops, lo, hi, stride, transposed = KMAP_CASES[case]
    ijk, off = synth.random_voxels(4, 150, 26, seed=81, origin=(-4100, 4085, -13), empty=(2,))
    b_in = tb.from_ijk(dev(ijk), dev(off))
    b_out = tb.chain(b_in, ops) if ops else b_in
    got = tb.kernel_map(b_in, b_out, lo, hi, stride, transposed).cpu().numpy()
    exp = oracle.run_kernel_map(b_in.to_numpy(), b_out.to_numpy(), lo, hi, stride, transposed)
    assert got.shape == exp.shape
    assert np.array_equal(got, exp), "kernel map case %d (%s): %d of %d entries differ" % (
        case, kmap_form, int((got != exp).sum()), got.size)


@pytest.mark.parametrize("case", range(3))
def test_kernel_map_dense_leaves(case, kmap_form):
    """Full leaves (512 voxels each): the staged form cuts a warp's 32 leaves
    into batches by its listed-voxel capacity; odd map offsets (a map that
    does not start on 16 bytes) take the scalar head and tail."""
    ops, lo, hi, stride, transposed = [([], (-1,) * 3, (1,) * 3, 1, False),
                                       ([("refine", 2)], (0,) * 3, (1,) * 3, 2, True),
                                       ([("coarsen", 2)], (0,) * 3, (1,) * 3, 2, False)][case]
    ijk, off = synth.random_voxels(2, 6, 6, seed=3, origin=(-20, 5, 9))
    b_in = tb.chain(tb.from_ijk(dev(ijk), dev(off)), [("refine", 8)])
    b_out = tb.chain(b_in, ops) if ops else b_in
    exp = oracle.run_kernel_map(b_in.to_numpy(), b_out.to_numpy(), lo, hi, stride, transposed)
    got = tb.kernel_map(b_in, b_out, lo, hi, stride, transposed).cpu().numpy()
    assert np.array_equal(got, exp), (kmap_form, int((got != exp).sum()))
    # the same map written one int32 past a 16-byte boundary
    v = b_out._view()
    K = exp.shape[1]
    buf = torch.full((int(v.num_voxels) * K + 8,), 7, dtype=torch.int32, device="cuda")
    lo_a = (ctypes.c_int32 * 3)(*lo)
    hi_a = (ctypes.c_int32 * 3)(*hi)
    st = tb.lib().tb_kernel_map(b_in.handle, b_out.handle, lo_a, hi_a, stride, 1 if transposed else 0,
                                ctypes.c_void_p(buf.data_ptr() + 4), int(v.num_voxels) * K, None)
    assert st == 0
    torch.cuda.synchronize()
    out = buf.cpu().numpy()
    assert out[0] == 7 and (out[1 + exp.size:] == 7).all()
    assert np.array_equal(out[1:1 + exp.size].reshape(exp.shape), exp)


def test_kernel_map_shells_sampled_rows():
    # full size: the B=16 shells, k3s1 same topology; rows sampled against the oracle's definition
    ijk, off = synth.make("shells_b16_res64")
    b = tb.from_ijk(dev(ijk), dev(off))
    got = tb.kernel_map(b, b).cpu().numpy()
    res = b.to_numpy()
    vox, voffs = oracle.batch_voxels(res)
    assert got.shape == (len(vox), 27)
    assert b.num_voxels == len(vox) == int(res["voxel_counts"].sum())
    assert (got[:, 13] == np.arange(len(vox))).all()
    rng = np.random.default_rng(5)
    for j in rng.choice(len(vox), 400, replace=False):
        g = int(np.searchsorted(voffs, j, side="right") - 1)
        where = {tuple(int(c) for c in vox[i]): i for i in range(voffs[g], voffs[g + 1])}
        p = vox[j]
        k = 0
        for dx in (-1, 0, 1):
            for dy in (-1, 0, 1):
                for dz in (-1, 0, 1):
                    q = (int(p[0]) + dx, int(p[1]) + dy, int(p[2]) + dz)
                    assert got[j, k] == where.get(q, -1)
                    k += 1


def _popcount_below(mask_words, bn):
    return sum(bin(int(mask_words[w])).count("1") for w in range(bn >> 6)) + \
        bin(int(mask_words[bn >> 6]) & ((1 << (bn & 63)) - 1)).count("1")


def test_kernel_map_stress_k2s2_transpose_sampled_leaves():
    """Full stress size, the form the library picks there (the staged map,
    chunks of 16 output leaves per warp): the k2s2 transpose map from the
    stress batch to its refinement.  The rows
    of sampled output leaves are checked against the map's definition
    (q = (p - d) / 2 where p - d is even), written out from the batches' own
    leaf arrays."""
    ijk, off = synth.make("stress_b64_res512")
    b = tb.from_ijk(dev(ijk), dev(off))
    fine = tb.refine(b)
    got = tb.kernel_map(b, fine, (0,) * 3, (1,) * 3, 2, True)
    ri, rf = b.to_numpy(), fine.to_numpy()
    vin = np.concatenate([[0], np.cumsum(ri["voxel_counts"])])
    vout = np.concatenate([[0], np.cumsum(rf["voxel_counts"])])
    index = {(int(ri["leaf_grid"][i]),) + tuple(int(c) for c in ri["origins"][i]): i
             for i in range(len(ri["origins"]))}
    rng = np.random.default_rng(7)
    for i in rng.choice(len(rf["origins"]), 150, replace=False):
        g, o, m = int(rf["leaf_grid"][i]), [int(c) for c in rf["origins"][i]], rf["masks"][i]
        rows = []
        for n in range(512):
            if not (int(m[n >> 6]) >> (n & 63)) & 1:
                continue
            p = (o[0] + (n >> 6), o[1] + ((n >> 3) & 7), o[2] + (n & 7))
            row = []
            for d in [(dx, dy, dz) for dx in (0, 1) for dy in (0, 1) for dz in (0, 1)]:
                t = [p[a] - d[a] for a in range(3)]
                if any(x % 2 for x in t):
                    row.append(-1)
                    continue
                q = [x // 2 for x in t]
                leaf = index.get((g, q[0] & ~7, q[1] & ~7, q[2] & ~7))
                bn = ((q[0] & 7) << 6) | ((q[1] & 7) << 3) | (q[2] & 7)
                if leaf is None or not (int(ri["masks"][leaf][bn >> 6]) >> (bn & 63)) & 1:
                    row.append(-1)
                    continue
                row.append(int(vin[g] + ri["voxel_offset"][leaf] + _popcount_below(ri["masks"][leaf], bn)))
            rows.append(row)
        r0 = int(vout[g] + rf["voxel_offset"][i])
        assert np.array_equal(got[r0:r0 + len(rows)].cpu().numpy(), np.array(rows, np.int32)), "leaf %d" % i


# ---------------------------------------------------------- failure detection

def test_bounded_wait_gives_up_and_leaves_the_device_usable():
    # a wait on a flag that nothing sets ends with TB_ERR_DEVICE_TIMEOUT after
    # its poll limit (no hang, no fault); a preset flag passes
    import time
    t0 = time.time()
    with pytest.raises(tb.TBError) as e:
        tb.selftest_wait(False, spin_limit=1 << 14)
    assert e.value.status == 6
    assert time.time() - t0 < 30
    tb.selftest_wait(True, spin_limit=1 << 14)
    check(*synth.make("pr1_b2_res32"), [("refine", 2)], "after a timed-out wait")


def test_export_many_matches_arrays():
    import torch
    ijk, off = synth.make("pr1_b2_res32")
    b0 = tb.from_ijk(dev(ijk), dev(off))
    bs = [b0, tb.refine(b0), tb.box_dilate(b0)]
    ref = [b.to_numpy(["origins", "masks", "voxel_offset", "leaf_offsets"]) for b in bs]
    # pinned host, device and pageable (numpy) destinations, one batch skipped per list
    o = [torch.empty((b.num_leaves, 3), dtype=torch.int32).pin_memory() for b in bs]
    m = [torch.empty((b.num_leaves, 8), dtype=torch.int64, device="cuda") for b in bs]
    v = [np.zeros(b.num_leaves, np.int64) for b in bs]
    lo = [torch.empty(b.num_grids + 1, dtype=torch.int64).pin_memory() for b in bs[:2]] + [None]
    tb.export_many(bs, o, m, v, lo)
    torch.cuda.synchronize()
    for i, r in enumerate(ref):
        assert np.array_equal(o[i].numpy(), r["origins"])
        assert np.array_equal(m[i].cpu().numpy().view(np.uint64), r["masks"])
        assert np.array_equal(v[i], r["voxel_offset"])
        if lo[i] is not None:
            assert np.array_equal(lo[i].numpy(), r["leaf_offsets"])
    # the same through a prepared plan, into cleared buffers, twice
    plan = tb.ExportPlan(o, m, v, lo)
    for _ in range(2):
        for x in o + m:
            x.zero_()
        for x in v:
            x[:] = 0
        plan(bs)
        torch.cuda.synchronize()
        for i, r in enumerate(ref):
            assert np.array_equal(o[i].numpy(), r["origins"])
            assert np.array_equal(m[i].cpu().numpy().view(np.uint64), r["masks"])
            assert np.array_equal(v[i], r["voxel_offset"])


def test_export_many_large_arrays():
    """Arrays of 1 MiB and more (here the masks, 5.6 MB, and the origins) go
    through the copy engines, the small ones through the copy kernel, in the
    same call."""
    import torch
    ijk, off = synth.make("shells_b16_res64")
    b0 = tb.from_ijk(dev(ijk), dev(off))
    bs = [tb.chain(b0, [("refine", 2), ("refine", 2)]), b0]
    ref = [b.to_numpy(["origins", "masks", "voxel_offset", "leaf_offsets"]) for b in bs]
    assert bs[0].num_leaves * 64 >= 1 << 20 and bs[1].num_leaves * 64 < 1 << 20
    o = [torch.zeros((b.num_leaves, 3), dtype=torch.int32).pin_memory() for b in bs]
    m = [torch.zeros((b.num_leaves, 8), dtype=torch.int64).pin_memory() for b in bs]
    v = [torch.zeros(b.num_leaves, dtype=torch.int64).pin_memory() for b in bs]
    lo = [torch.zeros(b.num_grids + 1, dtype=torch.int64).pin_memory() for b in bs]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    tb.export_many(bs, o, m, v, lo, stream=stream)
    stream.synchronize()
    for i, r in enumerate(ref):
        assert np.array_equal(o[i].numpy(), r["origins"])
        assert np.array_equal(m[i].numpy().view(np.uint64), r["masks"])
        assert np.array_equal(v[i].numpy(), r["voxel_offset"])
        assert np.array_equal(lo[i].numpy(), r["leaf_offsets"])


def test_pipelined_steps_export_what_they_built():
    """The bench's end-to-end pattern: each step's outputs exported to pinned
    host memory on a copy stream while the next step runs, and freed on the
    compute stream once their export is done.  Every step's host arrays
    equal the oracle's for that step."""
    import torch
    ijk, off = synth.make("shells_b16_res64")
    chains = [[("refine", 2)], [("coarsen", 2)], [DIL]]
    want = [oracle.run_voxels(ijk, off, ops) for ops in chains]
    plan = tb.MultiPlan(chains)
    ijk_h, off_h = torch.from_numpy(ijk).pin_memory(), torch.from_numpy(off).pin_memory()
    copy = torch.cuda.Stream()
    stream = torch.cuda.current_stream()
    steps, pending = 4, None
    host = [[(torch.zeros((len(w["origins"]), 3), dtype=torch.int32).pin_memory(),
              torch.zeros((len(w["origins"]), 8), dtype=torch.int64).pin_memory(),
              torch.zeros((len(w["origins"]),), dtype=torch.int64).pin_memory(),
              torch.zeros((len(off),), dtype=torch.int64).pin_memory()) for w in want] for _ in range(steps)]
    for i in range(steps):
        b0 = tb.from_ijk(ijk_h, off_h)
        outs = plan(b0)
        ready = torch.cuda.Event()
        ready.record(stream)
        copy.wait_event(ready)
        tb.export_many(outs, *[[h[j] for h in host[i]] for j in range(4)], stream=copy)
        done = torch.cuda.Event()
        done.record(copy)
        if pending is not None:
            stream.wait_event(pending[1])
            for b in pending[0]:
                b.free()
        pending = (outs + [b0], done)
    stream.wait_event(pending[1])
    for b in pending[0]:
        b.free()
    torch.cuda.synchronize()
    for i in range(steps):
        for j, w in enumerate(want):
            o, m, v, lo = host[i][j]
            assert np.array_equal(o.numpy(), w["origins"]), (i, j)
            assert np.array_equal(m.numpy().view(np.uint64), w["masks"]), (i, j)
            assert np.array_equal(v.numpy(), w["voxel_offset"]), (i, j)
            assert np.array_equal(lo.numpy(), w["leaf_offsets"]), (i, j)


def test_pyramid_b48_one_multi_call():
    # the same eight pyramid levels as one tb_multi call (one launch, fused passes)
    import bench
    ijk, off = synth.make("pyramid_b48_res64")
    L0 = tb.from_ijk(dev(ijk), dev(off))
    outs = tb.multi(L0, [ops for _, ops in bench.PYRAMID])
    for (name, ops), b in zip(bench.PYRAMID, outs):
        assert_same(b.to_numpy(), oracle.run_voxels(ijk, off, ops), "multi " + name)
        b.validate()
