"""The allocation-free refinement entry point, tb_refine_static.

Some callers cannot call cudaMalloc: applications that reserve all device
memory in their own arena, or code that runs where the CUDA allocator must not
be entered.  tb_refine_static takes the input leaves and caller-owned output
buffers and keeps its scratch in a static device array.  These tests call it
through the C ABI, twice in a row where the result is compared (the array
keeps the previous call's contents), and require every output array to equal
the CPU oracle's refinement and tb_refine's bit for bit -- the tolerance of
every parity test in this suite, since the result is a unique set in a total
order.  They also cover its promises on unsorted input with duplicates, empty
batches, inputs too large for the array and host-resident pointers.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from sparse_voxel_grid_leaf_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import sparse_voxel_grid_leaf_gb300 as tb  # noqa: E402

PER_LEAF = [("origins", torch.int32, (3,)), ("masks", torch.int64, (8,)), ("voxel_offset", torch.int64, ()),
            ("word_prefix", torch.int64, ()), ("leaf_bbox", torch.int32, (6,)), ("leaf_grid", torch.int32, ()),
            ("leaf_parent", torch.int32, ())]


class OutBuffers(ctypes.Structure):
    _fields_ = [("leaf_capacity", ctypes.c_int64), ("lower_capacity", ctypes.c_int64),
                ("upper_capacity", ctypes.c_int64)] + \
               [(n, ctypes.c_void_p) for n in (
                   "leaf_offsets", "lower_offsets", "upper_offsets", "voxel_counts", "grid_bbox", "node_counts",
                   "origins", "masks", "voxel_offset", "word_prefix", "leaf_bbox", "leaf_grid", "leaf_parent",
                   "lower_origins", "lower_parent", "upper_origins")]


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    L = tb.lib()
    L.tb_refine_static.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                   ctypes.c_int64, ctypes.POINTER(OutBuffers), ctypes.c_void_p, ctypes.c_void_p]
    L.tb_refine_static.restype = ctypes.c_int
    return L


def caller_buffers(B, leaf_cap, node_cap):
    """Output buffers the caller owns (allocated here by torch, i.e. by the caller)."""
    t = {"leaf_offsets": torch.full((B + 1,), -7, dtype=torch.int64, device="cuda"),
         "lower_offsets": torch.full((B + 1,), -7, dtype=torch.int64, device="cuda"),
         "upper_offsets": torch.full((B + 1,), -7, dtype=torch.int64, device="cuda"),
         "voxel_counts": torch.full((B,), -7, dtype=torch.int64, device="cuda"),
         "grid_bbox": torch.full((B, 6), -7, dtype=torch.int32, device="cuda"),
         "node_counts": torch.full((B, 3), -7, dtype=torch.int32, device="cuda"),
         "lower_origins": torch.full((node_cap, 3), -7, dtype=torch.int32, device="cuda"),
         "lower_parent": torch.full((node_cap,), -7, dtype=torch.int32, device="cuda"),
         "upper_origins": torch.full((node_cap, 3), -7, dtype=torch.int32, device="cuda")}
    for name, dt, shape in PER_LEAF:
        t[name] = torch.full((leaf_cap,) + shape, -7, dtype=dt, device="cuda")
    ob = OutBuffers()
    ob.leaf_capacity, ob.lower_capacity, ob.upper_capacity = leaf_cap, node_cap, node_cap
    for k, v in t.items():
        setattr(ob, k, v.data_ptr())
    return ob, t


def call_static(lib, src, ob):
    origins, masks, offs = src.tensor("origins"), src.tensor("masks"), src.tensor("leaf_offsets")
    return call_static_raw(lib, origins, masks, offs, src.num_grids, src.num_leaves, ob)


def call_static_raw(lib, origins, masks, offs, B, L, ob):
    """One call through the C ABI; origins/masks/offsets are torch tensors or
    numpy arrays (host memory)."""
    counts = (ctypes.c_int64 * 3)(-1, -1, -1)
    ptr = lambda x: 0 if x is None else (x.ctypes.data if isinstance(x, np.ndarray) else x.data_ptr())
    st = lib.tb_refine_static(ctypes.c_void_p(ptr(origins) if L else 0), ctypes.c_void_p(ptr(masks) if L else 0),
                              ctypes.c_void_p(ptr(offs)), B, L, ctypes.byref(ob), counts,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, [int(c) for c in counts]


def untouched(t):
    return all(int(v.min()) == -7 and int(v.max()) == -7 for v in t.values() if v.numel())


def assert_matches(t, counts, ref):
    """ref: a tb batch, or the oracle's arrays (a dict)."""
    exp = ref if isinstance(ref, dict) else ref.to_numpy()
    L, NL, NU = counts
    assert (L, NL, NU) == (len(exp["origins"]), len(exp["lower_origins"]), len(exp["upper_origins"]))
    got = {k: v.cpu().numpy() for k, v in t.items()}
    for name, _, _ in PER_LEAF:
        g = got[name][:L]
        e = exp[name].view(g.dtype) if exp[name].dtype != g.dtype else exp[name]
        assert np.array_equal(g, e), name
    for name in ("lower_origins", "lower_parent"):
        assert np.array_equal(got[name][:NL], exp[name]), name
    assert np.array_equal(got["upper_origins"][:NU], exp["upper_origins"])
    for name in ("leaf_offsets", "lower_offsets", "upper_offsets", "voxel_counts", "grid_bbox", "node_counts"):
        assert np.array_equal(got[name], exp[name]), name


@pytest.mark.parametrize("workload", ["shells_b16_res64", "mixed"])
def test_static_refine_equals_refine_twice(lib, workload):
    if workload == "mixed":   # empty members, negative octants, +-4096 tile crossings
        ijk, off = synth.random_voxels(6, 500, 70, seed=17, origin=(-4130, -40, 4060), empty=(0, 3))
    else:
        ijk, off = synth.make(workload)
    src = tb.from_ijk(torch.from_numpy(ijk).cuda(), torch.from_numpy(off).cuda())
    ref = tb.refine(src, 2)
    want = oracle.run_voxels(ijk, off, [("refine", 2)])
    cap = 8 * src.num_leaves
    for _ in range(2):   # the scratch array keeps the previous call's contents
        ob, t = caller_buffers(src.num_grids, cap, cap)
        st, counts = call_static(lib, src, ob)
        assert st == 0, tb.lib().tb_last_error()
        assert_matches(t, counts, want)
        assert_matches(t, counts, ref)


def test_static_refine_unsorted_duplicates_against_oracle(lib):
    """Input in any order with duplicate origins merges: leaves shuffled, each
    split into two half masks, plus all-zero leaves."""
    ijk, off = synth.random_voxels(5, 600, 40, seed=23, origin=(-4110, 4070, -30), empty=(2,))
    base = oracle.run_voxels(ijk, off)
    o, m, lo = base["origins"], base["masks"], base["leaf_offsets"]
    rng = np.random.default_rng(3)
    origins, masks, offs = [], [], [0]
    for g in range(len(lo) - 1):
        for i in rng.permutation(np.arange(lo[g], lo[g + 1])):
            half = m[i] & np.uint64(0x3333333333333333)
            origins += [o[i], o[i]]
            masks += [m[i] ^ half, half]
        origins.append(np.array([-16, 8, 4088], np.int32))
        masks.append(np.zeros(8, np.uint64))
        offs.append(len(origins))
    origins, masks = np.array(origins, np.int32), np.array(masks, np.uint64)
    offs = np.array(offs, np.int64)
    want = oracle.run_leaves(origins, masks, offs, [("refine", 2)])
    assert np.array_equal(want["origins"], oracle.run_voxels(ijk, off, [("refine", 2)])["origins"])
    d_o, d_m, d_off = (torch.from_numpy(x).cuda() for x in (origins, masks.view(np.int64), offs))
    B, L = len(offs) - 1, len(origins)
    for _ in range(2):
        ob, t = caller_buffers(B, 8 * L, 8 * L)
        st, counts = call_static_raw(lib, d_o, d_m, d_off, B, L, ob)
        assert st == 0, tb.lib().tb_last_error()
        assert_matches(t, counts, want)


def test_static_refine_empty_batches(lib):
    # B = 0; and B = 3 grids with no leaves: valid empty grids
    for B in (0, 3):
        offs = torch.zeros(B + 1, dtype=torch.int64, device="cuda")
        ob, t = caller_buffers(B, 4, 4)
        st, counts = call_static_raw(lib, None, None, offs, B, 0, ob)
        assert st == 0, tb.lib().tb_last_error()
        assert_matches(t, counts, oracle.run_voxels(np.zeros((0, 3), np.int32), np.zeros(B + 1, np.int64),
                                                     [("refine", 2)]))


def test_static_refine_too_large_writes_nothing(lib):
    # 80,660 leaves need more than the 32 MiB array (52 bytes per candidate,
    # 8 candidates per leaf): rejected before any launch
    L = 80660
    origins = torch.zeros((L, 3), dtype=torch.int32, device="cuda")
    origins[:, 0] = 8 * torch.arange(L, dtype=torch.int32, device="cuda")
    masks = torch.full((L, 8), -1, dtype=torch.int64, device="cuda")   # full leaves: 8 children each
    offs = torch.tensor([0, L], dtype=torch.int64, device="cuda")
    ob, t = caller_buffers(1, 16, 16)
    st, counts = call_static_raw(lib, origins, masks, offs, 1, L, ob)
    assert st == 7 and b"32 MiB" in tb.lib().tb_last_error()
    assert untouched(t) and counts == [-1, -1, -1]
    # a smaller prefix of the same leaves runs
    ob, t = caller_buffers(1, 16000, 16000)
    st, counts = call_static_raw(lib, origins[:2000], masks[:2000], torch.tensor([0, 2000], device="cuda"), 1,
                                 2000, ob)
    assert st == 0, tb.lib().tb_last_error()
    assert counts[0] == 16000


def test_static_refine_rejects_host_pointers(lib):
    ijk, off = synth.make("pr1_b2_res32")
    src = tb.from_ijk(torch.from_numpy(ijk).cuda(), torch.from_numpy(off).cuda())
    host_offs = src.tensor("leaf_offsets").cpu().numpy()
    ob, t = caller_buffers(src.num_grids, 8 * src.num_leaves, 8 * src.num_leaves)
    st, _ = call_static_raw(lib, src.tensor("origins"), src.tensor("masks"), host_offs, src.num_grids,
                            src.num_leaves, ob)
    assert st == 1 and b"device memory" in tb.lib().tb_last_error()
    host_out = np.zeros(8 * src.num_leaves * 3, np.int32)
    ob.origins = host_out.ctypes.data
    st, _ = call_static(lib, src, ob)
    assert st == 1 and b"device memory" in tb.lib().tb_last_error()
    assert untouched(t)


def test_static_refine_reports_small_capacity(lib):
    ijk, off = synth.make("pr1_b2_res32")
    src = tb.from_ijk(torch.from_numpy(ijk).cuda(), torch.from_numpy(off).cuda())
    ob, t = caller_buffers(src.num_grids, 10, 10)
    st, counts = call_static(lib, src, ob)
    assert st == 7 and counts[0] == tb.refine(src).num_leaves
    assert untouched(t)   # nothing written
    ob, t = caller_buffers(src.num_grids, counts[0], counts[0])
    st, counts2 = call_static(lib, src, ob)
    assert st == 0 and counts2 == counts
    assert_matches(t, counts2, tb.refine(src))
