"""The allocation-free refinement entry point, tb_refine_static.

Some callers cannot call cudaMalloc: applications that reserve all device
memory in their own arena, or code that runs where the CUDA allocator must not
be entered.  tb_refine_static takes the input leaves and caller-owned output
buffers and keeps its scratch in a static device array.  These tests call it
through the C ABI twice in a row and require both results to equal
tb_refine's bit for bit -- the tolerance of every parity test in this suite,
since the result is a unique set in a total order.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

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
    counts = (ctypes.c_int64 * 3)()
    origins, masks, offs = src.tensor("origins"), src.tensor("masks"), src.tensor("leaf_offsets")
    st = lib.tb_refine_static(ctypes.c_void_p(origins.data_ptr() if src.num_leaves else 0),
                              ctypes.c_void_p(masks.data_ptr() if src.num_leaves else 0),
                              ctypes.c_void_p(offs.data_ptr()), src.num_grids, src.num_leaves,
                              ctypes.byref(ob), counts, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, [int(c) for c in counts]


def assert_matches(t, counts, ref):
    L, NL, NU = counts
    assert (L, NL, NU) == (ref.num_leaves, ref.num_lowers, ref.num_uppers)
    exp = ref.to_numpy()
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
    cap = 8 * src.num_leaves
    for _ in range(2):   # the scratch array keeps the previous call's contents
        ob, t = caller_buffers(src.num_grids, cap, cap)
        st, counts = call_static(lib, src, ob)
        assert st == 0, tb.lib().tb_last_error()
        assert_matches(t, counts, ref)


def test_static_refine_reports_small_capacity(lib):
    ijk, off = synth.make("pr1_b2_res32")
    src = tb.from_ijk(torch.from_numpy(ijk).cuda(), torch.from_numpy(off).cuda())
    ob, t = caller_buffers(src.num_grids, 10, 10)
    st, counts = call_static(lib, src, ob)
    assert st == 7 and counts[0] == tb.refine(src).num_leaves
    assert int(t["origins"].min()) == -7 and int(t["origins"].max()) == -7   # nothing written
    ob, t = caller_buffers(src.num_grids, counts[0], counts[0])
    st, counts2 = call_static(lib, src, ob)
    assert st == 0 and counts2 == counts
    assert_matches(t, counts2, tb.refine(src))
