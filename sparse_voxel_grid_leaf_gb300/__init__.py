"""Batched generated-topology passes for sparse voxel grids on GB300.

Python binding of ``libtb.so`` (C ABI in ``include/tb.h``).  Every step of a
pass runs in the library's CUDA kernels; this module only marshals arguments
(pointers, sizes, the current torch CUDA stream) and exposes the resulting
device arrays as zero-copy torch tensors.  There is no CPU fallback: calling
any op without the built library raises ``TBError``.

Operations follow fVDB PR #757 ("Batched leaf-mask topology construction for
generated conv grids", Summary items 1-2) and the ijk front end named in its
Follow-ups paragraph:

* ``from_ijk(ijk, offsets)``  jagged voxel coordinates -> batch
* ``from_leaves(origins, masks, offsets)``  jagged leaves -> batch
* ``refine(b, f)``, ``coarsen(b, f)``  f in {2, 4, 8}
* ``box_dilate(b, lo, hi)``  Minkowski sum with [lo, hi]^3 (unit boxes)
* ``chain(b, ops)``  several passes with intermediate results on the device
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, Iterable, Optional, Sequence, Tuple

import numpy as np

from . import synth  # noqa: F401  (seeded workloads; no method arithmetic)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtb.so")

TB_OK = 0
STATUS_NAMES = {0: "TB_OK", 1: "TB_ERR_INVALID_ARG", 2: "TB_ERR_OOM", 3: "TB_ERR_CUDA",
                4: "TB_ERR_COORD_OVERFLOW", 5: "TB_ERR_NOT_CANONICAL", 6: "TB_ERR_DEVICE_TIMEOUT",
                7: "TB_ERR_TOO_LARGE", 8: "TB_ERR_INTERNAL"}
OP_REFINE, OP_COARSEN, OP_BOX_DILATE = 0, 1, 2


class TBError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class _Op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("factor", ctypes.c_int32),
                ("lo", ctypes.c_int32 * 3), ("hi", ctypes.c_int32 * 3)]


class _View(ctypes.Structure):
    _fields_ = [("num_grids", ctypes.c_int32), ("device", ctypes.c_int32),
                ("num_leaves", ctypes.c_int64), ("num_lowers", ctypes.c_int64),
                ("num_uppers", ctypes.c_int64), ("leaf_offsets_host", ctypes.c_void_p),
                ("bbox", ctypes.c_int32 * 6)] + \
               [(n, ctypes.c_void_p) for n in (
                   "leaf_offsets", "origins", "masks", "voxel_offset", "word_prefix", "leaf_bbox",
                   "leaf_grid", "leaf_parent", "voxel_counts", "grid_bbox", "node_counts",
                   "lower_offsets", "upper_offsets", "lower_origins", "lower_parent", "upper_origins")] + \
               [("build_slots", ctypes.c_int64), ("build_source_leaves", ctypes.c_int64),
                ("build_key_bits", ctypes.c_int32), ("build_digit_passes", ctypes.c_int32),
                ("num_voxels", ctypes.c_int64), ("build_member_ctas", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class _KStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


_lib = None
_lib_lock = threading.Lock()


def lib():
    """The loaded ``libtb.so`` (raises ``TBError`` if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise TBError(-1, "libtb.so is not built (run __graft_entry__.build() or "
                                  "python -m sparse_voxel_grid_leaf_gb300._build)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            pp = ctypes.POINTER(ctypes.c_void_p)
            sig = {
                "tb_from_ijk": [vp, vp, i32, i64, vp, vp, pp],
                "tb_from_leaves": [vp, vp, vp, i32, i64, vp, vp, pp],
                "tb_refine": [vp, i32, vp, vp, pp],
                "tb_coarsen": [vp, i32, vp, vp, pp],
                "tb_box_dilate": [vp, vp, vp, vp, vp, pp],
                "tb_chain": [vp, vp, i32, vp, vp, pp],
                "tb_multi": [vp, vp, vp, i32, vp, vp, pp],
                "tb_refine_masked": [vp, vp, i32, vp, vp, pp],
                "tb_kernel_map": [vp, vp, vp, vp, i32, i32, vp, i64, vp],
                "tb_stride1_box": [i32, i32, vp, vp],
                "tb_selftest_wait": [i32, i32, vp],
                "tb_batch_export_many": [vp, i32, vp, vp, vp, vp, vp],
                "tb_validate": [vp, vp],
                "tb_batch_get_view": [vp, ctypes.POINTER(_View)],
                "tb_batch_export": [vp, vp, vp, vp, vp, vp],
                "tb_batch_free": [vp, vp],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.tb_last_error.restype = ctypes.c_char_p
            L.tb_last_error.argtypes = []
            L.tb_version.restype = ctypes.c_int32
            L.tb_kernel_launch_count.restype = ctypes.c_int64
            L.tb_profile_enable.argtypes = [ctypes.c_int32]
            L.tb_profile_enable.restype = ctypes.c_int
            L.tb_profile_read.argtypes = [ctypes.POINTER(_KStat), ctypes.c_int32]
            L.tb_profile_read.restype = ctypes.c_int32
            L.tb_set_launch_mode.argtypes = [ctypes.c_int32]
            L.tb_set_launch_mode.restype = ctypes.c_int32
            L.tb_set_node_mode.argtypes = [ctypes.c_int32]
            L.tb_set_node_mode.restype = ctypes.c_int32
            L.tb_set_kmap_mode.argtypes = [ctypes.c_int32]
            L.tb_set_kmap_mode.restype = ctypes.c_int32
            _lib = L
        return _lib


def _check(st: int):
    if st != TB_OK:
        raise TBError(st, lib().tb_last_error().decode())


_RAW_STREAM = None


def _stream(stream=None) -> int:
    """Raw cudaStream_t of `stream` (default: torch's current stream)."""
    global _RAW_STREAM
    if stream is not None:
        return int(getattr(stream, "cuda_stream", stream) or 0)
    if _RAW_STREAM is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        dev = torch._C._cuda_getDevice
        if raw is not None:
            _RAW_STREAM = lambda: raw(dev())
        else:
            _RAW_STREAM = lambda: torch.cuda.current_stream().cuda_stream
    return int(_RAW_STREAM())


def selftest_wait(set_flag: bool, spin_limit: int = 1 << 16, stream=None):
    """Failure-detection self-test: a bounded device wait on a flag that is
    preset or never set; raises TBError(TB_ERR_DEVICE_TIMEOUT) when it ran out."""
    _check(lib().tb_selftest_wait(1 if set_flag else 0, int(spin_limit), ctypes.c_void_p(_stream(stream))))


def kernel_launch_count() -> int:
    """Kernels launched through the library by the calling thread so far."""
    return int(lib().tb_kernel_launch_count())


LAUNCH_MODES = {"auto": 0, "grid": 1, "member": 2}


def set_launch_mode(mode: str) -> str:
    """Launch shape of the pass kernel for the whole process: "auto" (member
    launches -- one cluster per grid of every chain -- where every grid is
    small, else the whole-grid kernel), "grid" or "member".  Returns the
    previous mode."""
    prev = lib().tb_set_launch_mode(LAUNCH_MODES[mode])
    if prev < 0:
        raise ValueError("launch mode %r" % (mode,))
    return {v: k for k, v in LAUNCH_MODES.items()}[prev]


def set_node_mode(mode: str) -> str:
    """How the whole-grid kernel orders a pass's output leaves, for the whole
    process: "auto" (lower-node child masks where the output's lower nodes are
    few, else the radix sort) or "sort".  Returns the previous mode."""
    prev = lib().tb_set_node_mode({"auto": 0, "sort": 1}[mode])
    if prev < 0:
        raise ValueError("node mode %r" % (mode,))
    return {0: "auto", 1: "sort"}[prev]


KMAP_MODES = {"auto": 0, "staged": 1, "staged_prepass": 2, "tabulated": 3, "per_entry": 4}


def set_kmap_mode(mode: str) -> str:
    """Which kernel writes ``kernel_map``, for the whole process: "auto",
    "staged", "staged_prepass", "tabulated" or "per_entry" (each where the box
    allows it, else per entry).  Returns the previous mode."""
    prev = lib().tb_set_kmap_mode(KMAP_MODES[mode])
    if prev < 0:
        raise ValueError("kmap mode %r" % (mode,))
    return {v: k for k, v in KMAP_MODES.items()}[prev]


def profile_enable(on=True):
    """Times every library kernel of this thread with CUDA events on its stream
    (``on`` = 2 also stamps the pass kernel's phase boundaries)."""
    lib().tb_profile_enable(int(on))


def profile_read() -> Dict[str, Tuple[int, float]]:
    """{kernel name: (launches, total ms)} since the last read; waits for the events."""
    arr = (_KStat * 64)()
    n = lib().tb_profile_read(arr, 64)
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(min(n, 64))}


class _CAI:
    """__cuda_array_interface__ holder that keeps its batch alive."""

    def __init__(self, owner, ptr, shape, typestr):
        self._owner = owner
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 2, "strides": None}


_ARRAYS = {
    # name: (dtype typestr, numpy dtype, shape function of (B, L, NL, NU))
    "leaf_offsets": ("<i8", np.int64, lambda B, L, NL, NU: (B + 1,)),
    "origins": ("<i4", np.int32, lambda B, L, NL, NU: (L, 3)),
    "masks": ("<i8", np.uint64, lambda B, L, NL, NU: (L, 8)),
    "voxel_offset": ("<i8", np.int64, lambda B, L, NL, NU: (L,)),
    "word_prefix": ("<i8", np.uint64, lambda B, L, NL, NU: (L,)),
    "leaf_bbox": ("<i4", np.int32, lambda B, L, NL, NU: (L, 6)),
    "leaf_grid": ("<i4", np.int32, lambda B, L, NL, NU: (L,)),
    "leaf_parent": ("<i4", np.int32, lambda B, L, NL, NU: (L,)),
    "voxel_counts": ("<i8", np.int64, lambda B, L, NL, NU: (B,)),
    "grid_bbox": ("<i4", np.int32, lambda B, L, NL, NU: (B, 6)),
    "node_counts": ("<i4", np.int32, lambda B, L, NL, NU: (B, 3)),
    "lower_offsets": ("<i8", np.int64, lambda B, L, NL, NU: (B + 1,)),
    "upper_offsets": ("<i8", np.int64, lambda B, L, NL, NU: (B + 1,)),
    "lower_origins": ("<i4", np.int32, lambda B, L, NL, NU: (NL, 3)),
    "lower_parent": ("<i4", np.int32, lambda B, L, NL, NU: (NL,)),
    "upper_origins": ("<i4", np.int32, lambda B, L, NL, NU: (NU, 3)),
}
ARRAY_NAMES = tuple(_ARRAYS)


class Batch:
    """A batch of grids produced by the library (owns its device memory).

    Sizes and device arrays are read lazily from the library's view of the
    batch, so passing batches from one call to the next costs nothing here."""

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)
        self._v = None

    def _view(self) -> _View:
        if self._v is None:
            v = _View()
            _check(lib().tb_batch_get_view(self.handle, ctypes.byref(v)))
            self._v = v
        return self._v

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise TBError(1, "batch already freed")
        return self._h

    num_grids = property(lambda self: int(self._view().num_grids))
    num_leaves = property(lambda self: int(self._view().num_leaves))
    num_lowers = property(lambda self: int(self._view().num_lowers))
    num_uppers = property(lambda self: int(self._view().num_uppers))
    device = property(lambda self: int(self._view().device))
    bbox = property(lambda self: tuple(int(x) for x in self._view().bbox))
    build_slots = property(lambda self: int(self._view().build_slots))
    build_source_leaves = property(lambda self: int(self._view().build_source_leaves))
    build_key_bits = property(lambda self: int(self._view().build_key_bits))
    build_digit_passes = property(lambda self: int(self._view().build_digit_passes))
    # CTAs per member of the member launch that built the batch; 0: whole-grid kernel
    build_member_ctas = property(lambda self: int(self._view().build_member_ctas))
    num_voxels = property(lambda self: int(self._view().num_voxels))

    @property
    def leaf_offsets_host(self) -> np.ndarray:
        v = self._view()
        return np.ctypeslib.as_array(ctypes.cast(v.leaf_offsets_host, ctypes.POINTER(ctypes.c_int64)),
                                     shape=(v.num_grids + 1,)).copy()

    def tensor(self, name: str):
        """Zero-copy torch CUDA tensor of one device array of the batch (64-bit
        masks and word prefixes are exposed as int64 bit patterns)."""
        import torch
        typestr, npdt, shp = _ARRAYS[name]
        v = self._view()
        shape = shp(v.num_grids, v.num_leaves, v.num_lowers, v.num_uppers)
        ptr = getattr(v, name)
        dev = "cuda:%d" % v.device
        if not ptr or int(np.prod(shape)) == 0:
            return torch.empty(shape, dtype=_torch_dtype(npdt), device=dev)
        return torch.as_tensor(_CAI(self, ptr, shape, typestr), device=dev)

    def __getattr__(self, name):
        if name in _ARRAYS:
            return self.tensor(name)
        raise AttributeError(name)

    def to_numpy(self, names: Sequence[str] = ARRAY_NAMES) -> Dict[str, np.ndarray]:
        """Copies arrays to host numpy (synchronizes the current stream)."""
        import torch
        out = {}
        for n in names:
            out[n] = self.tensor(n).cpu().numpy()
            if _ARRAYS[n][1] == np.uint64:
                out[n] = out[n].view(np.uint64)
        torch.cuda.current_stream().synchronize()
        return out

    def validate(self, stream=None):
        _check(lib().tb_validate(self.handle, ctypes.c_void_p(_stream(stream))))

    def free(self, stream=None):
        if self._h is not None:
            lib().tb_batch_free(self._h, ctypes.c_void_p(_stream(stream)))
            self._h = None
            self._v = None

    def __del__(self):
        try:
            if self._h is not None and _lib is not None:
                _lib.tb_batch_free(self._h, None)
                self._h = None
        except Exception:
            pass


def _torch_dtype(npdt):
    import torch
    return {np.int32: torch.int32, np.int64: torch.int64, np.uint64: torch.int64}[npdt]


def _ptr(x) -> Tuple[int, object]:
    """(address, keep-alive) of a torch tensor or numpy array, C-contiguous."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if not x.is_contiguous():
                x = x.contiguous()
            return x.data_ptr(), x
    except ImportError:
        pass
    a = np.ascontiguousarray(x)
    return a.ctypes.data, a


def _new(fn, *args) -> Batch:
    out = ctypes.c_void_p()
    _check(fn(*args, ctypes.byref(out)))
    return Batch(out.value)


def from_ijk(ijk, offsets, stream=None) -> Batch:
    """Batch from int32 voxel coordinates ``ijk [N,3]`` and int64 ``offsets [B+1]``
    (torch tensors on the GPU or the host, or numpy arrays)."""
    pi, ki = _ptr(ijk)
    po, ko = _ptr(offsets)
    B = int(ko.shape[0]) - 1
    N = int(ki.shape[0]) if ki.ndim else 0
    _dtype_check(ki, "int32")
    _dtype_check(ko, "int64")
    return _new(lib().tb_from_ijk, ctypes.c_void_p(pi), ctypes.c_void_p(po), B, N, None,
                ctypes.c_void_p(_stream(stream)))


def from_leaves(origins, masks, offsets, stream=None) -> Batch:
    """Batch from leaves: int32 ``origins [L,3]``, uint64 ``masks [L,8]``, int64 ``offsets [B+1]``."""
    po, ko = _ptr(origins)
    pm, km = _ptr(masks)
    pf, kf = _ptr(offsets)
    _dtype_check(ko, "int32")
    _dtype_check(km, "uint64", "int64")
    _dtype_check(kf, "int64")
    return _new(lib().tb_from_leaves, ctypes.c_void_p(po), ctypes.c_void_p(pm), ctypes.c_void_p(pf),
                int(kf.shape[0]) - 1, int(ko.shape[0]), None, ctypes.c_void_p(_stream(stream)))


def _dtype_check(x, *names):
    n = str(x.dtype).replace("torch.", "")
    if n not in names:
        raise TBError(1, "expected dtype %s, got %s" % ("/".join(names), n))


def refine(b: Batch, factor: int = 2, stream=None) -> Batch:
    return _new(lib().tb_refine, b.handle, int(factor), None, ctypes.c_void_p(_stream(stream)))


def refine_masked(b: Batch, voxel_mask, factor: int = 2, stream=None) -> Batch:
    """Refinement of the voxels whose flag is set: ``voxel_mask`` holds one
    bool/uint8 per active voxel of ``b`` in the batch's voxel order (grid by
    grid, leaf by leaf, ascending bit index), on the GPU or the host."""
    import torch
    if isinstance(voxel_mask, torch.Tensor) and voxel_mask.dtype == torch.bool:
        voxel_mask = voxel_mask.view(torch.uint8)
    elif isinstance(voxel_mask, np.ndarray) and voxel_mask.dtype == np.bool_:
        voxel_mask = voxel_mask.view(np.uint8)
    pm, km = _ptr(voxel_mask)
    _dtype_check(km, "uint8")
    return _new(lib().tb_refine_masked, b.handle, ctypes.c_void_p(pm), int(factor), None,
                ctypes.c_void_p(_stream(stream)))


def coarsen(b: Batch, factor: int = 2, stream=None) -> Batch:
    return _new(lib().tb_coarsen, b.handle, int(factor), None, ctypes.c_void_p(_stream(stream)))


def box_dilate(b: Batch, lo=(-1, -1, -1), hi=(1, 1, 1), stream=None) -> Batch:
    lo_a = (ctypes.c_int32 * 3)(*lo)
    hi_a = (ctypes.c_int32 * 3)(*hi)
    return _new(lib().tb_box_dilate, b.handle, lo_a, hi_a, None, ctypes.c_void_p(_stream(stream)))


_OPS_CACHE: Dict[Tuple, Tuple] = {}


def make_ops(ops: Iterable[Tuple]):
    """Op tuples ``("refine", f)``, ``("coarsen", f)``, ``("dilate", lo, hi)`` -> C array."""
    ops = tuple((o[0],) + tuple(tuple(x) if isinstance(x, (list, tuple)) else x for x in o[1:]) for o in ops)
    hit = _OPS_CACHE.get(ops)
    if hit is not None:
        return hit
    arr = (_Op * max(1, len(ops)))()
    for i, op in enumerate(ops):
        if op[0] == "refine":
            arr[i].kind, arr[i].factor = OP_REFINE, int(op[1])
        elif op[0] == "coarsen":
            arr[i].kind, arr[i].factor = OP_COARSEN, int(op[1])
        elif op[0] == "dilate":
            arr[i].kind, arr[i].factor = OP_BOX_DILATE, 1
            for a in range(3):
                arr[i].lo[a], arr[i].hi[a] = int(op[1][a]), int(op[2][a])
        else:
            raise TBError(1, "unknown op %r" % (op[0],))
    if len(_OPS_CACHE) < 1024:
        _OPS_CACHE[ops] = (arr, len(ops))
    return arr, len(ops)


def chain(b: Batch, ops: Iterable[Tuple], stream=None) -> Batch:
    arr, n = make_ops(ops)
    return _new(lib().tb_chain, b.handle, arr, n, None, ctypes.c_void_p(_stream(stream)))


class MultiPlan:
    """Chains of ops marshalled once, for repeated tb_multi calls over
    different batches: ``plan = MultiPlan(chains); outs = plan(batch)``."""

    def __init__(self, chains: Sequence[Iterable[Tuple]]):
        chains = [list(c) for c in chains]
        flat = [op for c in chains for op in c]
        self.n = len(chains)
        self._arr, _ = make_ops(flat)
        self._lens = (ctypes.c_int32 * self.n)(*[len(c) for c in chains])
        self._outs = (ctypes.c_void_p * self.n)()
        self._outs_p = ctypes.cast(self._outs, ctypes.POINTER(ctypes.c_void_p))
        self._fn = lib().tb_multi

    def __call__(self, b: Batch, stream=None) -> list:
        _check(self._fn(b.handle, self._arr, self._lens, self.n, None, ctypes.c_void_p(_stream(stream)),
                        self._outs_p))
        outs = self._outs
        return [Batch(outs[i]) for i in range(self.n)]


def multi(b: Batch, chains: Sequence[Iterable[Tuple]], stream=None) -> list:
    """Several chains of ops over the same batch in one call (one launch, one
    readback); returns one batch per chain."""
    return MultiPlan(chains)(b, stream)


# Convolution-topology aliases named by fVDB PR #757 (Summary and Measurements).
def conv_grid_k2s2(b: Batch, stream=None) -> Batch:
    """conv_grid with kernel 2, stride 2: coarsening by 2."""
    return coarsen(b, 2, stream)


def conv_transpose_grid_k2s2(b: Batch, stream=None) -> Batch:
    """conv_transpose_grid with kernel 2, stride 2: refinement by 2."""
    return refine(b, 2, stream)


def conv_grid_k3s1(b: Batch, stream=None) -> Batch:
    """conv_grid with kernel 3, stride 1: dilation by [-1, 1]^3."""
    return box_dilate(b, (-1, -1, -1), (1, 1, 1), stream)


def conv_transpose_grid_k3s2(b: Batch, stream=None) -> Batch:
    """conv_transpose_grid with kernel 3, stride 2: refine by 2, then the {-1,0}^3 pad."""
    return chain(b, [("refine", 2), ("dilate", (-1, -1, -1), (0, 0, 0))], stream)


def kernel_map(b_in: Batch, b_out: Batch, lo=(-1, -1, -1), hi=(1, 1, 1), stride: int = 1,
               transposed: bool = False, stream=None):
    """Kernel map of a sparse convolution from ``b_in`` to ``b_out``: an int32
    CUDA tensor ``[V_out, K]`` (K = box volume, offsets x-major) of input voxel
    indices, -1 where the input voxel is absent.  Input voxel for output voxel
    p and offset d: p + d (stride 1), 2 p + d (stride 2), or (p - d) / 2 when
    even (stride 2, transposed)."""
    import torch
    K = 1
    for a in range(3):
        K *= int(hi[a]) - int(lo[a]) + 1
    v = b_out._view()
    out = torch.empty((int(v.num_voxels), K), dtype=torch.int32, device="cuda:%d" % v.device)
    lo_a = (ctypes.c_int32 * 3)(*lo)
    hi_a = (ctypes.c_int32 * 3)(*hi)
    _check(lib().tb_kernel_map(b_in.handle, b_out.handle, lo_a, hi_a, int(stride), 1 if transposed else 0,
                               ctypes.c_void_p(out.data_ptr() if out.numel() else 0), int(out.numel()),
                               ctypes.c_void_p(_stream(stream))))
    return out


def stride1_box(kernel_size: int, transpose: bool = False) -> Tuple[Tuple[int, int, int], Tuple[int, int, int]]:
    """Box of the stride-1 topology of a uniform kernel of size K (1..15), from
    the library (tb_stride1_box): [-floor((K-1)/2), ceil((K-1)/2)] per axis
    for conv_grid (for even K the extra offset is on the positive side, a
    reading the pages leave open), and its mirror image for
    conv_transpose_grid."""
    lo = (ctypes.c_int32 * 3)()
    hi = (ctypes.c_int32 * 3)()
    _check(lib().tb_stride1_box(int(kernel_size), 1 if transpose else 0, lo, hi))
    return tuple(lo), tuple(hi)


def conv_grid_stride1(b: Batch, kernel_size: int, stream=None) -> Batch:
    """conv_grid with a uniform kernel of size K and stride 1 (PR #757 Summary
    item 2): one box dilation."""
    lo, hi = stride1_box(kernel_size)
    return box_dilate(b, lo, hi, stream)


def conv_transpose_grid_stride1(b: Batch, kernel_size: int, stream=None) -> Batch:
    """conv_transpose_grid with a uniform kernel of size K and stride 1: the
    mirrored box."""
    lo, hi = stride1_box(kernel_size, transpose=True)
    return box_dilate(b, lo, hi, stream)


def dilated_grid(b: Batch, radius: int, stream=None) -> Batch:
    """Dilation by an integer radius r (0..7): the box [-r, r]^3."""
    r = int(radius)
    return box_dilate(b, (-r, -r, -r), (r, r, r), stream)


def export_host(b: Batch, origins: np.ndarray, masks: np.ndarray, voxel_offset: Optional[np.ndarray] = None,
                leaf_offsets: Optional[np.ndarray] = None, stream=None):
    """Enqueues copies of leaf records into host buffers (caller synchronizes)."""
    def p(x):
        return None if x is None else ctypes.c_void_p(_ptr(x)[0])
    _check(lib().tb_batch_export(b.handle, p(origins), p(masks), p(voxel_offset), p(leaf_offsets),
                                 ctypes.c_void_p(_stream(stream))))


class ExportPlan:
    """Destinations of tb_batch_export_many marshalled once, for repeated
    exports of different batches into the same buffers:
    ``plan = ExportPlan(origins, masks, voxel_offset, leaf_offsets)``, then
    ``plan(batches)``.  Each argument is a list with one buffer (or None) per
    batch, or None to skip that array; the buffers must stay alive."""

    def __init__(self, origins=None, masks=None, voxel_offset=None, leaf_offsets=None):
        lists = [x for x in (origins, masks, voxel_offset, leaf_offsets) if x is not None]
        self.n = len(lists[0]) if lists else 0
        self._keep = []

        def plist(xs):
            if xs is None:
                return None
            arr = (ctypes.c_void_p * self.n)()
            for i, x in enumerate(xs):
                if x is not None:
                    p, k = _ptr(x)
                    self._keep.append(k)
                    arr[i] = p
            return arr
        self._lists = [plist(origins), plist(masks), plist(voxel_offset), plist(leaf_offsets)]
        self._hs = (ctypes.c_void_p * self.n)()
        self._fn = lib().tb_batch_export_many

    def __call__(self, batches: Sequence[Batch], stream=None):
        if len(batches) != self.n:
            raise TBError(1, "export plan for %d batches called with %d" % (self.n, len(batches)))
        for i, b in enumerate(batches):
            self._hs[i] = b.handle.value
        _check(self._fn(self._hs, self.n, *self._lists, ctypes.c_void_p(_stream(stream))))


def export_many(batches: Sequence[Batch], origins=None, masks=None, voxel_offset=None, leaf_offsets=None,
                stream=None):
    """Enqueues the copies of several batches' leaf records (one list entry per
    batch; a list, or an entry, may be None to skip): arrays of 1 MiB or more
    through the copy engines, the smaller ones whose destination the device
    can write (device or pinned host memory) through one copy kernel."""
    n = len(batches)
    keep = []

    def plist(xs):
        if xs is None:
            return None
        arr = (ctypes.c_void_p * n)()
        for i, x in enumerate(xs):
            if x is not None:
                p, k = _ptr(x)
                keep.append(k)
                arr[i] = p
        return arr
    hs = (ctypes.c_void_p * n)(*[b.handle.value for b in batches])
    _check(lib().tb_batch_export_many(hs, n, plist(origins), plist(masks), plist(voxel_offset),
                                      plist(leaf_offsets), ctypes.c_void_p(_stream(stream))))
