"""CPU oracle of the batched generated-topology pass (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does.

The arithmetic lives in ``oracle.cpp`` (plain single-threaded C++ over
``std::set``, compiled with g++ into ``liboracle.so``); this module only builds
it and marshals numpy arrays.  Function provenance (fVDB PR #757, "Batched
leaf-mask topology construction for generated conv grids"):

* ``run_voxels`` / ``run_leaves`` -- the per-voxel definition of refine,
  coarsen and box dilation (Summary items 1 and 2), grouped into 8^3 leaves in
  canonical node order (Summary item 1, sort bullet) with the derived per-leaf
  and per-grid arrays (Summary item 1, writer bullet).
* Ops are given as tuples: ``("refine", f)``, ``("coarsen", f)`` with
  f in {2, 4, 8}, and ``("dilate", lo, hi)`` with per-axis integer bounds.

Parity pins: see ``tests/test_oracle_pins.py``.  The conventions r9-r11 of the
design notes (0-based per-grid voxel offsets, the 9-bit word-prefix packing and
the empty-grid bbox) are fixed readings with no worked example on the pages:
parity unpinned against the original library for those three conventions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Iterable, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OP_REFINE, OP_COARSEN, OP_DILATE = 0, 1, 2
STATUS_OK, STATUS_BAD_ARG, STATUS_OVERFLOW = 0, 1, 4


class _Op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("factor", ctypes.c_int32),
                ("lo", ctypes.c_int32 * 3), ("hi", ctypes.c_int32 * 3)]


def build(force: bool = False, extra_flags: Sequence[str] = (), out: str = _LIB, src: str = _SRC) -> str:
    """Compiles ``oracle.cpp`` with g++ (no GPU involved)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", *extra_flags, src, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def load(path: str = _LIB):
    lib = ctypes.CDLL(path)
    vp, i32p, i64p, u64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), \
        ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_uint64)
    lib.oracle_run_voxels.restype = vp
    lib.oracle_run_voxels.argtypes = [vp, vp, ctypes.c_int32, vp, ctypes.c_int32]
    lib.oracle_run_leaves.restype = vp
    lib.oracle_run_leaves.argtypes = [vp, vp, vp, ctypes.c_int32, vp, ctypes.c_int32]
    lib.oracle_status.restype = ctypes.c_int32
    lib.oracle_status.argtypes = [vp]
    lib.oracle_sizes.restype = None
    lib.oracle_sizes.argtypes = [vp, vp]
    lib.oracle_fill.restype = None
    lib.oracle_fill.argtypes = [vp] * 17
    lib.oracle_free.restype = None
    lib.oracle_free.argtypes = [vp]
    del i32p, i64p, u64p
    return lib


def _get():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
        return _lib


def make_ops(ops: Iterable[Tuple]) -> "ctypes.Array":
    ops = list(ops)
    arr = (_Op * max(1, len(ops)))()
    for i, op in enumerate(ops):
        name = op[0]
        if name == "refine":
            arr[i].kind, arr[i].factor = OP_REFINE, int(op[1])
        elif name == "coarsen":
            arr[i].kind, arr[i].factor = OP_COARSEN, int(op[1])
        elif name == "dilate":
            arr[i].kind, arr[i].factor = OP_DILATE, 1
            for a in range(3):
                arr[i].lo[a] = int(op[1][a])
                arr[i].hi[a] = int(op[2][a])
        else:
            raise ValueError("unknown op %r" % (name,))
    return arr, len(ops)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _collect(lib, h, B: int) -> Dict[str, np.ndarray]:
    st = lib.oracle_status(h)
    if st != STATUS_OK:
        lib.oracle_free(h)
        raise OracleError(st)
    sizes = np.zeros(3, np.int64)
    lib.oracle_sizes(h, _ptr(sizes))
    L, NL, NU = (int(s) for s in sizes)
    out = {
        "leaf_offsets": np.zeros(B + 1, np.int64),
        "origins": np.zeros((L, 3), np.int32),
        "masks": np.zeros((L, 8), np.uint64),
        "voxel_offset": np.zeros(L, np.int64),
        "word_prefix": np.zeros(L, np.uint64),
        "leaf_bbox": np.zeros((L, 6), np.int32),
        "leaf_grid": np.zeros(L, np.int32),
        "leaf_parent": np.zeros(L, np.int32),
        "voxel_counts": np.zeros(B, np.int64),
        "grid_bbox": np.zeros((B, 6), np.int32),
        "node_counts": np.zeros((B, 3), np.int32),
        "lower_offsets": np.zeros(B + 1, np.int64),
        "upper_offsets": np.zeros(B + 1, np.int64),
        "lower_origins": np.zeros((NL, 3), np.int32),
        "lower_parent": np.zeros(NL, np.int32),
        "upper_origins": np.zeros((NU, 3), np.int32),
    }
    order = ["leaf_offsets", "origins", "masks", "voxel_offset", "word_prefix", "leaf_bbox",
             "leaf_grid", "leaf_parent", "voxel_counts", "grid_bbox", "node_counts",
             "lower_offsets", "upper_offsets", "lower_origins", "lower_parent", "upper_origins"]
    lib.oracle_fill(h, *[_ptr(out[k]) for k in order])
    lib.oracle_free(h)
    return out


class OracleError(RuntimeError):
    def __init__(self, status: int):
        super().__init__("oracle status %d" % status)
        self.status = status


def run_voxels(ijk: np.ndarray, offsets: np.ndarray, ops: Iterable[Tuple] = (),
               lib=None) -> Dict[str, np.ndarray]:
    """Jagged voxels -> chain of ops -> canonical leaf topology (numpy arrays)."""
    lib = lib or _get()
    ijk = np.ascontiguousarray(ijk, np.int32).reshape(-1, 3)
    offsets = np.ascontiguousarray(offsets, np.int64)
    B = offsets.shape[0] - 1
    arr, n = make_ops(ops)
    h = lib.oracle_run_voxels(_ptr(ijk), _ptr(offsets), B, ctypes.cast(arr, ctypes.c_void_p), n)
    return _collect(lib, h, B)


def run_leaves(origins: np.ndarray, masks: np.ndarray, offsets: np.ndarray,
               ops: Iterable[Tuple] = (), lib=None) -> Dict[str, np.ndarray]:
    """Jagged leaves (origin, 512-bit mask) -> chain of ops -> canonical topology."""
    lib = lib or _get()
    origins = np.ascontiguousarray(origins, np.int32).reshape(-1, 3)
    masks = np.ascontiguousarray(masks, np.uint64).reshape(-1, 8)
    offsets = np.ascontiguousarray(offsets, np.int64)
    B = offsets.shape[0] - 1
    arr, n = make_ops(ops)
    h = lib.oracle_run_leaves(_ptr(origins), _ptr(masks), _ptr(offsets), B,
                              ctypes.cast(arr, ctypes.c_void_p), n)
    return _collect(lib, h, B)


def batch_voxels(result: Dict[str, np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
    """The active voxels of a result in the batch's voxel order -- grid by
    grid, leaf by leaf in canonical order, within a leaf by ascending bit
    index n = 64 x + 8 y + z (fVDB PR #757: every build path enumerates voxels
    identically) -- as ``(ijk [V,3], offsets [B+1])``."""
    origins, masks, lo = result["origins"], result["masks"], result["leaf_offsets"]
    L = origins.shape[0]
    # bit n of a leaf is bit n & 63 of word n >> 6; the little-endian bytes of
    # the eight words, unpacked low bit first, list the bits in ascending n
    bits = np.unpackbits(np.ascontiguousarray(masks, np.uint64).view(np.uint8).reshape(L, 64), axis=1,
                         bitorder="little")
    leaf, n = np.nonzero(bits)            # row-major: leaf by leaf, ascending n
    local = np.stack([n >> 6, (n >> 3) & 7, n & 7], axis=1)
    ijk = (origins[leaf].astype(np.int64) + local).astype(np.int32).reshape(-1, 3)
    per_leaf = bits.sum(axis=1, dtype=np.int64)
    first = np.concatenate([[0], np.cumsum(per_leaf)])
    offs = first[np.asarray(lo, np.int64)]
    return ijk, offs.astype(np.int64)


def run_masked_refine(result: Dict[str, np.ndarray], voxel_mask: np.ndarray, factor: int,
                      lib=None) -> Dict[str, np.ndarray]:
    """Masked refinement (PR #757 test plan; masked subdivision prunes, then
    refines): the refinement by ``factor`` of the voxels of ``result`` whose
    flag in ``voxel_mask`` (batch voxel order, see batch_voxels) is set."""
    ijk, offs = batch_voxels(result)
    keep = np.asarray(voxel_mask).astype(bool).reshape(-1)
    assert keep.shape[0] == ijk.shape[0]
    counts = [int(keep[offs[g]:offs[g + 1]].sum()) for g in range(len(offs) - 1)]
    new_offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return run_voxels(ijk[keep], new_offs, [("refine", factor)], lib)


def run_kernel_map(in_result: Dict[str, np.ndarray], out_result: Dict[str, np.ndarray], lo, hi,
                   stride: int = 1, transposed: bool = False) -> np.ndarray:
    """Kernel map from its definition: for every voxel p of ``out_result`` (rows
    in batch voxel order) and every offset d of the box [lo, hi] (columns
    x-major), the batch voxel index in ``in_result`` of p + d (stride 1),
    stride * p + d (forward) or (p - d) / stride when divisible (transposed),
    within the same grid; -1 where there is no such voxel."""
    vin, oin = batch_voxels(in_result)
    vout, oout = batch_voxels(out_result)
    offs = [(dx, dy, dz) for dx in range(lo[0], hi[0] + 1) for dy in range(lo[1], hi[1] + 1)
            for dz in range(lo[2], hi[2] + 1)]
    res = np.full((len(vout), len(offs)), -1, np.int32)
    for g in range(len(oin) - 1):
        where = {tuple(int(c) for c in vin[i]): i for i in range(oin[g], oin[g + 1])}
        for j in range(oout[g], oout[g + 1]):
            p = [int(c) for c in vout[j]]
            for k, d in enumerate(offs):
                if transposed:
                    t = [p[a] - d[a] for a in range(3)]
                    if any(x % stride for x in t):
                        continue
                    q = tuple(x // stride for x in t)
                else:
                    q = tuple(stride * p[a] + d[a] for a in range(3))
                i = where.get(q)
                if i is not None:
                    res[j, k] = i
    return res


def member(result: Dict[str, np.ndarray], g: int) -> Dict[str, np.ndarray]:
    """The arrays of grid ``g`` alone, as if it had been run as a batch of one."""
    lo, hi = int(result["leaf_offsets"][g]), int(result["leaf_offsets"][g + 1])
    nlo, nhi = int(result["lower_offsets"][g]), int(result["lower_offsets"][g + 1])
    ulo, uhi = int(result["upper_offsets"][g]), int(result["upper_offsets"][g + 1])
    out = {k: result[k][lo:hi] for k in ("origins", "masks", "voxel_offset", "word_prefix",
                                         "leaf_bbox", "leaf_parent")}
    out["leaf_grid"] = result["leaf_grid"][lo:hi] - g
    out["lower_origins"] = result["lower_origins"][nlo:nhi]
    out["lower_parent"] = result["lower_parent"][nlo:nhi]
    out["upper_origins"] = result["upper_origins"][ulo:uhi]
    for k in ("voxel_counts", "grid_bbox", "node_counts"):
        out[k] = result[k][g:g + 1]
    out["leaf_offsets"] = np.array([0, hi - lo], np.int64)
    out["lower_offsets"] = np.array([0, nhi - nlo], np.int64)
    out["upper_offsets"] = np.array([0, uhi - ulo], np.int64)
    return out
