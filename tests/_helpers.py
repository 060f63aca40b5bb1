"""Test helpers written independently of both the oracle and the CUDA path.

They restate the pages' definitions directly on python sets of voxel tuples,
so that the oracle's grouping, bit layout and ordering code can be checked
against something other than itself.
"""
import os
from typing import Dict, List, Sequence, Set, Tuple

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

Vox = Tuple[int, int, int]


def read_sections(name: str) -> Dict[str, List[List[str]]]:
    out: Dict[str, List[List[str]]] = {}
    cur = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("[") and line.endswith("]"):
                cur = line[1:-1]
                out[cur] = []
                continue
            out[cur].append(line.split())
    return out


def leaves_to_voxels(origins: np.ndarray, masks: np.ndarray) -> Set[Vox]:
    """Voxel set of a leaf list; bit b of word w is local (w, b // 8, b % 8)."""
    s: Set[Vox] = set()
    for o, m in zip(origins.tolist(), masks.tolist()):
        for w in range(8):
            word = int(m[w])
            for b in range(64):
                if (word >> b) & 1:
                    s.add((o[0] + w, o[1] + b // 8, o[2] + b % 8))
    return s


def grid_voxels(res: Dict[str, np.ndarray], g: int) -> Set[Vox]:
    lo, hi = int(res["leaf_offsets"][g]), int(res["leaf_offsets"][g + 1])
    return leaves_to_voxels(res["origins"][lo:hi], res["masks"][lo:hi])


def jagged_sets(ijk: np.ndarray, offsets: np.ndarray) -> List[Set[Vox]]:
    return [set(map(tuple, ijk[offsets[g]:offsets[g + 1]].tolist())) for g in range(len(offsets) - 1)]


def pack_sets(sets: Sequence[Set[Vox]]):
    """python voxel sets -> (ijk int32 [N,3], offsets int64 [B+1])."""
    offsets = np.zeros(len(sets) + 1, np.int64)
    rows = []
    for g, s in enumerate(sets):
        rows.extend(sorted(s))
        offsets[g + 1] = len(rows)
    ijk = np.array(rows, np.int32).reshape(-1, 3)
    return ijk, offsets


def brute_refine(s: Set[Vox], f: int) -> Set[Vox]:
    return {(f * x + a, f * y + b, f * z + c) for (x, y, z) in s
            for a in range(f) for b in range(f) for c in range(f)}


def brute_coarsen(s: Set[Vox], f: int) -> Set[Vox]:
    # python's // is floor division
    return {(x // f, y // f, z // f) for (x, y, z) in s}


def brute_dilate(s: Set[Vox], lo: Sequence[int], hi: Sequence[int]) -> Set[Vox]:
    return {(x + a, y + b, z + c) for (x, y, z) in s
            for a in range(lo[0], hi[0] + 1) for b in range(lo[1], hi[1] + 1)
            for c in range(lo[2], hi[2] + 1)}


def popcount(w: int) -> int:
    return bin(int(w)).count("1")


def canon_tuple(o) -> Tuple[int, ...]:
    """Canonical sort tuple of an origin: signed root tile floor(v/4096), then
    the x-major upper child offset floor(v/128) mod 32, then the x-major lower
    child offset floor(v/8) mod 16 (fVDB PR #757, Summary item 1, sort bullet)."""
    o = [int(v) for v in o]
    return tuple(v // 4096 for v in o) + tuple((v // 128) % 32 for v in o) + tuple((v // 8) % 16 for v in o)


def check_derived(res: Dict[str, np.ndarray]):
    """Per-leaf/per-grid arrays against a direct recomputation from the masks."""
    B = len(res["leaf_offsets"]) - 1
    L = res["origins"].shape[0]
    assert res["leaf_offsets"][0] == 0 and res["leaf_offsets"][-1] == L
    for g in range(B):
        lo, hi = int(res["leaf_offsets"][g]), int(res["leaf_offsets"][g + 1])
        run = 0
        gmin = [2 ** 31 - 1] * 3
        gmax = [-2 ** 31] * 3
        for i in range(lo, hi):
            assert res["leaf_grid"][i] == g
            pcs = [popcount(w) for w in res["masks"][i]]
            assert sum(pcs) > 0, "empty leaf emitted"
            assert res["voxel_offset"][i] == run
            run += sum(pcs)
            wp = int(res["word_prefix"][i])
            for k in range(1, 8):
                assert (wp >> (9 * (k - 1))) & 511 == sum(pcs[:k])
            assert wp >> 63 == 0
            vox = leaves_to_voxels(res["origins"][i:i + 1], res["masks"][i:i + 1])
            mn = [min(v[a] for v in vox) for a in range(3)]
            mx = [max(v[a] for v in vox) for a in range(3)]
            assert list(res["leaf_bbox"][i]) == mn + mx
            gmin = [min(a, b) for a, b in zip(gmin, mn)]
            gmax = [max(a, b) for a, b in zip(gmax, mx)]
            assert all(int(o) % 8 == 0 for o in res["origins"][i])
        assert res["voxel_counts"][g] == run
        assert list(res["grid_bbox"][g]) == gmin + gmax
        # nodes: distinct 128^3 and 4096^3 blocks holding a leaf
        origins = res["origins"][lo:hi].astype(np.int64)
        lowers = {tuple((o // 128 * 128).tolist()) for o in origins}
        uppers = {tuple((o // 4096 * 4096).tolist()) for o in origins}
        assert list(res["node_counts"][g]) == [len(uppers), len(lowers), hi - lo]
        nlo = int(res["lower_offsets"][g])
        ulo = int(res["upper_offsets"][g])
        assert res["lower_offsets"][g + 1] - nlo == len(lowers)
        assert res["upper_offsets"][g + 1] - ulo == len(uppers)
        for i in range(lo, hi):
            p = int(res["leaf_parent"][i])
            assert 0 <= p < len(lowers)
            assert tuple(res["lower_origins"][nlo + p]) == tuple((origins[i - lo] // 128 * 128).tolist())
        # every node list strictly increasing in canonical order
        for name, first, n in (("origins", lo, hi - lo), ("lower_origins", nlo, len(lowers)),
                               ("upper_origins", ulo, len(uppers))):
            keys = [canon_tuple(o) for o in res[name][first:first + n]]
            assert all(a < b for a, b in zip(keys, keys[1:])), name + " not in canonical order"
        for j in range(len(lowers)):
            p = int(res["lower_parent"][nlo + j])
            assert 0 <= p < len(uppers)
            lo_o = res["lower_origins"][nlo + j].astype(np.int64)
            assert tuple(res["upper_origins"][ulo + p]) == tuple((lo_o // 4096 * 4096).tolist())
