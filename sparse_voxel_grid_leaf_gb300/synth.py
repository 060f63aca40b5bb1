"""Seeded synthetic voxel batches shaped like the workloads of fVDB PR #757.

The PR ("Batched leaf-mask topology construction for generated conv grids",
Measurements section) times its batched builder on synthetic shell batches of
about 7.8k voxels per member at resolution 64.  This module produces such
batches (and the other workload shapes used for testing) as a jagged list of
int32 voxel coordinates: ``ijk`` of shape ``[N, 3]`` plus ``offsets`` of shape
``[B + 1]`` (int64, ``offsets[0] == 0``, ``offsets[B] == N``).

It holds none of the topology method's arithmetic: it only draws coordinates.
Both the CUDA path and the CPU oracle consume its output.

Determinism: every random number comes from splitmix64 (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", 2014) evaluated in numpy
uint64 arithmetic, and uniforms are ``(x >> 11) * 2**-53``.  Floating-point
steps are plain IEEE float64 operations in a fixed order, so the same seed
gives the same voxels on x86-64 and aarch64.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


class SplitMix64:
    """Sequential splitmix64 stream: state += golden; output = mix(state)."""

    def __init__(self, seed: int):
        self.state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)

    def next_u64(self, n: int = 1) -> np.ndarray:
        k = np.arange(1, n + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            states = self.state + k * _GOLDEN
            self.state = self.state + np.uint64(n) * _GOLDEN
        return _mix(states)

    def uniform(self, n: int = 1) -> np.ndarray:
        return (self.next_u64(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def member_seed(base_seed: int, member: int) -> int:
    return base_seed * 1000 + member


def shell_voxels(rng: SplitMix64, res: int, r_lo: float, r_hi: float,
                 scale: float = 1.0) -> np.ndarray:
    """One-voxel-thick ellipsoid shell.

    Semi-axes ``r ~ U[r_lo, r_hi] * res`` (times ``scale``), drawn first, then
    centre ``c ~ U[0.45, 0.55] * res``, per axis.  (In this order the B=16
    shells at res 64 average 7,861 voxels per member and the B=48 batch has
    378,382, matching the "~7.8k voxels/member" and "~375k" the workloads are
    sized by.)  With ``p = ijk + 0.5`` and
    ``q = |(p - c) / r|``, the radial implicit value is
    ``f = |p - c| * (q - 1) / q`` (signed distance to the surface along the
    ray from the centre); a voxel is active iff ``|f| <= 0.5``.
    """
    r = (r_lo + (r_hi - r_lo) * rng.uniform(3)) * res * scale
    c = (0.45 + 0.10 * rng.uniform(3)) * res
    half = float(np.max(r)) + 2.0
    lo = np.floor(c - half).astype(np.int64)
    hi = np.ceil(c + half).astype(np.int64)
    out = []
    xs = np.arange(lo[0], hi[0] + 1, dtype=np.int64)
    ys = np.arange(lo[1], hi[1] + 1, dtype=np.int64)
    zs = np.arange(lo[2], hi[2] + 1, dtype=np.int64)
    Y, Z = np.meshgrid(ys, zs, indexing="ij")
    py = (Y.astype(np.float64) + 0.5 - c[1])
    pz = (Z.astype(np.float64) + 0.5 - c[2])
    for x in xs:  # one x-slab at a time keeps memory small at res 512
        px = float(x) + 0.5 - c[0]
        d2 = px * px + py * py + pz * pz
        qx, qy, qz = px / r[0], py / r[1], pz / r[2]
        q = np.sqrt(qx * qx + qy * qy + qz * qz)
        dist = np.sqrt(d2)
        with np.errstate(divide="ignore", invalid="ignore"):
            f = dist * (q - 1.0) / q
        act = np.abs(f) <= 0.5
        act &= q > 0.0
        if act.any():
            yy, zz = Y[act], Z[act]
            out.append(np.stack([np.full(yy.shape, x, np.int64), yy, zz], axis=1))
    if not out:
        return np.zeros((0, 3), np.int32)
    return np.concatenate(out).astype(np.int32)


def blob_voxels(rng: SplitMix64, res: int, p: float = 0.02,
                side_lo: int = 64, side_hi: int = 128) -> np.ndarray:
    """Bernoulli(p) voxels inside an axis-aligned box with sides U{side_lo..side_hi}."""
    c = (0.45 + 0.10 * rng.uniform(3)) * res
    sides = side_lo + (rng.next_u64(3) % np.uint64(side_hi - side_lo + 1)).astype(np.int64)
    lo = np.floor(c).astype(np.int64) - sides // 2
    n = int(np.prod(sides))
    keep = rng.uniform(n) < p
    idx = np.nonzero(keep)[0].astype(np.int64)
    sx, sy, sz = (int(s) for s in sides)
    x = idx // (sy * sz)
    y = (idx // sz) % sy
    z = idx % sz
    return (np.stack([x, y, z], axis=1) + lo[None, :]).astype(np.int32)


def _pack(members: Sequence[np.ndarray]) -> Tuple[np.ndarray, np.ndarray]:
    counts = np.array([m.shape[0] for m in members], dtype=np.int64)
    offsets = np.zeros(len(members) + 1, dtype=np.int64)
    np.cumsum(counts, out=offsets[1:])
    if len(members) and offsets[-1] > 0:
        ijk = np.ascontiguousarray(np.concatenate(members).astype(np.int32))
    else:
        ijk = np.zeros((0, 3), np.int32)
    return ijk, offsets


def shells(B: int, res: int, r_lo: float, r_hi: float, seed: int = 0,
           empty: Sequence[int] = (), size_range_log2: Optional[Tuple[float, float]] = None
           ) -> Tuple[np.ndarray, np.ndarray]:
    """A batch of B shells; members listed in ``empty`` have no voxels.

    With ``size_range_log2 = (a, b)`` each member's semi-axes are scaled by
    ``sqrt(2**U[a, b])`` so that its voxel count (proportional to the shell's
    area) varies by the factor ``2**U[a, b]``.
    """
    members: List[np.ndarray] = []
    for m in range(B):
        rng = SplitMix64(member_seed(seed, m))
        scale = 1.0
        if size_range_log2 is not None:
            a, b = size_range_log2
            # drawn first so that it does not perturb the shell's own draws
            s = 2.0 ** (a + (b - a) * float(rng.uniform(1)[0]))
            scale = float(np.sqrt(s))
        v = shell_voxels(rng, res, r_lo, r_hi, scale)
        if m in empty:
            v = np.zeros((0, 3), np.int32)
        members.append(v)
    return _pack(members)


def stress_mix(B: int = 64, res: int = 512, seed: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Mixed shells (even members) and Bernoulli(0.02) blobs (odd members).

    Each member is moved so that it straddles a root-tile boundary (a multiple
    of 4096 per axis): its voxels are re-centred on ``T = 4096 * (s * k)`` per
    axis, with the sign pattern ``s`` cycling through all eight octants and
    ``k`` in {1, 2}.
    """
    members: List[np.ndarray] = []
    for m in range(B):
        rng = SplitMix64(member_seed(seed, m))
        if m % 2 == 0:
            v = shell_voxels(rng, res, 0.05, 0.12)
        else:
            v = blob_voxels(rng, res)
        octant = (m // 2) % 8
        k = 1 + (m // 16) % 2
        sgn = np.array([-1 if (octant >> a) & 1 else 1 for a in range(3)], np.int64)
        T = 4096 * k * sgn
        centre = res // 2
        v = (v.astype(np.int64) - centre + T[None, :]).astype(np.int32)
        members.append(v)
    return _pack(members)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    res: int
    description: str


WORKLOADS = {
    "pr1_b2_res32": Workload("pr1_b2_res32", 2, 32,
                             "B=2 shells, res 32, semi-axes U[0.30,0.45]*res, seed 0"),
    "shells_b16_res64": Workload("shells_b16_res64", 16, 64,
                                 "B=16 shells, res 64, semi-axes U[0.30,0.48]*res, seed 0"),
    "shells_b48_res64": Workload("shells_b48_res64", 48, 64,
                                 "B=48 shells, res 64, semi-axes U[0.30,0.48]*res, seed 0"),
    "pyramid_b48_res64": Workload("pyramid_b48_res64", 48, 64,
                                  "B=48 shells, res 64, sizes 0.25x-4x, members 0/24/47 empty"),
    "stress_b64_res512": Workload("stress_b64_res512", 64, 512,
                                  "B=64 res 512: shells + Bernoulli(0.02) blobs across +-4096 tiles"),
}


def make(name: str, seed: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Voxel batch of a named workload: ``(ijk int32 [N,3], offsets int64 [B+1])``."""
    if name == "pr1_b2_res32":
        return shells(2, 32, 0.30, 0.45, seed)
    if name == "shells_b16_res64":
        return shells(16, 64, 0.30, 0.48, seed)
    if name == "shells_b48_res64":
        return shells(48, 64, 0.30, 0.48, seed)
    if name == "pyramid_b48_res64":
        return shells(48, 64, 0.30, 0.48, seed, empty=(0, 24, 47), size_range_log2=(-2.0, 2.0))
    if name == "stress_b64_res512":
        return stress_mix(64, 512, seed)
    raise KeyError(name)


def random_voxels(B: int, n_per: int, span: int, seed: int, origin: Sequence[int] = (0, 0, 0),
                  empty: Sequence[int] = ()) -> Tuple[np.ndarray, np.ndarray]:
    """Uniform random voxels (with duplicates) in ``origin + [0, span)^3`` per member."""
    members = []
    for m in range(B):
        rng = SplitMix64(member_seed(seed, m) + 7)
        n = 0 if m in empty else n_per
        v = (rng.next_u64(3 * n) % np.uint64(span)).astype(np.int64).reshape(n, 3)
        members.append((v + np.asarray(origin, np.int64)[None, :]).astype(np.int32))
    return _pack(members)
