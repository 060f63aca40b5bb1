"""The benchmark's byte model on CPU: the step's pass list follows the passes
the library ran (k3s2 fused into one pass for small inputs, two passes
above 32,768 leaves), and the §8(d) bytes of a pass are
76 L_in + 116 L_out + 24 S P + 100 B."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class FakeBatch:
    """The batch properties the pass list reads."""

    def __init__(self, leaves, slots, sources, key_bits=40, grids=4):
        self.num_leaves = leaves
        self.build_slots = slots
        self.build_source_leaves = sources
        self.build_key_bits = key_bits
        self.build_digit_passes = 0
        self.build_member_ctas = 0
        self.num_lowers = leaves // 10
        self.num_uppers = 2
        self.num_grids = grids


def step_outputs(k3s2_sources):
    b0 = FakeBatch(100, 1000, 1000)
    return {"from_ijk": b0, "refine2": FakeBatch(450, 450, 100), "coarsen2": FakeBatch(20, 100, 100),
            "dilate_k3s1": FakeBatch(130, 900, 100), "pad_neg": FakeBatch(120, 400, 100),
            "pad_pos": FakeBatch(120, 400, 100), "k3s2": FakeBatch(600, 1500, k3s2_sources),
            "coarsen4": FakeBatch(5, 100, 100)}


def test_fused_k3s2_is_one_pass():
    ps = bench.pass_stats(step_outputs(k3s2_sources=100))
    assert [p["kind"] for p in ps] == ["ijk", "refine", "coarsen", "dilate", "dilate", "dilate",
                                       "refine_dilate", "coarsen"]
    assert not any(p.get("inter") for p in ps)


def test_two_pass_k3s2_counts_its_refine_pass():
    ps = bench.pass_stats(step_outputs(k3s2_sources=-1))
    assert [p["kind"] for p in ps] == ["ijk", "refine", "coarsen", "dilate", "dilate", "dilate",
                                       "refine", "dilate", "coarsen"]
    first, second = ps[6], ps[7]
    # the first pass is the refine x2 call's: same input, same op
    assert first["inter"] and (first["L_in"], first["S"], first["L_out"]) == (100, 450, 450)
    # the pad pass reads the refined leaves and writes the k3s2 output
    assert (second["L_in"], second["S"], second["L_out"]) == (450, 1500, 600)
    # the intermediate pass hands its leaves on: no writer bytes for it
    by_fused = bench.kernel_bytes(bench.pass_stats(step_outputs(100)))
    by_split = bench.kernel_bytes(ps)
    assert by_split["chain"] > by_fused["chain"]


def test_pass_bytes_formula():
    p = {"kind": "refine", "L_in": 10, "L_out": 80, "S": 80, "P": 3, "B": 2}
    assert bench.pass_bytes(p) == 76 * 10 + 116 * 80 + 24 * 80 * 3 + 100 * 2
    p = {"kind": "ijk", "L_in": 1000, "L_out": 40, "S": 1000, "P": 2, "B": 2}
    assert bench.pass_bytes(p) == 12 * 1000 + 116 * 40 + 24 * 1000 * 2 + 100 * 2
    assert bench.model_digit_passes(FakeBatch(1, 1, 1, key_bits=41)) == 6
