"""Host-side check of the compressed sort key (no GPU): builds
tests/cpp/key_layout_check.cpp against the library's own headers with g++ and
runs it.  Canonical order per fVDB PR #757, Summary item 1 (sort bullet)."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_key_layout_orders_decodes_and_identifies_nodes(tmp_path):
    exe = tmp_path / "key_layout_check"
    cuda_inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", cuda_inc,
                    "-I", os.path.join(ROOT, "sparse_voxel_grid_leaf_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "cpp", "key_layout_check.cpp"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK")
    assert int(r.stdout.split()[1]) > 1000


def test_member_carve_holds_every_member(tmp_path):
    """The member launch's per-member shares of a chain's arrays, checked on
    the host against the library's own header: large enough, disjoint, in
    order, within the allocation."""
    exe = tmp_path / "member_carve_check"
    cuda_inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", cuda_inc,
                    "-I", os.path.join(ROOT, "sparse_voxel_grid_leaf_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "cpp", "member_carve_check.cpp"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK")
    assert int(r.stdout.split()[1]) > 100000
