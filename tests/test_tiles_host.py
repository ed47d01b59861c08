"""The decode kernels' tiling, run on the host over whole grids (CPU only).

tests/tiles_check.cu includes csrc/decode_tiles.cuh -- the same functions the
two tcgen05 decode kernels call to cut a CTA's outputs into pieces, slots and
TMA boxes -- and checks, for the launch configurations of the 70B decode
shapes and of ragged test shapes, that the ranges partition the outputs, that
pieces respect shard and gate/up-group boundaries, that boxes stay inside the
stage the launcher sized, and that row-side ranks partition the k-blocks
(inside one shard each where the FP8 kernels need it).  It is compiled with
nvcc as host code; nothing runs on a GPU.
"""
import os
import shutil
import subprocess
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_decode_tiling_invariants():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    assert os.path.exists(nvcc), "nvcc is required (it also builds the library)"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "tiles_check")
        subprocess.run([nvcc, "-std=c++17", "-x", "cu",
                        "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(ROOT, "tensor_column_linear_gelu_b300", "csrc"),
                        os.path.join(ROOT, "tests", "tiles_check.cu"), "-o", exe],
                       check=True, capture_output=True, text=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
