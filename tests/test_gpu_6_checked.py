"""The checked build (libtpla_checked.so, kernels compiled with TPLA_CHECKED):
every kernel's computed shared-memory, tensor-memory and weight-row indices,
and every output store against the extent of the output it writes, are
checked; a failed check records TP_ERR_DEVICE_CHECK and skips the access (no
assert, no trap).  This runs the small-shape parity suites -- all kernel
families: GEMV, the decode kernel in bf16 and FP8 modes, the FP8 kernel with
the weights in tensor memory, the prefill GEMM, the ring and uneven modes, and
the no-alloc FFN whose h lives in the library's fixed device buffer -- in
a child process that loads the checked library; every test there also asserts
that the device status is clear afterwards, so one failed index check fails
the run.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_1_small.py", "tests/test_gpu_4_modes.py", "tests/test_gpu_5_fp8.py",
          "tests/test_zz_no_alloc.py"]


def test_parity_suites_under_the_checked_build():
    from tensor_column_linear_gelu_b300 import build
    build.build(checked=True)
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-m", "gpu", "-q", "-x",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, capture_output=True, text=True, timeout=1200,
                       env=dict(os.environ, TPLA_CHECKED="1"))
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-25:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
