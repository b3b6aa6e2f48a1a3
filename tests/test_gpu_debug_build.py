"""The debug build (-DMOE_DEBUG: every caller-given index, segment bound and
tile start checked in the kernels, a failure recorded as MOE_ERR_ARG with
its site instead of an access outside a buffer) is built and the layer's
oracle tests and the debug checks' own tests run against it in a child
process, with the guard regions of the test helpers around every buffer.
Together they stand in for compute-sanitizer's memcheck, which this
machine pool does not offer."""
import os
import subprocess
import sys

import pytest

from combine_fp32_softmax_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_layer_tests_pass_under_the_debug_build():
    build.build(debug=True)
    env = dict(os.environ, MOE_GB300_DEBUG_LIB="1")
    env.pop("MOE_MARGINS_OUT", None)
    cmd = [sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_debug_checks.py",
           "tests/test_gpu_layer.py::test_layer_matches_oracle",
           "tests/test_gpu_layer.py::test_megakernel_bitwise_equals_kernel_chain",
           "tests/test_gpu_layer.py::test_bwd_megakernel_bitwise_equals_kernel_chain",
           "tests/test_gpu_layer.py::test_cta_pair_tiles_equal_single_cta_tiles_bitwise",
           "tests/test_gpu_layer.py::test_fused_routing_tables_equal_three_kernels_and_oracle",
           "tests/test_gpu_kernels.py"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    summary = [ln for ln in r.stdout.splitlines() if ln.strip()][-1]
    assert " passed" in summary and "skipped" not in summary, tail
