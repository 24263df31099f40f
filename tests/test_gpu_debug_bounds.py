"""GPU tests of the debug-bounds library (libmoe_route_debug.so: the same
sources compiled with MOE_DEBUG_BOUNDS, the kernels' internal index, size and
alignment checks compiled in).

1. Its self-test kernel runs one check that is false by construction and
   guards no access: the device error word must then read MOE_DEVERR_BOUNDS,
   and nothing else.
2. The parity suites of the bulk-store expand kernels, the chained and decode
   paths, the canaries and the shape fuzz run again in a child process with
   MOE_DEBUG_BOUNDS=1, so every kernel they launch carries its checks: every
   result must still match the oracle and no check may fail (each module
   asserts a clean device error word at its end, and every test that expects
   a data error checks the exact bits).
"""
import os
import subprocess
import sys

import pytest
import torch

from moe_routing_precision_gb300 import _build, ops

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def D():
    torch.cuda.set_device(0)
    return ops.load_library(_build.build(debug_bounds=True))


def _status(L):
    import ctypes
    bits = ctypes.c_uint32(0)
    rc = L.moe_get_device_status(None, ctypes.byref(bits))
    return rc, bits.value


def test_selftest_sets_only_the_bounds_bit(D):
    assert D.moe_debug_bounds_enabled() == 1
    assert _status(D) == (ops.MOE_OK, 0)
    assert D.moe_debug_bounds_selftest(None) == ops.MOE_OK
    assert _status(D) == (ops.MOE_ERR_DEVICE, ops.MOE_DEVERR_BOUNDS)
    assert _status(D) == (ops.MOE_OK, 0)   # read and cleared


def test_parity_suites_pass_with_the_checks_compiled_in(D):
    env = dict(os.environ, MOE_DEBUG_BOUNDS="1")
    probe = subprocess.run(
        [sys.executable, "-c",
         "from moe_routing_precision_gb300 import ops; "
         "print(ops.lib().moe_debug_bounds_enabled())"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip() == "1", probe.stderr
    suites = ["tests/test_gpu_parity.py", "tests/test_gpu_cast_opts.py", "tests/test_gpu_fp4.py",
              "tests/test_gpu_chain.py", "tests/test_gpu_decode.py", "tests/test_gpu_canary.py",
              "tests/test_gpu_fuzz.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu",
                        "-p", "no:cacheprovider", *suites],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
