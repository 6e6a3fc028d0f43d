"""The debug build as a stand-in for a memory sanitizer.

libtps_debug.so is the library compiled with TPS_DEBUG=1: every epilogue
store of the GEMM kernels (direct stores, TMA-store boxes, the CE tile
statistics) and every store of the CE core kernels checks that it lies
inside its output; a store outside is skipped and reported as
TPS_ERR_BOUNDS by tps_last_device_error.  This test runs the guard-band
file -- every entry point at ragged shapes, each call followed by a check
of the device error word, canaries and bit-identity -- against the debug
build in a child process (the binding loads the library named by
TPS_LIBRARY)."""
import os
import subprocess
import sys

import pytest

from backward_tcgen05_tma_gemms_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.gpu
def test_guard_cases_under_the_bounds_checked_build():
    so = build.build(debug=True)
    env = dict(os.environ, TPS_LIBRARY=so)
    check = ("from backward_tcgen05_tma_gemms_gb300 import api; "
             "assert api.library().tps_build_flags() & api.BUILD_DEBUG, 'not the debug build'")
    r = subprocess.run([sys.executable, "-c", check], env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_gpu_guard.py"), "-q", "-m", "gpu",
                        "-p", "no:cacheprovider"], env=env, cwd=ROOT, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "failed" not in r.stdout, r.stdout[-2000:]
