"""The preprocess suites under the checked build (libws_bounds.so, the same
sources compiled with WS_BOUNDS_CHECK).  Its kernels test every index into
the ring kernel's shared stage slots and column-tap table and every source
tap of both preprocess kernels; an index out of range sets device error bit
0x4 and is clamped into its buffer, so nothing traps.  The suites run in a
child process that loads the checked build (WS_BOUNDS_CHECK=1): the odd
shapes (ragged strides, unaligned bases, one-stage rings, rows too long for
a ring), the full-size workloads on both kernels, the typed outputs, and
lanes in every input mode.  Each preprocess test there asserts that the
bounds bit stayed clear, and a lane reports it as WS_ERR_DEVICE."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def checked_env():
    return dict(os.environ, WS_BOUNDS_CHECK="1")


def test_checked_build_is_loaded():
    import __graft_entry__
    __graft_entry__.build()
    code = ("from post_processing_gb300 import binding as B; "
            "assert B.ws_build_features() & B.WS_FEATURE_BOUNDS_CHECK; "
            "assert B.LIBRARY_PATH.endswith('libws_bounds.so'); print('ok')")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=checked_env(), capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


@pytest.mark.parametrize("target,select", [
    ("tests/test_gpu_preprocess.py", "odd_shapes or extreme or repeat or no_device_error or half_outputs or bgr"),
    ("tests/test_gpu_preprocess.py", "workload_parity"),
    ("tests/test_gpu_lane.py", "lane_parity or mapped_input"),
], ids=["odd-shapes", "workloads", "lanes"])
def test_suite_under_bounds_checks(target, select):
    import __graft_entry__
    __graft_entry__.build()
    cmd = [sys.executable, "-m", "pytest", target, "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider", "-k", select]
    r = subprocess.run(cmd, cwd=ROOT, env=checked_env(), capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
