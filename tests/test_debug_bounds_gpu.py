"""The debug build (SS_DEBUG_BOUNDS, libssscan_debug.so): every kernel family checks the index
ranges it derives against the sizes in ss_dims and records a failed check in the device status
word instead of trapping.  The GPU test runs tests/debug_bounds_run.py in a child process that
loads the debug build (SS_LIBRARY=debug): small problems through every entry point, against the
oracle, then a clean status word, then the self-test check that records SS_EBOUNDS.  The CPU
tests check that the debug build exports the same entry points and says which build it is."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

import selective_state_space_117_b300 as ss

HERE = os.path.dirname(os.path.abspath(__file__))
DEBUG_LIB = os.path.join(os.path.dirname(ss.library_path()), "libssscan_debug.so")
NORMAL_LIB = os.path.join(os.path.dirname(ss.library_path()), "libssscan.so")

needs_debug = pytest.mark.skipif(not os.path.exists(DEBUG_LIB), reason="debug build not built (build() makes it)")


def _exports(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    return set(re.findall(r"\bT (ss_\w+)", out))


@needs_debug
def test_debug_build_exports_the_same_entry_points():
    assert _exports(DEBUG_LIB) == _exports(NORMAL_LIB)
    assert ctypes.CDLL(DEBUG_LIB).ss_debug_bounds_build() == 1
    assert ctypes.CDLL(NORMAL_LIB).ss_debug_bounds_build() == 0


@needs_debug
@pytest.mark.gpu
def test_debug_build_every_kernel_in_bounds():
    env = dict(os.environ, SS_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_run.py")], capture_output=True, text=True,
                       env=env, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "ok selftest records SS_EBOUNDS" in r.stdout
