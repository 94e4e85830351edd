"""The TA_DEBUG build on the GPU: with every page-table lookup, TMA pool row and output row
checked on the device, forward and backward still match the fp64 oracle element by element and
no check fires on valid plans (tree_attn_check would report TA_ERR_DEVICE_BOUNDS).  The library
is chosen when the binding is imported, so the comparison runs in a child process with
TREEATTN_DEBUG=1 (tests/debug_child.py)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_matches_oracle_without_bounds_flags():
    env = dict(os.environ, TREEATTN_DEBUG="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_child.py")], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("no bounds flag") == 7, r.stdout
