"""Child process of tests/test_gpu_debug.py: loads the TA_DEBUG library (TREEATTN_DEBUG=1 must be
set before the binding is imported), runs forward and backward on the given episodes and
compares every output element with the fp64 oracle; tree_attn_check inside the runs fails on any
device-side bounds flag.  Prints one line per episode; exits non-zero on a mismatch."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

assert os.environ.get("TREEATTN_DEBUG") == "1"

from dag_packed_paged_gb300 import _native, build  # noqa: E402

build.build(debug=True)
assert _native.LIB == build.LIB_DEBUG

import oracle  # noqa: E402
from dag_packed_paged_gb300 import workloads as W  # noqa: E402
from gpu_helpers import Run, assert_close  # noqa: E402


def episodes():
    yield "tiny", W.tiny()
    yield "balanced/16", W.scaled(1, 16)
    yield "mount_heavy/64", W.scaled(4, 64)
    # 16-row pages (a packed slot is two pages) with D = 64 (the single-SM forward), and 128-row
    # pages with D = 128 (the CTA-pair forward)
    yield "random D=64 P=16", W.random_small(2001, max_branches=8, max_len=700, heads=(16, 2), head_dim=64,
                                             page_size=16, n_mounts=2)
    yield "random D=128 P=128", W.random_small(2002, max_branches=8, max_len=700, heads=(8, 1), head_dim=128,
                                               page_size=128, n_mounts=3)
    # split-KV forward: work items over parts of blocks, partial slots and the combine (checked
    # slot indexes), on both forwards
    yield "split D=128 cap 2", W.random_small(2003, max_branches=8, max_len=900, heads=(8, 2), head_dim=128,
                                              page_size=64, n_mounts=3)
    yield "split D=64 cap 2", W.random_small(2004, max_branches=8, max_len=900, heads=(8, 2), head_dim=64,
                                             page_size=32, n_mounts=3)


for name, ep in episodes():
    run = Run(ep, fwd_split_tiles=2) if name.startswith("split") else Run(ep)
    o, lse = run.fwd()                 # tree_attn_check raises on a bounds flag
    dq, dk, dv = run.bwd()
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    assert_close("O", o, ref.o)
    assert_close("dQ", dq, ref.dq)
    assert_close("dK", dk, ref.dk)
    assert_close("dV", dv, ref.dv)
    print(f"{name}: debug build matches the oracle, no bounds flag", flush=True)
