"""dK/dV parity where a key tile has many readers: the path full-size runs take.

The dK/dV kernel walks a key tile's readers in chunks; the loader and the elementwise warps
refill their copies of the reader list every 32 entries, and the Q/dO rings wrap around many
times on a long chunk.  These tests compare every element of dQ, dK and dV with the fp64 oracle on
episodes whose chunks are long -- by shape (the mount-heavy workload at 1/8 size, a wide fan),
by forcing unsplit chunks through ta_config.dkdv_chunk_entries, and at full size on the rows of
one mount-heavy DAG that gather from the most readers and of the balanced tree's root and first
depth-1 edge (stored oracle values, written by tests/golden/make_mount_heavy_dkdv.py and
make_balanced_tree_dkdv.py).  References: Octopus Section 3.4 (differentiable mount
edges) and HARTS Section 3.4 (the gather backward accumulates every consumer into the unique
compact row)."""
import hashlib
import os

import numpy as np
import pytest

import dag_packed_paged_gb300 as ta
import oracle
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "mount_heavy_dag0_dkdv.npz")
GOLDEN_BT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "balanced_tree_dkdv.npz")


def _longest_chunk(plan):
    ch = ta.tree_attn_plan_export(plan)["chunks"]
    return int((ch[:, 2] - ch[:, 1]).max())


_REF = {}


def _oracle(ep, t):
    key = (ep.name, ep.seed)
    if key not in _REF:
        _REF[key] = oracle.run(ep.branches, ep.mounts, t.q, t.k, t.v, t.do, ep.softmax_scale)
    return _REF[key]


@pytest.mark.parametrize("chunk", [0, 1 << 20], ids=["default_chunks", "unsplit_tiles"])
def test_mount_heavy_eighth_whole_strip(chunk):
    """The mount-heavy shape at 1/8 size (32,768 rows): with the default chunking 160 chunks
    hold more than 32 entries; unsplit, the longest holds 164.  Every row of O, dQ, dK, dV."""
    ep = W.scaled(4, 8)
    run = Run(ep, dkdv_chunk_entries=chunk)
    longest = _longest_chunk(run.plan)
    assert longest > 32 if chunk == 0 else longest >= 160
    ref = _oracle(ep, run.t)
    o, _ = run.fwd()
    dq, dk, dv = run.bwd()
    assert_close("O", o, ref.o)
    assert_close("dQ", dq, ref.dq)
    assert_close("dK", dk, ref.dk)
    assert_close("dV", dv, ref.dv)


@pytest.mark.parametrize("chunk", [0, 1 << 20, 7, 1], ids=["default", "unsplit", "7", "1"])
@pytest.mark.parametrize("dist", ["config", "realistic"])
def test_wide_fan_long_reader_lists(chunk, dist):
    """A 128-row root read by 256 one-block children (half of them mounting a sibling's tail):
    unsplit, the root tile's chunk holds every one of the 322 query blocks; split into chunks of
    7 or 1 entries, the fixed-order reduction sums up to 322 partial slots per tile."""
    ep = W.wide_fan()
    run = Run(ep, dist=dist, dkdv_chunk_entries=chunk)
    if chunk == 1 << 20:
        assert _longest_chunk(run.plan) >= 300
        assert ta.tree_attn_plan_stats(run.plan)["n_partial_slots"] == 0
    ref = _oracle(ep, run.t) if dist == "config" else oracle.run(
        ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    o, _ = run.fwd()
    dq, dk, dv = run.bwd()
    assert_close("O", o, ref.o)
    assert_close("dQ", dq, ref.dq)
    assert_close("dK", dk, ref.dk)
    assert_close("dV", dv, ref.dv)


def test_mount_heavy_full_size_shared_rows():
    """Full-size mount-heavy in the benchmark's launch configuration: dK and dV of 32 rows of
    the first DAG's mounted producer span and 32 rows of its root -- rows that gather from 32
    mount readers plus the producer's descendants, and from all 65,536 rows of the DAG -- against
    the oracle over every reader of that DAG."""
    if not os.path.exists(GOLDEN):
        pytest.fail(f"{GOLDEN} is missing; run tests/golden/make_mount_heavy_dkdv.py")
    g = np.load(GOLDEN)
    ep = W.config(4)
    run = Run(ep)
    dag_rows = int(g["dag_rows"])
    sel = ep.branches["row_start"] < dag_rows
    nb = int(sel.sum())
    mt = ep.mounts[(ep.mounts["reader"] < nb) & (ep.mounts["source"] < nb)]
    h = hashlib.sha256()
    for a in (ep.branches[sel], mt, run.t.q[:dag_rows], run.t.k[:dag_rows], run.t.v[:dag_rows],
              run.t.do[:dag_rows]):
        h.update(np.ascontiguousarray(a).tobytes())
    assert h.hexdigest() == str(g["input_sha256"]), "the stored oracle values are for other inputs"
    assert _longest_chunk(run.plan) >= 1000          # the root tile's readers in one chunk
    run.fwd()
    dq, dk, dv = run.bwd()
    rows = g["rows"]
    lo, hi = (int(x) for x in g["span"])
    span = (rows >= lo) & (rows < hi)
    assert span.sum() == 32 and (rows < 8192).sum() == 32
    for name, got, want in (("dK", dk, g["dk"]), ("dV", dv, g["dv"])):
        assert_close(name + " span", got[rows[span]], want[span].astype(np.float64))
        assert_close(name + " root", got[rows[~span]], want[~span].astype(np.float64))


def test_balanced_tree_full_size_shared_rows():
    """Full-size balanced tree in the benchmark's launch configuration: dK and dV of 32 rows of
    the 4,096-row root (read by all 45,056 rows) and 32 rows of the first depth-1 edge (read by
    its 10,240-row subtree), against the oracle over the whole tree."""
    if not os.path.exists(GOLDEN_BT):
        pytest.fail(f"{GOLDEN_BT} is missing; run tests/golden/make_balanced_tree_dkdv.py")
    g = np.load(GOLDEN_BT)
    ep = W.config(1)
    run = Run(ep)
    h = hashlib.sha256()
    for a in (ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do):
        h.update(np.ascontiguousarray(a).tobytes())
    assert h.hexdigest() == str(g["input_sha256"]), "the stored oracle values are for other inputs"
    run.fwd()
    dq, dk, dv = run.bwd()
    rows = g["rows"]
    lo, hi = (int(x) for x in g["edge"])
    edge = (rows >= lo) & (rows < hi)
    assert edge.sum() == 32 and (rows < int(ep.branches["length"][0])).sum() == 32
    for name, got, want in (("dK", dk, g["dk"]), ("dV", dv, g["dv"])):
        assert_close(name + " root", got[rows[~edge]], want[~edge].astype(np.float64))
        assert_close(name + " edge", got[rows[edge]], want[edge].astype(np.float64))
