"""Writes balanced_tree_dkdv.npz: the oracle's dK and dV on key rows of the full-size balanced
tree that gather from the most readers -- rows of the 4,096-row root, which all 45,056 rows of
the tree read, and rows of the first depth-1 edge, which its 10,240-row subtree reads (HARTS
Section 3.4: the gather backward accumulates every consumer into the unique compact row; Octopus
Section 3.3: every node attends to its ancestors).

Only the oracle runs here (fp64 CPU), over every row of the tree.  The file records the seed, a
SHA-256 over the tree's topology and its Q, K, V, dO bits, and the rows; the GPU test
regenerates the inputs, checks the hash, and compares.  It takes about a quarter of an hour on
eight host cores.

    python tests/golden/make_balanced_tree_dkdv.py
"""
import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from dag_packed_paged_gb300 import workloads as W  # noqa: E402

OUT = os.path.join(HERE, "balanced_tree_dkdv.npz")


def inputs_digest(ep, t):
    h = hashlib.sha256()
    for a in (ep.branches, ep.mounts, t.q, t.k, t.v, t.do):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def key_rows(ep):
    """32 rows of the root and 32 of the first depth-1 edge, seeded, ends included."""
    br = ep.branches
    root_len = int(br["length"][0])
    child = int(np.nonzero(br["parent"] == 0)[0][0])
    lo = int(br["row_start"][child])
    hi = lo + int(br["length"][child])
    rng = np.random.default_rng(np.random.SeedSequence([0, 6006]))
    root = np.concatenate([[0, root_len - 1], rng.choice(np.arange(1, root_len - 1), 30, replace=False)])
    edge = np.concatenate([[lo, hi - 1], rng.choice(np.arange(lo + 1, hi - 1), 30, replace=False)])
    return np.sort(np.concatenate([root, edge])).astype(np.int64), (lo, hi)


def main():
    ep = W.config(1)
    t = W.make_tensors(ep)
    digest = inputs_digest(ep, t)
    rows, edge = key_rows(ep)
    t0 = time.time()
    res = oracle.run(ep.branches, ep.mounts, t.q, t.k, t.v, t.do, ep.softmax_scale)
    dt = time.time() - t0
    np.savez_compressed(OUT, rows=rows, edge=np.array(edge), dk=res.dk[rows].astype(np.float32),
                        dv=res.dv[rows].astype(np.float32), seed=np.int64(ep.seed), input_sha256=digest,
                        workload=ep.name)
    print(f"wrote {OUT}: {len(rows)} key rows, oracle {dt:.0f} s on {res.threads} threads")


if __name__ == "__main__":
    main()
