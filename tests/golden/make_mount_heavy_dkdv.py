"""Writes mount_heavy_dag0_dkdv.npz: the oracle's dK and dV on key rows of the full-size
mount-heavy episode whose gradients gather from the most readers -- rows of the producer span
[4096, 8192) that 32 readers mount (Octopus Section 3.4, differentiable mount edges: gradients
flow back through mounts into the producer's K/V) and rows of the 8,192-row root that every row
of the DAG reads (HARTS Section 3.4: the gather backward accumulates every consumer into the
unique compact row).

Only the oracle runs here (fp64 CPU), over every row of the first of the episode's four
independent DAGs: those rows are all the readers of that DAG's keys.  The other three DAGs are
independent and are not needed.  The file records the seed, the generator's inputs (a SHA-256
over the DAG's Q, K, V, dO bits and its topology) and the rows; the GPU test regenerates the
inputs, checks the hash, and compares.  It takes about ten minutes on eight host cores.

    python tests/golden/make_mount_heavy_dkdv.py
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

OUT = os.path.join(HERE, "mount_heavy_dag0_dkdv.npz")
DAG_ROWS = 65_536          # rows of one of the four DAGs (the first one: rows [0, 65536))


def dag0_inputs(ep, t):
    """DAG 0's topology and tensors, and their hash."""
    sel = (ep.branches["row_start"] < DAG_ROWS)
    br = ep.branches[sel]
    nb = int(sel.sum())
    mt = ep.mounts[(ep.mounts["reader"] < nb) & (ep.mounts["source"] < nb)]
    h = hashlib.sha256()
    for a in (br, mt, t.q[:DAG_ROWS], t.k[:DAG_ROWS], t.v[:DAG_ROWS], t.do[:DAG_ROWS]):
        h.update(np.ascontiguousarray(a).tobytes())
    return br, mt, h.hexdigest()


def key_rows(ep):
    """32 rows of the mounted producer span and 32 of the root, seeded, ends included."""
    producer = 1                                      # branch 1 of DAG 0 (its first worker)
    m0 = ep.mounts[ep.mounts["source"] == producer][0]
    s0 = int(ep.branches["row_start"][producer])
    lo, hi = s0 + int(m0["src_begin"]), s0 + int(m0["src_end"])
    rng = np.random.default_rng(np.random.SeedSequence([0, 5005]))
    span = np.concatenate([[lo, hi - 1], rng.choice(np.arange(lo + 1, hi - 1), 30, replace=False)])
    root = np.concatenate([[0, 8191], rng.choice(np.arange(1, 8191), 30, replace=False)])
    return np.sort(np.concatenate([span, root])).astype(np.int64), (lo, hi)


def main():
    ep = W.config(4)
    t = W.make_tensors(ep)
    br, mt, digest = dag0_inputs(ep, t)
    rows, span = key_rows(ep)
    sl = slice(0, DAG_ROWS)
    t0 = time.time()
    res = oracle.run(br, mt, t.q[sl], t.k[sl], t.v[sl], t.do[sl], ep.softmax_scale)
    dt = time.time() - t0
    np.savez_compressed(OUT, rows=rows, span=np.array(span), dk=res.dk[rows].astype(np.float32),
                        dv=res.dv[rows].astype(np.float32), seed=np.int64(ep.seed), input_sha256=digest,
                        workload=ep.name, dag_rows=np.int64(DAG_ROWS))
    print(f"wrote {OUT}: {len(rows)} key rows, oracle {dt:.0f} s on {res.threads} threads")


if __name__ == "__main__":
    main()
