"""Forward parity on the GPU: libtreeattn (through its C ABI) against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import dag
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close, metrics

pytestmark = pytest.mark.gpu


def _oracle_fwd(ep, t, rows=None):
    return oracle.forward(ep.branches, ep.mounts, t.q, t.k, t.v, ep.softmax_scale, rows=rows)


SMALL = [
    ("tiny", lambda: W.tiny()),
    ("balanced/16", lambda: W.scaled(1, 16)),
    ("commander/32", lambda: W.scaled(2, 32)),
    ("irregular/32", lambda: W.scaled(3, 32)),
    ("mount_heavy/64", lambda: W.scaled(4, 64)),
]


@pytest.mark.parametrize("name,make", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("dist", ["config", "realistic", "sharp"])
def test_fwd_small_configs(name, make, dist):
    ep = make()
    run = Run(ep, dist=dist)
    o, lse = run.fwd()
    ref = _oracle_fwd(ep, run.t)
    assert_close("O", o, ref.o)
    ma, _ = metrics(lse, ref.lse)
    assert ma <= 2e-3, f"lse max_abs {ma}"


SHAPES = [((4, 1), 64, 16), ((1, 1), 128, 64), ((2, 1), 64, 32), ((8, 1), 128, 128),
          ((16, 1), 128, 64), ((16, 2), 64, 16), ((32, 8), 128, 64), ((8, 4), 128, 32)]


@pytest.mark.parametrize("seed", range(16))
def test_fwd_random_dags(seed):
    heads, D, P = SHAPES[seed % len(SHAPES)]
    ep = W.random_small(1000 + seed, max_branches=8, max_len=700, heads=heads, head_dim=D,
                        page_size=P, n_mounts=seed % 4)
    run = Run(ep, dist="realistic")
    o, lse = run.fwd()
    ref = _oracle_fwd(ep, run.t)
    assert_close("O", o, ref.o)
    assert metrics(lse, ref.lse)[0] <= 2e-3


@pytest.mark.parametrize("ep", [W.tiny(), W.scaled(4, 64), W.random_small(7, heads=(8, 1), head_dim=128)],
                         ids=lambda e: e.name)
def test_fwd_zero_queries_closed_form(ep):
    """Q = 0: every visible key gets the same weight, so lse = ln |vis(r)| and O is the mean
    of V over vis(r) -- this pins the visible-set sizes on the GPU."""
    t = W.make_tensors(ep)
    t.q[...] = 0
    run = Run(ep, tensors=t)
    o, lse = run.fwd()
    rows, ptr, lo, hi = dag.visible_intervals(ep.branches, ep.mounts)
    counts = np.array([int((hi[ptr[r]:ptr[r + 1]] - lo[ptr[r]:ptr[r + 1]]).sum()) for r in rows])
    assert np.abs(lse - np.log(counts)[:, None]).max() < 1e-5
    ref = _oracle_fwd(ep, t)
    assert_close("O", o, ref.o, max_abs=2e-3, rel_rms=5e-3)


def test_fwd_deterministic():
    ep = W.scaled(2, 32)
    run = Run(ep)
    o1, l1 = run.fwd()
    o2, l2 = run.fwd()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


FULL = [1, 2, 3, 4]


@pytest.mark.parametrize("cfg", FULL)
def test_fwd_full_size_sampled_rows(cfg):
    """The full-size workloads in the benchmark's launch configuration; the oracle checks a
    seeded sample of rows (deepest rows included) one by one."""
    ep = W.config(cfg)
    run = Run(ep)
    o, lse = run.fwd()
    rng = np.random.default_rng(cfg)
    N = ep.n_rows
    rows = np.unique(np.concatenate([rng.choice(N, 48, replace=False), [0, N - 1],
                                     ep.branches["row_start"] + ep.branches["length"] - 1]))[:96]
    ref = _oracle_fwd(ep, run.t, rows=rows)
    assert_close("O", o[rows], ref.o)
    assert metrics(lse[rows], ref.lse)[0] <= 2e-3
    assert np.isfinite(o).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("heads,page", [((4, 1), 16), ((16, 4), 16), ((8, 1), 32)], ids=["G4-P16", "G4x4-P16", "G8-P32"])
def test_fwd_bwd_head_dim_128_small_pages(heads, page):
    """Head dim 128 (the CTA-pair forward) on 16- and 32-row pages: a 32-row slot of a packed key
    tile is then two pages (two TMA boxes per CTA half), or one box per slot with no 64-row
    halves -- the load paths the page-64 workloads do not take."""
    ep = W.random_small(3000 + page + heads[0], max_branches=8, max_len=700, heads=heads, head_dim=128,
                        page_size=page, n_mounts=3)
    run = Run(ep, dist="realistic")
    o, lse = run.fwd()
    dq, dk, dv = run.bwd()
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    assert_close("O", o, ref.o)
    assert metrics(lse, ref.lse)[0] <= 2e-3
    assert_close("dQ", dq, ref.dq)
    assert_close("dK", dk, ref.dk)
    assert_close("dV", dv, ref.dv)
