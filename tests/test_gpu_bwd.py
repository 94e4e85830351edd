"""Backward parity on the GPU: dQ, dK, dV from libtreeattn against the fp64 oracle."""
import numpy as np
import pytest

import dag_packed_paged_gb300 as ta
import oracle
from oracle import dag
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close, metrics

pytestmark = pytest.mark.gpu

SMALL = [
    ("tiny", lambda: W.tiny()),
    ("balanced/16", lambda: W.scaled(1, 16)),
    ("commander/32", lambda: W.scaled(2, 32)),
    ("irregular/32", lambda: W.scaled(3, 32)),
    ("mount_heavy/64", lambda: W.scaled(4, 64)),
]


def _check_all(ep, run, ref):
    o, lse = run.fwd()
    dq, dk, dv = run.bwd()
    assert_close("O", o, ref.o)
    assert_close("dQ", dq, ref.dq)
    assert_close("dK", dk, ref.dk)
    assert_close("dV", dv, ref.dv)
    return dq, dk, dv


@pytest.mark.parametrize("name,make", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("dist", ["config", "realistic", "sharp"])
def test_bwd_small_configs(name, make, dist):
    ep = make()
    run = Run(ep, dist=dist)
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    _check_all(ep, run, ref)


def test_split_tiles_use_partials():
    """The tiny tree's root tile is read by every block; the plan splits its readers into
    several chunks whose partial sums are reduced -- make sure that path ran."""
    ep = W.tiny()
    run = Run(ep, dist="realistic")
    st = ta.tree_attn_plan_stats(run.plan)
    assert st["n_partial_slots"] >= 2
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    _check_all(ep, run, ref)


SHAPES = [((4, 1), 64, 16), ((1, 1), 128, 64), ((2, 1), 64, 32), ((8, 1), 128, 128),
          ((16, 1), 128, 64), ((16, 2), 64, 16), ((32, 8), 128, 64), ((8, 4), 128, 32)]


@pytest.mark.parametrize("seed", range(16))
def test_bwd_random_dags(seed):
    heads, D, P = SHAPES[seed % len(SHAPES)]
    ep = W.random_small(2000 + seed, max_branches=8, max_len=600, heads=heads, head_dim=D,
                        page_size=P, n_mounts=seed % 4)
    run = Run(ep, dist="realistic")
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    _check_all(ep, run, ref)


def test_bwd_deterministic():
    ep = W.scaled(4, 64)
    run = Run(ep)
    run.fwd()
    a = run.bwd()
    b = run.bwd()
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_untouched_pool_rows():
    """Spare pages (not in the page table) are never written by the backward."""
    ep = W.scaled(2, 32)
    run = Run(ep)
    run.fwd()
    run.bwd()
    spare = np.setdiff1d(np.arange(run.pool.k_pool.shape[0]), run.pool.page_table)
    assert len(spare) > 0
    assert (run.dk_pool[spare].abs().sum().item() == 0.0) and (run.dv_pool[spare].abs().sum().item() == 0.0)


def _cheap_key_rows(ep, max_reader_pairs=4_000_000, n=32):
    """Key rows whose readers' visible sets are small enough for the oracle to recompute
    every reader exactly (rows near the ends of unmounted leaf branches), with their readers."""
    rows, ptr, lo, hi = dag.visible_intervals(ep.branches, ep.mounts)
    owner = np.repeat(rows, np.diff(ptr))
    vis = np.array([int((hi[ptr[r]:ptr[r + 1]] - lo[ptr[r]:ptr[r + 1]]).sum()) for r in rows])
    br = ep.branches
    has_child_at_end = set()
    for b in range(len(br)):
        p = int(br["parent"][b])
        if p >= 0:
            has_child_at_end.add(p)
    mounted = {int(m["source"]) for m in ep.mounts}
    cand = []
    for b in range(len(br)):
        if b in has_child_at_end or b in mounted:
            continue
        end = int(br["row_start"][b] + br["length"][b])
        for k in (1, 3, 17, 64):
            if k <= int(br["length"][b]):
                cand.append(end - k)
    cols, readers = [], set()
    for j in cand:
        rd = owner[(lo <= j) & (j < hi)]
        cost = int(vis[rd].sum()) * ep.num_q_heads
        if cost * ep.head_dim <= max_reader_pairs * 128:
            cols.append(j)
            readers.update(rd.tolist())
        if len(cols) >= n:
            break
    return np.array(cols, dtype=np.int64), np.array(sorted(readers), dtype=np.int64)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_bwd_full_size(cfg):
    """Full-size workloads in the benchmark's launch configuration.  The oracle checks dQ on
    a seeded sample of rows, and dK/dV exactly on key rows near branch ends (computed from
    all of their readers); the whole-strip identities sum_j dK[j] = 0 and
    sum_j dV[j, g] = sum over rows and the heads of g of dO hold for every row."""
    ep = W.config(cfg)
    run = Run(ep)
    o, lse = run.fwd()
    dq, dk, dv = run.bwd()
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()
    N = ep.n_rows
    rng = np.random.default_rng(cfg)
    rows = np.unique(np.concatenate([rng.choice(N, 40, replace=False), [0, N - 1]]))
    f = oracle.forward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, ep.softmax_scale, rows=rows)
    b = oracle.backward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale, f,
                        with_dkdv=False)
    assert_close("O", o[rows], f.o)
    assert_close("dQ", dq[rows], b.dq)
    cols, rd = _cheap_key_rows(ep)
    assert len(cols) >= 4
    f2 = oracle.forward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, ep.softmax_scale, rows=rd)
    b2 = oracle.backward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale, f2)
    assert_close("dK", dk[cols], b2.dk[cols])
    assert_close("dV", dv[cols], b2.dv[cols])
    G = ep.num_q_heads // ep.num_kv_heads
    dof = W.bf16_bits_to_f32(run.t.do).astype(np.float64)
    want = dof.reshape(N, ep.num_kv_heads, G, ep.head_dim).sum((0, 2))
    got = dv.sum(0)
    assert np.linalg.norm(got - want) <= 1e-2 * np.linalg.norm(want)
    assert np.linalg.norm(dk.sum(0)) <= 1e-2 * np.abs(dk).sum(0).max()
