"""GPU parity for the mount-free (TA_NO_MOUNTS) and transitive-mount (TA_TRANSITIVE_MOUNTS)
views: forward and backward through the C ABI against the fp64 oracle with the same view."""
import numpy as np
import pytest

import dag_packed_paged_gb300 as ta
import oracle
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close, metrics
from test_oracle_views import crafted

pytestmark = pytest.mark.gpu

VIEWS = [(ta.TA_NO_MOUNTS, "no_mounts"), (ta.TA_TRANSITIVE_MOUNTS, "transitive")]


def _crafted_episode():
    br, mts = crafted()
    return W.Episode("crafted_views", br, mts, 8, 2, 128, 16, 0)


def _chain_episode(seed):
    """Random DAG whose mount sources are themselves readers, so closures are non-trivial."""
    rng = np.random.default_rng(seed)
    n = 6
    lens = [int(rng.integers(60, 400)) for _ in range(n)]
    parents = [-1] + [0] * (n - 1)
    forks = [0] + [lens[0]] * (n - 1)
    mounts = []
    for r in range(2, n):                      # branch r mounts a span of branch r-1 ...
        s = r - 1
        lo = int(rng.integers(0, lens[s] // 2))
        mounts.append((r, int(rng.integers(1, lens[r])), s, lo, lens[s]))
    return W.Episode(f"chain{seed}", W.make_branches(parents, forks, lens), W.make_mounts(mounts),
                     16, 4, 128, 64, seed)


EPISODES = [("crafted", _crafted_episode), ("commander/32", lambda: W.scaled(2, 32)),
            ("mount_heavy/64", lambda: W.scaled(4, 64)), ("chain7", lambda: _chain_episode(7)),
            ("chain8", lambda: _chain_episode(8)),
            ("random", lambda: W.random_small(911, max_branches=8, max_len=500, heads=(8, 2), head_dim=64,
                                              page_size=32, n_mounts=3))]


@pytest.mark.parametrize("name,make", EPISODES, ids=[e[0] for e in EPISODES])
@pytest.mark.parametrize("flags,view", VIEWS, ids=[v for _, v in VIEWS])
def test_views_fwd_bwd(name, make, flags, view):
    ep = make()
    run = Run(ep, dist="realistic", flags=flags)
    o, lse = run.fwd()
    dq, dk, dv = run.bwd()
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale, view=view)
    assert_close("O", o, ref.o)
    assert metrics(lse, ref.lse)[0] <= 2e-3
    assert_close("dQ", dq, ref.dq)
    assert_close("dK", dk, ref.dk)
    assert_close("dV", dv, ref.dv)


def test_transitive_differs_from_mounted_on_chains():
    """The chain episodes really exercise the closure (otherwise the test above proves little)."""
    from oracle import dag
    ep = _chain_episode(7)
    a = dag.count_pairs(ep.branches, ep.mounts, view="transitive")
    b = dag.count_pairs(ep.branches, ep.mounts)
    assert a > b
