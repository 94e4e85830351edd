"""The host index of the compact log-probability backward (tree_attn_logprob_index) and the
semantic positions of the synthetic workloads (no GPU)."""
import numpy as np
import pytest

import dag_packed_paged_gb300 as ta
from dag_packed_paged_gb300 import workloads as W
from oracle import dag


def test_index_groups_by_row_then_target():
    rng = np.random.default_rng(0)
    C, V, S = 50, 1000, 700
    pr = rng.integers(0, C, S)
    pt = rng.integers(0, 20, S).astype(np.int32)      # many repeated targets
    ptr, pos = ta.tree_attn_logprob_index(pr, pt, C, V)
    assert ptr[0] == 0 and ptr[-1] == S and np.all(np.diff(ptr) >= 0)
    assert sorted(pos.tolist()) == list(range(S))
    for c in range(C):
        seg = pos[ptr[c]:ptr[c + 1]]
        assert np.all(pr[seg] == c) and len(seg) == int((pr == c).sum())
        keys = list(zip(pt[seg].tolist(), seg.tolist()))
        assert keys == sorted(keys)                      # by target, then by position


def test_index_rejects_out_of_range():
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_logprob_index(np.array([0, 5]), np.array([1, 1], np.int32), 5, 10)
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_logprob_index(np.array([0, 1]), np.array([1, 10], np.int32), 5, 10)


@pytest.mark.parametrize("make", [W.tiny, lambda: W.scaled(1, 16), lambda: W.scaled(3, 32)])
def test_semantic_positions_follow_the_trajectories(make):
    ep = make()
    V = 512
    pr, pt, tok = W.semantic_positions(ep, V)
    # independent path: the oracle's trajectories (query rows only) give the same positions
    want_rows, want_tgt = [], []
    for traj in dag.trajectories(ep.branches, ep.mounts):
        q = [r for r, is_q in traj if is_q]
        want_rows += q[:-1]
        want_tgt += [int(tok[r]) for r in q[1:]]
    assert np.array_equal(pr, np.array(want_rows)) and np.array_equal(pt, np.array(want_tgt))
    assert len(pr) > ep.n_rows - len(ep.branches)    # forks make rows serve several positions
