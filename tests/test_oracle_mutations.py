"""The pins must catch plausible mistakes: plant each one in the oracle's DAG semantics (on
the CPU, by monkeypatching) and check that the trajectory pin then fails."""
import numpy as np
import pytest

import oracle
from oracle import dag
from dag_packed_paged_gb300 import workloads as W
from test_oracle_pins import TRAJ_EPS, _traj_attention, crafted, f64


def _trajectory_pin_holds(eps):
    for ep in eps:
        t = W.make_tensors(ep, dist="realistic")
        qf, kf, vf = f64(t.q), f64(t.k), f64(t.v)
        res = oracle.forward(ep.branches, ep.mounts, t.q, t.k, t.v, ep.softmax_scale)
        G = ep.num_q_heads // ep.num_kv_heads
        for traj in dag.trajectories(ep.branches, ep.mounts):
            qrows, o, _ = _traj_attention(traj, qf, kf, vf, ep.softmax_scale, G)
            if np.abs(res.o[qrows] - o).max() > 1e-12:
                return False
    return True


def test_unmutated_holds():
    assert _trajectory_pin_holds([crafted()] + TRAJ_EPS[:6])


def _drop_parent_mounts(branches, mounts, b):
    B = dag._br(branches)
    out = []
    while B[b][0] >= 0:
        p, f = B[b][0], B[b][1]
        if f > 0:
            out.append((p, 0, f))
        b = p
    return out


def _prefix_off_by_one(branches, mounts, b):
    B = dag._br(branches)
    return [(p, lo, min(hi + 1, B[p][2])) if x == 0 else (p, lo, hi)
            for x, (p, lo, hi) in enumerate(_orig_inherited(branches, mounts, b))]


def _mount_activates_late(branches, mounts, b, i):
    M = dag._mt(mounts)
    out = [(b, 0, i + 1)]
    for (r, t, s, lo, hi) in M:
        if r == b and t < i and hi > lo:          # should be t <= i
            out.append((s, lo, hi))
    out += dag.inherited_pieces(branches, mounts, b)
    return out


def _no_own_row(branches, mounts, b, i):
    return [(b, 0, i) if x == 0 else p for x, p in enumerate(_orig_visible(branches, mounts, b, i))
            if not (x == 0 and i == 0)] or [(b, 0, 1)]


_orig_inherited = dag.inherited_pieces
_orig_visible = dag.visible_pieces


@pytest.mark.parametrize("name,attr,fn", [
    ("parent mounts not inherited", "inherited_pieces", _drop_parent_mounts),
    ("parent prefix one row too long", "inherited_pieces", _prefix_off_by_one),
    ("mount seen one row late", "visible_pieces", _mount_activates_late),
    ("query does not see itself", "visible_pieces", _no_own_row),
])
def test_planted_mistake_is_caught(monkeypatch, name, attr, fn):
    monkeypatch.setattr(dag, attr, fn)
    assert not _trajectory_pin_holds([crafted()] + TRAJ_EPS[:6]), name
