"""Pins for the oracle's two other visibility views (same rows, same Eq. 2 positions):

* ``no_mounts`` -- the unmounted layers of Octopus Section 3.2 / Appendix C Table 8: equal to
  the same episode with its mount list emptied, an independent path through the oracle;
* ``transitive`` -- Octopus Section 3.3 item 1, active mounts "including transitive mounts":
  visible sets derived by hand for a crafted episode (a two-level chain of mounts, a span that
  ends just before its source's own mount, a source whose mount is inherited from its
  parent), plus inclusion properties on random episodes; planted mistakes must fail the pin.
"""
import numpy as np
import pytest

import oracle
from oracle import dag
from dag_packed_paged_gb300 import workloads as W


def crafted():
    # branch: (parent, fork, length, row_start)
    br = W.make_branches([-1, 0, 0, 0, 0, 3, 0], [0, 8, 8, 8, 8, 4, 8], [8, 8, 8, 8, 8, 4, 6])
    # branches 0 root, 1 B, 2 A, 3 C, 4 D, 5 E (child of C at 4), 6 F
    #        reader, offset, source, [begin, end)
    mts = W.make_mounts([(2, 3, 1, 2, 6),    # A mounts B [2, 6) at A's row 3
                         (3, 2, 2, 1, 7),    # C mounts A [1, 7) at C's row 2
                         (4, 5, 3, 0, 4),    # D mounts C [0, 4) at D's row 5
                         (4, 1, 2, 0, 3),    # D mounts A [0, 3) at D's row 1 (ends before A's mount)
                         (6, 2, 5, 0, 3)])   # F mounts E [0, 3) at F's row 2
    return br, mts


R = lambda a, b: set(range(a, b))   # noqa: E731
# rows (DFS layout): root 0..7, B 8..15, A 16..23, C 24..31, E 32..35, D 36..43, F 44..49
ROOT = R(0, 8)
# row -> (visible set, mounted view ; visible set, transitive view), derived by hand
EXPECTED = {
    42: (ROOT | R(16, 19) | R(24, 28) | R(36, 43),            # D@6: D, root, A[0,3), C[0,4)
         ROOT | R(10, 14) | R(16, 23) | R(24, 28) | R(36, 43)),  # + C's mount A[1,7) + A's B[2,6)
    39: (ROOT | R(16, 19) | R(36, 40),                        # D@3: A[0,3) only
         ROOT | R(16, 19) | R(36, 40)),                       # A's row 2 < its mount offset 3
    34: (ROOT | R(17, 23) | R(24, 28) | R(32, 35),            # E@2 inherits C[0,4) and C's A[1,7)
         ROOT | R(10, 14) | R(17, 23) | R(24, 28) | R(32, 35)),
    48: (ROOT | R(32, 35) | R(44, 49),                        # F@4: E[0,3) (no E ancestors)
         ROOT | R(10, 14) | R(17, 23) | R(32, 35) | R(44, 49)),  # E's inherited A[1,7), then B
    25: (ROOT | R(24, 26), ROOT | R(24, 26)),                 # C@1: before its mount
    21: (ROOT | R(10, 14) | R(16, 22), ROOT | R(10, 14) | R(16, 22)),  # A@5: B's span, B has none
}


def _pin_holds():
    br, mts = crafted()
    for row, (want_m, want_t) in EXPECTED.items():
        if dag.visible_set(br, mts, row) != want_m or dag.visible_set(br, mts, row, view="transitive") != want_t:
            return False
    return True


def test_crafted_transitive_and_mounted_sets():
    assert _pin_holds()
    br, mts = crafted()
    # the no-mounts view keeps only the ancestor path and the row's own predecessors
    assert dag.visible_set(br, mts, 42, view="no_mounts") == ROOT | R(36, 43)
    assert dag.visible_set(br, mts, 34, view="no_mounts") == ROOT | R(24, 28) | R(32, 35)


def _no_recursion(branches, mounts, spans):
    return list(spans) + [sp for (s, lo, hi) in spans for sp in dag.mounts_in_effect(branches, mounts, s, hi - 1)]


def _end_inclusive(branches, mounts, spans):
    out, seen, stack = [], set(), list(spans)
    while stack:
        sp = stack.pop()
        if sp in seen:
            continue
        seen.add(sp)
        out.append(sp)
        stack.extend(dag.mounts_in_effect(branches, mounts, sp[0], sp[2]))   # should be hi - 1
    return out


def _own_only(branches, mounts, spans):
    M = dag._mt(mounts)
    out, seen, stack = [], set(), list(spans)
    while stack:
        sp = stack.pop()
        if sp in seen:
            continue
        seen.add(sp)
        out.append(sp)
        s, lo, hi = sp
        stack.extend((src, a, z) for (r, t, src, a, z) in M if r == s and t <= hi - 1 and z > a)
    return out


@pytest.mark.parametrize("name,fn", [("closure not recursive", _no_recursion),
                                     ("source row e instead of e-1", _end_inclusive),
                                     ("source's inherited mounts ignored", _own_only)])
def test_planted_closure_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(dag, "_closure", fn)
    assert not _pin_holds(), name


EPISODES = [lambda: W.tiny(), lambda: W.scaled(2, 64), lambda: W.scaled(4, 128)] + \
    [(lambda s=s: W.random_small(300 + s, max_branches=10, max_len=120, n_mounts=1 + s % 5)) for s in range(12)]


@pytest.mark.parametrize("make", EPISODES)
def test_no_mounts_equals_empty_mount_list(make):
    ep = make()
    a = dag.visible_intervals(ep.branches, ep.mounts, view="no_mounts")
    b = dag.visible_intervals(ep.branches, ep.mounts[:0])
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("make", EPISODES)
def test_view_inclusions(make):
    ep = make()
    rows = np.arange(ep.n_rows)[:: max(1, ep.n_rows // 200)]
    for r in rows:
        nm = dag.visible_set(ep.branches, ep.mounts, int(r), view="no_mounts")
        m = dag.visible_set(ep.branches, ep.mounts, int(r))
        t = dag.visible_set(ep.branches, ep.mounts, int(r), view="transitive")
        assert nm <= m <= t


def test_transitive_equals_mounted_without_chains():
    # mount_heavy: every source (the producer) has no mounts of its own -> nothing to close over
    ep = W.scaled(4, 128)
    a = dag.visible_intervals(ep.branches, ep.mounts, view="transitive")
    b = dag.visible_intervals(ep.branches, ep.mounts)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_oracle_forward_no_mounts_is_the_mount_free_episode():
    ep = W.scaled(2, 64)
    t = W.make_tensors(ep, dist="realistic")
    a = oracle.forward(ep.branches, ep.mounts, t.q, t.k, t.v, ep.softmax_scale, view="no_mounts")
    b = oracle.forward(ep.branches, ep.mounts[:0], t.q, t.k, t.v, ep.softmax_scale)
    assert np.array_equal(a.o, b.o) and np.array_equal(a.lse, b.lse)
