"""Oracle: compact work and the replica-placement objective of HARTS (arXiv 2608.28158) Section 3.2.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Written from the definitions:

* compact work of a set of trajectories -- the number of distinct non-empty token prefixes,
  i.e. of nodes of their compact trie (HARTS Section 2.1: one compact row per distinct prefix;
  Section 3.2: the work of a microbatch is that count);
* the objective of Eq. 4, evaluated on a fully assigned plan: total work, the sum over slots of
  the slot's heaviest microbatch, and the heaviest replica's cumulative work, compared
  lexicographically;
* brute force over partitions: every way to cut the lexicographically sorted trajectories into
  contiguous groups (the space Eq. 9 searches exactly), and every set partition on tiny inputs.
"""
from __future__ import annotations


def compact_work(trajs) -> int:
    """Distinct non-empty prefixes of the trajectories (nodes of their trie)."""
    seen = set()
    for t in trajs:
        t = tuple(int(x) for x in t)
        for i in range(1, len(t) + 1):
            seen.add(t[:i])
    return len(seen)


def objective(work, replica, slot):
    """Eq. 4 terms of an assigned plan: (sum of work, sum over slots of the slot maximum,
    maximum over replicas of the replica's total)."""
    slots, reps = {}, {}
    for w, r, s in zip(work, replica, slot):
        slots[s] = max(slots.get(s, 0), int(w))
        reps[r] = reps.get(r, 0) + int(w)
    return (sum(int(w) for w in work), sum(slots.values()), max(reps.values()))


def contiguous_partitions(n, k):
    """All ways to cut range(n) into k non-empty contiguous groups (lists of start indices)."""
    if k == 1:
        yield [0]
        return
    def rec(start, left):
        if left == 1:
            yield []
            return
        for c in range(start + 1, n - left + 2):
            for rest in rec(c, left - 1):
                yield [c] + rest
    for cuts in rec(0, k):
        yield [0] + cuts


def set_partitions(items):
    """All set partitions of a small list."""
    if not items:
        yield []
        return
    first, rest = items[0], items[1:]
    for p in set_partitions(rest):
        for i in range(len(p)):
            yield p[:i] + [[first] + p[i]] + p[i + 1:]
        yield [[first]] + p
