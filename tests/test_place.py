"""Compact-work placement across data-parallel replicas (HARTS Section 3.2), CPU tests.

The planner's plans are checked against the oracle's definitions (oracle/placement.py): every
microbatch's work is the number of distinct prefixes of its trajectories, the Eq. 4 terms are
recomputed from the assignment, the contiguous exact search reaches the brute-force minimum over
all contiguous partitions (the space Eq. 9 searches), and no plan beats the brute-force optimum
over every set partition on tiny inputs."""

import numpy as np
import pytest

import dag_packed_paged_gb300 as ta
from oracle import placement as O


def rollouts(seed, n_traj, vocab=5, max_len=40):
    """Token trajectories of a random rollout forest: each new trajectory copies a prefix of an
    earlier one (a fork at a uniform point) or starts fresh, then continues with random tokens;
    a few exact duplicates and prefixes of others are mixed in."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 6006]))
    out = []
    for i in range(n_traj):
        r = rng.random()
        if out and r < 0.1:
            out.append(out[int(rng.integers(len(out)))].copy())                   # duplicate
        elif out and r < 0.2:
            src = out[int(rng.integers(len(out)))]
            out.append(src[: max(1, int(rng.integers(1, len(src) + 1)))].copy())  # a prefix
        elif out and r < 0.85:
            src = out[int(rng.integers(len(out)))]
            f = int(rng.integers(0, len(src) + 1))
            tail = rng.integers(0, vocab, size=int(rng.integers(1, max_len // 2 + 1)))
            out.append(np.concatenate([src[:f], tail]).astype(np.int32))
        else:
            out.append(rng.integers(0, vocab, size=int(rng.integers(1, max_len + 1))).astype(np.int32))
    return out


def check_plan(trajs, res, D, T):
    K = res["n_microbatches"]
    assert K % D == 0 and K == len(res["work"]) and res["n_slots"] == K // D
    mb = res["microbatch_of"]
    assert sorted(set(mb.tolist())) == list(range(K))                  # every microbatch non-empty
    for m in range(K):
        members = [trajs[i] for i in np.nonzero(mb == m)[0]]
        assert res["work"][m] == O.compact_work(members) <= T
    # one microbatch per replica per slot
    pairs = set(zip(res["replica_of"].tolist(), res["slot_of"].tolist()))
    assert len(pairs) == K and {r for r, _ in pairs} == set(range(D))
    assert (res["total_work"], res["slot_critical_work"], res["max_replica_work"]) == O.objective(
        res["work"], res["replica_of"], res["slot_of"])
    assert res["merged_work"] == O.compact_work(trajs)
    # slots hold the microbatches in descending work order, heavier ones on lighter replicas
    order = np.argsort(-res["work"], kind="stable")
    load = np.zeros(D, dtype=np.int64)
    for s in range(K // D):
        ms = order[s * D:(s + 1) * D]
        assert all(res["slot_of"][m] == s for m in ms)
        before = load.copy()
        for m in ms:
            load[res["replica_of"][m]] += res["work"][m]
        reps = [res["replica_of"][m] for m in ms]
        assert all(before[a] <= before[b] for a, b in zip(reps, reps[1:]))


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("D", [1, 2, 4])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_plans_are_valid_and_their_work_exact(seed, D, mode):
    trajs = rollouts(seed, 12 + 5 * seed)
    T = max(len(t) for t in trajs) + (seed % 4) * 20
    res = ta.tree_attn_place(trajs, replicas=D, capacity=T, mode=mode)
    check_plan(trajs, res, D, T)
    G = O.compact_work(trajs)
    assert res["k_min"] == D * max(1, -(-G // (T * D)))                   # Eq. 7


@pytest.mark.parametrize("seed", range(25))
def test_contiguous_search_reaches_the_contiguous_minimum(seed):
    """Eq. 9 is exact over partitions contiguous in lexicographic order: brute force over every
    such partition with K in the planner's range finds no smaller total work."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(3, 10))
    trajs = rollouts(100 + seed, n, vocab=3, max_len=12)
    D = int(rng.integers(1, 4))
    if n < D:
        D = 1
    T = max(len(t) for t in trajs) + int(rng.integers(0, 25))
    res = ta.tree_attn_place(trajs, replicas=D, capacity=T, mode=1)
    check_plan(trajs, res, D, T)
    srt = sorted(trajs, key=lambda t: tuple(t.tolist()))
    best = None
    for K in range(res["k_min"], res["k_max"] + 1, D):
        if K > n:
            continue
        for starts in O.contiguous_partitions(n, K):
            bounds = starts + [n]
            ws = [O.compact_work(srt[a:b]) for a, b in zip(bounds, bounds[1:])]
            if max(ws) <= T and (best is None or sum(ws) < best):
                best = sum(ws)
    assert best is not None and res["total_work"] == best


@pytest.mark.parametrize("seed", range(10))
def test_no_plan_beats_the_global_optimum(seed):
    """Tiny inputs: brute force over every set partition with K a multiple of D within capacity.
    The planner's total work is never below that optimum, and combining both candidate kinds
    is never worse than either kind alone under Eq. 4."""
    rng = np.random.default_rng(1000 + seed)
    n = int(rng.integers(2, 7))
    trajs = rollouts(200 + seed, n, vocab=3, max_len=10)
    D = 2 if n >= 2 else 1
    T = max(len(t) for t in trajs) + int(rng.integers(0, 15))
    opt = None
    for part in O.set_partitions(list(range(n))):
        if len(part) % D:
            continue
        ws = [O.compact_work([trajs[i] for i in g]) for g in part]
        if max(ws) <= T and (opt is None or sum(ws) < opt):
            opt = sum(ws)
    res = {m: ta.tree_attn_place(trajs, replicas=D, capacity=T, mode=m) for m in (0, 1, 2)}
    for r in res.values():
        check_plan(trajs, r, D, T)
        assert r["total_work"] >= opt
    key = lambda r: (r["total_work"], r["slot_critical_work"], r["max_replica_work"])
    assert key(res[0]) == min(key(res[1]), key(res[2]))


def test_greedy_shares_prefixes():
    """Two rollout trees whose trajectories share long prefixes within a tree and nothing across:
    with room for one tree per microbatch and two replicas, the plan keeps each tree together
    (total work = the merged trie's work, each replica one tree)."""
    rng = np.random.default_rng(3)
    trees = []
    for root_tok in (1, 2):
        root = np.concatenate([[root_tok], rng.integers(3, 9, size=200)]).astype(np.int32)
        trees.append([np.concatenate([root[:150 + 10 * k], rng.integers(3, 9, size=30)]).astype(np.int32)
                      for k in range(5)])
    trajs = trees[0] + trees[1]
    one_tree = O.compact_work(trees[0])
    for mode in (0, 2):
        res = ta.tree_attn_place(trajs, replicas=2, capacity=max(one_tree, O.compact_work(trees[1])), mode=mode)
        check_plan(trajs, res, 2, 10 ** 9)
        assert res["total_work"] == O.compact_work(trajs)
        assert res["n_microbatches"] == 2
        assert len(set(res["microbatch_of"][:5])) == 1 and len(set(res["microbatch_of"][5:])) == 1


def test_microbatches_ingest_to_their_work():
    """Each microbatch's compact work is the row count tree_attn_ingest builds for it (Eq. 5)."""
    trajs = rollouts(7, 40, vocab=4, max_len=60)
    res = ta.tree_attn_place(trajs, replicas=4, capacity=400)
    for m in range(res["n_microbatches"]):
        members = [trajs[i] for i in np.nonzero(res["microbatch_of"] == m)[0]]
        br, rows, _ = ta.tree_attn_ingest(members)
        assert len(rows) == res["work"][m]


def test_large_input_uses_evolved_partitions():
    """Above the exact-search threshold the contiguous candidates come from the evolved natural
    partition; plans stay valid."""
    trajs = rollouts(11, 90, vocab=4, max_len=30)
    T = 200
    res = ta.tree_attn_place(trajs, replicas=3, capacity=T, mode=1, exact_max_traj=16)
    check_plan(trajs, res, 3, T)
    exact = ta.tree_attn_place(trajs, replicas=3, capacity=T, mode=1)
    assert exact["total_work"] <= res["total_work"]


def test_place_units():
    rng = np.random.default_rng(5)
    for n, D in [(16, 4), (7, 3), (1, 2), (9, 1)]:
        w = rng.integers(1, 1000, size=n)
        res = ta.tree_attn_place_units(w, D)
        assert (res["total_work"], res["slot_critical_work"], res["max_replica_work"]) == O.objective(
            w, res["replica_of"], res["slot_of"])
        for s in set(res["slot_of"].tolist()):
            reps = res["replica_of"][res["slot_of"] == s]
            assert len(reps) == len(set(reps.tolist())) <= D
        order = np.argsort(-w, kind="stable")
        assert (res["slot_of"][order] == np.arange(n) // D).all()
    # equal units: each replica gets the same number
    res = ta.tree_attn_place_units(np.full(16, 65536), 4)
    assert np.bincount(res["replica_of"]).tolist() == [4, 4, 4, 4] and res["max_replica_work"] == 4 * 65536


def test_rejects_bad_inputs():
    trajs = rollouts(1, 6)
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_place(trajs, replicas=2, capacity=3)                    # a trajectory beyond capacity
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_place(trajs[:1], replicas=2, capacity=1000)            # fewer trajectories than replicas
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_place([np.zeros(0, np.int32)] + trajs, replicas=1, capacity=1000)
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_place_units(np.array([-1, 2]), 2)


def test_natural_partition_splits_at_the_lowest_valleys():
    """Three rollout trees that share nothing across (adjacent LCP 0 at the two tree boundaries)
    and long prefixes within: with capacity for exactly one tree, splitting heavy intervals at
    their lowest adjacent-LCP valley cuts exactly at the tree boundaries -- three microbatches."""
    rng = np.random.default_rng(9)
    trajs = []
    for root_tok in (1, 2, 3):
        root = np.concatenate([[root_tok], rng.integers(4, 9, size=120)]).astype(np.int32)
        trajs += [np.concatenate([root[:60 + 15 * k], rng.integers(4, 9, size=20)]).astype(np.int32)
                  for k in range(4)]
    works = [O.compact_work(trajs[4 * i:4 * i + 4]) for i in range(3)]
    res = ta.tree_attn_place(trajs, replicas=1, capacity=max(works), mode=1)
    assert res["k_natural"] == 3
    check_plan(trajs, res, 1, max(works))
