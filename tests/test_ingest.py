"""Trajectory ingestion (HARTS Section 2.1 compact map m: S -> C, Eq. 3; Section 3.2 Eq. 5):
raw token trajectories -> compact prefix-tree episode, checked against the oracle's Eq. 5
count and DAG visibility (no GPU needed)."""
import numpy as np
import pytest

import dag_packed_paged_gb300 as ta
from oracle import dag


def random_trajectories(seed, n=24, vocab=4, max_len=40):
    """Trajectories with many shared prefixes: random walks in a small-vocabulary token tree,
    plus exact duplicates, strict prefixes of others and an empty one."""
    rng = np.random.default_rng(seed)
    trajs = []
    for _ in range(n):
        if trajs and rng.random() < 0.5:
            base = trajs[int(rng.integers(len(trajs)))]
            cut = int(rng.integers(0, len(base) + 1))
            tail = rng.integers(0, vocab, size=int(rng.integers(0, max_len // 2)))
            trajs.append(np.concatenate([base[:cut], tail]).astype(np.int32))
        else:
            trajs.append(rng.integers(0, vocab, size=int(rng.integers(1, max_len))).astype(np.int32))
    trajs.append(trajs[int(rng.integers(len(trajs)))].copy())          # duplicate
    b = trajs[int(rng.integers(len(trajs)))]
    trajs.append(b[: len(b) // 2].copy())                                # strict prefix
    trajs.append(np.zeros(0, dtype=np.int32))                             # empty
    order = rng.permutation(len(trajs))
    return [trajs[i] for i in order]


def _plan(br):
    n = int((br["row_start"] + br["length"]).max()) if len(br) else 0
    pt = np.arange(max(1, -(-n // 16)), dtype=np.int32)
    return ta.tree_attn_plan(br, np.zeros(0, dtype=dag_mount_dtype()), pt, num_q_heads=4, num_kv_heads=1,
                             head_dim=64, page_size=16, num_pages=len(pt) + 1, flags=ta.TA_PLAN_HOST_ONLY)


def dag_mount_dtype():
    from dag_packed_paged_gb300 import workloads as W
    return W.MOUNT_DTYPE


@pytest.mark.parametrize("seed", range(20))
def test_ingest_matches_eq5_and_visibility(seed):
    trajs = random_trajectories(seed)
    br, row_tokens, row_of = ta.tree_attn_ingest(trajs)
    n = len(row_tokens)
    assert n == dag.compact_rows_eq5(trajs)                      # Eq. 5
    for t, rows in zip(trajs, row_of):                            # m maps every token to its row
        assert np.array_equal(row_tokens[rows], t)
    # a compact row sees exactly its trajectory's prefix (no mounts)
    rng = np.random.default_rng(seed)
    for i in rng.choice(len(trajs), 6, replace=False):
        rows = row_of[i]
        for t in range(len(rows)):
            assert dag.visible_set(br, [], int(rows[t])) == set(rows[: t + 1].tolist())
    # equal prefixes share rows; different tokens at a position never share a row
    for a in range(len(trajs)):
        for b in range(a):
            x, y = trajs[a], trajs[b]
            m = min(len(x), len(y))
            lcp = int(np.argmax(x[:m] != y[:m])) if m and (x[:m] != y[:m]).any() else m
            assert np.array_equal(row_of[a][:lcp], row_of[b][:lcp])
            if lcp < m:
                assert row_of[a][lcp] != row_of[b][lcp]
    # the episode plans as is; its positions are the trajectory offsets
    plan = _plan(br)
    pos = ta.tree_attn_plan_export(plan)["pos_ids"]
    for t, rows in zip(trajs, row_of):
        assert np.array_equal(pos[rows], np.arange(len(t)))
    assert np.array_equal(pos, dag.positions(br, []))


def test_ingest_is_independent_of_input_order():
    trajs = [t for t in random_trajectories(3) if len(t)]
    uniq = {tuple(t): t for t in trajs}
    trajs = list(uniq.values())
    a = ta.tree_attn_ingest(trajs)
    b = ta.tree_attn_ingest(trajs[::-1])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    for x, y in zip(a[2], b[2][::-1]):
        assert np.array_equal(x, y)


def test_ingest_edge_cases():
    br, rt, ro = ta.tree_attn_ingest([])
    assert len(br) == 0 and len(rt) == 0 and ro == []
    br, rt, ro = ta.tree_attn_ingest([np.zeros(0, np.int32)] * 3)
    assert len(br) == 0 and len(rt) == 0
    br, rt, ro = ta.tree_attn_ingest([[5, 6, 7]])
    assert br.tolist() == [(-1, 0, 3, 0)] and rt.tolist() == [5, 6, 7]
    # a trajectory extending another forks at the parent's end
    br, rt, ro = ta.tree_attn_ingest([[1, 2], [1, 2, 3]])
    assert br.tolist() == [(-1, 0, 2, 0), (0, 2, 1, 2)]


def test_ingest_rejects_bad_arguments():
    import ctypes
    L = ta._native.lib()
    tok = np.array([1, 2, 3], dtype=np.int32)
    bad = np.array([0, 2, 1], dtype=np.int64)                  # decreasing offsets
    nb, nr = ctypes.c_int32(0), ctypes.c_int64(0)
    out = np.zeros(4, dtype=ta._native.BRANCH_DTYPE)
    rows = np.zeros(4, dtype=np.int64)
    rc = L.tree_attn_ingest(tok.ctypes.data, bad.ctypes.data, 2, out.ctypes.data, 4, ctypes.byref(nb), None, 4,
                            ctypes.byref(nr), rows.ctypes.data, None)
    assert rc == ta.TA_ERR_INVALID
    good = np.array([0, 3], dtype=np.int64)
    rc = L.tree_attn_ingest(tok.ctypes.data, good.ctypes.data, 1, out.ctypes.data, 0, ctypes.byref(nb), None, 4,
                            ctypes.byref(nr), rows.ctypes.data, None)    # no branch capacity
    assert rc == ta.TA_ERR_INVALID


# ------------------------------------------------------------------ Octopus Eq. 6 owner mask
def _prefix_value(prefix):
    """A deterministic stand-in for log p(last token | rest) of a raw token prefix."""
    return (hash(tuple(int(x) for x in prefix)) % 10007) / 10007.0 - 0.5


@pytest.mark.parametrize("seed", range(12))
def test_owner_mask_counts_every_generated_prefix_once(seed):
    """Eq. 7: the masked sum over all trajectories' positions equals the sum over the distinct
    generated token prefixes (each counted once) -- checked against raw token tuples."""
    trajs = random_trajectories(seed)
    br, row_tokens, row_of, row_owner = ta.tree_attn_ingest(trajs, with_owner=True)
    # generated flag as a function of the raw prefix ending at the token (consistent across
    # trajectories sharing it): prompts / tool outputs are the other tokens
    generated = [np.array([hash(tuple(int(x) for x in t[: k + 1])) % 3 != 0 for k in range(len(t))], dtype=np.uint8)
                 for t in trajs]
    mask = ta.tree_attn_owner_mask(row_of, row_owner, generated)
    got = sum(_prefix_value(t[: k + 2]) for t, m in zip(trajs, mask) for k in np.nonzero(m)[0])
    distinct = {tuple(int(x) for x in t[: k + 1]) for t, g in zip(trajs, generated) for k in range(1, len(t)) if g[k]}
    want = sum(_prefix_value(p) for p in distinct)
    assert abs(got - want) < 1e-9
    assert sum(int(m.sum()) for m in mask) == len(distinct)
    # every masked position sits in the trajectory that owns the predicted token's row
    for l, (rows, m) in enumerate(zip(row_of, mask)):
        for k in np.nonzero(m)[0]:
            assert row_owner[rows[k + 1]] == l
        if len(m):
            assert m[-1] == 0
    # owners pass through the rows they own
    for c, l in enumerate(row_owner):
        assert c in set(row_of[l].tolist())
