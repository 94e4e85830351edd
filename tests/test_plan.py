"""Planner tests (CPU): the plan's positions, visible intervals, key-tile entries and
transpose are compared bit-exactly with the oracle's explicit enumeration from the DAG."""
import numpy as np
import pytest

import oracle
from oracle import dag
import dag_packed_paged_gb300 as ta
from dag_packed_paged_gb300 import workloads as W

T = 128


def host_plan(ep, mounts=None, page_table=None, flags=0, **over):
    mounts = ep.mounts if mounts is None else mounts
    n_logical = -(-ep.n_rows // ep.page_size)
    pt = np.arange(n_logical, dtype=np.int32) if page_table is None else page_table
    kw = dict(num_q_heads=ep.num_q_heads, num_kv_heads=ep.num_kv_heads, head_dim=ep.head_dim,
              page_size=ep.page_size, num_pages=max(n_logical, 1) + 3)
    kw.update(over)
    return ta.tree_attn_plan(ep.branches, mounts, pt, flags=flags | ta.TA_PLAN_HOST_ONLY, **kw)


def _merge(iv):
    out = []
    for a, z in sorted(iv):
        if out and a <= out[-1][1]:
            out[-1] = (out[-1][0], max(out[-1][1], z))
        else:
            out.append((a, z))
    return out


def _intervals_to_set_runs(lo, hi):
    return [(int(a), int(b)) for a, b in zip(lo, hi)]


def check_plan_against_oracle(ep, rows_to_check=None, flags=0, view="mounted"):
    plan = host_plan(ep, flags=flags)
    ex = ta.tree_attn_plan_export(plan)
    st = ta.tree_attn_plan_stats(plan)
    N = ep.n_rows
    # positions (Eq. 2): bit-exact
    assert (ex["pos_ids"] == dag.positions(ep.branches, ep.mounts)).all()
    assert (plan.pos_ids == ex["pos_ids"]).all()
    # visible sets: per row, block intervals + own rows [diag_lo, r] == oracle enumeration
    rows, ptr, olo, ohi = dag.visible_intervals(ep.branches, ep.mounts, view=view)
    blocks, diag, ivp = ex["blocks"], ex["diag"], ex["blk_iv_ptr"]
    covered = np.zeros(N, dtype=np.int64)
    check = set(range(N)) if rows_to_check is None else set(rows_to_check)
    for b in range(len(blocks)):
        r0, n, e0, e1 = (int(x) for x in blocks[b])
        assert diag[b, 0] == r0 and diag[b, 1] == r0 + n and n <= plan_block_rows(ep)
        ivs = _intervals_to_set_runs(ex["iv_lo"][ivp[b]:ivp[b + 1]], ex["iv_hi"][ivp[b]:ivp[b + 1]])
        # sorted, disjoint, maximal, none touching the diagonal from above
        for (a, z), (a2, z2) in zip(ivs, ivs[1:]):
            assert a < z < a2 < z2
        ents = ex["entries"][e0:e1]
        for r in range(r0, r0 + n):
            covered[r] += 1
            if r not in check:
                continue
            want = _intervals_to_set_runs(olo[ptr[r]:ptr[r + 1]], ohi[ptr[r]:ptr[r + 1]])
            got = _merge(ivs + [(r0, r + 1)])
            assert got == want, (r, got, want)
            # the key-tile entries cover exactly the same rows, once each
            mark = np.zeros(N, dtype=np.int32)
            for tile, lo, hi, fl in ents:
                assert tile * T <= lo < hi <= (tile + 1) * T
                assert bool(fl & 2) == (lo != tile * T or hi != (tile + 1) * T)
                top = min(hi, r + 1) if fl & 1 else hi
                mark[lo:max(lo, top)] += 1
            wmask = np.zeros(N, dtype=np.int32)
            for a, z in want:
                wmask[a:z] = 1
            assert (mark == wmask).all(), r
            # the packed tiles of the query-major kernels cover the same rows, once each
            assert (packed_marks(ex, b, r, N) == wmask).all(), r
    assert (covered == 1).all()
    # causal flag only where some key lies above the block's first row
    for b in range(len(blocks)):
        r0, n, e0, e1 = (int(x) for x in blocks[b])
        for tile, lo, hi, fl in ex["entries"][e0:e1]:
            if fl & 1:
                assert hi - 1 > r0
    # transpose: same entries grouped by key tile; chunks cover every tile's range once
    ents, te = ex["entries"], ex["t_entries"]
    assert len(ents) == len(te) == st["n_entries"]
    fwd = sorted((int(b), int(lo), int(hi), int(fl)) for b in range(len(blocks))
                 for (_, lo, hi, fl) in ents[blocks[b, 2]:blocks[b, 3]])
    assert sorted(map(tuple, te.tolist())) == fwd
    tiles_of_te = np.empty(len(te), dtype=np.int64)
    for i, (b, lo, hi, fl) in enumerate(te):
        tiles_of_te[i] = lo // T
    assert (np.diff(tiles_of_te) >= 0).all()
    seen = np.zeros(len(te), dtype=np.int32)
    slots = []
    for tile, a, z, slot in ex["chunks"]:
        assert (tiles_of_te[a:z] == tile).all() and z > a
        seen[a:z] += 1
        if slot >= 0:
            slots.append(int(slot))
    assert (seen == 1).all()
    assert sorted(slots) == list(range(len(slots))) and len(slots) == st["n_partial_slots"]
    assert sorted(ex["fwd_order"].tolist()) == list(range(len(blocks)))
    check_packed_flags(ex, ep.page_size)
    fp = ex["fblk_ptr"]
    assert fp[0] == 0 and (np.diff(fp) >= 1).all() and fp[-1] == len(ex["ftiles"]) == st["n_ftiles"]
    ntile = np.diff(fp)[ex["fwd_order"]]
    assert (np.diff(ntile) <= 0).all()       # longest blocks first
    # pair count
    assert st["pairs"] == int((ohi - olo).sum()) == dag.count_pairs(ep.branches, ep.mounts, view=view)
    assert st["n_rows"] == N
    return plan, ex, st


def _slots(rec):
    """(piece, lo, hi, causal) of the 4 slots of a packed tile record."""
    out = []
    for k in range(4):
        w = int(rec[4 + k // 2]) >> (12 * (k % 2))
        out.append((int(rec[k]), w & 63, (w >> 6) & 63, bool((int(rec[6]) >> (1 + k)) & 1)))
    return out


def packed_marks(ex, b, r, N):
    """How often each key row is visible to row r through block b's packed tiles."""
    mark = np.zeros(N + 4 * 32, dtype=np.int32)
    for rec in ex["ftiles"][ex["fblk_ptr"][b]:ex["fblk_ptr"][b + 1]]:
        for p, lo, hi, causal in _slots(rec):
            if p < 0:
                assert lo == hi == 0
                continue
            assert 0 <= lo < hi <= 32
            a, z = 32 * p + lo, 32 * p + hi
            if causal:
                z = min(z, r + 1)
            mark[a:max(a, z)] += 1
    assert not mark[N:].any()
    return mark[:N]


def check_packed_flags(ex, page_size):
    for rec in ex["ftiles"]:
        sl = _slots(rec)
        need = any(p < 0 or lo != 0 or hi != 32 or c for p, lo, hi, c in sl)
        assert bool(rec[6] & 1) == need
        for h in range(2):
            if rec[6] & (32 << h):
                assert page_size >= 64 and rec[2 * h] % 2 == 0 and rec[2 * h + 1] == rec[2 * h] + 1
        assert rec[7] == 0 and (rec[6] & ~0x7F) == 0


def plan_block_rows(ep):
    return 256 // (ep.num_q_heads // ep.num_kv_heads)


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_full_configs(cfg):
    ep = W.config(cfg)
    rng = np.random.default_rng(cfg)
    rows = None if ep.n_rows < 50_000 else rng.choice(ep.n_rows, 3000, replace=False)
    check_plan_against_oracle(ep, rows)


@pytest.mark.parametrize("seed", range(60))
def test_random_small(seed):
    ep = W.random_small(seed, max_branches=8, max_len=300, n_mounts=int(seed % 4))
    check_plan_against_oracle(ep)


@pytest.mark.parametrize("seed", range(6))
def test_random_gqa_shapes(seed):
    heads = [(1, 1), (2, 1), (8, 1), (16, 1), (16, 2), (32, 8)][seed]
    ep = W.random_small(100 + seed, max_branches=6, max_len=400, heads=heads, head_dim=128,
                        page_size=[16, 32, 64, 128][seed % 4])
    check_plan_against_oracle(ep)


def test_crafted():
    from test_oracle_pins import crafted
    check_plan_against_oracle(crafted())


def test_wide_fan():
    check_plan_against_oracle(W.wide_fan())


@pytest.mark.parametrize("seed", range(6))
def test_zero_length_mounts_give_identical_plan(seed):
    ep = W.random_small(seed, max_len=200)
    rng = np.random.default_rng(seed)
    rows = [tuple(int(x) for x in m) for m in ep.mounts]
    for _ in range(5):
        r = int(rng.integers(0, len(ep.branches)))
        s = int(rng.integers(0, len(ep.branches)))
        b = int(rng.integers(0, int(ep.branches["length"][s]) + 1))
        rows.append((r, int(rng.integers(0, int(ep.branches["length"][r]))), s, b, b))
    rng.shuffle(rows)
    a = ta.tree_attn_plan_export(host_plan(ep))
    b = ta.tree_attn_plan_export(host_plan(ep, mounts=W.make_mounts(rows)))
    for k in a:
        assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k


def test_planner_matches_eq2_example():
    # the worked example after Octopus Eq. 2, through the library planner
    br = W.make_branches([-1, 0, 0], [0, 1500, 1500], [1500, 2501, 505])
    mt = W.make_mounts([(2, 500, 1, 0, 2501)])
    ep = W.Episode("eq2", br, mt, 4, 1, 64, 16)
    ex = ta.tree_attn_plan_export(host_plan(ep))
    b0 = int(br["row_start"][2])
    assert ex["pos_ids"][b0 + 499] == 1999 and ex["pos_ids"][b0 + 500] == 4001


def test_empty_dag():
    ep = W.Episode("empty", W.make_branches([], [], []), W.make_mounts([]), 4, 1, 64, 16)
    plan = host_plan(ep, page_table=np.zeros(0, np.int32))
    st = ta.tree_attn_plan_stats(plan)
    assert st["n_rows"] == 0 and st["n_blocks"] == 0 and st["pairs"] == 0
    assert st["n_fwd_items"] == 0 and st["n_fwd_split"] == 0
    # a forced split cap on an empty DAG: still no work items
    forced = host_plan(ep, page_table=np.zeros(0, np.int32), fwd_split_tiles=1)
    stf, exf = ta.tree_attn_plan_stats(forced), ta.tree_attn_plan_export(forced)
    assert stf["n_fwd_items"] == 0 and stf["n_fwd_split"] == 0
    assert exf["fwd_items"].shape == (0, 4) and exf["fwd_combine"].shape == (0, 4)


def _expect(code, ep, **kw):
    with pytest.raises(ta.TreeAttnError) as ei:
        host_plan(ep, **kw)
    assert ei.value.code == code, str(ei.value)


def _raw_branches(parents, forks, lens, starts=None):
    br = np.zeros(len(parents), dtype=W.BRANCH_DTYPE)
    br["parent"], br["fork_offset"], br["length"] = parents, forks, lens
    br["row_start"] = np.concatenate([[0], np.cumsum(lens)[:-1]]) if starts is None else starts
    return br


def test_rejects_invalid_dags():
    mk = _raw_branches
    base = W.tiny()
    E = lambda br, mt=None: W.Episode("x", br, W.make_mounts(mt or []), 4, 1, 64, 16)
    _expect(ta.TA_ERR_INVALID, E(mk([-1, 5], [0, 1], [10, 10])))                  # bad parent
    _expect(ta.TA_ERR_INVALID, E(mk([-1, 0], [0, 11], [10, 10])))                 # fork > parent length
    _expect(ta.TA_ERR_INVALID, E(mk([-1], [3], [10])))                            # root with a fork offset
    br = mk([1, 0], [4, 4], [10, 10])                                            # parent cycle
    _expect(ta.TA_ERR_INVALID, E(br))
    br = mk([-1, 0], [0, 4], [10, 10]); br["row_start"][1] = 8                     # overlapping rows
    _expect(ta.TA_ERR_INVALID, E(br))
    br = mk([-1, 0], [0, 4], [10, 10]); br["row_start"][1] = 12                    # gap
    _expect(ta.TA_ERR_INVALID, E(br))
    br = mk([-1, 0, 0], [0, 4, 4], [10, 10, 10])
    _expect(ta.TA_ERR_INVALID, E(br, [(1, 2, 2, 0, 11)]))                         # span beyond source
    _expect(ta.TA_ERR_INVALID, E(br, [(1, 10, 2, 0, 3)]))                         # offset beyond reader
    _expect(ta.TA_ERR_INVALID, E(br, [(1, 2, 7, 0, 3)]))                          # bad source index
    _expect(ta.TA_ERR_INVALID, E(br, [(1, 2, 1, 0, 5)]))                          # reads its own future
    br = mk([-1, 0, 1], [0, 4, 6], [10, 10, 10])
    _expect(ta.TA_ERR_INVALID, E(br, [(1, 3, 2, 0, 2)]))                          # reads a descendant forked after the mount
    _expect(ta.TA_ERR_INVALID, E(br, [(1, 3, 2, 0, 2)]))
    br = mk([-1, 0, 0], [0, 4, 4], [10, 10, 10])
    _expect(ta.TA_ERR_INVALID, E(br, [(1, 3, 2, 0, 5), (2, 2, 1, 0, 5)]))         # mutual mounts
    # a mount that only becomes non-causal through another mount (transitively)
    br = mk([-1, 0, 0, 0], [0, 4, 4, 4], [10, 10, 10, 10])
    _expect(ta.TA_ERR_INVALID, E(br, [(2, 1, 1, 0, 9), (3, 1, 2, 0, 5), (1, 2, 3, 0, 4)]))
    # short page table, duplicate page, page out of range
    n_log = -(-base.n_rows // base.page_size)
    _expect(ta.TA_ERR_INVALID, base, page_table=np.arange(n_log - 1, dtype=np.int32))
    pt = np.arange(n_log, dtype=np.int32); pt[3] = pt[4]
    _expect(ta.TA_ERR_INVALID, base, page_table=pt)
    pt = np.arange(n_log, dtype=np.int32); pt[3] = 10_000
    _expect(ta.TA_ERR_INVALID, base, page_table=pt)


def test_valid_edge_mounts_accepted():
    mk = W.make_branches
    E = lambda br, mt=None: W.Episode("x", br, W.make_mounts(mt or []), 4, 1, 64, 16)
    br = mk([-1, 0, 1], [0, 4, 6], [10, 10, 10])
    host_plan(E(br, [(1, 7, 2, 0, 2)]))            # reads a descendant forked before the mount
    host_plan(E(br, [(1, 5, 1, 0, 5)]))            # reads its own completed past
    br = mk([-1, 0, 0], [0, 10, 10], [10, 10, 10])
    host_plan(E(br, [(1, 3, 2, 0, 5), (2, 6, 1, 0, 3)]))  # mutual, but each span is complete


def test_clamp_flag():
    mk = W.make_branches
    br = mk([-1, 0, 0], [0, 4, 4], [10, 10, 10])
    ep = W.Episode("x", br, W.make_mounts([(1, 2, 2, 5, 40)]), 4, 1, 64, 16)
    _expect(ta.TA_ERR_INVALID, ep)
    a = ta.tree_attn_plan_export(host_plan(ep, flags=ta.TA_CLAMP_MOUNTS))
    ep2 = W.Episode("x", br, W.make_mounts([(1, 2, 2, 5, 10)]), 4, 1, 64, 16)
    b = ta.tree_attn_plan_export(host_plan(ep2))
    for k in a:
        assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k
    ep3 = W.Episode("x", br, W.make_mounts([(1, 2, 2, 20, 40)]), 4, 1, 64, 16)   # emptied by the clamp
    c = ta.tree_attn_plan_export(host_plan(ep3, flags=ta.TA_CLAMP_MOUNTS))
    d = ta.tree_attn_plan_export(host_plan(W.Episode("x", br, W.make_mounts([]), 4, 1, 64, 16)))
    for k in c:
        assert np.array_equal(np.asarray(c[k]), np.asarray(d[k])), k


def test_rejects_unsupported_shapes():
    ep = W.tiny()
    _expect(ta.TA_ERR_UNSUPPORTED, ep, head_dim=96)
    _expect(ta.TA_ERR_UNSUPPORTED, ep, page_size=8)
    _expect(ta.TA_ERR_UNSUPPORTED, ep, num_q_heads=6, num_kv_heads=4)
    _expect(ta.TA_ERR_UNSUPPORTED, ep, num_q_heads=96, num_kv_heads=3)


def test_fwd_rejects_host_only_plan():
    plan = host_plan(W.tiny())
    with pytest.raises(ta.TreeAttnError) as ei:
        ta.tree_attn_fwd(plan, 16, 16, 16, 16, 16, stream=0)
    assert ei.value.code == ta.TA_ERR_INVALID


# ------------------------------------------------------------------ the two other views
VIEW_FLAGS = [(ta.TA_NO_MOUNTS, "no_mounts"), (ta.TA_TRANSITIVE_MOUNTS, "transitive")]


@pytest.mark.parametrize("flags,view", VIEW_FLAGS, ids=[v for _, v in VIEW_FLAGS])
@pytest.mark.parametrize("cfg", [0, 2, 4])
def test_views_full_configs(cfg, flags, view):
    ep = W.config(cfg)
    rng = np.random.default_rng(100 + cfg)
    rows = None if ep.n_rows < 50_000 else rng.choice(ep.n_rows, 2000, replace=False)
    check_plan_against_oracle(ep, rows, flags=flags, view=view)


@pytest.mark.parametrize("flags,view", VIEW_FLAGS, ids=[v for _, v in VIEW_FLAGS])
@pytest.mark.parametrize("seed", range(24))
def test_views_random_small(seed, flags, view):
    ep = W.random_small(500 + seed, max_branches=10, max_len=200, n_mounts=1 + seed % 5)
    check_plan_against_oracle(ep, flags=flags, view=view)


def test_views_crafted_transitive_chain():
    from test_oracle_views import crafted
    br, mts = crafted()
    ep = W.Episode("crafted_views", br, mts, 4, 1, 64, 16, 0)
    for flags, view in [(0, "mounted")] + VIEW_FLAGS:
        check_plan_against_oracle(ep, flags=flags, view=view)


def test_views_exclusive():
    ep = W.tiny()
    with pytest.raises(ta.TreeAttnError):
        host_plan(ep, flags=ta.TA_NO_MOUNTS | ta.TA_TRANSITIVE_MOUNTS)


def test_no_mounts_plan_equals_mount_free_plan_except_positions():
    ep = W.scaled(4, 64)
    a = ta.tree_attn_plan_export(host_plan(ep, flags=ta.TA_NO_MOUNTS))
    b = ta.tree_attn_plan_export(host_plan(ep, mounts=ep.mounts[:0]))
    for key in ("blocks", "blk_iv_ptr", "iv_lo", "iv_hi", "diag", "entries", "t_entries", "chunks"):
        assert np.array_equal(a[key], b[key]), key
    assert np.array_equal(a["pos_ids"], dag.positions(ep.branches, ep.mounts))


def test_stream_ordered_flag_leaves_the_plan_unchanged():
    """TA_PLAN_STREAM_ORDERED changes only how the device copy is made: the host plan (every
    exported array and the stats) is the same as without it."""
    ep = W.scaled(2, 32)
    a = host_plan(ep)
    b = host_plan(ep, flags=ta.TA_PLAN_STREAM_ORDERED)
    ea, eb = ta.tree_attn_plan_export(a), ta.tree_attn_plan_export(b)
    assert ea.keys() == eb.keys()
    for k in ea:
        assert np.array_equal(np.asarray(ea[k]), np.asarray(eb[k])), k
    sa, sb = ta.tree_attn_plan_stats(a), ta.tree_attn_plan_stats(b)
    for k in sa:
        if k != "plan_ms":
            assert sa[k] == sb[k], k


def _chunk_lengths(ex):
    ch = ex["chunks"]
    return ch[:, 2] - ch[:, 1]


@pytest.mark.parametrize("make", [lambda: W.config(1), lambda: W.scaled(4, 8)], ids=["balanced", "mount_heavy/8"])
def test_chunk_cap_follows_sm_count(make):
    """Without an explicit cap, a key tile's readers are split into chunks of at most
    max(8, entries * Hkv / (4 * SMs)) entries: fewer SMs give longer chunks and fewer of them."""
    ep = make()
    counts = {}
    for sms in (38, 76, 152, 304):
        plan = host_plan(ep, num_sms=sms)
        st = ta.tree_attn_plan_stats(plan)
        ex = ta.tree_attn_plan_export(plan)
        cap = max(8, st["n_entries"] * ep.num_kv_heads // (4 * sms))
        assert st["chunk_cap"] == cap and st["num_sms"] == sms
        assert _chunk_lengths(ex).max() <= cap
        counts[sms] = st["n_chunks"]
    assert counts[38] <= counts[76] <= counts[152] <= counts[304]
    assert counts[38] < counts[304]
    # a host-only plan has no device: 152 SMs unless the config names a count
    st = ta.tree_attn_plan_stats(host_plan(ep))
    assert st["num_sms"] == 152 and st["device"] == -1


def test_chunk_cap_override_gives_unsplit_long_chunks():
    """dkdv_chunk_entries forces the chunk length: a large cap leaves every key tile unsplit
    (no partial slots); a cap of 1 splits every tile into single entries."""
    ep = W.wide_fan()
    big = host_plan(ep, dkdv_chunk_entries=1 << 20)
    st, ex = ta.tree_attn_plan_stats(big), ta.tree_attn_plan_export(big)
    assert st["n_partial_slots"] == 0 and st["chunk_cap"] == 1 << 20
    assert st["n_chunks"] == len(np.unique(ex["t_entries"][:, 1] // T))
    assert _chunk_lengths(ex).max() >= 200
    one = host_plan(ep, dkdv_chunk_entries=1)
    st1, ex1 = ta.tree_attn_plan_stats(one), ta.tree_attn_plan_export(one)
    assert (_chunk_lengths(ex1) == 1).all() and st1["n_chunks"] == st1["n_entries"]
    # the chunking changes nothing else in the plan
    for key in ("blocks", "entries", "t_entries"):
        assert np.array_equal(ex[key], ex1[key])


def _check_fwd_items(st, ex, cap):
    """The forward's work items cover each query block's packed tiles exactly once, in parts of
    at most `cap` tiles, longest first; split blocks' parts own consecutive partial slots."""
    items, comb, fblk = ex["fwd_items"], ex["fwd_combine"], ex["fblk_ptr"]
    nb = len(fblk) - 1
    assert st["n_fwd_items"] == len(items) and st["n_fwd_split"] == len(comb)
    lens = items[:, 2] - items[:, 1]
    assert (lens >= 1).all() and (lens <= cap).all()
    assert (np.diff(lens) <= 0).all()                        # longest first
    seen = np.zeros(int(fblk[-1]), dtype=np.int32)
    for b, a, z, slot in items:
        assert fblk[b] <= a < z <= fblk[b + 1]
        seen[a:z] += 1
    assert (seen == 1).all()
    split = {int(c[0]): c for c in comb}
    slots = []
    for b in range(nb):
        mine = items[items[:, 0] == b]
        if b in split:
            _, s0, parts, zero = split[b]
            assert zero == 0 and len(mine) == parts >= 2
            assert sorted(mine[:, 3].tolist()) == list(range(s0, s0 + parts))
            # slot order follows the tiles
            by_slot = mine[np.argsort(mine[:, 3])]
            assert (by_slot[1:, 1] == by_slot[:-1, 2]).all()
            slots += by_slot[:, 3].tolist()
        else:
            assert len(mine) == 1 and mine[0, 3] == -1
            assert (mine[0, 1], mine[0, 2]) == (fblk[b], fblk[b + 1])
    assert sorted(slots) == list(range(len(slots)))


@pytest.mark.parametrize("cap", [1, 3, 7])
def test_fwd_split_items_cover_every_tile_once(cap):
    """fwd_split_tiles forces split-KV: every block longer than the cap becomes parts of at most
    cap tiles, nothing is visited twice, and the rest of the plan is unchanged."""
    ep = W.Episode(name="chain", branches=W.make_branches([-1, 0, 0], [0, 700, 1500], [2048, 600, 900]),
                   mounts=W.make_mounts([]), num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=64)
    forced = host_plan(ep, fwd_split_tiles=cap)
    st, ex = ta.tree_attn_plan_stats(forced), ta.tree_attn_plan_export(forced)
    assert st["fwd_split_cap"] == cap
    _check_fwd_items(st, ex, cap)
    lens = np.diff(ex["fblk_ptr"])
    assert st["n_fwd_split"] == int((lens > cap).sum()) > 0
    assert st["n_fwd_items"] == int(np.where(lens > cap, -(-lens // cap), 1).sum())
    whole = host_plan(ep, fwd_split_tiles=-1)
    stw, exw = ta.tree_attn_plan_stats(whole), ta.tree_attn_plan_export(whole)
    assert stw["n_fwd_split"] == 0 and stw["n_fwd_items"] == len(lens)
    _check_fwd_items(stw, exw, int(lens.max()))
    for key in ("blocks", "entries", "t_entries", "chunks", "ftiles", "fblk_ptr", "fwd_order"):
        assert np.array_equal(ex[key], exw[key]), key


def test_fwd_split_auto_only_when_the_longest_block_dominates():
    """The automatic cap splits only when the longest block exceeds 1.5x one worker's share of
    the tile work and by at least 32 tiles (workers: SMs for head dim 64, SM pairs for 128),
    into parts of at most max(16, share) tiles; otherwise it keeps every block whole."""
    def chain(n, d, heads):
        return W.Episode(name="chain", branches=W.make_branches([-1], [0], [n]), mounts=W.make_mounts([]),
                         num_q_heads=heads[0], num_kv_heads=heads[1], head_dim=d, page_size=64)

    ep = W.wide_fan()
    st = ta.tree_attn_plan_stats(host_plan(ep, num_sms=152))
    assert st["n_fwd_split"] == 0 and st["n_fwd_items"] == st["n_blocks"]
    cases = [(8192, 64, (4, 1), True), (16384, 128, (1, 1), True), (4096, 128, (4, 1), False),
             (16384, 128, (4, 1), False), (8192, 128, (16, 4), False)]
    for n, d, heads, splits in cases:
        p = host_plan(chain(n, d, heads), num_sms=152)
        st, ex = ta.tree_attn_plan_stats(p), ta.tree_attn_plan_export(p)
        lens = np.diff(ex["fblk_ptr"])
        workers = 152 if d == 64 else 76
        share = -(-int(lens.sum()) * heads[1] // workers)
        assert (2 * lens.max() > 3 * share and lens.max() - share >= 32) == splits, (n, d, heads)
        if splits:
            assert st["fwd_split_cap"] == max(16, share) and st["n_fwd_split"] > 0
        else:
            assert st["fwd_split_cap"] == lens.max() and st["n_fwd_split"] == 0
        _check_fwd_items(st, ex, st["fwd_split_cap"])
