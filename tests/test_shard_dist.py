"""Per-DAG sharding of a global batch over data-parallel ranks (gloo, CPU, world size 2 and 4).

The independent DAGs of `world` episodes are placed on the ranks by the replica assignment of
HARTS Section 3.2 (bench.rank_episode): every DAG lands on exactly one rank, the load imbalance
is reported, and each rank's plan equals the single-rank plan of the whole batch restricted to
the rank's DAGs -- bit for bit, rows shifted -- so no rank needs another rank's rows and the
attention has no collective."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _host_plan(ep):
    import dag_packed_paged_gb300 as ta
    n_logical = -(-ep.n_rows // ep.page_size)
    pt = np.arange(n_logical, dtype=np.int32)
    plan = ta.tree_attn_plan(ep.branches, ep.mounts, pt, num_q_heads=ep.num_q_heads, num_kv_heads=ep.num_kv_heads,
                             head_dim=ep.head_dim, page_size=ep.page_size, num_pages=n_logical,
                             flags=ta.TA_PLAN_HOST_ONLY)
    return ta.tree_attn_plan_export(plan)


def _dag_slices(ex, row_ranges):
    """Per DAG (given its row range in the strip), the plan arrays of its blocks, rows made
    relative to the DAG's first row."""
    out = []
    b = ex["blocks"]
    for lo, hi in row_ranges:
        sel = np.nonzero((b[:, 0] >= lo) & (b[:, 0] < hi))[0]
        ivp = ex["blk_iv_ptr"]
        ivs = [(ex["iv_lo"][ivp[i]:ivp[i + 1]] - lo).tolist() + (ex["iv_hi"][ivp[i]:ivp[i + 1]] - lo).tolist()
               for i in sel]
        ents = [ex["entries"][b[i, 2]:b[i, 3]].copy() for i in sel]
        for e in ents:
            e[:, 0] -= lo // 128
            e[:, 1:3] -= lo
        fts = []
        for i in sel:
            f = ex["ftiles"][ex["fblk_ptr"][i]:ex["fblk_ptr"][i + 1]].copy()
            f[:, :4] = np.where(f[:, :4] >= 0, f[:, :4] - lo // 32, -1)
            fts.append(f)
        out.append({"pos": ex["pos_ids"][lo:hi].tolist(), "rows": (b[sel, :2] - [lo, 0]).tolist(),
                    "diag": (ex["diag"][sel] - lo).tolist(), "ivs": ivs,
                    "entries": [e.tolist() for e in ents], "ftiles": [f.tolist() for f in fts]})
    return out


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import bench
    from dag_packed_paged_gb300 import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        make = lambda: W.scaled(4, 16)
        ep, info, mine = bench.rank_episode(make, world, rank)
        taken = [None] * world
        dist.all_gather_object(taken, mine)
        # the single-rank plan of the whole batch, and this rank's own plan
        units = []
        for s in range(world):
            e = make()
            e.seed = s
            units += W.split_dags(e)
        whole = W.concat_episodes(units)
        starts = np.cumsum([0] + [u.n_rows for u in units])
        full = _dag_slices(_host_plan(whole), [(starts[i], starts[i + 1]) for i in mine])
        lstarts = np.cumsum([0] + [units[i].n_rows for i in mine])
        local = _dag_slices(_host_plan(ep), [(lstarts[k], lstarts[k + 1]) for k in range(len(mine))])
        out.put((rank, taken, info, full == local, all(s % 128 == 0 for s in lstarts), len(mine)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_dags_placed_once_and_plans_restrict(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    taken = res[0][1]
    assert all(r[1] == taken for r in res)                       # every rank sees the same placement
    flat = sorted(i for t in taken for i in t)
    assert flat == list(range(4 * world))                        # every DAG exactly once
    for rank, _, info, same, aligned, n in res:
        assert same and aligned, rank                            # bit-exact restriction of the full plan
        assert n == 4 and info["dags_per_rank"] == [4] * world and info["imbalance"] == 1.0


def test_one_rank_is_the_episode():
    import bench
    from dag_packed_paged_gb300 import workloads as W
    ep, info, mine = bench.rank_episode(lambda: W.config(4), 1, 0)
    ref = W.config(4)
    assert np.array_equal(ep.branches, ref.branches) and np.array_equal(ep.mounts, ref.mounts)
    assert ep.seed == ref.seed and mine == [0, 1, 2, 3] and info["dags"] == 4


def test_uneven_dags_balance():
    """Episodes of one DAG each with different sizes: the heaviest rank is the LPT bound."""
    import bench
    from dag_packed_paged_gb300 import workloads as W
    sizes = []
    for r in range(3):
        ep, info, mine = bench.rank_episode(lambda: W.scaled(2, 8), 3, r)
        sizes.append(ep.n_rows)
    assert max(sizes) == info["max_rank_rows"] and info["dags"] == 3
