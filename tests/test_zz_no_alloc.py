"""tree_attn_bwd_noalloc: the backward for callers that cannot hand the library device
scratch (plugin hosts that pass only input and output buffers; loops that forbid device
allocation while running).  Its output must match the oracle and tree_attn_bwd's, call after
call, although every call reuses the library's fixed scratch array.  This file is collected
last so that a run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
import oracle
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close

pytestmark = pytest.mark.gpu


def _noalloc(run):
    dq = torch.full_like(run.dq, float("nan"))
    dk_pool = torch.zeros_like(run.dk_pool)
    dv_pool = torch.zeros_like(run.dv_pool)
    ta.tree_attn_bwd_noalloc(run.plan, run.q, run.k_pool, run.v_pool, run.o, run.lse, run.d_o,
                             dq, dk_pool, dv_pool)
    ta.tree_attn_check(run.plan)
    pt, n = run.pool.page_table, run.ep.n_rows
    dk = W.pool_rows(dk_pool.cpu().numpy(), pt, n).astype(np.float64)
    dv = W.pool_rows(dv_pool.cpu().numpy(), pt, n).astype(np.float64)
    return dq.cpu().numpy().astype(np.float64), dk, dv


@pytest.mark.parametrize("make", [W.tiny, lambda: W.scaled(1, 16), lambda: W.scaled(4, 64)],
                         ids=["tiny", "balanced/16", "mount_heavy/64"])
def test_noalloc_matches_oracle_and_workspace_backward_twice(make):
    ep = make()
    run = Run(ep, dist="realistic")
    run.fwd()
    ws_ref = run.bwd()                                 # tree_attn_bwd with a caller workspace
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    for _ in range(2):                                 # two calls in a row share the scratch
        got = _noalloc(run)
        for name, g, w, o in zip(("dQ", "dK", "dV"), got, ws_ref, (ref.dq, ref.dk, ref.dv)):
            assert_close(name + " vs oracle", g, o)
            assert_close(name + " vs tree_attn_bwd", g, w)


def test_noalloc_full_balanced_tree():
    """The full balanced tree needs 56.5 MiB of the 64 MiB scratch, the most of the five
    workloads: every element against tree_attn_bwd, and the oracle on sampled query rows (dQ)
    and on key rows whose readers it can recompute (dK, dV)."""
    from test_gpu_bwd import _cheap_key_rows
    ep = W.config(1)
    run = Run(ep)
    assert ta.tree_attn_bwd_workspace_size(run.plan) > (48 << 20)
    run.fwd()
    ws_ref = run.bwd()
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([rng.choice(ep.n_rows, 24, replace=False), [0, ep.n_rows - 1]]))
    f = oracle.forward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, ep.softmax_scale, rows=rows)
    b = oracle.backward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale, f,
                        with_dkdv=False)
    cols, rd = _cheap_key_rows(ep, n=16)
    f2 = oracle.forward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, ep.softmax_scale, rows=rd)
    b2 = oracle.backward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale, f2)
    for _ in range(2):
        dq, dk, dv = _noalloc(run)
        for name, g, w in zip(("dQ", "dK", "dV"), (dq, dk, dv), ws_ref):
            assert_close(name + " vs tree_attn_bwd", g, w)
        assert_close("dQ vs oracle", dq[rows], b.dq)
        assert_close("dK vs oracle", dk[cols], b2.dk[cols])
        assert_close("dV vs oracle", dv[cols], b2.dv[cols])


def test_noalloc_rejects_plans_beyond_its_scratch():
    # 2,097,152 rows x 16 query heads need 128 MiB of delta alone: more than the 64 MiB held
    n = 4096
    br = W.make_branches([-1] * n, [0] * n, [512] * n)
    pt = np.arange(n * 512 // 64, dtype=np.int32)
    plan = ta.tree_attn_plan(br, W.make_mounts([]), pt, num_q_heads=16, num_kv_heads=4, head_dim=128,
                             page_size=64, num_pages=len(pt), flags=ta.TA_PLAN_HOST_ONLY)
    assert ta.tree_attn_bwd_workspace_size(plan) > (64 << 20)
    with pytest.raises(ta.TreeAttnError) as ei:
        ta.tree_attn_bwd_noalloc(plan, 256, 256, 256, 256, 256, 256, 256, 256, 256, stream=0)
    assert ei.value.code == ta.TA_ERR_UNSUPPORTED
    assert "bytes of backward scratch" in str(ei.value)
