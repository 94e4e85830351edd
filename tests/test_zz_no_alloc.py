"""tree_attn_bwd_noalloc: the backward for callers that cannot hand the library device
scratch (plugin hosts that pass only input and output buffers; loops that forbid device
allocation while running).  Its output must match tree_attn_bwd's, call after call, although
every call reuses the library's fixed scratch array.  This file is collected last so that a
run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [W.tiny, lambda: W.scaled(1, 16), lambda: W.scaled(4, 64)],
                         ids=["tiny", "balanced/16", "mount_heavy/64"])
def test_noalloc_matches_workspace_backward_twice(make):
    ep = make()
    run = Run(ep, dist="realistic")
    run.fwd()
    dq_ref, dk_ref, dv_ref = run.bwd()                 # tree_attn_bwd with a caller workspace
    pt = run.pool.page_table
    for _ in range(2):                                 # two calls in a row share the scratch
        dq = torch.full_like(run.dq, float("nan"))
        dk_pool = torch.zeros_like(run.dk_pool)
        dv_pool = torch.zeros_like(run.dv_pool)
        ta.tree_attn_bwd_noalloc(run.plan, run.q, run.k_pool, run.v_pool, run.o, run.lse, run.d_o,
                                 dq, dk_pool, dv_pool)
        ta.tree_attn_check(run.plan)
        dk = W.pool_rows(dk_pool.cpu().numpy(), pt, ep.n_rows).astype(np.float64)
        dv = W.pool_rows(dv_pool.cpu().numpy(), pt, ep.n_rows).astype(np.float64)
        assert_close("dQ", dq.cpu().numpy().astype(np.float64), dq_ref)
        assert_close("dK", dk, dk_ref)
        assert_close("dV", dv, dv_ref)


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
