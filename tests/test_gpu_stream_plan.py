"""TA_PLAN_STREAM_ORDERED: a plan allocated, uploaded and freed in the order of one stream
(no host synchronisation).  Results on that stream, or on another stream ordered after it by
an event, must match the oracle, and freeing a plan in stream order must not disturb work
enqueued before the free or a plan built after it."""
import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
import oracle
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import as_f64, assert_close, bf16_tensor, metrics

pytestmark = pytest.mark.gpu


def _setup(ep, dev):
    t = W.make_tensors(ep, dist="realistic")
    pool = W.make_pool(ep, t)
    ins = [bf16_tensor(a, dev) for a in (t.q, pool.k_pool, pool.v_pool, t.do)]
    torch.cuda.synchronize(dev)
    return t, pool, ins


def _plan(ep, pool, stream):
    return ta.tree_attn_plan(ep.branches, ep.mounts, pool.page_table, num_q_heads=ep.num_q_heads,
                             num_kv_heads=ep.num_kv_heads, head_dim=ep.head_dim, page_size=ep.page_size,
                             num_pages=pool.k_pool.shape[0], flags=ta.TA_PLAN_STREAM_ORDERED, stream=stream)


def _outputs(ep, pool, dev):
    N, Hq, D = ep.n_rows, ep.num_q_heads, ep.head_dim
    o = torch.empty((N, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, N), dtype=torch.float32, device=dev)
    dq = torch.empty((N, Hq, D), dtype=torch.float32, device=dev)
    dk = torch.zeros(pool.k_pool.shape, dtype=torch.float32, device=dev)
    dv = torch.zeros(pool.v_pool.shape, dtype=torch.float32, device=dev)
    return o, lse, dq, dk, dv


def _check(ep, t, pool, o, lse, dq, dk_pool, dv_pool):
    ref = oracle.run(ep.branches, ep.mounts, t.q, t.k, t.v, t.do, ep.softmax_scale)
    N = ep.n_rows
    assert_close("O", as_f64(o), ref.o)
    assert metrics(as_f64(lse).T, ref.lse)[0] <= 2e-3
    assert_close("dQ", dq.cpu().numpy().astype(np.float64), ref.dq)
    assert_close("dK", W.pool_rows(dk_pool.cpu().numpy(), pool.page_table, N).astype(np.float64), ref.dk)
    assert_close("dV", W.pool_rows(dv_pool.cpu().numpy(), pool.page_table, N).astype(np.float64), ref.dv)


@pytest.mark.parametrize("make", [W.tiny, lambda: W.scaled(4, 64)], ids=["tiny", "mount_heavy/64"])
@pytest.mark.parametrize("other_stream", [False, True], ids=["same_stream", "event_ordered_stream"])
def test_stream_ordered_plan_matches_oracle(make, other_stream):
    ep = make()
    dev = torch.device("cuda:0")
    t, pool, (q, k_pool, v_pool, d_o) = _setup(ep, dev)
    s = torch.cuda.Stream(dev)
    plan = _plan(ep, pool, s)
    run_s = s
    if other_stream:
        ready = torch.cuda.Event()
        ready.record(s)
        run_s = torch.cuda.Stream(dev)
        run_s.wait_event(ready)
    o, lse, dq, dk, dv = _outputs(ep, pool, dev)
    torch.cuda.synchronize(dev)
    ws = torch.empty(max(ta.tree_attn_bwd_workspace_size(plan), 256), dtype=torch.uint8, device=dev)
    ta.tree_attn_fwd(plan, q, k_pool, v_pool, o, lse, stream=run_s)
    ta.tree_attn_bwd(plan, q, k_pool, v_pool, o, lse, d_o, dq, dk, dv, ws, stream=run_s)
    ta.tree_attn_check(plan, run_s)
    torch.cuda.synchronize(dev)
    _check(ep, t, pool, o, lse, dq, dk, dv)


def test_plan_freed_in_stream_order_then_rebuilt():
    ep = W.scaled(2, 32)
    dev = torch.device("cuda:0")
    t, pool, (q, k_pool, v_pool, d_o) = _setup(ep, dev)
    s = torch.cuda.Stream(dev)
    outs = [_outputs(ep, pool, dev) for _ in range(3)]
    torch.cuda.synchronize(dev)
    ws = None
    for i in range(3):            # each plan is freed (in s order) right after its launches
        plan = _plan(ep, pool, s)
        if ws is None:
            ws = torch.empty(max(ta.tree_attn_bwd_workspace_size(plan), 256), dtype=torch.uint8, device=dev)
        o, lse, dq, dk, dv = outs[i]
        ta.tree_attn_fwd(plan, q, k_pool, v_pool, o, lse, stream=s)
        ta.tree_attn_bwd(plan, q, k_pool, v_pool, o, lse, d_o, dq, dk, dv, ws, stream=s)
        if i == 2:
            ta.tree_attn_check(plan, s)
        del plan
    torch.cuda.synchronize(dev)
    _check(ep, t, pool, *outs[0])
    for i in (1, 2):              # identical inputs: identical (deterministic) outputs
        for a, b in zip(outs[0], outs[i]):
            assert torch.equal(a, b)
