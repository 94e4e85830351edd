"""Split-KV forward on the GPU: a query block whose packed-tile list is cut into parts (each a
work item writing a partial O and lse, merged by the combine kernel) gives the oracle's O and
lse, and the backward that reads them the oracle's gradients -- on both forwards (head dim 64,
the single-SM kernel; 128, the CTA pair), with forced caps down to one tile per part and with
the automatic cap on chains whose longest block dominates the forward."""
import numpy as np
import pytest

import oracle
import dag_packed_paged_gb300 as ta
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close, metrics

pytestmark = pytest.mark.gpu


def _check(run, ep, bwd=True):
    o, lse = run.fwd()
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    assert_close("O", o, ref.o)
    assert metrics(lse, ref.lse)[0] <= 2e-3
    if bwd:
        dq, dk, dv = run.bwd()
        assert_close("dQ", dq, ref.dq)
        assert_close("dK", dk, ref.dk)
        assert_close("dV", dv, ref.dv)
    return o, lse


def _chain(n_rows, head_dim, heads=(4, 1), page=64):
    return W.Episode(name=f"chain{n_rows}", branches=W.make_branches([-1], [0], [n_rows]),
                     mounts=W.make_mounts([]), num_q_heads=heads[0], num_kv_heads=heads[1],
                     head_dim=head_dim, page_size=page)


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("cap", [1, 2, 5])
def test_forced_split_matches_oracle(head_dim, cap):
    ep = W.random_small(4100 + cap + head_dim, max_branches=8, max_len=900, heads=(8, 2), head_dim=head_dim,
                        page_size=64, n_mounts=3)
    run = Run(ep, dist="realistic", fwd_split_tiles=cap)
    st = ta.tree_attn_plan_stats(run.plan)
    assert st["n_fwd_split"] > 0 and st["fwd_split_cap"] == cap
    o, lse = _check(run, ep)
    # the same inputs unsplit: the parts' merge moves O by rounding only
    whole = Run(ep, tensors=run.t, pool=run.pool, fwd_split_tiles=-1)
    assert ta.tree_attn_plan_stats(whole.plan)["n_fwd_split"] == 0
    o1, lse1 = whole.fwd()
    assert np.abs(lse - lse1).max() <= 1e-4
    assert np.abs(o - o1).max() <= 1.6e-2 * max(1.0, np.abs(o1).max())


@pytest.mark.parametrize("n,head_dim,heads", [(8192, 64, (4, 1)), (16384, 128, (1, 1))])
def test_auto_split_on_a_short_chain(n, head_dim, heads):
    """A single causal chain with few query blocks x KV heads against the workers: its longest
    block is well above a worker's share, so the automatic cap splits the longer blocks."""
    ep = _chain(n, head_dim, heads)
    run = Run(ep, dist="realistic")
    st = ta.tree_attn_plan_stats(run.plan)
    assert st["n_fwd_split"] > 0
    o, lse = run.fwd()
    ref = oracle.forward(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, ep.softmax_scale)
    assert_close("O", o, ref.o)
    assert metrics(lse, ref.lse)[0] <= 2e-3


@pytest.mark.parametrize("page", [16, 32])
def test_forced_split_small_pages(page):
    """Parts of blocks on 16- and 32-row pages (several TMA boxes per packed slot)."""
    ep = W.random_small(4200 + page, max_branches=6, max_len=600, heads=(4, 1), head_dim=128, page_size=page,
                        n_mounts=2)
    run = Run(ep, dist="sharp", fwd_split_tiles=2)
    assert ta.tree_attn_plan_stats(run.plan)["n_fwd_split"] > 0
    _check(run, ep, bwd=False)


def test_split_forward_in_a_graph_and_stream_ordered():
    """A plan with split blocks: the forward (work items and combine) captured in a CUDA graph
    replays bit-identically, and a stream-ordered plan (its partial buffer allocated in stream
    order) gives the same O and lse as the ordinary plan, bit for bit."""
    import torch
    ep = W.random_small(4300, max_branches=8, max_len=900, heads=(8, 2), head_dim=128, page_size=64, n_mounts=3)
    run = Run(ep, dist="realistic", fwd_split_tiles=2)
    assert ta.tree_attn_plan_stats(run.plan)["n_fwd_split"] > 0
    o, lse = run.fwd()
    eager_o, eager_lse = run.o.clone(), run.lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ta.tree_attn_fwd(run.plan, run.q, run.k_pool, run.v_pool, run.o, run.lse)
    for _ in range(2):
        run.o.fill_(float("nan"))
        run.lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        ta.tree_attn_check(run.plan)
        assert torch.equal(run.o.view(torch.int16), eager_o.view(torch.int16))
        assert torch.equal(run.lse.view(torch.int32), eager_lse.view(torch.int32))
    so = Run(ep, tensors=run.t, pool=run.pool, flags=ta.TA_PLAN_STREAM_ORDERED, fwd_split_tiles=2)
    o2, lse2 = so.fwd()
    assert np.array_equal(o2, o) and np.array_equal(lse2, lse)
