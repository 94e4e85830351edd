"""A whole multi-layer step in one CUDA graph.  One plan drives every mounted layer's launches
(Octopus Section 3.2: the mounted layers share the episode's DAG, positions and page table; only
Q, K, V and dO differ per layer).  The library's launches take plain stream arguments and do no
host synchronisation, so the forward and backward of all layers can be captured once and replayed
with a single graph launch: the GPU-side form of "one launch for all mounted layers sharing one
plan".  Replays must reproduce the eager results bit for bit (every kernel is deterministic)."""
import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import bf16_tensor

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [lambda: W.scaled(2, 32), lambda: W.tiny()], ids=["commander/32 D128", "tiny D64"])
def test_multi_layer_step_in_one_graph(make):
    ep = make()
    dev = torch.device("cuda:0")
    N, Hq, D = ep.n_rows, ep.num_q_heads, ep.head_dim
    layers = []
    for layer in range(3):
        t = W.make_tensors(ep, seed=200 + layer, dist="realistic")
        pool = W.make_pool(ep, t)
        ins = [bf16_tensor(a, dev) for a in (t.q, pool.k_pool, pool.v_pool, t.do)]
        outs = [torch.empty((N, Hq, D), dtype=torch.bfloat16, device=dev),
                torch.empty((Hq, N), dtype=torch.float32, device=dev),
                torch.empty((N, Hq, D), dtype=torch.float32, device=dev),
                torch.zeros(pool.k_pool.shape, dtype=torch.float32, device=dev),
                torch.zeros(pool.v_pool.shape, dtype=torch.float32, device=dev)]
        layers.append((ins, outs))
    plan = ta.tree_attn_plan(ep.branches, ep.mounts, pool.page_table, num_q_heads=Hq, num_kv_heads=ep.num_kv_heads,
                             head_dim=D, page_size=ep.page_size, num_pages=pool.k_pool.shape[0])
    ws = torch.empty(max(ta.tree_attn_bwd_workspace_size(plan), 256), dtype=torch.uint8, device=dev)

    def step():
        for (q, k, v, d_o), (o, lse, dq, dk, dv) in layers:
            ta.tree_attn_fwd(plan, q, k, v, o, lse)
            ta.tree_attn_bwd(plan, q, k, v, o, lse, d_o, dq, dk, dv, ws)

    step()                                          # eager
    torch.cuda.synchronize()
    ta.tree_attn_check(plan)
    eager = [[x.clone() for x in outs] for _, outs in layers]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for _, outs in layers:                      # replays must write every output again
            for x in outs:
                x.fill_(float("nan") if x.dtype != torch.float32 or x.dim() != 4 else 0.0)
        g.replay()
        torch.cuda.synchronize()
        ta.tree_attn_check(plan)
        for li, (_, outs) in enumerate(layers):
            for name, a, b in zip(("O", "lse", "dQ", "dK", "dV"), outs, eager[li]):
                assert torch.equal(a.view(torch.int8 if a.dtype == torch.bfloat16 else torch.int32),
                                   b.view(torch.int8 if b.dtype == torch.bfloat16 else torch.int32)), \
                    f"layer {li} {name} differs after replay"
