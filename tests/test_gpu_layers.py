"""One plan serves every mounted attention layer of a model step (Octopus Section 3.2: the
mounted layers share the episode's DAG, positions and page table; only Q, K, V and dO differ
per layer).  Layers run as successive launches on the same plan, since each layer's inputs
come from the previous layer's output.  Each layer's forward and backward must match the
oracle run on that layer's own tensors."""
import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
import oracle
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import as_f64, assert_close, bf16_tensor, metrics

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("flags", [0, ta.TA_NO_MOUNTS], ids=["mounted", "mount_free"])
def test_one_plan_many_layers(flags):
    ep = W.scaled(2, 32)
    dev = torch.device("cuda:0")
    N, Hq, D = ep.n_rows, ep.num_q_heads, ep.head_dim
    pool0 = W.make_pool(ep, W.make_tensors(ep, seed=100))
    plan = ta.tree_attn_plan(ep.branches, ep.mounts, pool0.page_table, num_q_heads=Hq,
                             num_kv_heads=ep.num_kv_heads, head_dim=D, page_size=ep.page_size,
                             num_pages=pool0.k_pool.shape[0], flags=flags)
    ws = torch.empty(max(ta.tree_attn_bwd_workspace_size(plan), 256), dtype=torch.uint8, device=dev)
    view = "no_mounts" if flags & ta.TA_NO_MOUNTS else "mounted"
    for layer in range(3):
        t = W.make_tensors(ep, seed=100 + layer, dist="realistic")
        pool = W.make_pool(ep, t)
        assert np.array_equal(pool.page_table, pool0.page_table)     # same pages, new contents
        q, k_pool, v_pool, d_o = (bf16_tensor(a, dev) for a in (t.q, pool.k_pool, pool.v_pool, t.do))
        o = torch.empty((N, Hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((Hq, N), dtype=torch.float32, device=dev)
        dq = torch.empty((N, Hq, D), dtype=torch.float32, device=dev)
        dk = torch.zeros(pool.k_pool.shape, dtype=torch.float32, device=dev)
        dv = torch.zeros(pool.v_pool.shape, dtype=torch.float32, device=dev)
        ta.tree_attn_fwd(plan, q, k_pool, v_pool, o, lse)
        ta.tree_attn_bwd(plan, q, k_pool, v_pool, o, lse, d_o, dq, dk, dv, ws)
        ta.tree_attn_check(plan)
        ref = oracle.run(ep.branches, ep.mounts, t.q, t.k, t.v, t.do, ep.softmax_scale, view=view)
        assert_close(f"O[{layer}]", as_f64(o), ref.o)
        assert metrics(as_f64(lse).T, ref.lse)[0] <= 2e-3
        assert_close(f"dQ[{layer}]", dq.cpu().numpy().astype(np.float64), ref.dq)
        assert_close(f"dK[{layer}]", W.pool_rows(dk.cpu().numpy(), pool.page_table, N).astype(np.float64), ref.dk)
        assert_close(f"dV[{layer}]", W.pool_rows(dv.cpu().numpy(), pool.page_table, N).astype(np.float64), ref.dv)
