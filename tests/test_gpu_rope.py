"""RoPE of Q and the K pool at the plan's Eq. 2 positions, through the C ABI, against the fp64
oracle (oracle/rope.py); spare pool pages and V must stay bit-identical."""
import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, as_f64, assert_close
from oracle.rope import rope

pytestmark = pytest.mark.gpu


def _long_root(n=262_144):
    """One 262,144-row root: positions up to 2^18, where an fp32 angle would be ~1e-2 rad off."""
    return W.Episode("long_root", W.make_branches([-1], [0], [n]), np.zeros(0, dtype=W.MOUNT_DTYPE),
                     4, 1, 64, 64, 0)


CASES = [("tiny", W.tiny, 10000.0), ("commander/32", lambda: W.scaled(2, 32), 1e6),
         ("mount_heavy/64", lambda: W.scaled(4, 64), 10000.0),
         ("random_d64_p16", lambda: W.random_small(77, heads=(16, 2), head_dim=64, page_size=16, n_mounts=2), 5e5),
         ("long_root", _long_root, 10000.0), ("mount_heavy", lambda: W.config(4), 1e6)]


@pytest.mark.parametrize("name,make,base", CASES, ids=[c[0] for c in CASES])
def test_rope_matches_oracle(name, make, base):
    ep = make()
    run = Run(ep)
    k_before = run.k_pool.clone()
    v_before = run.v_pool.clone()
    ta.tree_attn_rope(run.plan, run.q, run.k_pool, base)
    torch.cuda.synchronize()
    N = ep.n_rows
    pos = run.plan.pos_ids
    rows = np.arange(N) if N <= 20_000 else np.unique(np.concatenate(
        [np.random.default_rng(1).choice(N, 4000, replace=False), [0, N - 1]]))
    q0 = W.bf16_bits_to_f32(run.t.q[rows]).astype(np.float64)
    assert_close("Q", as_f64(run.q)[rows], rope(q0, pos[rows], base), max_abs=2e-2, rel_rms=5e-3)
    pt = run.pool.page_table
    k_all = W.pool_rows(run.k_pool.float().cpu().numpy(), pt, N)
    k0 = W.pool_rows(W.bf16_bits_to_f32(run.pool.k_pool), pt, N)
    assert_close("K", k_all[rows].astype(np.float64), rope(k0[rows].astype(np.float64), pos[rows], base),
                 max_abs=2e-2, rel_rms=5e-3)
    spare = np.setdiff1d(np.arange(run.k_pool.shape[0]), pt)
    assert torch.equal(run.k_pool[spare].view(torch.int16), k_before[spare].view(torch.int16))
    assert torch.equal(run.v_pool.view(torch.int16), v_before.view(torch.int16))


def test_rope_rejects_bad_base():
    ep = W.tiny()
    run = Run(ep)
    with pytest.raises(ta.TreeAttnError):
        ta.tree_attn_rope(run.plan, run.q, run.k_pool, 0.5)
