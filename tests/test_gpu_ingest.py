"""End to end on the GPU from raw trajectories: ingest (HARTS Eq. 3 / Eq. 5) -> plan ->
forward and backward through the C ABI, against the fp64 oracle on the ingested episode."""
import numpy as np
import pytest

import dag_packed_paged_gb300 as ta
import oracle
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close, metrics
from test_ingest import random_trajectories

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", [0, 1])
def test_ingested_episode_fwd_bwd(seed):
    trajs = [np.concatenate([t, t, t, t]) for t in random_trajectories(seed, n=16, max_len=120)]
    br, _, _ = ta.tree_attn_ingest(trajs)
    ep = W.Episode(f"ingested{seed}", br, np.zeros(0, dtype=W.MOUNT_DTYPE), 16, 4, 128, 64, seed)
    run = Run(ep, dist="realistic")
    o, lse = run.fwd()
    dq, dk, dv = run.bwd()
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    assert_close("O", o, ref.o)
    assert metrics(lse, ref.lse)[0] <= 2e-3
    assert_close("dQ", dq, ref.dq)
    assert_close("dK", dk, ref.dk)
    assert_close("dV", dv, ref.dv)
