"""The bounded-wait error path.  Every pipelined kernel waits on mbarriers with a time limit;
when one runs out the kernel records a status bit and returns, and tree_attn_check reports
TA_ERR_DEVICE_TIMEOUT.  tree_attn_selftest_timeout makes such a wait run out on purpose (one
thread, a barrier nothing arrives on, a short limit), so the path is exercised without any
fault: afterwards the status must read as a timeout, be cleared by the check, and leave the
context able to run an ordinary forward that still matches the oracle."""
import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
import oracle
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, assert_close


def _host_plan():
    ep = W.tiny()
    pt = np.arange(64, dtype=np.int32)
    return ta.tree_attn_plan(ep.branches, ep.mounts, pt, num_q_heads=ep.num_q_heads,
                             num_kv_heads=ep.num_kv_heads, head_dim=ep.head_dim, page_size=ep.page_size,
                             num_pages=len(pt), flags=ta.TA_PLAN_HOST_ONLY)


@pytest.mark.parametrize("limit_us", [0, 99, 1_000_001])
def test_selftest_rejects_limits_out_of_range(limit_us):
    plan = _host_plan()
    with pytest.raises(ta.TreeAttnError) as ei:
        ta.tree_attn_selftest_timeout(plan, limit_us, stream=0)
    assert ei.value.code == ta.TA_ERR_INVALID
    assert "limit_us" in str(ei.value)


def test_selftest_rejects_host_only_plans():
    plan = _host_plan()
    with pytest.raises(ta.TreeAttnError) as ei:
        ta.tree_attn_selftest_timeout(plan, 1000, stream=0)
    assert ei.value.code == ta.TA_ERR_INVALID


@pytest.mark.gpu
@pytest.mark.parametrize("limit_us", [200, 5000])
def test_expired_wait_is_reported_cleared_and_survivable(limit_us):
    ep = W.tiny()
    run = Run(ep, dist="realistic")
    o0, lse0 = run.fwd()                                   # status clean before the self-test
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    start.record(stream)
    ta.tree_attn_selftest_timeout(run.plan, limit_us)
    end.record(stream)
    with pytest.raises(ta.TreeAttnError) as ei:
        ta.tree_attn_check(run.plan)
    assert ei.value.code == ta.TA_ERR_DEVICE_TIMEOUT
    # the kernel waited for its limit and then returned on its own
    elapsed_us = start.elapsed_time(end) * 1e3
    assert limit_us <= elapsed_us < limit_us + 1e6, elapsed_us
    ta.tree_attn_check(run.plan)                           # the check cleared the status
    o, lse = run.fwd()                                     # the context still computes
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    assert_close("O", o, ref.o)
    assert np.array_equal(o, o0) and np.array_equal(lse, lse0)
