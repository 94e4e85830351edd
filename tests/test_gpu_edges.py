"""Degenerate episodes on the GPU: the empty DAG (N = 0: every call is a no-op) and DAGs of
one row and of one row per branch, whose attention has a closed form: a row that sees only
itself has P = 1, so O = V of that row, lse = scale * <q, k>, dQ = dK = 0 (dS = P (dP - delta)
with delta = <dO, O> = <dO, V> = dP) and dV = dO summed over its readers."""

import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
import oracle
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import Run, as_f64, assert_close, metrics

pytestmark = pytest.mark.gpu


def test_empty_dag_calls_are_noops():
    br = W.make_branches([], [], [])
    plan = ta.tree_attn_plan(br, W.make_mounts([]), np.zeros(1, dtype=np.int32), num_q_heads=4,
                             num_kv_heads=1, head_dim=64, page_size=16, num_pages=1)
    assert ta.tree_attn_plan_stats(plan)["n_rows"] == 0
    ta.tree_attn_fwd(plan, None, None, None, None, None)
    ta.tree_attn_bwd(plan, None, None, None, None, None, None, None, None, None, None, ws_bytes=0)
    ta.tree_attn_check(plan)


@pytest.mark.parametrize("heads,D,P", [((4, 1), 64, 16), ((16, 4), 128, 64)])
def test_single_row_closed_form(heads, D, P):
    ep = W.Episode("one_row", W.make_branches([-1], [0], [1]), W.make_mounts([]), heads[0], heads[1], D, P, 3)
    run = Run(ep, dist="realistic")
    o, lse = run.fwd()
    dq, dk, dv = run.bwd()
    t = run.t
    G = heads[0] // heads[1]
    q = W.bf16_bits_to_f32(t.q).astype(np.float64)[0]                        # [Hq, D]
    k = W.bf16_bits_to_f32(t.k).astype(np.float64)[0]                        # [Hkv, D]
    v = W.bf16_bits_to_f32(t.v).astype(np.float64)[0]
    do = W.bf16_bits_to_f32(t.do).astype(np.float64)[0]
    kv = np.repeat(np.arange(heads[1]), G)
    assert_close("O", o[0], v[kv], max_abs=8e-3, rel_rms=4e-3)          # bf16 rounding of V only
    assert metrics(lse[0], ep.softmax_scale * np.einsum("hd,hd->h", q, k[kv]))[0] <= 1e-3
    assert np.abs(dq).max() <= 1e-3 and np.abs(dk).max() <= 1e-3
    want_dv = np.zeros_like(v)
    np.add.at(want_dv, kv, do)
    assert_close("dV", dv[0], want_dv)


def test_rows_that_see_only_themselves():
    """Eight one-row roots: every row is its own DAG, so each row's result is the closed form."""
    n = 8
    ep = W.Episode("singletons", W.make_branches([-1] * n, [0] * n, [1] * n), W.make_mounts([]), 8, 2, 128, 16, 5)
    run = Run(ep, dist="realistic")
    o, lse = run.fwd()
    dq, dk, dv = run.bwd()
    ref = oracle.run(ep.branches, ep.mounts, run.t.q, run.t.k, run.t.v, run.t.do, ep.softmax_scale)
    assert_close("O", o, ref.o)
    assert metrics(lse, ref.lse)[0] <= 2e-3
    assert np.abs(dq).max() <= 1e-3 and np.abs(dk).max() <= 1e-3
    assert_close("dV", dv, ref.dv)
