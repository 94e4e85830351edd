"""Shared helpers for the GPU tests: move a synthetic episode to the device, run the library
through its C ABI, and compare with the oracle at the stated tolerances."""
import math

import numpy as np
import torch

import dag_packed_paged_gb300 as ta
from dag_packed_paged_gb300 import workloads as W

# tolerances for floating-point outputs (max-abs and relative RMS against the fp64 oracle)
MAX_ABS = 2e-2
REL_RMS = 1e-2


def bf16_tensor(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def as_f64(x: torch.Tensor) -> np.ndarray:
    return x.detach().float().cpu().numpy().astype(np.float64)


def metrics(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    d = got - want
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    rel = float(np.linalg.norm(d.ravel()) / max(np.linalg.norm(want.ravel()), 1e-30)) if d.size else 0.0
    return max_abs, rel


def assert_close(name, got, want, max_abs=MAX_ABS, rel_rms=REL_RMS):
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    ma, rr = metrics(got, want)
    assert ma <= max_abs and rr <= rel_rms, f"{name}: max_abs={ma:.3e} rel_rms={rr:.3e}"
    return ma, rr


class Run:
    """One episode on the device: inputs, plan, and the library's outputs."""

    def __init__(self, ep, dist="config", tensors=None, pool=None, dev="cuda:0", flags=0, **plan_kw):
        self.ep = ep
        self.t = tensors if tensors is not None else W.make_tensors(ep, dist=dist)
        self.pool = pool if pool is not None else W.make_pool(ep, self.t)
        self.dev = torch.device(dev)
        N, Hq, D = ep.n_rows, ep.num_q_heads, ep.head_dim
        self.q = bf16_tensor(self.t.q, self.dev)
        self.k_pool = bf16_tensor(self.pool.k_pool, self.dev)
        self.v_pool = bf16_tensor(self.pool.v_pool, self.dev)
        self.d_o = bf16_tensor(self.t.do, self.dev)
        self.plan = ta.tree_attn_plan(ep.branches, ep.mounts, self.pool.page_table,
                                      num_q_heads=Hq, num_kv_heads=ep.num_kv_heads, head_dim=D,
                                      page_size=ep.page_size, num_pages=self.pool.k_pool.shape[0],
                                      flags=flags, **plan_kw)
        self.o = torch.empty((N, Hq, D), dtype=torch.bfloat16, device=self.dev)
        self.lse = torch.empty((Hq, N), dtype=torch.float32, device=self.dev)

    def fwd(self):
        ta.tree_attn_fwd(self.plan, self.q, self.k_pool, self.v_pool, self.o, self.lse)
        ta.tree_attn_check(self.plan)
        return as_f64(self.o), as_f64(self.lse).T          # [N,Hq,D], [N,Hq]

    def bwd(self):
        ep = self.ep
        N, Hq, D = ep.n_rows, ep.num_q_heads, ep.head_dim
        ws = torch.empty(max(ta.tree_attn_bwd_workspace_size(self.plan), 256), dtype=torch.uint8,
                         device=self.dev)
        self.dq = torch.empty((N, Hq, D), dtype=torch.float32, device=self.dev)
        self.dk_pool = torch.zeros(self.k_pool.shape, dtype=torch.float32, device=self.dev)
        self.dv_pool = torch.zeros(self.v_pool.shape, dtype=torch.float32, device=self.dev)
        ta.tree_attn_bwd(self.plan, self.q, self.k_pool, self.v_pool, self.o, self.lse, self.d_o,
                         self.dq, self.dk_pool, self.dv_pool, ws)
        ta.tree_attn_check(self.plan)
        pt = self.pool.page_table
        dk = W.pool_rows(self.dk_pool.cpu().numpy(), pt, N).astype(np.float64)
        dv = W.pool_rows(self.dv_pool.cpu().numpy(), pt, N).astype(np.float64)
        return self.dq.cpu().numpy().astype(np.float64), dk, dv
