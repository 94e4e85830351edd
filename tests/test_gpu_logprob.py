"""Compact-to-semantic log-probabilities on the GPU (HARTS Section 4, Eq. 17-20) through the C
ABI, against the fp64 oracle (oracle/logprob.py): small cases element by element, and the
full-size configuration (the balanced tree's 45,056 compact rows x a 151,936-token vocabulary,
logits generated on the device) on sampled rows and positions."""
import numpy as np
import pytest
import torch

import dag_packed_paged_gb300 as ta
from dag_packed_paged_gb300 import workloads as W
from gpu_helpers import metrics
from oracle import logprob as LP

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def assert_bf16_close(name, got, want):
    """dlogits is bf16: round-to-nearest leaves at most 2^-9 relative error per element; allow
    2^-8 relative (plus 1e-5 absolute) for the fp32 exponentials and sums before the rounding,
    and the spec relative RMS over the whole array."""
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    bad = np.abs(got - want) > 2.0 ** -8 * np.abs(want) + 1e-5
    assert not bad.any(), f"{name}: {int(bad.sum())} elements beyond 2^-8 relative, e.g. got {got[bad][:3]} want {want[bad][:3]}"
    assert metrics(got, want)[1] <= 1e-2


def _run(logits_bf16, pos_row, pos_target, g):
    C, V = logits_bf16.shape
    pr = torch.from_numpy(pos_row).to(DEV)
    pt = torch.from_numpy(pos_target).to(DEV)
    lse = torch.empty(C, dtype=torch.float32, device=DEV)
    lp = torch.empty(len(pos_row), dtype=torch.float32, device=DEV)
    ta.tree_attn_logprob_fwd(logits_bf16, pr, pt, lse, lp)
    ptr, pos = ta.tree_attn_logprob_index(pos_row, pos_target, C, V)
    dz = torch.empty_like(logits_bf16)
    ta.tree_attn_logprob_bwd(logits_bf16, lse, torch.from_numpy(ptr).to(DEV), torch.from_numpy(pos).to(DEV), pt,
                             torch.from_numpy(g).to(DEV), dz)
    torch.cuda.synchronize()
    return lse, lp, dz


CASES = [("tiny_v4096", W.tiny, 4096), ("balanced16_v32000", lambda: W.scaled(1, 16), 32000),
         ("irregular32_v8192", lambda: W.scaled(3, 32), 8192)]


@pytest.mark.parametrize("name,make,V", CASES, ids=[c[0] for c in CASES])
def test_logprob_small(name, make, V):
    ep = make()
    pr, pt, _ = W.semantic_positions(ep, V, seed=1)
    rng = np.random.default_rng(2)
    z = (rng.standard_normal((ep.n_rows, V)) * 3.0).astype(np.float32)
    zb = torch.from_numpy(z).to(DEV).to(torch.bfloat16)
    z64 = zb.float().cpu().numpy().astype(np.float64)          # the bf16 values the kernel reads
    g = rng.standard_normal(len(pr)).astype(np.float32)
    g[rng.random(len(pr)) < 0.3] = 0.0                           # outside the action mask
    lse, lp, dz = _run(zb, pr, pt, g)
    want_lp, want_lse = LP.logprob(z64, pr, pt)
    assert metrics(lse.cpu().numpy(), want_lse)[0] <= 2e-3
    assert metrics(lp.cpu().numpy(), want_lp)[0] <= 2e-3
    want_dz = LP.dlogits(z64, pr, pt, g.astype(np.float64))
    assert_bf16_close("dlogits", dz.float().cpu().numpy().astype(np.float64), want_dz)
    untouched = np.setdiff1d(np.arange(ep.n_rows), pr)
    assert torch.count_nonzero(dz[torch.from_numpy(untouched).to(DEV)]).item() == 0
    # deterministic
    _, lp2, dz2 = _run(zb, pr, pt, g)
    assert torch.equal(lp, lp2) and torch.equal(dz.view(torch.int16), dz2.view(torch.int16))


def test_logprob_full_size_sampled():
    ep = W.config(1)                       # balanced tree: 45,056 compact rows
    V = 151_936
    pr, pt, _ = W.semantic_positions(ep, V, seed=5)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(11)
    zb = (torch.randn((ep.n_rows, V), generator=gen, device=DEV) * 3.0).to(torch.bfloat16)
    rng = np.random.default_rng(6)
    g = rng.standard_normal(len(pr)).astype(np.float32)
    lse, lp, dz = _run(zb, pr, pt, g)
    rows = np.unique(np.concatenate([rng.choice(ep.n_rows, 24, replace=False), pr[:4], [0, ep.n_rows - 1]]))
    z64 = zb[torch.from_numpy(rows).to(DEV)].float().cpu().numpy().astype(np.float64)
    remap = -np.ones(ep.n_rows, dtype=np.int64)
    remap[rows] = np.arange(len(rows))
    sel = np.nonzero(remap[pr] >= 0)[0]
    want_lp, want_lse = LP.logprob(z64, remap[pr[sel]], pt[sel])
    assert metrics(lse.cpu().numpy()[rows], want_lse)[0] <= 2e-3
    assert metrics(lp.cpu().numpy()[sel], want_lp)[0] <= 2e-3
    want_dz = LP.dlogits(z64, remap[pr[sel]], pt[sel], g[sel].astype(np.float64))
    got_dz = dz[torch.from_numpy(rows).to(DEV)].float().cpu().numpy().astype(np.float64)
    assert_bf16_close("dlogits", got_dz, want_dz)
