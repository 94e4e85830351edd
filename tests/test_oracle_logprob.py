"""Pins for the compact log-probability oracle (oracle/logprob.py): against the expanded
computation it replaces -- torch.log_softmax and autograd on S x V logits copied row by row
from the compact ones (HARTS Section 4, Eq. 17-20) -- and closed forms."""
import numpy as np
import torch

from oracle import logprob as LP


def _case(seed, C=37, V=211, S=120):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((C, V)) * 3.0
    pos_row = rng.integers(0, C, S)
    pos_row[:5] = 0                                   # one row shared by several positions
    pos_target = rng.integers(0, V, S)
    pos_target[1] = pos_target[0]                     # two positions, same row, same target
    g = rng.standard_normal(S)
    return z, pos_row, pos_target, g


def test_logprob_equals_expanded_log_softmax():
    for seed in range(4):
        z, pr, pt, _ = _case(seed)
        lam, lse = LP.logprob(z, pr, pt)
        zt = torch.tensor(z, dtype=torch.float64)
        want = torch.log_softmax(zt[torch.tensor(pr)], dim=1)[torch.arange(len(pr)), torch.tensor(pt)]
        assert np.allclose(lam, want.numpy(), atol=1e-12, rtol=0)
        assert np.allclose(lse, torch.logsumexp(zt, dim=1).numpy(), atol=1e-12, rtol=0)


def test_gradient_equals_autograd_of_expanded_objective():
    for seed in range(4):
        z, pr, pt, g = _case(seed)
        zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
        lam = torch.log_softmax(zt[torch.tensor(pr)], dim=1)[torch.arange(len(pr)), torch.tensor(pt)]
        (lam * torch.tensor(g)).sum().backward()
        assert np.allclose(LP.dlogits(z, pr, pt, g), zt.grad.numpy(), atol=1e-12, rtol=0)


def test_closed_forms():
    V = 64
    z = np.full((3, V), 0.7)
    lam, lse = LP.logprob(z, np.array([0, 1, 2]), np.array([5, 6, 7]))
    assert np.allclose(lam, -np.log(V), atol=1e-14) and np.allclose(lse, 0.7 + np.log(V), atol=1e-14)
    z, pr, pt, g = _case(7)
    d = LP.dlogits(z, pr, pt, g)
    assert np.allclose(d.sum(axis=1), 0.0, atol=1e-10)          # rows of dz sum to zero
    untouched = np.setdiff1d(np.arange(len(z)), pr)
    assert np.all(d[untouched] == 0)                              # rows no position reads
