"""Oracle: rotary position embedding of compact rows (fp64).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Octopus (arXiv 2611.06956) Section 3.2 uses RoPE's phase relation
<R_p q, R_s k> = <q, R_{s-p} k> (Eq. 1); HARTS (arXiv 2608.28158) Section 4.2 applies RoPE once
per compact row before attention.  The pages do not print the rotation itself; this follows
the common definition with the half-split pair layout (a reading listed in the design notes):
for i < D/2, (x_i, x_{i+D/2}) is rotated by the angle p * theta_i, theta_i = base^(-2i/D).
"""
from __future__ import annotations

import numpy as np


def rope(x, pos, base=10000.0):
    """x: float array [N, H, D]; pos: int [N].  Returns the rotated copy in fp64."""
    x = np.asarray(x, dtype=np.float64)
    n, h, d = x.shape
    half = d // 2
    theta = base ** (-2.0 * np.arange(half, dtype=np.float64) / d)        # [D/2]
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]    # [N, D/2]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)
