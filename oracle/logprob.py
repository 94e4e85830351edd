"""Oracle: compact-to-semantic log-probabilities and their gradient (fp64).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

HARTS (arXiv 2608.28158) Section 4: a compact logit row z_c serves every semantic position s
with m(s) = c; the log-probability of position s with next token y_s is
    lambda_s = z_{m(s), y_s} - log sum_v exp z_{m(s), v}                       (Eq. 17)
with the row maximum and sum-exp formed once per compact row; backward accumulates every
position's contribution into its compact row,
    grad z_c = sum_{s: m(s) = c} (dL/dlambda_s) grad_{z_c} lambda_s              (Eq. 19-20)
and grad_{z_c} lambda_s = e_{y_s} - softmax(z_c).
"""
from __future__ import annotations

import numpy as np


def row_lse(z):
    """Natural-log sum-exp of every compact row: z [C, V] -> [C] (fp64)."""
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def logprob(z, pos_row, pos_target):
    """lambda_s for every semantic position (Eq. 17)."""
    z = np.asarray(z, dtype=np.float64)
    lse = row_lse(z)
    return z[pos_row, pos_target] - lse[pos_row], lse


def dlogits(z, pos_row, pos_target, g):
    """grad of sum_s g_s lambda_s with respect to the compact logits (Eq. 19-20): [C, V]."""
    z = np.asarray(z, dtype=np.float64)
    lse = row_lse(z)
    p = np.exp(z - lse[:, None])
    out = np.zeros_like(z)
    G = np.zeros(len(z))
    np.add.at(G, pos_row, g)
    out -= G[:, None] * p
    np.add.at(out, (pos_row, pos_target), g)
    return out
