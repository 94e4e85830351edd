"""Pins for the oracle: checks against what the pages and the mathematics fix.

None of these compares the oracle with a retyped copy of its own formulas.  The references
are: a library routine (torch's scaled_dot_product_attention in fp64) run on every expanded
root-to-leaf trajectory; closed forms; finite differences; the worked example printed after
Octopus Eq. 2; HARTS Eq. 5 (compact rows) and Eq. 21-22 (visible pairs of a branch).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import dag
from dag_packed_paged_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _small_eps(seeds, **kw):
    out = []
    for s in seeds:
        ep = W.random_small(s, **kw)
        trajs = dag.trajectories(ep.branches, ep.mounts)
        if all(len({r for r, _ in t}) == len(t) for t in trajs):   # no row twice on a path
            out.append(ep)
    return out


def _traj_attention(traj, qf, kf, vf, scale, G, dof=None):
    """Causal attention over one expanded trajectory with torch's SDPA (fp64).

    Returns (query rows, O [nq,Hq,D], lse [nq,Hq], and if dof is given the autograd
    gradients dq [nq,Hq,D], dk/dv [L,Hkv,D] together with the KV rows)."""
    rows = np.array([r for r, _ in traj])
    isq = np.array([q for _, q in traj])
    L = len(rows)
    qpos = np.nonzero(isq)[0]
    qrows = rows[qpos]
    q = torch.tensor(qf[qrows], dtype=torch.float64).permute(1, 0, 2)       # [Hq, nq, D]
    k = torch.tensor(kf[rows], dtype=torch.float64).permute(1, 0, 2)        # [Hkv, L, D]
    v = torch.tensor(vf[rows], dtype=torch.float64).permute(1, 0, 2)
    k = k.repeat_interleave(G, 0)
    v = v.repeat_interleave(G, 0)
    mask = torch.tensor(np.arange(L)[None, :] <= qpos[:, None])             # causal in sequence order
    if dof is not None:
        q.requires_grad_(True); k.requires_grad_(True); v.requires_grad_(True)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    s = (q @ k.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    out = [qrows, o.detach().permute(1, 0, 2).numpy(), lse.detach().T.numpy()]
    if dof is not None:
        do = torch.tensor(dof, dtype=torch.float64).permute(1, 0, 2)
        (o * do).sum().backward()
        Hkv = kf.shape[1]
        dk = k.grad.reshape(Hkv, G, L, -1).sum(1).permute(1, 0, 2).numpy()
        dv = v.grad.reshape(Hkv, G, L, -1).sum(1).permute(1, 0, 2).numpy()
        out += [q.grad.permute(1, 0, 2).numpy(), rows, dk, dv]
    return out


def rel(a, b):
    return np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(np.asarray(b).ravel()), 1e-300)


# -------------------------------------------------------------------- positions (Eq. 2)

def test_eq2_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "eq2_worked_example.json")))
    first, last, nxt = g["mounted_first_pos"], g["mounted_last_pos"], g["reader_pos_next"]
    # root rows 0..first-1; A forks at `first` and covers positions first..last;
    # B forks at `first` and has reached position `nxt` when it mounts all of A.
    a_len = last - first + 1
    b_pre = nxt - first
    br = W.make_branches([-1, 0, 0], [0, first, first], [first, a_len, b_pre + 5])
    mt = W.make_mounts([(2, b_pre, 1, 0, a_len)])
    pos = dag.positions(br, mt)
    b0 = int(br["row_start"][2])
    a0 = int(br["row_start"][1])
    assert pos[a0] == first and pos[a0 + a_len - 1] == last
    assert pos[b0 + b_pre - 1] == nxt - 1
    assert pos[b0 + b_pre] == g["expected_next_pos"]
    assert pos[b0 + b_pre + 1] == g["expected_next_pos"] + 1


def test_tiny_positions_jump():
    ep = W.tiny()
    pos = dag.positions(ep.branches, ep.mounts)
    # branch 2 starts after the 256-row root; its row 64 mounts branch 1's rows 64..127,
    # whose positions end at 256+127 = 383, so it continues at 384 instead of 320.
    b2 = int(ep.branches["row_start"][2])
    assert list(pos[b2 + 62:b2 + 66]) == [318, 319, 384, 385]
    assert pos[b2 + 127] == 384 + 63
    assert list(pos[:256]) == list(range(256))


@pytest.mark.parametrize("seed", range(40))
def test_positions_strictly_precede_queries(seed):
    """Eq. 2's guarantee: every visible key other than the query's own row has a smaller
    position than the query."""
    ep = W.random_small(seed, max_len=40)
    pos = dag.positions(ep.branches, ep.mounts)
    for r in range(ep.n_rows):
        for j in dag.visible_set(ep.branches, ep.mounts, r):
            if j != r:
                assert pos[j] < pos[r], (r, j)


# -------------------------------------------------------------------- counts (Eq. 5, Eq. 21-22)

@pytest.mark.parametrize("cfg", [1, 3])
def test_compact_rows_eq5_and_pairs_eq22(cfg):
    ep = W.config(cfg)
    br = ep.branches
    trajs = dag.trajectories(br, ep.mounts)
    assert dag.compact_rows_eq5([[r for r, _ in t] for t in trajs]) == ep.n_rows
    # Eq. 21-22: a branch with h ancestor rows and l own rows contributes l*h + l(l+1)/2 pairs
    expect = 0
    for b in range(len(br)):
        h, x = 0, b
        while br["parent"][x] >= 0:
            h += int(br["fork_offset"][x])
            x = int(br["parent"][x])
        l = int(br["length"][b])
        expect += l * h + l * (l + 1) // 2
    assert dag.count_pairs(br, ep.mounts) == expect
    if cfg == 3:
        assert sum(len(t) for t in trajs) == ep.info["expanded_rows"]


def test_irregular_search_matches_recorded():
    seed, rho, ratio = W.irregular_search()
    assert (seed, rho) == (W.IRREGULAR_SEED, W.IRREGULAR_RHO)
    ep = W.irregular()
    assert 126_000 <= ep.n_rows <= 130_000
    assert len(ep.branches) == 64
    # the shape statistic the irregular tree copies: about 5.6 expanded rows per compact row
    assert abs(ep.info["expanded_rows"] / ep.n_rows - 5.6) <= 0.1


def test_tiny_pair_count():
    ep = W.tiny()
    # root: 256*257/2; 3 branches: 128 rows seeing 256 + own prefix; mount: 64 rows x 64 rows
    assert dag.count_pairs(ep.branches, ep.mounts) == 256 * 257 // 2 + 3 * (128 * 256 + 128 * 129 // 2) + 64 * 64


# -------------------------------------------------------------------- check (i): trajectories

def crafted():
    """Mounts inherited by children forking after the mount point, interior and zero-offset
    forks, two mounts on one reader, a mount at the reader's first row."""
    br = W.make_branches([-1, 0, 0, 2, 2, 0, 2, 1],
                         [0, 30, 30, 25, 5, 12, 0, 20],
                         [30, 20, 40, 15, 9, 11, 7, 6])
    mt = W.make_mounts([(2, 10, 1, 5, 15), (3, 3, 1, 15, 20), (3, 0, 5, 2, 4), (6, 2, 1, 0, 3),
                        (7, 1, 5, 0, 11)])
    return W.Episode("crafted", br, mt, 4, 2, 64, 16, 17)


def crafted_p64():
    ep = crafted()
    ep.name, ep.num_q_heads, ep.num_kv_heads, ep.head_dim = "crafted_gqa8", 8, 1, 128
    return ep


TRAJ_EPS = ([crafted(), crafted_p64()]
            + _small_eps(range(60), max_len=48, sibling_mounts_only=True)[:20]
            + _small_eps(range(200, 300), max_branches=8, max_len=40, n_mounts=3,
                         sibling_mounts_only=True)[:10])


@pytest.mark.parametrize("ep", [W.tiny()] + TRAJ_EPS, ids=lambda e: e.name)
def test_packed_equals_trajectory_attention(ep):
    t = W.make_tensors(ep, dist="realistic")
    qf, kf, vf = f64(t.q), f64(t.k), f64(t.v)
    res = oracle.forward(ep.branches, ep.mounts, t.q, t.k, t.v, ep.softmax_scale)
    G = ep.num_q_heads // ep.num_kv_heads
    seen = np.zeros(ep.n_rows, bool)
    for traj in dag.trajectories(ep.branches, ep.mounts):
        qrows, o, lse = _traj_attention(traj, qf, kf, vf, ep.softmax_scale, G)
        assert np.abs(res.o[qrows] - o).max() <= 1e-12 * max(1.0, np.abs(o).max())
        assert np.abs(res.lse[qrows] - lse).max() <= 1e-12 * max(1.0, np.abs(lse).max())
        seen[qrows] = True
    assert seen.all()


# -------------------------------------------------------------------- check (iii): gradients

GRAD_EPS = ([crafted()] + _small_eps(range(60, 120), max_len=40, sibling_mounts_only=True)[:8]
            + _small_eps(range(300, 400), max_branches=8, max_len=32, n_mounts=3,
                         sibling_mounts_only=True)[:6])


@pytest.mark.parametrize("ep", [W.tiny()] + GRAD_EPS, ids=lambda e: e.name)
def test_shared_row_gradients_sum_over_trajectories(ep):
    t = W.make_tensors(ep, dist="realistic")
    qf, kf, vf = f64(t.q), f64(t.k), f64(t.v)
    N, Hq, D, Hkv = ep.n_rows, ep.num_q_heads, ep.head_dim, ep.num_kv_heads
    G = Hq // Hkv
    rng = np.random.default_rng(ep.seed + 99)
    trajs = dag.trajectories(ep.branches, ep.mounts)
    # an independent upstream gradient per semantic position, in multiples of 1/16 so that
    # their per-compact-row sums are exact in bf16
    dos = [rng.integers(-4, 5, size=(sum(q for _, q in tr), Hq, D)) / 16.0 for tr in trajs]
    do_packed = np.zeros((N, Hq, D))
    for tr, d in zip(trajs, dos):
        qrows = np.array([r for r, q in tr if q])
        np.add.at(do_packed, qrows, d)
    assert np.abs(do_packed).max() < 256 / 16
    do_bits = W.f32_to_bf16_bits(do_packed.astype(np.float32))
    assert (f64(do_bits) == do_packed).all()
    res = oracle.run(ep.branches, ep.mounts, t.q, t.k, t.v, do_bits, ep.softmax_scale)
    dq = np.zeros((N, Hq, D)); dk = np.zeros((N, Hkv, D)); dv = np.zeros((N, Hkv, D))
    for tr, d in zip(trajs, dos):
        qrows, _, _, gq, kvrows, gk, gv = _traj_attention(tr, qf, kf, vf, ep.softmax_scale, G, d)
        np.add.at(dq, qrows, gq)
        np.add.at(dk, kvrows, gk)
        np.add.at(dv, kvrows, gv)
    for got, want in ((res.dq, dq), (res.dk, dk), (res.dv, dv)):
        assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())


# -------------------------------------------------------------------- check (ii): empty mounts

@pytest.mark.parametrize("seed", range(8))
def test_zero_length_mounts_change_nothing(seed):
    ep = W.random_small(seed, max_len=64)
    rng = np.random.default_rng(seed)
    extra = []
    for _ in range(4):
        r = int(rng.integers(0, len(ep.branches)))
        s = int(rng.integers(0, len(ep.branches)))
        t = int(rng.integers(0, int(ep.branches["length"][r])))
        b = int(rng.integers(0, int(ep.branches["length"][s]) + 1))
        extra.append((r, t, s, b, b))
    rows = [tuple(int(x) for x in m) for m in ep.mounts] + extra
    rng.shuffle(rows)
    mt2 = W.make_mounts(rows)
    tn = W.make_tensors(ep)
    assert (dag.positions(ep.branches, ep.mounts) == dag.positions(ep.branches, mt2)).all()
    a = dag.visible_intervals(ep.branches, ep.mounts)
    b = dag.visible_intervals(ep.branches, mt2)
    for x, y in zip(a, b):
        assert (x == y).all()
    r1 = oracle.run(ep.branches, ep.mounts, tn.q, tn.k, tn.v, tn.do, ep.softmax_scale)
    r2 = oracle.run(ep.branches, mt2, tn.q, tn.k, tn.v, tn.do, ep.softmax_scale)
    for f in ("o", "lse", "dq", "dk", "dv"):
        assert (getattr(r1, f) == getattr(r2, f)).all()


# -------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("ep", [W.tiny(), W.random_small(3), W.random_small(11)], ids=lambda e: e.name)
def test_zero_queries_give_uniform_attention(ep):
    t = W.make_tensors(ep)
    q0 = np.zeros_like(t.q)
    res = oracle.forward(ep.branches, ep.mounts, q0, t.k, t.v, ep.softmax_scale)
    vf = f64(t.v)
    G = ep.num_q_heads // ep.num_kv_heads
    for r in range(ep.n_rows):
        vis = sorted(dag.visible_set(ep.branches, ep.mounts, r))
        assert np.allclose(res.lse[r], math.log(len(vis)), rtol=0, atol=1e-13)
        mean = vf[vis].mean(0)                                   # [Hkv, D]
        assert np.abs(res.o[r] - np.repeat(mean, G, 0)).max() < 1e-13


@pytest.mark.parametrize("ep", [W.tiny(), W.scaled(4, 64), W.scaled(2, 256)], ids=lambda e: e.name)
def test_gradient_sum_identities(ep):
    """Each row of dS sums to zero, so sum_j dK[j] = 0; the probabilities of a row sum to one,
    so sum_j dV[j, g] = sum over rows and the heads of group g of dO."""
    t = W.make_tensors(ep, dist="realistic")
    res = oracle.run(ep.branches, ep.mounts, t.q, t.k, t.v, t.do, ep.softmax_scale)
    G = ep.num_q_heads // ep.num_kv_heads
    dof = f64(t.do)
    want = dof.reshape(ep.n_rows, ep.num_kv_heads, G, ep.head_dim).sum((0, 2))
    assert np.abs(res.dk.sum(0)).max() < 1e-12 * max(1.0, np.abs(res.dk).max()) * ep.n_rows
    assert np.abs(res.dv.sum(0) - want).max() < 1e-10


def test_single_root_is_causal_attention():
    br = W.make_branches([-1], [0], [200])
    ep = W.Episode("root", br, W.make_mounts([]), 4, 2, 64, 16, 5)
    t = W.make_tensors(ep, dist="realistic")
    res = oracle.forward(br, ep.mounts, t.q, t.k, t.v, ep.softmax_scale)
    q = torch.tensor(f64(t.q)).permute(1, 0, 2)
    k = torch.tensor(f64(t.k)).permute(1, 0, 2).repeat_interleave(2, 0)
    v = torch.tensor(f64(t.v)).permute(1, 0, 2).repeat_interleave(2, 0)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=ep.softmax_scale)
    assert np.abs(res.o - o.permute(1, 0, 2).numpy()).max() < 1e-13


# -------------------------------------------------------------------- finite differences

def test_backward_matches_finite_differences():
    """Richardson-extrapolated central differences of L = sum dO . O, stepping inputs by one
    and two bf16 ulps (both exactly representable), against the oracle's dQ/dK/dV."""
    ep = W.random_small(5, max_len=48, n_mounts=2)
    t = W.make_tensors(ep, dist="realistic")
    res = oracle.run(ep.branches, ep.mounts, t.q, t.k, t.v, t.do, ep.softmax_scale)
    dof = f64(t.do)
    iv = res.intervals

    def loss(q, k, v):
        r = oracle.forward(ep.branches, ep.mounts, q, k, v, ep.softmax_scale, intervals=iv)
        return float((r.o * dof).sum())

    rng = np.random.default_rng(0)
    checked = 0
    for name, grad in (("q", res.dq), ("k", res.dk), ("v", res.dv)):
        arr = getattr(t, name)
        for _ in range(200):
            idx = tuple(int(rng.integers(0, s)) for s in arr.shape)
            bits = int(arr[idx])
            mant = bits & 0x7F
            if not (8 <= mant <= 119) or (bits & 0x7F80) == 0:
                continue                                  # keep +-2 ulps inside the binade
            x0 = f64(np.uint16(bits))
            steps = {}
            for k_ in (1, 2):
                vals = []
                for sgn in (+1, -1):
                    a = arr.copy()
                    a[idx] = np.uint16(bits + sgn * k_)
                    vals.append((f64(a[idx]), loss(*(a if n == name else getattr(t, n) for n in "qkv"))))
                (xp, lp), (xm, lm) = vals
                steps[k_] = (lp - lm) / (xp - xm)
            fd = (4 * steps[1] - steps[2]) / 3
            g = grad[idx]
            assert abs(fd - g) <= 1e-6 * max(abs(g), 1e-3 * np.abs(grad).max()), (name, idx, fd, g, x0)
            checked += 1
            if checked % 4 == 0:
                break
    assert checked >= 12
