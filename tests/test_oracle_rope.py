"""Pins for the RoPE oracle (oracle/rope.py) from the mathematics, not from its own formula:
identity at position 0, a closed form that fixes the pair layout and the frequencies, the
relative-position phase relation of Octopus Eq. 1, the rotation group law, norm preservation."""
import numpy as np

from oracle.rope import rope


def test_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((5, 3, 16))
    assert np.array_equal(rope(x, np.zeros(5, np.int64)), x)


def test_closed_form_d4():
    # D = 4: pairs (0, 2) at theta_0 = 1 and (1, 3) at theta_1 = base^(-1/2)
    base, p = 10000.0, 37
    e1 = np.zeros((1, 1, 4)); e1[0, 0, 1] = 1.0
    y = rope(e1, np.array([p]), base)[0, 0]
    t1 = p * base ** -0.5
    assert np.allclose(y, [0.0, np.cos(t1), 0.0, np.sin(t1)], atol=1e-15, rtol=0)
    e0 = np.zeros((1, 1, 4)); e0[0, 0, 0] = 1.0
    assert np.allclose(rope(e0, np.array([p]), base)[0, 0], [np.cos(p), 0.0, np.sin(p), 0.0], atol=1e-15, rtol=0)


def test_relative_position_phase_relation():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((2, 1, 1, 128))
    for p, s, c in [(5, 3, 100), (1000, 20, 7), (262000, 1, 4096)]:
        a = np.sum(rope(q, [p]) * rope(k, [s]))
        b = np.sum(rope(q, [p + c]) * rope(k, [s + c]))
        z = np.sum(q * rope(k, [s - p]))                       # <q, R_{s-p} k>
        assert abs(a - b) <= 1e-9 * (1 + abs(a)) and abs(a - z) <= 1e-9 * (1 + abs(a))


def test_group_law_and_norms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 2, 64))
    p, s = np.array([3, 70, 1000, 5]), np.array([11, 0, 29, 123456])
    assert np.allclose(rope(rope(x, p), s), rope(x, p + s), atol=1e-10, rtol=0)
    y = rope(x, p)
    half = 32
    assert np.allclose(x[..., :half] ** 2 + x[..., half:] ** 2, y[..., :half] ** 2 + y[..., half:] ** 2, atol=1e-12)
