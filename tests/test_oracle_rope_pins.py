"""Pins for the oracle's rotate-half rotary embedding (ferrotensor
engine/attention.rs, rope / rope_theta) -- facts of a rotation that any
mistake in the pairing, the sign or the frequency breaks."""
import numpy as np


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_position_zero_is_identity(oracle):
    x = rnd((2, 1, 3 * 8), 1)
    np.testing.assert_array_equal(oracle.rope(x, head_dim=8, pos=0), x)


def test_rotation_keeps_every_pair_length(oracle):
    x = rnd((2, 5, 2 * 16), 2)
    y = oracle.rope(x, head_dim=16, pos=7)
    xs = x.reshape(2, 5, 2, 16)
    ys = y.reshape(2, 5, 2, 16)
    np.testing.assert_allclose(xs[..., :8] ** 2 + xs[..., 8:] ** 2, ys[..., :8] ** 2 + ys[..., 8:] ** 2, atol=1e-12)


def test_two_dimensional_closed_form(oracle):
    """head_dim 2: one pair, frequency theta**0 = 1, angle = position."""
    x = np.array([[[1.0, 0.0], [1.0, 0.0], [0.0, 1.0]]])
    y = oracle.rope(x, head_dim=2, pos=3)
    for s, (a, b) in enumerate([(1.0, 0.0), (1.0, 0.0), (0.0, 1.0)]):
        ang = 3.0 + s
        np.testing.assert_allclose(y[0, s], [a * np.cos(ang) - b * np.sin(ang), b * np.cos(ang) + a * np.sin(ang)],
                                   atol=1e-15)


def test_frequencies_follow_theta(oracle):
    """Unit vector on pair i at position 1 turns by theta**(-2i/hd)."""
    hd, theta = 8, 500.0
    for i in range(hd // 2):
        x = np.zeros((1, 1, hd))
        x[0, 0, i] = 1.0
        y = oracle.rope(x, head_dim=hd, pos=1, theta=theta)
        ang = theta ** (-2.0 * i / hd)
        np.testing.assert_allclose([y[0, 0, i], y[0, 0, i + hd // 2]], [np.cos(ang), np.sin(ang)], atol=1e-15)


def test_scores_depend_on_relative_position_only(oracle):
    """(R_m q) . (R_n k) = (R_{m+d} q) . (R_{n+d} k): the property RoPE exists for."""
    hd = 16
    q, k = rnd((1, 1, hd), 3), rnd((1, 1, hd), 4)
    s1 = float((oracle.rope(q, head_dim=hd, pos=5) * oracle.rope(k, head_dim=hd, pos=2)).sum())
    s2 = float((oracle.rope(q, head_dim=hd, pos=105) * oracle.rope(k, head_dim=hd, pos=102)).sum())
    np.testing.assert_allclose(s1, s2, rtol=1e-10)


def test_token_positions_count_within_each_sequence(oracle):
    x = rnd((2, 4, 8), 5)
    y = oracle.rope(x, head_dim=8, pos=10)
    np.testing.assert_allclose(y[1, 2], oracle.rope(x[1:2, 2:3], head_dim=8, pos=12)[0, 0], atol=1e-15)
