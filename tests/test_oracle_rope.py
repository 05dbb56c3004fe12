"""Pins of the RoPE oracle (oracle/ida_rope.py) against properties of the rotation."""
import numpy as np

from oracle import ida_rope as ro


def test_two_channels_rotate_by_the_position():
    """R = 2: the pair is rotated by exactly p radians."""
    x = np.array([[[[1.0, 0.0]]], [[[0.3, -2.0]]]]).reshape(2, 1, 1, 2)
    for p in (0, 1, 5, 1000):
        got = ro.rope(x, pos0=p)
        c, s = np.cos(p), np.sin(p)
        np.testing.assert_allclose(got[..., 0], x[..., 0] * c - x[..., 1] * s, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(got[..., 1], x[..., 0] * s + x[..., 1] * c, rtol=1e-14, atol=1e-14)


def test_rotation_keeps_pair_norms_and_position_zero_is_identity():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 9, 3, 16))
    y = ro.rope(x, pos0=17)
    np.testing.assert_allclose(y[..., 0::2] ** 2 + y[..., 1::2] ** 2, x[..., 0::2] ** 2 + x[..., 1::2] ** 2, rtol=1e-12)
    np.testing.assert_allclose(ro.rope(x[:, :1], pos0=0), x[:, :1], rtol=0, atol=0)


def test_scores_depend_on_the_relative_position_only():
    """<rope(q, m), rope(k, n)> = <rope(q, m - n), k>: the property rotary embeddings exist for."""
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((1, 1, 1, 32)), rng.standard_normal((1, 1, 1, 32))
    for m, n in ((5, 2), (100, 37), (3, 3)):
        lhs = (ro.rope(q, m) * ro.rope(k, n)).sum()
        rhs = (ro.rope(q, m - n) * k).sum()
        np.testing.assert_allclose(lhs, rhs, rtol=1e-11)


def test_rotations_compose_and_frequencies_follow_the_base():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 1, 2, 8))
    np.testing.assert_allclose(ro.rope(ro.rope(x, 7), 5), ro.rope(x, 12), rtol=1e-12)
    th = ro.angles(np.array([1.0]), 8, base=16.0)
    np.testing.assert_allclose(th[0], [1.0, 0.5, 0.25, 0.125], rtol=1e-15)
    # positions advance along axis 1
    y = ro.rope(np.repeat(x, 3, axis=1), pos0=4)
    np.testing.assert_allclose(y[:, 2], ro.rope(x, 6)[:, 0], rtol=1e-14)


def test_adjacent_channels_form_the_pairs():
    """The reading: channels (2i, 2i + 1) rotate together (not i and i + R/2)."""
    x = np.zeros((1, 1, 1, 4))
    x[..., 0] = 1.0
    np.testing.assert_allclose(ro.rope(x, 1)[0, 0, 0], [np.cos(1.0), np.sin(1.0), 0.0, 0.0], atol=1e-15)
