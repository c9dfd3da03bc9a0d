"""Pins for the oracle's rotary embedding, attention and RMSNorm.

Rotary embedding: identity at position 0; an isometry; a plane rotation by
exactly pos * base^(-2i/Dh) on the pair (i, i + Dh/2); scores depend only on
the relative position.  Attention: uniform scores give the mean of V; one
key gives that value row; two keys follow the closed-form two-point softmax.
RMSNorm: unit root-mean-square output, invariant to positive scaling.
"""
import numpy as np

from oracle.model import attend, rmsnorm, rope
from oracle.numerics import Arith

AR = Arith(np.float64)


def test_rope_identity_and_isometry():
    g = np.random.default_rng(0)
    x = g.standard_normal((3, 16))
    assert np.array_equal(rope(x, 0, 10000.0, AR), x)
    for pos in (1, 7, 1000, 262143):
        y = rope(x, pos, 10000.0, AR)
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_explicit_pair_rotation():
    Dh = 8
    for i in range(Dh // 2):
        x = np.zeros((1, Dh))
        x[0, i] = 1.0                      # unit vector on the first element of pair i
        pos = 3
        ang = pos * 10000.0 ** (-2.0 * i / Dh)
        y = rope(x, pos, 10000.0, AR)
        want = np.zeros((1, Dh))
        want[0, i] = np.cos(ang)
        want[0, i + Dh // 2] = np.sin(ang)
        np.testing.assert_allclose(y, want, atol=1e-15)


def test_rope_relative_position():
    g = np.random.default_rng(1)
    q = g.standard_normal((1, 32))
    k = g.standard_normal((1, 32))
    for m, n, c in ((5, 2, 11), (100, 37, 4000)):
        a = rope(q, m, 10000.0, AR) @ rope(k, n, 10000.0, AR).T
        b = rope(q, m + c, 10000.0, AR) @ rope(k, n + c, 10000.0, AR).T
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9)


def test_attention_special_cases():
    g = np.random.default_rng(2)
    H, Dh, T = 2, 8, 9
    K = g.standard_normal((T, H, Dh))
    V = g.standard_normal((T, H, Dh))
    # zero query: uniform weights -> mean of values
    o = attend(np.zeros((H, Dh)), K, V, AR)
    np.testing.assert_allclose(o, V.mean(axis=0), rtol=1e-13, atol=1e-13)
    # one key: the value row itself
    q = g.standard_normal((H, Dh))
    np.testing.assert_allclose(attend(q, K[:1], V[:1], AR), V[0], rtol=1e-13)
    # two keys: weight of key 1 is 1 / (1 + exp(-(s1 - s0)))
    s = np.einsum("thd,hd->th", K[:2], q) / np.sqrt(Dh)
    w1 = 1.0 / (1.0 + np.exp(-(s[1] - s[0])))
    want = (1 - w1)[:, None] * V[0] + w1[:, None] * V[1]
    np.testing.assert_allclose(attend(q, K[:2], V[:2], AR), want, rtol=1e-12)


def test_rmsnorm():
    g = np.random.default_rng(3)
    x = g.standard_normal(4096) * 3.7
    y = rmsnorm(x, 0.0, AR)
    assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    np.testing.assert_allclose(rmsnorm(5.0 * x, 0.0, AR), y, rtol=1e-14)
