"""Pins for how one oracle layer routes its mixer inputs and outputs.

The mixer reading (EvSpark discussion post, "What we implemented": Hyena
layers with short / medium FIR and modal IIR filters, attention layers with
an append-only KV cache) is [a | b | v] = W_in xn, z = b * v, y = filter(z),
out-projection of a * y; attention takes [q | k | v] = W_in xn, rotates q and
k, attends causally with scale 1/sqrt(D_h) and projects the head outputs.
The filters, RoPE, attention and RMSNorm have pins of their own; these tests
tie down the wiring around them with one-hot weights, where a layer's update
has a closed form on one output column:

* FIR (2 taps, two steps): x1_out[c] - x1[c] = a1 (h0 b1 v1 + h1 b0 v0).
  Swapping the outer gate a with b or v, dropping the history, swapping the
  taps or misrouting the out-projection each change the value.
* IIR (one complex pole): x1_out[c] - x1[c] = a1 Re(R (lam z0 + z1)).
* Attention: a first token attends only to itself, so its update is its own
  v (unrotated); a second token whose predecessor's key is zero weighs
  (v0, v1) by softmax(0, q1 . k1 / sqrt(D_h)), the dot product of two keys
  rotated at one position being rotation-invariant.

Each closed form is also checked to reject the same oracle layer with a
planted misrouting (gate streams swapped, taps reversed, q / k or k / v
blocks swapped).

The MLP weights are zero, so the MLP adds exactly zero.
"""
import numpy as np
import pytest

from oracle.model import LayerState, Model, rmsnorm
from oracle.numerics import Arith

A64 = Arith(np.float64)
D, F = 8, 2


class _Shape:
    d_model, d_ffn, norm_eps = D, F, 1e-6
    n_heads, head_dim, rope_base = 1, D, 10000.0


def _model():
    m = Model.__new__(Model)
    m.shape, m.ar = _Shape(), A64
    return m


def _layer(kind, routes, col, out_row, **filt):
    """One-hot routing: block r of W_in (r = 0, 1, 2) reads input column
    routes[r] into component col; W_out row out_row reads component col."""
    w_in = np.zeros((3 * D, D))
    for r, i in enumerate(routes):
        w_in[r * D + col, i] = 1.0
    w_out = np.zeros((D, D))
    w_out[out_row, col] = 1.0
    M = {"kind": kind, "param": 0, "w_in": w_in, "w_out": w_out,
         "w_gu": np.zeros((2 * F, D)), "w_down": np.zeros((D, F))}
    M.update(filt)
    return M


def _two_steps(M, kind, x0, x1):
    """A fresh layer state, two tokens; the second token's layer output."""
    m = _model()
    if kind == "SE":
        L = LayerState("SE", window=np.zeros((M["taps"].shape[0] - 1, D)))
    else:
        L = LayerState("ATT", K=np.zeros((4, 1, D)), V=np.zeros((4, 1, D)), length=0)
    m.layer_forward(M, L, x0, 0)
    return m.layer_forward(M, L, x1, 1)


def _xs(seed, n=2):
    g = np.random.default_rng(seed)
    return [g.standard_normal(D) * 2 for _ in range(n)]


@pytest.mark.parametrize("routes,col,out_row", [((1, 4, 6), 2, 5), ((7, 0, 3), 5, 0), ((2, 2, 6), 1, 1)])
def test_fir_layer_gates(routes, col, out_row):
    ia, ib, iv = routes
    h = np.random.default_rng(1).standard_normal((2, D))
    M = _layer("SE", routes, col, out_row, taps=h)
    m = _model()
    L = LayerState("SE", window=np.zeros((1, D)))
    x0, x1 = _xs(sum(routes) + col)
    o0 = m.layer_forward(M, L, x0, 0)
    o1 = m.layer_forward(M, L, x1, 1)
    n0, n1 = rmsnorm(x0, 1e-6, A64), rmsnorm(x1, 1e-6, A64)
    z0, z1 = n0[ib] * n0[iv], n1[ib] * n1[iv]
    want0 = x0.copy()
    want0[out_row] += n0[ia] * h[0, col] * z0
    want1 = x1.copy()
    want1[out_row] += n1[ia] * (h[0, col] * z1 + h[1, col] * z0)
    np.testing.assert_allclose(o0, want0, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(o1, want1, rtol=1e-13, atol=1e-14)
    # planted slips (the same oracle layer misrouted) miss the closed form
    if ia != ib:
        assert abs(_two_steps(_layer("SE", (ib, ia, iv), col, out_row, taps=h), "SE", x0, x1)[out_row]
                   - want1[out_row]) > 1e-9                                  # a and b swapped
    assert abs(_two_steps(_layer("SE", routes, col, out_row, taps=h[::-1].copy()), "SE", x0, x1)[out_row]
               - want1[out_row]) > 1e-9                                      # taps reversed


def test_iir_layer_gates():
    ia, ib, iv, col, out_row = 3, 6, 1, 4, 2
    lam = np.full((D, 1), 0.6 + 0.3j)
    R = np.full((D, 1), 1.5 - 0.7j)
    M = _layer("LI", (ia, ib, iv), col, out_row, lam=lam, res=R)
    m = _model()
    L = LayerState("LI", s=np.zeros((D, 1), np.complex128))
    x0, x1 = _xs(9)
    o0 = m.layer_forward(M, L, x0, 0)
    o1 = m.layer_forward(M, L, x1, 1)
    n0, n1 = rmsnorm(x0, 1e-6, A64), rmsnorm(x1, 1e-6, A64)
    z0, z1 = n0[ib] * n0[iv], n1[ib] * n1[iv]
    lam_c, R_c = complex(lam[0, 0]), complex(R[0, 0])
    want0 = x0.copy()
    want0[out_row] += n0[ia] * (R_c * z0).real
    want1 = x1.copy()
    want1[out_row] += n1[ia] * (R_c * (lam_c * z0 + z1)).real
    np.testing.assert_allclose(o0, want0, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(o1, want1, rtol=1e-13, atol=1e-14)
    # the real part of the product, not the product of real parts
    assert abs(n1[ia] * (R_c.real * (lam_c.real * z0 + z1)) - (want1[out_row] - x1[out_row])) > 1e-6


@pytest.mark.parametrize("col", [1, 6])
def test_attention_layer_routing(col):
    iq, ik, iv, out_row = 2, 5, 7, 3
    M = _layer("ATT", (iq, ik, iv), col, out_row)
    m = _model()
    L = LayerState("ATT", K=np.zeros((4, 1, D)), V=np.zeros((4, 1, D)), length=0)
    x0, x1 = _xs(col + 20)
    x0[ik] = 0.0  # the first token's key is zero
    o0 = m.layer_forward(M, L, x0, 0)
    o1 = m.layer_forward(M, L, x1, 1)
    n0, n1 = rmsnorm(x0, 1e-6, A64), rmsnorm(x1, 1e-6, A64)
    want0 = x0.copy()
    want0[out_row] += n0[iv]  # one key: weight exactly 1; v is not rotated
    s1 = n1[iq] * n1[ik] / np.sqrt(D)
    w0, w1 = 1.0 / (1.0 + np.exp(s1)), np.exp(s1) / (1.0 + np.exp(s1))
    want1 = x1.copy()
    want1[out_row] += w0 * n0[iv] + w1 * n1[iv]
    np.testing.assert_allclose(o0, want0, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(o1, want1, rtol=1e-12, atol=1e-13)
    assert L.length == 2
    # planted slips: q and k blocks swapped, or k and v swapped
    for wrong in ((ik, iq, iv), (iq, iv, ik)):
        got = _two_steps(_layer("ATT", wrong, col, out_row), "ATT", x0, x1)
        assert abs(got[out_row] - want1[out_row]) > 1e-9, wrong
