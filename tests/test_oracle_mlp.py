"""Pins for the oracle's SiLU and gated-MLP branch.

The pages say nothing about the MLP; the oracle reads it as the gated form
x += W_down (silu(W_gate xn) * W_up xn), xn = RMSNorm(x).  These tests tie
that reading down independently of the oracle's own formula:

* SiLU equals g * expit(g) (scipy's logistic function, a library routine),
  and satisfies silu(g) - silu(-g) = g and silu(0) = 0 (closed forms that a
  sign slip such as g * sigmoid(-g) breaks).
* With the mixer weights zero and one-hot rows in W_gate, W_up and W_down,
  one layer's update is exactly silu(xn_i) * xn_j on one output column and
  zero elsewhere (a closed form built from the pinned RMSNorm): swapping the
  gate and up halves, dropping a term or misrouting a row fails it.  In the
  bf16 storage mode the hidden value is rounded to bf16 before the down
  projection, which the same closed form with the rounding applied checks.
"""
import numpy as np
import pytest
from scipy.special import expit

from oracle.model import LayerState, Model, rmsnorm, silu
from oracle.numerics import Arith, round_bf16

A64 = Arith(np.float64)
A32 = Arith(np.float32, bf16_points=True)


def test_silu_is_g_times_logistic():
    g = np.concatenate([np.linspace(-30, 30, 2001), [-700.0, -80.0, 80.0, 700.0]])
    got = silu(g, A64)
    want = g * expit(g)
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-300)


def test_silu_closed_forms():
    g = np.linspace(-12, 12, 97)
    s = silu(g, A64)
    np.testing.assert_allclose(s - silu(-g, A64), g, rtol=0, atol=1e-13)
    assert silu(np.float64(0.0), A64) == 0.0
    assert abs(silu(np.float64(40.0), A64) - 40.0) < 1e-15 * 40
    assert abs(silu(np.float64(-40.0), A64)) < 1e-15
    # float32 mode keeps the same function to float32 accuracy
    np.testing.assert_allclose(silu(g.astype(np.float32), A32), g * expit(g), rtol=2e-6, atol=1e-6)


class _Shape:
    def __init__(self, d, F):
        self.d_model, self.d_ffn, self.norm_eps = d, F, 1e-6
        self.n_heads, self.head_dim, self.rope_base = 1, d, 10000.0


def _mlp_only_layer(d, F, gate_rows, up_rows, down_cols, kind="SE"):
    """Mixer weights zero (so the mixer adds exactly zero); W_gate row f is
    one-hot at gate_rows[f], W_up row f at up_rows[f], W_down row
    down_cols[f] one-hot at column f (hidden unit f feeds one output)."""
    w_gu = np.zeros((2 * F, d))
    w_down = np.zeros((d, F))
    for f, (i, j, c) in enumerate(zip(gate_rows, up_rows, down_cols)):
        w_gu[f, i] = 1.0
        w_gu[F + f, j] = 1.0
        w_down[c, f] = 1.0
    return {"kind": kind, "param": 3, "w_in": np.zeros((3 * d, d)), "w_out": np.zeros((d, d)),
            "w_gu": w_gu, "w_down": w_down, "taps": np.ones((3, d))}


def _run_layer(ar, d, F, M, x):
    m = Model.__new__(Model)
    m.shape, m.ar = _Shape(d, F), ar
    L = LayerState("SE", window=np.zeros((2, d), ar.dt))
    return m.layer_forward(M, L, np.asarray(x, ar.dt), 0)


@pytest.mark.parametrize("i,j,c", [(1, 5, 0), (5, 1, 7), (3, 3, 2)])
def test_mlp_one_hot_closed_form_fp64(i, j, c):
    d, F = 8, 4
    g = np.random.default_rng(i * 31 + j)
    x = g.standard_normal(d) * 3
    M = _mlp_only_layer(d, F, [i], [j], [c])
    got = _run_layer(A64, d, F, M, x) - x
    xn = rmsnorm(x, 1e-6, A64)
    want = np.zeros(d)
    want[c] = xn[i] * expit(xn[i]) * xn[j]
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)
    if i != j:
        # gate and up are not interchangeable: the swapped reading differs
        assert abs(want[c] - xn[j] * expit(xn[j]) * xn[i]) > 1e-6


def test_mlp_several_hidden_units_add():
    d, F = 16, 6
    g = np.random.default_rng(7)
    x = g.standard_normal(d)
    gi, uj, dc = [0, 3, 9, 12, 3, 15], [2, 2, 11, 0, 7, 1], [4, 4, 5, 15, 0, 4]
    M = _mlp_only_layer(d, F, gi, uj, dc)
    got = _run_layer(A64, d, F, M, x) - x
    xn = rmsnorm(x, 1e-6, A64)
    want = np.zeros(d)
    for i, j, c in zip(gi, uj, dc):
        want[c] += xn[i] * expit(xn[i]) * xn[j]
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


def test_mlp_one_hot_bf16_points():
    # bf16 storage mode: xn and the hidden value h are bf16 storage points;
    # the gate/up sums themselves stay float32 (the GPU sums them in fp32)
    d, F = 8, 2
    g = np.random.default_rng(3)
    for trial in range(50):
        x = (g.standard_normal(d) * 2).astype(np.float32)
        M = _mlp_only_layer(d, F, [2], [6], [1])
        got = _run_layer(A32, d, F, M, x)
        xn = round_bf16(rmsnorm(x, 1e-6, A32)).astype(np.float64)
        h = np.float32(round_bf16(np.float32(xn[2] * expit(xn[2]) * xn[6])).ravel()[0])
        want = x.copy()
        want[1] = np.float32(x[1] + h)
        np.testing.assert_allclose(got, want, rtol=2e-6, atol=1e-7)
    # the unrounded hidden value differs from the stored one in most draws,
    # so a missing storage point on h would show up above
    xs = (g.standard_normal((200, d)) * 2).astype(np.float32)
    diffs = 0
    for x in xs:
        xn = round_bf16(rmsnorm(x, 1e-6, A32)).astype(np.float64)
        hv = np.float32(xn[2] * expit(xn[2]) * xn[6])
        diffs += int(round_bf16(hv).ravel()[0] != hv)
    assert diffs > 150
