"""Pins for the oracle's Hyena filters.

* FIR with a unit tap at j is a pure delay by j (special case).
* FIR over a sequence equals numpy.convolve per channel (library routine).
* The modal IIR recurrence equals the explicit convolution with its impulse
  response h[t] = Re sum_m R_m lam_m^t (closed form of a geometric series),
  and with lam = 0 it reduces to y = Re(sum R) z.
"""
import numpy as np

from oracle.model import LayerState, Model
from oracle.numerics import Arith

AR = Arith(np.float64)


class _Shim(Model):
    """Model whose methods are used without a weight set."""

    def __init__(self):
        self.ar = AR


def _run_fir(taps, zs):
    L, d = taps.shape
    st = LayerState("MR", window=np.zeros((L - 1, d)))
    m = _Shim()
    return np.stack([m.fir_step({"taps": taps}, st, z) for z in zs])


def _run_iir(lam, res, zs):
    st = LayerState("LI", s=np.zeros(lam.shape, np.complex128))
    m = _Shim()
    M = {"lam": lam, "res": res}
    return np.stack([m.iir_step(M, st, z) for z in zs])


def test_fir_delta_is_delay():
    g = np.random.default_rng(1)
    d, L, T = 5, 7, 20
    zs = g.standard_normal((T, d))
    for j in range(L):
        taps = np.zeros((L, d))
        taps[j] = 1.0
        y = _run_fir(taps, zs)
        want = np.zeros_like(zs)
        want[j:] = zs[:T - j]
        assert np.array_equal(y, want), j


def test_fir_matches_numpy_convolve():
    g = np.random.default_rng(2)
    d, L, T = 6, 128, 300
    taps = g.standard_normal((L, d))
    zs = g.standard_normal((T, d))
    y = _run_fir(taps, zs)
    for c in range(d):
        ref = np.convolve(zs[:, c], taps[:, c])[:T]
        np.testing.assert_allclose(y[:, c], ref, rtol=1e-12, atol=1e-12)


def test_fir_window_carries_history():
    # splitting a sequence in two with the window carried over changes nothing
    g = np.random.default_rng(3)
    d, L, T = 3, 9, 40
    taps = g.standard_normal((L, d))
    zs = g.standard_normal((T, d))
    full = _run_fir(taps, zs)
    st = LayerState("MR", window=np.zeros((L - 1, d)))
    m = _Shim()
    part = [m.fir_step({"taps": taps}, st, z) for z in zs[:17]]
    saved = st.window.copy()
    assert np.array_equal(saved, np.concatenate([np.zeros((L - 1 - 8, d)), zs[9:17]])[-(L - 1):])
    part += [m.fir_step({"taps": taps}, st, z) for z in zs[17:]]
    assert np.array_equal(np.stack(part), full)


def test_iir_equals_modal_impulse_response():
    g = np.random.default_rng(4)
    d, M, T = 4, 8, 64
    r = g.uniform(0.9, 0.99, (d, M))
    th = g.uniform(-np.pi, np.pi, (d, M))
    lam = r * np.exp(1j * th)
    res = g.standard_normal((d, M)) * 0.25 + 1j * g.standard_normal((d, M)) * 0.25
    zs = g.standard_normal((T, d))
    y_rec = _run_iir(lam, res, zs)
    t = np.arange(T)
    h = np.real(np.einsum("cm,tcm->tc", res, lam[None, :, :] ** t[:, None, None]))   # [T][d]
    y_conv = _run_fir(h, zs)
    np.testing.assert_allclose(y_rec, y_conv, rtol=1e-10, atol=1e-10)


def test_iir_zero_poles():
    g = np.random.default_rng(5)
    d, M = 6, 16
    lam = np.zeros((d, M), np.complex128)
    res = g.standard_normal((d, M)) + 1j * g.standard_normal((d, M))
    zs = g.standard_normal((10, d))
    y = _run_iir(lam, res, zs)
    np.testing.assert_allclose(y, zs * np.real(res.sum(axis=1))[None, :], rtol=1e-13, atol=1e-13)


def test_iir_single_real_pole_geometric():
    # one pole lam = 0.5, residue 1: impulse response 0.5^t
    lam = np.full((1, 1), 0.5 + 0j)
    res = np.ones((1, 1), np.complex128)
    zs = np.zeros((6, 1))
    zs[0, 0] = 1.0
    y = _run_iir(lam, res, zs)
    assert np.allclose(y[:, 0], 0.5 ** np.arange(6))
