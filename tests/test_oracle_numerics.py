"""Pins for the oracle's bf16 rounding: hand cases from the IEEE layout and
agreement with torch's float32 -> bfloat16 conversion (a library routine)."""
import numpy as np
import torch

from oracle.numerics import Arith, round_bf16


def f(bits):
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def test_hand_cases():
    one = 1.0
    ulp = 2.0 ** -7                       # bf16 spacing in [1, 2)
    assert round_bf16(one)[()] == one
    assert round_bf16(one + ulp / 2)[()] == one              # tie -> even (1.0)
    assert round_bf16(one + 3 * ulp / 2)[()] == one + 2 * ulp  # tie -> even (1 + 2ulp)
    assert round_bf16(one + ulp / 2 + 2.0 ** -20)[()] == one + ulp
    assert round_bf16(-(one + ulp / 4))[()] == -one
    assert np.isinf(round_bf16(f(0x7F7FFFFF))[()])           # rounds up past max bf16
    assert np.isnan(round_bf16(np.float32(np.nan))[()])
    assert round_bf16(np.float32(np.inf))[()] == np.inf


def test_matches_torch_bfloat16():
    g = np.random.default_rng(0)
    x = np.concatenate([
        g.standard_normal(200000).astype(np.float32) * 10.0,
        # exact ties: low 16 bits = 0x8000 on finite values
        ((g.standard_normal(20000).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000))
         | np.uint32(0x8000)).view(np.float32),
        np.float32([0.0, -0.0, 1e-40, -1e-40, 3.0e38]),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = round_bf16(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_arith_points():
    a32 = Arith(np.float32, bf16_points=True)
    assert a32.r(1.0 + 2.0 ** -9) == 1.0
    a64 = Arith(np.float64)
    assert a64.r(1.0 + 2.0 ** -30) == 1.0 + 2.0 ** -30


def test_matvec_orders_agree():
    # the two summation orders are the same sum: exact on integer-valued
    # data (every partial sum representable), and within float64 rounding
    # of each other on random data
    g = np.random.default_rng(4)
    W = g.integers(-50, 50, size=(37, 200)).astype(np.float64)
    x = g.integers(-50, 50, size=200).astype(np.float64)
    a, b = Arith(np.float64), Arith(np.float64, order="k64_reversed")
    assert np.array_equal(a.mv(W, x), b.mv(W, x))
    assert np.array_equal(a.mv(W, x), np.array([sum(int(W[i, k]) * int(x[k]) for k in range(200))
                                                for i in range(37)], dtype=np.float64))
    W = g.standard_normal((64, 300))
    x = g.standard_normal(300)
    np.testing.assert_allclose(b.mv(W, x), a.mv(W, x), rtol=1e-12, atol=1e-12)
    c = Arith(np.float32, order="k64_reversed")
    assert c.mv(W.astype(np.float32), x.astype(np.float32)).dtype == np.float32
