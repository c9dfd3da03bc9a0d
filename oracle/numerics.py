"""bf16 rounding for the oracle (test infrastructure only).

bf16 keeps the top 16 bits of an IEEE-754 binary32 value: sign, 8 exponent
bits, 7 fraction bits.  Round-to-nearest-even on the dropped 16 bits:
add 0x7FFF plus the lowest kept bit, then clear the low half.  NaNs stay
NaN (quiet bit forced); infinities pass through; overflow rounds to inf,
as the IEEE definition of RNE requires.
"""
import numpy as np


def round_bf16(x) -> np.ndarray:
    """float32 array whose values are ``x`` rounded to bf16 (RNE)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = a.view(np.uint32).astype(np.uint64)
    is_nan = np.isnan(a)
    keep_lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + keep_lsb) & np.uint64(0xFFFF0000)
    out = bits.astype(np.uint32).view(np.float32).reshape(a.shape)
    if is_nan.any():
        out = out.copy()
        out[is_nan] = np.float32(np.nan)
    return out


class Arith:
    """Arithmetic mode of the oracle.

    ``Arith(np.float64)``                 - exact-ish reference (tiny config).
    ``Arith(np.float32, bf16_points=True)`` - fp32 with values rounded to bf16
        wherever the bf16 path stores them: GEMM inputs (normed activations,
        gated mixer output, attention output, MLP hidden), the in-projection
        outputs a|b|v and q|k|v, and the rotated q and k (k is what the KV
        cache holds).  Weights are bf16 values already.

    ``order`` picks the summation order of the matrix-vector products:
    ``"blas"`` (default) is numpy's ``W @ x``; ``"k64_reversed"`` forms the
    partial products of 64-column blocks of W (each by ``W @ x``) and adds
    them one at a time from the last block to the first.  Both are valid
    orders of the same sum in the arithmetic dtype; comparing them measures
    how far rounding alone moves the oracle's own results.
    """

    ORDERS = ("blas", "k64_reversed")

    def __init__(self, dtype=np.float64, bf16_points: bool = False, order: str = "blas"):
        if order not in self.ORDERS:
            raise ValueError(f"order must be one of {self.ORDERS}")
        self.dt = np.dtype(dtype)
        self.bf16 = bool(bf16_points)
        self.cdt = np.complex128 if self.dt == np.float64 else np.complex64
        self.order = order

    def mv(self, W, x):
        """W [N][K] times x [K] in the arithmetic dtype, in this mode's order."""
        if self.order == "blas":
            return W @ x
        K = W.shape[1]
        acc = None
        for b in reversed(range((K + 63) // 64)):
            part = W[:, 64 * b:64 * b + 64] @ x[64 * b:64 * b + 64]
            acc = part if acc is None else acc + part
        return acc.astype(self.dt, copy=False)

    def r(self, x):
        """A bf16 storage point (identity unless bf16_points)."""
        x = np.asarray(x, dtype=self.dt)
        if self.bf16:
            return round_bf16(x).astype(self.dt)
        return x
