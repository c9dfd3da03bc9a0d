"""Operator-level GPU parity at the single-layer sizes (d_model 4096, blocks of
13 tokens, bf16 activations / fp32 state) against the oracle's own filter,
rotary and attention code.

* FIR short (L 7) and medium (L 128), IIR (16 poles): block outputs within
  2e-2 of max |ref| (bf16 outputs); the retained per-position state (FIR
  ext rows, IIR states) within 1e-5 (fp32 state); then commit at a random
  keep and a second block from the sliced state.
* Attention (32 heads x 128 over 8192 cached positions; 8 x 64 over 3000;
  4 x 32 over 700; caches ~ N(0,1)): appended rotated keys / values and the
  block-causal outputs, then commit and a second block.
* Skinny GEMM (tcgen05 path for bf16, SIMT path for f32) at every weight
  shape of the 7B-shaped stack, n = 1, 13, 16.
Edge cases: n = 1, keep = 0, keep = n, window offset > 0, zero initial IIR.
"""
import numpy as np
import pytest

import synth
from gpu_util import book_zero, fir_ext, fir_set_window, rel_err, to_np, torch, up, wrap
from oracle.model import LayerState, Model as OModel, attend, rope
from oracle.numerics import Arith, round_bf16

AR = Arith(np.float32, bf16_points=True)
D = 4096


class _Ops(OModel):
    def __init__(self):
        self.ar = AR


def _abv(seed, n, d):
    return synth.abv_block(seed, n, d, "bf16")


def _f(bits):
    return synth.bf16_bits_to_f32(bits)


@pytest.mark.gpu
@pytest.mark.parametrize("L,pos0", [(7, 40), (128, 300), (7, 2)])
def test_fir_op_block_and_slice(L, pos0):
    # The ring holds the input of position p at row p mod (L-1+n_max): at
    # pos0 = 300 with L = 128 the window wraps around the ring; at pos0 = 2
    # the window reaches before position 0 (zero rows, never written).
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    n_max, d = 13, D
    taps = synth.mixer_params(1, "MR", L, d)["taps"]
    win = synth.layer_state(1, "MR", L, d)["window"].copy()
    win[:max(0, L - 1 - pos0)] = 0.0
    ring = t.zeros((L - 1 + n_max, d), dtype=t.float32, device="cuda")
    fir_set_window(ring, L, n_max, pos0, up(win))
    book = book_zero(t)
    book[0] = pos0
    taps_d = up(taps)
    ops = _Ops()
    st = LayerState("MR", window=win.copy())
    rng = np.random.default_rng(L)
    pos = pos0
    for rnd, n in enumerate((13, 1, 13)):
        abv = _abv(10 + rnd, n, d)
        g = t.empty((n, d), dtype=t.bfloat16, device="cuda")
        evs.evs_op_fir(L, d, n, n_max, evs.EVS_BF16, up(abv), taps_d, ring, book, g)
        a, b, v = _f(abv[:, :d]), _f(abv[:, d:2 * d]), _f(abv[:, 2 * d:])
        recs, gref = [], []
        work = LayerState("MR", window=st.window.copy())
        for i in range(n):
            z = b[i] * v[i]
            y = ops.fir_step({"taps": taps}, work, z)
            gref.append(round_bf16(a[i] * y))
            recs.append(work.window.copy())
        assert rel_err(to_np(g), np.stack(gref)) <= 2e-2
        ext = fir_ext(to_np(ring), L, n_max, pos, n)
        for i in range(n):
            assert np.array_equal(ext[i + 1:i + L], recs[i]), (rnd, i)
        keep = int(rng.integers(0, n + 1)) if rnd != 1 else 0
        evs.evs_op_commit(book, keep, n)
        if keep:
            st.window = recs[keep - 1]
        pos += keep
        assert int(book[0].item()) == pos


@pytest.mark.gpu
def test_iir_op_block_and_slice():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    n_max, d, M = 13, D, 16
    prm = synth.mixer_params(2, "LI", M, d)
    s0 = synth.layer_state(2, "LI", M, d)["s"]
    st0 = t.zeros((n_max, d, M, 2), dtype=t.float32, device="cuda")
    st1 = t.zeros_like(st0)
    st0[4] = up(s0).view(d, M, 2)
    book = book_zero(t)
    book[4] = 4                      # current state: bank 0 slot 4
    lam, res = up(prm["lam"]), up(prm["res"])
    ops = _Ops()
    cur = s0.astype(np.complex64)
    rng = np.random.default_rng(3)
    for rnd, n in enumerate((13, 13, 1, 13)):
        abv = _abv(20 + rnd, n, d)
        g = t.empty((n, d), dtype=t.bfloat16, device="cuda")
        evs.evs_op_iir(M, d, n, n_max, evs.EVS_BF16, up(abv), lam, res, st0, st1, book, g)
        a, b, v = _f(abv[:, :d]), _f(abv[:, d:2 * d]), _f(abv[:, 2 * d:])
        work = LayerState("LI", s=cur.copy())
        recs, gref = [], []
        for i in range(n):
            y = ops.iir_step({"lam": prm["lam"], "res": prm["res"]}, work, b[i] * v[i])
            gref.append(round_bf16(a[i] * y))
            recs.append(work.s.copy())
        assert rel_err(to_np(g), np.stack(gref)) <= 2e-2
        bank, slot = int(book[3].item()), int(book[4].item())
        S = to_np(st1 if bank == 0 else st0)
        for i in range(n):
            got = S[i, :, :, 0] + 1j * S[i, :, :, 1]
            assert rel_err(got.real, recs[i].real) <= 1e-5 and rel_err(got.imag, recs[i].imag) <= 1e-5
        keep = [0, n, 1, int(rng.integers(0, n + 1))][rnd]
        evs.evs_op_commit(book, keep, n)
        if keep:
            cur = recs[keep - 1]
        bk = book.cpu().numpy()
        assert (bk[3], bk[4]) == ((1 - bank, keep - 1) if keep else (bank, slot))


@pytest.mark.gpu
@pytest.mark.parametrize("H,Dh,P,chunk", [(32, 128, 8192, 256), (8, 64, 9210, 64), (8, 64, 3066, 64),
                                           (4, 32, 700, 32)])
def test_attention_op_cache(H, Dh, P, chunk):
    # Dh 128 / 64: the tensor-map kernel, fused with rotary / append / fold
    # for caches above 8192 positions, between the rotary and combine kernels
    # at or below (Dh 64: one box per key row; the first block straddles a
    # split boundary: 9216 and 3072, both at span 256); Dh 32: the SIMT
    # kernel on bf16 caches
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    n_max = 13
    d = H * Dh
    ctx = P + 3 * n_max
    ls = synth.layer_state(3, "ATT", 0, d, P=P, n_heads=H, head_dim=Dh)
    kc = t.zeros((H, ctx, Dh), dtype=t.bfloat16, device="cuda")
    vc = t.zeros_like(kc)
    kc[:, :P] = up(ls["k"]).transpose(0, 1)
    vc[:, :P] = up(ls["v"]).transpose(0, 1)
    Kf = np.zeros((ctx, H, Dh), np.float32)
    Vf = np.zeros((ctx, H, Dh), np.float32)
    Kf[:P], Vf[:P] = _f(ls["k"]), _f(ls["v"])
    book = book_zero(t)
    book[0] = P
    scratch = t.empty(evs.evs_op_attention_scratch_bytes(H, Dh, ctx, chunk, n_max), dtype=t.uint8, device="cuda")
    pos = P
    for rnd, (n, keep) in enumerate(((13, 5), (1, 1), (13, 13))):
        qkv = _abv(30 + rnd, n, d)
        g = t.empty((n, d), dtype=t.bfloat16, device="cuda")
        evs.evs_op_attention(H, Dh, n, n_max, ctx, chunk, 10000.0, evs.EVS_BF16, up(qkv), kc, vc, book, g, scratch)
        qf = _f(qkv)
        outs = []
        for i in range(n):
            q = round_bf16(rope(qf[i, :d].reshape(H, Dh), pos + i, 10000.0, AR))
            k = round_bf16(rope(qf[i, d:2 * d].reshape(H, Dh), pos + i, 10000.0, AR))
            Kf[pos + i], Vf[pos + i] = k, qf[i, 2 * d:].reshape(H, Dh)
        for i in range(n):
            q = round_bf16(rope(qf[i, :d].reshape(H, Dh), pos + i, 10000.0, AR))
            outs.append(attend(q, Kf[:pos + i + 1], Vf[:pos + i + 1], AR).reshape(d))
        assert rel_err(to_np(g), np.stack(outs)) <= 2e-2
        kg = to_np(kc[:, pos:pos + n]).transpose(1, 0, 2)
        vg = to_np(vc[:, pos:pos + n]).transpose(1, 0, 2)
        assert rel_err(kg, Kf[pos:pos + n]) <= 1e-2 and np.array_equal(vg, Vf[pos:pos + n])
        evs.evs_op_commit(book, keep, n)
        pos += keep
        assert int(book[0].item()) == pos


@pytest.mark.gpu
@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 4096), (22016, 4096), (4096, 11008), (512, 4096), (128, 64)])
def test_gemm_op_tensor_cores(N, K):
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    g = np.random.default_rng(N + K)
    Wb = synth._to_bf16_bits_trunc(g.standard_normal((N, K), dtype=np.float32) * 0.02)
    W = up(Wb)
    scratch = t.empty(evs.evs_op_gemm_scratch_bytes(N, K, evs.EVS_BF16), dtype=t.uint8, device="cuda")
    for n in (1, 13, 16):
        Xb = synth._to_bf16_bits_trunc(g.standard_normal((n, K), dtype=np.float32))
        y = t.empty((n, N), dtype=t.float32, device="cuda")
        evs.evs_op_gemm(W, up(Xb), N, K, n, evs.EVS_BF16, y, scratch)
        ref = _f(Xb).astype(np.float64) @ _f(Wb).astype(np.float64).T
        assert rel_err(to_np(y), ref) <= 1e-4, (N, K, n)
        assert int(scratch[-256:].view(t.int32)[0].item()) == 0   # no pipeline timeout


@pytest.mark.gpu
def test_gemm_op_simt_f32_ragged():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    g = np.random.default_rng(5)
    for N, K, n in ((192, 64, 5), (16, 64, 1), (300, 100, 16)):
        W = g.standard_normal((N, K)).astype(np.float32)
        X = g.standard_normal((n, K)).astype(np.float32)
        scratch = t.empty(evs.evs_op_gemm_scratch_bytes(N, K, evs.EVS_F32), dtype=t.uint8, device="cuda")
        y = t.empty((n, N), dtype=t.float32, device="cuda")
        evs.evs_op_gemm(up(W), up(X), N, K, n, evs.EVS_F32, y, scratch)
        assert rel_err(to_np(y), X.astype(np.float64) @ W.astype(np.float64).T) <= 1e-5
