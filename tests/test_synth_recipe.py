"""The seeded input generators follow the stated input recipe.

Both sides of every parity test read their inputs from `synth`, so a slip in
it (a wrong standard deviation, a shifted layer pattern, a keep law off by
one) would go unseen by parity.  These checks pin the recipe itself: the
7B-shaped layer pattern, the distribution parameters of weights, filter taps,
poles, residues, state, noise and commit lengths (sample statistics against
tolerances of several standard errors), the prompt alphabet, determinism per
seed, the bf16 truncation used to make bf16 draws, and the inverse-CDF draft
draw.
"""
import numpy as np
import pytest

import synth


def test_7b_layer_pattern():
    # attention iff i mod 6 = 5; the Hyena layers cycle SE 7, MR 128, LI 16
    sh = synth.stack_7b()
    kinds = [k for k, _ in sh.layers]
    assert len(kinds) == 32
    assert [i for i, k in enumerate(kinds) if k == synth.ATT] == [5, 11, 17, 23, 29]
    hy = [lp for lp in sh.layers if lp[0] != synth.ATT]
    assert hy == [[(synth.SE, 7), (synth.MR, 128), (synth.LI, 16)][j % 3] for j in range(27)]
    assert (sh.d_model, sh.d_ffn, sh.n_heads, sh.head_dim, sh.vocab, sh.gamma) == (4096, 11008, 32, 128, 512, 12)
    assert sh.n_block == 13 and sh.dtype == "bf16"


def _small(dtype="bf16"):
    return synth.ModelShape(name="recipe", vocab=256, d_model=256, layers=[(synth.SE, 7), (synth.MR, 128),
                            (synth.LI, 16), (synth.ATT, 0)], n_heads=2, head_dim=128, d_ffn=512, gamma=12,
                            dtype=dtype)


def _within(x, want, rel):
    return abs(x - want) <= rel * want


def test_weights_shapes_and_distributions():
    sh = _small()
    W = synth.make_weights(sh, 3)
    d, F, V = 256, 512, 256
    assert W["embed"].shape == (V, d) and W["lm_head"].shape == (V, d) and W["embed"].dtype == np.uint16
    dense = []
    for L, (kind, param) in zip(W["layers"], sh.layers):
        assert L["w_in"].shape == (3 * d, d) and L["w_out"].shape == (d, d)
        assert L["w_gu"].shape == (2 * F, d) and L["w_down"].shape == (d, F)
        dense.append(synth.bf16_bits_to_f32(L["w_gu"]).ravel())
        if kind in (synth.SE, synth.MR):
            t = L["taps"]
            assert t.shape == (param, d) and t.dtype == np.float32
            # N(0, 1/sqrt(L)): sample std within 5% (>= 1,792 draws)
            assert _within(float(t.std()), 1 / np.sqrt(param), 0.05), kind
            assert abs(float(t.mean())) < 4 / np.sqrt(param) / np.sqrt(t.size)
        elif kind == synth.LI:
            lam, res = L["lam"], L["res"]
            assert lam.shape == (d, param) and lam.dtype == np.complex64
            r = np.abs(lam)
            assert r.min() >= 0.9 - 1e-6 and r.max() <= 0.999 + 1e-6
            # |lambda| ~ U(0.9, 0.999), arg ~ U(-pi, pi): means and spreads
            assert abs(float(r.mean()) - 0.9495) < 0.003
            th = np.angle(lam)
            assert abs(float(th.mean())) < 0.1 and _within(float(th.std()), np.pi / np.sqrt(3), 0.03)
            assert _within(float(res.real.std()), 0.25, 0.04) and _within(float(res.imag.std()), 0.25, 0.04)
        else:
            assert "taps" not in L and "lam" not in L
    w = np.concatenate(dense)
    # N(0, 0.02) truncated to bf16 (toward zero, at most 2^-8 relative): std
    # within 1% of 0.02 over 1M draws, mean near 0
    assert _within(float(w.std()), 0.02, 0.01)
    assert abs(float(w.mean())) < 1e-4


def test_f32_weights_and_determinism():
    sh = _small("f32")
    a, b, c = synth.make_weights(sh, 9), synth.make_weights(sh, 9), synth.make_weights(sh, 10)
    assert a["embed"].dtype == np.float32
    assert np.array_equal(a["embed"], b["embed"]) and np.array_equal(a["layers"][2]["lam"], b["layers"][2]["lam"])
    assert not np.array_equal(a["embed"], c["embed"])
    # weights_f32 of a bf16 dict widens exactly; of an f32 dict it is the dict
    wb = synth.make_weights(_small(), 9)
    wf = synth.weights_f32(wb)
    assert np.array_equal(wf["layers"][0]["w_in"].view(np.uint32) >> 16, wb["layers"][0]["w_in"].astype(np.uint32))
    assert synth.weights_f32(a) is a


def test_bf16_truncation_keeps_the_high_half():
    g = np.random.default_rng(1)
    x = (g.standard_normal(10000) * 3).astype(np.float32)
    bits = synth._to_bf16_bits_trunc(x)
    y = synth.bf16_bits_to_f32(bits)
    assert np.array_equal(y.view(np.uint32), x.view(np.uint32) & 0xFFFF0000)
    assert np.all(np.abs(y) <= np.abs(x)) and np.all(np.sign(y) == np.sign(x))
    assert np.all(np.abs(x - y) <= np.abs(x) * 2.0 ** -7)


def test_prompts_uniforms_and_noise():
    p = synth.prompt(synth.stack_7b(), 4, 4096)
    assert p.dtype == np.int32 and set(np.unique(p)) == set(synth.ACGT_IDS)
    counts = np.bincount(p, minlength=85)[list(synth.ACGT_IDS)]
    assert counts.min() > 4096 / 4 - 4 * np.sqrt(4096 * 3 / 16)
    assert np.array_equal(p, synth.prompt(synth.stack_7b(), 4, 4096))
    t = synth.prompt(synth.tiny(), 4, 1000)
    assert t.min() >= 0 and t.max() < 16
    u = synth.uniforms(2, 300, 13)
    assert u.shape == (300, 13) and u.dtype == np.float32 and u.min() >= 0 and u.max() < 1
    assert abs(float(u.mean()) - 0.5) < 0.02
    z = synth.logit_noise(5, 4, 12, 512)
    assert z.shape == (4, 12, 512) and _within(float(z.std()), 0.5, 0.02)
    m = synth.markov_matrix(6, 512)
    assert _within(float(m.std()), 1.0, 0.01)


def test_keep_draws_laws():
    n = 13
    k = synth.keep_draws(7, 20000, n, kind="uniform")
    assert k.min() == 0 and k.max() == n and abs(float(k.mean()) - n / 2) < 0.1
    k = synth.keep_draws(7, 20000, n, kind="geometric")
    assert k.min() == 1 and k.max() == n
    # Geometric(1/3) on {1, 2, ...} clipped to n: P(K = 1) = 1/3,
    # E K = sum_{j=0}^{n-1} (2/3)^j = 3 (1 - (2/3)^n)
    assert abs(float(np.mean(k == 1)) - 1 / 3) < 0.015
    assert abs(float(k.mean()) - 3 * (1 - (2 / 3) ** n)) < 0.08
    assert abs(float(np.mean(k == n)) - (2 / 3) ** (n - 1)) < 0.01


@pytest.mark.parametrize("u,want", [(0.0, 0), (0.24, 0), (0.25, 1), (0.49, 1), (0.5, 2), (0.999, 2)])
def test_draw_from_is_the_inverse_cdf(u, want):
    # dyadic masses: the interval edges 0.25 and 0.5 are exact; entry j holds
    # [c_{j-1}, c_j)
    q = np.array([0.25, 0.25, 0.5], np.float32)
    assert synth.draw_from(q, u) == want
    # a zero-mass entry is never drawn
    assert synth.draw_from(np.array([0.25, 0.0, 0.75], np.float32), u) != 1


def test_synthesised_state_recipe():
    sh = _small()
    s = synth.synth_state(sh, 11, 300)
    assert s["P"] == 300
    se, mr, li, att = s["layers"]
    assert se["window"].shape == (6, 256) and mr["window"].shape == (127, 256)
    assert _within(float(mr["window"].std()), 1.0, 0.02)
    assert li["s"].shape == (256, 16) and li["s"].dtype == np.complex64
    assert _within(float(li["s"].real.std()), np.sqrt(2), 0.04) and _within(float(li["s"].imag.std()), np.sqrt(2), 0.04)
    assert att["k"].shape == (300, 2, 128) and att["k"].dtype == np.uint16
    kf = synth.bf16_bits_to_f32(att["k"])
    assert _within(float(kf.std()), 1.0, 0.02)
    e = synth.synth_state(sh, 11, 0)["layers"][3]
    assert e["k"].shape == (0, 2, 128)
    kh, vh = synth.kv_head(3, 5, 1000, 128)
    assert kh.shape == (1000, 128) and not np.array_equal(kh, vh)
    assert np.array_equal(kh, synth.kv_head(3, 5, 1000, 128)[0])
