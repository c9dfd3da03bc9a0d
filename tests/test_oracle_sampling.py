"""Pins for the oracle's distribution, sampler and accept rule.

* top-k with k = V is the plain softmax (scipy.special.softmax, a library
  routine); k = 1 is one-hot at the argmax; ties go to the lower index.
* sample(): hand-built ladders - all mass on one index, uniform mass, u at
  0 and just below 1, a zero-weight entry is never drawn.
* accept(): p == q accepts every draft; greedy hand cases; the exact
  losslessness of the rule by brute-force enumeration over every draft pair
  at vocab 16, gamma 2 (first emitted token ~ p_0; first two emitted tokens
  ~ p_0(x) p(y | x)) to 1e-12 (preprint abstract: "in exact arithmetic the
  scheme preserves the target distribution"); and a Monte-Carlo check that
  accept() with float32 uniforms realises the enumerated law.
"""
import numpy as np
import pytest
import scipy.special
import scipy.stats

import synth
from oracle.model import Model
from oracle.numerics import Arith
from oracle.sampling import GREEDY, SAMPLE, accept, argmax_low, sample, topk_probs


def test_topk_full_is_softmax():
    g = np.random.default_rng(0)
    for T in (1.0, 0.7, 2.0):
        l = g.standard_normal(512).astype(np.float64) * 3
        p = topk_probs(l, T, 0, dtype=np.float64)
        np.testing.assert_allclose(p, scipy.special.softmax(l / T), rtol=1e-12, atol=1e-15)
        p = topk_probs(l, T, 512, dtype=np.float64)
        np.testing.assert_allclose(p, scipy.special.softmax(l / T), rtol=1e-12, atol=1e-15)


def test_topk_k1_and_ties():
    l = np.array([0.5, 2.0, 2.0, -1.0, 2.0], np.float32)
    p = topk_probs(l, 1.0, 1)
    assert p.tolist() == [0, 1, 0, 0, 0]
    p = topk_probs(l, 1.0, 2)
    np.testing.assert_allclose(p, [0, 0.5, 0.5, 0, 0])
    p = topk_probs(l, 1.0, 4)
    e = np.exp(np.float32(0.5) - np.float32(2.0))
    np.testing.assert_allclose(p, np.array([e, 1, 1, 0, 1]) / (3 + e), rtol=1e-6)


def test_topk4_support():
    g = np.random.default_rng(1)
    l = g.standard_normal(512).astype(np.float32)
    p = topk_probs(l, 1.0, 4)
    assert (p > 0).sum() == 4
    assert set(np.flatnonzero(p)) == set(np.argsort(-l)[:4])
    assert abs(p.sum() - 1) < 1e-6


def test_sample_hand_cases():
    one = np.zeros(8, np.float32)
    one[5] = 1.0
    for u in (0.0, 0.3, np.float32(1 - 2 ** -24)):
        assert sample(one, u) == 5
    uni = np.full(4, 0.25, np.float32)           # W = 2^22 each, S = 2^24
    assert sample(uni, 0.0) == 0
    assert sample(uni, 0.25 - 2 ** -24) == 0
    assert sample(uni, 0.25) == 1
    assert sample(uni, 0.5) == 2
    assert sample(uni, np.float32(1 - 2 ** -24)) == 3
    w = np.array([0.5, 0.0, 0.5], np.float32)    # zero weight never drawn
    assert sample(w, 0.5 - 2 ** -24) == 0 and sample(w, 0.5) == 2
    tiny = np.array([2 ** -30, 1.0], np.float32)  # mass below 2^-24 is dropped
    assert sample(tiny, 0.0) == 1
    with pytest.raises(ValueError):
        sample(np.zeros(3, np.float32), 0.1)


def test_sample_unnormalised_weights():
    # the ladder only needs relative integer mass: w and w / 2 draw alike
    g = np.random.default_rng(2)
    w = g.random(16).astype(np.float32) / 16
    for u in g.random(200).astype(np.float32):
        assert sample(w, u) == sample(w / np.float32(2), u)


def test_accept_p_equals_q_accepts_all():
    g = np.random.default_rng(3)
    V, gamma = 16, 6
    p = g.dirichlet(np.ones(V), size=gamma + 1).astype(np.float32)
    q = p[:gamma].copy()
    for _ in range(100):
        drafts = [int(g.choice(V, p=p[i] / p[i].sum())) for i in range(gamma)]
        u = g.random(gamma + 1).astype(np.float32)
        a, tok = accept(p, q, drafts, u, SAMPLE)
        assert a == gamma
        assert tok == sample(p[gamma], u[gamma])


def test_accept_greedy_cases():
    V = 5
    logits = np.array([[0, 3, 1, 0, 0], [2, 0, 0, 0, 2], [0, 0, 0, 0, 9]], np.float32)
    q = np.zeros((2, V), np.float32)
    assert accept(logits, q, [1, 0], np.zeros(3), GREEDY) == (2, 4)   # all accepted, bonus argmax
    assert accept(logits, q, [1, 4], np.zeros(3), GREEDY) == (1, 0)   # tie at row 1 -> index 0
    assert accept(logits, q, [2, 0], np.zeros(3), GREEDY) == (0, 1)


def test_accept_sample_rejects_and_resamples_residual():
    # q puts mass on token 0 where p has none: always rejected; residual = p
    p = np.array([[0.0, 0.5, 0.5], [0.2, 0.3, 0.5]], np.float32)
    q = np.array([[1.0, 0.0, 0.0]], np.float32)
    for u in (0.0, 0.4, 0.99):
        a, tok = accept(p, q, [0], np.float32([0.5, u]), SAMPLE)
        assert a == 0 and tok == (1 if u < 0.5 else 2)


# ---------------------------------------------------------------- enumeration

def _tiny_target():
    shape = synth.tiny()
    W = synth.make_weights(shape, 0)
    m = Model(shape, W, Arith(np.float64))
    st = m.new_state(64)
    for t in synth.prompt(shape, 0, 6)[:-1]:
        m.step(st, int(t))
    pending = int(synth.prompt(shape, 0, 6)[-1])
    return shape, m, st, pending


def _probs(m, st, toks):
    logits, _ = m.verify(st, toks)
    return np.stack([topk_probs(l, 1.0, 0, dtype=np.float64) for l in logits])


@pytest.fixture(scope="module")
def enum_setup():
    shape, m, st, pending = _tiny_target()
    V = shape.vocab
    q = synth.fixed_logit_drafter(0, 2, V).astype(np.float64)
    q /= q.sum(axis=1, keepdims=True)            # exact distributions for the enumeration
    P = {}
    for d1 in range(V):
        for d2 in range(V):
            P[d1, d2] = _probs(m, st, [pending, d1, d2])
    nxt = {x: _probs(m, st, [pending, x])[1] for x in range(V)}
    return V, q, P, nxt


def _residual(p, q):
    r = np.maximum(p - q, 0.0)
    s = r.sum()
    return r / s if s > 0 else None


def test_enumeration_lossless(enum_setup):
    V, q, P, nxt = enum_setup
    p0 = P[0, 0][0]
    first = np.zeros(V)
    joint = np.zeros((V, V))
    acc_law = np.zeros(3)
    for d1 in range(V):
        for d2 in range(V):
            w = q[0, d1] * q[1, d2]
            p_0, p_1, p_2 = P[d1, d2]
            a1 = min(1.0, p_0[d1] / q[0, d1])
            r1 = _residual(p_0, q[0])
            if r1 is not None:
                first += w * (1 - a1) * r1
                joint += w * (1 - a1) * np.outer(r1, np.ones(V)) * np.stack([nxt[x] for x in range(V)])
            acc_law[0] += w * (1 - a1)
            first[d1] += w * a1
            a2 = min(1.0, p_1[d2] / q[1, d2])
            r2 = _residual(p_1, q[1])
            if r2 is not None:
                joint[d1] += w * a1 * (1 - a2) * r2
            joint[d1, d2] += w * a1 * a2
            acc_law[1] += w * a1 * (1 - a2)
            acc_law[2] += w * a1 * a2
    np.testing.assert_allclose(first, p0, atol=1e-12)
    want = p0[:, None] * np.stack([nxt[x] for x in range(V)])
    np.testing.assert_allclose(joint, want, atol=1e-12)
    assert abs(acc_law.sum() - 1) < 1e-12


def test_accept_monte_carlo_matches_enumeration(enum_setup):
    V, q64, P, nxt = enum_setup
    q = q64.astype(np.float32)
    P32 = {k: v.astype(np.float32) for k, v in P.items()}
    p0 = P[0, 0][0]
    g = np.random.default_rng(7)
    N = 60000
    du = g.random((N, 2))
    u = g.random((N, 3)).astype(np.float32)
    first = np.zeros(V)
    for r in range(N):
        d1 = synth.draw_from(q[0], du[r, 0])
        d2 = synth.draw_from(q[1], du[r, 1])
        a, tok = accept(P32[d1, d2], q, [d1, d2], u[r], SAMPLE)
        x = d1 if a >= 1 else tok
        first[x] += 1
    exp = p0 * N
    mask = exp > 5
    chi2 = (((first - exp) ** 2)[mask] / exp[mask]).sum()
    pval = scipy.stats.chi2.sf(chi2, mask.sum() - 1)
    assert pval > 1e-4, (chi2, pval)


def test_argmax_low():
    assert argmax_low([1, 3, 3, 2]) == 1
    assert argmax_low([5]) == 0
