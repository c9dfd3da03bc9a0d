"""Pins for the oracle's drafter-side Markov head.

* With a zero trunk, the first slot's distribution is the softmax of the
  Markov row picked by the pending token: scipy.special.softmax of M[prev] / T
  (a library routine), and not of the column M[:, prev] (M is asymmetric).
* With a zero Markov matrix, every slot's distribution is the softmax of
  its trunk row, whatever the previous tokens.
* With a zero trunk and one-hot rows M[a] peaking at f(a), greedy drafts
  follow the chain f(prev), f(f(prev)), ... (the previous draft feeds the
  next slot).
* Sampled drafts are the integer-ladder sample of each slot's q with its
  own uniform; over a grid of uniforms the first draft's frequencies match
  q_1 (inverse-CDF property).
"""
import numpy as np
from scipy.special import softmax

from oracle.drafter import markov_draft
from oracle.sampling import GREEDY, SAMPLE


def test_zero_trunk_first_slot_is_softmax_of_markov_row():
    g = np.random.default_rng(1)
    V, gamma = 32, 5
    M = (g.standard_normal((V, V)) * 2).astype(np.float32)
    assert not np.allclose(M, M.T)
    for prev in (0, 7, 31):
        for T in (1.0, 0.5):
            _, q = markov_draft(np.zeros((gamma, V), np.float32), M, prev, np.zeros(gamma), T, 0, GREEDY)
            np.testing.assert_allclose(q[0], softmax(M[prev].astype(np.float64) / T), rtol=2e-6, atol=1e-9)
            assert np.abs(q[0] - softmax(M[:, prev].astype(np.float64) / T)).max() > 1e-3


def test_zero_markov_is_trunk_softmax():
    g = np.random.default_rng(2)
    V, gamma = 40, 6
    trunk = (g.standard_normal((gamma, V)) * 3).astype(np.float32)
    d, q = markov_draft(trunk, np.zeros((V, V), np.float32), 3, g.random(gamma), 1.0, 0, SAMPLE)
    np.testing.assert_allclose(q, softmax(trunk.astype(np.float64), axis=1), rtol=2e-6, atol=1e-9)
    dg, _ = markov_draft(trunk, np.zeros((V, V), np.float32), 3, np.zeros(gamma), 1.0, 0, GREEDY)
    assert dg == [int(np.argmax(r)) for r in trunk]


def test_greedy_drafts_follow_the_markov_chain():
    V, gamma = 16, 8
    f = [(5 * a + 3) % V for a in range(V)]
    M = np.full((V, V), -4.0, np.float32)
    for a in range(V):
        M[a, f[a]] = 4.0
    d, q = markov_draft(np.zeros((gamma, V), np.float32), M, 2, np.zeros(gamma), 1.0, 4, GREEDY)
    want, x = [], 2
    for _ in range(gamma):
        x = f[x]
        want.append(x)
    assert d == want
    assert all((qi > 0).sum() == 4 for qi in q)


def test_sampled_first_draft_frequencies_match_q():
    g = np.random.default_rng(3)
    V, gamma = 8, 2
    trunk = g.standard_normal((gamma, V)).astype(np.float32)
    M = g.standard_normal((V, V)).astype(np.float32)
    _, q = markov_draft(trunk, M, 1, np.zeros(gamma), 1.0, 0, SAMPLE)
    N = 4096
    counts = np.zeros(V)
    for k in range(N):
        u = np.array([(k + 0.5) / N, 0.5], np.float32)
        d, _ = markov_draft(trunk, M, 1, u, 1.0, 0, SAMPLE)
        counts[d[0]] += 1
    np.testing.assert_allclose(counts / N, q[0], atol=2.0 / N)
