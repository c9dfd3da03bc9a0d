"""Accept / probs kernels against the oracle's rule, bit-exact.

Given identical p, q, drafts and float32 uniforms, the GPU's accepted
length and output token must equal the oracle's exactly (both take the
u*q < p decision in float32 and sample on the same integer ladder).
Cases: vocab 16 and 512, n = 1 (native: bonus sample only) to 16, greedy
and sampled, q == p (all accepted), q disjoint from p (first draft always
rejected, residual == p), drafts outside the vocabulary (rejected, with the
rejection's output token), ties in greedy argmax, rows without mass.
The top-k distribution kernel is checked against the oracle's top-k softmax
up to vocab 8192, with ties straddling the top-k cut.
"""
import numpy as np
import pytest

from gpu_util import to_np, torch, up
from oracle.sampling import GREEDY, SAMPLE, TWO24, accept, argmax_low, sample, topk_probs


def _gpu_accept(evs, p, q, d, u, mode):
    t = torch()
    n, V = p.shape
    acc = t.full((1,), -7, dtype=t.int32, device="cuda")
    tok = t.full((1,), -7, dtype=t.int32, device="cuda")
    qd = up(q.astype(np.float32)) if q is not None and q.size else t.zeros((1, V), dtype=t.float32, device="cuda")
    dd = up(np.asarray(d, np.int32)) if len(d) else t.zeros(1, dtype=t.int32, device="cuda")
    evs.evs_accept(up(p.astype(np.float32)), qd, dd, up(u.astype(np.float32)), n, V, mode, acc, tok)
    return int(acc.item()), int(tok.item())


def _dist(g, V, k=None):
    x = g.standard_normal(V).astype(np.float32) * 2
    return topk_probs(x, 1.0, k or 0, dtype=np.float32)


@pytest.mark.gpu
@pytest.mark.parametrize("V", [16, 512])
def test_accept_bit_exact_random(V):
    import hybrid_ssm_attention_gb300 as evs
    g = np.random.default_rng(V)
    cases = 0
    for trial in range(300):
        n = int(g.integers(1, 17))
        k = int(g.choice([0, 4, 1])) if V > 16 else 0
        p = np.stack([_dist(g, V, k) for _ in range(n)])
        kind = trial % 4
        if kind == 0:
            q = p[:-1].copy()                                   # identity drafter
        elif kind == 1:
            q = np.stack([_dist(g, V, k) for _ in range(n - 1)]) if n > 1 else np.zeros((0, V), np.float32)
        else:
            q = np.stack([0.5 * p[i] + 0.5 * _dist(g, V, k) for i in range(n - 1)]).astype(np.float32) \
                if n > 1 else np.zeros((0, V), np.float32)
        d = [int(g.choice(V, p=q[i] / q[i].sum())) for i in range(n - 1)]
        if kind == 3 and n > 2:
            d[1] = V + 3 if trial % 8 == 3 else -1            # outside the vocabulary
        u = g.random(n).astype(np.float32)
        for mode in (SAMPLE, GREEDY):
            got = _gpu_accept(evs, p, q, d, u, mode)
            dd = [x if 0 <= x < V else 0 for x in d]
            want = accept(p, q, dd, u, mode)
            if any(not (0 <= x < V) for x in d):
                # an out-of-range draft is rejected: if the rule had not
                # stopped before it, the round ends there with the rule's
                # rejection output (argmax p_a, or a sample of the residual
                # (p_a - q_{a+1})^+, falling back to p_a without mass)
                bad = next(i for i, x in enumerate(d) if not (0 <= x < V))
                if want[0] < bad:
                    assert got == want, (trial, mode, got, want)
                else:
                    a = bad
                    if mode == GREEDY:
                        tok = argmax_low(p[a])
                    else:
                        r = np.maximum(p[a] - q[a], np.float32(0)).astype(np.float32)
                        mass = sum(int(np.floor(np.float64(x) * TWO24)) for x in r)
                        tok = sample(r if mass > 0 else p[a], np.float32(u[n - 1]))
                    assert got == (a, tok), (trial, mode, got, (a, tok))
                cases += 1
                continue
            assert got == want, (trial, mode, n, got, want)
            cases += 1
            if kind == 0 and mode == SAMPLE:
                assert got[0] == n - 1
    assert cases > 400


@pytest.mark.gpu
def test_accept_disjoint_rejects_and_residual_is_p():
    import hybrid_ssm_attention_gb300 as evs
    V = 16
    p = np.zeros((3, V), np.float32)
    p[0, 8:] = 1 / 8
    p[1:, :] = 1 / V
    q = np.zeros((2, V), np.float32)
    q[:, :8] = 1 / 8
    for uu in np.linspace(0, 0.999, 17, dtype=np.float32):
        u = np.array([0.1, 0.2, uu], np.float32)
        got = _gpu_accept(evs, p, q, [2, 3], u, SAMPLE)
        assert got == accept(p, q, [2, 3], u, SAMPLE)
        assert got[0] == 0 and 8 <= got[1] < 16


@pytest.mark.gpu
def test_greedy_ties_lowest_index():
    import hybrid_ssm_attention_gb300 as evs
    V = 512
    p = np.zeros((2, V), np.float32)
    p[0, [7, 300, 9]] = 5.0
    p[1, [511, 3]] = 2.0
    got = _gpu_accept(evs, p, np.zeros((1, V), np.float32), [7], np.zeros(2, np.float32), GREEDY)
    assert got == (1, 3)
    got = _gpu_accept(evs, p, np.zeros((1, V), np.float32), [9], np.zeros(2, np.float32), GREEDY)
    assert got == (0, 7)


@pytest.mark.gpu
def test_probs_topk_support_and_values():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    g = np.random.default_rng(9)
    for V, n in ((512, 13), (16, 5), (100, 1)):
        L = (g.standard_normal((n, V)) * 3).astype(np.float32)
        L[0, :5] = L[0, 0]                       # ties
        for T, k in ((1.0, 4), (0.5, 1), (2.0, 0), (1.0, V), (1.0, V - 1)):
            p = t.empty((n, V), dtype=t.float32, device="cuda")
            evs.evs_probs(up(L), n, V, T, k, p)
            want = np.stack([topk_probs(r, T, k, dtype=np.float32) for r in L])
            got = to_np(p)
            assert np.array_equal(got > 0, want > 0), (V, T, k)
            assert np.abs(got - want).max() <= 2e-6


@pytest.mark.gpu
def test_probs_nan_logits_rank_below_every_number():
    # NaN entries stay out of a top-k support while the row holds k numbers
    # (the oracle's stable descending sort puts them last)
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    g = np.random.default_rng(29)
    for V in (16, 512, 4096):
        n = 4
        L = (g.standard_normal((n, V)) * 3).astype(np.float32)
        L[0, :3] = np.nan
        L[1, g.choice(V, V // 4, replace=False)] = np.nan
        L[2, V - 1] = np.nan
        L[3, 1::2] = np.nan
        for T, k in ((1.0, 4), (1.0, 1), (0.7, 5)):
            p = t.empty((n, V), dtype=t.float32, device="cuda")
            evs.evs_probs(up(L), n, V, T, k, p)
            want = np.stack([topk_probs(r, T, k, dtype=np.float32) for r in L])
            got = to_np(p)
            assert not np.isnan(got).any()
            assert np.array_equal(got > 0, want > 0), (V, T, k)
            assert np.abs(got - want).max() <= 2e-6


@pytest.mark.gpu
def test_probs_topk_large_vocab_and_ties_at_the_cut():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    g = np.random.default_rng(19)
    for V in (1000, 4096, 8192):
        n = 5
        L = (g.standard_normal((n, V)) * 3).astype(np.float32)
        # row 1: a block of equal values straddling every cut below
        L[1, 100:140] = 7.0
        L[1, 3000 % V] = 9.0
        # row 2: coarse values so that many ties exist everywhere
        L[2] = np.round(L[2])
        # row 3: -0 and +0 are equal values
        L[3, :] = -1.0
        L[3, 5], L[3, 9] = -0.0, 0.0
        for T, k in ((1.0, 4), (1.0, 1), (0.7, 37), (1.0, 100), (1.3, V - 1), (1.0, V // 2)):
            p = t.empty((n, V), dtype=t.float32, device="cuda")
            evs.evs_probs(up(L), n, V, T, k, p)
            want = np.stack([topk_probs(r, T, k, dtype=np.float32) for r in L])
            got = to_np(p)
            assert np.array_equal(got > 0, want > 0), (V, T, k)
            assert np.abs(got - want).max() <= 2e-6, (V, T, k)


@pytest.mark.gpu
def test_sample_rows_without_mass_and_unit_uniform():
    # a sampled row with no integer mass (all zero) yields its argmax; a
    # uniform of 1.0 (outside [0, 1)) lands on the last entry with mass
    import hybrid_ssm_attention_gb300 as evs
    V = 64
    p = np.zeros((1, V), np.float32)
    got = _gpu_accept(evs, p, np.zeros((0, V), np.float32), [], np.array([0.5], np.float32), SAMPLE)
    assert got == (0, 0)
    p[0, 17] = 0.25
    p[0, 40] = 0.75
    got = _gpu_accept(evs, p, np.zeros((0, V), np.float32), [], np.array([1.0], np.float32), SAMPLE)
    assert got == (0, 40)
    got = _gpu_accept(evs, p, np.zeros((0, V), np.float32), [], np.array([np.float32(1 - 2 ** -24)], np.float32),
                      SAMPLE)
    assert got == accept(p, None, [], np.array([np.float32(1 - 2 ** -24)]), SAMPLE) == (0, 40)
