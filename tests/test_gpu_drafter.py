"""The drafter-side Markov-head kernel (evs_markov_draft) against the oracle.

Each slot's q equals the oracle's top-k softmax of the trunk row plus the
Markov row of the previous token (support exact, values within 2e-6); each
draft equals the oracle's decision on that same q and uniform (integer-ladder
sample, bit-exact) or, greedy, the oracle's argmax; the greedy chain equals
the oracle's whole chain.  Vocab 16, 510, 512, 1000, 2000 and 8192; top_k
0, 1, 4, 7 and V - 1 (top_k 1 .. 8: the one-warp kernel for V <= 1024 and
V % 4 == 0, the merged-list kernel otherwise; other top_k: the radix
select); T 1, 0.8 and 0.7; integer logits whose ties straddle the top-k cut;
a one-hot Markov chain; a pending token outside the vocabulary; a slot whose
logits are all NaN (empty support: q zero, draft 0).
The drafter trunk stand-in (one attention layer at d_model 1024) scores the
gamma slots in one verify pass whose rows feed the kernel.
"""
import numpy as np
import pytest

import synth
from gpu_util import to_np, torch, up
from oracle.drafter import markov_draft
from oracle.sampling import GREEDY, SAMPLE, argmax_low, sample, topk_probs


def _gpu(evs, trunk, M, prev, u, T, k, mode):
    t = torch()
    gamma, V = trunk.shape
    d = t.full((gamma,), -7, dtype=t.int32, device="cuda")
    q = t.empty((gamma, V), dtype=t.float32, device="cuda")
    pv = t.tensor([prev], dtype=t.int32, device="cuda")
    evs.evs_markov_draft(up(trunk), up(M), V, pv, up(u.astype(np.float32)), gamma, T, k, mode, d, q)
    return [int(x) for x in d.cpu().numpy()], to_np(q)


@pytest.mark.gpu
@pytest.mark.parametrize("V", [16, 510, 512, 1000, 2000, 8192])
def test_markov_draft_matches_oracle(V):
    import hybrid_ssm_attention_gb300 as evs
    g = np.random.default_rng(V + 1)
    gamma = 12
    M = (g.standard_normal((V, V)) * 2).astype(np.float32)
    for trial in range(4 if V == 8192 else 10):
        trunk = (g.standard_normal((gamma, V)) * 2).astype(np.float32)
        prev = int(g.integers(0, V))
        u = g.random(gamma).astype(np.float32)
        for T, k in ((1.0, 4), (0.7, 0), (1.0, V - 1), (0.8, 7), (1.0, 1)):
            for mode in (SAMPLE, GREEDY):
                d, q = _gpu(evs, trunk, M, prev, u, T, k, mode)
                p = prev
                for i in range(gamma):
                    logits = trunk[i] + M[p]
                    ref = topk_probs(logits, T, k, dtype=np.float32)
                    assert np.array_equal(q[i] > 0, ref > 0), (trial, T, k, mode, i)
                    assert np.abs(q[i] - ref).max() <= 2e-6
                    want = argmax_low(logits) if mode == GREEDY else sample(q[i], u[i])
                    assert d[i] == want, (trial, T, k, mode, i)
                    p = d[i]
                if mode == GREEDY:
                    assert d == markov_draft(trunk, M, prev, u, T, k, GREEDY)[0]


@pytest.mark.gpu
@pytest.mark.parametrize("V", [16, 510, 1000, 2000, 8192])
def test_markov_draft_ties_take_lower_indices(V):
    # small integer logits: most entries tie with others, and ties straddle
    # the top-k cut; the support keeps the lower indices (the oracle's
    # stable order) for every k, in both kernels (k <= 8 and k = V - 1)
    import hybrid_ssm_attention_gb300 as evs
    g = np.random.default_rng(V + 3)
    gamma = 12
    M = g.integers(-2, 3, (V, V)).astype(np.float32)
    for k in (1, 3, 4, 8, V - 1):
        trunk = g.integers(-1, 2, (gamma, V)).astype(np.float32)
        prev = int(g.integers(0, V))
        u = g.random(gamma).astype(np.float32)
        for mode in (SAMPLE, GREEDY):
            d, q = _gpu(evs, trunk, M, prev, u, 1.0, k, mode)
            want_d, want_q = markov_draft(trunk, M, prev, u, 1.0, k, GREEDY) if mode == GREEDY else (None, None)
            p = prev
            for i in range(gamma):
                logits = trunk[i] + M[p]
                ref = topk_probs(logits, 1.0, k, dtype=np.float32)
                assert np.array_equal(q[i] > 0, ref > 0), (k, mode, i)
                assert np.abs(q[i] - ref).max() <= 2e-6
                want = argmax_low(logits) if mode == GREEDY else sample(q[i], u[i])
                assert d[i] == want, (k, mode, i)
                p = d[i]
            if mode == GREEDY:
                assert d == want_d


@pytest.mark.gpu
@pytest.mark.parametrize("V", [16, 512, 1000, 2000])
def test_markov_draft_nan_logits_stay_out_of_the_support(V):
    # NaN trunk entries rank below every number: q and the sampled drafts
    # match the oracle's rule on the same logits (top_k 1, 4, 8)
    import hybrid_ssm_attention_gb300 as evs
    g = np.random.default_rng(V + 7)
    gamma = 12
    M = (g.standard_normal((V, V)) * 2).astype(np.float32)
    for k in (1, 4, 8):
        trunk = (g.standard_normal((gamma, V)) * 2).astype(np.float32)
        trunk[:, g.choice(V, V // 4, replace=False)] = np.nan
        trunk[0, :2] = np.nan
        prev = int(g.integers(0, V))
        u = g.random(gamma).astype(np.float32)
        d, q = _gpu(evs, trunk, M, prev, u, 1.0, k, SAMPLE)
        assert not np.isnan(q).any()
        p = prev
        for i in range(gamma):
            ref = topk_probs(trunk[i] + M[p], 1.0, k, dtype=np.float32)
            assert np.array_equal(q[i] > 0, ref > 0), (k, i)
            assert np.abs(q[i] - ref).max() <= 2e-6
            assert d[i] == sample(q[i], u[i]), (k, i)
            p = d[i]


@pytest.mark.gpu
@pytest.mark.parametrize("V", [16, 512, 1000, 2000])
def test_markov_draft_row_without_a_number(V):
    # a slot whose logits are all NaN has an empty support (top_k 1 .. 8):
    # its q row is zero and its draft 0, so the next slot reads Markov row 0
    import hybrid_ssm_attention_gb300 as evs
    g = np.random.default_rng(V + 11)
    gamma, bad = 6, 2
    M = (g.standard_normal((V, V)) * 2).astype(np.float32)
    for k in (1, 4, 8):
        for mode in (GREEDY, SAMPLE):
            trunk = (g.standard_normal((gamma, V)) * 2).astype(np.float32)
            trunk[bad] = np.nan
            u = g.random(gamma).astype(np.float32)
            prev = int(g.integers(0, V))
            d, q = _gpu(evs, trunk, M, prev, u, 1.0, k, mode)
            assert d[bad] == 0 and not q[bad].any(), (k, mode)
            p = prev
            for i in range(gamma):
                if i != bad:
                    ref = topk_probs(trunk[i] + M[p], 1.0, k, dtype=np.float32)
                    assert np.array_equal(q[i] > 0, ref > 0), (k, mode, i)
                    assert np.abs(q[i] - ref).max() <= 2e-6
                    want = sample(q[i], u[i]) if mode == SAMPLE else argmax_low(trunk[i] + M[p])
                    assert d[i] == want, (k, mode, i)
                p = d[i]


@pytest.mark.gpu
def test_markov_draft_chain_and_bad_pending_token():
    import hybrid_ssm_attention_gb300 as evs
    V, gamma = 64, 10
    f = [(7 * a + 5) % V for a in range(V)]
    M = np.full((V, V), -3.0, np.float32)
    for a in range(V):
        M[a, f[a]] = 3.0
    z = np.zeros((gamma, V), np.float32)
    d, _ = _gpu(evs, z, M, 9, np.zeros(gamma), 1.0, 4, GREEDY)
    assert d == markov_draft(z, M, 9, np.zeros(gamma), 1.0, 4, GREEDY)[0]
    x, want = 9, []
    for _ in range(gamma):
        x = f[x]
        want.append(x)
    assert d == want
    d, _ = _gpu(evs, z, M, V + 5, np.zeros(gamma), 1.0, 4, GREEDY)  # outside: row 0
    assert d[0] == f[0]


@pytest.mark.gpu
def test_trunk_standin_feeds_the_markov_head():
    # the trunk stand-in scores gamma slots in one verify pass; its rows feed
    # the head kernel, whose q and drafts match the oracle's rule on them
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    shape = synth.drafter_trunk_standin()
    m = evs.Model(shape, synth.make_weights(shape, 5))
    st = evs.State(m, 256)
    gamma, V = shape.gamma, shape.vocab
    toks = t.tensor(synth.prompt(shape, 5, gamma), dtype=t.int32, device="cuda")
    trunk = t.empty((gamma, V), dtype=t.float32, device="cuda")
    evs.evs_verify_block(st, toks, gamma, trunk)
    evs.evs_commit(st, 1)
    M = synth.markov_matrix(5, V)
    u = synth.uniforms(5, 1, gamma)[0]
    d = t.zeros(gamma, dtype=t.int32, device="cuda")
    q = t.empty((gamma, V), dtype=t.float32, device="cuda")
    evs.evs_markov_draft(trunk, up(M), V, toks[:1], up(u), gamma, 1.0, 4, evs.EVS_SAMPLE, d, q)
    T_, Q, D = to_np(trunk), to_np(q), [int(x) for x in d.cpu().numpy()]
    p = int(toks[0].item())
    for i in range(gamma):
        ref = topk_probs(T_[i] + M[p], 1.0, 4, dtype=np.float32)
        assert np.array_equal(Q[i] > 0, ref > 0) and np.abs(Q[i] - ref).max() <= 2e-6
        assert D[i] == sample(Q[i], u[i])
        p = D[i]
    assert st.check() == 0
