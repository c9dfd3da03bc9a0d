"""Pins for the oracle's hybrid stack, block verify, commit and decode loops.

* Zero mixer and MLP weights: logits = W_lm RMSNorm(E[token]) whatever the
  history (special case of the residual stack).
* Block verify rows == successive native steps; the state committed at
  every keep in [0, n] equals the native state after keep steps, exactly
  (discussion post, "What we implemented": slicing to the accepted boundary
  with zero recomputation).
* Greedy speculative output == native output token for token, with a
  random fixed-logit drafter and with the identity drafter; the identity
  drafter has every draft accepted (model card, "Library" example;
  discussion post, identity-drafter overhead).
* Sampled speculative decoding with drafter q == target p accepts all.
"""
import numpy as np
import pytest

import synth
from oracle.decode import identity_greedy_drafter, native_generate, prefill, spec_generate
from oracle.model import ATT, LI, Model, rmsnorm
from oracle.numerics import Arith
from oracle.sampling import GREEDY, SAMPLE, topk_probs

AR = Arith(np.float64)


@pytest.fixture(scope="module")
def tiny():
    shape = synth.tiny()
    W = synth.make_weights(shape, 0)
    return shape, W, Model(shape, W, AR)


def _state_equal(a, b):
    assert a.pos == b.pos
    for x, y in zip(a.layers, b.layers):
        if x.window is not None:
            assert np.array_equal(x.window, y.window)
        if x.s is not None:
            assert np.array_equal(x.s, y.s)
        if x.K is not None:
            assert x.length == y.length
            assert np.array_equal(x.K[:x.length], y.K[:y.length])
            assert np.array_equal(x.V[:x.length], y.V[:y.length])


def test_zero_mixers_reduce_to_embedding_head(tiny):
    shape, W, _ = tiny
    Z = {"embed": W["embed"], "lm_head": W["lm_head"], "dtype": "f32", "layers": []}
    for L in W["layers"]:
        M = dict(L)
        for k in ("w_in", "w_out", "w_gu", "w_down"):
            M[k] = np.zeros_like(L[k])
        Z["layers"].append(M)
    m = Model(shape, Z, AR)
    st = m.new_state(16)
    for t in (3, 7, 1, 15):
        got = m.step(st, t)
        want = W["lm_head"].astype(np.float64) @ rmsnorm(W["embed"][t], shape.norm_eps, AR)
        np.testing.assert_allclose(got, want, rtol=1e-13)


def test_verify_rows_are_native_steps_and_commit_slices(tiny):
    shape, W, m = tiny
    st = m.new_state(64)
    pend = prefill(m, st, synth.prompt(shape, 0, 10))
    toks = [pend, 3, 9, 0, 12]
    logits, rec = m.verify(st, toks)
    ref = st.copy()
    for i, t in enumerate(toks):
        np.testing.assert_array_equal(logits[i], m.step(ref, t))
    for keep in range(len(toks) + 1):
        got = Model.commit(st, rec, keep)
        nat = st.copy()
        for t in toks[:keep]:
            m.step(nat, t)
        _state_equal(got, nat)
        # the source state is untouched by verify (rows < P of the KV unchanged)
        assert got.pos == st.pos + keep


def test_commit_rejects_bad_keep(tiny):
    shape, W, m = tiny
    st = m.new_state(16)
    _, rec = m.verify(st, [1, 2])
    with pytest.raises(ValueError):
        Model.commit(st, rec, 3)
    with pytest.raises(ValueError):
        Model.commit(st, rec, -1)


def test_kv_capacity_error(tiny):
    shape, W, m = tiny
    st = m.new_state(2)
    m.step(st, 1)
    m.step(st, 2)
    with pytest.raises(ValueError):
        m.step(st, 3)


def _drafter_fixed(shape, rounds):
    q = synth.fixed_logit_drafter(0, shape.gamma, shape.vocab)
    du = synth.draft_uniforms(0, rounds, shape.gamma)

    def drafter(emitted, rnd):
        return [synth.draw_from(q[i], du[rnd, i]) for i in range(shape.gamma)], q
    return drafter


def test_greedy_spec_equals_native(tiny):
    shape, W, m = tiny
    prompt = synth.prompt(shape, 0, 32)
    n_tok = 40
    st = m.new_state(128)
    pend = prefill(m, st, prompt)
    nat, _ = native_generate(m, st.copy(), pend, n_tok)
    for drafter in (_drafter_fixed(shape, 64), identity_greedy_drafter(nat, shape.gamma, shape.vocab)):
        spec, acc, _ = spec_generate(m, st.copy(), pend, n_tok, shape.gamma, drafter)
        assert spec[:n_tok] == nat
    _, acc, _ = spec_generate(m, st.copy(), pend, n_tok, shape.gamma,
                              identity_greedy_drafter(nat, shape.gamma, shape.vocab))
    assert all(a == shape.gamma for a in acc)


def test_final_state_after_spec_equals_native(tiny):
    shape, W, m = tiny
    prompt = synth.prompt(shape, 0, 32)
    st = m.new_state(128)
    pend = prefill(m, st, prompt)
    spec, acc, st_spec = spec_generate(m, st.copy(), pend, 23, shape.gamma, _drafter_fixed(shape, 64))
    # replay natively: every emitted token but the last (still pending) was consumed
    consumed = sum(a + 1 for a in acc)
    assert consumed == len(spec)
    nat = st.copy()
    seq = [pend] + spec
    for t in seq[:consumed]:
        m.step(nat, t)
    _state_equal(st_spec, nat)


def test_sample_with_q_equal_p_accepts_all(tiny):
    shape, W, m = tiny
    st = m.new_state(128)
    pend = prefill(m, st, synth.prompt(shape, 1, 8))
    U = synth.uniforms(1, 16, shape.n_block)
    du = synth.draft_uniforms(1, 16, shape.gamma)

    def drafter(emitted, rnd):
        # q_i := p_{i-1} along its own drafted path (identity drafter, sampling)
        work = st_box[0].copy()
        tok = pend_box[0]
        d, q = [], []
        for i in range(shape.gamma):
            p = topk_probs(m.step(work, tok), 1.0, 0, dtype=np.float32)
            x = synth.draw_from(p, du[rnd, i])
            d.append(x)
            q.append(p)
            tok = x
        return d, np.stack(q)

    st_box, pend_box = [st.copy()], [pend]
    out = []
    for rnd in range(4):
        drafts, q = drafter(out, rnd)
        logits, rec = m.verify(st_box[0], [pend_box[0]] + drafts)
        P = np.stack([topk_probs(l, 1.0, 0, dtype=np.float32) for l in logits])
        from oracle.sampling import accept
        a, tok = accept(P, q, drafts, U[rnd], SAMPLE)
        assert a == shape.gamma
        st_box[0] = Model.commit(st_box[0], rec, a + 1)
        pend_box[0] = tok


def test_bf16_points_mode_runs_and_is_close():
    shape = synth.single_layer(LI, 16, d_model=256, d_ffn=512, vocab=64, gamma=4, n_heads=2, head_dim=128)
    W = synth.weights_f32(synth.make_weights(shape, 5))
    m64 = Model(shape, W, Arith(np.float64))
    m32 = Model(shape, W, Arith(np.float32, bf16_points=True))
    s64, s32 = m64.new_state(8), m32.new_state(8)
    for t in (1, 2, 3):
        a, b = m64.step(s64, t), m32.step(s32, t)
        assert np.max(np.abs(a - b)) <= 2e-2 * np.max(np.abs(a))
