"""GPU parity on the fp32 tiny hybrid (vocab 16, d 64; FIR short 4, IIR 8 poles,
attention 2x32; gamma 4), through the C ABI, against the fp64 oracle.

Tolerance: 1e-5 of max |ref| per tensor (fp32 path).  Checked: prompt
prefill, block-verify logits, the per-position retained state of every
layer (FIR windows, IIR states, KV rows), greedy accept/commit rounds
token for token against oracle native greedy decoding, GPU speculative ==
GPU native (bitwise logits at every emitted position), and the sampled
path's probabilities.
"""
import numpy as np
import pytest

import synth
from gpu_util import fir_ext, rel_err, to_np, torch, wrap

TOL = 1e-5


def _setup(ctx=256, seed=0):
    import hybrid_ssm_attention_gb300 as evs
    from oracle.model import Model as OModel
    from oracle.numerics import Arith
    shape = synth.tiny()
    W = synth.make_weights(shape, seed)
    m = evs.Model(shape, W)
    st = evs.State(m, ctx)
    om = OModel(shape, W, Arith(np.float64))
    return evs, shape, W, m, st, om, om.new_state(ctx)


def _verify(evs, st, toks, V):
    t = torch()
    tt = t.tensor(np.asarray(toks, np.int32), device="cuda")
    lg = t.empty((len(toks), V), dtype=t.float32, device="cuda")
    evs.evs_verify_block(st, tt, len(toks), lg)
    return lg, tt


def _check_retained(shape, st, book, records, n):
    """GPU per-position state after a verify vs the oracle records."""
    d = shape.d_model
    for li, (kind, param) in enumerate(shape.layers):
        v = st.view(li)
        if kind in ("SE", "MR"):
            L = param
            ext = fir_ext(to_np(wrap(v.fir_ring, (L - 1 + v.n_max, d))), L, v.n_max, book["pos"], n)
            for i in range(n):
                assert rel_err(ext[i + 1:i + L], records[i].layers[li].window) <= TOL
        elif kind == "LI":
            M = param
            S = to_np(wrap(v.iir_all[1 - book["iir_bank"]], (v.n_max, d, M, 2)))
            for i in range(n):
                ref = records[i].layers[li].s
                got = S[i, :, :, 0] + 1j * S[i, :, :, 1]
                assert rel_err(got.real, ref.real) <= TOL and rel_err(got.imag, ref.imag) <= TOL
        else:
            H, Dh = shape.n_heads, shape.head_dim
            K = to_np(wrap(v.k_cache, (H, v.ctx_max, Dh)))
            Vc = to_np(wrap(v.v_cache, (H, v.ctx_max, Dh)))
            P = book["pos"]
            ref = records[n - 1].layers[li]
            assert rel_err(K[:, :P + n, :].transpose(1, 0, 2), ref.K[:P + n]) <= TOL
            assert rel_err(Vc[:, :P + n, :].transpose(1, 0, 2), ref.V[:P + n]) <= TOL


@pytest.mark.gpu
def test_tiny_prefill_verify_retained_state_and_commit():
    from oracle.model import Model as OModel
    evs, shape, W, m, st, om, ost = _setup()
    nb = shape.n_block
    prompt = [int(x) for x in synth.prompt(shape, 0, 32)]
    rng = np.random.default_rng(0)
    for s0 in range(0, len(prompt) - 1, nb):
        chunk = prompt[s0:min(s0 + nb, len(prompt) - 1)]
        lg, _ = _verify(evs, st, chunk, shape.vocab)
        ref, rec = om.verify(ost, chunk)
        assert rel_err(to_np(lg), ref) <= TOL
        book = st.book()
        assert book["pending_n"] == len(chunk)
        _check_retained(shape, st, book, rec, len(chunk))
        keep = len(chunk) if s0 + nb < len(prompt) - 1 else int(rng.integers(0, len(chunk) + 1))
        evs.evs_commit(st, keep)
        ost = OModel.commit(ost, rec, keep)
        book = st.book()
        assert book["pos"] == ost.pos and book["pending_n"] == 0
    # every keep in [0, n] on one block: slice == native state after keep steps
    block = [1, 2, 3, 4, 5][:nb]
    for keep in range(nb + 1):
        st2 = evs.State(m, 256)
        st.clone_into(st2)
        lg, _ = _verify(evs, st2, block, shape.vocab)
        ref, rec = om.verify(ost, block)
        assert rel_err(to_np(lg), ref) <= TOL
        evs.evs_commit(st2, keep)
        ost2 = OModel.commit(ost, rec, keep)
        # the next verify reads the sliced state: its logits pin the slice
        lg2, _ = _verify(evs, st2, [7], shape.vocab)
        ref2, _ = om.verify(ost2, [7])
        assert rel_err(to_np(lg2), ref2) <= TOL, keep
        assert st2.check() == 0
        st2.close()


@pytest.mark.gpu
def test_tiny_greedy_rounds_match_oracle_native():
    from oracle.decode import native_generate, prefill
    evs, shape, W, m, st, om, ost = _setup()
    t = torch()
    prompt = [int(x) for x in synth.prompt(shape, 0, 32)]
    pend = prefill(om, ost, prompt)
    nat, _ = native_generate(om, ost.copy(), pend, 40)
    nb = shape.n_block
    for s0 in range(0, len(prompt) - 1, nb):
        chunk = prompt[s0:min(s0 + nb, len(prompt) - 1)]
        _verify(evs, st, chunk, shape.vocab)
        evs.evs_commit(st, len(chunk))
    q = synth.fixed_logit_drafter(0, shape.gamma, shape.vocab)
    du = synth.draft_uniforms(0, 64, shape.gamma)
    acc = t.zeros(1, dtype=t.int32, device="cuda")
    tok = t.zeros(1, dtype=t.int32, device="cuda")
    out, rnd = [], 0
    while len(out) < 40:
        drafts = [synth.draw_from(q[i], du[rnd, i]) for i in range(shape.gamma)]
        lg, tt = _verify(evs, st, [pend] + drafts, shape.vocab)
        evs.evs_accept(lg, None, tt[1:], None, nb, shape.vocab, evs.EVS_GREEDY, acc, tok)
        evs.evs_commit_dev(st, acc)
        a, x = int(acc.item()), int(tok.item())
        out += drafts[:a] + [x]
        pend = x
        rnd += 1
    assert out[:40] == nat[:40]
    assert st.check() == 0


@pytest.mark.gpu
def test_tiny_gpu_spec_equals_gpu_native_bitwise():
    """GPU speculative rounds reproduce GPU native decoding exactly: every
    emitted position's logits row is bit-identical (block size does not
    change a row's arithmetic), hence identical greedy tokens."""
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    shape = synth.tiny()
    W = synth.make_weights(shape, 0)
    m = evs.Model(shape, W)
    prompt = [int(x) for x in synth.prompt(shape, 0, 32)]
    nb = shape.n_block

    def prefill(st):
        for s0 in range(0, len(prompt) - 1, nb):
            chunk = prompt[s0:min(s0 + nb, len(prompt) - 1)]
            _verify(evs, st, chunk, shape.vocab)
            evs.evs_commit(st, len(chunk))

    nat_st = evs.State(m, 256)
    prefill(nat_st)
    pend = prompt[-1]
    nat_tok, nat_lg = [], []
    for _ in range(40):
        lg, _ = _verify(evs, nat_st, [pend], shape.vocab)
        evs.evs_commit(nat_st, 1)
        row = to_np(lg)[0]
        nat_lg.append(row)
        pend = int(np.argmax(row))
        nat_tok.append(pend)
    sp = evs.State(m, 256)
    prefill(sp)
    pend = prompt[-1]
    q = synth.fixed_logit_drafter(1, shape.gamma, shape.vocab)
    du = synth.draft_uniforms(1, 64, shape.gamma)
    acc = t.zeros(1, dtype=t.int32, device="cuda")
    tok = t.zeros(1, dtype=t.int32, device="cuda")
    out, rows, rnd = [], [], 0
    while len(out) < 40:
        drafts = [synth.draw_from(q[i], du[rnd, i]) for i in range(shape.gamma)]
        if rnd % 3 == 0:   # mix in identity-drafted rounds
            k = len(out)
            drafts = (nat_tok[k:k + shape.gamma] + [0] * shape.gamma)[:shape.gamma]
        lg, tt = _verify(evs, sp, [pend] + drafts, shape.vocab)
        evs.evs_accept(lg, None, tt[1:], None, nb, shape.vocab, evs.EVS_GREEDY, acc, tok)
        evs.evs_commit_dev(sp, acc)
        a, x = int(acc.item()), int(tok.item())
        L = to_np(lg)
        rows += [L[i] for i in range(a + 1)]
        out += drafts[:a] + [x]
        pend = x
        rnd += 1
    assert out[:40] == nat_tok
    for i in range(40):
        assert np.array_equal(rows[i].view(np.uint32), nat_lg[i].view(np.uint32)), i


@pytest.mark.gpu
def test_tiny_sampled_probs_match_oracle():
    from oracle.sampling import topk_probs
    evs, shape, W, m, st, om, ost = _setup()
    t = torch()
    toks = [int(x) for x in synth.prompt(shape, 2, shape.n_block)]
    lg, _ = _verify(evs, st, toks, shape.vocab)
    ref, _ = om.verify(ost, toks)
    for T, k in ((1.0, 0), (0.7, 4), (1.3, 1), (1.0, 16)):
        p = t.empty_like(lg)
        evs.evs_probs(lg, len(toks), shape.vocab, T, k, p)
        want = np.stack([topk_probs(r, T, k, dtype=np.float64) for r in ref])
        got = to_np(p)
        assert rel_err(got, want) <= 1e-5
        assert np.array_equal(got > 0, want > 0)
