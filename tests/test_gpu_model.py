"""bf16 stacks through the C ABI (tensor-core GEMMs, split-K partials,
graphs with programmatic dependent launch) against the fp32 oracle with
bf16 storage points; tolerance 2e-2 of max |ref| on logits.

* small 6-layer bf16 stack (d 256): prefill, block verify, commit; GPU
  speculative == GPU native, bitwise, at every emitted position.
* 7B-shaped stack (32 layers, d 4096, F 11008, vocab 512, gamma 12), at
  full size from a synthesised state at context 1024: teacher-forced block
  logits vs the oracle's 13 native steps; greedy decisions compared where
  the oracle's top-2 gap exceeds 4x the observed logit error (non-ties).
"""
import numpy as np
import pytest

import synth
from gpu_util import rel_err, to_np, torch, up, wrap

TOL = 2e-2


def small_shape():
    return synth.ModelShape(name="small-bf16", vocab=128, d_model=256,
                            layers=[("SE", 7), ("MR", 128), ("LI", 16), ("SE", 7), ("MR", 32), ("ATT", 0)],
                            n_heads=2, head_dim=128, d_ffn=512, gamma=12, dtype="bf16", attn_chunk=64)


def _verify(evs, st, toks, V):
    t = torch()
    tt = t.tensor(np.asarray(toks, np.int32), device="cuda")
    lg = t.empty((len(toks), V), dtype=t.float32, device="cuda")
    evs.evs_verify_block(st, tt, len(toks), lg)
    return lg, tt


@pytest.mark.gpu
def test_small_bf16_stack_matches_oracle():
    import hybrid_ssm_attention_gb300 as evs
    from oracle.model import Model as OModel
    from oracle.numerics import Arith
    shape = small_shape()
    W = synth.make_weights(shape, 11)
    m = evs.Model(shape, W)
    st = evs.State(m, 512)
    om = OModel(shape, synth.weights_f32(W), Arith(np.float32, bf16_points=True))
    ost = om.new_state(512)
    prompt = [int(x) for x in synth.prompt(shape, 11, 100)]
    nb = shape.n_block
    rng = np.random.default_rng(1)
    for s0 in range(0, len(prompt), nb):
        chunk = prompt[s0:s0 + nb]
        lg, _ = _verify(evs, st, chunk, shape.vocab)
        ref, rec = om.verify(ost, chunk)
        assert rel_err(to_np(lg), ref) <= TOL, s0
        keep = len(chunk) if s0 + nb < len(prompt) else int(rng.integers(0, len(chunk) + 1))
        evs.evs_commit(st, keep)
        ost = OModel.commit(ost, rec, keep)
    assert st.check() == 0
    assert st.book()["pos"] == ost.pos


@pytest.mark.gpu
@pytest.mark.parametrize("graphs", [True, False])
def test_small_bf16_spec_equals_native_bitwise(graphs):
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    shape = small_shape()
    W = synth.make_weights(shape, 12)
    m = evs.Model(shape, W)
    prompt = [int(x) for x in synth.prompt(shape, 12, 40)]
    nb = shape.n_block

    def prefill(st):
        st.use_graphs(graphs)
        for s0 in range(0, len(prompt) - 1, nb):
            chunk = prompt[s0:min(s0 + nb, len(prompt) - 1)]
            _verify(evs, st, chunk, shape.vocab)
            evs.evs_commit(st, len(chunk))

    nat = evs.State(m, 512)
    prefill(nat)
    pend, ntok, nlg = prompt[-1], [], []
    for _ in range(60):
        lg, _ = _verify(evs, nat, [pend], shape.vocab)
        evs.evs_commit(nat, 1)
        row = to_np(lg)[0]
        nlg.append(row)
        pend = int(np.argmax(row))
        ntok.append(pend)
    sp = evs.State(m, 512)
    prefill(sp)
    pend = prompt[-1]
    acc = t.zeros(1, dtype=t.int32, device="cuda")
    tok = t.zeros(1, dtype=t.int32, device="cuda")
    g = np.random.default_rng(5)
    out, rows, rnd = [], [], 0
    while len(out) < 60:
        k = len(out)
        drafts = (ntok[k:k + shape.gamma] + [0] * shape.gamma)[:shape.gamma]
        cut = int(g.integers(0, shape.gamma + 1))          # corrupt the tail: partial acceptance
        drafts = drafts[:cut] + [int(x) for x in g.integers(0, shape.vocab, shape.gamma - cut)]
        lg, tt = _verify(evs, sp, [pend] + drafts, shape.vocab)
        evs.evs_accept(lg, None, tt[1:], None, nb, shape.vocab, evs.EVS_GREEDY, acc, tok)
        evs.evs_commit_dev(sp, acc)
        a, x = int(acc.item()), int(tok.item())
        L = to_np(lg)
        rows += [L[i] for i in range(a + 1)]
        out += drafts[:a] + [x]
        pend = x
        rnd += 1
    assert out[:60] == ntok
    for i in range(60):
        assert np.array_equal(rows[i].view(np.uint32), nlg[i].view(np.uint32)), i
    assert sp.check() == 0 and nat.check() == 0


def _load_synth_state(evs, shape, st, S, P):
    t = torch()
    for li, (kind, param) in enumerate(shape.layers):
        v = st.view(li)
        L = S["layers"][li]
        d = shape.d_model
        if kind in ("SE", "MR"):
            wrap(v.fir_ext[0], (param - 1 + v.n_max, d))[:param - 1] = up(L["window"])
        elif kind == "LI":
            wrap(v.iir_all[0], (v.n_max, d, param, 2))[0] = up(L["s"]).view(d, param, 2)
        else:
            H, Dh = shape.n_heads, shape.head_dim
            kc = wrap(v.k_cache, (H, v.ctx_max, Dh), "<i2").view(t.bfloat16)
            vc = wrap(v.v_cache, (H, v.ctx_max, Dh), "<i2").view(t.bfloat16)
            kc[:, :P] = up(L["k"]).transpose(0, 1)
            vc[:, :P] = up(L["v"]).transpose(0, 1)
    t.cuda.synchronize()
    st.set_book(pos=P, fir_bank=0, fir_off=0, iir_bank=0, iir_slot=0, pending_n=0, status=0)


@pytest.mark.gpu
def test_7b_block_verify_full_size():
    import hybrid_ssm_attention_gb300 as evs
    from oracle.model import Model as OModel
    from oracle.numerics import Arith
    shape = synth.stack_7b()
    P = 1024
    W = synth.make_weights(shape, 3)
    S = synth.synth_state(shape, 3, P)
    m = evs.Model(shape, W)
    st = evs.State(m, P + 64)
    _load_synth_state(evs, shape, st, S, P)
    toks = [int(x) for x in synth.prompt(shape, 3, shape.n_block)]
    lg, _ = _verify(evs, st, toks, shape.vocab)
    got = to_np(lg)
    assert st.check() == 0
    del m.tensors[:]   # free device weights before the host oracle runs
    Wf = synth.weights_f32(W)
    del W
    om = OModel(shape, Wf, Arith(np.float32, bf16_points=True))
    del Wf
    Sf = dict(S)
    Sf["layers"] = [dict(L, k=None if L["k"] is None else synth.bf16_bits_to_f32(L["k"]),
                         v=None if L["v"] is None else synth.bf16_bits_to_f32(L["v"])) for L in S["layers"]]
    ost = om.state_from(Sf, P + 64)
    ref, _ = om.verify(ost, toks)
    err = rel_err(got, ref)
    assert err <= TOL, err
    gap_tol = 4 * np.abs(got - ref).max()
    for i in range(len(toks)):
        srt = np.sort(ref[i])
        if srt[-1] - srt[-2] > gap_tol:
            assert int(np.argmax(got[i])) == int(np.argmax(ref[i])), i
