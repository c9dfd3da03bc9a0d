"""The persistent engine against the separate kernels, bit for bit.

The engine (one persistent kernel per span of layers between attention
mixers) keeps every reduction order of the separate kernels, which the other
GPU tests compare with the oracle.  Here two states of one model run the same
prefill and rounds, one through the engine and one through the separate
kernels: every verify's logits, every round's accepted count, output token
and target distribution, the bookkeeping and the retained FIR windows, IIR
states and KV rows must be identical bits.  Shapes: the small bf16 stack (blocks
of up to 13 and up to 16 rows) and a 7B-width stack with every layer kind
(FIR 7, FIR 128, IIR 16, attention); ragged blocks; greedy and sampled rounds.
"""
import numpy as np
import pytest

import synth
from gpu_util import to_np, torch, wrap


def small_shape(gamma=12):
    return synth.ModelShape(name="small-bf16", vocab=128, d_model=256,
                            layers=[("SE", 7), ("MR", 128), ("LI", 16), ("SE", 7), ("MR", 32), ("ATT", 0)],
                            n_heads=2, head_dim=128, d_ffn=512, gamma=gamma, dtype="bf16", attn_chunk=64)


def wide_shape():
    return synth.ModelShape(name="wide-bf16", vocab=512, d_model=4096,
                            layers=[("SE", 7), ("MR", 128), ("LI", 16), ("ATT", 0), ("MR", 128), ("SE", 7)],
                            n_heads=32, head_dim=128, d_ffn=11008, gamma=12, dtype="bf16", attn_chunk=64)


def _bits(x):
    return to_np(x).view(np.uint32)


def _state_bits(shape, st):
    t = torch()
    book = st.book()
    out = [np.array(list(book.values()), np.int64)]
    d = shape.d_model
    for li, (kind, param) in enumerate(shape.layers):
        v = st.view(li)
        if kind in ("SE", "MR"):
            out.append(to_np(wrap(v.fir_ring, (param - 1 + v.n_max, d))).view(np.uint32))
        elif kind == "LI":
            for b in (0, 1):
                out.append(to_np(wrap(v.iir_all[b], (v.n_max, d, param, 2))).view(np.uint32))
        else:
            H, Dh, P = shape.n_heads, shape.head_dim, book["pos"]
            for ptr in (v.k_cache, v.v_cache):
                out.append(to_np(wrap(ptr, (H, v.ctx_max, Dh), "<i2").view(t.bfloat16)[:, :P]).view(np.uint32))
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("which", ["small", "small16", "wide"])
def test_engine_equals_separate_kernels_bitwise(which):
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    shape = {"small": small_shape(), "small16": small_shape(15), "wide": wide_shape()}[which]
    W = synth.make_weights(shape, 81)
    m = evs.Model(shape, W)
    V, nb = shape.vocab, shape.n_block
    eng, sep = evs.State(m, 512), evs.State(m, 512)
    eng.use_engine(True)
    sep.use_engine(False)
    assert evs.evs_verify_kernel_count(eng, nb) < evs.evs_verify_kernel_count(sep, nb)
    prompt = [int(x) for x in synth.prompt(shape, 81, 3 * nb + 4)]
    g = np.random.default_rng(7)
    for s0 in range(0, len(prompt), nb):
        chunk = prompt[s0:s0 + nb]
        outs = []
        for st in (eng, sep):
            tt = t.tensor(np.asarray(chunk, np.int32), device="cuda")
            lg = t.empty((len(chunk), V), dtype=t.float32, device="cuda")
            evs.evs_verify_block(st, tt, len(chunk), lg)
            outs.append(_bits(lg))
        assert np.array_equal(outs[0], outs[1]), s0
        keep = int(g.integers(0, len(chunk) + 1)) if s0 else len(chunk)
        for st in (eng, sep):
            evs.evs_commit(st, keep)
    acc = [t.zeros(1, dtype=t.int32, device="cuda") for _ in range(2)]
    tok = [t.zeros(1, dtype=t.int32, device="cuda") for _ in range(2)]
    pend = prompt[-1]
    for rnd in range(6):
        n = [nb, 1, 5, nb, 2, nb][rnd]
        sample = rnd % 2 == 1
        block = [pend] + [int(x) for x in g.integers(0, V, n - 1)]
        q = t.softmax(t.tensor(g.standard_normal((max(n - 1, 1), V)), dtype=t.float32, device="cuda"), dim=1)
        u = t.tensor(g.random(n), dtype=t.float32, device="cuda")
        res = []
        for i, st in enumerate((eng, sep)):
            tt = t.tensor(np.asarray(block, np.int32), device="cuda")
            lg = t.empty((n, V), dtype=t.float32, device="cuda")
            p = t.empty((n, V), dtype=t.float32, device="cuda")
            evs.evs_round(st, tt, n, lg, p if sample else None, q if sample else None, u if sample else None,
                          1.0, 4, evs.EVS_SAMPLE if sample else evs.EVS_GREEDY, acc[i], tok[i])
            res.append((_bits(lg), _bits(p) if sample else None, int(acc[i].item()), int(tok[i].item())))
        assert np.array_equal(res[0][0], res[1][0]), rnd
        if sample:
            assert np.array_equal(res[0][1], res[1][1]), rnd
        assert res[0][2:] == res[1][2:], rnd
        pend = res[0][3]
    assert eng.check() == 0 and sep.check() == 0
    for a, b in zip(_state_bits(shape, eng), _state_bits(shape, sep)):
        assert np.array_equal(a, b)


@pytest.mark.gpu
def test_engine_7b_rounds_equal_separate_kernels_bitwise():
    # the full 7B-shaped stack: prefill of 64 tokens, then 4 identity-like
    # rounds of 13; logits, accepted counts, tokens and bookkeeping identical
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    shape = synth.stack_7b()
    W = synth.make_weights(shape, 3)
    m = evs.Model(shape, W)
    V, nb = shape.vocab, shape.n_block
    eng, sep = evs.State(m, 256), evs.State(m, 256)
    eng.use_engine(True)
    sep.use_engine(False)
    prompt = [int(x) for x in synth.prompt(shape, 3, 64)]
    for s0 in range(0, len(prompt), nb):
        chunk = prompt[s0:s0 + nb]
        outs = []
        for st in (eng, sep):
            tt = t.tensor(np.asarray(chunk, np.int32), device="cuda")
            lg = t.empty((len(chunk), V), dtype=t.float32, device="cuda")
            evs.evs_verify_block(st, tt, len(chunk), lg)
            evs.evs_commit(st, len(chunk))
            outs.append(_bits(lg))
        assert np.array_equal(outs[0], outs[1]), s0
    g = np.random.default_rng(11)
    acc = [t.zeros(1, dtype=t.int32, device="cuda") for _ in range(2)]
    tok = [t.zeros(1, dtype=t.int32, device="cuda") for _ in range(2)]
    pend = int(synth.prompt(shape, 4, 1)[0])
    for rnd in range(4):
        block = [pend] + [int(x) for x in g.integers(0, V, nb - 1)]
        res = []
        for i, st in enumerate((eng, sep)):
            tt = t.tensor(np.asarray(block, np.int32), device="cuda")
            lg = t.empty((nb, V), dtype=t.float32, device="cuda")
            evs.evs_round(st, tt, nb, lg, None, None, None, 1.0, 0, evs.EVS_GREEDY, acc[i], tok[i])
            res.append((_bits(lg), int(acc[i].item()), int(tok[i].item())))
        assert np.array_equal(res[0][0], res[1][0]), rnd
        assert res[0][1:] == res[1][1:], rnd
        pend = res[0][2]
    assert eng.book() == sep.book()
    assert eng.check() == 0 and sep.check() == 0


@pytest.mark.gpu
def test_engine_refused_where_the_model_does_not_fit():
    import hybrid_ssm_attention_gb300 as evs
    shape = synth.tiny()  # float32 storage: separate kernels only
    m = evs.Model(shape, synth.make_weights(shape, 1))
    st = evs.State(m, 64)
    with pytest.raises(evs.EvsError) as e:
        st.use_engine(True)
    assert e.value.code == evs.EVS_ERR_UNSUPPORTED
    st.use_engine(False)
