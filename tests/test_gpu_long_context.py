"""Block-causal attention at long context (the long-context configuration:
32 heads x 128, a cache of 262,144 committed positions ~ N(0, 1)) through
the operator entry point, the launch configuration the model uses at that
size (fixed key spans of 8,192 keys, 33 splits per head, 1,056 work units
over one CTA per SM).

The full cache is 4.3 GB; the oracle evaluates two sampled heads (0 and 29),
whose rows are synthesised on the host, while the other heads' rows are
device-side filler.  Heads are independent, so the sampled heads' outputs,
their appended rotated keys and values, and the commit are checked exactly
as at 8192 positions: a block of 13 queries, commit, then a single query.
"""
import numpy as np
import pytest

import synth
from gpu_util import book_zero, fir_ext, fir_set_window, rel_err, to_np, torch, up, wrap
from oracle.model import attend, rope
from oracle.numerics import Arith, round_bf16

AR = Arith(np.float32, bf16_points=True)


def _f(bits):
    return synth.bf16_bits_to_f32(bits)


@pytest.mark.gpu
def test_attention_op_262144_cache_sampled_heads():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    H, Dh, P, n_max, chunk = 32, 128, 262144, 13, 64
    d = H * Dh
    ctx = P + 2 * n_max
    heads = (0, 29)
    kc = t.empty((H, ctx, Dh), dtype=t.bfloat16, device="cuda")
    vc = t.empty_like(kc)
    gen = t.Generator(device="cuda").manual_seed(5)
    kc.normal_(generator=gen)
    vc.normal_(generator=gen)
    Kh, Vh = {}, {}
    for h in heads:
        kb, vb = synth.kv_head(4, h, P, Dh)
        kc[h, :P] = up(kb)
        vc[h, :P] = up(vb)
        Kh[h] = np.zeros((ctx, 1, Dh), np.float32)
        Vh[h] = np.zeros((ctx, 1, Dh), np.float32)
        Kh[h][:P, 0], Vh[h][:P, 0] = _f(kb), _f(vb)
    book = book_zero(t)
    book[0] = P
    scratch = t.empty(evs.evs_op_attention_scratch_bytes(H, Dh, ctx, chunk, n_max), dtype=t.uint8, device="cuda")
    pos = P
    for rnd, (n, keep) in enumerate(((13, 6), (1, 1))):
        qkv = synth.abv_block(50 + rnd, n, d, "bf16")
        g = t.empty((n, d), dtype=t.bfloat16, device="cuda")
        evs.evs_op_attention(H, Dh, n, n_max, ctx, chunk, 10000.0, evs.EVS_BF16, up(qkv), kc, vc, book, g,
                             scratch)
        qf = _f(qkv)
        gout = to_np(g)
        for h in heads:
            sl = slice(h * Dh, (h + 1) * Dh)
            for i in range(n):
                k = round_bf16(rope(qf[i, d:2 * d].reshape(H, Dh), pos + i, 10000.0, AR))[h]
                Kh[h][pos + i, 0], Vh[h][pos + i, 0] = k, qf[i, 2 * d:].reshape(H, Dh)[h]
            ref = []
            for i in range(n):
                q = round_bf16(rope(qf[i, :d].reshape(H, Dh), pos + i, 10000.0, AR))[h:h + 1]
                ref.append(attend(q, Kh[h][:pos + i + 1], Vh[h][:pos + i + 1], AR)[0])
            assert rel_err(gout[:, sl], np.stack(ref)) <= 2e-2, (rnd, h)
            kg = to_np(kc[h, pos:pos + n])
            vg = to_np(vc[h, pos:pos + n])
            assert rel_err(kg, Kh[h][pos:pos + n, 0]) <= 1e-2 and np.array_equal(vg, Vh[h][pos:pos + n, 0])
        assert np.isfinite(gout).all()
        evs.evs_op_commit(book, keep, n)
        pos += keep
        assert int(book[0].item()) == pos


def _kv_layer_from_synth(seed, P, H, Dh):
    """All heads of one attention layer's cache rows [P][H][Dh] (bf16 patterns)."""
    k = np.empty((P, H, Dh), np.uint16)
    v = np.empty((P, H, Dh), np.uint16)
    for h in range(H):
        k[:, h], v[:, h] = synth.kv_head(seed, h, P, Dh)
    return k, v


@pytest.mark.gpu
def test_7b_stack_262144_context_rounds():
    """The full 7B-shaped stack at 262,144 cached positions (long-context
    configuration): one traced block verify of 13 tokens from a synthesised
    state, then greedy and sampled (T = 1, top_k = 4) rounds whose commit
    lengths are drawn geometric with mean 3.

    The first attention layer's cache holds N(0, 1) rows from the input
    generators for every head; the other four attention layers hold device
    filler (their values reach the checks only through the residual stream,
    which the checks take from the GPU).  Teacher-forced against the oracle:
    every Hyena layer's update and retained state, the first attention
    layer's update over all 32 heads and 262,157 keys, its appended rows,
    and the head; each round's accept decision on the GPU's p, q, u."""
    import hybrid_ssm_attention_gb300 as evs
    from oracle.model import LayerState, Model as OModel
    from oracle.sampling import GREEDY, SAMPLE, accept
    t = torch()
    shape = synth.stack_7b()
    H, Dh, d, V = shape.n_heads, shape.head_dim, shape.d_model, shape.vocab
    P, n, R = 262144, shape.n_block, 4
    ctx = P + 64
    seed = 4
    W = synth.make_weights(shape, seed)
    m = evs.Model(shape, W)
    st = evs.State(m, ctx)
    S = synth.synth_state(shape, seed, 0)  # FIR windows and IIR states (no KV rows)
    att = [i for i, (k, _) in enumerate(shape.layers) if k == "ATT"]
    checked = att[0]
    gen = t.Generator(device="cuda").manual_seed(seed)
    kb, vb = _kv_layer_from_synth(seed, P, H, Dh)
    for li, (kind, param) in enumerate(shape.layers):
        v = st.view(li)
        L = S["layers"][li]
        if kind in ("SE", "MR"):
            fir_set_window(wrap(v.fir_ring, (param - 1 + v.n_max, d)), param, v.n_max, P, up(L["window"]))
        elif kind == "LI":
            wrap(v.iir_all[0], (v.n_max, d, param, 2))[0] = up(L["s"]).view(d, param, 2)
        else:
            kc = wrap(v.k_cache, (H, ctx, Dh), "<i2").view(t.bfloat16)
            vc = wrap(v.v_cache, (H, ctx, Dh), "<i2").view(t.bfloat16)
            if li == checked:
                for h in range(H):
                    kc[h, :P] = up(np.ascontiguousarray(kb[:, h]))
                    vc[h, :P] = up(np.ascontiguousarray(vb[:, h]))
            else:
                kc.normal_(generator=gen)
                vc.normal_(generator=gen)
    t.cuda.synchronize()
    st.set_book(pos=P, iir_bank=0, iir_slot=0, pending_n=0, status=0)
    toks = [int(x) for x in synth.prompt(shape, seed, n)]
    tt = t.tensor(np.asarray(toks, np.int32), device="cuda")
    lg = t.empty((n, V), dtype=t.float32, device="cuda")
    p = t.empty((n, V), dtype=t.float32, device="cuda")
    trace = t.empty((len(shape.layers) + 1, n, d), dtype=t.float32, device="cuda")
    evs.evs_verify_block_trace(st, tt, n, lg, trace)
    X, got = to_np(trace), to_np(lg)
    book = st.book()
    assert book["pending_n"] == n and book["status"] == 0
    ret = {}
    for li, (kind, param) in enumerate(shape.layers):
        v = st.view(li)
        if kind in ("SE", "MR"):
            ret[li] = fir_ext(to_np(wrap(v.fir_ring, (param - 1 + v.n_max, d))), param, v.n_max, P, n)
        elif kind == "LI":
            ret[li] = to_np(wrap(v.iir_all[1 - book["iir_bank"]], (v.n_max, d, param, 2)))
        elif li == checked:
            kc = wrap(v.k_cache, (H, ctx, Dh), "<i2").view(t.bfloat16)
            vc = wrap(v.v_cache, (H, ctx, Dh), "<i2").view(t.bfloat16)
            ret[li] = (to_np(kc[:, P:P + n]).transpose(1, 0, 2), to_np(vc[:, P:P + n]).transpose(1, 0, 2))
    # rounds: accept (greedy, then sampled), commit a drawn geometric keep
    keeps = synth.keep_draws(seed, R, n, kind="geometric")
    q = synth.fixed_logit_drafter(seed, n - 1, V)
    U = synth.uniforms(seed, R, n)
    acc = t.zeros(1, dtype=t.int32, device="cuda")
    tok = t.zeros(1, dtype=t.int32, device="cuda")
    pos = P
    for r in range(R):
        if r > 0:
            toks_r = [int(x) for x in synth.prompt(shape, seed + 10 * r, n)]
            evs.evs_verify_block(st, t.tensor(np.asarray(toks_r, np.int32), device="cuda"), n, lg)
        else:
            toks_r = toks
        if r % 2 == 0:
            evs.evs_accept(lg, None, t.tensor(np.asarray(toks_r[1:], np.int32), device="cuda"), None, n, V,
                           evs.EVS_GREEDY, acc, tok)
            want = accept(to_np(lg), None, toks_r[1:], np.zeros(n, np.float32), GREEDY)
        else:
            evs.evs_probs(lg, n, V, 1.0, 4, p)
            evs.evs_accept(p, up(q), t.tensor(np.asarray(toks_r[1:], np.int32), device="cuda"), up(U[r]), n, V,
                           evs.EVS_SAMPLE, acc, tok)
            want = accept(to_np(p), q, toks_r[1:], U[r], SAMPLE)
        assert (int(acc.item()), int(tok.item())) == want, r
        evs.evs_commit(st, int(keeps[r]))
        pos += int(keeps[r])
        assert st.book()["pos"] == pos
    assert st.check() == 0
    st.close()
    m.close()
    # the oracle, teacher-forced on the GPU's residual stream
    Wf = synth.weights_f32(W)
    del W
    om = OModel(shape, Wf, Arith(np.float32, bf16_points=True))
    del Wf
    for li, (M, (kind, param)) in enumerate(zip(om.layers, shape.layers)):
        Ls = S["layers"][li]
        if kind in ("SE", "MR"):
            L = LayerState(kind, window=Ls["window"].astype(np.float32).copy())
        elif kind == "LI":
            L = LayerState(kind, s=Ls["s"].astype(np.complex64).copy())
        elif li == checked:
            K = np.zeros((P + n, H, Dh), np.float32)
            Vv = np.zeros((P + n, H, Dh), np.float32)
            K[:P], Vv[:P] = _f(kb), _f(vb)
            L = LayerState(kind, K=K, V=Vv, length=P)
        else:
            continue
        d_ref, d_gpu = [], []
        for i in range(n):
            x_out = om.layer_forward(M, L, X[li][i].copy(), P + i)
            d_ref.append(x_out - X[li][i])
            d_gpu.append(X[li + 1][i] - X[li][i])
            if kind in ("SE", "MR"):
                assert rel_err(ret[li][i + 1:i + param], L.window) <= 2e-2, (li, i)
            elif kind == "LI":
                Rr = ret[li][i]
                assert rel_err(Rr[..., 0], L.s.real) <= 2e-2 and rel_err(Rr[..., 1], L.s.imag) <= 2e-2, (li, i)
        if kind == "ATT":
            assert rel_err(ret[li][0], L.K[P:P + n]) <= 2e-2 and rel_err(ret[li][1], L.V[P:P + n]) <= 2e-2
        e = rel_err(np.stack(d_gpu), np.stack(d_ref))
        assert e <= 2e-2, (li, kind, e)
    head = np.stack([om.head(X[-1][i]) for i in range(n)])
    assert rel_err(got, head) <= 1e-3
