"""evs_round_host (block and result in host memory) against evs_round on
device buffers: two clones of one state run the same rounds, one through
each entry point; every round's logits, accepted count, output token and
the bookkeeping are identical bits.  Greedy and sampled rounds, ragged block
sizes 1 .. 13; the host-memory round's graph is reused across calls.
"""
import numpy as np
import pytest

import synth
from gpu_util import to_np, torch


def _shape():
    return synth.ModelShape(name="small-bf16", vocab=128, d_model=256,
                            layers=[("SE", 7), ("MR", 32), ("LI", 16), ("ATT", 0)],
                            n_heads=2, head_dim=128, d_ffn=512, gamma=12, dtype="bf16", attn_chunk=64)


@pytest.mark.gpu
def test_round_host_equals_round_on_device_buffers():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    shape = _shape()
    m = evs.Model(shape, synth.make_weights(shape, 41))
    V, nb = shape.vocab, shape.n_block
    a, b = evs.State(m, 512), evs.State(m, 512)
    prompt = [int(x) for x in synth.prompt(shape, 41, 2 * nb)]
    lg = t.empty((nb, V), dtype=t.float32, device="cuda")
    for s0 in range(0, len(prompt), nb):
        chunk = t.tensor(np.asarray(prompt[s0:s0 + nb], np.int32), device="cuda")
        evs.evs_verify_block(a, chunk, chunk.numel(), lg[:chunk.numel()])
        evs.evs_commit(a, chunk.numel())
    a.clone_into(b)
    g = np.random.default_rng(5)
    acc = t.zeros(1, dtype=t.int32, device="cuda")
    tok = t.zeros(1, dtype=t.int32, device="cuda")
    pend = prompt[-1]
    for rnd, n in enumerate([nb, 1, 5, nb, 2, nb, nb, 7]):
        sample = rnd % 2 == 1
        block = np.asarray([pend] + [int(x) for x in g.integers(0, V, n - 1)], np.int32)
        q = t.softmax(t.tensor(g.standard_normal((max(n - 1, 1), V)), dtype=t.float32, device="cuda"), dim=1)
        u = t.tensor(g.random(n), dtype=t.float32, device="cuda")
        mode = evs.EVS_SAMPLE if sample else evs.EVS_GREEDY
        la = t.empty((n, V), dtype=t.float32, device="cuda")
        lb = t.empty((n, V), dtype=t.float32, device="cuda")
        pa = t.empty((n, V), dtype=t.float32, device="cuda") if sample else None
        pb = t.empty((n, V), dtype=t.float32, device="cuda") if sample else None
        evs.evs_round(a, t.tensor(block, device="cuda"), n, la, pa, q if sample else None, u if sample else None,
                      1.0, 4, mode, acc, tok)
        got = evs.evs_round_host(b, block, n, lb, pb, q if sample else None, u if sample else None, 1.0, 4, mode)
        want = (int(acc.item()), int(tok.item()))
        assert got == want, rnd
        assert np.array_equal(to_np(la).view(np.uint32), to_np(lb).view(np.uint32)), rnd
        if sample:
            assert np.array_equal(to_np(pa).view(np.uint32), to_np(pb).view(np.uint32)), rnd
        assert a.book() == b.book(), rnd
        pend = want[1]
    assert a.check() == 0 and b.check() == 0


@pytest.mark.gpu
def test_round_host_rejects_bad_arguments():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    shape = _shape()
    m = evs.Model(shape, synth.make_weights(shape, 2))
    st = evs.State(m, 128)
    lg = t.empty((shape.n_block, shape.vocab), dtype=t.float32, device="cuda")
    with pytest.raises(evs.EvsError) as e:
        evs.evs_round_host(st, np.zeros(17, np.int32), 17, lg, None, None, None, 1.0, 0, evs.EVS_GREEDY)
    assert e.value.code == evs.EVS_ERR_ARG
    with pytest.raises(evs.EvsError) as e:
        evs.evs_round_host(st, np.zeros(3, np.int32), 3, lg, None, None, None, 1.0, 0, evs.EVS_SAMPLE)
    assert e.value.code == evs.EVS_ERR_ARG
