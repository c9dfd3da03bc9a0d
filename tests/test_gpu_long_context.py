"""Block-causal attention at long context (the long-context configuration:
32 heads x 128, a cache of 262,144 committed positions ~ N(0, 1)) through
the operator entry point, the launch configuration the model uses at that
size (fixed key spans of 32,768 keys, nine splits per head).

The full cache is 4.3 GB; the oracle evaluates two sampled heads (0 and 29),
whose rows are synthesised on the host, while the other heads' rows are
device-side filler.  Heads are independent, so the sampled heads' outputs,
their appended rotated keys and values, and the commit are checked exactly
as at 8192 positions: a block of 13 queries, commit, then a single query.
"""
import numpy as np
import pytest

import synth
from gpu_util import book_zero, rel_err, to_np, torch, up
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
