"""Small, self-contained launches of one kernel for profiler captures.

    python -m hybrid_ssm_attention_gb300.profile_case gemm 22016 4096 13
        bf16 tensor-core GEMM of a [N][K] weight (N(0,0.02)) against n tokens,
        repeated `--reps` times (default 4); the weight (180 MB for the
        default shape) is larger than L2, so each launch streams it from HBM.
    python -m hybrid_ssm_attention_gb300.profile_case fir 128 4096 13
    python -m hybrid_ssm_attention_gb300.profile_case iir 16 4096 13
    python -m hybrid_ssm_attention_gb300.profile_case attn 8192 13   (split-KV chunks of 64 keys)
    python -m hybrid_ssm_attention_gb300.profile_case stack 2 13
        the first L layers (default 2) of the 7B-shaped stack with the
        library's packed weights: one warm-up verify of n tokens (4L+1 GEMM
        launches and the row / mixer kernels), then every weight GEMM of a
        step once more, each launched alone (in, out, gate/up, down per
        layer, then the head).
    python -m hybrid_ssm_attention_gb300.profile_case batch 2 8 13
        the first L layers of the 7B-shaped stack, B sequences of n rows each
        verified in one batched pass (B * n rows: 16-row chunks side by side
        in the GEMMs' N dimension), each sequence committing its block;
        repeated `--reps` times.
"""
from __future__ import annotations

import argparse

import numpy as np


def main():
    import torch

    import hybrid_ssm_attention_gb300 as evs
    from hybrid_ssm_attention_gb300 import build as b
    b.build()
    ap = argparse.ArgumentParser()
    ap.add_argument("kind", choices=["gemm", "fir", "iir", "attn", "stack", "batch"])
    ap.add_argument("args", type=int, nargs="*")
    ap.add_argument("--reps", type=int, default=4)
    a = ap.parse_args()
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(0)
    book = torch.zeros(8, dtype=torch.int32, device=dev)
    book[4] = -1
    if a.kind == "batch":
        import synth
        L, B, n = (a.args + [2, 8, 13][len(a.args):])[:3]
        full = synth.stack_7b()
        shape = synth.ModelShape(name=f"7b-first-{L}", vocab=full.vocab, d_model=full.d_model,
                                 layers=full.layers[:L], n_heads=full.n_heads, head_dim=full.head_dim,
                                 d_ffn=full.d_ffn, gamma=full.gamma, dtype="bf16", pole_mag=full.pole_mag)
        m = evs.Model(shape, synth.make_weights(shape, 3))
        sts = [evs.State(m, 256) for _ in range(B)]
        toks = torch.tensor([65 + (i % 4) for i in range(B * n)], dtype=torch.int32, device=dev)
        lg = torch.empty((B * n, shape.vocab), device=dev)
        for _ in range(a.reps):
            evs.evs_verify_batch(sts, toks, [n] * B, lg)
            for st in sts:
                evs.evs_commit(st, n)
    elif a.kind == "stack":
        import synth
        L, n = (a.args + [2, 13][len(a.args):])[:2]
        full = synth.stack_7b()
        shape = synth.ModelShape(name=f"7b-first-{L}", vocab=full.vocab, d_model=full.d_model,
                                 layers=full.layers[:L], n_heads=full.n_heads, head_dim=full.head_dim,
                                 d_ffn=full.d_ffn, gamma=full.gamma, dtype="bf16", pole_mag=full.pole_mag)
        m = evs.Model(shape, synth.make_weights(shape, 3))
        st = evs.State(m, 256)
        toks = torch.tensor([65 + (i % 4) for i in range(n)], dtype=torch.int32, device=dev)
        lg = torch.empty((n, shape.vocab), device=dev)
        evs.evs_verify_block(st, toks, n, lg)
        evs.evs_commit(st, n)
        evs.evs_profile_gemms(st, n)
    elif a.kind == "gemm":
        N, K, n = (a.args + [22016, 4096, 13][len(a.args):])[:3]
        W = (torch.randn(N, K, device=dev, generator=g) * 0.02).to(torch.bfloat16)
        X = torch.randn(n, K, device=dev, generator=g).to(torch.bfloat16)
        y = torch.empty(n, N, device=dev)
        s = torch.empty(evs.evs_op_gemm_scratch_bytes(N, K, evs.EVS_BF16), dtype=torch.uint8, device=dev)
        for _ in range(a.reps):
            evs.evs_op_gemm(W, X, N, K, n, evs.EVS_BF16, y, s)
    elif a.kind in ("fir", "iir"):
        P, d, n = (a.args + [128 if a.kind == "fir" else 16, 4096, 13][len(a.args):])[:3]
        abv = torch.randn(n, 3 * d, device=dev, generator=g).to(torch.bfloat16)
        gout = torch.empty(n, d, device=dev, dtype=torch.bfloat16)
        for r in range(a.reps):
            if a.kind == "fir":
                e0 = torch.randn(P - 1 + n, d, device=dev, generator=g)
                e1 = torch.empty_like(e0)
                taps = torch.randn(P, d, device=dev, generator=g)
                evs.evs_op_fir(P, d, n, n, evs.EVS_BF16, abv, taps, e0, e1, book, gout)
            else:
                s0 = torch.randn(n, d, P, 2, device=dev, generator=g)
                s1 = torch.empty_like(s0)
                lam = torch.rand(d, P, 2, device=dev, generator=g) * 0.7
                res = torch.randn(d, P, 2, device=dev, generator=g) * 0.25
                evs.evs_op_iir(P, d, n, n, evs.EVS_BF16, abv, lam, res, s0, s1, book, gout)
    else:
        P, n = (a.args + [8192, 13][len(a.args):])[:2]
        H, Dh, chunk = 32, 128, 64
        ctx = P + n
        kc = torch.randn(H, ctx, Dh, device=dev, generator=g).to(torch.bfloat16)
        vc = torch.randn(H, ctx, Dh, device=dev, generator=g).to(torch.bfloat16)
        qkv = torch.randn(n, 3 * H * Dh, device=dev, generator=g).to(torch.bfloat16)
        gout = torch.empty(n, H * Dh, device=dev, dtype=torch.bfloat16)
        s = torch.empty(evs.evs_op_attention_scratch_bytes(H, Dh, ctx, chunk, n), dtype=torch.uint8, device=dev)
        book[0] = P
        for _ in range(a.reps):
            evs.evs_op_attention(H, Dh, n, n, ctx, chunk, 10000.0, evs.EVS_BF16, qkv, kc, vc, book, gout, s)
    torch.cuda.synchronize()
    print("profile case done:", a.kind, a.args, float(np.float32(0)))


if __name__ == "__main__":
    main()
