"""Target distribution, sampler and the accept rule (oracle, test infrastructure only).

Sources.
* Preprint abstract and discussion post ("What we implemented"): sampling
  keeps the target distribution through exact rejection-sampling
  verification; greedy decoding reproduces native output token for token.
* Model card, "Library" example: default sampling is T = 1.0, top_k = 4.

The accept rule is the standard speculative-sampling rule the pages refer to:
draft d_i ~ q_i is accepted with probability min(1, p_{i-1}(d_i) / q_i(d_i));
at the first rejection the output token is drawn from the normalised residual
(p_{i-1} - q_i)^+; if every draft is accepted a bonus token is drawn from p_gamma.

Readings where the pages are silent (each fixed so that the GPU can match it
bit for bit given the same p, q and uniforms):
* accept test ``u_{i-1} * q_i(d_i) < p_{i-1}(d_i)`` in float32 (one rounded
  product, no division); u_{i-1} is the i-th uniform of the round;
* the output token always uses the last uniform u_gamma;
* sample(w, u) is an inverse CDF on integer weights W_j = floor(w_j 2^24),
  exact under any summation order; mass below 2^-24 per entry is dropped;
* a residual with zero integer mass falls back to p_{i-1};
* greedy: argmax with ties to the lowest index; top-k ties go to the lower
  index as well.
"""
from __future__ import annotations

import numpy as np

GREEDY, SAMPLE = 0, 1
TWO24 = 1 << 24


def topk_probs(logits, T: float = 1.0, top_k: int = 0, dtype=np.float32):
    """p = softmax(logits / T) restricted to the top_k largest logits
    (top_k <= 0 or >= V: all entries); zero elsewhere."""
    l = np.asarray(logits, dtype=dtype)
    V = l.shape[-1]
    keep = np.zeros(V, dtype=bool)
    if top_k <= 0 or top_k >= V:
        keep[:] = True
    else:
        order = np.argsort(-l, kind="stable")        # equal values keep index order
        keep[order[:top_k]] = True
    m = l[keep].max()
    w = np.zeros(V, dtype=dtype)
    w[keep] = np.exp((l[keep] - m) / dtype(T))
    return (w / w.sum(dtype=dtype)).astype(dtype)


def sample(w, u) -> int:
    """Smallest j with sum_{l<=j} W_l > floor(floor(u 2^24) * S / 2^24),
    W_l = floor(w_l 2^24), S = sum W_l (exact integers)."""
    w = np.asarray(w, dtype=np.float32)
    W = [int(np.floor(np.float64(x) * TWO24)) for x in w]
    S = sum(W)
    if S == 0:
        raise ValueError("sample: zero integer mass")
    U = int(np.floor(np.float64(np.float32(u)) * TWO24))
    t = (U * S) >> 24
    acc = 0
    for j, Wj in enumerate(W):
        acc += Wj
        if acc > t:
            return j
    raise AssertionError("unreachable: t < S")


def argmax_low(x) -> int:
    x = np.asarray(x)
    return int(np.flatnonzero(x == x.max())[0])


def accept(p, q, drafts, u, mode: int):
    """Accept rule for one verify block.

    p      [n][V]  target distributions (or, in greedy mode, any scores whose
                   argmax is the target token, e.g. logits); p[i] follows
                   block token i.
    q      [gamma][V] drafter distributions; q[i-1] proposed drafts[i-1].
    drafts [gamma] draft tokens d_1..d_gamma.
    u      [n]     uniforms in [0, 1).
    Returns (a, token): a in [0, gamma] accepted drafts, then the output token.
    """
    p = np.asarray(p, dtype=np.float32)
    n = p.shape[0]
    gamma = n - 1
    a = gamma
    for i in range(1, gamma + 1):
        d = int(drafts[i - 1])
        if mode == GREEDY:
            ok = d == argmax_low(p[i - 1])
        else:
            qi = np.asarray(q, dtype=np.float32)[i - 1]
            ok = np.float32(np.float32(u[i - 1]) * qi[d]) < p[i - 1][d]
        if not ok:
            a = i - 1
            break
    if mode == GREEDY:
        return a, argmax_low(p[a])
    u_last = np.float32(u[gamma])
    if a < gamma:
        qa = np.asarray(q, dtype=np.float32)[a]
        r = np.maximum(p[a] - qa, np.float32(0)).astype(np.float32)
        if sum(int(np.floor(np.float64(x) * TWO24)) for x in r) > 0:
            return a, sample(r, u_last)
    return a, sample(p[a], u_last)
