"""Native and speculative decode loops (oracle, test infrastructure only).

Round protocol (preprint abstract, (i); discussion post, "What we
implemented"): the block holds the pending token t_0 followed by drafts
d_1..d_gamma.  One verify pass scores the gamma + 1 tokens and retains each
position's state; the accept rule gives a accepted drafts and one output
token; the state is sliced to keep = a + 1 consumed tokens; the output token
becomes the next pending token.  Emitted per round: d_1..d_a, then the output
token.

Native decoding (model card, ``generate_native``) consumes one token per step.
The prompt's last token is the first pending token; the ones before it are
prefilled one step at a time.
"""
from __future__ import annotations

from typing import Callable, List, Sequence

import numpy as np

from .model import Model, State
from .sampling import GREEDY, accept, argmax_low, sample, topk_probs


def prefill(model: Model, st: State, prompt: Sequence[int]) -> int:
    for t in prompt[:-1]:
        model.step(st, int(t))
    return int(prompt[-1])


def choose(logits, mode, T, top_k, u, dtype=np.float32) -> int:
    if mode == GREEDY:
        return argmax_low(logits)
    return sample(topk_probs(logits, T, top_k, dtype=dtype), u)


def native_generate(model: Model, st: State, pending: int, n_tokens: int,
                    mode: int = GREEDY, T: float = 1.0, top_k: int = 0,
                    u: Sequence[float] = ()):
    """Returns (tokens, logits per step).  Sampling uses u[s] at step s."""
    toks, logs = [], []
    for s in range(n_tokens):
        logits = model.step(st, pending)
        tok = choose(logits, mode, T, top_k, u[s] if mode != GREEDY else 0.0)
        toks.append(tok)
        logs.append(logits)
        pending = tok
    return toks, logs


def spec_generate(model: Model, st: State, pending: int, n_tokens: int, gamma: int,
                  drafter: Callable, mode: int = GREEDY, T: float = 1.0,
                  top_k: int = 0, uniforms=None):
    """Speculative decoding with block verify + accept + commit.

    ``drafter(emitted, round)`` returns (drafts [gamma] ints, q [gamma][V]).
    ``uniforms[round]`` holds gamma + 1 float32 uniforms.
    Returns (tokens, accepted counts per round, final state).  The token list
    holds every token emitted by the rounds run, so it can exceed n_tokens by
    up to gamma; the final state has consumed all of them but the last."""
    out: List[int] = []
    acc: List[int] = []
    rnd = 0
    while len(out) < n_tokens:
        drafts, q = drafter(list(out), rnd)
        block = [pending] + [int(x) for x in drafts]
        logits, records = model.verify(st, block)
        if mode == GREEDY:
            P = logits
            u = np.zeros(gamma + 1, np.float32)
        else:
            P = np.stack([topk_probs(l, T, top_k, dtype=np.float32) for l in logits])
            u = uniforms[rnd]
        a, tok = accept(P, q, drafts, u, mode)
        st = Model.commit(st, records, a + 1)
        out += [int(x) for x in drafts[:a]] + [int(tok)]
        acc.append(a)
        pending = int(tok)
        rnd += 1
    return out, acc, st


def identity_greedy_drafter(native_tokens: Sequence[int], gamma: int, vocab: int):
    """Identity drafter (discussion post, "What we implemented"): proposes
    exactly the tokens native greedy decoding emits next."""
    def drafter(emitted, rnd):
        k = len(emitted)
        d = list(native_tokens[k:k + gamma])
        d += [0] * (gamma - len(d))
        q = np.zeros((gamma, vocab), np.float32)
        q[np.arange(gamma), d] = 1.0
        return d, q
    return drafter
