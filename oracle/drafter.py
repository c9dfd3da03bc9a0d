"""Drafter-side Markov head (oracle, test infrastructure only).

Sources.  The preprint abstract, contribution (ii), describes a distilled
drafter with a gamma-parallel trunk and a full-matrix Markov head; the model
card's checkpoint description adds one trunk layer at d_model 1024, the
target's layer-27 hidden state injected as a prefix, a full V x V Markov
head, a confidence head and a frozen embedding.  The pages print no
equations.  The plainest reading, used here:

  * the trunk scores all gamma draft slots in one pass: trunk_logits[i] is
    slot i's row (it cannot see the drafts it is about to propose);
  * the Markov head adds row M[prev] of a V x V matrix, prev being the
    token before the slot (the pending token for the first slot, the
    previous draft after that), so the drafts are sequential through the
    head alone;
  * draft i is drawn from q_i = top-k softmax((trunk_logits[i] + M[prev_i]) / T)
    with the same integer-ladder sampler as the accept rule and uniform u[i]
    (greedy: the argmax of the logits, ties to the lowest index).

The confidence head and the injection only shape the trained trunk's
inputs; with no trained weights here they are not restated.
"""
from __future__ import annotations

import numpy as np

from .sampling import GREEDY, argmax_low, sample, topk_probs


def markov_draft(trunk_logits, M, prev: int, u, T: float = 1.0, top_k: int = 0, mode: int = GREEDY):
    """Returns (drafts [gamma] ints, q [gamma][V] float32)."""
    trunk = np.asarray(trunk_logits, dtype=np.float32)
    M = np.asarray(M, dtype=np.float32)
    drafts, qs = [], []
    for i in range(trunk.shape[0]):
        logits = trunk[i] + M[int(prev)]
        q = topk_probs(logits, T, top_k, dtype=np.float32)
        d = argmax_low(logits) if mode == GREEDY else sample(q, np.float32(u[i]))
        drafts.append(int(d))
        qs.append(q)
        prev = d
    return drafts, np.stack(qs)
