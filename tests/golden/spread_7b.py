"""Writes spread_7b.json: how far the oracle's own logits move when only the
summation order of its matrix-vector products changes, on the full-size
7B-shaped block verify that the GPU test compares against (32 layers,
d_model 4096, weights of seed 3, a synthesised state at context 1024, the
13-token block of seed 3).

Both orders are valid float32 evaluations of the same method with the same
bf16 storage points; their difference is rounding alone, compounded through
32 layers (a bf16 storage point that lands on the other side of a rounding
boundary moves by one bf16 step, about 0.4% of the value, and the random-init
stack carries such flips forward).  The GPU's fp32 sums follow yet another
valid order, so its distance from the oracle is expected on the same scale;
the GPU test takes its free-running bound from this file.

Calls only the oracle and the seeded input generators.

    python tests/golden/spread_7b.py        # ~26 GB of host memory, a few minutes
"""
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle.model import Model  # noqa: E402
from oracle.numerics import Arith  # noqa: E402

SEED, P = 3, 1024


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.abs(a - b).max() / np.abs(b).max())


def main():
    shape = synth.stack_7b()
    n = shape.n_block
    t0 = time.time()
    W = synth.make_weights(shape, SEED)
    Wf = synth.weights_f32(W)
    del W
    S = synth.synth_state(shape, SEED, P)
    S["layers"] = [dict(L, k=None if L["k"] is None else synth.bf16_bits_to_f32(L["k"]),
                        v=None if L["v"] is None else synth.bf16_bits_to_f32(L["v"])) for L in S["layers"]]
    toks = [int(x) for x in synth.prompt(shape, SEED, n)]
    logits = {}
    for order in Arith.ORDERS:
        om = Model(shape, Wf, Arith(np.float32, bf16_points=True, order=order))
        st = om.state_from(S, P + 64)
        logits[order], _ = om.verify(st, toks)
        print(f"{order}: done at {time.time() - t0:.0f} s", flush=True)
    a, b = logits["blas"], logits["k64_reversed"]
    per_row = [rel(b[i], a[i]) for i in range(n)]
    out = {"what": "oracle vs oracle, float32 with bf16 storage points, two matrix-vector summation orders",
           "workload": {"shape": "7B-shaped stack (32 layers, d 4096, F 11008, vocab 512)", "weights_seed": SEED,
                        "state": f"synthesised at context {P}", "block_tokens": toks},
           "orders": list(Arith.ORDERS),
           "rel_err_logits": rel(b, a),
           "rel_err_logits_per_row": per_row,
           "max_abs_logit": float(np.abs(a).max())}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "spread_7b.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps({k: out[k] for k in ("rel_err_logits", "max_abs_logit")}))


if __name__ == "__main__":
    main()
