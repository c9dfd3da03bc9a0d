"""CPU oracle for the EvSpark block-verify / accept / commit path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
or run anything in this package.  The product path (``include/evs.h``, the
CUDA library and its Python binding) never imports it and shares no code
with it.

What it is: a plain, slow, obviously sequential restatement of the method
described in *EvSpark: Lossless Speculative Decoding for Hybrid DNA
Foundation Models* (preprint abstract; GitHub discussion "EvSpark: ~3x
lossless speculative decoding for Evo2 7B with hybrid-state rollback",
sections "The systems problem" and "What we implemented"; model card
"EvSpark - lossless speculative decoding for Evo2", "Library" example).

* ``model``    - the hybrid stack and native one-token decoding; block verify
                 defined as n native steps on a copy of the state, with the
                 per-position state recorded; commit = pick the record.
* ``sampling`` - temperature / top-k distribution, the integer-ladder
                 sampler, and the exact rejection-sampling accept rule.
* ``decode``   - native and speculative decode loops, identity drafter.
* ``numerics`` - bf16 round-to-nearest-even from the IEEE bit layout.

Parity status.  Every function is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` against a closed form, a special case that
reduces to a library routine, an invariant, or brute-force enumeration.
The layer *equations* themselves (FIR/IIR/attention/MLP forms) are a
reading: the pages name the three state classes but print no operator
equations and no weights exist here, so the operator definitions are
"parity unpinned" against the real Evo2 model.
"""
