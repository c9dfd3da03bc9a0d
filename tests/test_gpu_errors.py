"""Failure detection on the C ABI, all raised on the host or by in-kernel
checks that set a status bit and skip the access (nothing traps, faults or
hangs):

* protocol: commit without a pending verify, verify while one is pending
  (EVS_ERR_STATE); keep outside [0, n], n outside [1, gamma_max+1]
  (EVS_ERR_ARG); committed length + n > ctx_max (EVS_ERR_CAPACITY);
* device: a token outside the vocabulary (EVS_DEV_BAD_TOKEN), a device-side
  keep outside [0, n] (EVS_DEV_BAD_KEEP, state left as before the verify),
  an append past ctx_max after device-side commits (EVS_DEV_KV_OVERFLOW);
* injected faults: a device allocation limit (EVS_ALLOC_LIMIT) makes state
  creation fail with EVS_ERR_OOM and the library stays usable; a bounded
  pipeline wait on an mbarrier nothing arrives on expires after 2 ms and
  reports EVS_DEV_TIMEOUT in a status word, the kernel returning normally.
"""
import numpy as np
import pytest

import synth
from gpu_util import to_np, torch

ERR_ARG, ERR_STATE, ERR_CAPACITY, ERR_OOM = 1, 2, 3, 4
BAD_TOKEN, KV_OVERFLOW, BAD_KEEP, DEV_TIMEOUT = 1, 2, 4, 8


def _tiny(ctx):
    import hybrid_ssm_attention_gb300 as evs
    shape = synth.tiny()
    m = evs.Model(shape, synth.make_weights(shape, 0))
    return evs, shape, m, evs.State(m, ctx)


def _v(evs, st, toks, V):
    t = torch()
    tt = t.tensor(np.asarray(toks, np.int32), device="cuda")
    lg = t.empty((len(toks), V), dtype=t.float32, device="cuda")
    evs.evs_verify_block(st, tt, len(toks), lg)
    return lg


@pytest.mark.gpu
def test_protocol_errors():
    evs, shape, m, st = _tiny(64)
    with pytest.raises(evs.EvsError) as e:
        evs.evs_commit(st, 0)
    assert e.value.code == ERR_STATE
    _v(evs, st, [1, 2, 3], shape.vocab)
    with pytest.raises(evs.EvsError) as e:
        _v(evs, st, [1], shape.vocab)
    assert e.value.code == ERR_STATE
    with pytest.raises(evs.EvsError) as e:
        evs.evs_commit(st, 4)
    assert e.value.code == ERR_ARG
    with pytest.raises(evs.EvsError) as e:
        evs.evs_commit(st, -1)
    assert e.value.code == ERR_ARG
    evs.evs_commit(st, 3)
    for bad in ([], list(range(shape.n_block + 1))):
        with pytest.raises(evs.EvsError) as e:
            t = torch()
            tt = t.zeros(max(1, len(bad)), dtype=t.int32, device="cuda")
            lg = t.empty((max(1, len(bad)), shape.vocab), device="cuda")
            evs.evs_verify_block(st, tt, len(bad), lg)
        assert e.value.code == ERR_ARG
    assert st.check() == 0
    assert st.book()["pos"] == 3


@pytest.mark.gpu
def test_capacity_error_host_side():
    evs, shape, m, st = _tiny(12)
    _v(evs, st, [1, 2, 3, 4, 5], shape.vocab)
    evs.evs_commit(st, 5)
    _v(evs, st, [1, 2, 3, 4, 5], shape.vocab)
    evs.evs_commit(st, 5)
    with pytest.raises(evs.EvsError) as e:
        _v(evs, st, [1, 2, 3], shape.vocab)
    assert e.value.code == ERR_CAPACITY
    _v(evs, st, [1, 2], shape.vocab)     # exactly fills the cache
    evs.evs_commit(st, 2)
    assert st.check() == 0 and st.book()["pos"] == 12


@pytest.mark.gpu
def test_bad_token_sets_status():
    evs, shape, m, st = _tiny(64)
    lg = _v(evs, st, [1, shape.vocab + 5, 2], shape.vocab)
    assert np.isfinite(to_np(lg)).all()
    status = st.check()
    assert status & BAD_TOKEN


@pytest.mark.gpu
def test_device_keep_out_of_range_leaves_state():
    evs, shape, m, st = _tiny(64)
    t = torch()
    _v(evs, st, [1, 2, 3], shape.vocab)
    evs.evs_commit(st, 3)
    before = st.book()
    ref = to_np(_v(evs, st, [4], shape.vocab))
    evs.evs_commit(st, 0)
    _v(evs, st, [5, 6], shape.vocab)
    bad = t.tensor([20], dtype=t.int32, device="cuda")     # keep = 21 > n = 2
    evs.evs_commit_dev(st, bad)
    after = st.book()
    assert after["status"] & BAD_KEEP
    assert after["pos"] == before["pos"]
    assert after["pending_n"] == 0
    # the state is the one before the rejected block: same logits again
    st.set_book(status=0)
    got = to_np(_v(evs, st, [4], shape.vocab))
    assert np.array_equal(got, ref)


@pytest.mark.gpu
def test_kv_overflow_after_device_commits():
    evs, shape, m, st = _tiny(12)
    t = torch()
    acc = t.zeros(1, dtype=t.int32, device="cuda")
    tok = t.zeros(1, dtype=t.int32, device="cuda")
    n = shape.n_block
    for r in range(2):   # identity-style rounds committed on the device: pos 5, 10
        lg = _v(evs, st, [1, 2, 3, 4, 5], shape.vocab)
        acc.fill_(n - 1)
        evs.evs_commit_dev(st, acc)
    assert st.book()["pos"] == 10
    _v(evs, st, [1, 2, 3, 4, 5], shape.vocab)   # host no longer knows pos: device check
    status = st.check()
    assert status & KV_OVERFLOW


@pytest.mark.gpu
def test_allocation_limit_reports_oom_and_recovers(monkeypatch):
    import hybrid_ssm_attention_gb300 as evs
    shape = synth.tiny()
    m = evs.Model(shape, synth.make_weights(shape, 0))
    monkeypatch.setenv("EVS_ALLOC_LIMIT", "4096")
    with pytest.raises(evs.EvsError) as e:
        evs.State(m, 64)
    assert e.value.code == ERR_OOM
    monkeypatch.delenv("EVS_ALLOC_LIMIT")
    st = evs.State(m, 64)
    lg = _v(evs, st, [1, 2, 3], shape.vocab)
    assert np.isfinite(to_np(lg)).all() and st.check() == 0


@pytest.mark.gpu
def test_bounded_wait_expires_with_status():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    status = t.zeros(1, dtype=t.int32, device="cuda")
    evs.evs_selftest_wait_timeout(status, 2_000_000)
    t.cuda.synchronize()
    assert int(status.item()) == DEV_TIMEOUT
    # the context is still usable: a GEMM right after
    W = t.ones((128, 64), dtype=t.float32, device="cuda")
    X = t.ones((2, 64), dtype=t.float32, device="cuda")
    y = t.empty((2, 128), dtype=t.float32, device="cuda")
    scratch = t.empty(evs.evs_op_gemm_scratch_bytes(128, 64, evs.EVS_F32), dtype=t.uint8, device="cuda")
    evs.evs_op_gemm(W, X, 128, 64, 2, evs.EVS_F32, y, scratch)
    assert float(y.min().item()) == 64.0 and float(y.max().item()) == 64.0
    with pytest.raises(evs.EvsError):
        evs.evs_selftest_wait_timeout(status, 10_000_000_000)   # limit above 1 s is refused
