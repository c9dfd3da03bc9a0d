"""Operator GEMM on the library's static scratch (evs_op_gemm_static)
against evs_op_gemm on caller scratch: results within the GEMM tests'
tolerance of each other, on two calls in a row; no device memory taken
across calls; shapes whose scratch exceeds the static array are refused.

Collected last (file name) so that it runs after every other GPU test as
well as alone.
"""
import numpy as np
import pytest

import synth
from gpu_util import rel_err, to_np, torch, up


def _f(bits):
    return synth.bf16_bits_to_f32(bits)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,N,K,n", [("bf16", 22016, 4096, 13), ("bf16", 4096, 11008, 16),
                                         ("bf16", 128, 64, 1), ("f32", 300, 100, 16)])
def test_static_scratch_gemm_matches_caller_scratch_gemm(dtype, N, K, n):
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    g = np.random.default_rng(N * 7 + K)
    if dtype == "bf16":
        code = evs.EVS_BF16
        W = up(synth._to_bf16_bits_trunc(g.standard_normal((N, K), dtype=np.float32) * 0.02))
        X = up(synth._to_bf16_bits_trunc(g.standard_normal((n, K), dtype=np.float32)))
    else:
        code = evs.EVS_F32
        W = up(g.standard_normal((N, K)).astype(np.float32))
        X = up(g.standard_normal((n, K)).astype(np.float32))
    scratch = t.empty(evs.evs_op_gemm_scratch_bytes(N, K, code), dtype=t.uint8, device="cuda")
    assert scratch.numel() <= 4 << 20             # fits the static array
    ref = t.empty((n, N), dtype=t.float32, device="cuda")
    evs.evs_op_gemm(W, X, N, K, n, code, ref, scratch)
    ys = [t.full((n, N), float("nan"), dtype=t.float32, device="cuda") for _ in range(3)]
    evs.evs_op_gemm_static(W, X, N, K, n, code, ys[0])      # first call on the device: symbol lookup
    t.cuda.synchronize()
    free0 = t.cuda.mem_get_info()[0]
    evs.evs_op_gemm_static(W, X, N, K, n, code, ys[1])      # two calls in a row
    evs.evs_op_gemm_static(W, X, N, K, n, code, ys[2])
    t.cuda.synchronize()
    assert t.cuda.mem_get_info()[0] == free0
    r = to_np(ref).astype(np.float64)
    for y in ys:
        a = to_np(y)
        assert np.isfinite(a).all()
        assert rel_err(a, r) <= 1e-5


@pytest.mark.gpu
def test_static_scratch_gemm_refuses_oversized_plan():
    import hybrid_ssm_attention_gb300 as evs
    t = torch()
    N, K, n = 1024 * 128, 4096, 4          # 1024 column tiles: partial slots beyond the static array
    assert evs.evs_op_gemm_scratch_bytes(N, K, evs.EVS_BF16) > 4 << 20
    W = t.zeros((N, K), dtype=t.bfloat16, device="cuda")
    X = t.zeros((n, K), dtype=t.bfloat16, device="cuda")
    y = t.zeros((n, N), dtype=t.float32, device="cuda")
    with pytest.raises(evs.EvsError) as e:
        evs.evs_op_gemm_static(W, X, N, K, n, evs.EVS_BF16, y)
    assert "EVS_ERR_CAPACITY" in str(e.value)
    assert float(y.abs().max().item()) == 0.0
