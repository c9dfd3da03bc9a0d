"""The C ABI library loads and exports every function include/evs.h declares,
and the ctypes binding mirrors all of them (no GPU needed: no compute call)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "evs.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(evs_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from hybrid_ssm_attention_gb300 import build as b
    b.build()
    import hybrid_ssm_attention_gb300._abi as abi
    return abi.load()


def test_header_declares_the_path():
    names = declared_functions()
    for must in ("evs_verify_block", "evs_accept", "evs_commit", "evs_commit_dev", "evs_probs",
                 "evs_model_create", "evs_state_create", "evs_round", "evs_op_fir", "evs_op_iir",
                 "evs_op_attention", "evs_op_gemm"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    import hybrid_ssm_attention_gb300._abi as abi
    names = declared_functions()
    assert len(names) >= 25
    for n in names:
        assert hasattr(lib, n), n
        assert n in abi.PROTOTYPES, f"binding lacks {n}"
    assert set(abi.PROTOTYPES) <= set(names)


def test_version_and_error_without_gpu(lib):
    assert lib.evs_version().startswith(b"evs")
    # argument errors are reported before any device work
    import ctypes
    assert lib.evs_commit(None, 0, None) == 1
    assert b"null" in lib.evs_last_error()
    assert lib.evs_op_commit(None, 0, 1, None) == 1
    assert lib.evs_probs(None, 1, 1, 1.0, 0, None, None) == 1
    assert lib.evs_accept(ctypes.c_void_p(16), None, None, None, 2, 4, 9, ctypes.c_void_p(16),
                          ctypes.c_void_p(16), None) == 1


def test_struct_layouts_match_header():
    import ctypes
    import hybrid_ssm_attention_gb300._abi as abi
    assert ctypes.sizeof(abi.evs_book) == 32
    assert ctypes.sizeof(abi.evs_config) == 12 * 4 + 16   # 12 ints / floats, 2 pointers
    assert ctypes.sizeof(abi.evs_layer_weights) == 7 * 8
