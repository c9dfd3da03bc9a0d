"""ctypes mirror of include/evs.h (structures, constants, prototypes).

Argument marshalling only; every step of the path runs in libevs.  Loading
fails loudly if the library was not built: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libevs.so")

EVS_OK, EVS_ERR_ARG, EVS_ERR_STATE, EVS_ERR_CAPACITY = 0, 1, 2, 3
EVS_ERR_OOM, EVS_ERR_CUDA, EVS_ERR_DEVICE, EVS_ERR_UNSUPPORTED = 4, 5, 6, 7
EVS_DEV_BAD_TOKEN, EVS_DEV_KV_OVERFLOW, EVS_DEV_BAD_KEEP, EVS_DEV_TIMEOUT, EVS_DEV_BAD_PROBS = 1, 2, 4, 8, 16
EVS_F32, EVS_BF16 = 0, 1
EVS_LAYER_FIR, EVS_LAYER_IIR, EVS_LAYER_ATTN = 0, 1, 2
EVS_GREEDY, EVS_SAMPLE = 0, 1
EVS_OPT_SWIGLU_EPILOGUE, EVS_OPT_NORM_IN_GEMM, EVS_OPT_GEMM_SUMS_SLOTS = 1, 2, 4

ERR_NAMES = {0: "EVS_OK", 1: "EVS_ERR_ARG", 2: "EVS_ERR_STATE", 3: "EVS_ERR_CAPACITY",
             4: "EVS_ERR_OOM", 5: "EVS_ERR_CUDA", 6: "EVS_ERR_DEVICE", 7: "EVS_ERR_UNSUPPORTED"}

vp, i32, i64, f32, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t


class evs_config(C.Structure):
    _fields_ = [("vocab", i32), ("d_model", i32), ("n_layers", i32), ("n_heads", i32),
                ("head_dim", i32), ("d_ffn", i32), ("gamma_max", i32), ("dtype", i32),
                ("attn_chunk", i32), ("rope_base", f32), ("norm_eps", f32), ("options", i32),
                ("layer_kind_host", C.POINTER(i32)), ("layer_param_host", C.POINTER(i32))]


class evs_layer_weights(C.Structure):
    _fields_ = [("w_in", vp), ("w_out", vp), ("w_gu", vp), ("w_down", vp),
                ("fir_taps", vp), ("iir_lambda", vp), ("iir_residue", vp)]


class evs_weights(C.Structure):
    _fields_ = [("embed", vp), ("lm_head", vp), ("layers_host", C.POINTER(evs_layer_weights))]


class evs_book(C.Structure):
    _fields_ = [("pos", i32), ("reserved0", i32), ("reserved1", i32), ("iir_bank", i32),
                ("iir_slot", i32), ("pending_n", i32), ("status", i32), ("reserved", i32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class evs_layer_view(C.Structure):
    _fields_ = [("kind", i32), ("param", i32), ("fir_ring", vp), ("reserved", vp), ("iir_all", vp * 2),
                ("k_cache", vp), ("v_cache", vp), ("ctx_max", i64), ("n_max", i32)]


PP = C.POINTER(vp)
PROTOTYPES = {
    "evs_model_create": (i32, [C.POINTER(evs_config), C.POINTER(evs_weights), PP]),
    "evs_model_destroy": (i32, [vp]),
    "evs_state_create": (i32, [vp, i64, PP]),
    "evs_state_destroy": (i32, [vp]),
    "evs_state_reset": (i32, [vp, vp]),
    "evs_state_clone": (i32, [vp, vp, vp]),
    "evs_state_snapshot": (i32, [vp, vp, vp]),
    "evs_state_layer_view": (i32, [vp, i32, C.POINTER(evs_layer_view)]),
    "evs_state_book_dev": (i32, [vp, PP]),
    "evs_state_book_read": (i32, [vp, C.POINTER(evs_book), vp]),
    "evs_state_book_write": (i32, [vp, C.POINTER(evs_book), vp]),
    "evs_state_check": (i32, [vp, vp, C.POINTER(i32)]),
    "evs_state_use_graphs": (i32, [vp, i32]),
    "evs_state_use_engine": (i32, [vp, i32]),
    "evs_verify_block": (i32, [vp, vp, i32, vp, vp]),
    "evs_verify_block_trace": (i32, [vp, vp, i32, vp, vp, vp]),
    "evs_verify_batch": (i32, [vp, i32, vp, vp, vp, vp]),
    "evs_probs": (i32, [vp, i32, i32, f32, i32, vp, vp]),
    "evs_accept": (i32, [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]),
    "evs_markov_draft": (i32, [vp, vp, i32, vp, vp, i32, f32, i32, i32, vp, vp, vp]),
    "evs_commit": (i32, [vp, i32, vp]),
    "evs_commit_dev": (i32, [vp, vp, vp]),
    "evs_round": (i32, [vp, vp, i32, vp, vp, vp, vp, f32, i32, i32, vp, vp, vp]),
    "evs_round_host": (i32, [vp, vp, i32, vp, vp, vp, vp, f32, i32, i32, vp, vp, vp]),
    "evs_round_batch": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, f32, i32, i32, vp, vp, vp]),
    "evs_profile_gemm_chain": (i32, [vp, i32, i32, C.POINTER(C.c_float), C.POINTER(i64), C.POINTER(i32), vp]),
    "evs_op_fir": (i32, [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]),
    "evs_op_iir": (i32, [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]),
    "evs_op_attention_scratch_bytes": (sz, [i32, i32, i64, i32, i32]),
    "evs_op_attention": (i32, [i32, i32, i32, i32, i64, i32, f32, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
    "evs_op_commit": (i32, [vp, i32, i32, vp]),
    "evs_op_gemm_scratch_bytes": (sz, [i32, i32, i32]),
    "evs_op_gemm": (i32, [vp, vp, i32, i32, i32, i32, vp, vp, sz, vp]),
    "evs_op_gemm_static": (i32, [vp, vp, i32, i32, i32, i32, vp, vp]),
    "evs_selftest_wait_timeout": (i32, [vp, i64, vp]),
    "evs_profile_gemms": (i32, [vp, i32, C.POINTER(C.c_float), C.POINTER(i64), i32, C.POINTER(i32), vp]),
    "evs_last_error": (C.c_char_p, []),
    "evs_version": (C.c_char_p, []),
    "evs_kernel_launches": (i64, []),
    "evs_verify_kernel_count": (i32, [vp, i32]),
}

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """The loaded libevs (raises if it is missing - build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libevs is not built ({path} missing); run __graft_entry__.build()")
    lib = C.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
