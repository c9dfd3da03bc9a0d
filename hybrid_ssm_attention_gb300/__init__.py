"""Python binding of libevs: the block-verify / accept / commit path of lossless
speculative decoding for StripedHyena2-style hybrid models (EvSpark).

The functions below carry the C names of include/evs.h and only marshal
arguments (torch device tensors -> raw pointers, the current torch stream ->
cudaStream_t).  PyTorch provides device memory and streams; every step of the
path runs in the CUDA kernels of libevs.so.  If the library is missing the
first call raises - there is no fallback.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional, Sequence

import numpy as np

from . import _abi
from ._abi import (EVS_BF16, EVS_ERR_ARG, EVS_ERR_CAPACITY, EVS_ERR_CUDA, EVS_ERR_DEVICE,  # noqa: F401
                   EVS_ERR_OOM, EVS_ERR_STATE, EVS_ERR_UNSUPPORTED, EVS_F32, EVS_GREEDY, EVS_LAYER_ATTN,
                   EVS_LAYER_FIR, EVS_LAYER_IIR, EVS_OPT_GEMM_SUMS_SLOTS, EVS_OPT_NORM_IN_GEMM,
                   EVS_OPT_SWIGLU_EPILOGUE, EVS_SAMPLE, evs_book, evs_layer_view)

__all__ = ["EvsError", "Model", "State", "lib", "evs_verify_block", "evs_verify_block_trace", "evs_probs", "evs_accept",
           "evs_commit", "evs_commit_dev", "evs_markov_draft", "evs_round", "evs_round_host", "evs_round_batch", "evs_op_fir", "evs_op_iir",
           "evs_op_attention", "evs_op_commit", "evs_op_gemm", "evs_op_gemm_static", "evs_verify_batch",
           "evs_kernel_launches"]

KIND_CODES = {"SE": EVS_LAYER_FIR, "MR": EVS_LAYER_FIR, "FIR": EVS_LAYER_FIR,
              "LI": EVS_LAYER_IIR, "IIR": EVS_LAYER_IIR, "ATT": EVS_LAYER_ATTN, "ATTN": EVS_LAYER_ATTN}


class EvsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_abi.ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


def lib():
    return _abi.load()


def _check(rc: int, what: str):
    if rc != 0:
        raise EvsError(rc, f"{what}: {lib().evs_last_error().decode()}")


def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("device tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _to_device(a: np.ndarray, dtype_code: int):
    """numpy -> CUDA tensor: uint16 arrays are bf16 bit patterns."""
    torch = _torch()
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    if np.iscomplexobj(a):
        a = np.ascontiguousarray(a.astype(np.complex64)).view(np.float32)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


class Model:
    """An evs_model plus the device copies of its weights (kept alive here).

    ``shape`` needs vocab, d_model, layers [(kind, param)], n_heads, head_dim,
    d_ffn, gamma, dtype ("bf16" | "f32"), attn_chunk, rope_base, norm_eps;
    ``weights`` is the dict layout of the synthetic-input module (numpy)."""

    def __init__(self, shape, weights: dict, options: int = 0):
        self.shape = shape
        self.dtype = EVS_BF16 if shape.dtype == "bf16" else EVS_F32
        self.tensors = []
        up = lambda a: self._keep(_to_device(a, self.dtype))  # noqa: E731
        nl = len(shape.layers)
        kinds = (C.c_int32 * nl)(*[KIND_CODES[k] for k, _ in shape.layers])
        params = (C.c_int32 * nl)(*[int(p) for _, p in shape.layers])
        self._kinds, self._params = kinds, params
        cfg = _abi.evs_config(vocab=shape.vocab, d_model=shape.d_model, n_layers=nl,
                              n_heads=shape.n_heads, head_dim=shape.head_dim, d_ffn=shape.d_ffn,
                              gamma_max=shape.gamma, dtype=self.dtype, attn_chunk=shape.attn_chunk,
                              rope_base=shape.rope_base, norm_eps=shape.norm_eps, options=int(options),
                              layer_kind_host=kinds, layer_param_host=params)
        lw = (_abi.evs_layer_weights * nl)()
        for i, L in enumerate(weights["layers"]):
            lw[i].w_in = _ptr(up(L["w_in"]))
            lw[i].w_out = _ptr(up(L["w_out"]))
            lw[i].w_gu = _ptr(up(L["w_gu"]))
            lw[i].w_down = _ptr(up(L["w_down"]))
            if "taps" in L:
                lw[i].fir_taps = _ptr(up(L["taps"]))
            if "lam" in L:
                lw[i].iir_lambda = _ptr(up(L["lam"]))
                lw[i].iir_residue = _ptr(up(L["res"]))
        w = _abi.evs_weights(embed=_ptr(up(weights["embed"])), lm_head=_ptr(up(weights["lm_head"])),
                             layers_host=lw)
        h = C.c_void_p()
        _check(lib().evs_model_create(C.byref(cfg), C.byref(w), C.byref(h)), "evs_model_create")
        self.handle = h

    def _keep(self, t):
        self.tensors.append(t)
        return t

    def close(self):
        if getattr(self, "handle", None):
            lib().evs_model_destroy(self.handle)
            self.handle = None
        self.tensors = []

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


class State:
    """An evs_state (library-owned FIR / IIR banks, KV caches, workspaces)."""

    def __init__(self, model: Model, ctx_max: int):
        self.model = model
        h = C.c_void_p()
        _check(lib().evs_state_create(model.handle, int(ctx_max), C.byref(h)), "evs_state_create")
        self.handle = h
        self.ctx_max = int(ctx_max)

    def close(self):
        if getattr(self, "handle", None):
            lib().evs_state_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    def reset(self, stream=None):
        _check(lib().evs_state_reset(self.handle, _stream(stream)), "evs_state_reset")

    def view(self, layer: int) -> evs_layer_view:
        v = evs_layer_view()
        _check(lib().evs_state_layer_view(self.handle, layer, C.byref(v)), "evs_state_layer_view")
        return v

    def book(self, stream=None) -> dict:
        b = evs_book()
        _check(lib().evs_state_book_read(self.handle, C.byref(b), _stream(stream)), "evs_state_book_read")
        return b.as_dict()

    def set_book(self, stream=None, **fields):
        b = evs_book()
        cur = self.book(stream)
        cur.update(fields)
        for k, v in cur.items():
            setattr(b, k, int(v))
        _check(lib().evs_state_book_write(self.handle, C.byref(b), _stream(stream)), "evs_state_book_write")

    def book_dev(self) -> int:
        p = C.c_void_p()
        _check(lib().evs_state_book_dev(self.handle, C.byref(p)), "evs_state_book_dev")
        return p.value

    def check(self, stream=None) -> int:
        st = C.c_int32()
        rc = lib().evs_state_check(self.handle, _stream(stream), C.byref(st))
        if rc not in (0, _abi.EVS_ERR_DEVICE):
            _check(rc, "evs_state_check")
        return st.value

    def use_graphs(self, on: bool):
        _check(lib().evs_state_use_graphs(self.handle, int(bool(on))), "evs_state_use_graphs")

    def use_engine(self, on: bool):
        """Single-sequence verifies through the persistent engine (on by default where the model allows)."""
        _check(lib().evs_state_use_engine(self.handle, int(bool(on))), "evs_state_use_engine")

    def clone_into(self, dst: "State", stream=None):
        _check(lib().evs_state_clone(self.handle, dst.handle, _stream(stream)), "evs_state_clone")

    def snapshot_into(self, dst: "State", stream=None):
        """Recurrent state + bookkeeping only (KV caches are append-only)."""
        _check(lib().evs_state_snapshot(self.handle, dst.handle, _stream(stream)), "evs_state_snapshot")


# ------------------------------------------------------------------ C-named calls
def evs_verify_block(state: State, tokens, n: int, logits, stream=None):
    _check(lib().evs_verify_block(state.handle, _ptr(tokens), int(n), _ptr(logits), _stream(stream)),
           "evs_verify_block")


def evs_verify_block_trace(state: State, tokens, n: int, logits, x_trace, stream=None):
    _check(lib().evs_verify_block_trace(state.handle, _ptr(tokens), int(n), _ptr(logits), _ptr(x_trace),
                                        _stream(stream)), "evs_verify_block_trace")


def evs_probs(logits, n: int, V: int, T: float, top_k: int, p, stream=None):
    _check(lib().evs_probs(_ptr(logits), int(n), int(V), float(T), int(top_k), _ptr(p), _stream(stream)),
           "evs_probs")


def evs_accept(p, q, drafts, u, n: int, V: int, mode: int, out_accepted, out_token, stream=None):
    _check(lib().evs_accept(_ptr(p), _ptr(q), _ptr(drafts), _ptr(u), int(n), int(V), int(mode),
                            _ptr(out_accepted), _ptr(out_token), _stream(stream)), "evs_accept")


def evs_markov_draft(trunk_logits, markov, V: int, prev, u, gamma: int, T: float, top_k: int, mode: int, drafts, q,
                     stream=None):
    """Drafter-side Markov head: gamma sequential draws from trunk rows plus Markov rows."""
    _check(lib().evs_markov_draft(_ptr(trunk_logits), _ptr(markov), int(V), _ptr(prev), _ptr(u), int(gamma),
                                  float(T), int(top_k), int(mode), _ptr(drafts), _ptr(q), _stream(stream)),
           "evs_markov_draft")


def evs_commit(state: State, keep: int, stream=None):
    _check(lib().evs_commit(state.handle, int(keep), _stream(stream)), "evs_commit")


def evs_commit_dev(state: State, accepted, stream=None):
    _check(lib().evs_commit_dev(state.handle, _ptr(accepted), _stream(stream)), "evs_commit_dev")


def evs_round(state: State, tokens, n: int, logits, p, q, u, T: float, top_k: int, mode: int,
              out_accepted, out_token, stream=None):
    _check(lib().evs_round(state.handle, _ptr(tokens), int(n), _ptr(logits), _ptr(p), _ptr(q), _ptr(u),
                           float(T), int(top_k), int(mode), _ptr(out_accepted), _ptr(out_token),
                           _stream(stream)), "evs_round")


def evs_round_host(state: State, tokens, n: int, logits, p, q, u, T: float, top_k: int, mode: int, stream=None):
    """One round with the block in host memory (int32 numpy array or
    sequence); returns (accepted, token) as Python ints."""
    import numpy as _np
    tok = _np.ascontiguousarray(_np.asarray(tokens, dtype=_np.int32)[:n])
    acc = (C.c_int32 * 1)()
    otok = (C.c_int32 * 1)()
    _check(lib().evs_round_host(state.handle, tok.ctypes.data, int(n), _ptr(logits), _ptr(p), _ptr(q), _ptr(u),
                                float(T), int(top_k), int(mode), C.cast(acc, C.c_void_p), C.cast(otok, C.c_void_p),
                                _stream(stream)), "evs_round_host")
    return int(acc[0]), int(otok[0])


def evs_round_batch(states, tokens, ns, logits, p, q, u, T: float, top_k: int, mode: int, out_accepted, out_token,
                    stream=None):
    """One graph launch: batched verify, then every sequence's accept and commit on the device."""
    arr = (C.c_void_p * len(states))(*[st.handle for st in states])
    nh = (C.c_int32 * len(ns))(*[int(x) for x in ns])
    _check(lib().evs_round_batch(arr, len(states), _ptr(tokens), nh, _ptr(logits), _ptr(p), _ptr(q), _ptr(u),
                                 float(T), int(top_k), int(mode), _ptr(out_accepted), _ptr(out_token),
                                 _stream(stream)), "evs_round_batch")


def evs_op_fir(L, d, n, n_max, dtype, abv, taps, ring, book_dev, g, stream=None):
    _check(lib().evs_op_fir(L, d, n, n_max, dtype, _ptr(abv), _ptr(taps), _ptr(ring), _ptr(book_dev), _ptr(g),
                            _stream(stream)), "evs_op_fir")


def evs_op_iir(M, d, n, n_max, dtype, abv, lam, res, st0, st1, book_dev, g, stream=None):
    _check(lib().evs_op_iir(M, d, n, n_max, dtype, _ptr(abv), _ptr(lam), _ptr(res), _ptr(st0), _ptr(st1),
                            _ptr(book_dev), _ptr(g), _stream(stream)), "evs_op_iir")


def evs_op_attention_scratch_bytes(H, Dh, ctx_max, chunk, n_max) -> int:
    return int(lib().evs_op_attention_scratch_bytes(H, Dh, ctx_max, chunk, n_max))


def evs_op_attention(H, Dh, n, n_max, ctx_max, chunk, rope_base, dtype, qkv, kc, vc, book_dev, g,
                     scratch, stream=None):
    _check(lib().evs_op_attention(H, Dh, n, n_max, ctx_max, chunk, float(rope_base), dtype, _ptr(qkv),
                                  _ptr(kc), _ptr(vc), _ptr(book_dev), _ptr(g), _ptr(scratch),
                                  scratch.numel() * scratch.element_size(), _stream(stream)),
           "evs_op_attention")


def evs_op_commit(book_dev, keep: int, n: int, stream=None):
    _check(lib().evs_op_commit(_ptr(book_dev), int(keep), int(n), _stream(stream)), "evs_op_commit")


def evs_op_gemm_scratch_bytes(N, K, dtype) -> int:
    return int(lib().evs_op_gemm_scratch_bytes(N, K, dtype))


def evs_op_gemm(w, x, N, K, n, dtype, y, scratch, stream=None):
    _check(lib().evs_op_gemm(_ptr(w), _ptr(x), N, K, n, dtype, _ptr(y), _ptr(scratch),
                             scratch.numel() * scratch.element_size(), _stream(stream)), "evs_op_gemm")


def evs_op_gemm_static(w, x, N, K, n, dtype, y, stream=None):
    _check(lib().evs_op_gemm_static(_ptr(w), _ptr(x), N, K, n, dtype, _ptr(y), _stream(stream)),
           "evs_op_gemm_static")


def evs_selftest_wait_timeout(status, limit_ns, stream=None):
    _check(lib().evs_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)), "evs_selftest_wait_timeout")


def evs_verify_batch(states, tokens, ns, logits, stream=None):
    """One verify pass over several sequences' blocks (rows back to back)."""
    arr = (C.c_void_p * len(states))(*[st.handle for st in states])
    nh = (C.c_int32 * len(ns))(*[int(x) for x in ns])
    _check(lib().evs_verify_batch(arr, len(states), _ptr(tokens), nh, _ptr(logits), _stream(stream)),
           "evs_verify_batch")


def evs_kernel_launches() -> int:
    return int(lib().evs_kernel_launches())


def evs_verify_kernel_count(state: State, n: int) -> int:
    return int(lib().evs_verify_kernel_count(state.handle, int(n)))


def evs_profile_gemm_chain(state: State, n: int, reps: int = 10, stream=None):
    """(ms per chain, algorithmic bytes per chain, launches per chain) of the step's GEMMs back to back."""
    ms = C.c_float()
    by = C.c_int64()
    cnt = C.c_int32()
    _check(lib().evs_profile_gemm_chain(state.handle, int(n), int(reps), C.byref(ms), C.byref(by), C.byref(cnt),
                                        _stream(stream)), "evs_profile_gemm_chain")
    return float(ms.value), int(by.value), int(cnt.value)


def evs_profile_gemms(state: State, n: int, stream=None):
    """Per-launch (ms, algorithmic bytes) of one verify step's weight GEMMs."""
    cap = 4 * len(state.model.shape.layers) + 1
    ms = (C.c_float * cap)()
    by = (C.c_int64 * cap)()
    cnt = C.c_int32()
    _check(lib().evs_profile_gemms(state.handle, int(n), ms, by, cap, C.byref(cnt), _stream(stream)),
           "evs_profile_gemms")
    return [float(ms[i]) for i in range(cnt.value)], [int(by[i]) for i in range(cnt.value)]
