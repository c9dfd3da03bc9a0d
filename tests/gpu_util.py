"""Helpers for the -m gpu parity tests (no test functions here)."""
import numpy as np

BF16 = "<i2"


def torch():
    import torch as t
    return t


class _CAI:
    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def wrap(ptr, shape, typestr="<f4"):
    """Zero-copy torch view of library-owned device memory."""
    t = torch()
    return t.as_tensor(_CAI(ptr, shape, typestr), device="cuda")


def to_np(t_):
    t = torch()
    if t_.dtype == t.bfloat16:
        return (t_.contiguous().view(t.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32)
    return t_.detach().cpu().numpy()


def up(a, dtype=None):
    """numpy -> cuda tensor; uint16 arrays are bf16 bit patterns."""
    t = torch()
    if a.dtype == np.uint16:
        return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(t.bfloat16)
    if np.iscomplexobj(a):
        return t.from_numpy(np.ascontiguousarray(a.astype(np.complex64)).view(np.float32)).cuda()
    return t.from_numpy(np.ascontiguousarray(a, dtype=dtype or a.dtype)).cuda()


def rel_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def book_zero(t):
    """A device evs_book at position 0 (iir_slot = -1)."""
    b = t.zeros(8, dtype=t.int32, device="cuda")
    b[4] = -1
    return b


def noise_drafts(evs, st, snap, pending, noise, du, T=1.0, top_k=4):
    """The noise drafter: gamma = len(du) drafts along its own path.

    Draft i + 1 is drawn (inverse CDF, uniform du[i]) from q_i, the
    library's top-k softmax at temperature T of the target's native logits
    after the path so far plus noise[i] (N(0, 0.5) draws from the input
    generators).  The native steps run on st itself between a snapshot of
    its recurrent state and the restore (KV rows they append lie beyond the
    committed length and are rewritten by the next verify).  Returns
    (drafts, q as a [gamma][V] numpy array, q as a device tensor)."""
    import synth
    t = torch()
    gamma, V = noise.shape
    st.snapshot_into(snap)
    lg = t.empty((1, V), dtype=t.float32, device="cuda")
    tk = t.empty(1, dtype=t.int32, device="cuda")
    qd = t.empty((gamma, V), dtype=t.float32, device="cuda")
    drafts, cur = [], int(pending)
    for i in range(gamma):
        tk.fill_(cur)
        evs.evs_verify_block(st, tk, 1, lg)
        evs.evs_commit(st, 1)
        noisy = up((to_np(lg)[0] + noise[i]).astype(np.float32)[None])
        evs.evs_probs(noisy, 1, V, T, top_k, qd[i:i + 1])
        cur = synth.draw_from(to_np(qd[i]), float(du[i]))
        drafts.append(cur)
    snap.snapshot_into(st)
    return drafts, to_np(qd), qd


def fir_ext(ring, L, n_max, pos, n):
    """Positions pos-L+1 .. pos+n-1 of a FIR ring [L-1+n_max][d] (position p at
    row p mod (L-1+n_max)): the committed window followed by a block's n inputs,
    so row i+1 .. i+L-1 is the window after block position i."""
    R = L - 1 + n_max
    return ring[[p % R for p in range(pos - L + 1, pos + n)]]


def fir_set_window(ring_t, L, n_max, pos, window_t):
    """Place the window of a state at position pos (positions pos-L+1 .. pos-1)."""
    t = torch()
    R = L - 1 + n_max
    idx = t.tensor([(pos - L + 1 + r) % R for r in range(L - 1)], device=ring_t.device)
    ring_t[idx] = window_t
