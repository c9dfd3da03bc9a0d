"""Hybrid Hyena / attention stack and native decoding (oracle, test infrastructure only).

Source.  The EvSpark pages (preprint abstract; discussion post, "The systems
problem") describe the target as a StripedHyena2 hybrid whose inference state
mixes three classes:
  * fixed-length FIR sliding windows,
  * infinite-memory IIR recurrent states,
  * append-only attention KV caches.
They print no operator equations.  The plainest reading, used here:

  residual stream x (float), per layer
      x += Mixer(RMSNorm(x));   x += MLP(RMSNorm(x))
  RMSNorm(x) = x / sqrt(mean(x^2) + eps), unit gains.
  Hyena mixer: [a | b | v] = W_in xn;  z = b * v;  y = h (*) z  (causal,
      depthwise per channel);  out = W_out (a * y).
      FIR ("SE" short, "MR" medium): y_t = sum_{j<L} h[j] z_{t-j};
          state = the last L-1 values of z.
      IIR ("LI", modal): s_t = lam * s_{t-1} + z_t  (per channel, per pole,
          complex), y_t = Re sum_m R_m s_t[m];  state = s.
          Equivalent to the FIR with h[t] = Re sum_m R_m lam_m^t (pinned).
  Attention: [q | k | v] = W_in xn, heads contiguous; rotary embedding
      (rotate-half, base 10000, angle = position * base^(-2i/Dh)) on q and k;
      k, v appended to the cache; softmax(q k^T / sqrt(Dh)) over keys at
      positions <= own; out = W_out concat_heads.
  MLP: W_down (silu(W_gate xn) * W_up xn).
  Head: logits = W_lm RMSNorm(x).

Native decoding (the model card's ``generate_native``): one token per step.
Block verify (discussion post, "What we implemented"; reply, prerequisite 1)
is *defined* here as n native steps on a copy of the state, recording after
each step the logits and the FIR window, IIR state and KV length.  Commit
keeps the record after ``keep`` steps (``keep = 0``: the state before the
block) - the per-position state slicing of the preprint abstract, (i).
"""
from __future__ import annotations

import copy
from typing import List

import numpy as np

from .numerics import Arith

SE, MR, LI, ATT = "SE", "MR", "LI", "ATT"


def rmsnorm(x, eps, ar: Arith):
    x = np.asarray(x, dtype=ar.dt)
    ms = np.mean(x * x, dtype=ar.dt)
    return x / np.sqrt(ms + ar.dt.type(eps))


def silu(g, ar: Arith):
    g = np.asarray(g, dtype=ar.dt)
    return g / (ar.dt.type(1) + np.exp(-g))


def rope_tables(pos: int, head_dim: int, base: float, ar: Arith):
    """cos / sin of the rotary angles at one position, evaluated in float64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = np.power(np.float64(base), -2.0 * i / head_dim)
    ang = np.float64(pos) * inv_freq
    return np.cos(ang).astype(ar.dt), np.sin(ang).astype(ar.dt)


def rope(x, pos: int, base: float, ar: Arith):
    """Rotate-half rotary embedding of x [H][Dh] at one position: the pair
    (x[i], x[i + Dh/2]) is turned by angle pos * base^(-2i/Dh)."""
    x = np.asarray(x, dtype=ar.dt)
    half = x.shape[-1] // 2
    c, s = rope_tables(pos, x.shape[-1], base, ar)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def attend(qh, K, V, ar: Arith):
    """One query per head against keys / values [T][H][Dh]; softmax over T."""
    Dh = qh.shape[-1]
    scale = ar.dt.type(1.0 / np.sqrt(Dh))
    out = np.empty_like(qh)
    for h in range(qh.shape[0]):
        s = (K[:, h, :] @ qh[h]) * scale
        w = np.exp(s - s.max())
        out[h] = (w @ V[:, h, :]) / w.sum()
    return out


class LayerState:
    """Decoding state of one layer: FIR window (oldest first), IIR modal state,
    or the KV cache (rows [0, length) valid)."""

    def __init__(self, kind, window=None, s=None, K=None, V=None, length=0):
        self.kind, self.window, self.s = kind, window, s
        self.K, self.V, self.length = K, V, length

    def copy(self):
        # The KV arrays are shared, not copied: a copy only ever appends at
        # rows >= its own length, which the original never reads (append-only).
        return LayerState(self.kind,
                          None if self.window is None else self.window.copy(),
                          None if self.s is None else self.s.copy(),
                          self.K, self.V, self.length)


class State:
    def __init__(self, layers: List[LayerState], pos: int):
        self.layers, self.pos = layers, pos

    def copy(self):
        return State([L.copy() for L in self.layers], self.pos)


class Model:
    """Weights (a dict as produced by the synthetic-input module, float arrays)
    plus shape constants.  ``ar`` fixes the arithmetic."""

    def __init__(self, shape, W, ar: Arith):
        self.shape, self.ar = shape, ar
        dt = ar.dt
        self.embed = np.asarray(W["embed"], dtype=dt)
        self.lm_head = np.asarray(W["lm_head"], dtype=dt)
        self.layers = []
        for L in W["layers"]:
            M = {"kind": L["kind"], "param": L["param"]}
            for k in ("w_in", "w_out", "w_gu", "w_down"):
                M[k] = np.asarray(L[k], dtype=dt)
            if "taps" in L:
                M["taps"] = np.asarray(L["taps"], dtype=dt)
            if "lam" in L:
                M["lam"] = np.asarray(L["lam"], dtype=ar.cdt)
                M["res"] = np.asarray(L["res"], dtype=ar.cdt)
            self.layers.append(M)

    # ------------------------------------------------------------------ state
    def new_state(self, capacity: int) -> State:
        """Zero FIR windows, zero IIR states, empty KV caches of ``capacity`` rows."""
        sh, ar = self.shape, self.ar
        d = sh.d_model
        out = []
        for M in self.layers:
            k = M["kind"]
            if k in (SE, MR):
                out.append(LayerState(k, window=np.zeros((M["param"] - 1, d), ar.dt)))
            elif k == LI:
                out.append(LayerState(k, s=np.zeros((d, M["param"]), ar.cdt)))
            else:
                shp = (capacity, sh.n_heads, sh.head_dim)
                out.append(LayerState(k, K=np.zeros(shp, ar.dt), V=np.zeros(shp, ar.dt)))
        return State(out, 0)

    def state_from(self, synth: dict, capacity: int) -> State:
        """State at committed length P from synthesised per-layer arrays
        (FIR window [L-1][d], IIR s [d][M], K/V [P][H][Dh] as float arrays)."""
        st = self.new_state(capacity)
        P = int(synth["P"])
        for L, S in zip(st.layers, synth["layers"]):
            if L.window is not None:
                L.window[...] = S["window"]
            elif L.s is not None:
                L.s[...] = S["s"]
            else:
                L.K[:P] = S["k"]
                L.V[:P] = S["v"]
                L.length = P
        st.pos = P
        return st

    # ------------------------------------------------------------------ mixers
    def fir_step(self, M, L: LayerState, z):
        """y_t = sum_j h[j] z_{t-j}; the window holds z_{t-L+1} .. z_{t-1}."""
        seq = np.concatenate([L.window, z[None, :]], axis=0)      # [L][d], oldest first
        taps = M["taps"]                                           # [L][d], taps[j] weights z_{t-j}
        y = np.sum(taps[::-1] * seq, axis=0, dtype=self.ar.dt)
        L.window = seq[1:].copy()
        return y

    def iir_step(self, M, L: LayerState, z):
        """s <- lam * s + z ; y = Re sum_m R_m s_m."""
        L.s = M["lam"] * L.s + z[:, None].astype(self.ar.cdt)
        return np.real(np.sum(M["res"] * L.s, axis=1)).astype(self.ar.dt)

    def attn_step(self, M, L: LayerState, u, pos):
        sh, ar = self.shape, self.ar
        H, Dh, d = sh.n_heads, sh.head_dim, sh.d_model
        q = u[:d].reshape(H, Dh)
        k = u[d:2 * d].reshape(H, Dh)
        v = u[2 * d:].reshape(H, Dh)
        q = ar.r(rope(q, pos, sh.rope_base, ar))
        k = ar.r(rope(k, pos, sh.rope_base, ar))
        if L.length >= L.K.shape[0]:
            raise ValueError("KV capacity exceeded")
        L.K[L.length], L.V[L.length] = k, v
        L.length += 1
        o = attend(q, L.K[:L.length], L.V[:L.length], ar)
        return o.reshape(d)

    # ------------------------------------------------------------------ step
    def embed_token(self, token: int):
        if not (0 <= int(token) < self.shape.vocab):
            raise ValueError("token out of range")
        return self.embed[int(token)].astype(self.ar.dt).copy()

    def layer_forward(self, M, L: LayerState, x, pos: int):
        """One layer for one token: x + Mixer(RMSNorm(x)), then + MLP(RMSNorm(.)).
        Updates the layer's state L in place."""
        sh, ar = self.shape, self.ar
        d, F, eps = sh.d_model, sh.d_ffn, sh.norm_eps
        xn = ar.r(rmsnorm(x, eps, ar))
        u = ar.r(ar.mv(M["w_in"], xn))
        if M["kind"] == ATT:
            g = ar.r(self.attn_step(M, L, u, pos))
        else:
            a, b, v = u[:d], u[d:2 * d], u[2 * d:]
            z = b * v
            y = self.fir_step(M, L, z) if M["kind"] in (SE, MR) else self.iir_step(M, L, z)
            g = ar.r(a * y)
        x = x + ar.mv(M["w_out"], g)
        xn = ar.r(rmsnorm(x, eps, ar))
        gu = ar.mv(M["w_gu"], xn)
        h = ar.r(silu(gu[:F], ar) * gu[F:])
        return x + ar.mv(M["w_down"], h)

    def head(self, x):
        """Final RMSNorm and LM head."""
        return self.ar.mv(self.lm_head, self.ar.r(rmsnorm(x, self.shape.norm_eps, self.ar)))

    def step(self, st: State, token: int):
        """One native decode step: consumes ``token`` at position st.pos,
        updates every layer's state in place, returns the logits."""
        x = self.embed_token(token)
        for M, L in zip(self.layers, st.layers):
            x = self.layer_forward(M, L, x, st.pos)
        st.pos += 1
        return self.head(x)

    # ------------------------------------------------------------------ block
    def verify(self, st: State, tokens):
        """Block verify of tokens[0..n-1] from state ``st`` (unchanged).

        Returns (logits [n][V], records) where records[i] is the state after
        consuming tokens[0..i]; the GPU's single pass must reproduce both."""
        work = st.copy()
        logits, records = [], []
        for t in tokens:
            logits.append(self.step(work, int(t)))
            records.append(work.copy())
        return np.stack(logits), records

    @staticmethod
    def commit(st: State, records, keep: int) -> State:
        """State sliced to the accepted boundary: keep in [0, n] consumed tokens."""
        if not (0 <= keep <= len(records)):
            raise ValueError("keep out of range")
        return st.copy() if keep == 0 else records[keep - 1].copy()
