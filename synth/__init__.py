"""Seeded synthetic workloads for the block-verify / accept / commit path.

This module is shared by both sides of every parity test: it produces model
shapes, random-init weights, prompts, uniforms, drafter distributions and
synthesised decoding state. It holds none of the method's arithmetic (no
normalisation, projection, filter, attention, softmax of the target, accept
rule or state slicing); everything it returns is an input.

All randomness is NumPy PCG64 seeded through ``SeedSequence`` so that the CUDA
path and the CPU oracle see bit-identical inputs.

Shapes follow the workloads of *EvSpark: Lossless Speculative Decoding for
Hybrid DNA Foundation Models* (abstract; model-card "Numbers" paragraph): a
StripedHyena2-style stack of short/medium FIR, modal IIR and attention layers,
bf16 weights, gamma = 12. The real Evo2 weights and the genomic prompt suite
are not available; random-init weights and ACGT-uniform prompts stand in for
them.
"""
from __future__ import annotations

import dataclasses
import concurrent.futures as _cf
import os
from typing import List, Optional, Tuple

import numpy as np

# Layer kinds.  "SE" and "MR" are explicit causal FIR filters (short / medium),
# "LI" a modal IIR filter with diagonal complex poles, "ATT" multi-head
# attention over an append-only KV cache.
SE, MR, LI, ATT = "SE", "MR", "LI", "ATT"

# ASCII codes of A, C, G, T: the nucleotide token ids of a byte-level DNA LM.
ACGT_IDS = (65, 67, 71, 84)


@dataclasses.dataclass
class ModelShape:
    name: str
    vocab: int
    d_model: int
    layers: List[Tuple[str, int]]        # (kind, L for FIR | poles for LI | 0 for ATT)
    n_heads: int
    head_dim: int
    d_ffn: int
    gamma: int                            # draft length; a verify block holds gamma + 1 tokens
    dtype: str                            # "f32" or "bf16": storage type of weights / activations
    pole_mag: Tuple[float, float] = (0.9, 0.999)
    weight_std: float = 0.02
    residue_std: float = 0.25
    rope_base: float = 10000.0
    norm_eps: float = 1e-6
    attn_chunk: int = 64                  # keys per split-KV chunk on the GPU (absolute, fixed)

    @property
    def n_block(self) -> int:
        return self.gamma + 1


def tiny() -> ModelShape:
    """fp32 tiny hybrid: vocab 16, d 64, [FIR short 4, IIR 8 poles, attention 2x32]."""
    return ModelShape(name="tiny", vocab=16, d_model=64,
                      layers=[(SE, 4), (LI, 8), (ATT, 0)], n_heads=2, head_dim=32,
                      d_ffn=256, gamma=4, dtype="f32", pole_mag=(0.9, 0.99))


def stack_7b(n_layers: int = 32, d_model: int = 4096, d_ffn: int = 11008,
             n_heads: int = 32, head_dim: int = 128, vocab: int = 512,
             short_len: int = 7, medium_len: int = 128, poles: int = 16,
             gamma: int = 12, name: str = "7b") -> ModelShape:
    """7B-shaped stack: attention at every 6th layer (i % 6 == 5), the other
    layers cycle FIR-short / FIR-medium / IIR in that order."""
    layers: List[Tuple[str, int]] = []
    j = 0
    for i in range(n_layers):
        if i % 6 == 5:
            layers.append((ATT, 0))
        else:
            layers.append([(SE, short_len), (MR, medium_len), (LI, poles)][j % 3])
            j += 1
    return ModelShape(name=name, vocab=vocab, d_model=d_model, layers=layers,
                      n_heads=n_heads, head_dim=head_dim, d_ffn=d_ffn, gamma=gamma,
                      dtype="bf16", pole_mag=(0.9, 0.999))


def single_layer(kind: str, param: int = 0, d_model: int = 4096, d_ffn: int = 11008,
                 vocab: int = 512, gamma: int = 12, n_heads: int = 32,
                 head_dim: int = 128, dtype: str = "bf16") -> ModelShape:
    """One-layer bf16 model at d_model 4096 (Hyena layer or attention layer)."""
    return ModelShape(name=f"one-{kind}", vocab=vocab, d_model=d_model,
                      layers=[(kind, param)], n_heads=n_heads, head_dim=head_dim,
                      d_ffn=d_ffn, gamma=gamma, dtype=dtype, pole_mag=(0.9, 0.999))


# --------------------------------------------------------------------------
# random streams
# --------------------------------------------------------------------------

def _streams(seed: int, count: int) -> List[np.random.Generator]:
    return [np.random.Generator(np.random.PCG64(s))
            for s in np.random.SeedSequence(seed).spawn(count)]


def _normal_f32(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    out *= np.float32(std)
    return out


def _to_bf16_bits_trunc(x: np.ndarray) -> np.ndarray:
    """bf16 bit pattern of a float32 array by dropping the low 16 bits.
    Used only to *make* random bf16 inputs (a draw from a slightly
    zero-biased normal), never to round a computed value."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (an input-format decode)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


_POOL_THREADS = max(1, min(16, os.cpu_count() or 1))


def _big_normal_bf16(seed_seq: np.random.SeedSequence, shape, std: float) -> np.ndarray:
    """Large bf16 weight draw, row blocks filled by parallel PCG64 streams."""
    rows = shape[0]
    out = np.empty(shape, dtype=np.uint16)
    nblk = max(1, min(rows, 64))
    bounds = np.linspace(0, rows, nblk + 1).astype(np.int64)
    seeds = seed_seq.spawn(nblk)

    def work(b):
        r0, r1 = int(bounds[b]), int(bounds[b + 1])
        if r1 > r0:
            g = np.random.Generator(np.random.PCG64(seeds[b]))
            out[r0:r1] = _to_bf16_bits_trunc(_normal_f32(g, (r1 - r0,) + tuple(shape[1:]), std))

    with _cf.ThreadPoolExecutor(_POOL_THREADS) as ex:
        list(ex.map(work, range(nblk)))
    return out


def _dense(seed_seq, shape, std, dtype):
    if dtype == "bf16":
        return _big_normal_bf16(seed_seq, shape, std)
    g = np.random.Generator(np.random.PCG64(seed_seq))
    return _normal_f32(g, shape, std)


def make_weights(shape: ModelShape, seed: int) -> dict:
    """Random-init weights.

    Dense matrices are N(0, weight_std) in the shape's storage dtype
    (bf16 as uint16 bit patterns, f32 as float32), row-major [out][in]:
      embed [V][d], lm_head [V][d]; per layer w_in [3d][d] (rows a|b|v for
      Hyena, q|k|v for attention, heads contiguous), w_out [d][d],
      w_gu [2F][d] (rows 0..F-1 gate, F..2F-1 up), w_down [d][F].
    FIR taps [L][d] float32 ~ N(0, 1/sqrt(L)).
    IIR poles lam [d][M] complex64, |lam| ~ U(pole_mag), arg ~ U(-pi, pi);
    residues res [d][M] complex64 with Re, Im iid N(0, residue_std).
    """
    d, F, V = shape.d_model, shape.d_ffn, shape.vocab
    ss = np.random.SeedSequence(seed)
    top, *per_layer = ss.spawn(1 + len(shape.layers))
    s_embed, s_head = top.spawn(2)
    W = {"embed": _dense(s_embed, (V, d), shape.weight_std, shape.dtype),
         "lm_head": _dense(s_head, (V, d), shape.weight_std, shape.dtype),
         "dtype": shape.dtype, "layers": []}
    for (kind, param), lss in zip(shape.layers, per_layer):
        s_in, s_out, s_gu, s_dn, s_f = lss.spawn(5)
        L = {"kind": kind, "param": param,
             "w_in": _dense(s_in, (3 * d, d), shape.weight_std, shape.dtype),
             "w_out": _dense(s_out, (d, d), shape.weight_std, shape.dtype),
             "w_gu": _dense(s_gu, (2 * F, d), shape.weight_std, shape.dtype),
             "w_down": _dense(s_dn, (d, F), shape.weight_std, shape.dtype)}
        g = np.random.Generator(np.random.PCG64(s_f))
        if kind in (SE, MR):
            L["taps"] = _normal_f32(g, (param, d), 1.0 / np.sqrt(param))
        elif kind == LI:
            L["lam"], L["res"] = _poles(g, d, param, shape.pole_mag, shape.residue_std)
        W["layers"].append(L)
    return W


def _poles(g, d, M, mag, res_std):
    r = g.uniform(mag[0], mag[1], size=(d, M))
    th = g.uniform(-np.pi, np.pi, size=(d, M))
    lam = (r * np.cos(th) + 1j * r * np.sin(th)).astype(np.complex64)
    res = (g.standard_normal((d, M)) * res_std + 1j * g.standard_normal((d, M)) * res_std)
    return lam, res.astype(np.complex64)


def weights_f32(W: dict) -> dict:
    """A float32 view of a weight dict (bf16 patterns widened exactly)."""
    if W["dtype"] == "f32":
        return W
    conv = bf16_bits_to_f32
    out = {"embed": conv(W["embed"]), "lm_head": conv(W["lm_head"]), "dtype": "f32",
           "layers": []}
    for L in W["layers"]:
        M = dict(L)
        for k in ("w_in", "w_out", "w_gu", "w_down"):
            M[k] = conv(L[k])
        out["layers"].append(M)
    return out


# --------------------------------------------------------------------------
# prompts, uniforms, drafters
# --------------------------------------------------------------------------

def prompt(shape: ModelShape, seed: int, length: int) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1])))
    if shape.vocab > max(ACGT_IDS):
        return np.asarray(ACGT_IDS, dtype=np.int32)[g.integers(0, 4, size=length)]
    return g.integers(0, shape.vocab, size=length).astype(np.int32)


def uniforms(seed: int, rounds: int, n: int) -> np.ndarray:
    """float32 uniforms in [0, 1), one row of n per verify round."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 2])))
    return g.random((rounds, n), dtype=np.float32)


def fixed_logit_drafter(seed: int, gamma: int, vocab: int) -> np.ndarray:
    """Drafter with random fixed logits N(0, 1) per draft slot; returns its
    distributions q [gamma][V] (float32).  The drafter is not part of the
    verified path; its softmax lives here with its other inputs."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 3])))
    z = g.standard_normal((gamma, vocab))
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def draw_from(q_row: np.ndarray, u: float) -> int:
    """Inverse-CDF draw of a draft token from a drafter distribution."""
    c = np.cumsum(q_row.astype(np.float64))
    return int(min(np.searchsorted(c, u * c[-1], side="right"), len(q_row) - 1))


def draft_uniforms(seed: int, rounds: int, gamma: int) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 4])))
    return g.random((rounds, gamma))


def logit_noise(seed: int, rounds: int, gamma: int, vocab: int, std: float = 0.5) -> np.ndarray:
    """Noise of the noise drafter: float32 [rounds][gamma][vocab] ~ N(0, std)
    (std is the standard deviation).  The drafter proposes draft i from
    q_i = softmax(top-k(target logits along the draft path + noise[i])); the
    arithmetic of that softmax lives with the caller, the draws here."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 13])))
    return _normal_f32(g, (rounds, gamma, vocab), std)


def markov_matrix(seed: int, vocab: int, std: float = 1.0) -> np.ndarray:
    """Random-init full V x V Markov matrix of the drafter head, float32 ~ N(0, std)."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 14])))
    return _normal_f32(g, (vocab, vocab), std)


def drafter_trunk_standin(vocab: int = 512, gamma: int = 12) -> ModelShape:
    """Timing stand-in for the drafter trunk (random init, no trained
    weights exist): one attention layer at d_model 1024 (8 heads x 128,
    MLP 4096), scoring gamma draft slots in one pass."""
    return ModelShape(name="drafter-trunk-standin", vocab=vocab, d_model=1024, layers=[(ATT, 0)], n_heads=8,
                      head_dim=128, d_ffn=4096, gamma=gamma, dtype="bf16")


def keep_draws(seed: int, rounds: int, n: int, kind: str = "uniform") -> np.ndarray:
    """Commit lengths: U{0..n} or Geometric(1/3) on {1, 2, ...} clipped to n."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 5])))
    if kind == "uniform":
        return g.integers(0, n + 1, size=rounds).astype(np.int32)
    return np.minimum(g.geometric(1.0 / 3.0, size=rounds), n).astype(np.int32)


# --------------------------------------------------------------------------
# synthesised decoding state (stands in for a long prefill)
# --------------------------------------------------------------------------

def synth_state(shape: ModelShape, seed: int, P: int, ctx_max: Optional[int] = None) -> dict:
    """Random decoding state at committed length P.

    FIR windows [L-1][d] float32 ~ N(0, 1) (oldest first); IIR states [d][M]
    complex64 with Re, Im ~ N(0, sqrt 2) (standard deviation sqrt 2); KV caches [P][H][Dh] ~ N(0, 1) in the
    storage dtype.  Layers are listed in model order; a field is None where
    the layer kind has no such state."""
    ss = np.random.SeedSequence([seed, 6])
    streams = ss.spawn(len(shape.layers))
    d, H, Dh = shape.d_model, shape.n_heads, shape.head_dim
    out = {"P": P, "layers": []}
    for (kind, param), s in zip(shape.layers, streams):
        g = np.random.Generator(np.random.PCG64(s))
        st = {"kind": kind, "window": None, "s": None, "k": None, "v": None}
        if kind in (SE, MR):
            st["window"] = _normal_f32(g, (param - 1, d), 1.0)
        elif kind == LI:
            st["s"] = (g.standard_normal((d, param)) * np.sqrt(2.0)
                       + 1j * g.standard_normal((d, param)) * np.sqrt(2.0)).astype(np.complex64)
        else:
            sk, sv = s.spawn(2)
            st["k"] = _dense(sk, (P, H, Dh), 1.0, shape.dtype) if P else np.zeros((0, H, Dh), np.uint16 if shape.dtype == "bf16" else np.float32)
            st["v"] = _dense(sv, (P, H, Dh), 1.0, shape.dtype) if P else np.zeros((0, H, Dh), np.uint16 if shape.dtype == "bf16" else np.float32)
        out["layers"].append(st)
    return out


def mixer_params(seed: int, kind: str, param: int, d: int, pole_mag=(0.9, 0.999),
                 residue_std: float = 0.25) -> dict:
    """Filter parameters of one Hyena layer with the recipe of make_weights:
    FIR taps [L][d] ~ N(0, 1/sqrt(L)); IIR poles / residues [d][M] complex64."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 8])))
    if kind in (SE, MR):
        return {"taps": _normal_f32(g, (param, d), 1.0 / np.sqrt(param))}
    lam, res = _poles(g, d, param, pole_mag, residue_std)
    return {"lam": lam, "res": res}


def layer_state(seed: int, kind: str, param: int, d: int, P: int = 0, n_heads: int = 0,
                head_dim: int = 0, dtype: str = "bf16") -> dict:
    """Synthesised state of one layer with the recipe of synth_state."""
    shape = ModelShape(name="one", vocab=1, d_model=d, layers=[(kind, param)], n_heads=n_heads,
                       head_dim=head_dim, d_ffn=1, gamma=0, dtype=dtype)
    return synth_state(shape, seed, P)["layers"][0]


def kv_head(seed: int, head: int, P: int, head_dim: int) -> tuple:
    """Long-context cache rows of one attention head: K and V [P][head_dim]
    ~ N(0, 1), bf16 bit patterns (one head at a time, so a 262k-position
    cache can be synthesised for the heads a test samples)."""
    k = _dense(np.random.SeedSequence([seed, 11, head]), (P, head_dim), 1.0, "bf16")
    v = _dense(np.random.SeedSequence([seed, 12, head]), (P, head_dim), 1.0, "bf16")
    return k, v


def abv_block(seed: int, n: int, d: int, dtype: str = "bf16") -> np.ndarray:
    """Mixer inputs for an operator-level test: [n][3d] ~ N(0, 1) (a | b | v)."""
    ss = np.random.SeedSequence([seed, 7])
    return _dense(ss, (n, 3 * d), 1.0, dtype)
