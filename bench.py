#!/usr/bin/env python
"""Benchmark of the block-verify / accept / commit round at gamma = 12.

Workload: the 7B-shaped random-init hybrid stack (32 layers, d_model 4096,
gated MLP 11008, FIR-short / FIR-medium / IIR with attention every 6th
layer, vocab 512, bf16 weights ~13 GB), a 1024-token ACGT prompt, greedy
decoding with the identity drafter (drafts = the target's own native greedy
continuation, precomputed on the GPU outside the timed region, as in the
identity-drafter measurement of the EvSpark discussion post).

One step = one round: block verify of 13 tokens (pending + 12 drafts),
accept, commit - all in one CUDA graph on one stream.  Metric: accepted
tokens per second (emitted tokens / summed round time; drafter excluded),
plus verify-round latency and HBM bandwidth against the roofline.

Inputs (weights 13 GB, KV) are larger than L2, so no flush is needed.
Under torchrun every rank runs an independent replica (the path does not
shard); value = all ranks' tokens / the slowest rank's time.

--impl reference times the CPU oracle (test infrastructure) on the host
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "accepted tok/s at gamma=12 (block verify + accept + commit, identity drafter, greedy)"
UNIT = "tok/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="evs", choices=["evs", "reference"])
    ap.add_argument("--prompt", type=int, default=1024)
    ap.add_argument("--seed", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-replay", action="store_true")
    ap.add_argument("--no-batch", action="store_true")
    ap.add_argument("--long-gen", type=int, default=32768,
                    help="also generate this many tokens natively and speculatively (drafts with random "
                         "corrupted tails) and report whether the two sequences are identical (0: skip)")
    ap.add_argument("--no-sampled", action="store_true")
    ap.add_argument("--no-drafter", action="store_true")
    ap.add_argument("--no-long-context", action="store_true")
    ap.add_argument("--long-context", type=int, default=262144, help="cached positions of the long-context rounds")
    ap.add_argument("--cpu-one-thread-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--case", nargs="+", metavar=("KIND", "ARG"),
                    help="instead of the benchmark, launch one small profiler case and exit: "
                         "gemm N K n | fir L d n | iir M d n | attn P n | stack L n | batch L B n | markov V k")
    ap.add_argument("--reps", type=int, default=4, help="repetitions of a --case launch")
    return ap.parse_args()


# ------------------------------------------------------------------ ranks
def dist_setup(gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.lines, self.proc = gpu, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        return self.summarize(self.lines)

    @staticmethod
    def summarize(lines):
        """Median SM clock, the largest max clock and every throttle reason
        seen Active, from `--format=csv,noheader,nounits` lines of Q."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                a, b = float(f[1]), float(f[2])
            except ValueError:
                continue
            sm.append(a)
            mx.append(b)
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# DRAM traffic per GEMM launch (dram__bytes_read.sum + dram__bytes_write.sum,
# averaged over the 129 weight GEMMs of a step) from one ncu capture of the
# weight-streaming GEMM; valid only for the kernel source it was taken on
# (sha256 prefix of gemm.cu), else reported as null.
GEMM_TRAFFIC = {"gemm_cu_sha256": "1a29fdda8bf3055c", "bytes_per_launch": 100.88e6}


def gemm_traffic():
    import hashlib
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "hybrid_ssm_attention_gb300", "csrc", "gemm.cu")
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    return GEMM_TRAFFIC["bytes_per_launch"] if h == GEMM_TRAFFIC["gemm_cu_sha256"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ algorithmic bytes
def step_bytes(shape, P, n):
    """Bytes one verify round must move: weights once, each mixer's state
    read + retained per-position state written, KV read + append, logits."""
    d, F, V, es = shape.d_model, shape.d_ffn, shape.vocab, 2
    H, Dh = shape.n_heads, shape.head_dim
    b = (4 * d * d + 3 * d * F) * es * len(shape.layers) + V * d * es + n * d * es + n * V * 4
    for kind, prm in shape.layers:
        if kind in ("SE", "MR"):
            b += (prm - 1) * d * 4 + (prm - 1 + n) * d * 4 + prm * d * 4
        elif kind == "LI":
            b += prm * d * 8 * 3 + n * prm * d * 8
        else:
            b += (P + n) * H * Dh * es * 2 + n * H * Dh * es * 2
    return b


WORKLOAD = ("7B-shaped hybrid stack: 32 layers (FIR7/FIR128/IIR16, attention every 6th), d_model 4096, MLP 11008, "
            "vocab 512, bf16 weights 12.96 GB; 1024-token ACGT prompt; gamma=12; identity drafter, greedy")


def config(args, world, n, rounds):
    return {"workload": WORKLOAD, "gamma": 12, "context_start": args.prompt, "generated_tokens": n * rounds,
            "l2": "inputs larger than L2 (13 GB of weights per step), no flush",
            "parallelism": f"replicas x{world}"}


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: the
    implementer and part codes, plus the kernel's model string if any)."""
    fields = {}
    try:
        for ln in open("/proc/cpuinfo"):
            k, _, v = ln.partition(":")
            fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    for k in ("model name", "cpu model", "hardware"):
        if fields.get(k):
            return fields[k]
    if "cpu implementer" in fields:
        return f"Arm CPU implementer {fields['cpu implementer']} part {fields.get('cpu part', '?')}"
    import platform
    return platform.processor() or platform.machine()


def blas_threads():
    """Threads the oracle's matrix products run on (the BLAS pool)."""
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


# ------------------------------------------------------------------ oracle timing
def oracle_round_tokens_per_s(shape, W, seed, P, rounds, native_steps, warm=0):
    """The oracle's own speculative round on the same workload: a verify of
    the 13-token identity-drafter block (13 native steps on a copy, every
    position's state recorded), the accept rule and the commit; plus
    `native_steps` plain native steps.  The identity drafts (the oracle's own
    greedy continuation) are made outside the timed part, as on the GPU.
    Returns tok/s of the rounds (emitted tokens / round time), seconds per
    round and seconds per native step."""
    import synth
    from oracle.decode import native_generate
    from oracle.model import Model as OModel
    from oracle.numerics import Arith
    from oracle.sampling import GREEDY, accept
    om = OModel(shape, synth.weights_f32(W), Arith(np.float32, bf16_points=True))
    S = synth.synth_state(shape, seed, P)
    S["layers"] = [dict(L, k=None if L["k"] is None else synth.bf16_bits_to_f32(L["k"]),
                        v=None if L["v"] is None else synth.bf16_bits_to_f32(L["v"])) for L in S["layers"]]
    n = shape.n_block
    st = om.state_from(S, P + 2 * n * (warm + rounds + 1) + native_steps + 2)
    pend = int(synth.prompt(shape, seed, 1)[0])
    t0 = time.perf_counter()
    native_generate(om, st.copy(), pend, native_steps)
    t_native = (time.perf_counter() - t0) / max(native_steps, 1)
    t_round, emitted = 0.0, 0
    for r in range(warm + rounds):
        drafts, _ = native_generate(om, st.copy(), pend, n - 1)
        t0 = time.perf_counter()
        logits, rec = om.verify(st, [pend] + drafts)
        a, tok = accept(logits, None, drafts, np.zeros(n, np.float32), GREEDY)
        st = OModel.commit(st, rec, a + 1)
        if r >= warm:
            t_round += time.perf_counter() - t0
            emitted += a + 1
        pend = tok
    if rounds == 0:
        return None, None, t_native
    return emitted / t_round, t_round / rounds, t_native


def cpu_baseline(args, shape, W):
    """The oracle as the reported CPU baseline: all host cores, then one
    thread (a child process with one BLAS thread), on bounded samples."""
    rounds, native = 8, 16  # ~20 s timed on 16 cores (~35 s with the untimed drafts)
    tps, t_round, t_native = oracle_round_tokens_per_s(shape, W, args.seed, args.prompt, rounds, native)
    out = {"value": tps, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
           "cpu": cpu_model(), "host_cores": os.cpu_count(),
           "sample": f"{rounds} oracle rounds (13-token identity-drafter block verify = 13 native steps on a copy, "
                     f"accept, commit; drafts made outside the timed part) + {native} native steps of the same "
                     f"stack from context {args.prompt}, fp32 with bf16 storage points; value = emitted tokens / "
                     f"round time",
           "rounds": rounds, "round_s": t_round, "native_steps": native, "native_step_s": t_native,
           "native_tok_s": 1.0 / t_native}
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-one-thread-child", "--seed",
                            str(args.seed), "--prompt", str(args.prompt)], env=env, capture_output=True, text=True,
                           timeout=600)
        one = json.loads(r.stdout.strip().splitlines()[-1])
        out["one_thread"] = one
    except Exception as e:  # reported, not fatal: the all-cores figure stands
        out["one_thread"] = {"error": str(e)[:200]}
    return out


def run_cpu_one_thread_child(args):
    import synth
    shape = synth.stack_7b()
    W = synth.make_weights(shape, args.seed)
    _, _, t_native = oracle_round_tokens_per_s(shape, W, args.seed, args.prompt, 0, 1)
    print(json.dumps({"tok_s": 1.0 / t_native, "native_step_s": t_native, "threads": blas_threads(),
                      "sample": "1 oracle native step (a round of 13 costs 13 of them)"}))


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step one oracle round of the
    GPU arm's workload (identity-drafter block verify of 13 tokens, accept,
    commit), drafts made outside the timed part; rank 0 only."""
    if rank != 0:
        return
    import synth
    shape = synth.stack_7b()
    W = synth.make_weights(shape, args.seed)
    n = shape.n_block
    tps, t_round, t_native = oracle_round_tokens_per_s(shape, W, args.seed, args.prompt, args.steps, 1,
                                                       warm=args.warmup)
    sample = (f"{args.steps} oracle rounds after {args.warmup} warm-up rounds (13-token identity-drafter block "
              f"verify, accept, commit; fp32 with bf16 storage points) from context {args.prompt}")
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_round,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config(args, world, n, args.warmup + args.steps),
            "cpu_baseline": {"value": tps, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "cpu": cpu_model(), "sample": sample, "native_step_s": t_native},
            "e2e": {"value": tps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def long_generation(evs, torch, model, shape, prompt, ntok, seed, dev):
    """Greedy generation of ntok tokens twice from the same prompt: native
    (one token per round) and speculative (gamma=12 drafts = the native
    continuation with the tail after a random cut replaced by random tokens,
    so every round has an accepted prefix, a rejection or a bonus).  Also
    times the prompt's chunked prefill (block verify with keep = n)."""
    n = shape.n_block
    P0 = len(prompt)
    ctx = P0 + ntok + 2 * n
    st = evs.State(model, ctx)
    lg = torch.empty((n, shape.vocab), dtype=torch.float32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for s0 in range(0, P0 - 1, n):
        blk = torch.tensor(prompt[s0:min(s0 + n, P0 - 1)], dtype=torch.int32, device=dev)
        evs.evs_verify_block(st, blk, blk.numel(), lg[:blk.numel()])
        evs.evs_commit(st, blk.numel())
    e1.record()
    torch.cuda.synchronize()
    prefill_ms = e0.elapsed_time(e1)
    snap = evs.State(model, ctx)
    st.clone_into(snap)
    # native
    y = torch.empty(ntok + 1, dtype=torch.int32, device=dev)
    y[0] = prompt[-1]
    tok1 = y[:1].clone()
    lg1 = torch.empty((1, shape.vocab), dtype=torch.float32, device=dev)
    acc = torch.zeros(1, dtype=torch.int32, device=dev)
    otok = torch.zeros(1, dtype=torch.int32, device=dev)
    e0.record()
    for i in range(ntok):
        evs.evs_round(st, tok1, 1, lg1, None, None, None, 1.0, 0, evs.EVS_GREEDY, acc, otok)
        tok1.copy_(otok)
        y[i + 1:i + 2].copy_(otok)
    e1.record()
    torch.cuda.synchronize()
    native_ms = e0.elapsed_time(e1)
    native = y.cpu().numpy()
    # speculative, drafts built on the host from the native sequence
    snap.clone_into(st)
    g = np.random.default_rng(seed)
    out = []
    pend = int(native[0])
    toks = torch.empty(n, dtype=torch.int32, device=dev)
    rounds = 0
    accepted = 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    while len(out) < ntok:
        k = len(out)
        nxt = [int(v) for v in native[k + 1:k + n]]
        drafts = (nxt + [0] * (n - 1))[:n - 1]
        cut = int(g.integers(0, n))
        drafts = drafts[:cut] + [int(v) for v in g.integers(0, shape.vocab, n - 1 - cut)]
        toks.copy_(torch.tensor([pend] + drafts, dtype=torch.int32))
        evs.evs_round(st, toks, n, lg, None, None, None, 1.0, 0, evs.EVS_GREEDY, acc, otok)
        a, x = int(acc.item()), int(otok.item())
        out += drafts[:a] + [x]
        pend = x
        rounds += 1
        accepted += a
    spec_s = time.perf_counter() - t0
    out = np.asarray(out[:ntok], np.int64)
    ref = native[1:ntok + 1].astype(np.int64)
    mism = np.nonzero(out != ref)[0]
    st.close()
    snap.close()
    return {"tokens": ntok, "identical": bool(mism.size == 0),
            "first_mismatch": int(mism[0]) if mism.size else None,
            "native_ms_per_token": native_ms / ntok, "spec_rounds": rounds,
            "mean_accepted_per_round": accepted / rounds,
            "spec_tok_s_host_driven": ntok / spec_s,
            "prefill": {"tokens": P0 - 1, "ms": prefill_ms, "tok_s": (P0 - 1) / (prefill_ms / 1e3)},
            "context_end": P0 + ntok}


def batched_sweep(evs, torch, model, shape, post_prompt, ctx, dev, y, rounds=24, warm=4):
    """Batched rounds (evs_round_batch: one graph per round doing one verify
    pass over B sequences' blocks of n rows, then every sequence's accept and
    commit on the device).  Up to B * n = 16 rows the GEMMs take one 16-row
    chunk, beyond that 2..8 chunks side by side (up to 128 rows).  Every
    sequence starts from the post-prompt state and is fed the identity
    drafter's blocks (y: the target's own greedy continuation), so every
    draft is accepted (asserted).  Reports round time and verified rows per
    second for each (B, n)."""
    out = []
    V = shape.vocab
    for B, n in ((1, 13), (2, 8), (4, 4), (8, 2), (16, 1), (2, 13), (4, 13), (8, 13), (16, 8), (1, 1), (2, 1),
                 (4, 1), (8, 1)):
        states = [evs.State(model, ctx) for _ in range(B)]
        for st in states:
            post_prompt.clone_into(st)
        lg = torch.empty((B * n, V), dtype=torch.float32, device=dev)
        rounds = min(rounds, y.numel() // n - warm)  # the identity blocks available
        toks = y[: n * (rounds + warm)].view(rounds + warm, 1, n).expand(rounds + warm, B, n).reshape(
            rounds + warm, B * n).contiguous()
        acc = torch.zeros(B, dtype=torch.int32, device=dev)
        tok = torch.zeros(B, dtype=torch.int32, device=dev)
        acc_log = torch.zeros((rounds + warm, B), dtype=torch.int32, device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for r in range(rounds + warm):
            if r == warm:
                torch.cuda.synchronize()
                e0.record()
            evs.evs_round_batch(states, toks[r], [n] * B, lg, None, None, None, 1.0, 0, evs.EVS_GREEDY, acc, tok)
            acc_log[r].copy_(acc)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / rounds
        all_acc = bool((acc_log == n - 1).all().item())
        out.append({"B": B, "n": n, "rows": B * n, "ms_per_round": ms, "rows_per_s": B * n / (ms / 1e3),
                    "all_accepted": all_acc})
        for st in states:
            st.close()
    return out


def crossover(sweep):
    """Batched speculative verification against batched native decoding of
    the same B sequences: native = one row per sequence per pass (B x 1);
    speculative = the widest block pass per sequence measured (B x 13 up to
    104 rows, 16 x 8 at B = 16).  A speculative round emits (accepted + 1)
    tokens per sequence against one per native pass, so it wins once
    accepted + 1 > spec_ms / native_ms (the break-even tokens per round);
    at full acceptance the speedup is n * native_ms / spec_ms."""
    ms = {(r["B"], r["n"]): r["ms_per_round"] for r in sweep}
    out = []
    for B in (1, 2, 4, 8, 16):
        widths = [k[1] for k in ms if k[0] == B]
        if not widths:
            continue
        n = 13 if (B, 13) in ms else max(widths)
        if (B, 1) not in ms or n == 1:
            continue
        out.append({"B": B, "native_ms": ms[(B, 1)], "spec_n": n, "spec_ms": ms[(B, n)],
                    "break_even_tokens_per_round": ms[(B, n)] / ms[(B, 1)],
                    "speedup_all_accepted": n * ms[(B, 1)] / ms[(B, n)]})
    return out


def noise_drafts(evs, torch, st, snap, pending, noise, du, dev, T=1.0, top_k=4):
    """The noise drafter (outside every timed region): draft i + 1 is drawn
    (inverse CDF, uniform du[i]) from q_i, the library's top-k softmax of the
    target's native logits along the draft path plus noise[i].  The native
    steps run on st between a snapshot of its recurrent state and the
    restore; the KV rows they append lie beyond the committed length and are
    rewritten by the next verify.  Returns (drafts, q on the device)."""
    import synth
    gamma, V = noise.shape
    st.snapshot_into(snap)
    lg = torch.empty((1, V), dtype=torch.float32, device=dev)
    tk = torch.empty(1, dtype=torch.int32, device=dev)
    q = torch.empty((gamma, V), dtype=torch.float32, device=dev)
    drafts, cur = [], int(pending)
    for i in range(gamma):
        tk.fill_(cur)
        evs.evs_verify_block(st, tk, 1, lg)
        evs.evs_commit(st, 1)
        noisy = torch.from_numpy((lg.cpu().numpy()[0] + noise[i]).astype(np.float32)[None]).to(dev)
        evs.evs_probs(noisy, 1, V, T, top_k, q[i:i + 1])
        cur = synth.draw_from(q[i].cpu().numpy(), float(du[i]))
        drafts.append(cur)
    snap.snapshot_into(st)
    return drafts, q


def sampled_rounds(evs, torch, model, shape, post_prompt, ctx, dev, pending, seed, rounds=8, warm=2):
    """Sampled decoding (T = 1.0, top_k = 4) with the noise drafter (q = top-4
    softmax of the target's logits along the draft path plus N(0, 0.5)
    noise), from the post-prompt state.  A first pass alternates drafter and
    round (each round one graph launch: verify, target distribution, accept,
    commit), recording every round's block, q and uniforms; the timed pass
    restores the post-prompt state and runs the same rounds back to back
    (their results repeat the first pass bit for bit, asserted), with CUDA
    events around the whole sequence, as the greedy measurement does."""
    import synth
    n, V, gamma = shape.n_block, shape.vocab, shape.gamma
    st, snap = evs.State(model, ctx), evs.State(model, ctx)
    post_prompt.clone_into(st)
    R = warm + rounds
    noise = synth.logit_noise(seed, R, gamma, V)
    du = synth.draft_uniforms(seed, R, gamma)
    U = torch.from_numpy(synth.uniforms(seed, R, n)).to(dev)
    lg = torch.empty((n, V), dtype=torch.float32, device=dev)
    p = torch.empty((n, V), dtype=torch.float32, device=dev)
    q = torch.empty((gamma, V), dtype=torch.float32, device=dev)
    u = torch.empty(n, dtype=torch.float32, device=dev)
    acc = torch.zeros(1, dtype=torch.int32, device=dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    toks = torch.empty(n, dtype=torch.int32, device=dev)
    blocks = torch.empty((R, n), dtype=torch.int32, device=dev)
    qs = torch.empty((R, gamma, V), dtype=torch.float32, device=dev)
    results, draft_s = [], 0.0
    for r in range(R):
        t0 = time.perf_counter()
        drafts, qr = noise_drafts(evs, torch, st, snap, pending, noise[r], du[r], dev)
        torch.cuda.synchronize()
        draft_s += time.perf_counter() - t0 if r >= warm else 0.0
        blocks[r].copy_(torch.tensor([pending] + drafts, dtype=torch.int32))
        qs[r].copy_(qr)
        toks.copy_(blocks[r])
        q.copy_(qs[r])
        u.copy_(U[r])
        evs.evs_round(st, toks, n, lg, p, q, u, 1.0, 4, evs.EVS_SAMPLE, acc, tok)
        results.append((int(acc.item()), int(tok.item())))
        pending = results[-1][1]
    # timed pass: the same rounds back to back from the post-prompt state
    post_prompt.clone_into(st)
    acc_log = torch.zeros((R, 2), dtype=torch.int32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for r in range(R):
        if r == warm:
            torch.cuda.synchronize()
            e0.record()
        toks.copy_(blocks[r])
        q.copy_(qs[r])
        u.copy_(U[r])
        evs.evs_round(st, toks, n, lg, p, q, u, 1.0, 4, evs.EVS_SAMPLE, acc, tok)
        acc_log[r, 0:1].copy_(acc)
        acc_log[r, 1:2].copy_(tok)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    replay = [tuple(int(x) for x in row) for row in acc_log.cpu().numpy()]
    ok = st.check() == 0 and replay == results
    st.close()
    snap.close()
    accepted = [a for a, _ in results[warm:]]
    emitted = sum(a + 1 for a in accepted)
    return {"value": emitted / (ms / 1e3), "unit": UNIT, "rounds": rounds, "ms_per_round": ms / rounds,
            "mean_accepted_per_round": float(np.mean(accepted)), "accepted": accepted,
            "replay_identical_and_status_ok": ok, "drafter_ms_per_round_host": 1e3 * draft_s / rounds,
            "note": "T=1.0, top_k=4; noise drafter q_i = top-4 softmax(target logits along the draft path + "
                    "N(0, 0.5)); rounds (one graph each: verify 13, probs, accept, commit) timed back to back "
                    "with CUDA events on a replay of the drafter-driven pass; drafter untimed (12 native "
                    "steps + host draws per round)"}


def drafter_rounds(evs, torch, dev, seed, prompt_len, rounds=16, warm=4):
    """The drafter side, as a timing stand-in (no trained drafter exists):
    per round the trunk stand-in (one attention layer at d_model 1024,
    random init) scores the gamma draft slots in one verify pass and commits
    the pending token, then the Markov head kernel draws the gamma drafts
    from its rows (T = 1, top_k = 4).  Rounds back to back; CUDA events
    around each part of each round, read at the end."""
    import synth
    shape = synth.drafter_trunk_standin()
    gamma, V = shape.gamma, shape.vocab
    m = evs.Model(shape, synth.make_weights(shape, seed))
    st = evs.State(m, prompt_len + warm + rounds + 2 * gamma)
    pr = torch.from_numpy(synth.prompt(shape, seed, prompt_len)).to(dev)
    lg = torch.empty((gamma, V), dtype=torch.float32, device=dev)
    for s0 in range(0, prompt_len - 1, gamma):
        k = min(gamma, prompt_len - 1 - s0)
        evs.evs_verify_block(st, pr[s0:s0 + k], k, lg[:k])
        evs.evs_commit(st, k)
    M = torch.from_numpy(synth.markov_matrix(seed, V)).to(dev)
    U = torch.from_numpy(synth.uniforms(seed, warm + rounds, gamma)).to(dev)
    toks = torch.from_numpy(synth.prompt(shape, seed + 1, (warm + rounds) * gamma).reshape(-1, gamma)).to(dev)
    d = torch.zeros(gamma, dtype=torch.int32, device=dev)
    q = torch.empty((gamma, V), dtype=torch.float32, device=dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(rounds)]

    def one(r, e):
        if e:
            e[0].record()
        evs.evs_verify_block(st, toks[r], gamma, lg)
        evs.evs_commit(st, 1)
        if e:
            e[1].record()
        evs.evs_markov_draft(lg, M, V, toks[r, :1], U[r], gamma, 1.0, 4, evs.EVS_SAMPLE, d, q)
        if e:
            e[2].record()

    for r in range(warm):
        one(r, None)
    torch.cuda.synchronize()
    # the device sleeps while the host queues every timed round behind it,
    # so the events time the device, not the Python calls between them
    # (without torch's sleep kernel the rounds run as queued; queued_ahead
    # then reports false)
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(100_000_000)
    for r in range(rounds):
        one(warm + r, ev[r])
    queued_ahead = not ev[-1][2].query()
    torch.cuda.synchronize()
    trunk = sum(e[0].elapsed_time(e[1]) for e in ev) / rounds
    head = sum(e[1].elapsed_time(e[2]) for e in ev) / rounds
    total = ev[0][0].elapsed_time(ev[-1][2]) / rounds
    ok = st.check() == 0
    st.close()
    m.close()
    return {"us_per_round": 1e3 * total, "trunk_us": 1e3 * trunk, "markov_head_us": 1e3 * head, "status_ok": ok,
            "queued_ahead": queued_ahead,
            "note": "timing stand-in, random init: trunk = one attention layer at d_model 1024 (8x128 heads, MLP "
                    "4096, vocab 512) scoring 12 slots in one verify pass; Markov head = the evs_markov_draft "
                    "kernel (12 sequential top-4 draws over trunk row + V x V Markov row); the rounds are queued "
                    "behind a device sleep, so the events time the device (queued_ahead: the host had queued "
                    "the last round before the device reached it)"}


def long_context_rounds(evs, torch, model, shape, P, seed, dev, peak, rounds=6, warm=2):
    """The same stack over a synthesised long context: FIR windows and IIR
    states from the input generators, every attention layer's cache holding
    P rows of device filler N(0, 1) (the values do not change the work).
    Each round is a verify of 13 tokens, the accept rule (greedy, then
    sampled at T = 1, top_k = 4) and a commit of a length drawn geometric
    with mean 3; rounds run back to back, timed with CUDA events."""
    import synth
    n, V, d = shape.n_block, shape.vocab, shape.d_model
    H, Dh = shape.n_heads, shape.head_dim
    ctx = P + n * 2 * (warm + rounds) + n
    st = evs.State(model, ctx)
    S = synth.synth_state(shape, seed, 0)
    gen = torch.Generator(device=dev).manual_seed(seed)
    for li, (kind, param) in enumerate(shape.layers):
        v = st.view(li)
        L = S["layers"][li]
        if kind in ("SE", "MR"):
            # the window is positions P-L+1 .. P-1, ring row p mod (L-1+n_max)
            w = torch.from_numpy(L["window"]).to(dev)
            R = param - 1 + v.n_max
            idx = torch.tensor([(P - param + 1 + r) % R for r in range(param - 1)], device=dev)
            _dev_view(torch, v.fir_ring, (R, d), torch.float32)[idx] = w
        elif kind == "LI":
            s2 = torch.from_numpy(np.ascontiguousarray(L["s"]).view(np.float32)).to(dev)
            _dev_view(torch, v.iir_all[0], (v.n_max, d * param * 2), torch.float32)[0] = s2.reshape(-1)
        else:
            for ptr in (v.k_cache, v.v_cache):
                _dev_view(torch, ptr, (H, ctx, Dh), torch.bfloat16).normal_(generator=gen)
    torch.cuda.synchronize()
    st.set_book(pos=P, iir_bank=0, iir_slot=0, pending_n=0, status=0)
    keeps = synth.keep_draws(seed, 2 * (warm + rounds), n, kind="geometric")
    q = torch.from_numpy(synth.fixed_logit_drafter(seed, n - 1, V)).to(dev)
    U = torch.from_numpy(synth.uniforms(seed, 2 * (warm + rounds), n)).to(dev)
    toks = torch.from_numpy(synth.prompt(shape, seed, 2 * (warm + rounds) * n).reshape(-1, n)).to(dev)
    lg = torch.empty((n, V), dtype=torch.float32, device=dev)
    p = torch.empty((n, V), dtype=torch.float32, device=dev)
    acc = torch.zeros(1, dtype=torch.int32, device=dev)
    tok = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {}
    k = 0
    for mode in ("greedy", "sampled"):
        # rounds back to back (the commit lengths are known on the host, so
        # nothing waits between rounds); events around the timed rounds
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        kept = 0
        for r in range(warm + rounds):
            if r == warm:
                torch.cuda.synchronize()
                e0.record()
            tk = toks[k]
            evs.evs_verify_block(st, tk, n, lg)
            if mode == "greedy":
                evs.evs_accept(lg, None, tk[1:], None, n, V, evs.EVS_GREEDY, acc, tok)
            else:
                evs.evs_probs(lg, n, V, 1.0, 4, p)
                evs.evs_accept(p, q, tk[1:], U[k], n, V, evs.EVS_SAMPLE, acc, tok)
            evs.evs_commit(st, int(keeps[k]))
            if r >= warm:
                kept += int(keeps[k])
            k += 1
        e1.record()
        torch.cuda.synchronize()
        t_round = e0.elapsed_time(e1)
        out[mode] = {"ms_per_round": t_round / rounds, "tok_s": kept / (t_round / 1e3), "mean_keep": kept / rounds}
    book = st.book()
    ok = st.check() == 0
    st.close()
    sb = step_bytes(shape, P + n, n)
    ms = out["greedy"]["ms_per_round"]
    out.update({"context": P, "rounds_per_mode": rounds, "status_ok": ok, "pos_end": book["pos"],
                "step_hbm": {"bytes": sb, "achieved_gbs": sb / (ms / 1e3) / 1e9,
                             "frac": sb / (ms / 1e3) / 1e9 / peak},
                "note": "commit lengths drawn geometric (mean 3) override the accept result; attention caches "
                        "are device filler N(0,1), FIR/IIR state synthesised; verify (graph) + accept + commit "
                        "per round, rounds back to back"})
    return out


def _dev_view(torch, ptr, shape, dtype):
    """Zero-copy torch view of library-owned device memory (state setup)."""
    class _A:
        pass
    a = _A()
    ts = {torch.float32: "<f4", torch.bfloat16: "<i2"}[dtype]
    a.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": ts, "data": (int(ptr), False), "version": 3,
                                  "strides": None}
    t = torch.as_tensor(a, device="cuda")
    return t.view(torch.bfloat16) if dtype == torch.bfloat16 else t


def run_case(args):
    """Small, self-contained launches of one kernel for profiler captures.

    gemm N K n     bf16 tensor-core GEMM of a [N][K] weight (N(0, 0.02)) against
                   n tokens, --reps times; the default 22016 x 4096 weight
                   (180 MB) is larger than L2, so each launch streams it from HBM
    fir L d n      FIR mixer (L taps, d channels, n block rows), fresh inputs per rep
    iir M d n      IIR mixer (M poles)
    attn P n       split-KV attention over P cached positions (32 x 128, chunks of 64)
    stack L n      the first L layers of the 7B-shaped stack with the library's
                   packed weights: one warm-up verify of n tokens, then every
                   weight GEMM of a step once more, each launched alone
    batch L B n    the first L layers, B sequences of n rows verified in one
                   batched pass, each committing its block; --reps times
    markov V k     the Markov head: 12 sampled draws of top-k over a V-entry
                   trunk row plus a V x V Markov row, --reps times
    """
    import torch

    import hybrid_ssm_attention_gb300 as evs
    from hybrid_ssm_attention_gb300 import build as b
    b.build()
    kind, cargs = args.case[0], [int(x) for x in args.case[1:]]
    if kind not in ("gemm", "fir", "iir", "attn", "stack", "batch", "markov"):
        raise SystemExit(f"unknown case {kind}")

    class a:
        pass
    a.kind, a.args, a.reps = kind, cargs, args.reps
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(0)
    book = torch.zeros(8, dtype=torch.int32, device=dev)
    book[4] = -1
    if a.kind == "batch":
        import synth
        L, B, n = (a.args + [2, 8, 13][len(a.args):])[:3]
        full = synth.stack_7b()
        shape = synth.ModelShape(name=f"7b-first-{L}", vocab=full.vocab, d_model=full.d_model,
                                 layers=full.layers[:L], n_heads=full.n_heads, head_dim=full.head_dim,
                                 d_ffn=full.d_ffn, gamma=full.gamma, dtype="bf16", pole_mag=full.pole_mag)
        m = evs.Model(shape, synth.make_weights(shape, 3))
        sts = [evs.State(m, 256) for _ in range(B)]
        toks = torch.tensor([65 + (i % 4) for i in range(B * n)], dtype=torch.int32, device=dev)
        lg = torch.empty((B * n, shape.vocab), device=dev)
        for _ in range(a.reps):
            evs.evs_verify_batch(sts, toks, [n] * B, lg)
            for st in sts:
                evs.evs_commit(st, n)
    elif a.kind == "stack":
        import synth
        L, n = (a.args + [2, 13][len(a.args):])[:2]
        full = synth.stack_7b()
        shape = synth.ModelShape(name=f"7b-first-{L}", vocab=full.vocab, d_model=full.d_model,
                                 layers=full.layers[:L], n_heads=full.n_heads, head_dim=full.head_dim,
                                 d_ffn=full.d_ffn, gamma=full.gamma, dtype="bf16", pole_mag=full.pole_mag)
        m = evs.Model(shape, synth.make_weights(shape, 3))
        st = evs.State(m, 256)
        toks = torch.tensor([65 + (i % 4) for i in range(n)], dtype=torch.int32, device=dev)
        lg = torch.empty((n, shape.vocab), device=dev)
        evs.evs_verify_block(st, toks, n, lg)
        evs.evs_commit(st, n)
        evs.evs_profile_gemms(st, n)
    elif a.kind == "markov":
        V, k = (a.args + [512, 4][len(a.args):])[:2]
        gamma = 12
        trunk = torch.randn(gamma, V, device=dev, generator=g) * 2
        M = torch.randn(V, V, device=dev, generator=g) * 2
        u = torch.rand(gamma, device=dev, generator=g)
        prev = torch.tensor([3], dtype=torch.int32, device=dev)
        d = torch.zeros(gamma, dtype=torch.int32, device=dev)
        q = torch.empty(gamma, V, device=dev)
        for _ in range(a.reps):
            evs.evs_markov_draft(trunk, M, V, prev, u, gamma, 1.0, k, evs.EVS_SAMPLE, d, q)
    elif a.kind == "gemm":
        N, K, n = (a.args + [22016, 4096, 13][len(a.args):])[:3]
        W = (torch.randn(N, K, device=dev, generator=g) * 0.02).to(torch.bfloat16)
        X = torch.randn(n, K, device=dev, generator=g).to(torch.bfloat16)
        y = torch.empty(n, N, device=dev)
        s = torch.empty(evs.evs_op_gemm_scratch_bytes(N, K, evs.EVS_BF16), dtype=torch.uint8, device=dev)
        for _ in range(a.reps):
            evs.evs_op_gemm(W, X, N, K, n, evs.EVS_BF16, y, s)
    elif a.kind in ("fir", "iir"):
        P, d, n = (a.args + [128 if a.kind == "fir" else 16, 4096, 13][len(a.args):])[:3]
        abv = torch.randn(n, 3 * d, device=dev, generator=g).to(torch.bfloat16)
        gout = torch.empty(n, d, device=dev, dtype=torch.bfloat16)
        for r in range(a.reps):
            if a.kind == "fir":
                ring = torch.randn(P - 1 + n, d, device=dev, generator=g)
                taps = torch.randn(P, d, device=dev, generator=g)
                book[0] = 1000 + r  # the window wraps around the ring
                evs.evs_op_fir(P, d, n, n, evs.EVS_BF16, abv, taps, ring, book, gout)
            else:
                s0 = torch.randn(n, d, P, 2, device=dev, generator=g)
                s1 = torch.empty_like(s0)
                lam = torch.rand(d, P, 2, device=dev, generator=g) * 0.7
                res = torch.randn(d, P, 2, device=dev, generator=g) * 0.25
                evs.evs_op_iir(P, d, n, n, evs.EVS_BF16, abv, lam, res, s0, s1, book, gout)
    else:
        P, n = (a.args + [8192, 13][len(a.args):])[:2]
        H, Dh, chunk = 32, 128, 64
        ctx = P + n
        kc = torch.randn(H, ctx, Dh, device=dev, generator=g).to(torch.bfloat16)
        vc = torch.randn(H, ctx, Dh, device=dev, generator=g).to(torch.bfloat16)
        qkv = torch.randn(n, 3 * H * Dh, device=dev, generator=g).to(torch.bfloat16)
        gout = torch.empty(n, H * Dh, device=dev, dtype=torch.bfloat16)
        s = torch.empty(evs.evs_op_attention_scratch_bytes(H, Dh, ctx, chunk, n), dtype=torch.uint8, device=dev)
        book[0] = P
        for _ in range(a.reps):
            evs.evs_op_attention(H, Dh, n, n, ctx, chunk, 10000.0, evs.EVS_BF16, qkv, kc, vc, book, gout, s)
    torch.cuda.synchronize()
    print("profile case done:", a.kind, a.args)


def run_evs(args, rank, world, local):
    import torch

    import hybrid_ssm_attention_gb300 as evs
    import synth
    from hybrid_ssm_attention_gb300 import build as _build
    _build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    shape = synth.stack_7b()
    n = shape.n_block
    P0 = args.prompt
    rounds = args.warmup + args.steps
    ctx = P0 + n * rounds + 2 * n
    W = synth.make_weights(shape, args.seed)
    model = evs.Model(shape, W)
    st = evs.State(model, ctx)
    prompt = [int(x) for x in synth.prompt(shape, args.seed, P0)]

    # prefill prompt[:-1] in blocks of n, committing each block
    lg = torch.empty((n, shape.vocab), dtype=torch.float32, device=dev)
    for s0 in range(0, P0 - 1, n):
        blk = torch.tensor(prompt[s0:min(s0 + n, P0 - 1)], dtype=torch.int32, device=dev)
        evs.evs_verify_block(st, blk, blk.numel(), lg[:blk.numel()])
        evs.evs_commit(st, blk.numel())
    snap = evs.State(model, ctx)
    st.clone_into(snap)
    torch.cuda.synchronize()

    # native greedy decoding (n = 1 rounds): the identity drafter's tokens
    n_nat = n * rounds + 1
    y = torch.empty(n_nat + 1, dtype=torch.int32, device=dev)
    y[0] = prompt[-1]
    tok1 = torch.empty(1, dtype=torch.int32, device=dev)
    lg1 = torch.empty((1, shape.vocab), dtype=torch.float32, device=dev)
    acc = torch.zeros(1, dtype=torch.int32, device=dev)
    otok = torch.zeros(1, dtype=torch.int32, device=dev)
    tok1.copy_(y[:1])
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(n_nat):
        if i == 16:
            e0.record()
        evs.evs_round(st, tok1, 1, lg1, None, None, None, 1.0, 0, evs.EVS_GREEDY, acc, otok)
        tok1.copy_(otok)
        y[i + 1:i + 2].copy_(otok)
    e1.record()
    torch.cuda.synchronize()
    native_step_ms = e0.elapsed_time(e1) / (n_nat - 16)

    # speculative rounds from the post-prompt state: block r = y[n r : n r + n]
    snap.clone_into(st)
    blocks = y[: n * rounds].view(rounds, n).contiguous()
    tokens = torch.empty(n, dtype=torch.int32, device=dev)
    acc_log = torch.zeros(rounds, dtype=torch.int32, device=dev)
    launches0 = None
    clocks = ClockSampler(local).start()
    for r in range(rounds):
        if r == args.warmup:
            torch.cuda.synchronize()
            barrier(world)
            torch.cuda.synchronize()
            launches0 = evs.evs_kernel_launches()
            torch.cuda.nvtx.range_push("timed")
            e0.record()
        tokens.copy_(blocks[r])
        evs.evs_round(st, tokens, n, lg, None, None, None, 1.0, 0, evs.EVS_GREEDY, acc, otok)
        acc_log[r:r + 1].copy_(acc)
    e1.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    launches = evs.evs_kernel_launches() - launches0
    barrier(world)
    clk = clocks.stop()
    t_ms = e0.elapsed_time(e1)
    t_max_ms = reduce_max(t_ms, world)
    accepted = acc_log.cpu().numpy()
    book = st.book()
    ok = bool((accepted == n - 1).all()) and book["pos"] == P0 - 1 + n * rounds
    emitted = float(np.sum(accepted[args.warmup:] + 1))
    total_tokens = reduce_sum(emitted, world)
    value = total_tokens / (t_max_ms / 1e3)
    ms_per_step = t_ms / args.steps

    # dominant kernel: the weight-streaming GEMM.  achieved = its algorithmic
    # bytes / its launch time as it runs in the step (the step's 129 GEMMs
    # back to back in one graph, PDL between them, next-weight prefetch),
    # CUDA events around 10 chains; each launch timed alone is reported beside
    ms, by = evs.evs_profile_gemms(st, n)
    peak, peak_src = load_peaks()
    a_bytes, a_ms = float(sum(by)), float(sum(ms))
    c_ms, c_bytes, c_launches = evs.evs_profile_gemm_chain(st, n, 10)
    achieved = c_bytes / (c_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": gemm_traffic(), "kernel": "gemm_tc_kernel", "launches": c_launches,
                "avg_launch_us": 1e3 * c_ms / c_launches, "bytes_per_launch": c_bytes / c_launches,
                "peak_source": peak_src,
                "timing": "the step's GEMM launches back to back (one graph, PDL, next-weight prefetch), CUDA events",
                "alone": {"avg_launch_us": 1e3 * a_ms / len(ms), "achieved": a_bytes / (a_ms / 1e3) / 1e9,
                          "frac": a_bytes / (a_ms / 1e3) / 1e9 / peak}}
    sb = step_bytes(shape, P0 - 1 + n * (args.warmup + args.steps // 2), n)

    # snapshot-and-replay baseline: snapshot the recurrent state, verify,
    # accept, restore, verify the kept tokens again, commit (the second
    # forward pass that per-position slicing removes)
    replay = None
    R, Wr = min(args.steps, 16, rounds - 2), 2  # replayed blocks come from the same `rounds` blocks
    if not args.no_replay and R >= 1:
        snap.clone_into(st)
        rsnap = evs.State(model, ctx)
        emitted_r = 0
        for r in range(Wr + R):
            if r == Wr:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            tokens.copy_(blocks[r])
            st.snapshot_into(rsnap)
            evs.evs_verify_block(st, tokens, n, lg)
            evs.evs_accept(lg, None, tokens[1:], None, n, shape.vocab, evs.EVS_GREEDY, acc, otok)
            keep = int(acc.item()) + 1
            rsnap.snapshot_into(st)
            evs.evs_verify_block(st, tokens[:keep], keep, lg[:keep])
            evs.evs_commit(st, keep)
            if r >= Wr:
                emitted_r += keep
        torch.cuda.synchronize()
        dt_r = time.perf_counter() - t0
        rsnap.close()
        replay = {"value": emitted_r / dt_r, "unit": UNIT, "ms_per_round": 1e3 * dt_r / R, "rounds": R,
                  "slicing_speedup": (1e3 * dt_r / R) / ms_per_step,
                  "note": "host-driven: snapshot (FIR/IIR state + book), verify, accept, read keep, restore, "
                          "verify keep tokens, commit; identity drafter, so keep = 13"}

    # end to end through the C ABI with the block and the result in host
    # memory: evs_round_host copies the block in and the result out (both
    # inside the round's graph) and returns once the result is on the host
    e2e = None
    if not args.no_e2e:
        snap.clone_into(st)
        host_blocks = blocks.cpu().numpy()
        emitted_e2e = 0
        for r in range(rounds):
            if r == args.warmup:
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            a_r, _ = evs.evs_round_host(st, host_blocks[r], n, lg, None, None, None, 1.0, 0, evs.EVS_GREEDY)
            if r >= args.warmup:
                emitted_e2e += a_r + 1
        dt = time.perf_counter() - t0
        e2e = {"value": reduce_sum(emitted_e2e, world) / reduce_max(dt, world), "unit": UNIT,
               "h2d_bytes_per_step": 4 * n, "d2h_bytes_per_step": 8}

    batched = cross = None
    if not args.no_batch:
        batched = batched_sweep(evs, torch, model, shape, snap, ctx, dev, y)
        cross = crossover(batched)

    longgen = None
    if args.long_gen > 0:
        longgen = long_generation(evs, torch, model, shape, prompt, args.long_gen, args.seed + 100, dev)

    drafter = None
    if not args.no_drafter:
        drafter = drafter_rounds(evs, torch, dev, args.seed + 2, P0)

    sampled = None
    if not args.no_sampled:
        sampled = sampled_rounds(evs, torch, model, shape, snap, ctx, dev, prompt[-1], args.seed + 1)

    longctx = None
    if not args.no_long_context:
        longctx = long_context_rounds(evs, torch, model, shape, args.long_context, args.seed + 1, dev, peak)

    cpu = None
    if not args.no_cpu and rank == 0 and world == 1:
        st.close()
        snap.close()
        model.close()
        torch.cuda.empty_cache()
        cpu = cpu_baseline(args, shape, W)
    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config(args, world, n, rounds),
            "verify_round_us": 1e3 * ms_per_step,
            "native_step_us": 1e3 * native_step_ms,
            "identity_overhead": ms_per_step / (n * native_step_ms),
            "all_accepted": ok,
            "step_hbm": {"bytes": sb, "achieved_gbs": sb / (ms_per_step / 1e3) / 1e9,
                         "frac": sb / (ms_per_step / 1e3) / 1e9 / peak},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "snapshot_replay": replay,
            "long_generation": longgen, "batched_verify": batched, "batched_crossover": cross, "sampled": sampled,
            "long_context": longctx,
            "drafter": drafter,
            "gpu_launches": int(launches),
            "clocks": clk}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.cpu_one_thread_child:
        run_cpu_one_thread_child(args)
        return
    if args.case:
        run_case(args)
        return
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_evs(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
