"""Host-side logic of bench.py's multi-replica mode on CPU (gloo, world size 2):
the step time is the max over ranks, the token count the sum over ranks, and
rank 0 alone prints."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.reduce_max(10.0 + rank, world)
    s = bench.reduce_sum(13.0 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, t, s))
    dist.destroy_process_group()


def test_replica_aggregation_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [11.0, 11.0]
    assert [r[2] for r in res] == [39.0, 39.0]


def test_step_bytes_counts_weights_once():
    import bench
    import synth
    sh = synth.stack_7b()
    b = bench.step_bytes(sh, 1024, 13)
    w = 32 * (4 * 4096 * 4096 + 3 * 4096 * 11008) * 2
    assert w == 12952010752
    assert 13.0e9 < b < 13.3e9


def test_crossover_break_even_and_full_acceptance_speedup():
    # a speculative round of n rows emits accepted + 1 tokens per sequence
    # against one per native pass: break-even = spec_ms / native_ms tokens per
    # round, speedup at full acceptance = n * native_ms / spec_ms
    import bench
    sweep = [{"B": 1, "n": 1, "ms_per_round": 2.5}, {"B": 1, "n": 13, "ms_per_round": 2.75},
             {"B": 16, "n": 1, "ms_per_round": 3.2}, {"B": 16, "n": 8, "ms_per_round": 6.4},
             {"B": 4, "n": 13, "ms_per_round": 3.5}]  # B = 4 has no native pass: skipped
    out = bench.crossover(sweep)
    assert [r["B"] for r in out] == [1, 16]
    b1, b16 = out
    assert b1["spec_n"] == 13 and b1["break_even_tokens_per_round"] == 2.75 / 2.5
    assert abs(b1["speedup_all_accepted"] - 13 * 2.5 / 2.75) < 1e-12
    assert b16["spec_n"] == 8 and b16["break_even_tokens_per_round"] == 2.0
    assert b16["speedup_all_accepted"] == 4.0


def test_clock_summary_of_nvidia_smi_lines():
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active, then
    # hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    import bench
    ok = "0, 2070, 2070, 912.40, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
    cap = "0, 1980, 2070, 1398.10, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
    hot = "0, 1500, 2070, 1200.00, 0x0000000000000040, Not Active, Active, Not Active, Not Active"
    na = "0, 2070, [N/A], 900.00, 0x0, Not Active, Not Active, Not Active, Not Active"
    s = bench.ClockSampler.summarize([ok, ok, cap, "garbage", na, ""])
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    s = bench.ClockSampler.summarize([ok, hot, cap])
    assert s["sm_mhz"] == 1980.0 and s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert bench.ClockSampler.summarize([])["sm_mhz"] is None


def test_peak_denominator_measured_else_fallback(tmp_path, monkeypatch):
    import json
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")  # no file
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6743.6, "bf16_tflops": 1904.1}))
    assert bench.load_peaks() == (6743.6, "measured")
    (tmp_path / "MEASURED_PEAKS.json").write_text("{not json")
    assert bench.load_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
