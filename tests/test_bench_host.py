"""Host logic of bench.py: clock-sample parsing, whole-job aggregation, the max-over-ranks
reduction with two gloo ranks on CPU, and the reference (oracle) arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CSV = """index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], clocks_event_reasons.active, clocks_event_reasons.hw_slowdown, clocks_event_reasons.hw_thermal_slowdown, clocks_event_reasons.sw_thermal_slowdown, clocks_event_reasons.sw_power_cap
0, 1965 MHz, 2070 MHz, 180.12 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active
0, 1477 MHz, 2070 MHz, 1350.00 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active
0, 1500 MHz, 2070 MHz, 1390.00 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active
"""


def test_parse_clock_csv():
    c = bench.parse_clock_csv(CSV)
    assert c["samples"] == 3 and c["samples_under_load"] == 2
    assert c["sm_mhz"] == pytest.approx((1477 + 1500) / 2)
    assert c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_csv("")["samples"] == 0


def test_whole_job_rate_is_total_units_over_slowest_rank():
    assert bench.whole_job_rate(10.0, 4, 2.0) == 20.0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.reduce_max(1.5 + rank)       # each rank's step time
    bench.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=120,
                       cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_summary_pairs_every_workload_with_its_fraction_of_peak():
    import bench
    bd = {
        "fwd": {"tflops": 1400.0, "frac_of_peak": 0.72},
        "fwd_bwd": {"tflops": 1100.0}, "fwd_causal": {"tflops": 1240.0}, "fwd_bwd_causal": {"tflops": 980.0},
        "gpt2m_8x16x1024x64_causal": {"fwd_tflops": 350.0, "fwd_frac": 0.18, "fwd_bwd_tflops": 330.0,
                                      "fwd_bwd_frac": 0.17},
        "block_sparse": {"fwd_bwd_tflops": 520.0},
        "fwd_fp8": {"tflops": 1950.0, "frac_of_fp8_peak": 0.6},
        "gemm_peaks": {"fp8_peak_used": 3250.0},
        "decode": {"gbps": 6950.0, "frac_of_hbm": 1.02},
    }
    s = bench.summarize(bd, 2000.0)
    assert s["fwd"] == [1400.0, 0.72]
    assert s["fwd_bwd"] == [1100.0, 0.55] and s["fwd_bwd_causal"] == [980.0, 0.49]
    assert s["gpt2m_fwd"] == [350.0, 0.18] and s["gpt2m_fwd_bwd"] == [330.0, 0.17]
    assert s["block_sparse_fwd_bwd"] == [520.0, 0.26]
    assert s["fwd_fp8"] == [1950.0, 0.6] and s["fp8_peak"] == 3250.0
    assert s["decode"] == [6950.0, 1.02]
    assert "long_fwd" not in s and "varlen_fwd_bwd" not in s
    assert len(json.dumps(s)) < 1000
