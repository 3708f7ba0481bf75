"""Multi-process host logic of bench.py on CPU (gloo, world size 2): the replicas report the
slowest rank's time, the job's throughput sums the ranks' work, and the reference arm prints only
on rank 0. No GPU is involved."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(ws),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    r, local, w = bench.dist_setup(ws, "gloo")
    assert (r, local, w) == (rank, rank, ws)
    ms = bench.allreduce_max(10.0 + 5.0 * rank, w)   # rank 1 is the slow one
    bench.barrier(w)
    out[rank] = (ms, bench.job_tflops(10**12, 4, w, ms))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replicas_report_slowest_rank_and_summed_work():
    ws = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(ws, _free_port(), out), nprocs=ws, join=True)
    for rank in range(ws):
        ms, tflops = out[rank]
        assert ms == 15.0
        # 2 ranks x 4 steps x 1 TFLOP in 15 ms
        assert tflops == pytest.approx(2 * 4 * 1.0 / 0.015)


def test_job_tflops_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_tflops(2 * 10**12, 10, 1, 1000.0) == pytest.approx(20.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "single", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    env = dict(os.environ, RANK="0", LOCAL_RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "single", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["value"] > 0 and line["value"] == line["e2e"]["value"]


def test_peak_follows_the_sampled_clocks():
    """Burst peak when the timed region ran at the maximum SM clock with no cap; sustained
    otherwise (power cap, thermal reasons, or a clock well below its maximum)."""
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6000.0}
    free = {"sm_mhz": 2032.0, "sm_max_mhz": 2032.0, "reasons": []}
    assert bench.choose_peak(free, peaks, "measured")[:2] == (3600.0, "burst")
    capped = dict(free, reasons=["sw_power_cap"])
    assert bench.choose_peak(capped, peaks, "measured")[:2] == (2800.0, "sustained")
    slow = dict(free, sm_mhz=1500.0)
    assert bench.choose_peak(slow, peaks, "measured")[:2] == (2800.0, "sustained")
    unknown = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    assert bench.choose_peak(unknown, peaks, "measured")[1] == "sustained"
