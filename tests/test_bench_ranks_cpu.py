"""The multi-process path of bench.py on CPU (gloo, world size 2): the
requests of a decode step are independent, so ranks run replicas and meet
only to time the job; the slowest rank's time is the job's, and only rank 0
prints.  The GPU arms use the same helpers over NCCL."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks_worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        mine = 1.5 + rank              # this rank's duration
        got = bench.max_over_ranks(mine, world, torch.device("cpu"))
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"mine": mine, "max": got}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    world = 2
    mp.spawn(_ranks_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    assert [r["max"] for r in res] == [2.5, 2.5]          # every rank sees the slowest
    assert sorted(r["mine"] for r in res) == [1.5, 2.5]


def test_max_over_ranks_one_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    bench.rank_barrier(1)   # no process group needed


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference launched as the driver launches N > 1: rank 0
    alone times the oracle and prints one JSON line; rank 1 exits 0 quietly."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "16", "--warmup", "3",
           "--cpu-workers", "1", "--cpu-pairs", "48"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["cores"] == 1 and d["e2e"]["h2d_bytes_per_step"] == 0
    # the same config object our arm prints, and the same sample as its cpu_baseline
    sys.path.insert(0, ROOT)
    import bench
    assert d["config"] == bench.describe("decode_T4096", 2)
    assert d["cpu_baseline"]["sample"].startswith("48 seeded random (request, head) pairs")


def test_profile_summary_sections(tmp_path):
    """Each kernel's figures are read from its own section of an ncu summary:
    a later kernel's DRAM bytes never stand in for an earlier one's."""
    sys.path.insert(0, ROOT)
    import bench
    p = tmp_path / "s.md"
    p.write_text("# title\n\n- kernel_source_sha256_16: `abc`\n\n## first\n\n"
                 "- kernel: `prefill_tc_kernel`\n- dram_bytes_per_full_launch: 201862400\n\n"
                 "## second\n\n- kernel: `append_tc_kernel`\n"
                 "- dram_bytes_per_full_launch: 92373504  (the projection)\n")
    head, sec = bench.summary_sections(str(p))
    assert head == {"kernel_source_sha256_16": "abc"}
    assert sec["prefill_tc_kernel"]["dram_bytes_per_full_launch"] == "201862400"
    assert sec["append_tc_kernel"]["dram_bytes_per_full_launch"] == "92373504"


def test_nvml_clock_sampler_reads_and_decodes():
    """The in-process clock sampler: without NVML (this host) the bench falls
    back to nvidia-smi; with a fake NVML it polls the SM clock and decodes the
    clock-event reason bits (read-only queries)."""
    import ctypes
    import bench
    s = bench.clock_sampler(0)
    if not torch.cuda.is_available():
        assert isinstance(s, bench.ClockSampler)

    class FakeNvml:
        def __init__(self):
            self.n = 0

        def nvmlDeviceGetClockInfo(self, h, kind, out):
            assert kind == 1  # SM clock
            self.n += 1
            ctypes.cast(out, ctypes.POINTER(ctypes.c_uint))[0] = 1900 if self.n % 2 else 2000
            return 0

    fake = FakeNvml()
    smp = bench.NvmlClockSampler.__new__(bench.NvmlClockSampler)
    import threading
    smp.ct, smp.threading = ctypes, threading
    smp.samples, smp.max_mhz, smp.t0, smp.t1 = [], 2070.0, None, None
    smp.lib, smp.h = fake, None

    def reasons(h, out):
        ctypes.cast(out, ctypes.POINTER(ctypes.c_ulonglong))[0] = 0x4 | 0x40  # power cap, hw thermal
        return 0
    smp.reasons_fn = reasons
    smp.start()
    import time
    smp.begin()
    time.sleep(0.02)
    smp.end()
    time.sleep(0.01)  # samples after the region do not count
    r = smp.stop()
    assert r["samples"] >= 5 and r["samples"] < len(smp.samples)
    assert 1900.0 <= r["sm_mhz"] <= 2000.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert r["sampled_after_region"] is False
