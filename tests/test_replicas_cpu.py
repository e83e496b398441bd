"""Host logic of the benchmark's replica runs and its clock record, on CPU.

`bench.py --gpus N` under torchrun runs N independent replicas of the decode step (the path has
no exchange step, so no data-path collective): the ranks start each timed window together, the
job's window is the slowest rank's, and the whole-job figure counts every rank's tokens. These
tests run the same helpers as two `gloo` ranks on CPU; the reference arm's other ranks exit
without work; the clock record is parsed from nvidia-smi's CSV rows; the per-step spread is
computed from events recorded between consecutive steps (driven here by stand-ins for the CUDA
events and the plan).
"""
import json
import os
import socket
import subprocess
import sys
import time

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir, delays_s):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        res = {"max": bench.max_over_ranks(torch, 1.5 + rank, world, "cpu")}
        calls = []

        def step(i):
            calls.append(i)
            time.sleep(delays_s[rank])

        res["job_us"] = bench.host_timed_job(torch, step, 3, world, "cpu")
        res["calls"] = calls
        synced = []
        res["job_us_sync"] = bench.host_timed_job(torch, lambda i: None, 2, world, "cpu",
                                                  sync=lambda: synced.append(rank))
        res["synced"] = synced
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_window(tmp_path):
    world, delays = 2, [0.0, 0.02]  # rank 1 takes 20 ms per step, rank 0 none
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), delays), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(world)]
    assert res[0]["max"] == res[1]["max"] == 2.5
    # every rank reports the same whole-job figure, set by rank 1's 3 x 20 ms over 3 x 2 tokens
    assert res[0]["job_us"] == res[1]["job_us"]
    assert res[0]["job_us"] >= 3 * 20_000 / (3 * 2)
    assert res[0]["job_us"] < 3 * 20_000 / (3 * 2) * 50  # loose: only a gross miscount fails
    assert res[0]["calls"] == res[1]["calls"] == [0, 1, 2]
    assert res[0]["job_us_sync"] == res[1]["job_us_sync"]
    assert res[0]["synced"] == [0] and res[1]["synced"] == [1]


def test_one_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(torch, 7.25, 1, "cpu") == 7.25
    calls = []
    us = bench.host_timed_job(torch, calls.append, 4, 1, "cpu")
    assert calls == [0, 1, 2, 3] and us >= 0.0


@pytest.mark.parametrize("slowest_us,tokens,world,want", [(1000.0, 10, 1, 100.0), (1000.0, 10, 4, 25.0),
                                                          (331.3 * 20, 20, 8, 331.3 / 8)])
def test_whole_job_counts_every_rank_tokens(slowest_us, tokens, world, want):
    assert bench.job_us_per_token(slowest_us, tokens, world) == pytest.approx(want, rel=1e-12)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_clock_record_from_nvidia_smi_rows():
    rows = ("0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "0, 1965, 2070, 1399.8, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
            "0, 2070, 2070, 1100.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "0, [N/A], 2070, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]\n"
            "0, 2070, 20")  # a line cut off when the sampler was stopped
    got = bench.parse_clock_samples(rows)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    hot = bench.parse_clock_samples("0, 1500, 2070, 1400, 0x48, Active, Not Active, Active, Not Active\n")
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"] and hot["sm_mhz"] == 1500.0
    assert bench.parse_clock_samples("") == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_committed_traffic_profile_matches_the_kernel_sources():
    # the bench reports DRAM traffic only while the capture was taken on these exact sources
    assert bench.read_traffic() is not None, "profile's source hash differs: re-capture the traffic"
    assert abs(bench.read_traffic() / bench.step_bytes() - 1.0) < 0.01


class _FakeEvent:
    clock = [0.0]

    def __init__(self, enable_timing=False):
        assert enable_timing
        self.t = None

    def record(self, stream):
        assert stream == "launch-stream"
        self.t = _FakeEvent.clock[0]

    def elapsed_time(self, other):  # milliseconds, as CUDA events report
        return other.t - self.t


class _FakeCuda:
    Event = _FakeEvent

    @staticmethod
    def synchronize():
        pass


class _FakeTorch:
    cuda = _FakeCuda


class _FakePlan:
    def __init__(self, step_ms):
        self.step_ms, self.calls = step_ms, 0

    def nt_decode_step(self, stream):
        assert stream == "launch-stream"
        _FakeEvent.clock[0] += self.step_ms[self.calls]
        self.calls += 1


def test_step_distribution_times_each_step_between_its_events():
    step_ms = [0.330 + 0.001 * (i % 10) for i in range(60)]  # 330 ... 339 us, six times each
    _FakeEvent.clock[0] = 5.0
    plan = _FakePlan(step_ms)
    got = bench.step_distribution(_FakeTorch, plan, 60, "launch-stream")
    assert plan.calls == 60
    assert got["n"] == 60 and got["min"] == 330.0 and got["max"] == 339.0
    assert got["median"] == pytest.approx(334.5, abs=0.01)
    assert 330.0 <= got["p10"] <= 331.0 and 338.0 <= got["p90"] <= 339.0
