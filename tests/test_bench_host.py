"""The benchmark's CPU legs without a GPU: the one-thread oracle baseline and
the all-cores one (spawned processes) run on the small workload's inputs built
on the CPU, and report what the JSON line needs."""
import os

import torch

from paged_kv_cache_211_gb300 import workloads as wl


def test_cpu_baselines_one_thread_and_all_cores():
    import bench
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w, device=torch.device("cpu"), num_layers=1)
    one, seqs = bench.cpu_baseline(inp, w, budget_s=5.0)
    assert one["cores"] == 1 and one["kind"] == "oracle" and one["value"] > 0
    assert sorted(seqs) == list(range(w.num_seqs))          # the whole small batch
    assert len(one["runs"]) == 3 and one["value"] == sorted(one["runs"])[1]   # the median
    every = bench.cpu_baseline_all_cores(inp, w, seqs, timeout_s=120.0)
    assert every["cores"] == min(os.cpu_count() or 1, len(seqs))
    assert every["kind"] == "oracle" and every["unit"] == "GB/s" and every["value"] > 0
    assert f"the same {len(seqs)} sequences" in every["sample"]
    assert len(every["runs"]) == 3 and every["value"] == sorted(every["runs"])[1]


def test_clock_sampler_without_a_gpu_reports_nothing():
    import bench
    assert bench.ClockSampler(0).stop() is None


def test_all_cores_leg_gives_up_on_a_dead_or_silent_process():
    import queue

    import bench
    import pytest

    class Proc:
        def __init__(self, code):
            self.exitcode = code

    q = queue.Queue()
    q.put(0.5)
    assert bench._collect(q, [Proc(None)], 1, 5.0) == [0.5]
    with pytest.raises(RuntimeError, match="exited with code 1"):
        bench._collect(queue.Queue(), [Proc(None), Proc(1)], 2, 60.0)
    with pytest.raises(TimeoutError):
        bench._collect(queue.Queue(), [Proc(None)], 1, 1.5)
