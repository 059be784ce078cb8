#!/usr/bin/env python
"""Decode-step PagedAttention benchmark on GB300.

One step = one decode step of one layer over the workload's batch: the new
token of every sequence is written into the paged cache, then decode
attention runs (split-context partition pass + log-sum-exp merge).  All of it
runs in libpagedkv's CUDA kernels, called through the C ABI.

Prints ONE JSON line (rank 0).  Default workload: the Llama/Mistral-7B-shaped
long-context decode (32 sequences, lognormal lengths with median 8192,
32 query / 8 KV heads, head_dim 128, bf16).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn achieved HBM GB/s (% of GB300 peak) and tokens/s per layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
# the long-context workload the >= 70 %-of-peak target is stated on; the
# committed ncu summary covers its partition kernel
DEFAULT_WORKLOAD = "llama7b_long"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_partition_llama7b_long.md")
KERNEL_SOURCES = ["paged_kv_cache_211_gb300/csrc/pkv_decode.cu",
                  "paged_kv_cache_211_gb300/csrc/pkv_internal.cuh",
                  "paged_kv_cache_211_gb300/csrc/pkv_tma.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer loop")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other decode workloads and prefill")
    ap.add_argument("--prefill", action="store_true",
                    help="time chunked-prefill attention instead of the decode step")
    ap.add_argument("--pool-blocks", type=int, default=0,
                    help="shrink the physical pool (for small profiler captures)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers

def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def partition_kernel_name() -> str:
    """The partition kernel the library runs (the TMA pipeline unless the
    register-pipelined kernel is selected for comparison)."""
    if os.environ.get("PKV_DECODE_KERNEL") == "ldg":
        return "decode_partition_kernel"
    return "decode_partition_tma_kernel"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic():
    """DRAM bytes per launch of the partition kernel from the committed ncu summary,
    if the summary was taken on the current kernel source (else None)."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)\s*\(kernel_source_sha256:\s*([0-9a-f]+)",
                  text)
    if not m or m.group(2) != kernel_source_hash():
        return None
    return int(m.group(1))


def _smi_target(device_index: int) -> str:
    try:
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        return uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        return str(device_index)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons: one sample just before the timed
    region, samples every 100 ms while it runs, and one just after it, so that
    even a region of a few milliseconds carries a record."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.target = _smi_target(device_index)
        self.before = self._once()
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.target, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def _once(self) -> list:
        try:
            r = subprocess.run(["nvidia-smi", "-i", self.target, f"--query-gpu={self.FIELDS}",
                                "--format=csv,noheader,nounits"], capture_output=True,
                               text=True, timeout=10)
            return self._rows(r.stdout.splitlines())
        except Exception:
            return []

    @staticmethod
    def _rows(lines) -> list:
        rows = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        return rows

    def stop(self):
        during = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()
            during = self._rows(open(self.path))
            os.unlink(self.path)
        after = self._once()
        rows = self.before + during + after
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "samples_during": len(during),
                "sm_mhz_before_after": [num(r[1]) for r in self.before + after]}


def compact_host(inp, seq_ids, kv_heads=None, q_heads=None):
    """Host copies (bit patterns) of what the oracle needs for `seq_ids`
    (optionally only the first kv_heads KV heads and first q_heads query heads)."""
    from paged_kv_cache_211_gb300.workloads import BLOCK_SIZE as BS
    w = inp["workload"]
    tables, lens = inp["block_tables_host"], inp["context_lens_host"]
    need = (lens[seq_ids].astype(np.int64) + BS - 1) // BS
    used = sorted({int(b) for s, n in zip(seq_ids, need) for b in tables[s, :n]})
    remap = {b: i for i, b in enumerate(used)}
    dev = inp["k_cache"].device
    idx = torch.tensor(used, dtype=torch.long, device=dev)
    heads = slice(None) if kv_heads is None else slice(0, kv_heads)

    def bits(t):
        return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    kc = bits(inp["k_cache"][0].index_select(0, idx)[:, :, heads])
    vc = bits(inp["v_cache"][0].index_select(0, idx)[:, :, heads])
    tb = np.zeros((len(seq_ids), tables.shape[1]), np.int32)
    for r, (s, n) in enumerate(zip(seq_ids, need)):
        tb[r, :n] = [remap[int(b)] for b in tables[s, :n]]
    sel = torch.tensor(list(seq_ids), dtype=torch.long, device=dev)
    hq = slice(None) if kv_heads is None else slice(0, q_heads or kv_heads * w.group)
    q = bits(inp["q"].index_select(0, sel)[:, hq])
    kn = bits(inp["k_new"][0].index_select(0, sel)[:, heads])
    vn = bits(inp["v_new"][0].index_select(0, sel)[:, heads])
    return dict(q=q, kc=kc, vc=vc, kn=kn, vn=vn, tb=tb, ln=lens[seq_ids].astype(np.int32))


def oracle_step(h, w):
    """The oracle's decode step (write + attention) on compact host inputs."""
    import oracle
    dt = oracle.BF16 if w.dtype == "bf16" else oracle.F16
    slots = oracle.slot_mapping(h["tb"], h["ln"], 16, h["kc"].shape[0])
    kc, vc = oracle.reshape_and_cache(h["kn"], h["vn"], h["kc"], h["vc"], slots)
    return oracle.decode_attention(dt, h["q"], kc, vc, h["tb"], h["ln"], w.scale)


def sample_bytes(w, lens, kv_heads, q_heads=None):
    """Algorithmic bytes of a (sequences x first kv_heads KV heads) sample."""
    n = int(np.asarray(lens, np.int64).sum())
    B = len(lens)
    blocks = int(((np.asarray(lens, np.int64) + 15) // 16).sum())
    hq = q_heads or kv_heads * w.group
    return (n * kv_heads * w.head_dim * 4 + 2 * B * hq * w.head_dim * 2 + blocks * 4 + B * 4
            + 2 * B * kv_heads * w.head_dim * 4)


def cpu_baseline(inp, w, budget_s=10.0, runs=3):
    """The oracle as it stands, one thread, on whole sequences until ~budget_s
    (or the whole batch, whichever comes first); the same sequences are then
    run again, `runs` times in all, and the median is reported.  Returns the
    result and the sequences it covered."""
    lens = inp["context_lens_host"]
    order = [int(s) for s in np.random.default_rng(w.seed + 99).permutation(len(lens))]
    hosts, done = [], []
    values, secs = [], []
    for r in range(runs):
        t_total, nbytes = 0.0, 0
        todo = order if r == 0 else done
        for k, s in enumerate(todo):
            if r == 0:
                hosts.append(compact_host(inp, [s]))
            t0 = time.perf_counter()
            oracle_step(hosts[k], w)
            t_total += time.perf_counter() - t0
            nbytes += sample_bytes(w, lens[[s]], w.num_kv_heads)
            if r == 0:
                done.append(s)
                if t_total >= budget_s:
                    break
        values.append(nbytes / t_total / 1e9)
        secs.append(t_total)
    toks = int(lens[done].sum())
    med = statistics.median(values)
    return {"value": round(med, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "runs": [round(v, 4) for v in values],
            "sample": f"{len(done)} of {len(lens)} sequences ({toks} context tokens, all "
                      f"{w.num_q_heads} query heads), write + attention, fp64, 1 thread; "
                      f"median of {runs} runs of {statistics.median(secs):.1f} s"}, done


def _oracle_cores_worker(hs, w, ready, gos, results):
    """One process of the all-cores baseline: loads the oracle, reports ready,
    then for each round waits for the common start and runs the oracle over
    its share."""
    import oracle
    oracle.default()
    ready.put(os.getpid())
    for r, go in enumerate(gos):
        if not go.wait(timeout=600):
            return
        t0 = time.perf_counter()
        for h in hs:
            oracle_step(h, w)
        results.put((r, time.perf_counter() - t0))


def _collect(q, procs, k, timeout_s):
    """k items from q, giving up at once if a process died with an error, or
    after timeout_s."""
    import queue
    got, deadline = [], time.perf_counter() + timeout_s
    while len(got) < k:
        try:
            got.append(q.get(timeout=1.0))
        except queue.Empty:
            dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
            if dead:
                raise RuntimeError(f"an oracle process exited with code {dead[0]}")
            if time.perf_counter() > deadline:
                raise TimeoutError(f"{len(got)} of {k} oracle processes answered")
    return got


def cpu_baseline_all_cores(inp, w, seq_ids, timeout_s=180.0, runs=3):
    """The same oracle, unchanged, on every host core: one spawned process per
    core, each given whole sequences (longest first, to the least-loaded
    process).  In each of `runs` rounds all start together and the time runs
    from that start to the last process's end, so load imbalance counts
    against it; the median round is reported."""
    import multiprocessing as mp
    lens = inp["context_lens_host"]
    seq_ids = [int(s) for s in seq_ids]
    n = max(1, min(os.cpu_count() or 1, len(seq_ids)))
    shares, load = [[] for _ in range(n)], [0] * n
    for s in sorted(seq_ids, key=lambda s: -int(lens[s])):
        i = load.index(min(load))
        shares[i].append(compact_host(inp, [s]))
        load[i] += int(lens[s])
    ctx = mp.get_context("spawn")
    ready, results = ctx.Queue(), ctx.Queue()
    gos = [ctx.Event() for _ in range(runs)]
    procs = [ctx.Process(target=_oracle_cores_worker,
                         args=(shares[i], w, ready, gos, results), daemon=True)
             for i in range(n)]
    for p in procs:
        p.start()
    walls, busiest = [], []
    try:
        _collect(ready, procs, n, timeout_s)
        for go in gos:
            t0 = time.perf_counter()
            go.set()
            busy = _collect(results, procs, n, timeout_s)
            walls.append(time.perf_counter() - t0)
            busiest.append(max(b for _, b in busy))
    finally:
        for go in gos:
            go.set()
        for p in procs:
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()
    nbytes = sample_bytes(w, lens[seq_ids], w.num_kv_heads)
    values = [nbytes / t / 1e9 for t in walls]
    wall = statistics.median(walls)
    return {"value": round(statistics.median(values), 4), "unit": "GB/s", "cores": n,
            "kind": "oracle", "runs": [round(v, 4) for v in values],
            "sample": f"the same {len(seq_ids)} sequences as cpu_baseline, {n} processes "
                      f"(whole sequences each), median of {runs} rounds: {wall:.2f} s wall, "
                      f"busiest process {statistics.median(busiest):.2f} s"}


# ----------------------------------------------------------------------------- arms

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, dev=None) -> float:
    """The slowest rank's time (every rank gets it)."""
    if world == 1:
        return x
    import torch.distributed as dist
    on = dev if (dev is not None and dist.get_backend() == "nccl") else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(w, lens, per_step_bytes, flushed):
    layers = w.num_layers
    return {
        "workload": w.name, "description": w.description, "num_seqs": w.num_seqs,
        "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
        "block_size": 16, "num_blocks": w.num_blocks, "context_tokens": int(lens.sum()),
        "max_context_len": int(lens.max()), "layers_per_step": layers,
        "step": ("write 1 new token/seq + partition pass + LSE merge, one layer" if layers == 1
                 else f"{layers} layers x (write + partition pass + LSE merge), one CUDA graph"),
        "l2": ("L2 flushed (256 MB write) before every timed step" if flushed else
               "inputs larger than L2: %.2f GB touched per step vs 129 MB L2, no flush"
               % (per_step_bytes / 1e9)),
    }


def unique_kv_tokens(w, lens) -> int:
    """Context tokens counted once: with a shared prefix of P blocks every
    sequence reads the same first 16 P tokens (up to its own length)."""
    lens = lens.astype(np.int64)
    ptok = 16 * w.prefix_blocks
    if not ptok:
        return int(lens.sum())
    return int(np.maximum(lens - ptok, 0).sum() + min(int(lens.max()), ptok))


class DecodeStep:
    """One decode step of workload `w` through the library's public calls: the
    fused write + partition pass and the merge (paged_kv_decode_step), the
    cascade for a shared prefix (paged_kv_decode_step_cascade), or, for a
    multi-layer workload, every layer in one paged_kv_decode_step_layers call
    captured once into a CUDA graph and replayed."""

    def __init__(self, pkv, wl, w, inp, dev, stream):
        self.pkv, self.w, self.inp, self.stream = pkv, w, inp, stream
        lens = inp["context_lens_host"]
        B, Hq, D = w.num_seqs, w.num_q_heads, w.head_dim
        self.max_len = max_len = int(lens.max())
        self.L = L = w.num_layers
        self.P = P = w.prefix_blocks
        self.out = torch.empty_like(inp["q"])
        self.ws = (pkv.new_cascade_workspace(B, Hq, D, max_len, P, dev) if P
                   else pkv.new_workspace(B, Hq, D, max_len, dev))
        self.step_bytes = L * wl.algorithmic_bytes(w, lens, with_write=True)
        # unique bytes: the shared prefix's K/V counted once
        self.unique_bytes = self.step_bytes - L * (int(lens.sum()) - unique_kv_tokens(w, lens)) \
            * w.num_kv_heads * D * 4
        self.need_flush = self.unique_bytes <= 4 * L2_BYTES
        min_pb = pkv.paged_attention_min_partition_blocks(max_len)
        merges = int((max_len + 15) // 16 > max(min_pb, 8))
        self.launches = L * (3 if P else 1 + merges)
        self.eager_ms = None
        self.graph = None
        if L > 1:
            q_all = inp["q_layers"].contiguous()
            self.out_all = torch.empty_like(q_all)
            lay = (q_all, inp["k_new"], inp["v_new"], inp["k_cache"], inp["v_cache"],
                   inp["block_tables"], inp["context_lens"], max_len, w.scale, self.out_all,
                   self.ws)
            for _ in range(3):
                pkv.paged_kv_decode_step_layers(*lay, stream=stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(20):
                pkv.paged_kv_decode_step_layers(*lay, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            self.eager_ms = e0.elapsed_time(e1) / 20
            cap = torch.cuda.Stream()
            cap.wait_stream(stream)
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(self.graph, stream=cap, capture_error_mode="relaxed"):
                    pkv.paged_kv_decode_step_layers(*lay, stream=cap)
            stream.wait_stream(cap)
            torch.cuda.synchronize()

    def __call__(self):
        if self.graph is not None:
            self.graph.replay()
            return
        i, w, pkv = self.inp, self.w, self.pkv
        if self.P:
            pkv.paged_kv_decode_step_cascade(i["q"], i["k_new"][0], i["v_new"][0],
                                             i["k_cache"][0], i["v_cache"][0], i["block_tables"],
                                             i["context_lens"], self.max_len, self.P, w.scale,
                                             self.out, self.ws, stream=self.stream)
        else:
            pkv.paged_kv_decode_step(i["q"], i["k_new"][0], i["v_new"][0], i["k_cache"][0],
                                     i["v_cache"][0], i["block_tables"], i["context_lens"],
                                     self.max_len, w.scale, self.out, self.ws,
                                     stream=self.stream)


def time_loop(step, K, stream, flush=None):
    """Milliseconds per call of step() over K calls, CUDA events on `stream`:
    one pair around the whole loop, or, with an L2 flush before every call,
    one pair around each call (the flush outside)."""
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / K


# decode workloads timed beside the default line (steps, warm-up): the other
# four decode configurations
SECONDARY = {"tiny": (1000, 20), "qwen3_0p6b": (200, 5), "tinyllama_1p1b": (1000, 20),
             "prefix_shared": (1000, 20)}


def bytes_formula(w) -> str:
    f = ("sum_s n_s*Hkv*D*4 (K and V of every valid token) + 2*B*Hq*D*2 (q in, out) "
         "+ 4*sum_s ceil(n_s/16) (table entries) + 4*B (lengths) + 2*B*Hkv*D*2*2 "
         "(new K/V rows read and written)")
    if w.num_layers > 1:
        f = f"{w.num_layers} layers x [{f}]"
    if w.prefix_blocks:
        f += ("; unique: the shared prefix's 16*P tokens counted once, "
              "(sum_s max(n_s - 16P, 0) + 16P)*Hkv*D*4 in the first term")
    return f


def secondary_workload(pkv, wl, name, dev, stream, peak, flush):
    steps, warmup = SECONDARY[name]
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, device=dev, num_layers=w.num_layers)
    lens = inp["context_lens_host"]
    st = DecodeStep(pkv, wl, w, inp, dev, stream)
    fl = flush if st.need_flush else None
    for _ in range(warmup):
        if fl is not None:
            fl.zero_()
        st()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    ms = time_loop(st, steps, stream, fl)
    clk = clocks.stop()
    if pkv.pkv_device_status() != 0:
        raise SystemExit(f"device status flags set during the {name} benchmark")
    gbs = st.step_bytes / (ms / 1e3) / 1e9
    ent = {
        "description": w.description, "step_us": round(ms * 1e3, 2), "steps": steps,
        "value": round(gbs, 2), "unit": "GB/s",
        "frac_of_measured_hbm": round(gbs / peak, 4),
        "pct_of_nominal_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
        "tokens_per_s_per_layer": round(w.num_seqs / (ms / 1e3 / w.num_layers), 1),
        "us_per_layer": round(ms * 1e3 / w.num_layers, 2),
        "bytes_per_step": int(st.step_bytes), "bytes_formula": bytes_formula(w),
        "context_tokens": int(lens.sum()), "layers_per_step": w.num_layers,
        "gpu_launches_per_step": st.launches,
        "l2": ("L2 flushed (256 MB write) before every timed step" if fl is not None else
               "inputs larger than L2 (%.2f GB per step), no flush" % (st.step_bytes / 1e9)),
        "api": ("paged_kv_decode_step_layers, one CUDA graph replay per step" if st.graph else
                "paged_kv_decode_step_cascade" if st.P else "paged_kv_decode_step"),
        "clocks": clk,
    }
    if st.P:
        ugbs = st.unique_bytes / (ms / 1e3) / 1e9
        ent.update(unique_bytes_per_step=int(st.unique_bytes), unique_gbs=round(ugbs, 2),
                   unique_frac_of_measured_hbm=round(ugbs / peak, 4),
                   note="value counts the shared prefix once per sequence (logical bytes); "
                        "unique_gbs counts it once")
    if st.eager_ms is not None:
        ent["eager_us_per_step"] = round(st.eager_ms * 1e3, 2)
    del st, inp
    torch.cuda.empty_cache()
    return ent


def prefill_measure(pkv, wl, dev, K, warmup):
    """Chunked-prefill attention on the Llama-7B-shaped prompt batch."""
    w = wl.WORKLOADS["llama7b_prefill"]
    inp = wl.make_prefill_inputs(w, chunk=2048, device=dev)
    kc, vc = inp["k_cache"][0], inp["v_cache"][0]
    # the chunk's K/V go to their slots first: the slot of row r is that of the
    # last token of its sequence cut at row_pos[r] + 1 tokens (library call)
    row_tables = inp["block_tables"].index_select(0, inp["row_seq"].long()).contiguous()
    row_slots = pkv.paged_kv_slot_mapping(row_tables, inp["row_pos"] + 1, w.num_blocks)
    pkv.reshape_and_cache(inp["k_rows"], inp["v_rows"], kc, vc, row_slots)
    q, out = inp["q_rows"], torch.empty_like(inp["q_rows"])
    lens = inp["context_lens_host"]
    qlens = np.diff(inp["cu_q_lens_host"])
    flops = wl.prefill_flops(lens, qlens, w.num_q_heads, w.head_dim)

    def step():
        pkv.paged_attention_prefill(q, kc, vc, inp["block_tables"], inp["context_lens"],
                                    inp["cu_q_lens"], inp["max_q_len"], w.scale, out)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    # bytes one step touches: q read, out written, the chunks' K/V read
    touched = 2 * q.numel() * q.element_size() + \
        2 * int(lens.sum()) * w.num_kv_heads * w.head_dim * q.element_size()
    clocks = ClockSampler(dev.index)
    ms = time_loop(step, K, torch.cuda.current_stream())
    clk = clocks.stop()
    if pkv.pkv_device_status() != 0:
        raise SystemExit("device status flags set during the prefill benchmark")
    peak = None
    try:
        peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
    except Exception:
        pass
    tf = flops / (ms / 1e3) / 1e12
    res = dict(w=w, ms=ms, tf=tf, peak=peak, flops=flops, rows=int(qlens.sum()),
               touched=touched, clocks=clk)
    del inp, q, out
    torch.cuda.empty_cache()
    return res


def cow_measure(pkv, dev, stream, peak):
    """The prefix cache's copy-on-write: its device half (paged_kv_copy_blocks)
    on a Llama-7B-shaped layer pool, 2048 (source, destination) block pairs per
    call, and the host allocator's operations through the Python binding."""
    NB, Hkv, D, pairs = 65536, 8, 128, 2048
    g = torch.Generator(device=dev).manual_seed(2116)
    kc = torch.randn(NB, 16, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn(NB, 16, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
    perm = torch.from_numpy(np.random.default_rng(2116).permutation(NB)[:2 * pairs]
                            .astype(np.int32)).to(dev)
    src, dst = perm[:pairs].contiguous(), perm[pairs:].contiguous()

    def step():
        pkv.paged_kv_copy_blocks(kc, vc, src, dst, stream=stream)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    K = 200
    ms = time_loop(step, K, stream)
    clk = clocks.stop()
    if pkv.pkv_device_status() != 0:
        raise SystemExit("device status flags set during the copy-on-write benchmark")
    block_bytes = 16 * Hkv * D * 2
    moved = pairs * 2 * 2 * block_bytes  # K and V, read and written
    gbs = moved / (ms / 1e3) / 1e9
    del kc, vc
    torch.cuda.empty_cache()

    # host allocator: each operation timed over many calls (CPU wall clock)
    alloc = pkv.BlockAllocator(NB)
    ops = {}

    def timed(name, fn, n):
        t0 = time.perf_counter()
        for i in range(n):
            fn(i)
        ops[name] = round((time.perf_counter() - t0) / n * 1e6, 3)

    held = []
    timed("alloc_1_us", lambda i: held.append(alloc.alloc(1)[0]), 20000)
    timed("share_1_us", lambda i: alloc.share([held[i]]), 20000)
    timed("free_1_us", lambda i: alloc.free([held[i]]), 20000)   # drops the shared ref
    hashes = [pkv.paged_kv_block_hash(0 if i == 0 else i, list(range(16 * i, 16 * i + 16)))
              for i in range(64)]
    for i, h in enumerate(hashes):
        alloc.prefix_insert(held[i], h)
    timed("prefix_lookup_64_blocks_us",
          lambda i: alloc.free(alloc.prefix_lookup(hashes)), 2000)

    def share_cow_free(i):  # a writer moved off a shared block, then its copy freed
        b = held[100 + i % 1000]
        alloc.share([b])
        moved_to, _ = alloc.cow(b)
        alloc.free([moved_to])

    timed("share_cow_free_us", share_cow_free, 10000)
    alloc.close()
    return {
        "description": "copy-on-write of 2048 random blocks of a Llama-7B-shaped layer "
                       "(16 x 8 KV heads x 128, bf16, K and V) in a 65536-block pool; host "
                       "allocator operations",
        "step_us": round(ms * 1e3, 2), "steps": K, "value": round(gbs, 2), "unit": "GB/s",
        "frac_of_measured_hbm": round(gbs / peak, 4),
        "bytes_per_step": moved,
        "bytes_formula": "pairs * 2 (K, V) * 2 (read, write) * 16 * Hkv * D * 2",
        "gpu_launches_per_step": 1, "api": "paged_kv_copy_blocks",
        "l2": "256 MB moved per call from random blocks of 4.3 GB of pools, no flush",
        "host_allocator_us_per_op": ops,
        "host_note": "BlockAllocator through the Python binding (ctypes call included), "
                     "CPU wall clock",
        "clocks": clk,
    }


def prefill_kernel_name() -> str:
    return ("prefill_tma_kernel (mma.sync m16n8k16)"
            if os.environ.get("PKV_PREFILL_KERNEL") == "mma" else
            "prefill_tc_kernel (tcgen05.mma kind::f16)")


def run_ours(args):
    import paged_kv_cache_211_gb300 as pkv
    from paged_kv_cache_211_gb300 import workloads as wl

    world, rank, local = dist_init()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.lib()  # fail loudly if the library is missing
    w = wl.WORKLOADS[args.workload]
    if args.pool_blocks:
        w = w.with_(num_blocks=args.pool_blocks)
    L = w.num_layers
    inp = wl.make_inputs(w, device=dev, num_layers=L)
    lens = inp["context_lens_host"]
    B, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    q, kc, vc = inp["q"], inp["k_cache"][0], inp["v_cache"][0]
    kn, vn = inp["k_new"][0], inp["v_new"][0]
    bt, cl = inp["block_tables"], inp["context_lens"]
    stream = torch.cuda.current_stream()
    step = DecodeStep(pkv, wl, w, inp, dev, stream)
    max_len, out, ws, P = step.max_len, step.out, step.ws, step.P
    step_bytes = step.step_bytes
    blocks = int(((lens.astype(np.int64) + 15) // 16).sum())
    # the fused write + partition kernel: K/V of every valid token (the new row
    # read from k_new/v_new instead of the cache), q, table entries, lengths,
    # and the new rows written
    part_bytes = (wl.kv_bytes(w, lens) + B * Hq * D * 2 + blocks * 4 + B * 4
                  + 2 * B * Hkv * D * 2)
    need_flush = step.need_flush
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step_split(evs):
        # the same two kernels through their own entry points, with events
        # between (which also keeps the two from overlapping)
        if P:  # the cascade's three kernels are timed together
            evs[0].record(stream)
            step()
            evs[1].record(stream)
            evs[2].record(stream)
            return
        evs[0].record(stream)
        pkv.paged_kv_decode_step_partition_pass(q, kn, vn, kc, vc, bt, cl, max_len, w.scale,
                                                out, ws, stream=stream)
        evs[1].record(stream)
        pkv.paged_attention_merge_pass(q, kc, vc, bt, cl, max_len, w.scale, out, ws,
                                       stream=stream)
        evs[2].record(stream)

    K = args.steps
    for _ in range(max(args.warmup, 3)):
        if need_flush:
            flush.zero_()
        step()
    torch.cuda.synchronize()

    # timed region A: the step as a user calls it -> value, ms_per_step
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index) if rank == 0 else None
    ms = time_loop(step, K, stream, flush if need_flush else None)
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(ms, world, dev)

    # timed region B: per-kernel durations (roofline of the dominant kernel)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        if need_flush:
            flush.zero_()
        step_split(evs[i])
    torch.cuda.synchronize()
    barrier(world)
    if pkv.pkv_device_status() != 0:
        raise SystemExit("device status flags set during the benchmark")
    t_part = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    t_merge = sum(e[1].elapsed_time(e[2]) for e in evs) / K

    # end to end through the host-buffer entry point: pinned inputs in, output out
    e2e = None
    if not args.no_e2e and L == 1 and not P:
        pin = lambda t: t.cpu().pin_memory()
        qh, knh, vnh, bth, clh = pin(q), pin(kn), pin(vn), pin(bt), pin(cl)
        outh = torch.empty_like(qh).pin_memory()
        staging = torch.empty(pkv.paged_kv_decode_step_staging_bytes(B, Hq, Hkv, D, bt.shape[1]),
                              dtype=torch.uint8, device=dev)

        def host_step():
            pkv.paged_kv_decode_step_host(qh, knh, vnh, bth, clh, outh, staging, kc, vc, max_len,
                                          w.scale, ws, stream=stream)

        for _ in range(max(args.warmup, 3)):
            host_step()
        torch.cuda.synchronize()
        barrier(world)
        e_ms = time_loop(host_step, K, stream, flush if need_flush else None)
        barrier(world)
        e_ms = max_over_ranks(e_ms, world, dev)
        h2d = (qh.numel() * 2 + knh.numel() * 2 + vnh.numel() * 2 + bth.numel() * 4 +
               clh.numel() * 4)
        e2e = {"value": round(world * step_bytes / (e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e_ms, 5), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(outh.numel() * 2),
               "api": "paged_kv_decode_step_host (pinned host q, k_new, v_new, block tables, "
                      "lengths in; attention output out)"}

    peak, peak_kind = measured_peaks()
    launches, eager_ms = step.launches, step.eager_ms
    # the other decode workloads and prefill, each under its own clock record
    workloads = None
    if not args.no_workloads and rank == 0 and world == 1 and w.name == DEFAULT_WORKLOAD:
        del step
        workloads = {}
        for name in SECONDARY:
            workloads[name] = secondary_workload(pkv, wl, name, dev, stream, peak, flush)
        pf = prefill_measure(pkv, wl, dev, K=50, warmup=5)
        workloads["llama7b_prefill"] = {
            "description": pf["w"].description, "step_us": round(pf["ms"] * 1e3, 2),
            "steps": 50, "value": round(pf["tf"], 2), "unit": "TFLOP/s",
            "frac_of_measured_bf16": round(pf["tf"] / pf["peak"], 4) if pf["peak"] else None,
            "flops_per_step": pf["flops"], "query_rows": pf["rows"],
            "flops_formula": "4 * sum over query rows of (visible keys = position + 1) * Hq * D "
                             "(causal q.k and p.v)",
            "kernel": prefill_kernel_name(), "gpu_launches_per_step": 1,
            "l2": "inputs larger than L2: %.2f GB touched per step, no flush (compute-bound)"
                  % (pf["touched"] / 1e9),
            "api": "paged_attention_prefill", "clocks": pf["clocks"]}
        workloads["prefix_cache_cow"] = cow_measure(pkv, dev, stream, peak)

    if rank != 0:
        return
    value = world * step_bytes / (ms / 1e3) / 1e9
    achieved = part_bytes / (t_part / 1e3) / 1e9
    cpu, cpu_all = None, None
    if not args.no_cpu_baseline:
        cpu, seqs = cpu_baseline(inp, w)
        try:
            cpu_all = cpu_baseline_all_cores(inp, w, seqs)
        except Exception as e:  # the one-thread baseline stands on its own
            cpu_all = {"unavailable": f"{type(e).__name__}: {e}"[:200]}
    # the committed summary's DRAM bytes are those of the default workload only
    traffic = recorded_traffic() if w.name == DEFAULT_WORKLOAD else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded N(0,1) K/V/q, shuffled block tables)",
        "config": dict(workload_config(w, lens, step_bytes, need_flush),
                       **({"cascade_prefix_blocks": P} if P else {})),
        "tokens_per_s_per_layer": round(world * B / (ms / 1e3 / L), 1),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * value / world / peak, 2),
        "algorithmic_bytes_per_step": int(step_bytes),
        "kernels_ms": {"decode_partition_fused_write": round(t_part, 5),
                       "decode_merge": round(t_merge, 5),
                       "note": "each kernel between its own events, so the merge and the "
                               "next partition pass do not overlap the partition pass here"},
        "roofline": {"bound": "hbm", "kernel": partition_kernel_name(),
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": int(part_bytes),
                     "traffic": traffic},
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": e2e,
        "gpu_launches": K * launches,
        "eager_ms_per_step": None if eager_ms is None else round(eager_ms, 5),
        "clocks": clk,
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)


def run_prefill(args):
    """Chunked-prefill attention on the Llama-7B-shaped prompt batch: TFLOP/s."""
    import paged_kv_cache_211_gb300 as pkv
    from paged_kv_cache_211_gb300 import workloads as wl

    dev = torch.device("cuda", 0)
    pf = prefill_measure(pkv, wl, dev, K=max(1, min(args.steps, 200)), warmup=args.warmup)
    w, ms, tf, peak = pf["w"], pf["ms"], pf["tf"], pf["peak"]
    K = max(1, min(args.steps, 200))
    print(json.dumps({
        "metric": "chunked-prefill attention TFLOP/s (causal, paged cache)", "value": round(tf, 2),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "description": w.description,
                   "query_rows": pf["rows"], "flops": pf["flops"],
                   "l2": "inputs larger than L2: %.2f GB touched per step vs 129 MB L2, no "
                         "flush (compute-bound)" % (pf["touched"] / 1e9)},
        "roofline": {"bound": "tensor", "achieved": round(tf, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4) if peak else None,
                     "kernel": prefill_kernel_name(),
                     "note": "causal FLOPs (4 * visible pairs * D * query heads) against the "
                             "measured cuBLAS bf16 burst peak"},
        "gpu_launches": K, "clocks": pf["clocks"]}), flush=True)


def run_reference(args):
    """The CPU oracle, as it stands, on a bounded sample of the same workload per step."""
    from paged_kv_cache_211_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    inp = wl.make_inputs(w, device=dev, num_layers=1)
    lens = inp["context_lens_host"]
    order = [int(s) for s in np.random.default_rng(w.seed + 7).permutation(len(lens))]
    cache = {}

    def sample(s, kvh, nq):
        key = (s, kvh, nq)
        if key not in cache:
            cache.clear()  # one sequence's copies at a time
            cache[key] = compact_host(inp, [s], kv_heads=kvh, q_heads=nq)
        return cache[key]

    def sub(kvh, nq):  # the workload restricted to the sampled heads
        return w.with_(num_q_heads=nq, num_kv_heads=kvh)

    # calibrate on one KV head with its whole group of query heads, of one
    # sequence: the sample keeps the workload's arithmetic per K/V byte
    g = w.group
    t0 = time.perf_counter()
    oracle_step(sample(order[0], 1, g), sub(1, g))
    t1 = max(time.perf_counter() - t0, 1e-6)
    total_steps = args.steps + args.warmup
    per_step = min(2.0, 120.0 / max(total_steps, 1))
    kvh = max(1, min(w.num_kv_heads, int(round(per_step / t1))))
    nq = kvh * g
    times, nbytes = [], []
    for i in range(total_steps):
        s = order[i % len(order)]
        hs = sample(s, kvh, nq)
        t0 = time.perf_counter()
        oracle_step(hs, sub(kvh, nq))
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            nbytes.append(sample_bytes(w, lens[[s]], kvh, nq))
    secs = sum(times)
    value = sum(nbytes) / secs / 1e9
    ms = 1e3 * secs / len(times)
    sample_txt = (f"per step: 1 of {w.num_seqs} sequences (cycling), {kvh} of "
                  f"{w.num_kv_heads} KV head(s) with all {g} query heads of each; "
                  f"write + attention, fp64, 1 thread")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) K/V/q, shuffled block tables)",
        "config": workload_config(w, lens, wl.algorithmic_bytes(w, lens),
                                  wl.algorithmic_bytes(w, lens) <= 4 * L2_BYTES),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample_txt},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill:
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
