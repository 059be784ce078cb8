"""Helpers for the GPU parity tests: run the oracle on host copies of the
ORIGINAL inputs (never on anything the CUDA path produced)."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from pkv_testutil import bits

BS = 16


def dtype_code(w) -> int:
    return oracle.BF16 if w.dtype == "bf16" else oracle.F16


def _chunks(seq_ids, lens, k):
    """Split seq_ids into at most k groups of about equal token counts (longest
    first to the least-loaded group); each group keeps the input order."""
    seq_ids = [int(s) for s in seq_ids]
    k = max(1, min(k, len(seq_ids)))
    groups, load = [[] for _ in range(k)], [0] * k
    for s in sorted(seq_ids, key=lambda s: -int(lens[s])):
        i = load.index(min(load))
        groups[i].append(s)
        load[i] += int(lens[s]) + 1
    pos = {s: i for i, s in enumerate(seq_ids)}
    return [sorted(g, key=pos.get) for g in groups if g]


def _compact(inp, seq_ids, need_lens, layer):
    """Host copies (bit patterns) of the blocks the sequences `seq_ids` use up to
    need_lens tokens (ids remapped; attention does not depend on physical ids)
    and their remapped tables, taken from the device pools as they are now."""
    tables = inp["block_tables_host"]
    seq_ids = np.asarray(seq_ids)
    need = (need_lens[seq_ids].astype(np.int64) + BS - 1) // BS
    used = sorted({int(b) for s, n in zip(seq_ids, need) for b in tables[s, :n]})
    remap = {b: i for i, b in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=inp["k_cache"].device)
    kc = bits(inp["k_cache"][layer].index_select(0, idx))
    vc = bits(inp["v_cache"][layer].index_select(0, idx))
    tb = np.zeros((len(seq_ids), tables.shape[1]), np.int32)
    for r, (s, n) in enumerate(zip(seq_ids, need)):
        tb[r, :n] = [remap[int(b)] for b in tables[s, :n]]
    return kc, vc, tb


def oracle_steps(inp, seq_ids, steps, layer: int = 0, workers: int | None = None):
    """The oracle's consecutive decode steps on the sequences `seq_ids`.

    steps: dicts with host arrays over ALL sequences of the workload -- q
    [B,Hq,D], k_new / v_new [B,Hkv,D] (uint16 bit patterns) and lens [B]
    int32 -- applied in order: each step writes its new rows at position
    len-1, then attends with its q.  The pools are read from the device as
    they are when this is called (before the GPU touches them).  Work is
    split over threads by sequence (the oracle's C calls release the GIL).
    Returns one fp64 output [len(seq_ids), Hq, D] per step.
    """
    from concurrent.futures import ThreadPoolExecutor
    w = inp["workload"]
    code = dtype_code(w)
    seq_ids = np.asarray(seq_ids)
    need_lens = np.max(np.stack([np.asarray(st["lens"]) for st in steps]), axis=0)
    k = workers or max(1, min(16, os.cpu_count() or 1))
    parts = _chunks(seq_ids, need_lens, k)
    jobs = []
    for part in parts:
        kc, vc, tb = _compact(inp, part, need_lens, layer)
        jobs.append((part, kc, vc, tb))

    def run(job):
        part, kc, vc, tb = job
        outs = []
        for st in steps:
            ln = np.asarray(st["lens"])[part].astype(np.int32)
            slots = oracle.slot_mapping(tb, ln, BS, kc.shape[0])
            kc, vc = oracle.reshape_and_cache(st["k_new"][part], st["v_new"][part], kc, vc,
                                              slots)
            outs.append(oracle.decode_attention(code, st["q"][part], kc, vc, tb, ln, w.scale))
        return outs

    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(run, jobs))
    # back to the order of seq_ids
    row = {int(s): i for i, s in enumerate(seq_ids)}
    outs = []
    for i in range(len(steps)):
        o = np.empty((len(seq_ids),) + results[0][i].shape[1:], np.float64)
        for (part, _, _, _), r in zip(jobs, results):
            o[[row[s] for s in part]] = r[i]
        outs.append(o)
    return outs


def compact_oracle_step(inp, seq_ids, layer: int = 0):
    """Oracle decode step (write, then attention) of the workload's own step
    (q, and layer `layer`'s new rows and pools) for the sequences `seq_ids`.  Returns (out [len(seq_ids), Hq, D] fp64,
    written K rows, written V rows), the written rows [n, Hkv, D] uint16."""
    seq_ids = np.asarray(seq_ids)
    step = dict(q=bits(inp["q"]), k_new=bits(inp["k_new"][layer]),
                v_new=bits(inp["v_new"][layer]), lens=inp["context_lens_host"])
    out = oracle_steps(inp, seq_ids, [step], layer=layer)[0]
    return out, step["k_new"][seq_ids], step["v_new"][seq_ids]


def assert_attention_close(got_bits: np.ndarray, want: np.ndarray, dtype: int, what: str = ""):
    """Parity bar for decode attention with fp16/bf16 outputs:
    elementwise |gpu - oracle| <= max(4e-3, 1e-2 * |oracle|), and the largest
    error relative to the largest |oracle| <= 1e-2.  Returns the errors."""
    got = oracle.decode(dtype, got_bits)
    assert got.shape == want.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    bound = np.maximum(4e-3, 1e-2 * np.abs(want))
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert (err <= bound).all(), (
        f"{what}: error {err[worst]:.3e} at {worst} above {bound[worst]:.3e} "
        f"(gpu {got[worst]:.6f}, oracle {want[worst]:.6f})")
    scale = float(np.abs(want).max()) if want.size else 0.0
    norm_rel = float(err.max()) / scale if scale > 0 else float(err.max())
    assert norm_rel <= 1e-2, f"{what}: norm-relative error {norm_rel:.3e}"
    return float(err.max()), norm_rel


def sample_seqs(lens: np.ndarray, k: int, seed: int = 0) -> np.ndarray:
    """k sequences: the longest, the shortest and a seeded random rest."""
    B = len(lens)
    if k >= B:
        return np.arange(B)
    rng = np.random.default_rng(seed)
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    rest = [int(i) for i in rng.permutation(B) if int(i) not in pick]
    return np.array(sorted(pick | set(rest[:k - len(pick)])))
