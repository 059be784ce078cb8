"""Helpers for the GPU parity tests: run the oracle on host copies of the
ORIGINAL inputs (never on anything the CUDA path produced)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from pkv_testutil import bits

BS = 16


def dtype_code(w) -> int:
    return oracle.BF16 if w.dtype == "bf16" else oracle.F16


def compact_oracle_step(inp: dict, seq_ids, layer: int = 0):
    """Oracle decode step (write, then attention) for the sequences `seq_ids`.

    The blocks those sequences reference are copied from the untouched
    device pools into a compact host pool (ids remapped; attention does not
    depend on physical ids), the oracle writes the new tokens there, then
    computes attention.  Returns (out [len(seq_ids), Hq, D] fp64, written
    K rows, written V rows) where the written rows are [n, Hkv, D] uint16.
    """
    w = inp["workload"]
    tables = inp["block_tables_host"]
    lens = inp["context_lens_host"]
    seq_ids = np.asarray(seq_ids)
    need = (lens[seq_ids].astype(np.int64) + BS - 1) // BS
    used = sorted({int(b) for s, n in zip(seq_ids, need) for b in tables[s, :n]})
    remap = {b: i for i, b in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=inp["k_cache"].device)
    kc = bits(inp["k_cache"][layer].index_select(0, idx))
    vc = bits(inp["v_cache"][layer].index_select(0, idx))
    tb = np.zeros((len(seq_ids), tables.shape[1]), np.int32)
    for r, (s, n) in enumerate(zip(seq_ids, need)):
        tb[r, :n] = [remap[int(b)] for b in tables[s, :n]]
    ln = lens[seq_ids].astype(np.int32)
    sel = torch.tensor(seq_ids, dtype=torch.long, device=inp["q"].device)
    q = bits(inp["q"].index_select(0, sel))
    kn = bits(inp["k_new"][layer].index_select(0, sel))
    vn = bits(inp["v_new"][layer].index_select(0, sel))
    slots = oracle.slot_mapping(tb, ln, BS, len(used))
    kc2, vc2 = oracle.reshape_and_cache(kn, vn, kc, vc, slots)
    out = oracle.decode_attention(dtype_code(w), q, kc2, vc2, tb, ln, w.scale)
    return out, kn, vn


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
