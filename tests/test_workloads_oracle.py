"""The seeded workloads (structure, poison) and the oracle on workload-shaped
inputs against the library reference; golden fixtures."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_211_gb300 import workloads as wl
from pkv_testutil import host_inputs, sdpa_reference, token_slots

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _facts():
    with open(os.path.join(GOLDEN, "pages_facts.json")) as f:
        return json.load(f)


def test_pages_block_size_and_layout():
    facts = _facts()
    assert wl.BLOCK_SIZE == facts["block_size"]["value"] == facts["cache_block_size_cfg"]["value"]
    inp = wl.make_inputs(wl.WORKLOADS["tiny"], num_layers=2)
    w = inp["workload"]
    # layer-major, then [num_blocks, block_size, num_kv_heads, head_dim]
    assert tuple(inp["k_cache"].shape) == (2, w.num_blocks, 16, w.num_kv_heads, w.head_dim)
    assert inp["k_cache"].data_ptr() != inp["v_cache"].data_ptr()   # separate pools


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_workload_tables_and_lengths(name):
    w = wl.WORKLOADS[name]
    lens = wl.context_lens(w)
    tables, used, poison = wl.block_tables(w, lens)
    assert lens.shape == (w.num_seqs,) and lens.min() >= 1
    assert lens.max() <= w.max_blocks_per_seq * 16
    need = (lens + 15) // 16
    seen = {}
    for s in range(w.num_seqs):
        row = tables[s, :need[s]]
        assert ((row >= 0) & (row < w.num_blocks)).all()
        assert not used[poison] and (tables[s, need[s]:] == poison).all()
        for j, b in enumerate(row):
            if j < w.prefix_blocks:
                continue
            assert b not in seen, "private blocks must not be shared"
            seen[b] = s
    if w.prefix_blocks:
        assert (tables[:, :w.prefix_blocks] == tables[0, :w.prefix_blocks]).all()
    # the drawn lengths follow the stated recipe
    if name == "tiny":
        assert lens.tolist() == [17, 33, 64, 100]
    if name == "qwen3_0p6b":
        assert lens.min() >= 32 and lens.max() <= 512
    if name == "tinyllama_1p1b":
        assert (lens == 2048).all()
    if name == "llama7b_long":
        assert lens.max() <= 32768 and 4000 < np.median(lens) < 16000
    if name == "prefix_shared":
        assert (lens >= 1024 + 64).all() and (lens <= 1024 + 512).all()


def test_poison_placement_tiny():
    inp = wl.make_inputs(wl.WORKLOADS["tiny"])
    h = host_inputs(inp)
    kd = oracle.decode_f16(h["k_cache"])
    for s, n in enumerate(h["lens"]):
        valid = token_slots(h["tables"][s], int(n) - 1)
        flat = kd.reshape(-1, *kd.shape[2:])
        assert np.isfinite(flat[valid]).all()
        new_slot = token_slots(h["tables"][s], int(n))[-1]
        assert np.isnan(flat[new_slot]).all(), "the new token's slot must start poisoned"
    assert np.isnan(kd[inp["poison_block"]]).all()


@pytest.mark.parametrize("name,nseq", [("tiny", None), ("qwen3_0p6b", 12), ("prefix_shared", 6)])
def test_oracle_on_workload_vs_sdpa(name, nseq):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, num_layers=1)
    h = host_inputs(inp)
    sl = oracle.slot_mapping(h["tables"], h["lens"], 16, w.num_blocks)
    kc, vc = oracle.reshape_and_cache(h["k_new"], h["v_new"], h["k_cache"], h["v_cache"], sl)
    sel = slice(0, nseq)
    dt = oracle.BF16 if w.dtype == "bf16" else oracle.F16
    got = oracle.decode_attention(dt, h["q"][sel], kc, vc, h["tables"][sel], h["lens"][sel],
                                  w.scale)
    want = sdpa_reference(dt, h["q"][sel], kc, vc, h["tables"][sel], h["lens"][sel], w.scale)
    assert np.isfinite(got).all()
    assert np.allclose(got, want, rtol=1e-10, atol=1e-12)


def test_golden_oracle_regression():
    with open(os.path.join(GOLDEN, "oracle_small_case.json")) as f:
        g = json.load(f)
    B, Hq, D = len(g["context_lens"]), g["num_q_heads"], g["head_dim"]
    NB, BS, Hkv = g["num_blocks"], g["block_size"], g["num_kv_heads"]
    q = np.array(g["q_bits"], np.uint16).reshape(B, Hq, D)
    k = np.array(g["k_bits"], np.uint16).reshape(NB, BS, Hkv, D)
    v = np.array(g["v_bits"], np.uint16).reshape(NB, BS, Hkv, D)
    out = oracle.decode_attention(oracle.F16, q, k, v, g["block_tables"], g["context_lens"],
                                  g["scale"])
    want = np.array([float.fromhex(x) for x in g["expected_out"]]).reshape(out.shape)
    assert np.array_equal(out, want)
    assert oracle.slot_mapping(g["block_tables"], g["context_lens"], BS, NB).tolist() == \
        g["expected_slots"]
