"""Seeded synthetic decode workloads (inputs only; no attention arithmetic).

This module is the one piece the CUDA path and the CPU oracle share: it
makes the inputs (query rows, K/V pools, block tables, context lengths and
the step's new K/V rows) and nothing else.  It contains none of the method's
arithmetic: no gather, no dot product, no softmax, no slot computation.

Shapes follow the pages' workloads (model *shapes* only, no weights):
Qwen3-0.6B ("micro-vLLM" wiki quick start; "MinivLLM" 使用教程 step 3),
TinyLlama-1.1B ("mini-vllm 项目深度解析" 项目概述) and Llama/Mistral
("micro-vLLM" wiki feature list).  The cache is cut into 16-token blocks
("mini-vllm 项目深度解析" §2) and each layer's pool is laid out
[num_blocks][16][num_kv_heads][head_dim], separately for K and V
(§关键工程决策 item 3).

Poisoning: every slot that holds no valid token (unused blocks, slots past a
sequence's length in its last block, and the slot the step's new token is
about to be written to) is filled with NaN, and unused block-table entries
point at a poisoned block, so that a stray read shows up as NaN.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BLOCK_SIZE = 16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    num_blocks: int
    dtype: str                 # "f16" or "bf16"
    lens: str                  # how context lengths are drawn (see context_lens)
    max_blocks_per_seq: int
    num_layers: int = 1        # layers whose pools are laid out layer-major
    prefix_blocks: int = 0     # leading physical blocks shared by every sequence
    description: str = ""

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(
        "tiny", 2111, 4, 16, 8, 128, 64, "f16", "fixed:17,33,64,100", 7,
        description="4 seqs, lens {17,33,64,100}, 16q/8kv, D=128, fp16, 64-block pool"),
    "qwen3_0p6b": Workload(
        "qwen3_0p6b", 2112, 60, 16, 8, 128, 4096, "f16", "uniform:32,512", 32, num_layers=28,
        description="Qwen3-0.6B-shaped: 60 seqs, lens U[32,512], 16q/8kv, D=128, fp16, "
                    "4096-block pool per layer, 28 layers per step"),
    "tinyllama_1p1b": Workload(
        "tinyllama_1p1b", 2113, 256, 32, 4, 64, 40000, "f16", "fixed_all:2048", 128,
        description="TinyLlama-1.1B-shaped: 256 seqs x 2048, 32q/4kv (GQA 8), D=64, fp16, "
                    "40000-block pool"),
    "llama7b_long": Workload(
        "llama7b_long", 2114, 32, 32, 8, 128, 65536, "bf16", "lognormal:8192,0.5,32768", 2048,
        description="Llama/Mistral-7B-shaped long context: 32 seqs, lens lognormal "
                    "(median 8192, sigma 0.5, cap 32768), 32q/8kv, D=128, bf16, 65536-block pool"),
    "llama7b_prefill": Workload(
        "llama7b_prefill", 2116, 8, 32, 8, 128, 1536, "bf16", "fixed_all:2048", 128,
        description="Llama-7B-shaped chunked prefill: 8 prompts x 2048 tokens, the whole "
                    "prompt as one chunk, 32q/8kv, D=128, bf16"),
    "prefix_shared": Workload(
        "prefix_shared", 2115, 128, 16, 8, 128, 4096, "bf16", "prefix:1024,64,512", 96,
        prefix_blocks=64,
        description="128 seqs sharing the same first 64 physical blocks (1024-token prefix) "
                    "plus private suffixes U[64,512], 16q/8kv, D=128, bf16, 4096-block pool"),
}


def context_lens(w: Workload) -> np.ndarray:
    """Per-sequence context lengths (including this step's new token)."""
    rng = np.random.default_rng(w.seed)
    kind, _, arg = w.lens.partition(":")
    if kind == "fixed":
        vals = [int(x) for x in arg.split(",")]
        assert len(vals) == w.num_seqs
        lens = np.array(vals, np.int64)
    elif kind == "fixed_all":
        lens = np.full(w.num_seqs, int(arg), np.int64)
    elif kind == "uniform":
        lo, hi = (int(x) for x in arg.split(","))
        lens = rng.integers(lo, hi + 1, size=w.num_seqs)
    elif kind == "lognormal":
        med, sigma, cap = arg.split(",")
        z = rng.standard_normal(w.num_seqs)
        lens = np.clip(np.rint(np.exp(math.log(float(med)) + float(sigma) * z)), 1, int(cap))
        lens = lens.astype(np.int64)
    elif kind == "prefix":
        plen, lo, hi = (int(x) for x in arg.split(","))
        lens = plen + rng.integers(lo, hi + 1, size=w.num_seqs)
    else:
        raise ValueError(f"unknown length kind {w.lens!r}")
    assert lens.max() <= w.max_blocks_per_seq * BLOCK_SIZE
    return lens.astype(np.int32)


def block_tables(w: Workload, lens: np.ndarray):
    """Block tables drawn from a seeded random permutation of the pool.

    Returns (tables [B, MB] int32, used_mask [NB] bool, poison_block id).
    Sequences take physical blocks from the permutation in order; with
    ``prefix_blocks`` the first entries of every table are the same shared
    blocks.  Entries past a sequence's last block point at a poisoned block.
    """
    rng = np.random.default_rng(w.seed + 1)
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    need = (lens.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE
    tables = np.empty((w.num_seqs, w.max_blocks_per_seq), np.int32)
    used = np.zeros(w.num_blocks, bool)
    pos = 0
    shared = perm[:w.prefix_blocks]
    pos += w.prefix_blocks
    for s in range(w.num_seqs):
        n = int(need[s])
        own = n - w.prefix_blocks
        assert own >= 0
        row = np.concatenate([shared, perm[pos:pos + own]])
        pos += own
        if pos > w.num_blocks:
            raise ValueError("pool too small for the drawn lengths")
        tables[s, :n] = row
        used[row] = True
    unused = np.flatnonzero(~used)
    poison = int(unused[0]) if unused.size else -1
    if poison < 0:
        raise ValueError("workload leaves no free block to poison")
    for s in range(w.num_seqs):
        tables[s, int(need[s]):] = poison
    return tables, used, poison


def _randn(shape, dtype, device, gen, chunk=1 << 27):
    """Standard-normal values rounded to ``dtype`` (generated in fp32 chunks)."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out


def make_inputs(w: Workload, device="cpu", poison: bool = True,
                num_layers: Optional[int] = None) -> dict:
    """All inputs of one decode step of ``w`` as torch tensors on ``device``.

    Keys: q [B,Hq,D] (and q_layers [L,B,Hq,D], q_layers[0] = q), k_cache/v_cache
    [L,NB,16,Hkv,D] (layer-major; L=1 unless ``num_layers``), block_tables [B,MB]
    int32, context_lens [B] int32,
    k_new/v_new [L,B,Hkv,D] (the token at position len-1), plus host copies of
    lengths and tables and the poison bookkeeping.
    """
    L = w.num_layers if num_layers is None else num_layers
    lens = context_lens(w)
    tables, used, poison_block = block_tables(w, lens)
    dt = w.torch_dtype
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + 7)
    B, Hq, Hkv, D, NB = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_blocks
    q = _randn((B, Hq, D), dt, dev, gen)
    k_cache = _randn((L, NB, BLOCK_SIZE, Hkv, D), dt, dev, gen)
    v_cache = _randn((L, NB, BLOCK_SIZE, Hkv, D), dt, dev, gen)
    k_new = _randn((L, B, Hkv, D), dt, dev, gen)
    v_new = _randn((L, B, Hkv, D), dt, dev, gen)
    # per-layer queries for multi-layer steps (layer 0 is q itself)
    q_layers = torch.cat([q.unsqueeze(0), _randn((L - 1, B, Hq, D), dt, dev, gen)]) if L > 1 \
        else q.unsqueeze(0)
    if poison:
        nan = float("nan")
        unused_ids = torch.from_numpy(np.flatnonzero(~used)).to(dev)
        k_cache[:, unused_ids] = nan
        v_cache[:, unused_ids] = nan
        # slots past each sequence's length in its last block, and the new
        # token's slot (position len-1), hold no valid token before the write
        blk, off = [], []
        for s in range(B):
            n = int(lens[s])
            last = (n - 1) // BLOCK_SIZE
            b = int(tables[s, last])
            for o in range((n - 1) % BLOCK_SIZE, BLOCK_SIZE):
                blk.append(b)
                off.append(o)
        bi = torch.tensor(blk, dtype=torch.long, device=dev)
        oi = torch.tensor(off, dtype=torch.long, device=dev)
        k_cache[:, bi, oi] = nan
        v_cache[:, bi, oi] = nan
    return {
        "workload": w,
        "q": q,
        "q_layers": q_layers,
        "k_cache": k_cache,
        "v_cache": v_cache,
        "k_new": k_new,
        "v_new": v_new,
        "block_tables": torch.from_numpy(tables).to(dev),
        "context_lens": torch.from_numpy(lens).to(dev),
        "block_tables_host": tables,
        "context_lens_host": lens,
        "used_blocks": used,
        "poison_block": poison_block,
    }


def kv_bytes(w: Workload, lens: np.ndarray) -> int:
    """K+V bytes one decode call must read: every valid token's rows, all KV heads."""
    return int(lens.astype(np.int64).sum()) * w.num_kv_heads * w.head_dim * 2 * 2


def algorithmic_bytes(w: Workload, lens: np.ndarray, with_write: bool = True) -> int:
    """Bytes a decode step must move at minimum.

    K/V rows of every valid token, q in and out back (2 B/elem each), one
    int32 table entry per used block and one length per sequence, plus the
    new token's K/V read and write when the step includes the cache write.
    """
    B, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    blocks = int(((lens.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE).sum())
    total = kv_bytes(w, lens) + 2 * B * Hq * D * 2 + blocks * 4 + B * 4
    if with_write:
        total += 2 * B * Hkv * D * 2 * 2
    return total


def make_prefill_inputs(w: Workload, chunk: int, device="cpu") -> dict:
    """A chunked-prefill step of ``w``: every sequence's last ``chunk`` tokens
    (or all of them, if shorter) are query rows.  Keys as in make_inputs for
    the pools and tables, plus q_rows [R,Hq,D], k_rows/v_rows [R,Hkv,D] (the
    chunk's K/V), cu_q_lens [B+1] int32, and for every packed row its
    sequence (row_seq) and position in that sequence (row_pos), int32 [R]."""
    inp = make_inputs(w, device=device, num_layers=1, poison=False)
    lens = inp["context_lens_host"]
    qlens = np.minimum(lens, chunk).astype(np.int64)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    row_seq = np.repeat(np.arange(w.num_seqs), qlens).astype(np.int32)
    row_pos = np.concatenate([np.arange(int(n) - int(ql), int(n))
                              for n, ql in zip(lens, qlens)]).astype(np.int32)
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed * 1000 + 11)
    R = int(cu[-1])
    inp.update(
        q_rows=_randn((R, w.num_q_heads, w.head_dim), w.torch_dtype, dev, gen),
        k_rows=_randn((R, w.num_kv_heads, w.head_dim), w.torch_dtype, dev, gen),
        v_rows=_randn((R, w.num_kv_heads, w.head_dim), w.torch_dtype, dev, gen),
        cu_q_lens=torch.from_numpy(cu).to(dev), cu_q_lens_host=cu,
        row_seq=torch.from_numpy(row_seq).to(dev), row_pos=torch.from_numpy(row_pos).to(dev),
        max_q_len=int(qlens.max()))
    return inp


def prefill_flops(lens: np.ndarray, qlens: np.ndarray, num_q_heads: int, head_dim: int) -> int:
    """Multiply-adds x 2 of causal attention: row at position p reads p + 1 keys,
    for q.k and for p.v."""
    total = 0
    for n, ql in zip(lens.astype(np.int64), qlens.astype(np.int64)):
        # sum over p = n-ql .. n-1 of (p + 1)
        total += ql * (2 * n - ql + 1) // 2
    return int(4 * total * num_q_heads * head_dim)
