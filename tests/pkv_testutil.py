"""Test helpers: conversions and independent (library-based) references.

Nothing here imports the CUDA library; the references below are built from
numpy / torch library routines and plain enumeration, independently of the
C oracle, so that they can pin it.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

BS = 16


def bits(t: torch.Tensor) -> np.ndarray:
    """A 16-bit float tensor's bit patterns as a uint16 numpy array (host copy)."""
    assert t.dtype in (torch.float16, torch.bfloat16)
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)


def lib_decode(a: np.ndarray, dtype: int) -> np.ndarray:
    """Library decoders: numpy's float16 and torch's bfloat16 conversions."""
    if dtype == 0:
        return np.ascontiguousarray(a).view(np.float16).astype(np.float64)
    return from_bits(a, torch.bfloat16).to(torch.float64).numpy()


def token_slots(table_row, n: int, bs: int = BS) -> list:
    """Enumerate a sequence's tokens in order: every slot of every listed block, cut at n."""
    slots = []
    for b in table_row:
        for o in range(bs):
            slots.append(int(b) * bs + o)
            if len(slots) == n:
                return slots
    return slots[:n]


def sdpa_reference(dtype, q, k_cache, v_cache, tables, lens, scale):
    """torch scaled_dot_product_attention in float64 on contiguously gathered contexts.

    Decoding uses the library decoders, gathering uses token_slots and numpy
    fancy indexing, and grouped-query heads are expanded with
    repeat_interleave (query head i <- KV head i // group).
    """
    qd = lib_decode(q, dtype)
    B, Hq, D = qd.shape
    NB, bs, Hkv, _ = k_cache.shape
    g = Hq // Hkv
    kf = k_cache.reshape(NB * bs, Hkv, D)
    vf = v_cache.reshape(NB * bs, Hkv, D)
    out = np.zeros((B, Hq, D))
    for s in range(B):
        n = int(lens[s])
        if n == 0:
            continue
        sl = np.array(token_slots(tables[s], n, bs))
        K = torch.from_numpy(lib_decode(kf[sl], dtype)).permute(1, 0, 2)
        V = torch.from_numpy(lib_decode(vf[sl], dtype)).permute(1, 0, 2)
        K = K.repeat_interleave(g, dim=0)
        V = V.repeat_interleave(g, dim=0)
        qs = torch.from_numpy(qd[s]).unsqueeze(1)
        o = F.scaled_dot_product_attention(qs, K, V, scale=scale)
        out[s] = o.squeeze(1).numpy()
    return out


def host_inputs(inp: dict):
    """uint16 / int views of one layer of a make_inputs() dict, for the oracle."""
    return dict(
        q=bits(inp["q"]),
        k_cache=bits(inp["k_cache"][0]),
        v_cache=bits(inp["v_cache"][0]),
        k_new=bits(inp["k_new"][0]),
        v_new=bits(inp["v_new"][0]),
        tables=inp["block_tables_host"],
        lens=inp["context_lens_host"],
    )


def check_close(got, want, atol=4e-3, rtol_norm=1e-2):
    """The decode-attention parity bar: max abs error <= atol and
    max abs error / max |want| <= rtol_norm; returns (max_abs, norm_rel)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - want)
    max_abs = float(err.max()) if err.size else 0.0
    scale = float(np.abs(want).max()) if want.size else 0.0
    norm_rel = max_abs / scale if scale > 0 else max_abs
    assert max_abs <= atol, f"max abs error {max_abs:.3e} > {atol}"
    assert norm_rel <= rtol_norm, f"norm-relative error {norm_rel:.3e} > {rtol_norm}"
    return max_abs, norm_rel
