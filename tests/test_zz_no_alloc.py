"""paged_attention_decode_noalloc: decode attention for callers that cannot
allocate device memory (a plug-in inside a framework that owns all device
memory, or a runtime whose memory plan is fixed at start-up).  It keeps its
split-context partials in a static array inside the library instead of a
caller workspace.

Checked through the C ABI against paged_attention_decode on the same inputs,
within the tolerance the parity tests use, on two calls in a row (the second
call finds the first call's partials still in the shared array).  This file
sorts last so that a run stopping at the first failure has run every other
test first; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_211_gb300 as pkv
from paged_kv_cache_211_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _prepared(name, dev, **kw):
    """A workload whose step tokens are already written, so every row is valid."""
    w = wl.WORKLOADS[name].with_(**kw)
    inp = wl.make_inputs(w, device=dev, num_layers=1)
    kc, vc = inp["k_cache"][0], inp["v_cache"][0]
    pkv.paged_kv_write_new_tokens(inp["k_new"][0], inp["v_new"][0], kc, vc,
                                  inp["block_tables"], inp["context_lens"])
    return w, inp


def _close(got, want):
    g, r = got.float(), want.float()
    assert torch.isfinite(g).all()
    bound = torch.clamp(1e-2 * r.abs(), min=4e-3)
    err = (g - r).abs()
    assert bool((err <= bound).all()), f"max error {err.max().item():.3e}"


def test_noalloc_matches_workspace_entry_two_calls_in_a_row(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    cases = [_prepared("prefix_shared", cuda_device, num_seqs=48),   # 2+ partitions per seq
             _prepared("qwen3_0p6b", cuda_device)]                    # other sizes, fp16
    for w, inp in cases:
        q, kc, vc = inp["q"], inp["k_cache"][0], inp["v_cache"][0]
        bt, cl = inp["block_tables"], inp["context_lens"]
        max_len = int(inp["context_lens_host"].max())
        assert pkv.paged_attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                                   max_len) <= pkv.NOALLOC_SCRATCH_BYTES
        want = torch.empty_like(q)
        ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, cuda_device)
        pkv.paged_attention_decode(q, kc, vc, bt, cl, max_len, w.scale, want, ws)
        got = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode_noalloc(q, kc, vc, bt, cl, max_len, w.scale, got)
        torch.cuda.synchronize()
        _close(got, want)
    assert pkv.pkv_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    B, Hq, D, max_len = 4096, 32, 128, 32768
    assert pkv.paged_attention_workspace_bytes(B, Hq, D, max_len) > pkv.NOALLOC_SCRATCH_BYTES
    L = pkv.lib()
    p = pkv.ctypes.c_void_p(4096)   # never touched: the size check comes first
    rc = L.paged_attention_decode_noalloc(p, p, p, p, 2048, p, max_len, B, Hq, 8, D, 100, 0.1,
                                          p, 1, None)
    assert rc == 6
