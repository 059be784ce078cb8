"""paged_attention_decode_noalloc: decode attention for callers that cannot
allocate device memory (a plug-in inside a framework that owns all device
memory, or a runtime whose memory plan is fixed at start-up and must not call
cudaMalloc on the serving path).  It keeps its split-context partials in a
static array inside the library instead of a caller workspace.

Checked through the C ABI against the CPU oracle and against
paged_attention_decode on the same inputs, within the tolerance the parity
tests use, on two calls in a row per problem (the second call finds the first
call's partials still in the shared array), over two problems of different
sizes.  Every pointer passed is a real device tensor.  This file sorts last
so that a run stopping at the first failure has run every other test first;
it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_211_gb300 as pkv
from paged_kv_cache_211_gb300 import workloads as wl
from gpu_helpers import assert_attention_close, compact_oracle_step, dtype_code
from pkv_testutil import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    pkv.pkv_device_status(reset=True)


def _prepared(name, dev, **kw):
    """A workload, the oracle's answer for its decode step (computed on the
    untouched pools), and the pools with the step's tokens written."""
    w = wl.WORKLOADS[name].with_(**kw)
    inp = wl.make_inputs(w, device=dev, num_layers=1)
    want, _, _ = compact_oracle_step(inp, np.arange(w.num_seqs))
    pkv.paged_kv_write_new_tokens(inp["k_new"][0], inp["v_new"][0], inp["k_cache"][0],
                                  inp["v_cache"][0], inp["block_tables"], inp["context_lens"])
    return w, inp, want


def test_noalloc_matches_oracle_and_workspace_entry_two_calls_in_a_row(cuda_device):
    cases = [_prepared("prefix_shared", cuda_device, num_seqs=48),   # partials in the scratch
             _prepared("qwen3_0p6b", cuda_device)]                    # other sizes, fp16
    scratch = pkv.paged_attention_noalloc_scratch_bytes()
    assert scratch == 32 << 20
    for w, inp, want in cases:
        q, kc, vc = inp["q"], inp["k_cache"][0], inp["v_cache"][0]
        bt, cl = inp["block_tables"], inp["context_lens"]
        max_len = int(inp["context_lens_host"].max())
        assert pkv.paged_attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                                   max_len) <= scratch
        ref = torch.empty_like(q)
        ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, cuda_device)
        pkv.paged_attention_decode(q, kc, vc, bt, cl, max_len, w.scale, ref, ws)
        got = [torch.full_like(q, float("nan")) for _ in range(2)]
        for g in got:                          # two calls in a row on the shared array
            pkv.paged_attention_decode_noalloc(q, kc, vc, bt, cl, max_len, w.scale, g)
        torch.cuda.synchronize()
        assert pkv.pkv_device_status() == 0
        code = dtype_code(w)
        assert_attention_close(bits(ref), want, code, f"{w.name} workspace entry")
        for i, g in enumerate(got):
            assert_attention_close(bits(g), want, code, f"{w.name} no-alloc call {i + 1}")
            # against the existing entry point, within the same elementwise bar
            diff = (g.float() - ref.float()).abs()
            bound = torch.clamp(1e-2 * ref.float().abs(), min=4e-3)
            assert bool((diff <= bound).all()), f"{w.name} call {i + 1}: {diff.max():.3e}"


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_device):
    """A problem whose workspace would exceed the scratch is refused before
    anything is enqueued: the output keeps its contents.  The tensors are
    real and small (one-token contexts); only the length bound is large."""
    dev = cuda_device
    B, Hq, Hkv, D, max_len, NB = 64, 32, 8, 128, 32768, 4
    need = pkv.paged_attention_workspace_bytes(B, Hq, D, max_len)
    assert need > pkv.paged_attention_noalloc_scratch_bytes()
    q = torch.randn(B, Hq, D, device=dev).to(torch.bfloat16)
    kc = torch.randn(NB, 16, Hkv, D, device=dev).to(torch.bfloat16)
    vc = torch.randn(NB, 16, Hkv, D, device=dev).to(torch.bfloat16)
    bt = torch.zeros(B, max_len // 16, dtype=torch.int32, device=dev)
    cl = torch.ones(B, dtype=torch.int32, device=dev)
    out = torch.full_like(q, float("nan"))
    torch.cuda.synchronize()
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attention_decode_noalloc(q, kc, vc, bt, cl, max_len, D ** -0.5, out)
    assert e.value.status == pkv.PKV_ERR_WORKSPACE
    assert pkv.lib().pkv_status_string(e.value.status) == b"workspace missing or too small"
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
    assert pkv.pkv_device_status() == 0
