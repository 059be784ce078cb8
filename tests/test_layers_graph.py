"""The multi-layer decode step (one call for every layer of a layer-major
stack) against the oracle, and the same call captured in a CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_211_gb300 as pkv
from paged_kv_cache_211_gb300 import workloads as wl
from gpu_helpers import assert_attention_close, dtype_code
from pkv_testutil import bits

pytestmark = pytest.mark.gpu


def _oracle_layer(inp, layer):
    w = inp["workload"]
    h_q = bits(inp["q_layers"][layer])
    kc, vc = bits(inp["k_cache"][layer]), bits(inp["v_cache"][layer])
    tb, ln = inp["block_tables_host"], inp["context_lens_host"]
    slots = oracle.slot_mapping(tb, ln, 16, w.num_blocks)
    kc, vc = oracle.reshape_and_cache(bits(inp["k_new"][layer]), bits(inp["v_new"][layer]), kc,
                                      vc, slots)
    return oracle.decode_attention(dtype_code(w), h_q, kc, vc, tb, ln, w.scale)


# Each later layer's partition pass runs beside the previous layer's merge
# and waits for it only before its first workspace write: short contexts
# (items of whole or cut sequences, shared by the consumer warps or, with many
# sequences, taken whole by one warp each) and long ones (the even split, at
# D = 128 and at D = 64 with two heads per consumer).
CASES = [
    ("qwen3_0p6b", 4, {}),
    ("tiny", 3, {}),   # no merge: each layer's pass follows the previous layer's pass
    ("llama7b_long", 3, dict(num_seqs=4, num_blocks=8200)),
    ("tinyllama_1p1b", 3, dict(num_seqs=24, num_blocks=3200)),
    ("qwen3_0p6b", 3, dict(num_seqs=160)),   # consumer warps take whole items
    # 16 KV heads: the register-pipelined pass, which waits for the previous
    # layer's merge before it reads anything
    ("qwen3_0p6b", 3, dict(num_seqs=24, num_q_heads=32, num_kv_heads=16)),
]


@pytest.mark.parametrize("name,L,kw", CASES,
                         ids=[c[0] + "".join("_%s%d" % (k[4] if k.startswith("num_") else k[0], v)
                                             for k, v in c[2].items()) for c in CASES])
def test_layers_step_eager_and_graph(cuda_device, name, L, kw):
    import __graft_entry__
    __graft_entry__.build()
    w = wl.WORKLOADS[name].with_(**kw)
    inp = wl.make_inputs(w, device=cuda_device, num_layers=L)
    want = [_oracle_layer(inp, l) for l in range(L)]        # before the GPU writes anything
    max_len = int(inp["context_lens_host"].max())
    q = inp["q_layers"].contiguous()
    out = torch.empty_like(q)
    ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, cuda_device)
    args = (q, inp["k_new"], inp["v_new"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
            inp["context_lens"], max_len, w.scale)
    pkv.paged_kv_decode_step_layers(*args, out, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    for l in range(L):
        assert_attention_close(bits(out[l]), want[l], dtype_code(w), f"layer {l}")

    # capture the same step into a CUDA graph and replay it: identical results
    eager = out.clone()
    out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            pkv.paged_kv_decode_step_layers(*args, out, ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert pkv.pkv_device_status() == 0
