"""Cascade decode over a shared prefix against the oracle (GPU).

The oracle knows nothing of the cascade: it attends each sequence's whole
context through its block table, so these tests check that reading the
shared prefix once for all sharers changes nothing but the reads."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_211_gb300 as pkv
from paged_kv_cache_211_gb300 import workloads as wl
from gpu_helpers import assert_attention_close, compact_oracle_step, dtype_code
from pkv_testutil import bits

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    pkv.pkv_device_status(reset=True)


def test_cascade_step_on_prefix_shared_workload(cuda_device):
    w = wl.WORKLOADS["prefix_shared"]
    inp = wl.make_inputs(w, device=cuda_device, num_layers=1)
    lens = inp["context_lens_host"]
    ids = np.arange(w.num_seqs)                 # every sequence
    want, kn_rows, _ = compact_oracle_step(inp, ids)
    max_len = int(lens.max())
    out = torch.empty_like(inp["q"])
    ws = pkv.new_cascade_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len,
                                   w.prefix_blocks, cuda_device)
    slots = torch.empty(w.num_seqs, dtype=torch.int64, device=cuda_device)
    pkv.paged_kv_decode_step_cascade(inp["q"], inp["k_new"][0], inp["v_new"][0],
                                     inp["k_cache"][0], inp["v_cache"][0], inp["block_tables"],
                                     inp["context_lens"], max_len, w.prefix_blocks, w.scale, out,
                                     ws, slot_mapping_out=slots)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    want_slots = oracle.slot_mapping(inp["block_tables_host"], lens, 16, w.num_blocks)
    assert np.array_equal(slots.cpu().numpy(), want_slots)
    assert_attention_close(bits(out)[ids], want, dtype_code(w), "cascade step")
    # the plain path on the (now written) cache agrees with the cascade
    ref = torch.empty_like(out)
    ws2 = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, cuda_device)
    pkv.paged_attention_decode(inp["q"], inp["k_cache"][0], inp["v_cache"][0],
                               inp["block_tables"], inp["context_lens"], max_len, w.scale, ref,
                               ws2)
    torch.cuda.synchronize()
    assert torch.allclose(out.float(), ref.float(), atol=1e-2, rtol=1e-2)


def _shared_case(dev, dtype, lens, P, Hq, Hkv, D, seed):
    """Sequences whose tables all start with the same P full blocks; the rest
    of each context in private blocks; NaN in every slot past a sequence's
    own length outside the shared prefix."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    MB = max(P, max((n + 15) // 16 for n in lens))
    need_private = [max(0, (n + 15) // 16 - P) for n in lens]
    NB = P + sum(need_private) + 4
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, MB), perm[-1], np.int32)
    pos = P
    for s in range(B):
        tables[s, :P] = perm[:P]
        tables[s, P:P + need_private[s]] = perm[pos:pos + need_private[s]]
        pos += need_private[s]
    g = torch.Generator(device=dev).manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float16
    rnd = lambda *sh: torch.randn(*sh, generator=g, device=dev).to(dt)
    kc, vc, q = rnd(NB, 16, Hkv, D), rnd(NB, 16, Hkv, D), rnd(B, Hq, D)
    for s, n in enumerate(lens):            # poison private slots past each length
        for t in range(max(n, 16 * P), 16 * ((max(n, 16 * P) + 15) // 16)):
            b = int(tables[s, t // 16])
            kc[b, t % 16] = float("nan")
            vc[b, t % 16] = float("nan")
    return (torch.from_numpy(tables).to(dev), torch.tensor(lens, dtype=torch.int32, device=dev),
            tables, np.array(lens, np.int32), kc, vc, q)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B", [("bf16", 16, 8, 128, 14), ("f16", 32, 4, 64, 14),
                                               ("bf16", 8, 8, 128, 14), ("f16", 12, 4, 128, 14),
                                               ("bf16", 24, 8, 128, 50),
                                               ("f16", 32, 16, 64, 14)])  # register-pipelined pass
def test_cascade_attention_short_and_long_sequences(dtype, Hq, Hkv, D, B, cuda_device):
    """Sequences shorter than, equal to and longer than a 192-token prefix (12
    blocks: one full and one half key tile of the prefix pass); with B = 50 and
    3 query heads per KV head, 150 rows per KV head: two row tiles, the second
    partly empty.  16 KV heads take the register-pipelined partition pass,
    which waits for the prefix pass instead of running beside it."""
    P = 12
    base = [1, 5, 16, 100, 191, 192, 193, 250, 700, 1000, 64, 300, 2, 193]
    lens = [base[i % len(base)] + (i // len(base)) * 37 for i in range(B)]
    bt, cl, tables, ln, kc, vc, q = _shared_case(cuda_device, dtype, lens, P, Hq, Hkv, D, 17)
    code = oracle.BF16 if dtype == "bf16" else oracle.F16
    want = oracle.decode_attention(code, bits(q), bits(kc), bits(vc), tables, ln, D ** -0.5)
    out = torch.empty_like(q)
    ws = pkv.new_cascade_workspace(len(lens), Hq, D, max(lens), P, cuda_device)
    pkv.paged_attention_decode_cascade(q, kc, vc, bt, cl, max(lens), P, D ** -0.5, out, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    assert_attention_close(bits(out), want, code, f"cascade g={Hq // Hkv} D={D}")


def test_cascade_step_refuses_a_token_inside_the_prefix(cuda_device):
    P = 4
    lens = [64, 65, 200]                                # the first one's token is in block 3 < P
    bt, cl, tables, ln, kc, vc, q = _shared_case(cuda_device, "bf16", lens, P, 8, 8, 128, 5)
    kn = torch.randn(3, 8, 128, device=cuda_device).to(torch.bfloat16)
    vn = torch.randn(3, 8, 128, device=cuda_device).to(torch.bfloat16)
    k_before = kc.clone()
    out = torch.empty_like(q)
    ws = pkv.new_cascade_workspace(3, 8, 128, 200, P, cuda_device)
    slots = torch.empty(3, dtype=torch.int64, device=cuda_device)
    pkv.paged_kv_decode_step_cascade(q, kn, vn, kc, vc, bt, cl, 200, P, 128 ** -0.5, out, ws,
                                     slot_mapping_out=slots)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(reset=True) & pkv.DEV_BAD_LENGTH
    assert int(slots[0]) == -1
    assert torch.equal(kc[tables[0, 3]].view(torch.int16), k_before[tables[0, 3]].view(torch.int16))
    assert int(slots[1]) == int(tables[1, 4]) * 16 and int(slots[2]) >= 0


@pytest.mark.parametrize("switch", [{"PKV_WARP_ITEMS": "1"}, {"PKV_WARP_ITEMS": "0"},
                                    {"PKV_STREAM_FEED": "0"}],
                         ids=["even_stream_producer", "items", "even_self_feeding"])
def test_cascade_suffix_splits_in_child(switch, cuda_device):
    """The suffix pass split evenly over the consumer warps (the default when
    the workspace holds the slots) with its rings filled by the stream
    producer, the same split with self-feeding warps (PKV_STREAM_FEED=0), and
    dealt as items (PKV_WARP_ITEMS=0), on the same cases: 128 and 50
    sequences, lengths inside, at and past the prefix."""
    env = dict(os.environ, **switch)
    env["PYTHONPATH"] = os.pathsep.join([HERE, os.path.dirname(HERE), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.join(HERE, "cascade_case_check.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "ok" in r.stdout
