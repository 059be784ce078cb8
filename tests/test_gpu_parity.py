"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Cache writes and slot mapping are compared bit for bit; decode attention
within the stated tolerance (elementwise max(4e-3, 1e-2 |oracle|), and
1e-2 relative to the largest |oracle|).  Every workload runs in the launch
configuration the benchmark times (paged_kv_decode_step with the adaptive
partitioning), and the oracle checks every sequence of every workload (its
work is spread over the host cores by sequence).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_211_gb300 as pkv
from paged_kv_cache_211_gb300 import workloads as wl
from gpu_helpers import (assert_attention_close, compact_oracle_step, dtype_code,
                         oracle_steps, sample_seqs)
from pkv_testutil import bits

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    pkv.pkv_device_status(reset=True)


def _run_step(inp, dev):
    w = inp["workload"]
    q, kc, vc = inp["q"], inp["k_cache"][0], inp["v_cache"][0]
    max_len = int(inp["context_lens_host"].max())
    out = torch.empty_like(q)
    ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, dev)
    slots = torch.full((w.num_seqs,), -7, dtype=torch.int64, device=dev)
    pkv.paged_kv_decode_step(q, inp["k_new"][0], inp["v_new"][0], kc, vc, inp["block_tables"],
                             inp["context_lens"], max_len, w.scale, out, ws,
                             slot_mapping_out=slots)
    torch.cuda.synchronize()
    return out, slots


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_decode_step_parity(name, cuda_device):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, device=cuda_device, num_layers=1)
    lens, tables = inp["context_lens_host"], inp["block_tables_host"]
    k_orig, v_orig = inp["k_cache"][0].clone(), inp["v_cache"][0].clone()
    seq_ids = np.arange(w.num_seqs)
    want, kn_rows, vn_rows = compact_oracle_step(inp, seq_ids)   # before the GPU touches anything

    out, slots = _run_step(inp, cuda_device)
    assert pkv.pkv_device_status() == 0

    # block-table plumbing: bit-exact against the oracle on the full tables
    want_slots = oracle.slot_mapping(tables, lens, 16, w.num_blocks)
    assert np.array_equal(slots.cpu().numpy(), want_slots)

    # KV write: the written rows equal the oracle's, every other byte is unchanged
    kc, vc = inp["k_cache"][0], inp["v_cache"][0]
    flat = lambda t: t.view(-1, w.num_kv_heads, w.head_dim)
    sl = torch.from_numpy(want_slots).to(cuda_device)
    sel = torch.from_numpy(seq_ids).to(cuda_device)
    assert np.array_equal(bits(flat(kc)[sl][sel]), kn_rows)
    assert np.array_equal(bits(flat(vc)[sl][sel]), vn_rows)
    keep = torch.ones(w.num_blocks * 16, dtype=torch.bool, device=cuda_device)
    keep[sl] = False
    assert torch.equal(flat(kc)[keep].view(torch.int16), flat(k_orig)[keep].view(torch.int16))
    assert torch.equal(flat(vc)[keep].view(torch.int16), flat(v_orig)[keep].view(torch.int16))

    # attention
    got = bits(out)[seq_ids]
    err, rel = assert_attention_close(got, want, dtype_code(w), name)
    print(f"{name}: {len(seq_ids)} seqs checked, max abs err {err:.2e}, norm-rel {rel:.2e}")


@pytest.mark.parametrize("name", ["tiny", "qwen3_0p6b"])
def test_separate_entry_points(name, cuda_device):
    """reshape_and_cache + paged_attention_decode called one by one."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, device=cuda_device, num_layers=1)
    want, _, _ = compact_oracle_step(inp, np.arange(w.num_seqs))
    kc, vc = inp["k_cache"][0], inp["v_cache"][0]
    slots = pkv.paged_kv_slot_mapping(inp["block_tables"], inp["context_lens"], w.num_blocks)
    pkv.reshape_and_cache(inp["k_new"][0], inp["v_new"][0], kc, vc, slots)
    max_len = int(inp["context_lens_host"].max())
    out = torch.empty_like(inp["q"])
    ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, cuda_device)
    pkv.paged_attention_decode(inp["q"], kc, vc, inp["block_tables"], inp["context_lens"],
                               max_len, w.scale, out, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    assert_attention_close(bits(out), want, dtype_code(w), name)


@pytest.mark.parametrize("name", ["tiny", "qwen3_0p6b", "prefix_shared"])
def test_partition_length_invariance(name, cuda_device):
    """Partitions of 1, 2, 4, 32 blocks and one partition per sequence all match the
    oracle, and each other within fp32 rounding."""
    w = wl.WORKLOADS[name]
    if name == "prefix_shared":
        w = w.with_(num_seqs=24)
    inp = wl.make_inputs(w, device=cuda_device, num_layers=1)
    want, _, _ = compact_oracle_step(inp, np.arange(w.num_seqs))
    kc, vc = inp["k_cache"][0], inp["v_cache"][0]
    slots = pkv.paged_kv_slot_mapping(inp["block_tables"], inp["context_lens"], w.num_blocks)
    pkv.reshape_and_cache(inp["k_new"][0], inp["v_new"][0], kc, vc, slots)
    max_len = int(inp["context_lens_host"].max())
    ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, cuda_device)
    outs = {}
    min_pb = pkv.paged_attention_min_partition_blocks(max_len)
    for pb in sorted({max(min_pb, x) for x in (1, 2, 4, 32, w.max_blocks_per_seq)}):
        out = torch.empty_like(inp["q"])
        pkv.paged_attention_decode_partitioned(inp["q"], kc, vc, inp["block_tables"],
                                               inp["context_lens"], max_len, w.scale, out, ws,
                                               partition_blocks=pb)
        torch.cuda.synchronize()
        outs[pb] = out.float()
        assert_attention_close(bits(out), want, dtype_code(w), f"{name} pb={pb}")
    ref = outs[w.max_blocks_per_seq]
    for pb, o in outs.items():
        assert torch.allclose(o, ref, atol=2e-2, rtol=2e-2), pb
    assert pkv.pkv_device_status() == 0


def _custom(dev, dtype, lens, Hq, Hkv, D, NB, seed, poison=True, table_blocks=None):
    w = wl.Workload("custom", seed, len(lens), Hq, Hkv, D, NB, dtype,
                    "fixed:" + ",".join(str(n) for n in lens),
                    table_blocks or max(1, (max(lens) + 15) // 16))
    return w, wl.make_inputs(w, device=dev, num_layers=1, poison=poison)


@pytest.mark.parametrize("dtype,Hkv,D", [("bf16", 8, 128), ("f16", 2, 128), ("bf16", 4, 64)])
def test_even_split_edge_cases(dtype, Hkv, D, cuda_device):
    """The adaptive pass cuts the (sequence, head group, block) units evenly over
    the CTAs: fewer units than CTAs (a wide table and a large length bound, so
    most CTAs get nothing and a sequence's pieces sit in CTAs with empty ones
    between them), empty sequences, and one long sequence cut across many CTAs
    among short ones."""
    cases = (([17, 0, 5, 1, 300], 4096, 256),
             ([3000] + [1 + (7 * i) % 40 for i in range(50)], 3000, None))
    for k, (lens, bound, tb) in enumerate(cases):
        w, inp = _custom(cuda_device, dtype, lens, 4 * Hkv, Hkv, D, 600, seed=90 + k,
                         table_blocks=tb)
        keep = np.array([i for i, n in enumerate(lens) if n > 0])
        empty = [i for i, n in enumerate(lens) if n == 0]
        want, _, _ = compact_oracle_step(inp, keep)
        q = inp["q"]
        out = torch.full_like(q, float("nan"))
        ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, bound, cuda_device)
        pkv.paged_kv_decode_step(q, inp["k_new"][0], inp["v_new"][0], inp["k_cache"][0],
                                 inp["v_cache"][0], inp["block_tables"], inp["context_lens"],
                                 bound, w.scale, out, ws)
        torch.cuda.synchronize()
        assert pkv.pkv_device_status() == 0
        for i in empty:
            assert torch.count_nonzero(out[i]) == 0
        assert_attention_close(bits(out)[keep], want, dtype_code(w), f"case {k}")


@pytest.mark.parametrize("dtype,Hq,Hkv,D,lens", [("bf16", 8, 2, 128, [32768]),
                                                  ("f16", 4, 1, 64, [30000, 100])])
def test_even_split_segment_over_many_ctas(dtype, Hq, Hkv, D, lens, cuda_device):
    """A (sequence, head group) cut across far more than 32 CTAs (76 and about
    150 pieces): the merge reads row i < 32 in lane i and the rest in further
    rounds."""
    NB = sum((n + 15) // 16 for n in lens) + 8
    w, inp = _custom(cuda_device, dtype, lens, Hq, Hkv, D, NB, seed=len(lens) + Hkv)
    want, _, _ = compact_oracle_step(inp, np.arange(len(lens)))
    out, _ = _run_step(inp, cuda_device)
    assert pkv.pkv_device_status() == 0
    assert_attention_close(bits(out), want, dtype_code(w), f"{lens[0]} tokens, Hkv={Hkv}")


@pytest.mark.parametrize("dtype,Hq,Hkv,D", [("bf16", 8, 8, 128), ("f16", 8, 1, 64),
                                             ("bf16", 16, 4, 64), ("f16", 6, 3, 128),
                                             ("bf16", 14, 2, 128)])
def test_group_sizes_and_ragged_lengths(dtype, Hq, Hkv, D, cuda_device):
    """MHA (g=1), g=3, 4, 7, 8, D 64/128, lengths on and around block boundaries."""
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 1000]
    w, inp = _custom(cuda_device, dtype, lens, Hq, Hkv, D, 256, seed=77)
    want, _, _ = compact_oracle_step(inp, np.arange(len(lens)))
    out, _ = _run_step(inp, cuda_device)
    assert pkv.pkv_device_status() == 0
    assert_attention_close(bits(out), want, dtype_code(w), f"g={Hq // Hkv} D={D}")


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B", [("bf16", 32, 8, 128, 160), ("f16", 32, 4, 64, 200),
                                               ("bf16", 8, 8, 128, 96)])
def test_warp_items(dtype, Hq, Hkv, D, B, cuda_device):
    """Many short one-head items (at least half an item per consumer warp of
    the grid, contexts under 64 blocks): each consumer warp takes whole items
    of its own.  Lengths span empty, one token, block boundaries and 1000
    tokens, so some sequences stay whole and others are cut and merged."""
    rng = np.random.default_rng(1000 + B)
    lens = rng.integers(1, 1001, size=B)
    lens[:6] = [0, 1, 16, 17, 1000, 999]
    w, inp = _custom(cuda_device, dtype, [int(n) for n in lens], Hq, Hkv, D,
                     int((lens + 15).sum() // 16) + 64, seed=B)
    keep = np.flatnonzero(lens > 0)
    want, _, _ = compact_oracle_step(inp, keep)
    out, slots = _run_step(inp, cuda_device)
    assert pkv.pkv_device_status() == 0
    assert int(slots[0]) == -1
    assert torch.count_nonzero(out[0]) == 0
    assert_attention_close(bits(out)[keep], want, dtype_code(w), f"B={B} g={Hq // Hkv} D={D}")


def test_length_one_returns_v_exactly(cuda_device):
    w, inp = _custom(cuda_device, "bf16", [1, 1, 1], 8, 2, 128, 8, seed=5)
    out, _ = _run_step(inp, cuda_device)
    # out[s, i] == the new token's V row of KV head i // 4, bit for bit
    want = inp["v_new"][0].repeat_interleave(4, dim=1)
    assert torch.equal(out.view(torch.int16), want.view(torch.int16))


def test_empty_context_gives_zeros(cuda_device):
    w, inp = _custom(cuda_device, "f16", [5, 40, 7], 8, 4, 128, 16, seed=6)
    inp["context_lens"][1] = 0           # a padding row
    lens = inp["context_lens_host"].copy()
    lens[1] = 0
    inp["context_lens_host"] = lens
    keep = np.array([0, 2])
    want, _, _ = compact_oracle_step(inp, keep)
    out, slots = _run_step(inp, cuda_device)
    assert pkv.pkv_device_status() == 0
    assert int(slots[1]) == -1
    assert torch.count_nonzero(out[1]) == 0
    assert_attention_close(bits(out)[keep], want, oracle.F16, "non-empty rows")


def test_bad_device_values_are_flagged_not_read(cuda_device):
    """A table entry outside the pool and a length beyond the bound are skipped and
    flagged in the device status word; the other rows stay correct."""
    w, inp = _custom(cuda_device, "bf16", [40, 40, 40], 8, 4, 128, 16, seed=8)
    want, _, _ = compact_oracle_step(inp, np.array([0]))
    q, kc, vc = inp["q"], inp["k_cache"][0], inp["v_cache"][0]
    slots = pkv.paged_kv_slot_mapping(inp["block_tables"], inp["context_lens"], w.num_blocks)
    pkv.reshape_and_cache(inp["k_new"][0], inp["v_new"][0], kc, vc, slots)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    inp["block_tables"][1, 1] = 1 << 30          # out of range
    inp["context_lens"][2] = 999                 # beyond max_context_len and the table
    max_len = 40
    out = torch.empty_like(q)
    ws = pkv.new_workspace(3, 8, 128, max_len, cuda_device)
    pkv.paged_attention_decode(q, kc, vc, inp["block_tables"], inp["context_lens"], max_len,
                               w.scale, out, ws)
    torch.cuda.synchronize()
    flags = pkv.pkv_device_status(reset=False)
    assert flags & pkv.DEV_BAD_BLOCK_ID and flags & pkv.DEV_BAD_LENGTH
    assert pkv.paged_kv_last_error() == 4        # PKV_ERR_BAD_BLOCK_ID; clears the word
    assert pkv.paged_kv_last_error() == 0
    assert torch.isfinite(out.float()).all()
    assert torch.count_nonzero(out[2]) == 0      # an invalid length gives a zero row
    assert_attention_close(bits(out)[:1], want, oracle.BF16, "row without bad values")
    assert pkv.pkv_device_status() == 0


def test_reshape_and_cache_padding_and_bad_slots(cuda_device):
    NB, Hkv, D = 12, 8, 128
    g = torch.Generator(device=cuda_device).manual_seed(3)
    kc = torch.randn(NB, 16, Hkv, D, generator=g, device=cuda_device).to(torch.float16)
    vc = torch.randn(NB, 16, Hkv, D, generator=g, device=cuda_device).to(torch.float16)
    kn = torch.randn(5, Hkv, D, generator=g, device=cuda_device).to(torch.float16)
    vn = torch.randn(5, Hkv, D, generator=g, device=cuda_device).to(torch.float16)
    slots = torch.tensor([3, -1, 191, 17, NB * 16 + 5], dtype=torch.int64, device=cuda_device)
    hk, hv = bits(kc), bits(vc)
    wk, wv = oracle.reshape_and_cache(bits(kn)[[0, 2, 3]], bits(vn)[[0, 2, 3]], hk, hv,
                                      np.array([3, 191, 17]))
    pkv.reshape_and_cache(kn, vn, kc, vc, slots)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(reset=False) == pkv.DEV_BAD_SLOT
    assert pkv.paged_kv_last_error() == 1        # PKV_ERR_INVALID_ARG
    assert np.array_equal(bits(kc), wk) and np.array_equal(bits(vc), wv)


def test_maximum_batch_and_maximum_length(cuda_device):
    """8192 sequences (lengths and offsets fill 64 KB of shared memory) and two
    32768-token contexts (64 partitions of the minimum length)."""
    rng = np.random.default_rng(9)
    lens = [int(x) for x in rng.integers(1, 40, size=8192)]
    w, inp = _custom(cuda_device, "f16", lens, 4, 2, 64, 8192 * 3 + 8, seed=10)
    ids = sample_seqs(np.array(lens), 64, seed=1)
    want, _, _ = compact_oracle_step(inp, ids)
    out, _ = _run_step(inp, cuda_device)
    assert pkv.pkv_device_status() == 0
    assert_attention_close(bits(out)[ids], want, oracle.F16, "8192 seqs")

    w, inp = _custom(cuda_device, "bf16", [32768, 32768], 32, 8, 128, 4100, seed=11)
    want, _, _ = compact_oracle_step(inp, np.arange(2))
    out, _ = _run_step(inp, cuda_device)
    assert pkv.pkv_device_status() == 0
    assert_attention_close(bits(out), want, oracle.BF16, "32768 tokens")


def _two_steps(inp, dev, seed):
    """Two consecutive decode steps of the workload's sequences: the first at
    lengths n - 1 (its token at position n - 2), the second at n (the
    workload's own token position), each with fresh q and new K/V rows."""
    w = inp["workload"]
    lens2 = inp["context_lens_host"].astype(np.int32)
    lens1 = np.maximum(lens2 - 1, 0).astype(np.int32)
    g = torch.Generator(device=dev).manual_seed(seed)
    dt = inp["q"].dtype
    rnd = lambda *sh: torch.randn(*sh, generator=g, device=dev).to(dt)
    B, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    steps = []
    for ln in (lens1, lens2):
        steps.append(dict(q=rnd(B, Hq, D), k_new=rnd(B, Hkv, D), v_new=rnd(B, Hkv, D),
                          lens=ln, cl=torch.from_numpy(ln).to(dev)))
    return steps


def _host_steps(inp, steps, dev):
    """Runs the steps back to back through paged_kv_decode_step_host, each from
    its own pinned host buffers into its own pinned output; returns the outputs."""
    w = inp["workload"]
    pin = lambda t: t.cpu().pin_memory()
    max_len = int(max(int(st["lens"].max()) for st in steps))
    staging = torch.empty(pkv.paged_kv_decode_step_staging_bytes(w.num_seqs, w.num_q_heads,
                                                                 w.num_kv_heads, w.head_dim,
                                                                 w.max_blocks_per_seq),
                          dtype=torch.uint8, device=dev)
    ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, dev)
    bth = pin(inp["block_tables"])
    host = [dict(q=pin(st["q"]), kn=pin(st["k_new"]), vn=pin(st["v_new"]), cl=pin(st["cl"]))
            for st in steps]
    outs = [torch.full_like(h["q"], float("nan")).pin_memory() for h in host]
    torch.cuda.synchronize()
    for h, o in zip(host, outs):
        pkv.paged_kv_decode_step_host(h["q"], h["kn"], h["vn"], bth, h["cl"], o, staging,
                                      inp["k_cache"][0], inp["v_cache"][0], max_len, w.scale,
                                      ws)
    torch.cuda.current_stream().synchronize()
    return outs


@pytest.mark.parametrize("name", ["tiny", "qwen3_0p6b", "llama7b_long", "hkv16"])
def test_host_buffer_steps_back_to_back(name, cuda_device):
    """paged_kv_decode_step_host, the entry the end-to-end number times: two
    steps enqueued back to back (the second one's staging kernel follows the
    first one's kernels on the stream), inputs and outputs in pinned host
    memory, both outputs and the cache writes against the oracle, every
    sequence.  hkv16 has 16 KV heads, which the register-pipelined partition
    pass serves, with short contexts and no merge pass."""
    if name == "hkv16":
        w, inp = _custom(cuda_device, "f16", [17, 40, 5, 100, 64, 33, 2, 90], 32, 16, 64, 96,
                         seed=61)
    else:
        inp = wl.make_inputs(wl.WORKLOADS[name], device=cuda_device, num_layers=1)
        w = inp["workload"]
    steps = _two_steps(inp, cuda_device, seed=w.seed + 5)
    hsteps = [dict(q=bits(st["q"]), k_new=bits(st["k_new"]), v_new=bits(st["v_new"]),
                   lens=st["lens"]) for st in steps]
    seq_ids = np.arange(w.num_seqs)
    want1, want2 = oracle_steps(inp, seq_ids, hsteps)   # before the GPU touches anything
    out1, out2 = _host_steps(inp, steps, cuda_device)
    assert pkv.pkv_device_status() == 0
    code = dtype_code(w)
    assert_attention_close(bits(out1), want1, code, f"{name} step 1")
    assert_attention_close(bits(out2), want2, code, f"{name} step 2")
    rows = lambda t: t.view(-1, w.num_kv_heads, w.head_dim)
    for st, hs in zip(steps, hsteps):
        sl = oracle.slot_mapping(inp["block_tables_host"], st["lens"], 16, w.num_blocks)
        live = sl >= 0
        idx = torch.from_numpy(sl[live]).to(cuda_device)
        assert np.array_equal(bits(rows(inp["k_cache"][0])[idx]), hs["k_new"][live])
        assert np.array_equal(bits(rows(inp["v_cache"][0])[idx]), hs["v_new"][live])


def test_step_after_a_kernel_that_rewrites_lengths_and_tables(cuda_device):
    """A decode step right after a kernel that rewrites context_lens and
    block_tables on the same stream (a scheduler's per-step update): the step
    must use the new values.  Each sequence grows by one token and four of
    them cross into a block that the update kernel has just entered in the
    table (the entry named a poisoned block before).  Repeated with a long
    and a short context mix."""
    for k, lens in enumerate(([1500, 2100, 33, 700, 16, 32, 48, 6000],
                              [17, 64, 100, 31, 16, 32, 48, 80])):
        lens2 = [n + 1 for n in lens]
        w, inp = _custom(cuda_device, "bf16", lens2, 32, 8, 128, 1200, seed=81 + k)
        tables = inp["block_tables_host"]
        dev = cuda_device
        B = len(lens)
        # before the update, a sequence whose new token opens a block has that
        # table entry pointing at a poisoned block
        stale = tables.copy()
        for s, n in enumerate(lens):
            if n % 16 == 0:
                stale[s, n // 16] = inp["poison_block"]
        bt = torch.from_numpy(stale).to(dev)
        cl = torch.tensor(lens, dtype=torch.int32, device=dev)
        fresh_rows = torch.from_numpy(tables).to(dev)
        step = dict(q=bits(inp["q"]), k_new=bits(inp["k_new"][0]), v_new=bits(inp["v_new"][0]),
                    lens=np.array(lens2, np.int32))
        want = oracle_steps(inp, np.arange(B), [step])[0]
        max_len = max(lens2)
        ws = pkv.new_workspace(B, 32, 128, max_len, dev)
        out = torch.empty_like(inp["q"])
        torch.cuda.synchronize()
        for _ in range(3):       # a few spins of the same update + step
            bt.copy_(torch.from_numpy(stale).to(dev))
            cl.fill_(0)
            torch.cuda.synchronize()
            # the update: kernels on the stream right before the step
            cl.copy_(cl.new_tensor(lens))
            cl.add_(1)
            bt.mul_(0).add_(fresh_rows)
            pkv.paged_kv_decode_step(inp["q"], inp["k_new"][0], inp["v_new"][0],
                                     inp["k_cache"][0], inp["v_cache"][0], bt, cl, max_len,
                                     w.scale, out, ws)
            torch.cuda.synchronize()
            assert pkv.pkv_device_status() == 0
            assert_attention_close(bits(out), want, oracle.BF16, f"mix {k}")


def test_layer_views_of_a_layer_major_pool(cuda_device):
    """Each layer of a layer-major pool is addressed by its own base pointer (a view)."""
    w = wl.WORKLOADS["tiny"]
    inp = wl.make_inputs(w, device=cuda_device, num_layers=3)
    max_len = int(inp["context_lens_host"].max())
    ws = pkv.new_workspace(w.num_seqs, w.num_q_heads, w.head_dim, max_len, cuda_device)
    for layer in (2, 0, 1):
        want, _, _ = compact_oracle_step(inp, np.arange(w.num_seqs), layer=layer)
        out = torch.empty_like(inp["q"])
        pkv.paged_kv_decode_step(inp["q"], inp["k_new"][layer], inp["v_new"][layer],
                                 inp["k_cache"][layer], inp["v_cache"][layer],
                                 inp["block_tables"], inp["context_lens"], max_len, w.scale,
                                 out, ws)
        torch.cuda.synchronize()
        assert_attention_close(bits(out), want, oracle.F16, f"layer {layer}")
    assert pkv.pkv_device_status() == 0


@pytest.mark.parametrize("dtype,Hq,Hkv,D,lens", [
    ("bf16", 32, 8, 128, [1500, 2100, 33, 700]),     # long: partitions and a merge per step
    ("f16", 16, 8, 128, [17, 64, 100, 31]),          # short: no merge
])
def test_consecutive_steps_see_the_previous_token(dtype, Hq, Hkv, D, lens, cuda_device):
    """Two decode steps enqueued back to back, as a decoder runs them: the
    second step's partition pass may start while the first step's merge still
    runs, and its context includes the token the first step wrote."""
    lens2 = [n + 1 for n in lens]
    w, inp = _custom(cuda_device, dtype, lens2, Hq, Hkv, D, 512, seed=71)
    tables = inp["block_tables_host"]
    dev = cuda_device
    g = torch.Generator(device=dev).manual_seed(72)
    dt = inp["q"].dtype
    rnd = lambda *sh: torch.randn(*sh, generator=g, device=dev).to(dt)
    B = len(lens)
    q1, q2 = rnd(B, Hq, D), rnd(B, Hq, D)
    kn1, vn1, kn2, vn2 = rnd(B, Hkv, D), rnd(B, Hkv, D), rnd(B, Hkv, D), rnd(B, Hkv, D)
    cl1 = torch.tensor(lens, dtype=torch.int32, device=dev)
    cl2 = torch.tensor(lens2, dtype=torch.int32, device=dev)
    kc, vc = inp["k_cache"][0], inp["v_cache"][0]
    hk, hv = bits(kc), bits(vc)                        # the pools before either step
    max_len = max(lens2)
    ws = pkv.new_workspace(B, Hq, D, max_len, dev)
    out1, out2 = torch.empty_like(q1), torch.empty_like(q2)
    torch.cuda.synchronize()
    pkv.paged_kv_decode_step(q1, kn1, vn1, kc, vc, inp["block_tables"], cl1, max_len, w.scale,
                             out1, ws)
    pkv.paged_kv_decode_step(q2, kn2, vn2, kc, vc, inp["block_tables"], cl2, max_len, w.scale,
                             out2, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    code = dtype_code(w)
    nb = w.num_blocks
    s1 = oracle.slot_mapping(tables, np.array(lens, np.int32), 16, nb)
    hk, hv = oracle.reshape_and_cache(bits(kn1), bits(vn1), hk, hv, s1)
    s2 = oracle.slot_mapping(tables, np.array(lens2, np.int32), 16, nb)
    hk, hv = oracle.reshape_and_cache(bits(kn2), bits(vn2), hk, hv, s2)
    want = oracle.decode_attention(code, bits(q2), hk, hv, tables, np.array(lens2, np.int32),
                                   w.scale)
    assert_attention_close(bits(out2), want, code, "second step")
    assert np.array_equal(bits(kc).reshape(-1, Hkv, D)[s1], bits(kn1))
    assert np.array_equal(bits(kc).reshape(-1, Hkv, D)[s2], bits(kn2))


def test_bounded_wait_gives_up_and_reports(cuda_device):
    """A kernel waiting on an mbarrier that nothing arrives on gives up after its
    bound (~0.1 s here), flags PKV_DEV_TIMEOUT and returns; the context stays
    usable for the next call."""
    pkv.pkv_device_status(reset=True)
    pkv.pkv_selftest_bounded_wait()
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(reset=True) & pkv.DEV_TIMEOUT
    w, inp = _custom(cuda_device, "bf16", [40, 17, 300], 8, 4, 128, 64, seed=9)
    want, _, _ = compact_oracle_step(inp, np.arange(3))
    out, _ = _run_step(inp, cuda_device)
    assert pkv.pkv_device_status() == 0
    assert_attention_close(bits(out), want, oracle.BF16, "after a timed-out wait")


@pytest.mark.parametrize("wide", ["1", "0"])
def test_long_context_builds_in_child(wide, cuda_device):
    """The one-head producer-warp pass in 12 warps (the default: setmaxnreg
    hands the producer warpgroup's registers to the consumers) and in nine
    (PKV_WIDE=0), each in a child process, against the oracle."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PKV_WIDE=wide)
    env["PYTHONPATH"] = os.pathsep.join([here, os.path.dirname(here), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.join(here, "decode_case_check.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "ok" in r.stdout
