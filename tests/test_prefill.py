"""Chunked-prefill attention over the paged cache against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_211_gb300 as pkv
from gpu_helpers import assert_attention_close
from pkv_testutil import bits, token_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    pkv.pkv_device_status(reset=True)


def _case(dev, dtype, specs, Hq, Hkv, D, seed):
    """specs: (context_len n, chunk rows q_len) per sequence; the chunk is the
    last q_len tokens.  Slots past n are NaN; the chunk's slots start as NaN
    and are written with the chunk's K/V before attention."""
    rng = np.random.default_rng(seed)
    B = len(specs)
    need = [(n + 15) // 16 for n, _ in specs]
    MB, NB = max(need), sum(need) + 3
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, MB), perm[-1], np.int32)
    pos = 0
    for s, nb in enumerate(need):
        tables[s, :nb] = perm[pos:pos + nb]
        pos += nb
    g = torch.Generator(device=dev).manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float16
    rnd = lambda *sh: torch.randn(*sh, generator=g, device=dev).to(dt)
    kc, vc = rnd(NB, 16, Hkv, D), rnd(NB, 16, Hkv, D)
    slots = []
    for s, (n, ql) in enumerate(specs):
        sl = token_slots(tables[s], 16 * need[s])
        for t in range(n - ql, 16 * need[s]):           # the chunk and the tail: NaN
            kc.view(-1, Hkv, D)[sl[t]] = float("nan")
            vc.view(-1, Hkv, D)[sl[t]] = float("nan")
        slots += sl[n - ql:n]
    R = sum(ql for _, ql in specs)
    q, kn, vn = rnd(R, Hq, D), rnd(R, Hkv, D), rnd(R, Hkv, D)
    cu = np.concatenate([[0], np.cumsum([ql for _, ql in specs])]).astype(np.int32)
    lens = np.array([n for n, _ in specs], np.int32)
    return dict(kc=kc, vc=vc, q=q, kn=kn, vn=vn, tables=tables, lens=lens, cu=cu,
                slots=np.array(slots, np.int64), maxq=max(ql for _, ql in specs))


def _run(c, D, dev):
    code = oracle.BF16 if c["q"].dtype == torch.bfloat16 else oracle.F16
    hk, hv = oracle.reshape_and_cache(bits(c["kn"]), bits(c["vn"]), bits(c["kc"]),
                                      bits(c["vc"]), c["slots"])
    want = oracle.prefill_attention(code, bits(c["q"]), hk, hv, c["tables"], c["lens"], c["cu"],
                                    D ** -0.5)
    pkv.reshape_and_cache(c["kn"], c["vn"], c["kc"], c["vc"],
                          torch.from_numpy(c["slots"]).to(dev))
    bt = torch.from_numpy(c["tables"]).to(dev)
    cl = torch.from_numpy(c["lens"]).to(dev)
    cu = torch.from_numpy(c["cu"]).to(dev)
    out = torch.full_like(c["q"], float("nan"))
    pkv.paged_attention_prefill(c["q"], c["kc"], c["vc"], bt, cl, cu, c["maxq"], D ** -0.5, out)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    return out, want, code, bt, cl


@pytest.mark.parametrize("dtype,Hq,Hkv,D", [("bf16", 32, 8, 128), ("f16", 32, 4, 64),
                                             ("bf16", 8, 8, 128), ("f16", 16, 8, 64),
                                             ("bf16", 12, 4, 128), ("f16", 32, 2, 128)])
def test_prefill_matches_oracle(dtype, Hq, Hkv, D, cuda_device):
    specs = [(100, 100), (300, 64), (33, 1), (17, 17), (5, 3), (450, 160), (64, 16), (1, 1)]
    c = _case(cuda_device, dtype, specs, Hq, Hkv, D, seed=Hq + D)
    out, want, code, bt, cl = _run(c, D, cuda_device)
    assert_attention_close(bits(out), want, code, f"prefill g={Hq // Hkv} D={D}")
    if Hq // Hkv > 8:
        return                                    # decode attention serves g <= 8
    # the last row of every chunk sees the whole context: it is a decode row
    last = torch.from_numpy(c["cu"][1:] - 1).to(cuda_device).long()
    dec = torch.empty(len(specs), Hq, D, dtype=c["q"].dtype, device=cuda_device)
    ws = pkv.new_workspace(len(specs), Hq, D, int(c["lens"].max()), cuda_device)
    pkv.paged_attention_decode(c["q"][last].contiguous(), c["kc"], c["vc"], bt, cl,
                               int(c["lens"].max()), D ** -0.5, dec, ws)
    torch.cuda.synchronize()
    assert torch.allclose(dec.float(), out[last].float(), atol=1e-2, rtol=1e-2)


@pytest.mark.parametrize("dtype,Hq,Hkv,D", [("bf16", 32, 8, 128), ("f16", 16, 16, 64),
                                             ("bf16", 32, 2, 128), ("f16", 12, 4, 128)])
def test_prefill_rows_past_the_last_chunk_are_never_used(dtype, Hq, Hkv, D, cuda_device):
    """q and out hold more rows than the chunks, NaN past them.  A query tile
    of 128 / g tokens that runs past its chunk loads the rows after it (by
    tensor copies when g divides 128, zero-filled by cp.async otherwise):
    those rows see no key and are never stored, so the chunks match the
    oracle and the extra output rows stay as they were."""
    specs = [(300, 70), (190, 45)]          # chunks that end inside a tile
    c = _case(cuda_device, dtype, specs, Hq, Hkv, D, seed=53 + Hq)
    R = c["q"].shape[0]
    q = torch.full((R + 37, Hq, D), float("nan"), dtype=c["q"].dtype, device=cuda_device)
    q[:R] = c["q"]
    c["q"] = q
    out, want, code, _, _ = _run(c, D, cuda_device)
    assert_attention_close(bits(out[:R]), want[:R], code, f"rows past the chunks g={Hq // Hkv}")
    assert torch.isnan(out[R:].float()).all()


def test_prefill_flags_a_chunk_longer_than_its_context(cuda_device):
    c = _case(cuda_device, "bf16", [(40, 8), (30, 30)], 8, 2, 128, seed=3)
    _run(c, 128, cuda_device)                       # valid first
    bad = torch.tensor([40, 20], dtype=torch.int32, device=cuda_device)   # 30 rows > 20
    out = torch.zeros_like(c["q"])
    pkv.paged_attention_prefill(c["q"], c["kc"], c["vc"],
                                torch.from_numpy(c["tables"]).to(cuda_device), bad,
                                torch.from_numpy(c["cu"]).to(cuda_device), c["maxq"],
                                128 ** -0.5, out)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(reset=True) & pkv.DEV_BAD_LENGTH
    assert torch.count_nonzero(out[8:]) == 0       # the bad sequence was skipped


def test_prefill_flags_rows_outside_q_and_chunks_over_the_bound(cuda_device):
    """cu_q_lens is read on the device: rows past q's end, a negative start or
    a chunk longer than max_q_len are flagged and that sequence is skipped,
    while the valid one is still served."""
    c = _case(cuda_device, "bf16", [(40, 8), (30, 30)], 8, 2, 128, seed=5)
    good, _, _, bt, cl = _run(c, 128, cuda_device)
    cases = [
        ([0, 8, 54], [40, 46], c["maxq"]),          # 46 rows from row 8: past q's 38 rows
        ([0, 8, 38], [40, 30], 8),                  # 30 rows over a bound of 8
        ([-4, 8, 38], [40, 30], c["maxq"]),         # a negative first row
    ]
    for cu, lens, maxq in cases:
        out = torch.zeros_like(c["q"])
        pkv.paged_attention_prefill(c["q"], c["kc"], c["vc"], bt,
                                    torch.tensor(lens, dtype=torch.int32, device=cuda_device),
                                    torch.tensor(cu, dtype=torch.int32, device=cuda_device),
                                    maxq, 128 ** -0.5, out)
        torch.cuda.synchronize()
        assert pkv.pkv_device_status(reset=True) & pkv.DEV_BAD_LENGTH, cu
        if cu[0] == 0:
            assert np.array_equal(bits(out[:8]), bits(good[:8])), cu   # the valid sequence
            assert torch.count_nonzero(out[8:]) == 0, cu
        else:
            assert torch.count_nonzero(out[:8]) == 0, cu
            assert np.array_equal(bits(out[8:]), bits(good[8:])), cu


def test_prefill_long_chunk_over_a_cached_prefix(cuda_device):
    """Many 128-row tiles and key tiles: a 400-token chunk after 1600 cached
    tokens, beside a whole 1200-token prompt."""
    specs = [(2000, 400), (1200, 1200), (129, 129)]
    c = _case(cuda_device, "bf16", specs, 16, 4, 128, seed=41)
    out, want, code, _, _ = _run(c, 128, cuda_device)
    assert_attention_close(bits(out), want, code, "long chunk")


def test_prefill_rescales_when_scores_grow(cuda_device):
    """Scores that climb along the context move a row's running maximum by far
    more than the kernel lets P grow, so the output is rescaled between tiles."""
    specs = [(1100, 600), (700, 700)]
    c = _case(cuda_device, "f16", specs, 8, 2, 128, seed=43)
    # K of token t scaled by (1 + t / 64): later keys score ever higher
    need = [(n + 15) // 16 for n, _ in specs]
    for s, (n, _) in enumerate(specs):
        sl = token_slots(c["tables"][s], 16 * need[s])
        for t in range(n - specs[s][1]):
            row = c["kc"].view(-1, 2, 128)[sl[t]]
            c["kc"].view(-1, 2, 128)[sl[t]] = (row.float() * (1 + t / 64)).to(row.dtype)
    c["kn"] = (c["kn"].float() * 12).to(c["kn"].dtype)
    c["q"] = (c["q"].float() * 2).to(c["q"].dtype)
    out, want, code, _, _ = _run(c, 128, cuda_device)
    assert_attention_close(bits(out), want, code, "growing scores")


def test_prefill_flags_a_bad_block_id(cuda_device):
    c = _case(cuda_device, "bf16", [(300, 300)], 8, 2, 128, seed=47)
    _run(c, 128, cuda_device)
    tables = c["tables"].copy()
    tables[0, 5] = 1 << 30
    out = torch.full_like(c["q"], float("nan"))
    pkv.paged_attention_prefill(c["q"], c["kc"], c["vc"], torch.from_numpy(tables).to(cuda_device),
                                torch.from_numpy(c["lens"]).to(cuda_device),
                                torch.from_numpy(c["cu"]).to(cuda_device), c["maxq"],
                                128 ** -0.5, out)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status(reset=True) & pkv.DEV_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()
