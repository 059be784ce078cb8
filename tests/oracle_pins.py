"""Pins for the CPU oracle: each check compares the oracle with something
other than itself and raises AssertionError on a mismatch.

They take an ``oracle.Oracle`` so that the same battery can run against the
real oracle (tests/test_oracle_pins.py) and against copies of it with a
planted mistake (tests/test_oracle_mutants.py), which must each fail at
least one pin.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from pkv_testutil import BS, bits, lib_decode, sdpa_reference, token_slots

F16, BF16 = 0, 1


def _f16(x) -> np.ndarray:
    return np.asarray(x, np.float16).view(np.uint16)


def _bf16(x) -> np.ndarray:
    return bits(torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


def _small_case(seed, dtype, B=3, Hq=4, Hkv=2, D=8, NB=12, lens=(1, 17, 33), poison=True):
    """A small paged case with a shuffled pool and NaN in every unused slot."""
    rng = np.random.default_rng(seed)
    enc = _bf16 if dtype == BF16 else _f16
    MB = max(1, max((n + BS - 1) // BS for n in lens))
    perm = rng.permutation(NB)
    tables = np.zeros((B, MB), np.int32)
    used = np.zeros((NB, BS), bool)
    pos = 0
    for s, n in enumerate(lens):
        nb = (n + BS - 1) // BS
        tables[s, :nb] = perm[pos:pos + nb]
        for j in range(nb):
            for o in range(BS):
                if j * BS + o < n:
                    used[perm[pos + j], o] = True
        pos += nb
    free_block = perm[pos]
    for s, n in enumerate(lens):
        tables[s, (n + BS - 1) // BS:] = free_block
    q = enc(rng.standard_normal((B, Hq, D)))
    k = enc(rng.standard_normal((NB, BS, Hkv, D)))
    v = enc(rng.standard_normal((NB, BS, Hkv, D)))
    if poison:
        nan = enc(np.full(1, np.nan))[0]
        k[~used] = nan
        v[~used] = nan
    return q, k, v, tables, np.array(lens, np.int32)


# --- decoders ---------------------------------------------------------------

def pin_decoders_exhaustive(o):
    """All 65536 patterns against numpy float16 and torch bfloat16 conversions."""
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    for dt in (F16, BF16):
        got = o.decode(dt, allbits)
        want = lib_decode(allbits, dt)
        nan_g, nan_w = np.isnan(got), np.isnan(want)
        assert (nan_g == nan_w).all(), "NaN patterns differ"
        assert np.array_equal(got[~nan_g], want[~nan_w]), "decoded values differ"
        assert np.array_equal(np.signbit(got[~nan_g]), np.signbit(want[~nan_w])), "signs differ"


# --- block-table plumbing ----------------------------------------------------

def pin_slot_mapping_enumeration(o):
    """Slot of position len-1 equals the last element of the enumerated slot list."""
    rng = np.random.default_rng(7)
    NB, MB = 50, 6
    for trial in range(20):
        B = 8
        tables = rng.integers(0, NB, size=(B, MB)).astype(np.int32)
        lens = rng.integers(1, MB * BS + 1, size=B).astype(np.int32)
        lens[0] = 16   # last slot of block 0
        lens[1] = 17   # first slot of block 1
        lens[2] = 1
        got = o.slot_mapping(tables, lens, BS, NB)
        want = [token_slots(tables[s], int(lens[s]))[-1] for s in range(B)]
        assert np.array_equal(got, np.array(want)), (got, want)
    got = o.slot_mapping(tables[:1], np.zeros(1, np.int32), BS, NB)
    assert got[0] == -1, "empty sequence must give slot -1"


# --- reshape_and_cache ----------------------------------------------------

def pin_reshape_and_cache_scatter(o):
    """Oracle write == numpy fancy-index scatter over the flattened slot axis."""
    rng = np.random.default_rng(11)
    NB, Hkv, D, T = 9, 3, 8, 7
    k = rng.integers(0, 1 << 16, size=(NB, BS, Hkv, D)).astype(np.uint16)
    v = rng.integers(0, 1 << 16, size=(NB, BS, Hkv, D)).astype(np.uint16)
    kn = rng.integers(0, 1 << 16, size=(T, Hkv, D)).astype(np.uint16)
    vn = rng.integers(0, 1 << 16, size=(T, Hkv, D)).astype(np.uint16)
    slots = rng.choice(NB * BS, size=T, replace=False).astype(np.int64)
    slots[3] = -1  # padding token
    gk, gv = o.reshape_and_cache(kn, vn, k, v, slots)
    wk = k.copy().reshape(NB * BS, Hkv, D)
    wv = v.copy().reshape(NB * BS, Hkv, D)
    keep = slots >= 0
    wk[slots[keep]] = kn[keep]
    wv[slots[keep]] = vn[keep]
    assert np.array_equal(gk, wk.reshape(k.shape)), "K pool differs"
    assert np.array_equal(gv, wv.reshape(v.shape)), "V pool differs"


def pin_copy_blocks_whole_blocks(o):
    """Copy-on-write's device half: after the copy each destination block holds
    its source block's bytes in both pools, every other block is unchanged,
    and an id outside the pool is refused."""
    rng = np.random.default_rng(13)
    NB, Hkv, D = 11, 2, 8
    k = rng.integers(0, 1 << 16, size=(NB, BS, Hkv, D)).astype(np.uint16)
    v = rng.integers(0, 1 << 16, size=(NB, BS, Hkv, D)).astype(np.uint16)
    ids = rng.permutation(NB)
    src, dst = ids[:3].astype(np.int32), ids[3:6].astype(np.int32)   # disjoint lists
    gk, gv = o.copy_blocks(k, v, src, dst)
    wk, wv = k.copy(), v.copy()
    wk[dst], wv[dst] = k[src], v[src]
    assert np.array_equal(gk, wk), "K pool differs"
    assert np.array_equal(gv, wv), "V pool differs"
    try:
        o.copy_blocks(k, v, np.array([NB], np.int32), np.array([0], np.int32))
    except ValueError:
        pass
    else:
        raise AssertionError("an id past the pool was accepted")


# --- decode attention: library pin, brute force, closed forms ----------------

def pin_attention_vs_sdpa(o):
    """Oracle vs torch SDPA (float64) on independently gathered contexts."""
    for dt in (F16, BF16):
        for seed, (Hq, Hkv, D, lens) in enumerate([
                (4, 2, 8, (1, 17, 33)),
                (8, 8, 16, (5, 16, 40)),
                (8, 1, 4, (3, 48, 2)),
                (6, 3, 8, (31, 32, 33))]):
            q, k, v, tb, ln = _small_case(100 + seed, dt, Hq=Hq, Hkv=Hkv, D=D, lens=lens)
            scale = 1.0 / math.sqrt(D)
            got = o.decode_attention(dt, q, k, v, tb, ln, scale)
            want = sdpa_reference(dt, q, k, v, tb, ln, scale)
            assert np.isfinite(got).all(), "oracle output not finite"
            assert np.allclose(got, want, rtol=1e-11, atol=1e-12), np.abs(got - want).max()


def pin_attention_brute_force(o):
    """Pure-Python loops with math.exp on tiny inputs (no numpy arithmetic)."""
    q, k, v, tb, ln = _small_case(5, F16, B=2, Hq=2, Hkv=1, D=4, NB=4, lens=(3, 18))
    scale = 0.7
    got = o.decode_attention(F16, q, k, v, tb, ln, scale)
    qd = lib_decode(q, F16).tolist()
    kd = lib_decode(k, F16).tolist()
    vd = lib_decode(v, F16).tolist()
    for s in range(2):
        for i in range(2):
            zs = []
            rows = []
            for t in range(int(ln[s])):
                b = int(tb[s][t // BS])
                krow = kd[b][t % BS][0]
                rows.append(vd[b][t % BS][0])
                zs.append(scale * sum(qd[s][i][d] * krow[d] for d in range(4)))
            m = max(zs)
            e = [math.exp(z - m) for z in zs]
            tot = sum(e)
            for d in range(4):
                want = sum(e[t] / tot * rows[t][d] for t in range(len(e)))
                assert abs(got[s, i, d] - want) <= 1e-12, (s, i, d, got[s, i, d], want)


def _one_seq(dt, q_vals, k_rows, v_rows, table, NB, Hkv=1, scale=1.0):
    """A single-sequence case with explicit rows placed through `table`."""
    enc = _bf16 if dt == BF16 else _f16
    D = len(q_vals[0])
    n = len(k_rows)
    k = np.zeros((NB, BS, Hkv, D), np.float64)
    v = np.zeros((NB, BS, Hkv, D), np.float64)
    for t in range(n):
        b = table[t // BS]
        k[b, t % BS] = np.asarray(k_rows[t]).reshape(Hkv, D)
        v[b, t % BS] = np.asarray(v_rows[t]).reshape(Hkv, D)
    q = enc(np.asarray(q_vals, np.float64)[None])
    return (q, enc(k), enc(v), np.array([table], np.int32), np.array([n], np.int32), scale)


def pin_closed_forms(o):
    # (a) two tokens, scores (0, ln 3): weights 1/4, 3/4
    case = _one_seq(F16, [[1, 0]], [[0, 0], [1, 0]], [[4, -2], [8, 2]], [1], NB=2,
                    scale=math.log(3.0))
    got = o.decode_attention(F16, *case)
    assert np.allclose(got[0, 0], [7.0, 1.0], rtol=0, atol=1e-12), got
    # (b) 17 tokens across two physical blocks (table [2, 0]); token 16 sits in
    #     block 0 slot 0 and scores ln 48, the other 16 score 0:
    #     weights 1/64 each and 48/64; V_t = (t, 1)  ->  out = (120/64 + 12, 1)
    k_rows = [[0, 0]] * 16 + [[1, 0]]
    v_rows = [[t, 1] for t in range(17)]
    case = _one_seq(F16, [[1, 0]], k_rows, v_rows, [2, 0], NB=3, scale=math.log(48.0))
    got = o.decode_attention(F16, *case)
    assert np.allclose(got[0, 0], [120 / 64 + 12, 1.0], rtol=0, atol=1e-12), got
    # (c) a context of length 1 returns V exactly
    q, k, v, tb, ln = _small_case(9, BF16, lens=(1, 1, 1))
    got = o.decode_attention(BF16, q, k, v, tb, ln, 0.3)
    for s in range(3):
        b = tb[s, 0]
        want = lib_decode(v[b, 0], BF16)   # [Hkv, D]
        for i in range(4):
            assert np.array_equal(got[s, i], want[i // 2]), "length-1 context must return V"
    # (d) identical K rows: uniform weights, out = mean of V rows
    rng = np.random.default_rng(3)
    vr = rng.integers(-8, 9, size=(20, 4)).astype(np.float64)
    case = _one_seq(F16, [[0.5, -1, 2, 0.25]], [[1, 2, 3, 4]] * 20, vr, [4, 1], NB=5, scale=0.9)
    got = o.decode_attention(F16, *case)
    assert np.allclose(got[0, 0], vr.mean(0), rtol=0, atol=1e-12), (got, vr.mean(0))
    # (e) scores of 40000 (exp overflows unless the maximum is subtracted):
    #     token 0 dominates completely and out = V_0
    k_rows = [[100, 100, 100, 100]] + [[0, 0, 0, 0]] * 15
    v_rows = [[1, 2, 3, 4]] + [[-7, -7, -7, -7]] * 15
    case = _one_seq(F16, [[100, 100, 100, 100]], k_rows, v_rows, [0], NB=1, scale=1.0)
    got = o.decode_attention(F16, *case)
    assert np.array_equal(got[0, 0], [1.0, 2.0, 3.0, 4.0]), got
    # (f) GQA: V constant per KV head (value h+1): query head i returns i // g + 1
    Hq, Hkv, D = 8, 4, 4
    rng = np.random.default_rng(4)
    n = 21
    k_rows = [rng.standard_normal(Hkv * D) for _ in range(n)]
    v_rows = [np.repeat(np.arange(1, Hkv + 1, dtype=np.float64), D) for _ in range(n)]
    q_vals = rng.standard_normal((Hq, D))
    case = _one_seq(BF16, q_vals, k_rows, v_rows, [1, 0], NB=2, Hkv=Hkv, scale=0.5)
    got = o.decode_attention(BF16, *case)
    for i in range(Hq):
        assert np.allclose(got[0, i], i // (Hq // Hkv) + 1, rtol=0, atol=1e-12), (i, got[0, i])
    # (g) an empty context gives an all-zero output
    q, k, v, tb, ln = _small_case(10, F16, lens=(0, 5, 0))
    got = o.decode_attention(F16, q, k, v, tb, ln, 0.3)
    assert np.array_equal(got[0], np.zeros_like(got[0])) and np.array_equal(got[2], 0 * got[2])


# --- invariants ---------------------------------------------------------------

def pin_weights_sum_to_one(o):
    q, k, v, tb, ln = _small_case(21, BF16, lens=(1, 17, 40))
    out, w = o.decode_attention(BF16, q, k, v, tb, ln, 0.35, return_weights=True)
    for s, n in enumerate(ln):
        assert np.allclose(w[s, :, :n].sum(-1), 1.0, rtol=0, atol=1e-12)
        assert (w[s, :, :n] >= 0).all()
        assert np.all(w[s, :, n:] == 0)


def pin_block_permutation_invariance(o):
    """Relabelling physical blocks (pool and tables alike) changes nothing, bit for bit."""
    q, k, v, tb, ln = _small_case(31, F16, lens=(7, 33, 20))
    base = o.decode_attention(F16, q, k, v, tb, ln, 0.25)
    perm = np.random.default_rng(32).permutation(k.shape[0])
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    got = o.decode_attention(F16, q, k2, v2, perm[tb].astype(np.int32), ln, 0.25)
    assert np.array_equal(base, got)


def pin_shared_prefix_equals_private(o):
    """Sequences sharing prefix blocks == the same sequences with private copies."""
    rng = np.random.default_rng(41)
    NB, Hkv, D, B = 20, 2, 8, 3
    k = _bf16(rng.standard_normal((NB, BS, Hkv, D)))
    v = _bf16(rng.standard_normal((NB, BS, Hkv, D)))
    q = _bf16(rng.standard_normal((B, 4, D)))
    shared = [0, 1]                  # 32-token prefix
    tb = np.array([shared + [2, 3], shared + [4, 5], shared + [6, 7]], np.int32)
    ln = np.array([40, 64, 33], np.int32)
    a = o.decode_attention(BF16, q, k, v, tb, ln, 0.3)
    k2, v2 = k.copy(), v.copy()
    tb2 = tb.copy()
    nxt = 8
    for s in range(1, B):            # give sequences 1.. their own copies
        for j in range(2):
            k2[nxt] = k[shared[j]]
            v2[nxt] = v[shared[j]]
            tb2[s, j] = nxt
            nxt += 1
    b = o.decode_attention(BF16, q, k2, v2, tb2, ln, 0.3)
    assert np.array_equal(a, b)


def pin_poison_not_read(o):
    """NaN in every unused slot and block leaves the output finite and unchanged."""
    q, k, v, tb, ln = _small_case(51, BF16, lens=(3, 17, 30), poison=True)
    q2, k2, v2, _, _ = _small_case(51, BF16, lens=(3, 17, 30), poison=False)
    a = o.decode_attention(BF16, q, k, v, tb, ln, 0.3)
    b = o.decode_attention(BF16, q2, k2, v2, tb, ln, 0.3)
    assert np.isfinite(a).all() and np.array_equal(a, b)


ALL_PINS = [
    pin_decoders_exhaustive,
    pin_slot_mapping_enumeration,
    pin_reshape_and_cache_scatter,
    pin_copy_blocks_whole_blocks,
    pin_attention_vs_sdpa,
    pin_attention_brute_force,
    pin_closed_forms,
    pin_weights_sum_to_one,
    pin_block_permutation_invariance,
    pin_shared_prefix_equals_private,
    pin_poison_not_read,
]


def failing_pins(o) -> list:
    """Names of the pins that fail (or raise) for oracle build ``o``."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception:  # an assertion, or the oracle rejecting its inputs
            bad.append(pin.__name__)
    return bad


# --- prefill (causal, packed chunks) -------------------------------------------

def pin_prefill_vs_sdpa_causal(o):
    """Prefill oracle vs torch SDPA (float64) with an explicit causal mask built
    from positions, on contexts gathered by enumeration."""
    import torch.nn.functional as F
    from pkv_testutil import token_slots
    rng = np.random.default_rng(61)
    for dt, (Hq, Hkv, D) in [(F16, (4, 2, 8)), (BF16, (6, 3, 16)), (F16, (2, 2, 4))]:
        enc = _bf16 if dt == BF16 else _f16
        lens = [5, 33, 17, 1]
        qlens = [5, 7, 1, 1]          # a whole prompt, a chunk, and decode-like rows
        NB = 12
        perm = rng.permutation(NB)
        MB = 3
        tables = np.zeros((4, MB), np.int32)
        pos = 0
        for s, n in enumerate(lens):
            nb = (n + 15) // 16
            tables[s, :nb] = perm[pos:pos + nb]
            pos += nb
        k = enc(rng.standard_normal((NB, BS, Hkv, D)))
        v = enc(rng.standard_normal((NB, BS, Hkv, D)))
        cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
        q = enc(rng.standard_normal((cu[-1], Hq, D)))
        scale = 0.37
        got = o.prefill_attention(dt, q, k, v, tables, np.array(lens, np.int32), cu, scale)
        kf = k.reshape(NB * BS, Hkv, D)
        vf = v.reshape(NB * BS, Hkv, D)
        for s, (n, ql) in enumerate(zip(lens, qlens)):
            sl = np.array(token_slots(tables[s], n))
            K = torch.from_numpy(lib_decode(kf[sl], dt)).permute(1, 0, 2).repeat_interleave(
                Hq // Hkv, dim=0)
            V = torch.from_numpy(lib_decode(vf[sl], dt)).permute(1, 0, 2).repeat_interleave(
                Hq // Hkv, dim=0)
            Q = torch.from_numpy(lib_decode(q[cu[s]:cu[s + 1]], dt)).permute(1, 0, 2)
            qpos = torch.arange(n - ql, n).unsqueeze(1)
            kpos = torch.arange(n).unsqueeze(0)
            mask = kpos <= qpos                                   # [ql, n]
            ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
            want = ref.permute(1, 0, 2).numpy()
            assert np.allclose(got[cu[s]:cu[s + 1]], want, rtol=1e-11, atol=1e-12), s


def pin_prefill_last_row_is_decode(o):
    """The last row of a chunk sees the whole context: it equals decode attention."""
    q, k, v, tb, ln = _small_case(71, BF16, lens=(1, 17, 40))
    cu = np.array([0, 1, 2, 3], np.int32)
    a = o.prefill_attention(BF16, q, k, v, tb, ln, cu, 0.4)
    b = o.decode_attention(BF16, q, k, v, tb, ln, 0.4)
    assert np.array_equal(a, b)


def pin_prefill_large_scores(o):
    """Scores near 1e3 overflow exp in fp64 unless the row maximum is taken out
    first; the result must still match SDPA (which is overflow-safe)."""
    import torch.nn.functional as F
    rng = np.random.default_rng(67)
    n, ql, D = 20, 6, 4
    q = _f16(np.full((ql, 1, D), 4.0))
    kv = rng.choice([-4.0, 4.0], size=(2, BS, 1, D))
    kv[1, 0] = 4.0                                 # token 0: q . k = 64, the row maximum
    k = _f16(kv)
    v = _f16(rng.standard_normal((2, BS, 1, D)))
    tables = np.array([[1, 0]], np.int32)
    cu = np.array([0, ql], np.int32)
    scale = 20.0                                   # |score| up to 20 * 64 = 1280
    got = o.prefill_attention(F16, q, k, v, tables, np.array([n], np.int32), cu, scale)
    kf, vf = k.reshape(-1, 1, D), v.reshape(-1, 1, D)
    from pkv_testutil import token_slots
    sl = np.array(token_slots(tables[0], n))
    K = torch.from_numpy(lib_decode(kf[sl], F16)).permute(1, 0, 2)
    V = torch.from_numpy(lib_decode(vf[sl], F16)).permute(1, 0, 2)
    Q = torch.from_numpy(lib_decode(q, F16)).permute(1, 0, 2)
    mask = torch.arange(n).unsqueeze(0) <= torch.arange(n - ql, n).unsqueeze(1)
    want = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
    want = want.permute(1, 0, 2).numpy()
    assert np.isfinite(got).all(), "non-finite output"
    assert np.allclose(got, want, rtol=1e-11, atol=1e-12)


ALL_PINS += [pin_prefill_vs_sdpa_causal, pin_prefill_last_row_is_decode,
             pin_prefill_large_scores]
