"""Host allocator with prefix cache, copy-on-write and rollback, against the
plain Python policy model (oracle/prefix_cache_model.py), plus scenarios."""
import random

import numpy as np
import pytest

import oracle
import paged_kv_cache_211_gb300 as pkv
from oracle.prefix_cache_model import ModelError, PrefixCacheModel


def _run(fn):
    try:
        return ("ok", fn())
    except pkv.PagedKVError as e:
        return ("err", e.status)
    except ModelError as e:
        return ("err", e.code)


class _ModelAllocator:
    """The policy model behind the library allocator's Python API, so that the
    scripted scenarios below (expectations worked out by hand) pin the model
    as well as the library."""

    def __init__(self, num_blocks):
        self.m = PrefixCacheModel(num_blocks)

    def _call(self, fn, *args):
        try:
            return fn(*args)
        except ModelError as e:
            raise pkv.PagedKVError("model", e.code) from None

    def alloc(self, n):
        return self._call(self.m.alloc, n)

    def share(self, ids):
        return self._call(self.m.share, list(ids))

    def free(self, ids):
        return self._call(self.m.free_ids, list(ids))

    def num_free(self):
        return self.m.num_free()

    def refcount(self, b):
        return self.m.refs[b] if 0 <= b < self.m.n else -1

    def num_cached(self):
        return len(self.m.hash_of)

    def prefix_insert(self, b, h):
        return self._call(self.m.insert, b, h)

    def prefix_lookup(self, hashes):
        return self._call(self.m.lookup, list(hashes))

    def cow(self, b):
        return self._call(self.m.cow, b)

    def rollback(self, table, new_len):
        return self._call(self.m.rollback, list(table), new_len)


ALLOCATORS = pytest.mark.parametrize("make", [pkv.BlockAllocator, _ModelAllocator],
                                     ids=["library", "oracle_model"])


def test_differential_random_ops():
    rng = random.Random(2111)
    NB = 40
    for trial in range(6):
        a = pkv.BlockAllocator(NB)
        m = PrefixCacheModel(NB)
        hashes = [rng.getrandbits(64) for _ in range(30)]
        held = []          # block ids we hold a reference to (with repeats)
        for step in range(600):
            op = rng.choice(["alloc", "alloc", "free", "share", "insert", "lookup", "cow",
                             "rollback", "bad_free"])
            if op == "alloc":
                k = rng.randint(0, 6)
                r1, r2 = _run(lambda: a.alloc(k)), _run(lambda: m.alloc(k))
                if r1[0] == "ok":
                    held += r1[1]
            elif op == "free" and held:
                ids = rng.sample(held, rng.randint(1, min(4, len(held))))
                r1, r2 = _run(lambda: a.free(ids)), _run(lambda: m.free_ids(ids))
                if r1[0] == "ok":
                    for b in ids:
                        held.remove(b)
            elif op == "share" and held:
                ids = rng.sample(held, rng.randint(1, min(3, len(held))))
                r1, r2 = _run(lambda: a.share(ids)), _run(lambda: m.share(ids))
                if r1[0] == "ok":
                    held += ids
            elif op == "insert" and held:
                b, h = rng.choice(held), rng.choice(hashes)
                r1, r2 = _run(lambda: a.prefix_insert(b, h)), _run(lambda: m.insert(b, h))
            elif op == "lookup":
                hs = rng.sample(hashes, rng.randint(1, 4))
                r1, r2 = _run(lambda: a.prefix_lookup(hs)), _run(lambda: m.lookup(hs))
                if r1[0] == "ok":
                    held += r1[1]
            elif op == "cow" and held:
                b = rng.choice(held)
                r1, r2 = _run(lambda: a.cow(b)), _run(lambda: m.cow(b))
                if r1[0] == "ok":
                    held.remove(b)
                    held.append(r1[1][0])
            elif op == "rollback" and held:
                table = rng.sample(held, rng.randint(1, min(5, len(held))))
                if len(set(table)) != len(table):
                    continue
                new_len = rng.randint(0, 16 * len(table))
                r1 = _run(lambda: a.rollback(list(table), new_len))
                r2 = _run(lambda: m.rollback(list(table), new_len))
                if r1[0] == "ok":
                    for b in table[len(r1[1]):]:
                        held.remove(b)
            elif op == "bad_free":
                ids = [NB + 3]
                r1, r2 = _run(lambda: a.free(ids)), _run(lambda: m.free_ids(ids))
            else:
                continue
            assert r1 == r2, (trial, step, op, r1, r2)
            assert a.num_free() == m.num_free()
            assert a.num_cached() == len(m.by_hash)
            assert [a.refcount(b) for b in range(NB)] == m.refs


def test_block_hash_chains_and_is_sensitive():
    toks = list(range(100, 116))
    h0 = pkv.paged_kv_block_hash(0, toks)
    assert h0 == pkv.paged_kv_block_hash(0, toks)            # deterministic
    assert h0 != pkv.paged_kv_block_hash(1, toks)            # parent matters
    for i in range(16):
        t2 = list(toks)
        t2[i] += 1
        assert pkv.paged_kv_block_hash(0, t2) != h0          # every token matters
    assert pkv.paged_kv_block_hash(0, toks[::-1]) != h0      # order matters
    h1 = pkv.paged_kv_block_hash(h0, toks)
    assert h1 not in (h0, pkv.paged_kv_block_hash(0, toks + toks))


def _chain(tokens):
    hs, h = [], 0
    for i in range(0, len(tokens) - len(tokens) % 16, 16):
        h = pkv.paged_kv_block_hash(h, tokens[i:i + 16])
        hs.append(h)
    return hs


@ALLOCATORS
def test_prefix_reuse_release_and_eviction(make):
    a = make(8)
    prompt = list(range(48))                     # 3 full blocks
    hs = _chain(prompt)
    A = a.alloc(3)
    for b, h in zip(A, hs):
        a.prefix_insert(b, h)
    assert a.num_cached() == 3
    B = a.prefix_lookup(hs[:2] + [12345])        # shares the first two, stops at the miss
    assert B == A[:2] and [a.refcount(b) for b in A] == [2, 2, 1]
    a.free(A)
    a.free(B)
    # released but registered: cached, not free-listed, still found by hash
    assert a.num_free() == 8 and a.num_cached() == 3
    assert all(a.refcount(b) == 0 for b in A)
    C = a.prefix_lookup(hs)
    assert C == A and all(a.refcount(b) == 1 for b in A)
    a.free(C)
    # memory pressure: 5 never-used blocks go first, then cached ones, oldest first
    D = a.alloc(6)
    assert sorted(D[:5]) == [3, 4, 5, 6, 7] and D[5] == A[0]
    assert a.num_cached() == 2 and a.prefix_lookup(hs[:1]) == []


@ALLOCATORS
def test_rollback_refuses_a_bad_tail_whole(make):
    """A tail naming a block more often than it is referenced, or a length past
    the table (up to the largest int), is refused and nothing changes."""
    a = make(6)
    t = a.alloc(2)
    with pytest.raises(pkv.PagedKVError) as e:
        a.rollback(t + [t[1]], 16)                   # t[1] twice in the tail, held once
    assert e.value.status == 4
    assert [a.refcount(b) for b in t] == [1, 1] and a.num_free() == 4
    with pytest.raises(pkv.PagedKVError) as e:
        a.rollback(t, 2 ** 31 - 1)
    assert e.value.status == 1
    assert a.rollback(t, 16) == t[:1] and a.num_free() == 5


@ALLOCATORS
def test_copy_on_write_and_rollback(make):
    a = make(8)
    x = a.alloc(2)
    a.prefix_insert(x[1], 777)
    a.share(x)                                   # a second sequence forks
    new, copy = a.cow(x[1])                      # before writing into the shared block
    assert copy and new not in x and a.refcount(x[1]) == 1 and a.refcount(new) == 1
    same, copy2 = a.cow(x[0])                    # still shared: copy again
    assert copy2
    mine, copy3 = a.cow(new)                     # sole owner: write in place
    assert mine == new and not copy3
    # rollback of a 3-block sequence to 20 tokens keeps 2 blocks
    t = a.alloc(3)
    a.prefix_insert(t[1], 999)
    kept = a.rollback(t, 20)
    assert kept == t[:2] and a.refcount(t[2]) == 0
    assert a.prefix_lookup([999]) == []          # now-partial block left the cache
    with pytest.raises(pkv.PagedKVError):
        a.rollback(t[:2], 40)                    # longer than the table


@pytest.mark.gpu
def test_copy_blocks_bit_exact(cuda_device):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    g = torch.Generator(device=cuda_device).manual_seed(5)
    NB, Hkv, D = 20, 8, 128
    kc = torch.randn(NB, 16, Hkv, D, generator=g, device=cuda_device).to(torch.bfloat16)
    vc = torch.randn(NB, 16, Hkv, D, generator=g, device=cuda_device).to(torch.bfloat16)
    src = np.array([3, 7, 0, 11], np.int32)
    dst = np.array([12, 4, 19, 1], np.int32)
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    want_k, want_v = oracle.copy_blocks(bits(kc), bits(vc), src, dst)
    pkv.paged_kv_copy_blocks(kc, vc, torch.from_numpy(src).to(cuda_device),
                             torch.from_numpy(dst).to(cuda_device))
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0
    assert np.array_equal(bits(kc), want_k) and np.array_equal(bits(vc), want_v)


@pytest.mark.gpu
def test_copy_blocks_skips_clashing_pairs(cuda_device):
    """Pairs whose outcome would depend on the order of the copies are skipped
    and flagged: two pairs writing block 4, and a pair writing block 3, which
    pair 0 reads.  A pair copying a block onto itself changes nothing.  The
    other pairs are copied bit for bit, as the oracle copies them."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    g = torch.Generator(device=cuda_device).manual_seed(6)
    NB, Hkv, D = 24, 4, 64
    kc = torch.randn(NB, 16, Hkv, D, generator=g, device=cuda_device).to(torch.float16)
    vc = torch.randn(NB, 16, Hkv, D, generator=g, device=cuda_device).to(torch.float16)
    src = np.array([3, 7, 0, 11, 5, 9, 6, 13], np.int32)
    dst = np.array([12, 4, 19, 1, 4, 3, 6, 20], np.int32)
    copied = [2, 3, 7]                         # 0, 1, 4 and 5 clash; 6 is a self-copy
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    want_k, want_v = oracle.copy_blocks(bits(kc), bits(vc), src[copied], dst[copied])
    pkv.paged_kv_copy_blocks(kc, vc, torch.from_numpy(src).to(cuda_device),
                             torch.from_numpy(dst).to(cuda_device))
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == pkv.DEV_BAD_BLOCK_ID
    assert np.array_equal(bits(kc), want_k) and np.array_equal(bits(vc), want_v)


@pytest.mark.gpu
def test_parallel_sampling_fork_with_copy_on_write(cuda_device):
    """Two sequences forked from one 40-token prompt share its 3 blocks (the
    last one partial).  Before each appends its own token, copy-on-write gives
    the second one a private copy of the partial block; then one decode step
    writes both tokens and attends.  Checked against the oracle doing the same
    on host copies."""
    import torch
    import __graft_entry__
    from gpu_helpers import assert_attention_close
    __graft_entry__.build()
    NB, Hq, Hkv, D, prompt = 10, 8, 2, 128, 40
    g = torch.Generator(device=cuda_device).manual_seed(9)
    rnd = lambda *shape: torch.randn(*shape, generator=g, device=cuda_device).to(torch.bfloat16)
    kc, vc = rnd(NB, 16, Hkv, D), rnd(NB, 16, Hkv, D)
    q, kn, vn = rnd(2, Hq, D), rnd(2, Hkv, D), rnd(2, Hkv, D)
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    h_kc, h_vc = bits(kc), bits(vc)

    a = pkv.BlockAllocator(NB)
    shared = a.alloc(3)                        # the prompt's blocks (prefill wrote them)
    a.share(shared)                            # the fork: both sequences reference them
    tables = [list(shared), list(shared)]
    new_id, copy = a.cow(shared[2])            # sequence 1 writes next: copy first
    assert copy
    tables[1][2] = new_id
    src = torch.tensor([shared[2]], dtype=torch.int32, device=cuda_device)
    dst = torch.tensor([new_id], dtype=torch.int32, device=cuda_device)
    pkv.paged_kv_copy_blocks(kc, vc, src, dst)
    mine, copy0 = a.cow(shared[2])             # sequence 0 is now the sole owner
    assert mine == shared[2] and not copy0

    bt = torch.tensor(tables, dtype=torch.int32, device=cuda_device)
    cl = torch.tensor([prompt + 1, prompt + 1], dtype=torch.int32, device=cuda_device)
    out = torch.empty_like(q)
    ws = pkv.new_workspace(2, Hq, D, prompt + 1, cuda_device)
    pkv.paged_kv_decode_step(q, kn, vn, kc, vc, bt, cl, prompt + 1, D ** -0.5, out, ws)
    torch.cuda.synchronize()
    assert pkv.pkv_device_status() == 0

    # oracle: the same copy, write and attention on the host copies
    ok, ov = oracle.copy_blocks(h_kc, h_vc, [shared[2]], [new_id])
    tb = np.array(tables, np.int32)
    ln = np.array([prompt + 1] * 2, np.int32)
    slots = oracle.slot_mapping(tb, ln, 16, NB)
    ok, ov = oracle.reshape_and_cache(bits(kn), bits(vn), ok, ov, slots)
    want = oracle.decode_attention(oracle.BF16, bits(q), ok, ov, tb, ln, D ** -0.5)
    assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov)
    assert_attention_close(bits(out), want, oracle.BF16, "forked sequences")
    # the two sequences now differ only in their last token
    assert not torch.equal(out[0], out[1])
