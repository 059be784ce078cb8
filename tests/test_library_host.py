"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host logic (allocator, sizing, argument validation that
returns before any CUDA call) behaves as documented."""
import ctypes
import json
import os
import re
import subprocess

import pytest

import paged_kv_cache_211_gb300 as pkv
from paged_kv_cache_211_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def L():
    pkv_build.build()
    return pkv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("paged_kv_alloc", "reshape_and_cache", "paged_attention_decode",
                 "paged_kv_slot_mapping", "paged_kv_decode_step", "pkv_cache_bytes"):
        assert must in names
    assert len(names) >= 20


def test_every_declared_symbol_is_exported(L):
    nm = subprocess.run(["nm", "-D", "--defined-only", pkv.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = {line.split()[-1] for line in nm.splitlines() if " T " in line}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(L, n)


def declared_arity():
    """Parameter count of every function the header declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(([^)]*)\)\s*;",
                         text, flags=re.M):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_signatures_match_the_header():
    """Every ctypes signature the binding installs has the header's parameter count."""
    arity = declared_arity()
    assert set(arity) == set(declared_functions())
    for name, (argtypes, _) in pkv._SIGS.items():
        assert name in arity, f"{name} is bound but not declared"
        assert len(argtypes) == arity[name], (name, len(argtypes), arity[name])


def test_version_and_status_strings(L):
    assert pkv.pkv_version() >= 100
    assert L.pkv_status_string(0) == b"ok"
    assert L.pkv_status_string(3) == b"not enough free blocks"


def test_cache_bytes_layout():
    facts = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_facts.json")))
    bs = facts["block_size"]["value"]
    # one pool = layers x blocks x 16 x kv_heads x head_dim x 2 bytes
    assert pkv.pkv_cache_bytes(28, 4096, 8, 128, block_size=bs) == 28 * 4096 * 16 * 8 * 128 * 2
    assert pkv.pkv_cache_bytes(1, 10, 8, 128, block_size=32) == 0   # block size is fixed at 16
    assert pkv.pkv_cache_bytes(0, 10, 8, 128) == 0


def test_workspace_sizing():
    w1 = pkv.paged_attention_workspace_bytes(32, 32, 128, 32768)
    w2 = pkv.paged_attention_workspace_bytes(32, 32, 128, 100)   # 7 blocks -> <= 7 partitions
    assert w1 > w2 > 0 and w1 % 256 == 0
    # long contexts: the even split keeps two slots of up to 16 query-head rows
    # for each of up to 256 CTAs; short ones never use it and reserve nothing
    even_rows = 2 * 256 * 16 * (128 + 2) * 4
    assert pkv.paged_attention_workspace_bytes(1, 32, 128, 32768) >= even_rows
    assert pkv.paged_attention_workspace_bytes(1, 32, 128, 100) < even_rows
    assert pkv.paged_attention_workspace_bytes(1, 4, 128, 32768) >= 2 * 256 * 4 * (128 + 2) * 4
    assert pkv.paged_attention_workspace_bytes(32, 32, 128, 1024) == w1   # 64 partitions either way
    # at most 64 partitions per sequence: 32 seqs x 64 x 32 heads x (128 + 2) floats
    assert w1 <= 32 * 64 * 32 * 130 * 4 + 4096
    assert pkv.paged_attention_min_partition_blocks(32768) == 32
    assert pkv.paged_attention_min_partition_blocks(100) == 1
    assert pkv.paged_attention_workspace_bytes(0, 32, 128, 100) == 0


def test_admission_control_with_six_blocks():
    """The pages' pressure case: 6 blocks; a request needing more is refused whole."""
    facts = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_facts.json")))
    a = pkv.BlockAllocator(facts["admission_under_pressure"]["num_blocks"])
    first = a.alloc(4)
    assert sorted(first) == [0, 1, 2, 3] and a.num_free() == 2
    with pytest.raises(pkv.PagedKVError) as e:
        a.alloc(3)                   # all or nothing
    assert e.value.status == 3 and a.num_free() == 2
    a.free(first[:2])
    assert a.num_free() == 4
    second = a.alloc(4)
    assert len(set(second)) == 4 and not set(second) & set(first[2:])
    assert a.num_free() == 0


def test_prefix_sharing_refcounts():
    a = pkv.BlockAllocator(10)
    prefix = a.alloc(3)
    a.share(prefix)                  # a second sequence shares the prefix
    assert [a.refcount(b) for b in prefix] == [2, 2, 2]
    a.free(prefix)                   # first sequence finishes
    assert a.num_free() == 7 and [a.refcount(b) for b in prefix] == [1, 1, 1]
    a.free(prefix)                   # second one too: blocks return
    assert a.num_free() == 10 and a.refcount(prefix[0]) == 0


def test_allocator_rejects_bad_ids_whole():
    a = pkv.BlockAllocator(5)
    ids = a.alloc(2)
    for bad in ([ids[0], 7], [ids[0], -1], [ids[0], 4]):   # out of range / never allocated
        with pytest.raises(pkv.PagedKVError) as e:
            a.free(bad)
        assert e.value.status == 4
    assert [a.refcount(i) for i in ids] == [1, 1]        # nothing changed
    with pytest.raises(pkv.PagedKVError):
        a.free([ids[0], ids[0]])                         # more drops than references
    assert a.refcount(ids[0]) == 1
    with pytest.raises(pkv.PagedKVError):
        a.share([3])
    assert a.refcount(-1) == -1 and a.refcount(99) == -1
    assert a.alloc(0) == []


def test_host_validation_before_any_cuda_call(L):
    """Bad arguments are refused on the host with a status code (no device touched)."""
    p = ctypes.c_void_p(4096)   # never dereferenced: validation fails first
    # odd group (Hq % Hkv != 0)
    rc = L.paged_attention_decode(p, p, p, p, 4, p, 64, 2, 12, 8, 128, 10, 0.1, p, p, 1 << 20,
                                  0, None)
    assert rc == 1
    # head_dim 96 and group 16 are valid shapes the library has no kernel for
    assert L.paged_attention_decode(p, p, p, p, 4, p, 64, 2, 16, 8, 96, 10, 0.1, p, p, 1 << 20,
                                    0, None) == 2
    assert L.paged_attention_decode(p, p, p, p, 4, p, 64, 2, 32, 2, 128, 10, 0.1, p, p, 1 << 20,
                                    0, None) == 2
    # workspace too small
    assert L.paged_attention_decode(p, p, p, p, 4, p, 64, 2, 16, 8, 128, 10, 0.1, p, p, 8, 0,
                                    None) == 6
    # bad dtype, null q, non-finite scale
    assert L.paged_attention_decode(p, p, p, p, 4, p, 64, 2, 16, 8, 128, 10, 0.1, p, p, 1 << 20,
                                    7, None) == 1
    assert L.paged_attention_decode(None, p, p, p, 4, p, 64, 2, 16, 8, 128, 10, 0.1, p, p,
                                    1 << 20, 0, None) == 1
    assert L.paged_attention_decode(p, p, p, p, 4, p, 64, 2, 16, 8, 128, 10, float("inf"), p, p,
                                    1 << 20, 0, None) == 1
    # partition shorter than the workspace bound allows
    assert L.paged_attention_decode_partitioned(p, p, p, p, 2048, p, 32768, 2, 16, 8, 128, 10,
                                                0.1, p, p, 1 << 30, 1, 0, None) == 1
    # reshape_and_cache: head_dim whose rows are not 16-byte multiples; misaligned pointer
    assert L.reshape_and_cache(p, p, p, p, p, 3, 10, 1, 4, 0, None) == 2
    assert L.reshape_and_cache(ctypes.c_void_p(18), p, p, p, p, 3, 10, 8, 128, 0, None) == 1
    # zero work is fine and touches nothing
    assert L.reshape_and_cache(None, None, None, None, None, 0, 10, 8, 128, 0, None) == 0
    assert L.paged_attention_decode(None, None, None, None, 4, None, 64, 0, 16, 8, 128, 10, 0.1,
                                    None, None, 0, 0, None) == 0
    # prefill: negative row count of q
    assert L.paged_attention_prefill(p, p, p, p, 4, p, p, 2, 8, -1, 16, 8, 128, 10, 0.1, p, 0,
                                     None) == 1
    # host-buffer step: staging too small
    assert L.paged_kv_decode_step_host(p, p, p, p, p, p, p, 64, p, p, 4, 64, 2, 16, 8, 128, 10,
                                       0.1, p, 1 << 20, 0, None) == 6


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(pkv, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(pkv, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        pkv.lib()
