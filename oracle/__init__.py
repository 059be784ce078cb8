"""CPU oracle for the decode-step paged KV cache path (fp64).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's ``cpu_baseline`` / reference leg may import this package.
The product library (``paged_kv_cache_211_gb300``) never imports it and
shares no code with it; the oracle's arithmetic lives in
``pagedkv_oracle.c`` (plain C, gcc) and is wrapped here with ctypes.

Functions and the passages they follow (page title, section):

* ``slot_mapping`` -- "micro-vLLM" wiki, execution chain (KVCacheManager
  keeps each sequence's block table); "mini-vllm 项目深度解析" §2 (fixed
  16-token blocks).  slot = table[p // 16] * 16 + p % 16 for p = len - 1.
* ``reshape_and_cache`` -- "mini-vllm 项目深度解析" §关键工程决策 item 3
  (separate K/V pools, layer-major, block size before KV heads).
* ``decode_attention`` -- "MinivLLM" 使用教程 step 5 (PagedAttention for the
  decode stage) over the cache above; plain softmax attention in fp64.
* ``decode_f16`` / ``decode_bf16`` -- the IEEE binary16 and bfloat16 format
  definitions.
* ``copy_blocks`` -- the device half of copy-on-write (whole-block copies).
* ``prefill_attention`` -- "MinivLLM" 使用教程 step 4 / 核心亮点 (a self-written
  FlashAttention for the prefill stage) over the paged cache: packed query
  chunks, causal within each sequence.
* ``prefix_cache_model.PrefixCacheModel`` -- the allocator's policy (free
  stack, prefix cache by hash, LRU of released cached blocks, copy-on-write,
  rollback) in plain Python.

Every function is pinned by ``tests/test_oracle_pins.py`` against something
other than itself (library routines, brute force, closed forms, invariants);
the policy model by the hand-worked allocator scenarios of
``tests/test_prefix_cache.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")

F16 = 0
BF16 = 1

_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (default: into ``oracle/_build``)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", src, "-o", tmp, "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected 16-bit patterns as uint16, got {a.dtype}")
    return a


class Oracle:
    """One loaded build of the C oracle (the default one, or a test variant)."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        c_u16p = ctypes.POINTER(ctypes.c_uint16)
        c_i32p = ctypes.POINTER(ctypes.c_int32)
        c_i64p = ctypes.POINTER(ctypes.c_int64)
        c_f64p = ctypes.POINTER(ctypes.c_double)
        lib.pko_decode_array.argtypes = [ctypes.c_int, c_u16p, c_f64p, ctypes.c_int64]
        lib.pko_decode_array.restype = None
        lib.pko_slot_mapping.argtypes = [c_i32p, ctypes.c_int, c_i32p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, c_i64p]
        lib.pko_slot_mapping.restype = ctypes.c_int
        lib.pko_reshape_and_cache.argtypes = [c_u16p, c_u16p, c_u16p, c_u16p, c_i64p,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int]
        lib.pko_reshape_and_cache.restype = ctypes.c_int
        lib.pko_decode_attention.argtypes = [ctypes.c_int, c_u16p, c_u16p, c_u16p, c_i32p,
                                             ctypes.c_int, c_i32p, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double, c_f64p, c_f64p,
                                             ctypes.c_int64]
        lib.pko_decode_attention.restype = ctypes.c_int
        lib.pko_copy_blocks.argtypes = [c_u16p, c_u16p, c_i32p, c_i32p, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.pko_copy_blocks.restype = ctypes.c_int
        lib.pko_prefill_attention.argtypes = [ctypes.c_int, c_u16p, c_u16p, c_u16p, c_i32p,
                                              ctypes.c_int, c_i32p, c_i32p, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_double, c_f64p]
        lib.pko_prefill_attention.restype = ctypes.c_int
        self.lib = lib
        self.path = so_path

    def decode(self, dtype: int, bits) -> np.ndarray:
        """16-bit patterns (uint16) -> float64, by the oracle's own decoders."""
        b = _bits(bits)
        out = np.empty(b.shape, np.float64)
        self.lib.pko_decode_array(dtype, _ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double),
                                  b.size)
        return out

    def decode_f16(self, bits) -> np.ndarray:
        return self.decode(F16, bits)

    def decode_bf16(self, bits) -> np.ndarray:
        return self.decode(BF16, bits)

    def slot_mapping(self, block_tables, context_lens, block_size: int,
                     num_blocks: int) -> np.ndarray:
        """Slot of the token at position ``context_len - 1`` of every sequence."""
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        out = np.empty(cl.shape[0], np.int64)
        rc = self.lib.pko_slot_mapping(_ptr(bt, ctypes.c_int32), bt.shape[1],
                                       _ptr(cl, ctypes.c_int32), cl.shape[0], block_size,
                                       num_blocks, _ptr(out, ctypes.c_int64))
        if rc != 0:
            raise ValueError(f"oracle slot_mapping failed with code {rc}")
        return out

    def reshape_and_cache(self, k_new, v_new, k_cache, v_cache, slots):
        """Copies of the K and V pools after writing the new tokens.

        ``k_new``/``v_new``: [T, Hkv, D] uint16; pools: [NB, bs, Hkv, D] uint16.
        """
        kn, vn = _bits(k_new), _bits(v_new)
        kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
        sl = np.ascontiguousarray(slots, dtype=np.int64)
        nb, bs, hkv, d = kc.shape
        rc = self.lib.pko_reshape_and_cache(_ptr(kn, ctypes.c_uint16), _ptr(vn, ctypes.c_uint16),
                                            _ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16),
                                            _ptr(sl, ctypes.c_int64), sl.shape[0], nb, bs, hkv, d)
        if rc != 0:
            raise ValueError(f"oracle reshape_and_cache failed with code {rc}")
        return kc, vc

    def copy_blocks(self, k_cache, v_cache, src, dst):
        """Copies of the pools after block dst[i] receives block src[i] (K and V)."""
        kc, vc = _bits(k_cache).copy(), _bits(v_cache).copy()
        s = np.ascontiguousarray(src, dtype=np.int32)
        d = np.ascontiguousarray(dst, dtype=np.int32)
        nb, bs, hkv, hd = kc.shape
        rc = self.lib.pko_copy_blocks(_ptr(kc, ctypes.c_uint16), _ptr(vc, ctypes.c_uint16),
                                      _ptr(s, ctypes.c_int32), _ptr(d, ctypes.c_int32), s.shape[0],
                                      nb, bs, hkv, hd)
        if rc != 0:
            raise ValueError(f"oracle copy_blocks failed with code {rc}")
        return kc, vc

    def prefill_attention(self, dtype: int, q, k_cache, v_cache, block_tables, context_lens,
                          cu_q_lens, scale: float):
        """fp64 causal attention of packed query rows [R, Hq, D] over the paged cache."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        cu = np.ascontiguousarray(cu_q_lens, dtype=np.int32)
        r, hq, d = qb.shape
        nb, bs, hkv, _ = kc.shape
        out = np.zeros((r, hq, d), np.float64)
        rc = self.lib.pko_prefill_attention(
            dtype, _ptr(qb, ctypes.c_uint16), _ptr(kc, ctypes.c_uint16),
            _ptr(vc, ctypes.c_uint16), _ptr(bt, ctypes.c_int32), bt.shape[1],
            _ptr(cl, ctypes.c_int32), _ptr(cu, ctypes.c_int32), cl.shape[0], hq, hkv, d, nb, bs,
            float(scale), _ptr(out, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"oracle prefill_attention failed with code {rc}")
        return out

    def decode_attention(self, dtype: int, q, k_cache, v_cache, block_tables, context_lens,
                         scale: float, return_weights: bool = False):
        """fp64 decode attention; out [B, Hq, D] (and weights [B, Hq, MB*bs])."""
        qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        b, hq, d = qb.shape
        nb, bs, hkv, d2 = kc.shape
        if d2 != d or vc.shape != kc.shape or bt.shape[0] != b or cl.shape[0] != b:
            raise ValueError("shape mismatch")
        out = np.zeros((b, hq, d), np.float64)
        stride = bt.shape[1] * bs
        w = np.zeros((b, hq, stride), np.float64) if return_weights else None
        rc = self.lib.pko_decode_attention(
            dtype, _ptr(qb, ctypes.c_uint16), _ptr(kc, ctypes.c_uint16),
            _ptr(vc, ctypes.c_uint16), _ptr(bt, ctypes.c_int32), bt.shape[1],
            _ptr(cl, ctypes.c_int32), b, hq, hkv, d, nb, bs, float(scale),
            _ptr(out, ctypes.c_double), _ptr(w, ctypes.c_double) if w is not None else None,
            stride)
        if rc != 0:
            raise ValueError(f"oracle decode_attention failed with code {rc}")
        return (out, w) if return_weights else out


_default = None


def default() -> Oracle:
    """The oracle built from ``pagedkv_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def variant(src_text: str, workdir: str) -> Oracle:
    """Compile and load a modified copy of the oracle source (tests only)."""
    src = os.path.join(workdir, "oracle_variant.c")
    with open(src, "w") as f:
        f.write(src_text)
    return Oracle(build(force=True, src=src, out=os.path.join(workdir, "liboracle_variant.so")))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def decode_f16(bits):
    return default().decode_f16(bits)


def decode_bf16(bits):
    return default().decode_bf16(bits)


def decode(dtype: int, bits):
    return default().decode(dtype, bits)


def slot_mapping(block_tables, context_lens, block_size: int, num_blocks: int):
    return default().slot_mapping(block_tables, context_lens, block_size, num_blocks)


def reshape_and_cache(k_new, v_new, k_cache, v_cache, slots):
    return default().reshape_and_cache(k_new, v_new, k_cache, v_cache, slots)


def copy_blocks(k_cache, v_cache, src, dst):
    return default().copy_blocks(k_cache, v_cache, src, dst)


def prefill_attention(dtype: int, q, k_cache, v_cache, block_tables, context_lens, cu_q_lens,
                      scale: float):
    return default().prefill_attention(dtype, q, k_cache, v_cache, block_tables, context_lens,
                                       cu_q_lens, scale)


def decode_attention(dtype: int, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                     return_weights: bool = False):
    return default().decode_attention(dtype, q, k_cache, v_cache, block_tables, context_lens,
                                      scale, return_weights)
