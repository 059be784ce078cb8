"""Python binding of libpagedkv (decode-step PagedAttention on GB300).

Argument marshalling only: every step of the path runs in the CUDA library
(``csrc/``) behind the C ABI declared in ``include/pagedkv.h``.  The names
below are the C entry points; each takes torch tensors, checks their dtypes
and shapes, and passes raw pointers, sizes and the current CUDA stream.
There is no fallback: if the library is missing or cannot load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "PagedKVError", "lib", "BLOCK_SIZE", "pkv_version", "pkv_cache_bytes",
    "paged_kv_slot_mapping", "reshape_and_cache", "paged_attention_workspace_bytes",
    "paged_attention_min_partition_blocks", "paged_attention_decode",
    "paged_attention_decode_partitioned", "paged_attention_partition_pass",
    "paged_attention_merge_pass", "paged_kv_write_new_tokens", "paged_kv_decode_step",
    "paged_kv_decode_step_partition_pass", "paged_kv_decode_step_layers",
    "paged_attention_cascade_workspace_bytes", "paged_attention_decode_cascade",
    "paged_kv_decode_step_cascade", "new_cascade_workspace", "paged_attention_prefill",
    "paged_kv_decode_step_staging_bytes", "paged_kv_decode_step_host", "pkv_device_status",
    "paged_kv_last_error", "pkv_selftest_bounded_wait",
    "BlockAllocator", "new_workspace", "paged_kv_block_hash", "paged_kv_copy_blocks",
    "paged_attention_decode_noalloc", "paged_attention_noalloc_scratch_bytes",
    "PKV_OK", "PKV_ERR_INVALID_ARG", "PKV_ERR_UNSUPPORTED", "PKV_ERR_NO_BLOCKS",
    "PKV_ERR_BAD_BLOCK_ID", "PKV_ERR_CUDA", "PKV_ERR_WORKSPACE",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")
BLOCK_SIZE = 16

PKV_F16, PKV_BF16 = 0, 1
# pkv_status codes
(PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_NO_BLOCKS, PKV_ERR_BAD_BLOCK_ID,
 PKV_ERR_CUDA, PKV_ERR_WORKSPACE) = range(7)
DEV_BAD_BLOCK_ID, DEV_BAD_LENGTH, DEV_BAD_SLOT, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "not enough free blocks",
           4: "bad block id", 5: "CUDA error", 6: "workspace missing or too small"}


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_STATUS.get(status, 'unknown status')} (status {status})")
        self.status = status


_lib = None

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "pkv_version": ([], _i),
    "pkv_status_string": ([_i], ctypes.c_char_p),
    "pkv_cache_bytes": ([_i, _i, _i, _i, _i, _i], _sz),
    "paged_kv_alloc_create": ([_i, ctypes.POINTER(_vp)], _i),
    "paged_kv_alloc_destroy": ([_vp], None),
    "paged_kv_alloc": ([_vp, _i, _vp], _i),
    "paged_kv_share": ([_vp, _i, _vp], _i),
    "paged_kv_free": ([_vp, _i, _vp], _i),
    "paged_kv_num_free": ([_vp], _i),
    "paged_kv_refcount": ([_vp, ctypes.c_int32], _i),
    "paged_kv_slot_mapping": ([_vp, _i, _vp, _i, _i, _vp, _vp], _i),
    "reshape_and_cache": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp], _i),
    "paged_attention_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "paged_attention_min_partition_blocks": ([_i], _i),
    "paged_attention_decode": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _f, _vp,
                                _vp, _sz, _i, _vp], _i),
    "paged_attention_decode_partitioned": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i,
                                            _i, _f, _vp, _vp, _sz, _i, _i, _vp], _i),
    "paged_kv_decode_step": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                              _f, _vp, _vp, _vp, _sz, _i, _vp], _i),
    "paged_attention_partition_pass": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                        _f, _vp, _vp, _sz, _i, _i, _vp], _i),
    "paged_attention_merge_pass": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _f,
                                    _vp, _vp, _sz, _i, _i, _vp], _i),
    "paged_kv_write_new_tokens": ([_vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _i,
                                   _vp], _i),
    "paged_kv_decode_step_partition_pass": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i,
                                             _i, _i, _i, _f, _vp, _vp, _vp, _sz, _i, _vp], _i),
    "paged_kv_decode_step_layers": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i,
                                     _i, _i, _f, _vp, _vp, _sz, _i, _vp], _i),
    "paged_attention_cascade_workspace_bytes": ([_i, _i, _i, _i, _i], _sz),
    "paged_attention_decode_cascade": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _i,
                                        _f, _vp, _vp, _sz, _i, _vp], _i),
    "paged_kv_decode_step_cascade": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i,
                                      _i, _i, _f, _vp, _vp, _vp, _sz, _i, _vp], _i),
    "paged_attention_prefill": ([_vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                 _f, _vp, _i, _vp], _i),
    "paged_kv_decode_step_staging_bytes": ([_i, _i, _i, _i, _i], _sz),
    "paged_kv_decode_step_host": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp, _i, _i,
                                   _i, _i, _i, _i, _i, _f, _vp, _sz, _i, _vp], _i),
    "pkv_device_status": ([ctypes.POINTER(ctypes.c_uint), _i], _i),
    "paged_kv_last_error": ([ctypes.c_void_p], _i),
    "pkv_selftest_bounded_wait": ([ctypes.c_void_p], _i),
    "paged_kv_num_cached": ([_vp], _i),
    "paged_kv_block_hash": ([ctypes.c_uint64, _vp, _i], ctypes.c_uint64),
    "paged_kv_prefix_insert": ([_vp, ctypes.c_int32, ctypes.c_uint64], _i),
    "paged_kv_prefix_lookup": ([_vp, _i, _vp, _vp, ctypes.POINTER(_i)], _i),
    "paged_kv_cow": ([_vp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(_i)],
                     _i),
    "paged_kv_rollback": ([_vp, _vp, _i, _i, ctypes.POINTER(_i)], _i),
    "paged_kv_copy_blocks": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp], _i),
    "paged_attention_decode_noalloc": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _f,
                                        _vp, _i, _vp], _i),
    "paged_attention_noalloc_scratch_bytes": ([], _sz),
}


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(fn: str, rc: int):
    if rc != 0:
        raise PagedKVError(fn, rc)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PKV_F16
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (pass a view of one layer's pool)")
    return ctypes.c_void_p(t.data_ptr())


def _opt(t: Optional[torch.Tensor], name: str):
    return None if t is None else _dev(t, name)


def _check_slots(t: Optional[torch.Tensor], n: int, name: str):
    """An optional int64 [n] slot output (the kernels write n 8-byte slots)."""
    if t is not None and (t.dtype != torch.int64 or t.numel() != n):
        raise ValueError(f"{name} must be int64 [{n}]")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def pkv_version() -> int:
    return lib().pkv_version()


def pkv_cache_bytes(num_layers, num_blocks, num_kv_heads, head_dim, dtype=torch.bfloat16,
                    block_size=BLOCK_SIZE) -> int:
    code = PKV_BF16 if dtype == torch.bfloat16 else PKV_F16
    return lib().pkv_cache_bytes(num_layers, num_blocks, block_size, num_kv_heads, head_dim, code)


def paged_kv_slot_mapping(block_tables, context_lens, num_blocks, slot_mapping=None,
                          stream=None) -> torch.Tensor:
    """Slot of each sequence's token at position len-1 (int64, -1 for empty rows)."""
    B, MB = block_tables.shape
    _check_tables(block_tables, context_lens, B)
    _check_slots(slot_mapping, B, "slot_mapping")
    if slot_mapping is None:
        slot_mapping = torch.empty(B, dtype=torch.int64, device=block_tables.device)
    _check("paged_kv_slot_mapping", lib().paged_kv_slot_mapping(
        _dev(block_tables, "block_tables"), MB, _dev(context_lens, "context_lens"), B,
        num_blocks, _dev(slot_mapping, "slot_mapping"), _stream(stream)))
    return slot_mapping


def reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None):
    """Write k_new/v_new [T, Hkv, D] into one layer's pools [NB, 16, Hkv, D] at slot_mapping."""
    T, Hkv, D = k_new.shape
    NB = k_cache.shape[0]
    if tuple(k_cache.shape[1:]) != (BLOCK_SIZE, Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("pool shape must be [num_blocks, 16, num_kv_heads, head_dim]")
    _check_new_rows(k_new, v_new, (T, Hkv, D), k_new.dtype)
    if k_cache.dtype != k_new.dtype or v_cache.dtype != k_new.dtype:
        raise ValueError("the pools must have k_new's dtype")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T:
        raise ValueError("slot_mapping must be int64 [num_tokens]")
    _check("reshape_and_cache", lib().reshape_and_cache(
        _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(slot_mapping, "slot_mapping"), T, NB, Hkv, D,
        _dtype_code(k_new), _stream(stream)))


def paged_attention_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len) -> int:
    return lib().paged_attention_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                                 max_context_len)


def paged_attention_min_partition_blocks(max_context_len) -> int:
    return lib().paged_attention_min_partition_blocks(max_context_len)


def new_workspace(num_seqs, num_q_heads, head_dim, max_context_len, device) -> torch.Tensor:
    """A workspace tensor for paged_attention_decode (allocated by torch, caller-owned)."""
    n = paged_attention_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def _check_decode_shapes(q, k_cache, v_cache, block_tables, context_lens, out):
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if bs != BLOCK_SIZE or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("pool shape must be [num_blocks, 16, num_kv_heads, head_dim]")
    _check_tables(block_tables, context_lens, B)
    _check_dtypes(q, k_cache, v_cache, out)
    return B, Hq, Hkv, D, NB


def _check_tables(block_tables, context_lens, B):
    if (block_tables.dtype != torch.int32 or block_tables.dim() != 2
            or block_tables.shape[0] != B):
        raise ValueError("block_tables must be int32 [num_seqs, max_blocks_per_seq]")
    if context_lens.dtype != torch.int32 or context_lens.numel() != B:
        raise ValueError("context_lens must be int32 [num_seqs]")


def _check_new_rows(k_new, v_new, shape, dtype):
    if (tuple(k_new.shape) != shape or tuple(v_new.shape) != shape or k_new.dtype != dtype
            or v_new.dtype != dtype):
        raise ValueError(f"k_new/v_new must be shaped {shape} in q's dtype")


def _check_dtypes(q, k_cache, v_cache, out):
    if (out.shape != q.shape or out.dtype != q.dtype or k_cache.dtype != q.dtype
            or v_cache.dtype != q.dtype):
        raise ValueError("q, out and the pools must share one dtype; out shaped like q")


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                           scale, out, workspace, stream=None):
    """out[s, i] = softmax(scale * q[s, i] . K^T) V over the paged context of sequence s."""
    B, Hq, Hkv, D, NB = _check_decode_shapes(q, k_cache, v_cache, block_tables, context_lens,
                                             out)
    _check("paged_attention_decode", lib().paged_attention_decode(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), int(max_context_len), B, Hq, Hkv, D, NB,
        float(scale), _dev(out, "out"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return out


def _decode_pb(fn_name, q, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
               out, workspace, partition_blocks, stream):
    B, Hq, Hkv, D, NB = _check_decode_shapes(q, k_cache, v_cache, block_tables, context_lens,
                                             out)
    _check(fn_name, getattr(lib(), fn_name)(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), int(max_context_len), B, Hq, Hkv, D, NB,
        float(scale), _dev(out, "out"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), int(partition_blocks), _dtype_code(q),
        _stream(stream)))
    return out


def paged_attention_decode_partitioned(q, k_cache, v_cache, block_tables, context_lens,
                                       max_context_len, scale, out, workspace, partition_blocks,
                                       stream=None):
    """paged_attention_decode with a fixed partition length (blocks; 0 = adaptive)."""
    return _decode_pb("paged_attention_decode_partitioned", q, k_cache, v_cache, block_tables,
                      context_lens, max_context_len, scale, out, workspace, partition_blocks,
                      stream)


def paged_attention_partition_pass(q, k_cache, v_cache, block_tables, context_lens,
                                   max_context_len, scale, out, workspace, partition_blocks=0,
                                   stream=None):
    """First pass: per-partition (max, sum, unnormalised output); one-partition rows to out."""
    return _decode_pb("paged_attention_partition_pass", q, k_cache, v_cache, block_tables,
                      context_lens, max_context_len, scale, out, workspace, partition_blocks,
                      stream)


def paged_attention_merge_pass(q, k_cache, v_cache, block_tables, context_lens,
                               max_context_len, scale, out, workspace, partition_blocks=0,
                               stream=None):
    """Second pass: log-sum-exp merge of the partitions (same arguments as the first)."""
    return _decode_pb("paged_attention_merge_pass", q, k_cache, v_cache, block_tables,
                      context_lens, max_context_len, scale, out, workspace, partition_blocks,
                      stream)


def paged_kv_write_new_tokens(k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                              slot_mapping_out=None, stream=None):
    """Copy each sequence's new K/V row to the slot of position len-1."""
    B, Hkv, D = k_new.shape
    NB = k_cache.shape[0]
    if tuple(k_cache.shape[1:]) != (BLOCK_SIZE, Hkv, D) or v_cache.shape != k_cache.shape:
        raise ValueError("pool shape must be [num_blocks, 16, num_kv_heads, head_dim]")
    _check_new_rows(k_new, v_new, (B, Hkv, D), k_new.dtype)
    if k_cache.dtype != k_new.dtype or v_cache.dtype != k_new.dtype:
        raise ValueError("the pools must have k_new's dtype")
    _check_tables(block_tables, context_lens, B)
    _check_slots(slot_mapping_out, B, "slot_mapping_out")
    _check("paged_kv_write_new_tokens", lib().paged_kv_write_new_tokens(
        _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), B, NB, Hkv, D,
        _opt(slot_mapping_out, "slot_mapping_out"), _dtype_code(k_new), _stream(stream)))


def _decode_step(fn_name, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                 max_context_len, scale, out, workspace, slot_mapping_out, stream):
    B, Hq, Hkv, D, NB = _check_decode_shapes(q, k_cache, v_cache, block_tables, context_lens,
                                             out)
    _check_new_rows(k_new, v_new, (B, Hkv, D), q.dtype)
    _check_slots(slot_mapping_out, B, "slot_mapping_out")
    _check(fn_name, getattr(lib(), fn_name)(
        _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), int(max_context_len), B, Hq, Hkv, D, NB,
        float(scale), _dev(out, "out"), _opt(slot_mapping_out, "slot_mapping_out"),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dtype_code(q), _stream(stream)))
    return out


def paged_kv_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                         max_context_len, scale, out, workspace, slot_mapping_out=None,
                         stream=None):
    """Write each sequence's new K/V at position len-1, then decode attention."""
    return _decode_step("paged_kv_decode_step", q, k_new, v_new, k_cache, v_cache, block_tables,
                        context_lens, max_context_len, scale, out, workspace, slot_mapping_out,
                        stream)


def paged_kv_decode_step_partition_pass(q, k_new, v_new, k_cache, v_cache, block_tables,
                                        context_lens, max_context_len, scale, out, workspace,
                                        slot_mapping_out=None, stream=None):
    """The first kernel of paged_kv_decode_step (fused write + partition pass)."""
    return _decode_step("paged_kv_decode_step_partition_pass", q, k_new, v_new, k_cache,
                        v_cache, block_tables, context_lens, max_context_len, scale, out,
                        workspace, slot_mapping_out, stream)


def new_cascade_workspace(num_seqs, num_q_heads, head_dim, max_context_len, num_prefix_blocks,
                          device) -> torch.Tensor:
    n = lib().paged_attention_cascade_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                                      max_context_len, num_prefix_blocks)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def paged_attention_decode_cascade(q, k_cache, v_cache, block_tables, context_lens,
                                   max_context_len, num_prefix_blocks, scale, out, workspace,
                                   stream=None):
    """Decode attention when every sequence's table starts with the same
    num_prefix_blocks full blocks: the shared prefix is read once for all."""
    B, Hq, Hkv, D, NB = _check_decode_shapes(q, k_cache, v_cache, block_tables, context_lens,
                                             out)
    _check("paged_attention_decode_cascade", lib().paged_attention_decode_cascade(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), int(max_context_len), B, Hq, Hkv, D, NB,
        int(num_prefix_blocks), float(scale), _dev(out, "out"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return out


def paged_kv_decode_step_cascade(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                                 max_context_len, num_prefix_blocks, scale, out, workspace,
                                 slot_mapping_out=None, stream=None):
    """paged_kv_decode_step with the shared-prefix cascade."""
    B, Hq, Hkv, D, NB = _check_decode_shapes(q, k_cache, v_cache, block_tables, context_lens,
                                             out)
    _check_new_rows(k_new, v_new, (B, Hkv, D), q.dtype)
    _check_slots(slot_mapping_out, B, "slot_mapping_out")
    _check("paged_kv_decode_step_cascade", lib().paged_kv_decode_step_cascade(
        _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), int(max_context_len), B, Hq, Hkv, D, NB,
        int(num_prefix_blocks), float(scale), _dev(out, "out"),
        _opt(slot_mapping_out, "slot_mapping_out"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return out


def paged_attention_prefill(q, k_cache, v_cache, block_tables, context_lens, cu_q_lens,
                            max_q_len, scale, out, stream=None):
    """Causal attention of packed query chunks [rows, Hq, D] over the paged cache."""
    R, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if bs != BLOCK_SIZE or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("pool shape must be [num_blocks, 16, num_kv_heads, head_dim]")
    B = context_lens.numel()
    _check_tables(block_tables, context_lens, B)
    if cu_q_lens.dtype != torch.int32 or cu_q_lens.numel() != B + 1:
        raise ValueError("cu_q_lens must be int32 [num_seqs + 1]")
    _check_dtypes(q, k_cache, v_cache, out)
    _check("paged_attention_prefill", lib().paged_attention_prefill(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), _dev(cu_q_lens, "cu_q_lens"), B, int(max_q_len), R,
        Hq, Hkv, D, NB, float(scale), _dev(out, "out"), _dtype_code(q), _stream(stream)))
    return out


def paged_kv_decode_step_layers(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                                max_context_len, scale, out, workspace, stream=None):
    """One decode step of every layer: q/out [L,B,Hq,D], k_new/v_new [L,B,Hkv,D],
    pools [L,NB,16,Hkv,D] (layer-major); tables, lengths and workspace shared."""
    L, B, Hq, D = q.shape
    L2, NB, bs, Hkv, D2 = k_cache.shape
    if L2 != L or bs != BLOCK_SIZE or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [layers, num_blocks, 16, num_kv_heads, head_dim]")
    _check_new_rows(k_new, v_new, (L, B, Hkv, D), q.dtype)
    _check_dtypes(q, k_cache, v_cache, out)
    _check_tables(block_tables, context_lens, B)
    _check("paged_kv_decode_step_layers", lib().paged_kv_decode_step_layers(
        _dev(q, "q"), _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), int(max_context_len), B, Hq, Hkv, D, NB, L,
        float(scale), _dev(out, "out"), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dtype_code(q), _stream(stream)))
    return out


def paged_kv_decode_step_staging_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                       max_blocks_per_seq) -> int:
    return lib().paged_kv_decode_step_staging_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                    head_dim, max_blocks_per_seq)


def _host(t: torch.Tensor, name: str):
    if t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host tensor (pinned for async copies)")
    return ctypes.c_void_p(t.data_ptr())


def paged_kv_decode_step_host(q_host, k_new_host, v_new_host, block_tables_host,
                              context_lens_host, out_host, staging, k_cache, v_cache,
                              max_context_len, scale, workspace, stream=None):
    """paged_kv_decode_step with inputs/output in (pinned) host memory; enqueues only."""
    B, Hq, D = q_host.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if bs != BLOCK_SIZE or D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("pool shape must be [num_blocks, 16, num_kv_heads, head_dim]")
    _check_new_rows(k_new_host, v_new_host, (B, Hkv, D), q_host.dtype)
    _check_tables(block_tables_host, context_lens_host, B)
    _check_dtypes(q_host, k_cache, v_cache, out_host)
    _check("paged_kv_decode_step_host", lib().paged_kv_decode_step_host(
        _host(q_host, "q_host"), _host(k_new_host, "k_new_host"),
        _host(v_new_host, "v_new_host"), _host(block_tables_host, "block_tables_host"),
        _host(context_lens_host, "context_lens_host"), _host(out_host, "out_host"),
        _dev(staging, "staging"), staging.numel() * staging.element_size(),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), block_tables_host.shape[1],
        int(max_context_len), B, Hq, Hkv, D, NB, float(scale), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dtype_code(q_host), _stream(stream)))


def paged_attention_noalloc_scratch_bytes() -> int:
    """Bytes of the static scratch array paged_attention_decode_noalloc uses."""
    return int(lib().paged_attention_noalloc_scratch_bytes())


def paged_attention_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens,
                                   max_context_len, scale, out, stream=None):
    """paged_attention_decode without a workspace argument, for callers that cannot
    allocate device memory: the partials go to a static array inside the library
    (paged_attention_noalloc_scratch_bytes()).  Calls share that array, so calls
    overlapping on the GPU must not be issued; problems needing more scratch
    raise (PKV_ERR_WORKSPACE)."""
    B, Hq, Hkv, D, NB = _check_decode_shapes(q, k_cache, v_cache, block_tables, context_lens,
                                             out)
    _check("paged_attention_decode_noalloc", lib().paged_attention_decode_noalloc(
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), block_tables.shape[1],
        _dev(context_lens, "context_lens"), int(max_context_len), B, Hq, Hkv, D, NB,
        float(scale), _dev(out, "out"), _dtype_code(q), _stream(stream)))
    return out


def paged_kv_block_hash(parent_hash: int, tokens) -> int:
    """64-bit hash of one block's token ids chained with its parent block's hash."""
    arr = (ctypes.c_int32 * max(len(tokens), 1))(*[int(t) for t in tokens])
    return lib().paged_kv_block_hash(ctypes.c_uint64(parent_hash),
                                     ctypes.cast(arr, ctypes.c_void_p), len(tokens))


def paged_kv_copy_blocks(k_cache, v_cache, src_block_ids, dst_block_ids, stream=None):
    """Copy whole blocks src -> dst in both pools of one layer (device int32 id lists)."""
    NB, bs, Hkv, D = k_cache.shape
    if v_cache.shape != k_cache.shape or bs != BLOCK_SIZE:
        raise ValueError("pool shape must be [num_blocks, 16, num_kv_heads, head_dim]")
    if (src_block_ids.dtype != torch.int32 or dst_block_ids.dtype != torch.int32
            or dst_block_ids.shape != src_block_ids.shape):
        raise ValueError("block id lists must be int32 and of equal length")
    _check("paged_kv_copy_blocks", lib().paged_kv_copy_blocks(
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _dev(src_block_ids, "src"),
        _dev(dst_block_ids, "dst"), src_block_ids.numel(), NB, Hkv, D, _dtype_code(k_cache),
        _stream(stream)))


def pkv_device_status(reset: bool = True) -> int:
    """PKV_DEV_* bits set by kernels on the current device (synchronises)."""
    flags = ctypes.c_uint(0)
    _check("pkv_device_status", lib().pkv_device_status(ctypes.byref(flags), int(reset)))
    return flags.value


def paged_kv_last_error(stream=None) -> int:
    """Status code for the device checks of work on `stream` (waits for it; clears
    the device status word).  Returned, not raised: 0 means no flag was set."""
    return int(lib().paged_kv_last_error(_stream(stream)))


def pkv_selftest_bounded_wait(stream=None) -> None:
    """Enqueue the bounded-wait diagnostic (sets DEV_TIMEOUT after ~0.1 s)."""
    _check("pkv_selftest_bounded_wait", lib().pkv_selftest_bounded_wait(_stream(stream)))


class BlockAllocator:
    """Host block allocator (refcounted, all-or-nothing) over ids [0, num_blocks)."""

    def __init__(self, num_blocks: int):
        h = ctypes.c_void_p()
        _check("paged_kv_alloc_create", lib().paged_kv_alloc_create(num_blocks, ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks

    def close(self):
        if self._h:
            lib().paged_kv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _ids(ids):
        arr = (ctypes.c_int32 * len(ids))(*[int(i) for i in ids])
        return arr, ctypes.cast(arr, ctypes.c_void_p)

    def alloc(self, n: int) -> list:
        arr = (ctypes.c_int32 * max(n, 1))()
        _check("paged_kv_alloc", lib().paged_kv_alloc(self._h, n, ctypes.cast(arr, ctypes.c_void_p)))
        return list(arr[:n])

    def share(self, ids):
        arr, p = self._ids(ids)
        _check("paged_kv_share", lib().paged_kv_share(self._h, len(ids), p))

    def free(self, ids):
        arr, p = self._ids(ids)
        _check("paged_kv_free", lib().paged_kv_free(self._h, len(ids), p))

    def num_free(self) -> int:
        return lib().paged_kv_num_free(self._h)

    def refcount(self, block_id: int) -> int:
        return lib().paged_kv_refcount(self._h, block_id)

    def num_cached(self) -> int:
        return lib().paged_kv_num_cached(self._h)

    def prefix_insert(self, block_id: int, block_hash: int):
        _check("paged_kv_prefix_insert",
               lib().paged_kv_prefix_insert(self._h, block_id, ctypes.c_uint64(block_hash)))

    def prefix_lookup(self, hashes) -> list:
        """Ids of the leading cached blocks (each gains a reference); stops at a miss."""
        n = len(hashes)
        harr = (ctypes.c_uint64 * max(n, 1))(*[int(h) for h in hashes])
        out = (ctypes.c_int32 * max(n, 1))()
        hits = ctypes.c_int(0)
        _check("paged_kv_prefix_lookup", lib().paged_kv_prefix_lookup(
            self._h, n, ctypes.cast(harr, ctypes.c_void_p), ctypes.cast(out, ctypes.c_void_p),
            ctypes.byref(hits)))
        return list(out[:hits.value])

    def cow(self, block_id: int):
        """(block to write into, whether the caller must copy the old block's content)."""
        new_id = ctypes.c_int32(0)
        copy = ctypes.c_int(0)
        _check("paged_kv_cow", lib().paged_kv_cow(self._h, block_id, ctypes.byref(new_id),
                                                  ctypes.byref(copy)))
        return new_id.value, bool(copy.value)

    def rollback(self, table, new_len: int):
        """Drop the blocks past new_len tokens; returns the kept table."""
        arr = (ctypes.c_int32 * max(len(table), 1))(*[int(b) for b in table])
        keep = ctypes.c_int(0)
        _check("paged_kv_rollback", lib().paged_kv_rollback(
            self._h, ctypes.cast(arr, ctypes.c_void_p), len(table), new_len, ctypes.byref(keep)))
        return list(arr[:keep.value])
