"""ctypes binding of ``libpa.so`` (``include/pa.h``), same names as the C ABI.

Argument marshalling only: these functions check that tensors have the
dtype, device and contiguity the C ABI expects, pass raw pointers, sizes and
the current CUDA stream, and turn a non-OK status into an exception.  Every
step of the computation runs in the library's CUDA kernels; there is no
fallback.  If ``libpa.so`` has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

LIBRARY = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa.so")

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_WORKSPACE",
                4: "PA_ERR_CUDA", 5: "PA_ERR_DEVICE", 6: "PA_ERR_NO_BLOCKS", 7: "PA_ERR_NOT_FOUND",
                8: "PA_ERR_SWAPPED"}
PA_SWAP_OUT, PA_SWAP_IN = 0, 1
PA_DECODE_EARLY_METADATA = 0x1
DEVERR_BLOCK_ID, DEVERR_SLOT, DEVERR_SEQ_LEN, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
PA_DTYPE_BF16 = 0

# Every function declared in include/pa.h with (restype, argtypes).
_P, _I64, _I32, _U32, _F, _SZ = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                                  ctypes.c_float, ctypes.c_size_t)


class PaCapacity(ctypes.Structure):
    """``pa_capacity``: contiguous against paged capacity of a KV budget."""
    _fields_ = [("contiguous_requests", ctypes.c_int64), ("paged_requests", ctypes.c_int64),
                ("contiguous_waste", ctypes.c_double), ("paged_waste", ctypes.c_double),
                ("mean_tail_slots", ctypes.c_double), ("prefix_bytes_contiguous", ctypes.c_double),
                ("prefix_bytes_paged", ctypes.c_double)]


class PaKvPool(ctypes.Structure):
    """``pa_kv_pool``: one layer's view of the block pool (strides in elements)."""
    _fields_ = [("base", ctypes.c_void_p), ("num_blocks", ctypes.c_int64), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("block_stride", ctypes.c_int64), ("kv_stride", ctypes.c_int64)]


_POOL = ctypes.POINTER(PaKvPool)
SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [_I32]),
    "pa_version": (_I32, []),
    "pa_reshape_and_cache": (_I32, [_POOL, _P, _P, _P, _I64, _P]),
    "pa_decode_workspace_size": (_SZ, [_POOL, _I32, _I32, _I32, _I32]),
    "pa_decode_partition_tokens": (_I32, [_POOL, _I32, _I32, _I32, _I32]),
    "pa_decode": (_I32, [_P, _P, _POOL, _P, _I32, _P, _I32, _I32, _I32, _F, _I32, _P, _SZ, _P]),
    "pa_decode_ex": (_I32, [_P, _P, _POOL, _P, _I32, _P, _I32, _I32, _I32, _F, _I32, _P, _SZ, _P, _P, _U32, _P]),
    "pa_decode_host_staging_size": (_SZ, [_POOL, _I32, _I32, _I32]),
    "pa_decode_host": (_I32, [_P, _P, _POOL, _P, _I32, _P, _I32, _I32, _I32, _F, _I32, _P, _P, _U32, _P, _SZ, _P, _SZ,
                              _P]),
    "pa_decode_noalloc": (_I32, [_P, _P, _POOL, _P, _I32, _P, _I32, _I32, _I32, _F, _I32, _P]),
    "pa_copy_blocks": (_I32, [_POOL, _P, _I32, _P]),
    "pa_swap_blocks": (_I32, [_POOL, _P, _I64, _P, _I32, _I32, _P]),
    "pa_prefill_chunk": (_I32, [_P, _P, _POOL, _P, _I32, _P, _I32, _I32, _I32, _I32, _F, _P]),
    "pa_prefix_attention": (_I32, [_P, _P, _P, _POOL, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _F, _P]),
    "pa_decode_cascade": (_I32, [_P, _P, _POOL, _P, _I32, _P, _I32, _I32, _I32, _F, _I32, _P, _SZ, _P, _P, _P, _P,
                                 _U32, _P]),
    "pa_cascade_plan": (_I32, [_P, _I32, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "pa_decode_grouped": (_I32, [_P, _P, _POOL, _P, _I32, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _F,
                                 _P, _P, _U32, _P]),
    "pa_get_device_error": (_I32, [ctypes.POINTER(_U32), _I32, _P]),
    "pa_check_wait_timeout": (_I32, [ctypes.c_uint64, _P]),
    "pa_set_stream_k_ctas": (_I32, [_I32]),
    "pa_set_prefill_ctas": (_I32, [_I32]),
    "pa_block_layout": (_I32, [_I64, _I32, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "pa_slot_mapping": (_I32, [_P, _P, _I32, _I32, _P, _P, _I64, _I32, _I64]),
    "pa_bm_create": (_I32, [ctypes.POINTER(_P), _I64, _I32]),
    "pa_bm_destroy": (None, [_P]),
    "pa_bm_add_seq": (_I32, [_P, ctypes.POINTER(_I32)]),
    "pa_bm_append_tokens": (_I32, [_P, _I32, _I64, _P, _P, ctypes.POINTER(_I32)]),
    "pa_bm_fork": (_I32, [_P, _I32, ctypes.POINTER(_I32)]),
    "pa_bm_free_seq": (_I32, [_P, _I32]),
    "pa_bm_get_table": (_I32, [_P, _I32, _P, _I32, ctypes.POINTER(_I32), ctypes.POINTER(_I64)]),
    "pa_bm_num_free": (_I64, [_P]),
    "pa_bm_refcount": (_I32, [_P, _I64]),
    "pa_bm_can_admit": (_I32, [_P, _I64, _I64, ctypes.POINTER(_I32)]),
    "pa_bm_set_host_pool": (_I32, [_P, _I64]),
    "pa_bm_swap_out": (_I32, [_P, _I32, _P, _I32, ctypes.POINTER(_I32)]),
    "pa_bm_swap_in": (_I32, [_P, _I32, _P, _I32, ctypes.POINTER(_I32)]),
    "pa_bm_num_free_host": (_I64, [_P]),
    "pa_bm_is_swapped": (_I32, [_P, _I32]),
    "pa_bm_prefix_match": (_I32, [_P, _P, _I64, ctypes.c_uint64, ctypes.POINTER(_I64)]),
    "pa_bm_add_seq_cached": (_I32, [_P, _P, _I64, ctypes.c_uint64, ctypes.POINTER(_I32), ctypes.POINTER(_I64)]),
    "pa_bm_cache_seq": (_I32, [_P, _I32, _P, _I64, ctypes.c_uint64, ctypes.POINTER(_I64)]),
    "pa_bm_prefix_evict": (_I32, [_P, _I64, ctypes.POINTER(_I64)]),
    "pa_bm_num_cached": (_I64, [_P]),
    "pa_bm_num_evictable": (_I64, [_P]),
    "pa_bm_prefix_stats": (_I32, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "pa_capacity_estimate": (_I32, [_P, _I64, _I64, _I32, _I64, _I64, _I64, ctypes.POINTER(PaCapacity)]),
}


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(f"{LIBRARY} is missing: build it with paged_kv_cache_167_gb300.build.build()")
        handle = ctypes.CDLL(LIBRARY)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttentionError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _dev(t: torch.Tensor, dtype, name: str) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _host(t: torch.Tensor, dtype, name: str) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a CPU tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


# ---------------------------------------------------------------------------
# pool descriptor
# ---------------------------------------------------------------------------

def pool_desc(pool: torch.Tensor, layer: Optional[int] = None) -> PaKvPool:
    """Descriptor of a bf16 pool tensor.

    ``pool`` is [NB][2][Hkv][b][d] (one layer) or the layered
    [NB][2][L][Hkv][b][d]; for the latter ``layer`` picks the layer's view.
    """
    _dev(pool, torch.bfloat16, "pool")
    if pool.dim() == 5:
        nb, two, hkv, b, d = pool.shape
        base, bstride, kvstride = pool.data_ptr(), 0, 0
    elif pool.dim() == 6:
        if layer is None:
            raise ValueError("layer is required for a layered pool")
        nb, two, nl, hkv, b, d = pool.shape
        if not 0 <= layer < nl:
            raise ValueError("layer out of range")
        slab = hkv * b * d
        base = pool.data_ptr() + layer * slab * pool.element_size()
        bstride, kvstride = 2 * nl * slab, nl * slab
    else:
        raise ValueError("pool must be [NB][2][Hkv][b][d] or [NB][2][L][Hkv][b][d]")
    if two != 2:
        raise ValueError("pool dim 1 must be 2 (K, V)")
    return PaKvPool(base, nb, hkv, b, d, PA_DTYPE_BF16, bstride, kvstride)


# ---------------------------------------------------------------------------
# device calls
# ---------------------------------------------------------------------------

def reshape_and_cache(pool: torch.Tensor, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                      layer: Optional[int] = None, stream=None) -> None:
    desc = pool_desc(pool, layer)
    n = k.shape[0]
    if v.shape != k.shape or slot_mapping.numel() != n:
        raise ValueError("k, v and slot_mapping disagree on the token count")
    _check(lib().pa_reshape_and_cache(ctypes.byref(desc), _dev(k, torch.bfloat16, "k"),
                                      _dev(v, torch.bfloat16, "v"),
                                      _dev(slot_mapping, torch.int64, "slot_mapping"), n, _stream(stream)),
           "pa_reshape_and_cache")


def decode_workspace_size(pool: torch.Tensor, num_seqs: int, num_q_heads: int, max_seq_len: int,
                          partition_tokens: int = 0, layer: Optional[int] = None) -> int:
    desc = pool_desc(pool, layer)
    return int(lib().pa_decode_workspace_size(ctypes.byref(desc), num_seqs, num_q_heads, max_seq_len,
                                              partition_tokens))


def decode_partition_tokens(pool: torch.Tensor, num_seqs: int, num_q_heads: int, max_seq_len: int,
                            partition_tokens: int = 0, layer: Optional[int] = None) -> int:
    desc = pool_desc(pool, layer)
    return int(lib().pa_decode_partition_tokens(ctypes.byref(desc), num_seqs, num_q_heads, max_seq_len,
                                                partition_tokens))


def decode(out: torch.Tensor, q: torch.Tensor, pool: torch.Tensor, block_tables: torch.Tensor,
           seq_lens: torch.Tensor, max_seq_len: int, scale: float, partition_tokens: int = 0,
           workspace: Optional[torch.Tensor] = None, layer: Optional[int] = None, stream=None,
           flags: int = 0, new_k: Optional[torch.Tensor] = None, new_v: Optional[torch.Tensor] = None) -> None:
    """pa_decode (pa_decode_ex when ``flags``, ``new_k`` or ``new_v`` is given).
    ``workspace`` is a uint8 CUDA tensor of at least decode_workspace_size(...)
    bytes (None when that size is 0); ``new_k`` / ``new_v`` ([B][Hkv][d] bf16)
    are stored at each sequence's last position before attending."""
    desc = pool_desc(pool, layer)
    B, Hq, _ = q.shape
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("block_tables / seq_lens do not match the batch")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, torch.uint8, "workspace"), workspace.numel()
    args = (_dev(out, torch.bfloat16, "out"), _dev(q, torch.bfloat16, "q"), ctypes.byref(desc),
            _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
            _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, int(max_seq_len), float(scale), int(partition_tokens),
            ws_ptr, ws_bytes)
    if flags or new_k is not None or new_v is not None:
        nk = _dev(new_k, torch.bfloat16, "new_k") if new_k is not None else ctypes.c_void_p(0)
        nv = _dev(new_v, torch.bfloat16, "new_v") if new_v is not None else ctypes.c_void_p(0)
        for name, t in (("new_k", new_k), ("new_v", new_v)):
            if t is not None and (t.dim() != 3 or t.shape[0] != B or t.shape[1:] != (desc.num_kv_heads, desc.head_dim)):
                raise ValueError(f"{name} must be [num_seqs][num_kv_heads][head_dim]")
        _check(lib().pa_decode_ex(*args, nk, nv, int(flags), _stream(stream)), "pa_decode_ex")
    else:
        _check(lib().pa_decode(*args, _stream(stream)), "pa_decode")


def decode_host_staging_size(pool: torch.Tensor, num_seqs: int, num_q_heads: int, max_blocks_per_seq: int,
                             layer: Optional[int] = None) -> int:
    desc = pool_desc(pool, layer)
    return int(lib().pa_decode_host_staging_size(ctypes.byref(desc), num_seqs, num_q_heads, max_blocks_per_seq))


def decode_host(out_host: torch.Tensor, q_host: torch.Tensor, pool: torch.Tensor, tables_host: torch.Tensor,
                seq_lens_host: torch.Tensor, max_seq_len: int, scale: float, staging: torch.Tensor,
                partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None, layer: Optional[int] = None,
                stream=None, flags: int = 0, new_k_host: Optional[torch.Tensor] = None,
                new_v_host: Optional[torch.Tensor] = None) -> None:
    """pa_decode_host: one decode step from host (ideally pinned) tensors; the
    output lands in ``out_host`` once ``stream`` has been synchronised.
    ``staging`` is a uint8 CUDA tensor of decode_host_staging_size(...) bytes."""
    desc = pool_desc(pool, layer)
    B, Hq, _ = q_host.shape
    if out_host.shape != q_host.shape:
        raise ValueError("out_host must have q_host's shape")
    if tables_host.dim() != 2 or tables_host.shape[0] != B or seq_lens_host.numel() != B:
        raise ValueError("tables_host / seq_lens_host do not match the batch")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, torch.uint8, "workspace"), workspace.numel()
    nk = _host(new_k_host, torch.bfloat16, "new_k_host") if new_k_host is not None else ctypes.c_void_p(0)
    nv = _host(new_v_host, torch.bfloat16, "new_v_host") if new_v_host is not None else ctypes.c_void_p(0)
    _check(lib().pa_decode_host(_host(out_host, torch.bfloat16, "out_host"), _host(q_host, torch.bfloat16, "q_host"),
                                ctypes.byref(desc), _host(tables_host, torch.int32, "tables_host"),
                                tables_host.shape[1], _host(seq_lens_host, torch.int32, "seq_lens_host"), B, Hq,
                                int(max_seq_len), float(scale), int(partition_tokens), nk, nv, int(flags),
                                _dev(staging, torch.uint8, "staging"), staging.numel(), ws_ptr, ws_bytes,
                                _stream(stream)), "pa_decode_host")


def decode_noalloc(out: torch.Tensor, q: torch.Tensor, pool: torch.Tensor, block_tables: torch.Tensor,
                   seq_lens: torch.Tensor, max_seq_len: int, scale: float, partition_tokens: int = 0,
                   layer: Optional[int] = None, stream=None) -> None:
    """pa_decode_noalloc: pa_decode with its partials in the library's fixed
    8 MiB device array, for callers that cannot allocate a workspace."""
    desc = pool_desc(pool, layer)
    B, Hq, _ = q.shape
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("block_tables / seq_lens do not match the batch")
    _check(lib().pa_decode_noalloc(_dev(out, torch.bfloat16, "out"), _dev(q, torch.bfloat16, "q"),
                                   ctypes.byref(desc), _dev(block_tables, torch.int32, "block_tables"),
                                   block_tables.shape[1], _dev(seq_lens, torch.int32, "seq_lens"), B, Hq,
                                   int(max_seq_len), float(scale), int(partition_tokens), _stream(stream)),
           "pa_decode_noalloc")


def copy_blocks(pool: torch.Tensor, pairs: torch.Tensor, layer: Optional[int] = None, stream=None) -> None:
    desc = pool_desc(pool, layer)
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [n][2]")
    _check(lib().pa_copy_blocks(ctypes.byref(desc), _dev(pairs, torch.int32, "pairs"), pairs.shape[0],
                                _stream(stream)), "pa_copy_blocks")


def swap_blocks(pool: torch.Tensor, host: torch.Tensor, pairs: torch.Tensor, direction: int,
                layer: Optional[int] = None, stream=None) -> None:
    """pa_swap_blocks.  ``host`` is a pinned CPU bf16 tensor of
    [host_blocks][2][Hkv][b][d]; ``pairs`` a CUDA int32 [n][2] of
    (device block, host block); ``direction`` PA_SWAP_OUT or PA_SWAP_IN."""
    desc = pool_desc(pool, layer)
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [n][2]")
    if host.device.type != "cpu" or host.dtype != torch.bfloat16 or not host.is_contiguous():
        raise ValueError("host must be a contiguous bf16 CPU tensor")
    if host.dim() != 5 or tuple(host.shape[1:]) != (2, desc.num_kv_heads, desc.block_size, desc.head_dim):
        raise ValueError("host must be [host_blocks][2][Hkv][b][d]")
    _check(lib().pa_swap_blocks(ctypes.byref(desc), ctypes.c_void_p(host.data_ptr()), host.shape[0],
                                _dev(pairs, torch.int32, "pairs"), pairs.shape[0], int(direction),
                                _stream(stream)), "pa_swap_blocks")


def prefill_chunk(out: torch.Tensor, q: torch.Tensor, pool: torch.Tensor, block_tables: torch.Tensor,
                  ctx_lens: torch.Tensor, max_ctx_len: int, scale: float, layer: Optional[int] = None,
                  stream=None) -> None:
    desc = pool_desc(pool, layer)
    B, C, Hq, _ = q.shape
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or ctx_lens.numel() != B:
        raise ValueError("block_tables / ctx_lens do not match the batch")
    _check(lib().pa_prefill_chunk(_dev(out, torch.bfloat16, "out"), _dev(q, torch.bfloat16, "q"),
                                  ctypes.byref(desc), _dev(block_tables, torch.int32, "block_tables"),
                                  block_tables.shape[1], _dev(ctx_lens, torch.int32, "ctx_lens"), B, C, Hq,
                                  int(max_ctx_len), float(scale), _stream(stream)), "pa_prefill_chunk")


def prefix_attention(o_part: torch.Tensor, lse: torch.Tensor, q: torch.Tensor, pool: torch.Tensor,
                     prefix_tables: torch.Tensor, prefix_lens: torch.Tensor, group_size: int, max_prefix_len: int,
                     scale: float, group_order: Optional[torch.Tensor] = None, layer: Optional[int] = None,
                     stream=None) -> None:
    """pa_prefix_attention: q [num_groups * group_size][Hq][d] bf16 (sequences
    group by group); o_part fp32 of q's shape, lse fp32 [B][Hq]; group_order
    an int32 CUDA permutation of the groups (the order their CTAs start) or None."""
    desc = pool_desc(pool, layer)
    B, Hq, _ = q.shape
    if group_size <= 0 or B % group_size != 0:
        raise ValueError("the batch must be whole groups")
    G = B // group_size
    if o_part.shape != q.shape or tuple(lse.shape) != (B, Hq):
        raise ValueError("o_part must have q's shape and lse [B][Hq]")
    if prefix_tables.dim() != 2 or prefix_tables.shape[0] != G or prefix_lens.numel() != G:
        raise ValueError("prefix_tables / prefix_lens do not match the groups")
    if group_order is not None and group_order.numel() != G:
        raise ValueError("group_order must hold one entry per group")
    order = _dev(group_order, torch.int32, "group_order") if group_order is not None else ctypes.c_void_p(0)
    _check(lib().pa_prefix_attention(_dev(o_part, torch.float32, "o_part"), _dev(lse, torch.float32, "lse"),
                                     _dev(q, torch.bfloat16, "q"), ctypes.byref(desc),
                                     _dev(prefix_tables, torch.int32, "prefix_tables"), prefix_tables.shape[1],
                                     _dev(prefix_lens, torch.int32, "prefix_lens"), order, G, int(group_size), Hq,
                                     int(max_prefix_len), float(scale), _stream(stream)), "pa_prefix_attention")


def decode_cascade(out: torch.Tensor, q: torch.Tensor, pool: torch.Tensor, suffix_tables: torch.Tensor,
                   suffix_lens: torch.Tensor, max_suffix_len: int, scale: float, prefix_o: torch.Tensor,
                   prefix_lse: torch.Tensor, partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                   layer: Optional[int] = None, stream=None, flags: int = 0, new_k: Optional[torch.Tensor] = None,
                   new_v: Optional[torch.Tensor] = None) -> None:
    """pa_decode_cascade: decode over each sequence's suffix with the prefix
    partial (prefix_attention's o_part and lse) folded into every row."""
    desc = pool_desc(pool, layer)
    B, Hq, _ = q.shape
    if out.shape != q.shape or prefix_o.shape != q.shape or tuple(prefix_lse.shape) != (B, Hq):
        raise ValueError("out and prefix_o must have q's shape, prefix_lse [B][Hq]")
    if suffix_tables.dim() != 2 or suffix_tables.shape[0] != B or suffix_lens.numel() != B:
        raise ValueError("suffix_tables / suffix_lens do not match the batch")
    for name, t in (("new_k", new_k), ("new_v", new_v)):
        if t is not None and (t.dim() != 3 or t.shape[0] != B or t.shape[1:] != (desc.num_kv_heads, desc.head_dim)):
            raise ValueError(f"{name} must be [num_seqs][num_kv_heads][head_dim]")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, torch.uint8, "workspace"), workspace.numel()
    nk = _dev(new_k, torch.bfloat16, "new_k") if new_k is not None else ctypes.c_void_p(0)
    nv = _dev(new_v, torch.bfloat16, "new_v") if new_v is not None else ctypes.c_void_p(0)
    _check(lib().pa_decode_cascade(_dev(out, torch.bfloat16, "out"), _dev(q, torch.bfloat16, "q"),
                                   ctypes.byref(desc), _dev(suffix_tables, torch.int32, "suffix_tables"),
                                   suffix_tables.shape[1], _dev(suffix_lens, torch.int32, "suffix_lens"), B, Hq,
                                   int(max_suffix_len), float(scale), int(partition_tokens), ws_ptr, ws_bytes,
                                   _dev(prefix_o, torch.float32, "prefix_o"),
                                   _dev(prefix_lse, torch.float32, "prefix_lse"), nk, nv, int(flags),
                                   _stream(stream)), "pa_decode_cascade")


def decode_grouped(out: torch.Tensor, q: torch.Tensor, pool: torch.Tensor, prefix_tables: torch.Tensor,
                   prefix_lens: torch.Tensor, suffix_tables: torch.Tensor, suffix_lens: torch.Tensor, group_size: int,
                   max_prefix_len: int, max_suffix_len: int, scale: float,
                   group_order: Optional[torch.Tensor] = None, new_k: Optional[torch.Tensor] = None,
                   new_v: Optional[torch.Tensor] = None, layer: Optional[int] = None, flags: int = 0,
                   stream=None) -> None:
    """pa_decode_grouped: each group's queries over its shared prefix and each
    member's own suffix in one call (the cascade fused, for short suffixes).
    flags: 0 or PA_DECODE_EARLY_METADATA."""
    desc = pool_desc(pool, layer)
    B, Hq, _ = q.shape
    if group_size <= 0 or B % group_size != 0:
        raise ValueError("the batch must be whole groups")
    G = B // group_size
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if prefix_tables.dim() != 2 or prefix_tables.shape[0] != G or prefix_lens.numel() != G:
        raise ValueError("prefix_tables / prefix_lens do not match the groups")
    if suffix_tables.dim() != 2 or suffix_tables.shape[0] != B or suffix_lens.numel() != B:
        raise ValueError("suffix_tables / suffix_lens do not match the batch")
    if group_order is not None and group_order.numel() != G:
        raise ValueError("group_order must hold one entry per group")
    for name, t in (("new_k", new_k), ("new_v", new_v)):
        if t is not None and (t.dim() != 3 or t.shape[0] != B or t.shape[1:] != (desc.num_kv_heads, desc.head_dim)):
            raise ValueError(f"{name} must be [num_seqs][num_kv_heads][head_dim]")
    order = _dev(group_order, torch.int32, "group_order") if group_order is not None else ctypes.c_void_p(0)
    nk = _dev(new_k, torch.bfloat16, "new_k") if new_k is not None else ctypes.c_void_p(0)
    nv = _dev(new_v, torch.bfloat16, "new_v") if new_v is not None else ctypes.c_void_p(0)
    _check(lib().pa_decode_grouped(_dev(out, torch.bfloat16, "out"), _dev(q, torch.bfloat16, "q"),
                                   ctypes.byref(desc), _dev(prefix_tables, torch.int32, "prefix_tables"),
                                   prefix_tables.shape[1], _dev(prefix_lens, torch.int32, "prefix_lens"), order,
                                   _dev(suffix_tables, torch.int32, "suffix_tables"), suffix_tables.shape[1],
                                   _dev(suffix_lens, torch.int32, "suffix_lens"), G, int(group_size), Hq,
                                   int(max_prefix_len), int(max_suffix_len), float(scale), nk, nv, int(flags),
                                   _stream(stream)),
           "pa_decode_grouped")


def cascade_plan(tables, seq_lens, group_size: int, block_size: int) -> dict:
    """pa_cascade_plan on host arrays: the prefix each group of ``group_size``
    consecutive sequences shares (whole blocks, leaving every member at least
    one token) and the suffixes.  Returns numpy int32 arrays prefix_tables
    [G][W], prefix_lens [G], group_order [G] (longest prefix first),
    suffix_tables [B][W], suffix_lens [B]."""
    t = np.ascontiguousarray(np.asarray(tables, dtype=np.int32))
    L = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(-1))
    if t.ndim != 2 or t.shape[0] != L.shape[0]:
        raise ValueError("tables must be [B][W] with one length per row")
    B, W = t.shape
    if group_size <= 0 or B % group_size != 0:
        raise ValueError("the batch must be whole groups")
    G = B // group_size
    pt = np.empty((G, W), np.int32)
    pl = np.empty(G, np.int32)
    go = np.empty(G, np.int32)
    st = np.empty((B, W), np.int32)
    sl = np.empty(B, np.int32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    _check(lib().pa_cascade_plan(ptr(t), W, ptr(L), B, int(group_size), int(block_size), ptr(pt), ptr(pl), ptr(go),
                                 ptr(st), ptr(sl)), "pa_cascade_plan")
    return {"prefix_tables": pt, "prefix_lens": pl, "group_order": go, "suffix_tables": st, "suffix_lens": sl}


def check_wait_timeout(limit_ns: int, stream=None) -> None:
    """pa_check_wait_timeout: a wait that nothing completes gives up after
    ``limit_ns`` and records PA_DEVERR_TIMEOUT in the error word."""
    _check(lib().pa_check_wait_timeout(int(limit_ns), _stream(stream)), "pa_check_wait_timeout")


def set_stream_k_ctas(ctas: int) -> None:
    """pa_set_stream_k_ctas (testing hook): fix the balanced decode grid at
    ``ctas`` CTAs for later calls in this process; 0 restores the default."""
    _check(lib().pa_set_stream_k_ctas(int(ctas)), "pa_set_stream_k_ctas")


def set_prefill_ctas(ctas: int) -> None:
    """pa_set_prefill_ctas (testing hook): fix the persistent grid of the
    tensor-core prefill / prefix / grouped kernel at `ctas` CTAs (0 restores
    one per SM)."""
    _check(lib().pa_set_prefill_ctas(int(ctas)), "pa_set_prefill_ctas")


def get_device_error(clear: bool = True, stream=None) -> int:
    """The current device's error word (PA_DEVERR_* bits); synchronises."""
    word = ctypes.c_uint32(0)
    status = lib().pa_get_device_error(ctypes.byref(word), 1 if clear else 0, _stream(stream))
    if status not in (PA_OK, 5):
        raise PagedAttentionError(status, "pa_get_device_error")
    return int(word.value)


# ---------------------------------------------------------------------------
# host helpers
# ---------------------------------------------------------------------------

def block_layout(tokens: int, block_size: int):
    blocks, unused = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().pa_block_layout(tokens, block_size, ctypes.byref(blocks), ctypes.byref(unused)),
           "pa_block_layout")
    return blocks.value, unused.value


def slot_mapping(tables: np.ndarray, seq_idx: Sequence[int], positions: Sequence[int], block_size: int,
                 num_blocks: int) -> np.ndarray:
    """Host slot mapping (int64 numpy array) for (sequence, position) pairs."""
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    seq_idx = np.ascontiguousarray(seq_idx, dtype=np.int32)
    positions = np.ascontiguousarray(positions, dtype=np.int64)
    out = np.empty(len(positions), dtype=np.int64)
    _check(lib().pa_slot_mapping(out.ctypes.data_as(_P), tables.ctypes.data_as(_P), tables.shape[0],
                                 tables.shape[1], seq_idx.ctypes.data_as(_P), positions.ctypes.data_as(_P),
                                 len(positions), block_size, num_blocks), "pa_slot_mapping")
    return out


def capacity_estimate(lens: Sequence[int], shared_prefix_tokens: int, block_size: int, max_seq_len: int,
                      bytes_per_token: int, budget_bytes: int) -> dict:
    """Contiguous against paged capacity of a KV budget for the length mix
    ``lens`` (``pa_capacity_estimate``), as a dict of the struct's fields."""
    lens = np.ascontiguousarray(lens, dtype=np.int64)
    out = PaCapacity()
    _check(lib().pa_capacity_estimate(lens.ctypes.data_as(_P), len(lens), shared_prefix_tokens, block_size,
                                      max_seq_len, bytes_per_token, budget_bytes, ctypes.byref(out)),
           "pa_capacity_estimate")
    return {name: getattr(out, name) for name, _ in PaCapacity._fields_}
