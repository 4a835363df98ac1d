"""Python handle on the host block manager (``pa_bm_*`` in ``include/pa.h``).

Marshalling only; the free list, reference counts, forks, copy-on-write
planning, swapping and the prefix-cache index live in
``csrc/pa_block_manager.cpp``.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import numpy as np

from .binding import PagedAttentionError, _check, lib

_I32, _I64 = ctypes.c_int32, ctypes.c_int64


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        handle = ctypes.c_void_p()
        _check(lib().pa_bm_create(ctypes.byref(handle), num_blocks, block_size), "pa_bm_create")
        self._h = handle
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if self._h:
            lib().pa_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass

    def add_seq(self) -> int:
        sid = _I32()
        _check(lib().pa_bm_add_seq(self._h, ctypes.byref(sid)), "pa_bm_add_seq")
        return sid.value

    def append_tokens(self, seq: int, n: int) -> Tuple[np.ndarray, Optional[Tuple[int, int]]]:
        """Appends n tokens; returns their slots and the (src, dst) copy-on-write
        pair to run through copy_blocks first, if any."""
        slots = np.empty(n, dtype=np.int64)
        pair = (ctypes.c_int32 * 2)()
        ncow = _I32()
        _check(lib().pa_bm_append_tokens(self._h, seq, n, slots.ctypes.data_as(ctypes.c_void_p),
                                         ctypes.cast(pair, ctypes.c_void_p), ctypes.byref(ncow)),
               "pa_bm_append_tokens")
        return slots, ((pair[0], pair[1]) if ncow.value else None)

    def fork(self, parent: int) -> int:
        child = _I32()
        _check(lib().pa_bm_fork(self._h, parent, ctypes.byref(child)), "pa_bm_fork")
        return child.value

    def free_seq(self, seq: int) -> None:
        _check(lib().pa_bm_free_seq(self._h, seq), "pa_bm_free_seq")

    def table(self, seq: int) -> Tuple[np.ndarray, int]:
        """(physical block ids, token count) of a sequence."""
        nb, nt = _I32(), _I64()
        _check(lib().pa_bm_get_table(self._h, seq, None, 0, ctypes.byref(nb), ctypes.byref(nt)),
               "pa_bm_get_table")
        out = np.empty(max(nb.value, 1), dtype=np.int32)
        _check(lib().pa_bm_get_table(self._h, seq, out.ctypes.data_as(ctypes.c_void_p), nb.value, None, None),
               "pa_bm_get_table")
        return out[:nb.value], nt.value

    def num_free(self) -> int:
        return int(lib().pa_bm_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(lib().pa_bm_refcount(self._h, block))

    def can_admit(self, prompt_tokens: int, watermark_blocks: int = 0) -> bool:
        ok = _I32()
        _check(lib().pa_bm_can_admit(self._h, prompt_tokens, watermark_blocks, ctypes.byref(ok)),
               "pa_bm_can_admit")
        return bool(ok.value)

    # ---- swapping to a pinned host buffer (see pa_bm_swap_out / pa_bm_swap_in)

    def set_host_pool(self, host_blocks: int) -> None:
        _check(lib().pa_bm_set_host_pool(self._h, host_blocks), "pa_bm_set_host_pool")

    def _swap(self, fn, name: str, seq: int) -> np.ndarray:
        cap = self.num_blocks   # a sequence never holds more blocks than the pool
        pairs = np.empty((cap, 2), dtype=np.int32)
        n = _I32()
        _check(fn(self._h, seq, pairs.ctypes.data_as(ctypes.c_void_p), cap, ctypes.byref(n)), name)
        return pairs[:n.value]

    def swap_out(self, seq: int) -> np.ndarray:
        """Moves seq's blocks to host slots; returns the (device block, host
        block) pairs to run through swap_blocks(PA_SWAP_OUT)."""
        return self._swap(lib().pa_bm_swap_out, "pa_bm_swap_out", seq)

    def swap_in(self, seq: int) -> np.ndarray:
        """Gives seq fresh device blocks; returns the (device block, host block)
        pairs to run through swap_blocks(PA_SWAP_IN)."""
        return self._swap(lib().pa_bm_swap_in, "pa_bm_swap_in", seq)

    def num_free_host(self) -> int:
        return int(lib().pa_bm_num_free_host(self._h))

    def is_swapped(self, seq: int) -> bool:
        r = int(lib().pa_bm_is_swapped(self._h, seq))
        if r < 0:
            raise PagedAttentionError(7, "pa_bm_is_swapped")
        return r == 1

    # ---- prefix cache (see pa_bm_prefix_match .. pa_bm_prefix_stats)

    @staticmethod
    def _tokens(tokens) -> np.ndarray:
        return np.ascontiguousarray(tokens, dtype=np.int32)

    def prefix_match(self, tokens, condition: int = 0) -> int:
        """Tokens of the cached whole blocks at the head of ``tokens``."""
        t, m = self._tokens(tokens), _I64()
        _check(lib().pa_bm_prefix_match(self._h, t.ctypes.data_as(ctypes.c_void_p), len(t), condition,
                                        ctypes.byref(m)), "pa_bm_prefix_match")
        return m.value

    def add_seq_cached(self, tokens, condition: int = 0) -> Tuple[int, int]:
        """New sequence starting with the cached blocks of ``tokens``' head;
        returns (sequence id, matched tokens)."""
        t, sid, m = self._tokens(tokens), _I32(), _I64()
        _check(lib().pa_bm_add_seq_cached(self._h, t.ctypes.data_as(ctypes.c_void_p), len(t), condition,
                                          ctypes.byref(sid), ctypes.byref(m)), "pa_bm_add_seq_cached")
        return sid.value, m.value

    def cache_seq(self, seq: int, tokens, condition: int = 0) -> int:
        """Publishes seq's whole blocks holding ``tokens``; returns new entries."""
        t, n = self._tokens(tokens), _I64()
        _check(lib().pa_bm_cache_seq(self._h, seq, t.ctypes.data_as(ctypes.c_void_p), len(t), condition,
                                     ctypes.byref(n)), "pa_bm_cache_seq")
        return n.value

    def prefix_evict(self, n_blocks: int) -> int:
        freed = _I64()
        _check(lib().pa_bm_prefix_evict(self._h, n_blocks, ctypes.byref(freed)), "pa_bm_prefix_evict")
        return freed.value

    def num_cached(self) -> int:
        return int(lib().pa_bm_num_cached(self._h))

    def num_evictable(self) -> int:
        return int(lib().pa_bm_num_evictable(self._h))

    def prefix_stats(self) -> Tuple[int, int]:
        """(matched tokens, offered tokens) over all add_seq_cached calls."""
        hit, query = _I64(), _I64()
        _check(lib().pa_bm_prefix_stats(self._h, ctypes.byref(hit), ctypes.byref(query)), "pa_bm_prefix_stats")
        return hit.value, query.value


__all__ = ["BlockManager", "PagedAttentionError"]
