"""CPU oracle for paged KV-cache attention -- TEST INFRASTRUCTURE.

This package is the checker, not the product.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the CUDA path (``paged_kv_cache_167_gb300``) and
never imports it; the product never imports this package.

``pa_oracle.c`` holds the arithmetic (plain C, fp64).  This module only builds
it with gcc and marshals numpy arrays through ctypes.  bf16 tensors travel as
their raw 16-bit patterns (numpy ``uint16``).

Pinned against the pages by ``tests/test_oracle_pins.py`` (printed values of
the block-layout and address-map example, closed forms, invariants, a library
attention routine and brute force); ``tests/test_oracle_mutants.py`` shows that
planted mistakes in ``pa_oracle.c`` fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pa_oracle.c")
LIBRARY = os.path.join(HERE, "libpa_oracle.so")


def _gcc_has_openmp(cc: str) -> bool:
    probe = subprocess.run([cc, "-fopenmp", "-x", "c", "-E", "-", "-o", os.devnull],
                           input=b"#include <omp.h>\n", capture_output=True)
    return probe.returncode == 0


def build(source: str = SOURCE, output: str = LIBRARY, openmp: bool = True) -> str:
    """Compile the oracle into a shared library with gcc; returns its path."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", source, "-o", output, "-lm"]
    if openmp and _gcc_has_openmp(cc):
        cmd.insert(1, "-fopenmp")
    subprocess.run(cmd, check=True, capture_output=True)
    return output


class PoolGeom(ctypes.Structure):
    """One layer's view of the block pool, strides in elements."""
    _fields_ = [
        ("num_blocks", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int64),
        ("block_size", ctypes.c_int64),
        ("head_dim", ctypes.c_int64),
        ("block_stride", ctypes.c_int64),
        ("kv_stride", ctypes.c_int64),
    ]


def dense_geom(num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int,
               num_layers: int = 1) -> PoolGeom:
    """Geometry of a pool laid out [NB][2][layers][Hkv][b][d] (one layer's view)."""
    slab = num_kv_heads * block_size * head_dim
    return PoolGeom(num_blocks, num_kv_heads, block_size, head_dim,
                    2 * num_layers * slab, num_layers * slab)


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes handle on one build of ``pa_oracle.c``."""

    def __init__(self, library: str = LIBRARY):
        self.library = library
        lib = ctypes.CDLL(library)
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        G = ctypes.POINTER(PoolGeom)
        sig = {
            "orc_num_threads": (I32, []),
            "orc_set_num_threads": (I32, [I32]),
            "orc_block_layout": (I32, [I64, I64, ctypes.POINTER(I64), ctypes.POINTER(I64)]),
            "orc_address": (None, [P, I64, I64, ctypes.POINTER(I64), ctypes.POINTER(I64)]),
            "orc_slot": (I64, [P, I64, I64]),
            "orc_slot_mapping": (None, [P, P, I64, P, P, I64, I64]),
            "orc_reshape_and_cache": (None, [P, G, P, P, P, I64]),
            "orc_copy_blocks": (None, [P, G, P, I64]),
            "orc_swap_blocks": (None, [P, G, P, P, I64, I32]),
            "orc_capacity": (I32, [P, I64, I64, I64, I64, I64, I64, P]),
            "orc_paged_decode_rows": (None, [P, P, P, G, P, I64, P, I64, D, P, I64]),
            "orc_paged_decode": (None, [P, P, P, G, P, I64, P, I64, I64, D]),
            "orc_paged_decode_lse": (None, [P, P, P, P, G, P, I64, P, I64, I64, D]),
            "orc_prefill_rows": (None, [P, P, P, G, P, I64, P, I64, I64, D, P, I64]),
            "orc_prefill": (None, [P, P, P, G, P, I64, P, I64, I64, I64, D]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        self._lib = lib

    # -- capacity arithmetic and address map ---------------------------------
    def num_threads(self) -> int:
        return int(self._lib.orc_num_threads())

    def set_num_threads(self, n: int) -> int:
        """Threads the oracle's OpenMP loops use from now on; returns the count in force."""
        return int(self._lib.orc_set_num_threads(int(n)))

    def block_layout(self, tokens: int, block_size: int):
        blocks, unused = ctypes.c_int64(), ctypes.c_int64()
        rc = self._lib.orc_block_layout(tokens, block_size, ctypes.byref(blocks), ctypes.byref(unused))
        if rc != 0:
            raise ValueError("invalid size")
        return blocks.value, unused.value

    def address(self, table_row: Sequence[int], pos: int, block_size: int):
        row = _i32(table_row)
        phys, off = ctypes.c_int64(), ctypes.c_int64()
        self._lib.orc_address(_ptr(row), pos, block_size, ctypes.byref(phys), ctypes.byref(off))
        return phys.value, off.value

    def slot_mapping(self, tables, seq_idx, positions, block_size: int) -> np.ndarray:
        tables = _i32(tables)
        seq_idx, positions = _i32(seq_idx), _i64(positions)
        out = np.empty(len(positions), dtype=np.int64)
        self._lib.orc_slot_mapping(_ptr(out), _ptr(tables), tables.shape[1], _ptr(seq_idx),
                                   _ptr(positions), len(positions), block_size)
        return out

    # -- pool writes -----------------------------------------------------------
    def reshape_and_cache(self, pool: np.ndarray, geom: PoolGeom, k: np.ndarray, v: np.ndarray,
                          slots) -> None:
        """Writes k, v ([N][Hkv][d] bf16 bits) into ``pool`` in place."""
        if pool.dtype != np.uint16 or not pool.flags.c_contiguous:
            raise TypeError("pool must be a C-contiguous uint16 array")
        k, v, slots = _u16(k), _u16(v), _i64(slots)
        self._lib.orc_reshape_and_cache(_ptr(pool), ctypes.byref(geom), _ptr(k), _ptr(v),
                                        _ptr(slots), len(slots))

    def copy_blocks(self, pool: np.ndarray, geom: PoolGeom, pairs) -> None:
        if pool.dtype != np.uint16 or not pool.flags.c_contiguous:
            raise TypeError("pool must be a C-contiguous uint16 array")
        pairs = _i32(pairs).reshape(-1, 2)
        self._lib.orc_copy_blocks(_ptr(pool), ctypes.byref(geom), _ptr(pairs), pairs.shape[0])

    def swap_blocks(self, pool: np.ndarray, geom: PoolGeom, host: np.ndarray, pairs, direction: int) -> None:
        """Block copies between pool and host ([hb][2][Hkv][b][d]); pairs are
        (pool block, host block); direction 0 = pool -> host, 1 = host -> pool."""
        for name, a in (("pool", pool), ("host", host)):
            if a.dtype != np.uint16 or not a.flags.c_contiguous:
                raise TypeError(f"{name} must be a C-contiguous uint16 array")
        pairs = _i32(pairs).reshape(-1, 2)
        self._lib.orc_swap_blocks(_ptr(pool), ctypes.byref(geom), _ptr(host), _ptr(pairs), pairs.shape[0],
                                  int(direction))

    # -- capacity ---------------------------------------------------------------
    def capacity(self, lens, shared_prefix_tokens: int, block_size: int, max_seq_len: int,
                 bytes_per_token: int, budget_bytes: int) -> dict:
        """Contiguous against paged capacity of a KV budget for the length mix
        ``lens`` (requests taken from it in turn); see ``orc_capacity``."""
        lens = np.ascontiguousarray(lens, dtype=np.int64)
        out = np.zeros(7, np.float64)
        rc = self._lib.orc_capacity(_ptr(lens), len(lens), int(shared_prefix_tokens), int(block_size),
                                    int(max_seq_len), int(bytes_per_token), int(budget_bytes), _ptr(out))
        if rc != 0:
            raise ValueError("invalid capacity arguments")
        keys = ("contiguous_requests", "paged_requests", "contiguous_waste", "paged_waste", "mean_tail_slots",
                "prefix_bytes_contiguous", "prefix_bytes_paged")
        res = dict(zip(keys, out.tolist()))
        res["contiguous_requests"] = int(res["contiguous_requests"])
        res["paged_requests"] = int(res["paged_requests"])
        return res

    # -- attention -------------------------------------------------------------
    def paged_decode(self, q: np.ndarray, pool: np.ndarray, geom: PoolGeom, tables, seq_lens,
                     num_q_heads: int, scale: float, rows: Optional[np.ndarray] = None) -> np.ndarray:
        """Decode attention; q is [B][Hq][d].  Returns fp64 [B][Hq][d], or
        [n][d] for ``rows`` given as (s, h) pairs."""
        q, pool, tables, seq_lens = _u16(q), _u16(pool), _i32(tables), _i32(seq_lens)
        d = geom.head_dim
        if rows is None:
            B = seq_lens.shape[0]
            out = np.empty((B, num_q_heads, d), dtype=np.float64)
            self._lib.orc_paged_decode(_ptr(out), _ptr(q), _ptr(pool), ctypes.byref(geom),
                                       _ptr(tables), tables.shape[1], _ptr(seq_lens), B,
                                       num_q_heads, float(scale))
            return out
        rows = _i32(rows).reshape(-1, 2)
        out = np.empty((rows.shape[0], d), dtype=np.float64)
        self._lib.orc_paged_decode_rows(_ptr(out), _ptr(q), _ptr(pool), ctypes.byref(geom),
                                        _ptr(tables), tables.shape[1], _ptr(seq_lens),
                                        num_q_heads, float(scale), _ptr(rows), rows.shape[0])
        return out

    def paged_decode_lse(self, q: np.ndarray, pool: np.ndarray, geom: PoolGeom, tables, seq_lens,
                         num_q_heads: int, scale: float):
        """Decode attention with each row's log-sum-exp log(sum_t exp(scale q.K_t)):
        returns (out fp64 [B][Hq][d], lse fp64 [B][Hq]; -inf with no keys)."""
        q, pool, tables, seq_lens = _u16(q), _u16(pool), _i32(tables), _i32(seq_lens)
        B = seq_lens.shape[0]
        out = np.empty((B, num_q_heads, geom.head_dim), dtype=np.float64)
        lse = np.empty((B, num_q_heads), dtype=np.float64)
        self._lib.orc_paged_decode_lse(_ptr(out), _ptr(lse), _ptr(q), _ptr(pool), ctypes.byref(geom),
                                       _ptr(tables), tables.shape[1], _ptr(seq_lens), B, num_q_heads,
                                       float(scale))
        return out, lse

    def prefill(self, q: np.ndarray, pool: np.ndarray, geom: PoolGeom, tables, ctx_lens,
                num_q_heads: int, scale: float, rows: Optional[np.ndarray] = None) -> np.ndarray:
        """Chunked causal prefill; q is [B][C][Hq][d].  Returns fp64 of q's
        shape, or [n][d] for ``rows`` given as (s, j, h) triples."""
        q, pool, tables, ctx_lens = _u16(q), _u16(pool), _i32(tables), _i32(ctx_lens)
        B, C = q.shape[0], q.shape[1]
        d = geom.head_dim
        if rows is None:
            out = np.empty((B, C, num_q_heads, d), dtype=np.float64)
            self._lib.orc_prefill(_ptr(out), _ptr(q), _ptr(pool), ctypes.byref(geom),
                                  _ptr(tables), tables.shape[1], _ptr(ctx_lens), B, C,
                                  num_q_heads, float(scale))
            return out
        rows = _i32(rows).reshape(-1, 3)
        out = np.empty((rows.shape[0], d), dtype=np.float64)
        self._lib.orc_prefill_rows(_ptr(out), _ptr(q), _ptr(pool), ctypes.byref(geom),
                                   _ptr(tables), tables.shape[1], _ptr(ctx_lens), C,
                                   num_q_heads, float(scale), _ptr(rows), rows.shape[0])
        return out


_DEFAULT: Optional[Oracle] = None


def load() -> Oracle:
    """The oracle built from ``pa_oracle.c`` (rebuilt when the source is newer)."""
    global _DEFAULT
    if _DEFAULT is None:
        stale = (not os.path.exists(LIBRARY)
                 or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))
        if stale:
            build()
        _DEFAULT = Oracle(LIBRARY)
    return _DEFAULT

