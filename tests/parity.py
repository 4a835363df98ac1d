"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs, and compare.

Float acceptance rule for attention outputs (bf16 output, fp32 accumulate)
against the fp64 oracle: an element passes iff
    |gpu - ref| <= max(ATOL, RTOL * |ref|)
with ATOL = 4e-3 and RTOL = 1e-2, the max-abs / max-rel bounds the
specification of this path states, read as a per-element either/or because a
pure relative bound is meaningless where the reference crosses zero.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

import oracle
import pa_workloads as wl

ATOL = 4e-3
RTOL = 1e-2


def assert_close(got: torch.Tensor, ref: np.ndarray, what: str) -> Dict[str, float]:
    g = got.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    err = np.abs(g - ref)
    bad = err > np.maximum(ATOL, RTOL * np.abs(ref))
    big = np.abs(ref) >= 0.4
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "max_rel_ref_ge_0.4": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
             "n_bad": int(bad.sum())}
    assert not np.isnan(g).any(), f"{what}: NaN in output"
    assert stats["n_bad"] == 0, f"{what}: {stats['n_bad']} elements out of tolerance; {stats}"
    return stats


def geom_of(w: wl.Workload) -> oracle.PoolGeom:
    return oracle.dense_geom(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)


class Case:
    """One workload's tensors on the GPU and their host bit patterns."""

    def __init__(self, w: wl.Workload, device="cuda", tensors: Optional[dict] = None):
        self.w = w
        self.dev = torch.device(device)
        t = tensors if tensors is not None else wl.make_tensors(w, "cpu")
        self.cpu = t
        self.pool = t["pool"].to(self.dev)
        self.q = t["q"].to(self.dev)
        self.new_k = t["new_k"].to(self.dev)
        self.new_v = t["new_v"].to(self.dev)
        self.tables = torch.as_tensor(w.tables, device=self.dev)
        self.seq_lens = torch.as_tensor(w.seq_lens, device=self.dev)
        self.pool_ref = wl.bf16_bits(t["pool"]).copy()   # oracle's copy of the pool
        self.orc = oracle.load()
        self.geom = geom_of(w)
