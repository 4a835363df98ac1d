"""Capacity of a KV budget (pa_capacity_estimate, host arithmetic): the
library's closed form against the oracle's request-by-request, token-by-token
simulation on seeded length mixes, and against the worked numbers that
how-pagedattention-works (aiinfrainterviews.com) prints in "A strong answer"
(no GPU)."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "capacity_worked_example.json")
INT_FIELDS = ("contiguous_requests", "paged_requests")
REAL_FIELDS = ("contiguous_waste", "paged_waste", "mean_tail_slots", "prefix_bytes_contiguous", "prefix_bytes_paged")


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_167_gb300 as pa
    return pa


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def same(got, ref):
    for k in INT_FIELDS:
        assert got[k] == ref[k], (k, got, ref)
    for k in REAL_FIELDS:
        assert abs(got[k] - ref[k]) <= 1e-12 * max(1.0, abs(ref[k])), (k, got, ref)


def length_mix(rng, kind, n, prefix, max_len):
    if kind == "lognormal":        # chat-like: long right tail
        x = rng.lognormal(np.log(max(prefix, 1) + 400), 0.7, n)
    elif kind == "uniform":
        x = rng.uniform(prefix, max_len, n)
    else:                          # bimodal: short chats and long documents
        x = np.where(rng.random(n) < 0.8, rng.normal(prefix + 300, 60, n), rng.normal(max_len * 0.8, 200, n))
    return np.clip(np.rint(x), prefix, max_len).astype(np.int64)


@pytest.mark.parametrize("kind", ["lognormal", "uniform", "bimodal"])
@pytest.mark.parametrize("b", [8, 16, 32, 64])
@pytest.mark.parametrize("prefix", [0, 512, 700])
def test_matches_oracle(pa, orc, kind, b, prefix):
    rng = np.random.default_rng(b * 1000 + prefix + len(kind))
    max_len = 4096
    lens = length_mix(rng, kind, 300, prefix, max_len)
    for budget in (0, 5 * 10**8, 7 * 10**9, 40 * 10**9):
        args = (lens, prefix, b, max_len, 163840, budget)
        same(pa.capacity_estimate(*args), orc.capacity(*args))


def test_exact_budget_boundaries(pa, orc):
    """Budgets one byte either side of an exact fit of reservations or blocks."""
    for lens, b, max_len in (([12], 4, 12), ([3, 10, 7], 4, 16), ([33, 1, 64, 16], 16, 64)):
        for k in range(0, 40):
            for budget in (k * max_len - 1, k * max_len, k * b - 1, k * b, k * b + 1):
                if budget < 0:
                    continue
                same(pa.capacity_estimate(lens, 0, b, max_len, 1, budget), orc.capacity(lens, 0, b, max_len, 1, budget))


def test_worked_example_through_library(pa):
    g = json.load(open(GOLDEN))
    i, pr = g["inputs"], g["printed"]
    c = pa.capacity_estimate([i["request_tokens"]], 0, i["block_size"], i["max_seq_len"], i["bytes_per_token"],
                             i["budget_bytes"])
    assert c["contiguous_requests"] == pr["contiguous_requests"]
    assert round(c["contiguous_waste"], 2) == pr["waste_fraction"]
    assert abs(c["paged_requests"] - pr["paged_requests_about"]) <= pr["paged_requests_rel_tol"] * \
        pr["paged_requests_about"]
    assert round(c["paged_requests"] / c["contiguous_requests"]) == pr["gain_about"]
    sp = g["shared_prefix"]
    P, n = sp["prefix_tokens"], sp["conversations"]
    c = pa.capacity_estimate([P + 850] * n, P, 16, 8192, i["bytes_per_token"], i["budget_bytes"])
    assert round(c["prefix_bytes_contiguous"] / 1e9) == sp["contiguous_duplicate_gb"]
    assert round(c["prefix_bytes_paged"] / 1e6) == sp["paged_mb"]


def test_large_budget_is_closed_form(pa):
    """A budget far beyond what a token-by-token simulation could walk."""
    c = pa.capacity_estimate([850], 0, 16, 8192, 1, 10**18)
    assert c["contiguous_requests"] == 10**18 // 8192
    assert c["paged_requests"] == (10**18 // 16) // 54


def test_invalid_arguments(pa):
    bad = [
        ([], 0, 16, 64, 1, 100),          # no requests
        ([10], 0, 0, 64, 1, 100),         # block size
        ([10], 0, 16, 0, 1, 100),         # max_seq_len
        ([10], 0, 16, 64, 0, 100),        # bytes per token
        ([10], 0, 16, 64, 1, -1),         # budget
        ([10], -1, 16, 64, 1, 100),       # prefix
        ([65], 0, 16, 64, 1, 100),        # longer than max_seq_len
        ([10], 11, 16, 64, 1, 100),       # shorter than its prefix
        ([0, 0], 0, 16, 64, 1, 100),      # nothing to hold: admission would not end
        ([32], 32, 16, 64, 1, 100),       # all blocks shared: same
        ([10], 0, 16, 2**62, 4, 100),     # overflow of the reservation size
    ]
    for args in bad:
        with pytest.raises(pa.PagedAttentionError) as e:
            pa.capacity_estimate(*args)
        assert e.value.status == 1, args


def test_shared_prefix_workload_mix(pa, orc):
    """The 256-sequence shared-prompt workload's lengths (2,000-token prompt plus
    a lognormal suffix, at most 8,192 tokens) at Llama 3.1 70B's 328 KB a token:
    the library equals the oracle, and sharing the prompt's 125 blocks beats
    both private paging and contiguous reservation."""
    import pa_workloads as wl
    w = wl.CONFIGS["shared_prefix"]()
    lens = w.seq_lens.astype(np.int64)
    args = dict(block_size=16, max_seq_len=8192, bytes_per_token=328000, budget_bytes=435 * 10**9)
    shared = pa.capacity_estimate(lens, 2000, **args)
    private = pa.capacity_estimate(lens, 0, **args)
    same(shared, orc.capacity(lens, 2000, 16, 8192, 328000, 435 * 10**9))
    same(private, orc.capacity(lens, 0, 16, 8192, 328000, 435 * 10**9))
    assert shared["paged_requests"] > private["paged_requests"] > shared["contiguous_requests"]
    assert shared["contiguous_waste"] > 0.5 and shared["paged_waste"] < 0.01
