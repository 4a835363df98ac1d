"""Host planning of a cascade decode (pa_cascade_plan): which leading blocks a
group of sequences shares and what each keeps of its own (no GPU)."""
import numpy as np
import pytest

import pa_workloads as wl


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_167_gb300 as pa
    return pa


def by_scan(tables, lens, group_size, b):
    """Block by block: a block is shared while every member of the group has
    the same id there and every member still has a token after it."""
    B, W = tables.shape
    plens, suffix = [], np.full((B, W), -1, np.int32)
    for gi in range(B // group_size):
        rows = range(gi * group_size, (gi + 1) * group_size)
        n = 0
        while (n < W and tables[gi * group_size, n] >= 0
               and all(tables[s, n] == tables[gi * group_size, n] for s in rows)
               and all((n + 1) * b < lens[s] for s in rows)):
            n += 1
        plens.append(n * b)
        for s in rows:
            suffix[s, :W - n] = tables[s, n:]
    return np.asarray(plens, np.int32), suffix


def test_hand_example(pa):
    t = np.array([[5, 6, 7, 8], [5, 6, 9, -1], [5, 6, 7, 10], [1, 2, 3, 4]], np.int32)
    p = pa.cascade_plan(t, [64, 40, 61, 13], 2, 16)
    assert p["prefix_lens"].tolist() == [32, 0]
    assert p["prefix_tables"].tolist() == [[5, 6, -1, -1], [-1, -1, -1, -1]]
    assert p["suffix_tables"].tolist() == [[7, 8, -1, -1], [9, -1, -1, -1], [5, 6, 7, 10], [1, 2, 3, 4]]
    assert p["suffix_lens"].tolist() == [32, 8, 61, 13]
    assert p["group_order"].tolist() == [0, 1]


def test_whole_sequence_shared_keeps_last_token(pa):
    """Two sequences with identical 3-block tables and 48 tokens share two
    blocks, not three: the token being decoded stays in each suffix."""
    t = np.array([[3, 4, 5], [3, 4, 5]], np.int32)
    p = pa.cascade_plan(t, [48, 48], 2, 16)
    assert p["prefix_lens"].tolist() == [32] and p["suffix_lens"].tolist() == [16, 16]
    p = pa.cascade_plan(t, [33, 48], 2, 16)
    assert p["prefix_lens"].tolist() == [32]
    p = pa.cascade_plan(t, [32, 48], 2, 16)
    assert p["prefix_lens"].tolist() == [16]
    p = pa.cascade_plan(t, [0, 48], 2, 16)
    assert p["prefix_lens"].tolist() == [0] and p["suffix_lens"].tolist() == [0, 48]


@pytest.mark.parametrize("seed", range(6))
def test_random_against_scan(pa, seed):
    rng = np.random.default_rng(seed)
    b, gsz = int(rng.choice([4, 16])), int(rng.integers(1, 5))
    groups = int(rng.integers(1, 6))
    B, W = groups * gsz, 12
    tables = np.full((B, W), -1, np.int32)
    lens = np.zeros(B, np.int32)
    nxt = 0
    for gi in range(groups):
        common = int(rng.integers(0, 8))
        shared = list(range(nxt, nxt + common))
        nxt += common
        for k in range(gsz):
            s = gi * gsz + k
            own = int(rng.integers(0, W - common + 1))
            row = shared + list(range(nxt, nxt + own))
            nxt += own
            tables[s, :len(row)] = row
            lens[s] = int(rng.integers(max(0, (len(row) - 1) * b + 1), len(row) * b + 1)) if row else 0
    p = pa.cascade_plan(tables, lens, gsz, b)
    plens, suffix = by_scan(tables, lens, gsz, b)
    assert np.array_equal(p["prefix_lens"], plens)
    assert np.array_equal(p["suffix_tables"], suffix)
    assert np.array_equal(p["suffix_lens"], lens - np.repeat(plens, gsz))
    # groups by prefix length, longest first, ties in index order
    assert p["group_order"].tolist() == sorted(range(groups), key=lambda g: (-int(plens[g]), g))
    for gi in range(groups):
        n = plens[gi] // b
        assert np.array_equal(p["prefix_tables"][gi, :n], tables[gi * gsz, :n])
        assert (p["prefix_tables"][gi, n:] == -1).all()


def test_workloads(pa):
    w = wl.shared_prefix()
    p = pa.cascade_plan(w.tables, w.seq_lens, w.batch, w.block_size)
    assert p["prefix_lens"].tolist() == [2000]
    assert np.array_equal(p["prefix_tables"][0, :125], w.notes["shared_ids"])
    w = wl.beam_fork()
    p = pa.cascade_plan(w.tables, w.seq_lens, 4, w.block_size)
    assert np.array_equal(p["prefix_lens"], (w.notes["prompt_lens"] // 16) * 16)
    assert (p["suffix_lens"] >= 1).all() and (p["suffix_lens"] <= 16).all()


def test_invalid(pa):
    t = np.zeros((4, 2), np.int32)
    for args in ((t, [1, 1, 1, 1], 3, 16),        # not whole groups
                 (t, [1, 1, 1, 1], 0, 16),        # group size
                 (t, [1, 1, 1, 1], 2, 0),         # block size
                 (t, [1, -1, 1, 1], 2, 16),       # negative length
                 (t, [1, 33, 1, 1], 2, 16)):      # longer than the table
        with pytest.raises((pa.PagedAttentionError, ValueError)):
            pa.cascade_plan(*args)
