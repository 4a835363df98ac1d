"""The seeded workload generators produce what their recipes state (no GPU)."""
import numpy as np

import pa_workloads as wl


def _check_tables(w):
    valid = w.tables >= 0
    assert (w.tables[valid] < w.num_blocks).all()
    for s, L in enumerate(w.seq_lens):
        n = int(valid[s].sum())
        assert n * w.block_size >= L and (n - 1) * w.block_size < max(L, 1)
        assert valid[s, :n].all()


def test_configs_are_deterministic_and_valid():
    for name, make in wl.CONFIGS.items():
        a, b = make(), make()
        assert np.array_equal(a.tables, b.tables) and np.array_equal(a.seq_lens, b.seq_lens), name
        _check_tables(a)


def test_recipes():
    w = wl.tiny()
    assert w.seq_lens.tolist() == [1, 10, 16, 37] and w.num_blocks == 32 and w.block_size == 16
    assert len(np.unique(w.tables[w.tables >= 0])) == 6
    p = wl.tiny_page_example()
    assert p.tables.tolist() == [[5, 1, 7]] and p.block_size == 4 and p.seq_lens.tolist() == [10]
    w = wl.llama70b_decode()
    assert w.batch == 64 and (w.seq_lens >= 600).all() and (w.seq_lens <= 850).all()
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim, w.num_blocks) == (64, 8, 128, 16384)
    assert len(np.unique(w.tables[w.tables >= 0])) == int((w.tables >= 0).sum())   # no block shared
    w = wl.long_context()
    assert (w.seq_lens == 8192).all() and w.max_blocks == 512 and w.partition_tokens == 512
    w = wl.shared_prefix()
    assert w.batch == 256 and (w.tables[:, :125] == w.tables[0, :125]).all()
    assert (w.seq_lens - 2000 >= 1).all() and (w.seq_lens - 2000 <= 6192).all()
    assert 600 < np.median(w.seq_lens - 2000) < 1100
    private = w.tables[:, 125:]
    private = private[private >= 0]
    assert len(np.unique(private)) == len(private) and not np.isin(private, w.tables[0, :125]).any()
    w = wl.beam_fork()
    assert w.batch == 128 and len(w.copy_pairs) <= 96
    src, dst = w.copy_pairs[:, 0], w.copy_pairs[:, 1]
    assert len(np.unique(dst)) == len(dst) and not np.isin(dst, src).any()
    w = wl.prefill_chunk()
    assert w.kind == "prefill" and w.chunk == 512 and (w.ctx_lens == 4096).all() and w.max_blocks == 288


def test_tensors_shapes():
    w = wl.tiny()
    t = wl.make_tensors(w)
    assert t["pool"].shape == (32, 2, 2, 16, 64) and t["q"].shape == (4, 4, 64)
    assert t["new_k"].shape == (4, 2, 64)
    unused = np.setdiff1d(np.arange(32), w.referenced)
    assert not t["pool"][unused].any()
    assert np.array_equal(wl.bf16_bits(wl.make_tensors(w)["q"]), wl.bf16_bits(t["q"]))


def test_shared_groups():
    """Each group's tables start with the same prefix blocks; every other block
    is used by one table only; lengths are prefix + suffix."""
    prefix, suffix, gsz = [32, 0, 64], [1, 17, 5, 0, 40, 16], 2
    w = wl.shared_groups(prefix, suffix, gsz, 8, 2, 128, 16, seed=3)
    _check_tables(w)
    assert w.seq_lens.tolist() == [33, 49, 5, 0, 104, 80]
    seen = {}
    for s in range(w.batch):
        n_pre = prefix[s // gsz] // 16
        head = w.tables[s, :n_pre].tolist()
        first = w.tables[(s // gsz) * gsz, :n_pre].tolist()
        assert head == first
        for blk in w.tables[s, n_pre:][w.tables[s, n_pre:] >= 0].tolist():
            assert blk not in seen, blk
            seen[blk] = s
    shared = {b for g, p in enumerate(prefix) for b in w.tables[g * gsz, :p // 16].tolist()}
    assert not shared & set(seen)
