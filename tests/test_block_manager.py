"""Host block manager: allocation on demand, reference counts, forks,
copy-on-write planning and admission, checked against invariants and the
pages' counting claims (no GPU)."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_167_gb300 as pa
    return pa


def check_invariants(bm, live, orc):
    """refcount(b) == number of live tables holding b; free == refcount 0;
    each table holds exactly block_layout(tokens) blocks; slots agree with the oracle."""
    counts = np.zeros(bm.num_blocks, dtype=np.int64)
    for s in live:
        table, tokens = bm.table(s)
        assert len(table) == orc.block_layout(tokens, bm.block_size)[0]
        assert len(set(table.tolist())) == len(table)
        counts[table] += 1
    ref = np.asarray([bm.refcount(b) for b in range(bm.num_blocks)])
    assert np.array_equal(ref, counts)
    assert bm.num_free() == int((counts == 0).sum())


def test_random_operations(pa):
    orc = oracle.load()
    rng = np.random.default_rng(0)
    bm = pa.BlockManager(256, 16)
    live = []
    pending_cow = []
    for step in range(600):
        op = rng.choice(["add", "append", "fork", "free"], p=[0.15, 0.5, 0.15, 0.2])
        if op == "add" or not live:
            live.append(bm.add_seq())
        elif op == "append":
            s = int(rng.choice(live))
            table_before, tokens_before = bm.table(s)
            n = int(rng.integers(1, 40))
            try:
                slots, pair = bm.append_tokens(s, n)
            except pa.PagedAttentionError as e:
                assert e.status == 6  # PA_ERR_NO_BLOCKS, and nothing changed
                t2, n2 = bm.table(s)
                assert n2 == tokens_before and np.array_equal(t2, table_before)
                continue
            table, tokens = bm.table(s)
            assert tokens == tokens_before + n
            pos = np.arange(tokens_before, tokens, dtype=np.int64)
            ref = orc.slot_mapping(table[None, :], np.zeros(n, np.int32), pos, 16)
            assert np.array_equal(slots, ref)
            if pair is not None:
                src, dst = pair
                assert tokens_before % 16 != 0 and table_before[-1] == src and table[len(table_before) - 1] == dst
                pending_cow.append(pair)
        elif op == "fork":
            live.append(bm.fork(int(rng.choice(live))))
        else:
            s = int(rng.choice(live))
            bm.free_seq(s)
            live.remove(s)
        check_invariants(bm, live, orc)
    assert pending_cow, "the random walk never exercised copy-on-write"


def test_exhaustion_leaves_state_unchanged(pa):
    bm = pa.BlockManager(4, 16)
    s = bm.add_seq()
    bm.append_tokens(s, 60)
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.append_tokens(s, 10)
    assert e.value.status == 6
    assert bm.table(s)[1] == 60 and bm.num_free() == 0
    bm.append_tokens(s, 4)  # still fits in the last block
    assert bm.table(s)[1] == 64


def test_beam_fork_footprint(pa):
    """Beams share their prompt; a partly filled last block is copied for every
    beam but the first, so N beams cost the prompt's blocks plus one block per
    extra beam (common prefix + N x divergent blocks)."""
    orc = oracle.load()
    for prompt in (1024, 1030, 2999, 3000, 2048):
        bm = pa.BlockManager(4096, 16)
        root = bm.add_seq()
        bm.append_tokens(root, prompt)
        beams = [root] + [bm.fork(root) for _ in range(3)]
        original_tail = int(bm.table(root)[0][-1])
        pairs = []
        for s in beams:
            _, pair = bm.append_tokens(s, 1)
            if pair:
                pairs.append(pair)
        nblk, tail = orc.block_layout(prompt, 16)
        used = 4096 - bm.num_free()
        if tail:            # partly filled: 3 copies; the last beam to write keeps the original
            assert len(pairs) == 3 and used == nblk + 3
            assert len({d for _, d in pairs}) == 3 and {s for s, _ in pairs} == {original_tail}
            assert bm.table(beams[-1])[0][-1] == original_tail and bm.refcount(original_tail) == 1
        else:               # full: nothing to copy, every beam opens one new block
            assert not pairs and used == nblk + 4
        for b in bm.table(root)[0][:-1]:
            assert bm.refcount(int(b)) == 4


def test_shared_system_prompt(pa):
    """A 2,000-token system prompt shared by 256 sequences is held once: 125
    blocks with refcount 256, whatever the suffixes."""
    bm = pa.BlockManager(32768, 16)
    prompt = bm.add_seq()
    bm.append_tokens(prompt, 2000)
    prefix = bm.table(prompt)[0]
    assert len(prefix) == 125
    rng = np.random.default_rng(1)
    seqs = [bm.fork(prompt) for _ in range(256)]
    bm.free_seq(prompt)
    suffix = rng.integers(1, 2000, size=256)
    for s, n in zip(seqs, suffix):
        _, pair = bm.append_tokens(s, int(n))
        assert pair is None
    for b in prefix:
        assert bm.refcount(int(b)) == 256
    assert 32768 - bm.num_free() == 125 + int(sum(-(-n // 16) for n in suffix))


def test_admission(pa):
    bm = pa.BlockManager(10, 16)
    assert bm.can_admit(100, 2)          # ceil(100/16) + 1 + 2 = 10
    assert not bm.can_admit(100, 3)
    assert bm.can_admit(0, 9)
    s = bm.add_seq()
    bm.append_tokens(s, 17)
    assert bm.can_admit(100, 0)          # 8 free, 7 + 1 needed
    assert not bm.can_admit(100, 1)
    bm.free_seq(s)
    assert bm.can_admit(100, 2)


def test_unknown_sequence(pa):
    bm = pa.BlockManager(10, 16)
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.append_tokens(3, 1)
    assert e.value.status == 7
    s = bm.add_seq()
    bm.free_seq(s)
    with pytest.raises(pa.PagedAttentionError):
        bm.fork(s)
