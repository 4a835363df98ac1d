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


# ---------------------------------------------------------------------------
# swapping to host slots (how-pagedattention-works, feature table, preemption
# row; "What interviewers probe next")
# ---------------------------------------------------------------------------

def test_swap_out_and_in(pa):
    bm = pa.BlockManager(16, 4)
    bm.set_host_pool(8)
    s = bm.add_seq()
    bm.append_tokens(s, 10)                       # 3 blocks: 0, 1, 2
    table, tokens = bm.table(s)
    pairs = bm.swap_out(s)
    assert pairs[:, 0].tolist() == table.tolist() and pairs[:, 1].tolist() == [0, 1, 2]
    assert bm.is_swapped(s) and bm.num_free() == 16 and bm.num_free_host() == 5
    for call in (lambda: bm.append_tokens(s, 1), lambda: bm.table(s), lambda: bm.fork(s), lambda: bm.swap_out(s)):
        with pytest.raises(pa.PagedAttentionError) as e:
            call()
        assert e.value.status == 8                # PA_ERR_SWAPPED
    other = bm.add_seq()
    bm.append_tokens(other, 8)                    # reuses two of the released blocks meanwhile
    back = bm.swap_in(s)
    assert back[:, 1].tolist() == [0, 1, 2]       # same host slots, in table order
    t_other, _ = bm.table(other)
    assert set(back[:, 0].tolist()).isdisjoint(t_other.tolist()) and len(set(back[:, 0].tolist())) == 3
    table2, tokens2 = bm.table(s)
    assert tokens2 == tokens and table2.tolist() == back[:, 0].tolist()
    assert not bm.is_swapped(s) and bm.num_free_host() == 8
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.swap_in(s)
    assert e.value.status == 8


def test_swap_keeps_shared_blocks_for_other_tables(pa):
    orc = oracle.load()
    bm = pa.BlockManager(16, 4)
    bm.set_host_pool(4)
    parent = bm.add_seq()
    bm.append_tokens(parent, 6)                   # blocks 0, 1 (last partly filled)
    child = bm.fork(parent)
    pairs = bm.swap_out(child)
    assert pairs[:, 0].tolist() == [0, 1]
    assert bm.refcount(0) == 1 and bm.refcount(1) == 1   # the parent still holds both
    check_invariants(bm, [parent], orc)
    bm.swap_in(child)
    t_child, _ = bm.table(child)
    assert set(t_child.tolist()).isdisjoint({0, 1})     # private copies now
    check_invariants(bm, [parent, child], orc)
    slots, cow = bm.append_tokens(child, 1)
    assert cow is None                            # nothing shared left to copy


def test_swap_capacity_and_release(pa):
    bm = pa.BlockManager(6, 4)
    bm.set_host_pool(2)
    s = bm.add_seq()
    bm.append_tokens(s, 12)                       # 3 blocks > 2 host slots
    table, _ = bm.table(s)
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.swap_out(s)
    assert e.value.status == 6 and not bm.is_swapped(s) and bm.table(s)[0].tolist() == table.tolist()
    bm.set_host_pool(4)
    bm.swap_out(s)
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.set_host_pool(8)                       # slots in use
    assert e.value.status == 1
    fillers = [bm.add_seq() for _ in range(2)]
    for f in fillers:
        bm.append_tokens(f, 12)                   # 6 device blocks in use: none left
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.swap_in(s)
    assert e.value.status == 6 and bm.is_swapped(s)
    bm.free_seq(s)                                # a swapped-out sequence releases its host slots
    assert bm.num_free_host() == 4


def test_random_operations_with_swaps(pa):
    orc = oracle.load()
    rng = np.random.default_rng(7)
    bm = pa.BlockManager(96, 8)
    bm.set_host_pool(64)
    live, swapped = [], set()
    for step in range(500):
        op = rng.choice(["add", "append", "fork", "free", "out", "in"], p=[0.12, 0.4, 0.1, 0.13, 0.12, 0.13])
        on_device = [s for s in live if s not in swapped]
        if op == "add" or not live:
            live.append(bm.add_seq())
        elif op == "append" and on_device:
            s = int(rng.choice(on_device))
            try:
                bm.append_tokens(s, int(rng.integers(1, 30)))
            except pa.PagedAttentionError as e:
                assert e.status == 6
        elif op == "fork" and on_device:
            live.append(bm.fork(int(rng.choice(on_device))))
        elif op == "free":
            s = int(rng.choice(live))
            bm.free_seq(s)
            live.remove(s)
            swapped.discard(s)
        elif op == "out" and on_device:
            s = int(rng.choice(on_device))
            try:
                pairs = bm.swap_out(s)
                swapped.add(s)
                assert len(set(pairs[:, 1].tolist())) == len(pairs)
            except pa.PagedAttentionError as e:
                assert e.status == 6
        elif op == "in" and swapped:
            s = int(rng.choice(sorted(swapped)))
            try:
                pairs = bm.swap_in(s)
                swapped.discard(s)
                assert bm.table(s)[0].tolist() == pairs[:, 0].tolist()
            except pa.PagedAttentionError as e:
                assert e.status == 6
        check_invariants(bm, [s for s in live if s not in swapped], orc)
        assert all(bm.is_swapped(s) for s in swapped)
    for s in list(swapped):
        bm.free_seq(s)
    assert bm.num_free_host() == 64
