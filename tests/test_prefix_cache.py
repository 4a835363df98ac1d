"""Prefix cache of the host block manager (pa_bm_prefix_match .. pa_bm_prefix_stats)
against the reference model in ``oracle/prefix_cache.py``, which keys blocks by
their whole token prefix (how-pagedattention-works (aiinfrainterviews.com),
shared-system-prompt paragraph; auto-20261007-1900-en (lihaoran.work), "Shared
prefixes need matching computation").  Physical block ids are the library's
choice, so tables are compared through their sharing structure (no GPU)."""
import numpy as np
import pytest

from oracle import prefix_cache


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_167_gb300 as pa
    return pa


def same_structure(bm, model, lib_ids, model_ids):
    """Live tables agree up to one renaming of block ids; reference counts of
    the blocks they hold agree; the counters agree."""
    fwd, back = {}, {}
    for s in lib_ids:
        lt, ln = bm.table(lib_ids[s])
        mt, mn = model.seqs[model_ids[s]]
        assert ln == mn and len(lt) == len(mt), s
        for a, b in zip(lt.tolist(), mt):
            assert fwd.setdefault(a, b) == b and back.setdefault(b, a) == a, (s, a, b)
    for a, b in fwd.items():
        assert bm.refcount(a) == model.ref[b], (a, b)
    assert bm.num_free() == model.num_free()
    assert bm.num_cached() == len(model.entries)
    assert bm.num_evictable() == len(model.evictable())
    assert bm.prefix_stats() == (model.hit_tokens, model.query_tokens)


@pytest.mark.parametrize("seed,num_blocks,b", [(0, 64, 4), (1, 40, 2), (2, 200, 16), (3, 24, 8)])
def test_random_walk_against_model(pa, seed, num_blocks, b):
    rng = np.random.default_rng(seed)
    bm = pa.BlockManager(num_blocks, b)
    model = prefix_cache.PrefixCacheModel(num_blocks, b)
    prompts = [rng.integers(0, 3, int(rng.integers(1, 5 * b))).tolist() for _ in range(4)]
    lib_ids, model_ids, tokens = {}, {}, {}
    nxt = 0
    for step in range(700):
        op = rng.choice(["add", "append", "cache", "fork", "free", "evict", "probe"],
                        p=[0.2, 0.3, 0.15, 0.05, 0.15, 0.05, 0.1])
        if op == "add" or not lib_ids:
            toks = list(prompts[rng.integers(len(prompts))]) + rng.integers(0, 3, int(rng.integers(0, 3 * b))).tolist()
            cond = int(rng.integers(0, 2))
            ls, lm = bm.add_seq_cached(toks, cond)
            ms, mm = model.add_seq_cached(toks, cond)
            assert lm == mm, (step, toks)
            lib_ids[nxt], model_ids[nxt], tokens[nxt] = ls, ms, (toks, cond)
            nxt += 1
            continue
        s = list(lib_ids)[rng.integers(len(lib_ids))]
        if op == "append":
            toks, cond = tokens[s]
            _, have = model.seqs[model_ids[s]]
            n = int(rng.integers(1, 3 * b))
            extra = toks[have:have + n]
            extra += rng.integers(0, 3, n - len(extra)).tolist()
            try:
                model_pair = model.append(model_ids[s], n)
                model_ok = True
            except prefix_cache.NoBlocks:
                model_ok = False
            try:
                _, lib_pair = bm.append_tokens(lib_ids[s], n)
                lib_ok = True
            except pa.PagedAttentionError as e:
                assert e.status == 6
                lib_ok = False
            assert lib_ok == model_ok, step
            if lib_ok:
                assert (lib_pair is None) == (model_pair is None), step
                tokens[s] = (toks[:have] + extra, cond)
        elif op == "cache":
            toks, cond = tokens[s]
            _, have = model.seqs[model_ids[s]]
            n = int(rng.integers(0, have + 1))
            assert bm.cache_seq(lib_ids[s], toks[:n], cond) == model.cache_seq(model_ids[s], toks[:n], cond), step
        elif op == "fork":
            c = nxt
            nxt += 1
            lib_ids[c], model_ids[c] = bm.fork(lib_ids[s]), model.fork(model_ids[s])
            tokens[c] = (list(tokens[s][0]), tokens[s][1])
        elif op == "free":
            bm.free_seq(lib_ids.pop(s))
            model.free_seq(model_ids.pop(s))
            tokens.pop(s)
        elif op == "evict":
            n = int(rng.integers(0, 4))
            assert bm.prefix_evict(n) == model.evict(n), step
        else:
            toks = list(prompts[rng.integers(len(prompts))]) + rng.integers(0, 3, int(rng.integers(0, 2 * b))).tolist()
            cond = int(rng.integers(0, 2))
            assert bm.prefix_match(toks, cond) == model.prefix_match(toks, cond), step
        same_structure(bm, model, lib_ids, model_ids)
        if step % 50 == 0:
            for toks in prompts:
                for cond in (0, 1):
                    assert bm.prefix_match(toks * 3, cond) == model.prefix_match(toks * 3, cond)


def test_shared_system_prompt(pa):
    """The page's 2,000-token prompt over 200 conversations: 125 blocks held
    once, every table starting with them, each counting 200 tables + the cache."""
    P, n, b = 2000, 200, 16
    bm = pa.BlockManager(12000, b)
    rng = np.random.default_rng(5)
    prompt = rng.integers(0, 128000, P).tolist()
    s0, hit = bm.add_seq_cached(prompt)
    assert hit == 0
    bm.append_tokens(s0, P)
    assert bm.cache_seq(s0, prompt) == P // b
    heads = set()
    for _ in range(n - 1):
        s, hit = bm.add_seq_cached(prompt + rng.integers(0, 128000, 850).tolist())
        assert hit == P
        _, cow = bm.append_tokens(s, 850)
        assert cow is None                       # the shared blocks are full: nothing to copy
        heads.add(tuple(bm.table(s)[0][:P // b].tolist()))
    bm.append_tokens(s0, 850)
    heads.add(tuple(bm.table(s0)[0][:P // b].tolist()))
    assert len(heads) == 1
    assert all(bm.refcount(blk) == n + 1 for blk in next(iter(heads)))
    assert bm.num_free() == 12000 - P // b - n * 54
    assert bm.prefix_stats()[0] == (n - 1) * P


def test_swapped_sequence_keeps_cache(pa):
    """Swapping out a sequence that holds cached blocks leaves them cached and
    evictable; swapping it back gives it private blocks."""
    bm = pa.BlockManager(16, 4)
    bm.set_host_pool(8)
    toks = list(range(8))
    s, _ = bm.add_seq_cached(toks)
    bm.append_tokens(s, 8)
    bm.cache_seq(s, toks)
    assert bm.num_evictable() == 0
    pairs = bm.swap_out(s)
    assert len(pairs) == 2 and bm.num_evictable() == 2 and bm.num_cached() == 2
    assert bm.prefix_match(toks) == 8
    back = bm.swap_in(s)
    assert len(back) == 2 and not set(back[:, 0].tolist()) & set(pairs[:, 0].tolist())
    assert bm.num_evictable() == 2


def test_allocation_evicts_when_pool_is_dry(pa):
    bm = pa.BlockManager(4, 2)
    for toks in ([1, 2, 3, 4], [5, 6, 7, 8]):
        s, _ = bm.add_seq_cached(toks)
        bm.append_tokens(s, 4)
        bm.cache_seq(s, toks)
        bm.free_seq(s)
    assert bm.num_free() == 0 and bm.num_evictable() == 4
    assert bm.can_admit(5)                       # ceil(5/2) + 1 = 4 blocks, all evictable
    assert not bm.can_admit(7)
    d = bm.add_seq()
    bm.append_tokens(d, 6)
    assert bm.num_cached() == 1 and bm.num_evictable() == 1 and bm.num_free() == 0
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.append_tokens(d, 4)
    assert e.value.status == 6
    assert bm.table(d)[1] == 6                   # unchanged by the refused append


def test_errors(pa):
    bm = pa.BlockManager(8, 4)
    s = bm.add_seq()
    bm.append_tokens(s, 4)
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.cache_seq(s, list(range(5)))          # more tokens than the sequence holds
    assert e.value.status == 1
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.cache_seq(99, [1, 2, 3, 4])
    assert e.value.status == 7
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.prefix_evict(-1)
    assert e.value.status == 1
    bm.set_host_pool(4)
    bm.swap_out(s)
    with pytest.raises(pa.PagedAttentionError) as e:
        bm.cache_seq(s, [1, 2, 3, 4])
    assert e.value.status == 8
    assert bm.prefix_match([]) == 0 and bm.add_seq_cached([])[1] == 0
