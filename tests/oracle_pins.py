"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Every pin takes an ``oracle.Oracle`` handle and raises ``AssertionError`` when
the oracle disagrees, so the same pins run against the real oracle
(``test_oracle_pins.py``) and against deliberately broken builds of it
(``test_oracle_mutants.py``).  None of them re-types the oracle's formulas:
each compares it with something else --

* values the pages print (``tests/golden/*.json``, each with its citation),
* a library attention routine (``torch.nn.functional.scaled_dot_product_attention``
  in fp64 on the un-paged tensors),
* pure-Python brute force on tiny inputs (naive softmax, ``math.fsum``),
* closed forms (one key, zero query, constant values),
* invariants the pages state (output independent of physical placement; shared
  prefix blocks equal private copies; C=1 prefill equals decode).

The ``pin_prefix_*`` pins hold the prefix-cache reference model
(``oracle/prefix_cache.py``, the class in ``prefix_model``) to the pages'
shared-prompt example, to the rule that a block matches only after an equal
context, to brute-force longest-prefix search and to hand-worked eviction.

Run as ``python -m tests.oracle_pins --library PATH [--prefix-model FILE]`` to
print a JSON list of the pins that fail for the oracle built at PATH and the
prefix-cache model in FILE (exit status 1 if any fail).
"""
from __future__ import annotations

import json
import math
import os
import sys
from typing import Callable, Dict, List

import numpy as np
import torch
import torch.nn.functional as F

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle as oracle_pkg  # noqa: E402
from oracle import prefix_cache as prefix_model  # noqa: E402

BF16 = torch.bfloat16


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(BF16)


def randn(shape, gen) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(BF16)


def place(K: torch.Tensor, V: torch.Tensor, lens, tables, num_blocks: int, block_size: int,
          gen) -> torch.Tensor:
    """Test-side placement of contiguous K/V ([B][Lmax][Hkv][d]) into a fresh
    pool [NB][2][Hkv][b][d] (slots not covered stay random junk)."""
    B, _, H, d = K.shape
    pool = randn((num_blocks, 2, H, block_size, d), gen)
    for s in range(B):
        for t in range(int(lens[s])):
            blk, off = int(tables[s][t // block_size]), t % block_size
            pool[blk, 0, :, off, :] = K[s, t]
            pool[blk, 1, :, off, :] = V[s, t]
    return pool


def random_tables(rng, lens, num_blocks: int, block_size: int) -> np.ndarray:
    counts = [-(-int(L) // block_size) for L in lens]
    tables = np.full((len(lens), max(1, max(counts))), -1, dtype=np.int32)
    perm = rng.permutation(num_blocks)
    c = 0
    for s, n in enumerate(counts):
        tables[s, :n] = perm[c:c + n]
        c += n
    return tables


def sdpa_rows(q_rows: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float,
              mask=None) -> torch.Tensor:
    """Library attention in fp64.  q_rows [M][Hq][d], K/V [L][Hkv][d];
    GQA by repeating each kv-head over its consecutive group of q-heads."""
    Hq, Hkv = q_rows.shape[1], K.shape[1]
    G = Hq // Hkv
    qq = q_rows.double().permute(1, 0, 2).unsqueeze(0)                      # [1][Hq][M][d]
    kk = K.double().permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)  # [1][Hq][L][d]
    vv = V.double().permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
    return o.squeeze(0).permute(1, 0, 2)                                      # [M][Hq][d]


# ---------------------------------------------------------------------------
# capacity arithmetic and address map
# ---------------------------------------------------------------------------

def pin_block_layout_page_example(orc):
    g = golden("block_layout_page_example.json")
    b = g["block_size"]
    for tokens, expect in g["cases"]:
        assert orc.block_layout(tokens, b) == tuple(expect), (tokens, expect)
    assert orc.block_layout(g["printed"]["tokens"], b) == tuple(g["printed"]["layout"])
    tb = g["tail_bound"]
    for n in range(tb["tokens_from"], tb["tokens_to_exclusive"]):
        blocks, unused = orc.block_layout(n, b)
        assert blocks * b >= n and tb["unused_min"] <= unused < tb["unused_max_exclusive"], n
    for tokens, bs in g["invalid"]:
        try:
            orc.block_layout(tokens, bs)
        except ValueError:
            continue
        raise AssertionError(f"block_layout({tokens}, {bs}) accepted an invalid size")


def pin_block_layout_worked_example(orc):
    g = golden("worked_example_blocks.json")
    blocks, unused = orc.block_layout(g["tokens"], g["block_size"])
    assert blocks == g["blocks"], blocks
    for n in range(1, 2000):
        _, unused = orc.block_layout(n, g["block_size"])
        assert 0 <= unused <= g["max_idle_slots"], n
    # exactly-full sequences leave nothing idle, one more token opens a block
    assert orc.block_layout(32, 16) == (2, 0) and orc.block_layout(33, 16) == (3, 15)


def pin_address_page_example(orc):
    g = golden("address_page_example.json")
    phys, off = orc.address(g["table"], g["position"], g["block_size"])
    assert (phys, off) == (g["physical_block"], g["offset"]), (phys, off)
    # the first slot of each logical block lands at offset 0 of the next table entry
    for logical, blk in enumerate(g["table"]):
        assert orc.address(g["table"], logical * g["block_size"], g["block_size"]) == (blk, 0)


def pin_slot_writer_page_example(orc):
    """Write the page's 10 tokens through the slot writer with table [5,1,7] and
    b=4: token 9 must be found at physical block 7, offset 1, and the two tail
    slots of block 7 must stay untouched."""
    g = golden("address_page_example.json")
    b, table, T = g["block_size"], g["table"], g["tokens"]
    H, d, NB = 2, 8, 8
    gen = torch.Generator().manual_seed(11)
    geom = oracle_pkg.dense_geom(NB, H, b, d)
    pool = bits(randn((NB, 2, H, b, d), gen)).copy()
    before = pool.copy()
    k, v = bits(randn((T, H, d), gen)), bits(randn((T, H, d), gen))
    slots = orc.slot_mapping([table], np.zeros(T, np.int32), np.arange(T), b)
    orc.reshape_and_cache(pool, geom, k, v, slots)
    assert np.array_equal(pool[g["physical_block"], 0, :, g["offset"]], k[g["position"]])
    assert np.array_equal(pool[g["physical_block"], 1, :, g["offset"]], v[g["position"]])
    # tokens 0..3 fill block 5, 4..7 fill block 1, 8..9 the head of block 7
    for t in range(T):
        blk, off = table[t // b], t % b
        assert np.array_equal(pool[blk, 0, :, off], k[t]) and np.array_equal(pool[blk, 1, :, off], v[t])
    assert np.array_equal(pool[7, :, :, 2:], before[7, :, :, 2:])
    untouched = [i for i in range(NB) if i not in table]
    assert np.array_equal(pool[untouched], before[untouched])
    # a negative slot is padding: nothing is written
    pool2 = before.copy()
    orc.reshape_and_cache(pool2, geom, k[:3], v[:3], [-1, -1, -1])
    assert np.array_equal(pool2, before)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

DECODE_CASES = [
    # B, Hq, Hkv, d, b, lens, NB, seed
    (4, 4, 2, 16, 4, [1, 7, 13, 4], 24, 1),
    (2, 8, 1, 32, 16, [33, 5], 12, 2),
    (3, 8, 8, 8, 2, [9, 1, 6], 20, 3),
    (2, 6, 2, 64, 16, [70, 16], 10, 4),
]


def _decode_case(case):
    B, Hq, Hkv, d, b, lens, NB, seed = case
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    Lmax = max(lens)
    K, V = randn((B, Lmax, Hkv, d), gen), randn((B, Lmax, Hkv, d), gen)
    q = randn((B, Hq, d), gen)
    tables = random_tables(rng, lens, NB, b)
    pool = place(K, V, lens, tables, NB, b, gen)
    geom = oracle_pkg.dense_geom(NB, Hkv, b, d)
    return q, K, V, tables, pool, geom, np.asarray(lens, np.int32), 1.0 / math.sqrt(d)


def pin_decode_vs_sdpa(orc):
    for case in DECODE_CASES:
        q, K, V, tables, pool, geom, lens, scale = _decode_case(case)
        got = orc.paged_decode(bits(q), bits(pool), geom, tables, lens, q.shape[1], scale)
        for s in range(len(lens)):
            ref = sdpa_rows(q[s:s + 1], K[s, :lens[s]], V[s, :lens[s]], scale)[0].numpy()
            err = np.abs(got[s] - ref).max()
            assert err < 1e-10, (case, s, err)
        rows = np.asarray([[s, h] for s in range(len(lens)) for h in range(q.shape[1])][::3])
        sub = orc.paged_decode(bits(q), bits(pool), geom, tables, lens, q.shape[1], scale, rows=rows)
        assert np.array_equal(sub, got[rows[:, 0], rows[:, 1]])


def pin_decode_brute_force(orc):
    """Naive softmax in pure Python (no max subtraction, math.fsum) on tiny inputs."""
    B, Hq, Hkv, d, b, lens, NB = 2, 4, 2, 4, 2, [3, 5], 8
    rng = np.random.default_rng(5)
    gen = torch.Generator().manual_seed(5)
    K, V = randn((B, 5, Hkv, d), gen), randn((B, 5, Hkv, d), gen)
    q = randn((B, Hq, d), gen)
    tables = random_tables(rng, lens, NB, b)
    pool = place(K, V, lens, tables, NB, b, gen)
    scale = 0.37
    got = orc.paged_decode(bits(q), bits(pool), oracle_pkg.dense_geom(NB, Hkv, b, d), tables,
                           np.asarray(lens, np.int32), Hq, scale)
    Kf, Vf, qf = K.double().tolist(), V.double().tolist(), q.double().tolist()
    for s in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            w = [math.exp(scale * math.fsum(qf[s][h][i] * Kf[s][t][g][i] for i in range(d)))
                 for t in range(lens[s])]
            z = math.fsum(w)
            for i in range(d):
                ref = math.fsum(w[t] * Vf[s][t][g][i] for t in range(lens[s])) / z
                assert abs(got[s, h, i] - ref) <= 1e-12 * max(1.0, abs(ref)), (s, h, i)


def pin_decode_closed_forms(orc):
    B, Hq, Hkv, d, b, NB = 3, 4, 2, 16, 4, 16
    rng = np.random.default_rng(6)
    gen = torch.Generator().manual_seed(6)
    geom = oracle_pkg.dense_geom(NB, Hkv, b, d)
    # one key: the output is that key's value row, exactly
    lens = [1, 1, 1]
    K, V, q = randn((B, 1, Hkv, d), gen), randn((B, 1, Hkv, d), gen), randn((B, Hq, d), gen)
    tables = random_tables(rng, lens, NB, b)
    pool = place(K, V, lens, tables, NB, b, gen)
    out = orc.paged_decode(bits(q), bits(pool), geom, tables, np.asarray(lens, np.int32), Hq, 0.25)
    for s in range(B):
        for h in range(Hq):
            assert np.array_equal(out[s, h], V[s, 0, h // 2].double().numpy()), (s, h)
    # zero query: every key weighs the same, the output is the mean of V
    lens = [5, 9, 12]
    K, V = randn((B, 12, Hkv, d), gen), randn((B, 12, Hkv, d), gen)
    q = torch.zeros((B, Hq, d), dtype=BF16)
    tables = random_tables(rng, lens, NB, b)
    pool = place(K, V, lens, tables, NB, b, gen)
    out = orc.paged_decode(bits(q), bits(pool), geom, tables, np.asarray(lens, np.int32), Hq, 0.25)
    for s in range(B):
        mean = V[s, :lens[s]].double().mean(dim=0).numpy()
        for h in range(Hq):
            assert np.abs(out[s, h] - mean[h // 2]).max() < 1e-13, (s, h)
    # all value rows equal c: the output is c whatever the scores
    q = randn((B, Hq, d), gen)
    c = randn((Hkv, d), gen)
    V = c.unsqueeze(0).unsqueeze(0).expand(B, 12, Hkv, d).contiguous()
    pool = place(K, V, lens, tables, NB, b, gen)
    out = orc.paged_decode(bits(q), bits(pool), geom, tables, np.asarray(lens, np.int32), Hq, 0.25)
    for s in range(B):
        for h in range(Hq):
            assert np.abs(out[s, h] - c[h // 2].double().numpy()).max() < 1e-13, (s, h)


def pin_decode_placement_invariance(orc):
    """Same logical K/V under two random physical placements: identical output."""
    q, K, V, tables, pool, geom, lens, scale = _decode_case(DECODE_CASES[0])
    rng = np.random.default_rng(99)
    gen = torch.Generator().manual_seed(99)
    tables2 = random_tables(rng, lens, geom.num_blocks, geom.block_size)
    pool2 = place(K, V, lens, tables2, geom.num_blocks, geom.block_size, gen)
    a = orc.paged_decode(bits(q), bits(pool), geom, tables, lens, q.shape[1], scale)
    b = orc.paged_decode(bits(q), bits(pool2), geom, tables2, lens, q.shape[1], scale)
    assert not np.array_equal(tables, tables2)
    assert np.array_equal(a, b)


def pin_decode_shared_prefix(orc):
    """Tables sharing physical prefix blocks give the same result as tables
    holding private copies of the same prefix."""
    Hq, Hkv, d, b, NB = 4, 2, 8, 4, 40
    gen = torch.Generator().manual_seed(7)
    prefix_tokens, lens = 8, [11, 14, 8]
    B = len(lens)
    Kp, Vp = randn((prefix_tokens, Hkv, d), gen), randn((prefix_tokens, Hkv, d), gen)
    K, V = randn((B, 14, Hkv, d), gen), randn((B, 14, Hkv, d), gen)
    K[:, :prefix_tokens], V[:, :prefix_tokens] = Kp, Vp
    q = randn((B, Hq, d), gen)
    # private: every sequence has its own copy of the prefix blocks
    priv = np.asarray([[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, -1, -1]], np.int32)
    pool_priv = place(K, V, lens, priv, NB, b, gen)
    # shared: one copy of the two prefix blocks, every table starts with them
    shared = np.asarray([[20, 21, 30, -1], [20, 21, 31, 32], [20, 21, -1, -1]], np.int32)
    pool_sh = place(K, V, lens, shared, NB, b, gen)
    geom = oracle_pkg.dense_geom(NB, Hkv, b, d)
    a = orc.paged_decode(bits(q), bits(pool_priv), geom, priv, np.asarray(lens, np.int32), Hq, 0.3)
    c = orc.paged_decode(bits(q), bits(pool_sh), geom, shared, np.asarray(lens, np.int32), Hq, 0.3)
    assert np.array_equal(a, c)


def pin_decode_lse(orc):
    """The log-sum-exp log(sum_t exp(scale q.K_t)) that a cascade merges by:
    log(n) for a zero query; scale q.k + log(n) when every key is k; a naive
    pure-Python sum on tiny inputs; and the merge identity -- attention over
    a prefix and a suffix, weighted by exp(lse), is attention over both."""
    Hq, Hkv, d, b, NB = 4, 2, 8, 4, 32
    gen = torch.Generator().manual_seed(11)
    rng = np.random.default_rng(11)
    geom = oracle_pkg.dense_geom(NB, Hkv, b, d)
    lens = [3, 9, 16, 1]
    B = len(lens)
    K, V = randn((B, 16, Hkv, d), gen), randn((B, 16, Hkv, d), gen)
    tables = random_tables(rng, lens, NB, b)
    pool = place(K, V, lens, tables, NB, b, gen)
    L = np.asarray(lens, np.int32)
    out0, lse0 = orc.paged_decode_lse(np.zeros((B, Hq, d), np.uint16), bits(pool), geom, tables, L, Hq, 0.3)
    assert np.abs(lse0 - np.log(L)[:, None]).max() < 1e-13
    q = randn((B, Hq, d), gen)
    out, lse = orc.paged_decode_lse(bits(q), bits(pool), geom, tables, L, Hq, 0.3)
    assert np.array_equal(out, orc.paged_decode(bits(q), bits(pool), geom, tables, L, Hq, 0.3))
    qf, Kf = q.double().tolist(), K.double().tolist()
    for s in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            z = math.fsum(math.exp(0.3 * math.fsum(qf[s][h][i] * Kf[s][t][g][i] for i in range(d)))
                          for t in range(lens[s]))
            assert abs(lse[s, h] - math.log(z)) < 1e-12, (s, h)
    # every key equal to k: each score is scale q.k
    k = randn((Hkv, d), gen)
    Ke = k.unsqueeze(0).unsqueeze(0).expand(B, 16, Hkv, d).contiguous()
    pool_e = place(Ke, V, lens, tables, NB, b, gen)
    _, lse_e = orc.paged_decode_lse(bits(q), bits(pool_e), geom, tables, L, Hq, 0.3)
    for s in range(B):
        for h in range(Hq):
            dot = math.fsum(qf[s][h][i] * float(k[h // 2, i]) for i in range(d))
            assert abs(lse_e[s, h] - (0.3 * dot + math.log(lens[s]))) < 1e-12, (s, h)
    # merge identity: the first two blocks as a prefix, the rest as a suffix
    full = [16, 12, 9]
    Bf = len(full)
    tab = random_tables(rng, full, NB, b)
    Kf2, Vf2 = randn((Bf, 16, Hkv, d), gen), randn((Bf, 16, Hkv, d), gen)
    pool_f = place(Kf2, Vf2, full, tab, NB, b, gen)
    qm = randn((Bf, Hq, d), gen)
    o_all, l_all = orc.paged_decode_lse(bits(qm), bits(pool_f), geom, tab, np.asarray(full, np.int32), Hq, 0.3)
    o_a, l_a = orc.paged_decode_lse(bits(qm), bits(pool_f), geom, tab[:, :2], np.full(Bf, 2 * b, np.int32), Hq, 0.3)
    o_b, l_b = orc.paged_decode_lse(bits(qm), bits(pool_f), geom, np.ascontiguousarray(tab[:, 2:]),
                                    np.asarray(full, np.int32) - 2 * b, Hq, 0.3)
    M = np.maximum(l_a, l_b)
    wa, wb = np.exp(l_a - M)[..., None], np.exp(l_b - M)[..., None]
    assert np.abs((wa * o_a + wb * o_b) / (wa + wb) - o_all).max() < 1e-13
    assert np.abs(np.logaddexp(l_a, l_b) - l_all).max() < 1e-12
    # no keys: -inf and zeros
    o_z, l_z = orc.paged_decode_lse(bits(qm), bits(pool_f), geom, tab, np.zeros(Bf, np.int32), Hq, 0.3)
    assert np.all(np.isneginf(l_z)) and not o_z.any()


def pin_decode_layered_pool(orc):
    """The pages' pool shape [NB][2][layers][Hkv][b][d]: a layer's view through
    strides equals a dense pool holding only that layer."""
    B, Hq, Hkv, d, b, NB, layers = 2, 4, 2, 8, 4, 12, 3
    rng = np.random.default_rng(8)
    gen = torch.Generator().manual_seed(8)
    lens = np.asarray([7, 10], np.int32)
    tables = random_tables(rng, lens, NB, b)
    pool3 = bits(randn((NB, 2, layers, Hkv, b, d), gen))
    q = randn((B, Hq, d), gen)
    for layer in range(layers):
        dense = np.ascontiguousarray(pool3[:, :, layer])
        a = orc.paged_decode(bits(q), dense, oracle_pkg.dense_geom(NB, Hkv, b, d), tables, lens, Hq, 0.3)
        view = pool3.reshape(-1)[layer * Hkv * b * d:]
        geom = oracle_pkg.dense_geom(NB, Hkv, b, d, num_layers=layers)
        c = orc.paged_decode(bits(q), view, geom, tables, lens, Hq, 0.3)
        assert np.array_equal(a, c), layer


def pin_prefill_vs_sdpa(orc):
    """Chunk queries at positions ctx..ctx+C-1 against causal, paged keys."""
    Hq, Hkv, d, b, NB, C = 4, 2, 16, 4, 24, 5
    ctx = [0, 7, 3]
    B = len(ctx)
    rng = np.random.default_rng(9)
    gen = torch.Generator().manual_seed(9)
    total = [c + C for c in ctx]
    K, V = randn((B, max(total), Hkv, d), gen), randn((B, max(total), Hkv, d), gen)
    q = randn((B, C, Hq, d), gen)
    tables = random_tables(rng, total, NB, b)
    pool = place(K, V, total, tables, NB, b, gen)
    geom = oracle_pkg.dense_geom(NB, Hkv, b, d)
    scale = 1.0 / math.sqrt(d)
    got = orc.prefill(bits(q), bits(pool), geom, tables, np.asarray(ctx, np.int32), Hq, scale)
    for s in range(B):
        L = total[s]
        key_pos = torch.arange(L)
        mask = key_pos[None, :] <= (ctx[s] + torch.arange(C))[:, None]        # [C][L]
        ref = sdpa_rows(q[s], K[s, :L], V[s, :L], scale, mask=mask.unsqueeze(0).unsqueeze(0))
        err = np.abs(got[s] - ref.numpy()).max()
        assert err < 1e-10, (s, err)
    rows = np.asarray([[s, j, h] for s in range(B) for j in range(C) for h in range(Hq)][::5])
    sub = orc.prefill(bits(q), bits(pool), geom, tables, np.asarray(ctx, np.int32), Hq, scale, rows=rows)
    assert np.array_equal(sub, got[rows[:, 0], rows[:, 1], rows[:, 2]])


def pin_prefill_one_query_is_decode(orc):
    """A chunk of one query at position ctx is a decode step over ctx+1 keys."""
    q, K, V, tables, pool, geom, lens, scale = _decode_case(DECODE_CASES[3])
    ctx = lens - 1
    pre = orc.prefill(bits(q.unsqueeze(1)), bits(pool), geom, tables, ctx, q.shape[1], scale)
    dec = orc.paged_decode(bits(q), bits(pool), geom, tables, lens, q.shape[1], scale)
    assert np.array_equal(pre[:, 0], dec)


# ---------------------------------------------------------------------------
# copy-on-write
# ---------------------------------------------------------------------------

def pin_copy_blocks(orc):
    """After a fork copy, each dst block holds its src block's K and V; reading
    a sequence through dst gives what reading it through src gave."""
    for layers in (1, 2):
        NB, Hkv, b, d = 10, 2, 4, 8
        gen = torch.Generator().manual_seed(10 + layers)
        pool = bits(randn((NB, 2, layers, Hkv, b, d), gen)).copy()
        before = pool.copy()
        pairs = np.asarray([[3, 5], [0, 6], [9, 2]], np.int32)
        geom = oracle_pkg.dense_geom(NB, Hkv, b, d, num_layers=layers)
        flat = pool.reshape(-1)
        orc.copy_blocks(flat[(layers - 1) * Hkv * b * d:], geom, pairs)
        for src, dst in pairs:
            assert np.array_equal(pool[dst, :, layers - 1], before[src, :, layers - 1]), (src, dst)
            if layers > 1:
                assert np.array_equal(pool[dst, :, 0], before[dst, :, 0])
        others = [i for i in range(NB) if i not in pairs[:, 1]]
        assert np.array_equal(pool[others], before[others])
    q = randn((1, 4, d), gen)
    lens = np.asarray([4 * b], np.int32)
    pool1 = bits(randn((NB, 2, Hkv, b, d), gen)).copy()
    g1 = oracle_pkg.dense_geom(NB, Hkv, b, d)
    t_src = np.asarray([[3, 0, 9, 1]], np.int32)
    a = orc.paged_decode(bits(q), pool1, g1, t_src, lens, 4, 0.3)
    orc.copy_blocks(pool1, g1, [[3, 5], [0, 6], [9, 2], [1, 4]])
    c = orc.paged_decode(bits(q), pool1, g1, np.asarray([[5, 6, 2, 4]], np.int32), lens, 4, 0.3)
    assert np.array_equal(a, c)


# ---------------------------------------------------------------------------
# swapping to host memory
# ---------------------------------------------------------------------------

def pin_swap_blocks(orc):
    """Swap-out puts in host slot hb exactly the K and V rows of the tokens the
    test placed in device block blk; swap-in into other device blocks then
    reads back, through a table pointing at them, what the original table
    read (library attention on the un-paged tensors)."""
    rng = np.random.default_rng(31)
    gen = torch.Generator().manual_seed(31)
    NB, Hkv, Hq, b, d = 12, 2, 4, 4, 8
    lens = [11]
    tables = np.asarray([[7, 2, 9]], np.int32)
    K, V = randn((1, 12, Hkv, d), gen), randn((1, 12, Hkv, d), gen)
    pool = bits(place(K, V, lens, tables, NB, b, gen)).copy()
    geom = oracle_pkg.dense_geom(NB, Hkv, b, d)
    host = np.zeros((5, 2, Hkv, b, d), np.uint16)
    out_pairs = np.asarray([[7, 3], [2, 0], [9, 4]], np.int32)
    orc.swap_blocks(pool, geom, host, out_pairs, 0)
    for j, (blk, hb) in enumerate(out_pairs):
        for off in range(b):
            t = j * b + off
            if t < lens[0]:
                assert np.array_equal(host[hb, 0, :, off], bits(K[0, t])), (blk, hb, off)
                assert np.array_equal(host[hb, 1, :, off], bits(V[0, t])), (blk, hb, off)
    assert not host[1].any() and not host[2].any()        # unused host slots untouched
    before = pool.copy()
    in_pairs = np.asarray([[0, 3], [5, 0], [11, 4]], np.int32)
    orc.swap_blocks(pool, geom, host, in_pairs, 1)
    others = [i for i in range(NB) if i not in in_pairs[:, 0]]
    assert np.array_equal(pool[others], before[others])
    q = randn((1, Hq, d), gen)
    got = orc.paged_decode(bits(q), pool, geom, np.asarray([[0, 5, 11]], np.int32), np.asarray(lens, np.int32),
                           Hq, 0.5)
    ref = sdpa_rows(q, K[0, :lens[0]], V[0, :lens[0]], 0.5)[0].numpy()
    assert np.abs(got[0] - ref).max() < 1e-12


# ---------------------------------------------------------------------------
# capacity of a KV budget, contiguous against paged
# ---------------------------------------------------------------------------

def pin_capacity_worked_example(orc):
    """The page's Llama 3.1 70B arithmetic: 328 KB a token, 8,192-token
    reservations, an 850-token chat request, 16-token blocks, 435 GB."""
    g = golden("capacity_worked_example.json")
    i, pr = g["inputs"], g["printed"]
    bpt, L, b = i["bytes_per_token"], i["request_tokens"], i["block_size"]
    c = orc.capacity([L], 0, b, i["max_seq_len"], bpt, i["budget_bytes"])
    assert round(i["max_seq_len"] * bpt / 1e9, 2) == pr["contiguous_reservation_gb"]
    assert round(L * bpt / 1e9, 2) == pr["used_gb"]
    assert round((i["max_seq_len"] - L) * bpt / 1e9, 2) == pr["waste_gb"]
    assert c["contiguous_requests"] == pr["contiguous_requests"], c
    assert round(c["contiguous_waste"], 2) == pr["waste_fraction"], c
    assert (L + c["mean_tail_slots"]) / b == pr["blocks_per_request"], c
    assert round(b * bpt / 1e6, 1) == pr["block_mb"]
    assert abs(c["paged_requests"] - pr["paged_requests_about"]) <= pr["paged_requests_rel_tol"] * \
        pr["paged_requests_about"], c
    assert round(c["paged_requests"] / c["contiguous_requests"]) == pr["gain_about"], c


def pin_capacity_shared_prefix(orc):
    """A 2,000-token system prompt at 328 KB a token is 656 MB; 200
    conversations hold 131 GB of it when each keeps a copy, 656 MB when its
    blocks are shared.  Shared whole blocks also raise the paged concurrency
    to what the private blocks alone allow."""
    g = golden("capacity_worked_example.json")
    sp, bpt = g["shared_prefix"], g["inputs"]["bytes_per_token"]
    P, n, b = sp["prefix_tokens"], sp["conversations"], 16
    lens = [P + 850] * n
    c = orc.capacity(lens, P, b, 8192, bpt, 435 * 10**9)
    assert round(P * bpt / 1e6) == sp["prefix_mb"]
    assert round(c["prefix_bytes_contiguous"] / 1e9) == sp["contiguous_duplicate_gb"], c
    assert round(c["prefix_bytes_paged"] / 1e6) == sp["paged_mb"], c
    total = (435 * 10**9) // (b * bpt)
    assert c["paged_requests"] == (total - P // b) // -(-(P + 850 - (P // b) * b) // b), c
    # a prefix that ends inside a block: that block stays private to each request
    c2 = orc.capacity([P + 10 + 850] * n, P + 10, b, 8192, bpt, 435 * 10**9)
    assert c2["prefix_bytes_paged"] == ((P // b) * b + n * 10) * bpt, c2


def pin_capacity_small_by_hand(orc):
    """lens (3, 10), b = 4, 12-token reservations, 1 byte a token, 20 bytes:
    one reservation fits; five blocks serve 3 (1 block), 10 (3 blocks), 3 (1
    block), and the next 10 finds none.  Held slots 4 + 12 for 13 tokens."""
    c = orc.capacity([3, 10], 0, 4, 12, 1, 20)
    assert c["contiguous_requests"] == 1 and c["paged_requests"] == 3, c
    assert abs(c["contiguous_waste"] - (1 - 13 / 24)) < 1e-15, c
    assert abs(c["paged_waste"] - (1 - 13 / 16)) < 1e-15, c
    assert c["mean_tail_slots"] == 1.5, c
    # budgets that are exact multiples admit the last reservation / block
    assert orc.capacity([12], 0, 4, 12, 1, 24)["contiguous_requests"] == 2
    assert orc.capacity([12], 0, 4, 12, 1, 24)["paged_requests"] == 2
    assert orc.capacity([12], 0, 4, 12, 1, 23)["contiguous_requests"] == 1
    assert orc.capacity([12], 0, 4, 12, 1, 11)["paged_requests"] == 0
    # zero-token requests hold nothing; the tail bound of the block layout holds per request
    c = orc.capacity([0, 5], 0, 4, 12, 1, 8)
    assert c["paged_requests"] == 3 and c["mean_tail_slots"] == 1.5, c
    for bad in (([], 0), ([5], 6), ([13], 0), ([0], 0)):
        try:
            orc.capacity(bad[0], bad[1], 4, 12, 1, 20)
        except ValueError:
            continue
        raise AssertionError(f"capacity accepted {bad}")


def pin_capacity_chat_mix(orc):
    """Chats averaging about 500 tokens under a 4,096-token maximum leave
    80-95% of max-length reservations unused; with 16-token pages only tail
    slots are lost, under 5%."""
    g = golden("capacity_worked_example.json")["chat_mix"]
    rng = np.random.default_rng(500)
    lens = np.clip(np.rint(rng.lognormal(np.log(420), 0.6, 4000)), 1, g["max_context"]).astype(np.int64)
    assert abs(lens.mean() - g["mean_tokens_about"]) < 50
    c = orc.capacity(lens, 0, 16, g["max_context"], 328000, 435 * 10**9)
    lo, hi = g["reserved_unused_range"]
    assert lo <= c["contiguous_waste"] <= hi, c
    assert c["paged_waste"] < g["paged_waste_below"], c
    assert abs(c["mean_tail_slots"] - 7.5) < 0.5, c            # uniform tails average (b - 1) / 2
    assert c["paged_requests"] > 5 * c["contiguous_requests"], c


# ---------------------------------------------------------------------------
# prefix-cache reference model
# ---------------------------------------------------------------------------

def pin_prefix_shared_system_prompt(orc):
    """how-pagedattention-works, shared-system-prompt paragraph: a 2,000-token
    prompt shared by 200 conversations is one set of 125 blocks that every
    table points at, each block counting 200 tables plus the cache."""
    g = golden("capacity_worked_example.json")["shared_prefix"]
    P, n, b = g["prefix_tokens"], g["conversations"], 16
    m = prefix_model.PrefixCacheModel(12000, b)
    rng = np.random.default_rng(2000)
    prompt = rng.integers(0, 32000, P).tolist()
    s0, hit = m.add_seq_cached(prompt)
    assert hit == 0
    m.append(s0, P)
    assert m.cache_seq(s0, prompt) == P // b
    seqs = [s0]
    for _ in range(n - 1):
        own = rng.integers(0, 32000, 850).tolist()
        s, hit = m.add_seq_cached(prompt + own)
        assert hit == P, hit
        m.append(s, 850)
        seqs.append(s)
    m.append(s0, 850)
    heads = {tuple(m.seqs[s][0][:P // b]) for s in seqs}
    assert len(heads) == 1
    assert all(m.ref[blk] == n + 1 for blk in next(iter(heads)))
    assert m.num_free() == 12000 - P // b - n * (-(-850 // b))
    assert m.hit_tokens == (n - 1) * P


def pin_prefix_context_matters(orc):
    """auto-20261007-1900-en, "Shared prefixes need matching computation": equal
    tokens after another context, or under another condition, do not match."""
    b = 4
    m = prefix_model.PrefixCacheModel(64, b)
    x0, x1, y0, y1 = [1, 2, 3, 4], [5, 6, 7, 8], [9, 9, 9, 9], [8, 7, 6, 5]
    s, _ = m.add_seq_cached(x0 + x1)
    m.append(s, 8)
    assert m.cache_seq(s, x0 + x1) == 2
    assert m.prefix_match(y0 + x1) == 0
    assert m.prefix_match(x0 + y1) == b
    assert m.prefix_match(x0 + x1, condition=1) == 0
    assert m.prefix_match(x0 + x1 + [3, 3]) == 2 * b
    assert m.prefix_match(x0 + x1[:b - 1]) == b          # a partial block is never matched
    assert m.prefix_match(x0[:b - 1]) == 0
    assert m.prefix_match([]) == 0
    # content already cached keeps its entry; the chain continues from it
    t = m.add_seq()
    m.append(t, 12)
    assert m.cache_seq(t, x0 + x1 + y0) == 1
    assert m.prefix_match(x0 + x1 + y0) == 3 * b
    # a block already cached under other content ends publishing
    u = m.add_seq()
    m.append(u, 8)
    assert m.cache_seq(u, y1 + y1) == 2
    assert m.cache_seq(u, y0 + y1) == 0 and m.prefix_match(y0) == 0


def pin_prefix_brute_force(orc):
    """Longest cached prefix in whole blocks equals a direct scan of every
    published token list (no eviction: the pool never runs out)."""
    rng = np.random.default_rng(77)
    b = 2
    m = prefix_model.PrefixCacheModel(10000, b)
    published = []
    for _ in range(40):
        cond = int(rng.integers(0, 2))
        toks = rng.integers(0, 2, int(rng.integers(0, 12))).tolist()
        s = m.add_seq()
        m.append(s, len(toks))
        m.cache_seq(s, toks, cond)
        published.append((cond, toks))
    for _ in range(400):
        cond = int(rng.integers(0, 2))
        q = rng.integers(0, 2, int(rng.integers(0, 14))).tolist()
        best = 0
        for c, toks in published:
            if c != cond:
                continue
            k = 0
            while (k + 1) * b <= min(len(q), len(toks)) and q[:(k + 1) * b] == toks[:(k + 1) * b]:
                k += 1
            best = max(best, k)
        assert m.prefix_match(q, cond) == best * b, (q, cond)


def pin_prefix_lru_hand_worked(orc):
    """Four 2-token blocks.  A = [1,2,3,4] and B = [5,6,7,8] are cached and
    their sequences freed, then A is used again; a sequence needing two blocks
    evicts B's deeper block, then B's first; A stays."""
    m = prefix_model.PrefixCacheModel(4, 2)
    for toks in ([1, 2, 3, 4], [5, 6, 7, 8]):
        s, _ = m.add_seq_cached(toks)
        m.append(s, 4)
        m.cache_seq(s, toks)
        m.free_seq(s)
    assert m.num_free() == 0 and m.available() == 4
    s, hit = m.add_seq_cached([1, 2, 3, 4])
    assert hit == 4
    m.free_seq(s)
    d = m.add_seq()
    m.append(d, 2)
    assert m.prefix_match([5, 6, 7, 8]) == 2 and m.prefix_match([1, 2, 3, 4]) == 4
    m.append(d, 2)
    assert m.prefix_match([5, 6, 7, 8]) == 0 and m.prefix_match([1, 2, 3, 4]) == 4
    # three blocks, one free: a two-block need evicts A's deeper block only
    m = prefix_model.PrefixCacheModel(3, 2)
    s, _ = m.add_seq_cached([1, 2, 3, 4])
    m.append(s, 4)
    m.cache_seq(s, [1, 2, 3, 4])
    m.free_seq(s)
    d = m.add_seq()
    m.append(d, 4)
    assert m.prefix_match([1, 2, 3, 4]) == 2
    try:
        m.append(d, 3)                                   # needs 2 blocks, 1 can be had
    except prefix_model.NoBlocks:
        pass
    else:
        raise AssertionError("append beyond the pool succeeded")
    assert m.prefix_match([1, 2, 3, 4]) == 2


def pin_prefix_evict_subtree(orc):
    """Evicting an entry drops the entries that extend it, even one whose block
    a live sequence holds (the sequence keeps the block)."""
    m = prefix_model.PrefixCacheModel(8, 2)
    a = m.add_seq()
    m.append(a, 2)
    assert m.cache_seq(a, [1, 2]) == 1
    c = m.add_seq()
    m.append(c, 4)
    assert m.cache_seq(c, [1, 2, 3, 4]) == 1               # its block 1 hangs under A's entry
    m.free_seq(a)
    assert len(m.evictable()) == 1 and len(m.entries) == 2
    assert m.evict(1) == 1
    assert len(m.entries) == 0 and m.prefix_match([1, 2, 3, 4]) == 0
    assert m.num_free() == 6
    m.free_seq(c)
    assert m.num_free() == 8


PINS: Dict[str, Callable] = {name: fn for name, fn in globals().items() if name.startswith("pin_")}


def failing_pins(orc) -> List[str]:
    bad = []
    for name, fn in PINS.items():
        try:
            fn(orc)
        except Exception:  # noqa: BLE001 -- any exception means the pin did not hold
            bad.append(name)
    return bad


def main(argv=None) -> int:
    import argparse
    ap = argparse.ArgumentParser()
    ap.add_argument("--library", default=oracle_pkg.LIBRARY)
    ap.add_argument("--prefix-model", default=None)
    args = ap.parse_args(argv)
    if args.prefix_model:
        import importlib.util
        spec = importlib.util.spec_from_file_location("prefix_cache_under_test", args.prefix_model)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        globals()["prefix_model"] = mod
    bad = failing_pins(oracle_pkg.Oracle(args.library))
    print(json.dumps(bad))
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main())
