"""GPU parity of chunked causal prefill (tcgen05 path) against the oracle,
through the C ABI: the chunk's K/V are written by the slot writer, then the
chunk's queries attend the paged context causally."""
import numpy as np
import pytest
import torch

import pa_workloads as wl
from tests.parity import Case, assert_close

pytestmark = pytest.mark.gpu

bits = wl.bf16_bits


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_167_gb300 as pa
    assert torch.cuda.is_available(), "a CUDA device is required"
    pa.get_device_error(clear=True)
    return pa


def run_prefill(pa, c: Case, junk_tail: bool = False):
    w = c.w
    slots = pa.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size, w.num_blocks)
    oslots = c.orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size)
    assert np.array_equal(slots, oslots)
    if junk_tail:   # non-finite junk in every slot past each sequence's end
        nan = torch.full((w.head_dim,), float("nan"), dtype=torch.bfloat16, device=c.dev)
        for s, L in enumerate(w.seq_lens):
            if L % w.block_size:
                blk = int(w.tables[s, (L - 1) // w.block_size])
                c.pool[blk, :, :, L % w.block_size:, :] = nan
    pa.reshape_and_cache(c.pool, c.new_k, c.new_v, torch.as_tensor(slots, device=c.dev))
    c.orc.reshape_and_cache(c.pool_ref, c.geom, bits(c.cpu["new_k"]), bits(c.cpu["new_v"]), oslots)
    out = torch.full_like(c.q, float("nan"))
    ctx = torch.as_tensor(w.ctx_lens, device=c.dev)
    pa.prefill_chunk(out, c.q, c.pool, c.tables, ctx, int(w.ctx_lens.max()), w.scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    return out


def oracle_prefill(c: Case, rows=None):
    w = c.w
    return c.orc.prefill(bits(c.cpu["q"]), c.pool_ref, c.geom, w.tables, w.ctx_lens, w.num_q_heads, w.scale,
                         rows=rows)


@pytest.mark.parametrize("group,hkv,ctx,chunk", [
    (8, 2, [0, 37], 45),        # ragged last M-tile, empty context, context not a block multiple
    (8, 1, [130], 16),          # one full M-tile
    (4, 2, [7, 64], 40),
    (2, 2, [300, 1], 70),
    (1, 2, [5, 200], 130),      # 128 queries per M-tile, second tile ragged
])
def test_prefill_small(pa, group, hkv, ctx, chunk):
    w = wl.prefill_chunk(batch=len(ctx), ctx=ctx, chunk=chunk, num_blocks=128, num_q_heads=group * hkv,
                         num_kv_heads=hkv, seed=500 + group + chunk)
    c = Case(w)
    out = run_prefill(pa, c)
    assert_close(out, oracle_prefill(c), f"G={group} ctx={ctx} C={chunk}")


@pytest.mark.parametrize("bs", [8, 32, 64])
@pytest.mark.parametrize("group,hkv,ctx,chunk", [
    (8, 2, [0, 37], 45),
    (2, 2, [300, 1], 70),
    (1, 1, [129, 600], 130),
])
def test_prefill_block_sizes(pa, bs, group, hkv, ctx, chunk):
    """Block sizes other than 16: a 128-key tile spans 16, 4 or 2 blocks."""
    w = wl.prefill_chunk(batch=len(ctx), ctx=ctx, chunk=chunk, num_blocks=256, num_q_heads=group * hkv,
                         num_kv_heads=hkv, seed=700 + bs + group + chunk, block_size=bs)
    c = Case(w)
    out = run_prefill(pa, c, junk_tail=True)
    assert not torch.isnan(out).any()
    assert_close(out, oracle_prefill(c), f"b={bs} G={group} ctx={ctx} C={chunk}")


def test_prefill_junk_past_sequence_end(pa):
    w = wl.prefill_chunk(batch=2, ctx=[33, 100], chunk=21, num_blocks=64, num_q_heads=16, num_kv_heads=2, seed=77)
    c = Case(w)
    out = run_prefill(pa, c, junk_tail=True)
    assert not torch.isnan(out).any()
    assert_close(out, oracle_prefill(c), "junk tail")


def test_prefill_full_size(pa):
    """16 sequences x (4096 cached + 512 chunk tokens), 64/8 heads: sampled rows."""
    w = wl.prefill_chunk()
    c = Case(w)
    out = run_prefill(pa, c)
    rng = np.random.default_rng(9)
    n = 1536
    rows = np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.chunk, n), rng.integers(0, w.num_q_heads, n)], 1)
    rows[:64, 1] = w.chunk - 1            # include the last query of the chunk
    rows[64:128, 1] = 0                   # and the first
    ref = oracle_prefill(c, rows)
    assert_close(out[rows[:, 0], rows[:, 1], rows[:, 2]], ref, "prefill full size")


def test_prefill_repeatable_under_contention(pa):
    """Chunked prefill (4 sequences x (1,000 .. 3,000 cached + 256 chunk
    tokens), ragged last key tiles) twelve times, every other time while a
    second stream copies gigabytes: every output is bit-identical to the
    first, and the first matches the oracle on sampled rows.  Late K/V tiles
    must not let the epilogue read O before the last P.V has completed."""
    w = wl.prefill_chunk(batch=4, ctx=[1000, 3000, 2017, 1500], chunk=256, num_blocks=2048, seed=91)
    c = Case(w)
    first = run_prefill(pa, c)
    rng = np.random.default_rng(13)
    n = 512
    rows = np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.chunk, n), rng.integers(0, w.num_q_heads, n)], 1)
    rows[:32, 1] = w.chunk - 1
    assert_close(first[rows[:, 0], rows[:, 1], rows[:, 2]], oracle_prefill(c, rows), "prefill repeat")
    side = torch.cuda.Stream()
    src = torch.empty(1 << 30, dtype=torch.uint8, device=c.dev)
    dst = torch.empty_like(src)
    ctx = torch.as_tensor(w.ctx_lens, device=c.dev)
    for rep in range(12):
        if rep % 2:
            with torch.cuda.stream(side):
                for _ in range(3):
                    dst.copy_(src)
        out = torch.full_like(c.q, float("nan"))
        pa.prefill_chunk(out, c.q, c.pool, c.tables, ctx, int(w.ctx_lens.max()), w.scale)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        assert torch.equal(out, first), f"prefill output differs at run {rep}"


@pytest.mark.parametrize("group,hkv,ctx,chunk", [
    (4, 2, [0, 300, 1000], 70),      # 3 M-tiles x 2 heads x 3 sequences = 18 units, one of them empty of context
    (8, 2, [40] * 10, 256),          # 320 units: one CTA may hold at most 256, so a grid of 1 becomes 2
])
def test_prefill_persistent_grid_sweep(pa, group, hkv, ctx, chunk):
    """The persistent grid walks its units in rounds and hands the copy and
    tensor-core pipeline from one unit to the next inside a CTA.  Every grid
    size from one CTA (every unit in one CTA) to one per unit gives the same
    output bit for bit, and the default grid matches the oracle."""
    w = wl.prefill_chunk(batch=len(ctx), ctx=ctx, chunk=chunk, num_blocks=1024, num_q_heads=group * hkv,
                         num_kv_heads=hkv, seed=900 + group + chunk)
    c = Case(w)
    base = run_prefill(pa, c)
    if len(ctx) <= 3:
        assert_close(base, oracle_prefill(c), f"G={group} ctx={ctx} C={chunk}")
    ctxd = torch.as_tensor(w.ctx_lens, device=c.dev)
    n_units = -(-chunk // (128 // group)) * hkv * len(ctx)
    try:
        for ctas in (1, 2, 3, 5, 7, 17, n_units - 1, n_units, n_units + 5):
            pa.set_prefill_ctas(ctas)
            out = torch.full_like(c.q, float("nan"))
            pa.prefill_chunk(out, c.q, c.pool, c.tables, ctxd, int(w.ctx_lens.max()), w.scale)
            torch.cuda.synchronize()
            assert pa.get_device_error() == 0
            assert torch.equal(out, base), f"{ctas} CTAs: output differs from the default grid's"
    finally:
        pa.set_prefill_ctas(0)
