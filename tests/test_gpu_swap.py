"""GPU parity of block swapping between the pool and pinned host memory
(pa_swap_blocks) against the oracle, through the C ABI.  how-pagedattention-works
(aiinfrainterviews.com), feature table, preemption row, and "What interviewers
probe next": a preempted sequence's blocks go to pinned host memory and come
back at block granularity."""
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


def pinned_host(n, c: Case):
    w = c.w
    return torch.zeros((n, 2, w.num_kv_heads, w.block_size, w.head_dim), dtype=torch.bfloat16, pin_memory=True)


@pytest.mark.parametrize("name", ["tiny", "llama70b_decode"])
def test_swap_out_in_bit_exact(pa, name):
    w = wl.CONFIGS[name]()
    c = Case(w)
    rng = np.random.default_rng(3)
    referenced = np.unique(w.tables[w.tables >= 0])
    n = min(len(referenced), 200)
    dev_blocks = rng.choice(referenced, size=n, replace=False).astype(np.int32)
    host_slots = rng.permutation(n + 7)[:n].astype(np.int32)
    host = pinned_host(n + 7, c)
    host_ref = bits(host).copy()
    out_pairs = np.stack([dev_blocks, host_slots], 1)
    pa.swap_blocks(c.pool, host, torch.as_tensor(out_pairs, device=c.dev), pa.PA_SWAP_OUT)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    c.orc.swap_blocks(c.pool_ref, c.geom, host_ref, out_pairs, 0)
    assert np.array_equal(bits(host), host_ref), "swap-out is not bit-exact"
    # back into blocks nobody references, then the pool must equal the oracle's
    free_blocks = np.setdiff1d(np.arange(w.num_blocks), referenced)
    targets = rng.choice(free_blocks, size=n, replace=False).astype(np.int32)
    in_pairs = np.stack([targets, host_slots], 1)
    pa.swap_blocks(c.pool, host, torch.as_tensor(in_pairs, device=c.dev), pa.PA_SWAP_IN)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    c.orc.swap_blocks(c.pool_ref, c.geom, host_ref, in_pairs, 1)
    assert np.array_equal(bits(c.pool), c.pool_ref), "swap-in is not bit-exact"


def test_swapped_sequence_decodes_the_same(pa):
    """Decode of sequence 0 through its table, then after its blocks were
    swapped out, overwritten on the device and swapped back into other blocks."""
    w = wl.CONFIGS["llama70b_decode"]()
    c = Case(w)
    nb = int(-(-int(w.seq_lens[0]) // w.block_size))
    table0 = w.tables[0, :nb].copy()
    out_ref = c.orc.paged_decode(bits(c.cpu["q"][:1]), c.pool_ref, c.geom, w.tables[:1], w.seq_lens[:1],
                                 w.num_q_heads, w.scale)
    host = pinned_host(nb, c)
    pa.swap_blocks(c.pool, host, torch.as_tensor(np.stack([table0, np.arange(nb, dtype=np.int32)], 1),
                                                 device=c.dev), pa.PA_SWAP_OUT)
    c.pool[torch.as_tensor(table0.astype(np.int64), device=c.dev)] = 0   # the device blocks are reused
    referenced = np.unique(w.tables[w.tables >= 0])
    fresh = np.setdiff1d(np.arange(w.num_blocks), referenced)[:nb].astype(np.int32)
    pa.swap_blocks(c.pool, host, torch.as_tensor(np.stack([fresh, np.arange(nb, dtype=np.int32)], 1),
                                                 device=c.dev), pa.PA_SWAP_IN)
    tables = torch.full((1, w.tables.shape[1]), -1, dtype=torch.int32, device=c.dev)
    tables[0, :nb] = torch.as_tensor(fresh, device=c.dev)
    out = torch.empty_like(c.q[:1])
    nbytes = pa.decode_workspace_size(c.pool, 1, w.num_q_heads, int(w.seq_lens[0]), 0)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=c.dev)
    pa.decode(out, c.q[:1].contiguous(), c.pool, tables, c.seq_lens[:1].contiguous(), int(w.seq_lens[0]), w.scale,
              0, ws)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert_close(out, out_ref, "decode after swap out / in")


def test_swap_layered_pool(pa):
    """Swapping one layer of a layered pool touches only that layer."""
    gen = torch.Generator().manual_seed(11)
    NB, L, Hkv, b, d = 20, 3, 2, 16, 64
    pool = torch.randn((NB, 2, L, Hkv, b, d), generator=gen).to(torch.bfloat16).cuda()
    before = bits(pool).copy()
    host = torch.zeros((4, 2, Hkv, b, d), dtype=torch.bfloat16, pin_memory=True)
    pairs = np.asarray([[5, 2], [17, 0], [3, 3]], np.int32)
    pa.swap_blocks(pool, host, torch.as_tensor(pairs, device="cuda"), pa.PA_SWAP_OUT, layer=1)
    torch.cuda.synchronize()
    for blk, hb in pairs:
        assert np.array_equal(bits(host)[hb], before[blk, :, 1])
    pa.swap_blocks(pool, host, torch.as_tensor([[9, 2]], dtype=torch.int32, device="cuda"), pa.PA_SWAP_IN, layer=2)
    torch.cuda.synchronize()
    after = bits(pool)
    assert np.array_equal(after[9, :, 2], before[5, :, 1])
    mask = np.ones(after.shape, bool)
    mask[9, :, 2] = False
    assert np.array_equal(after[mask], before[mask])
    assert pa.get_device_error() == 0


def test_swap_errors(pa):
    w = wl.CONFIGS["tiny"]()
    c = Case(w)
    host = pinned_host(2, c)
    before = bits(c.pool).copy()
    bad = torch.as_tensor([[w.num_blocks, 0], [1, 5], [-1, 1], [2, 1]], dtype=torch.int32, device=c.dev)
    pa.swap_blocks(c.pool, host, bad, pa.PA_SWAP_IN)
    torch.cuda.synchronize()
    assert pa.get_device_error(clear=True) & pa.binding.DEVERR_BLOCK_ID
    after = bits(c.pool)
    assert np.array_equal(after[2], bits(host)[1]) and np.array_equal(np.delete(after, 2, 0), np.delete(before, 2, 0))
    # Pageable memory: refused before any launch unless this GPU addresses host
    # memory through the host's page tables, in which case the copy must be right.
    pageable = torch.zeros_like(host).contiguous()
    assert not pageable.is_pinned()
    try:
        pa.swap_blocks(c.pool, pageable, torch.as_tensor([[0, 0]], dtype=torch.int32, device=c.dev), pa.PA_SWAP_OUT)
        torch.cuda.synchronize()
        assert np.array_equal(bits(pageable)[0], bits(c.pool)[0])
    except pa.PagedAttentionError as e:
        assert e.status == 1
    with pytest.raises(pa.PagedAttentionError):
        pa.swap_blocks(c.pool, host, torch.as_tensor([[0, 0]], dtype=torch.int32, device=c.dev), 7)
    assert pa.get_device_error() == 0
