"""GPU parity of the decode path (slot writer, paged decode, split-context
reduce, copy-on-write copies) against the oracle, through the C ABI."""
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


def write_new_tokens(pa, c: Case):
    w = c.w
    if w.new_positions is None or len(w.new_positions) == 0:
        return
    slots = pa.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size, w.num_blocks)
    oslots = c.orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size)
    assert np.array_equal(slots, oslots), "host slot mapping differs from the oracle"
    pa.reshape_and_cache(c.pool, c.new_k, c.new_v, torch.as_tensor(slots, device=c.dev))
    c.orc.reshape_and_cache(c.pool_ref, c.geom, bits(c.cpu["new_k"]), bits(c.cpu["new_v"]), oslots)


def run_decode(pa, c: Case, partition_tokens=None, flags=0):
    w = c.w
    part = w.partition_tokens if partition_tokens is None else partition_tokens
    out = torch.empty_like(c.q)
    nbytes = pa.decode_workspace_size(c.pool, w.batch, w.num_q_heads, w.max_seq_len, part)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=c.dev) if nbytes else None
    pa.decode(out, c.q, c.pool, c.tables, c.seq_lens, w.max_seq_len, w.scale, part, ws, flags=flags)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    return out


def oracle_decode(c: Case, rows=None):
    return c.orc.paged_decode(bits(c.cpu["q"]), c.pool_ref, c.geom, c.w.tables, c.w.seq_lens,
                              c.w.num_q_heads, c.w.scale, rows=rows)


# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "tiny_page_example"])
@pytest.mark.parametrize("part_blocks", [0, 1, 2])
def test_tiny_configs(pa, name, part_blocks):
    w = wl.CONFIGS[name]()
    c = Case(w)
    write_new_tokens(pa, c)
    assert np.array_equal(bits(c.pool), c.pool_ref), "slot writer is not bit-exact"
    out = run_decode(pa, c, part_blocks * w.block_size)
    assert_close(out, oracle_decode(c), f"{name} part={part_blocks}")


def test_page_example_slot(pa):
    """Token 9 of the page example lands in physical block 7, offset 1."""
    w = wl.tiny_page_example()
    c = Case(w)
    write_new_tokens(pa, c)
    pool = bits(c.pool)
    assert np.array_equal(pool[7, 0, :, 1], bits(c.cpu["new_k"])[9])
    assert np.array_equal(pool[7, 1, :, 1], bits(c.cpu["new_v"])[9])


SWEEP_LENS = [1, 3, 16, 17, 63, 64, 65, 200, 331]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("bs", [4, 8, 16, 32, 64])
def test_shape_sweep(pa, d, group, bs):
    hkv = 2
    w = wl.custom(SWEEP_LENS, hkv * group, hkv, d, bs, seed=1000 + d + group * 10 + bs)
    c = Case(w)
    write_new_tokens(pa, c)
    assert np.array_equal(bits(c.pool), c.pool_ref)
    ref = oracle_decode(c)
    for part in (0, bs, 4 * bs, 64 if 64 % bs == 0 else bs):
        assert_close(run_decode(pa, c, part), ref, f"d={d} G={group} b={bs} part={part}")
    assert_close(run_decode(pa, c, 0, pa.PA_DECODE_EARLY_METADATA), ref, f"d={d} G={group} b={bs} early")


@pytest.mark.parametrize("name,sample", [("llama70b_decode", None), ("long_context", None),
                                         ("shared_prefix", 2048), ("beam_fork", 2048)])
def test_full_size(pa, name, sample):
    """The full-size workloads, in the launch configuration the bench times."""
    w = wl.CONFIGS[name]()
    c = Case(w)
    if w.copy_pairs is not None and len(w.copy_pairs):
        pa.copy_blocks(c.pool, torch.as_tensor(w.copy_pairs, device=c.dev))
        c.orc.copy_blocks(c.pool_ref, c.geom, w.copy_pairs)
    write_new_tokens(pa, c)
    assert np.array_equal(bits(c.pool), c.pool_ref), "pool after copies and writes is not bit-exact"
    out = run_decode(pa, c)
    if sample is None:
        assert_close(out, oracle_decode(c), name)
    else:
        rng = np.random.default_rng(5)
        flat = rng.choice(w.batch * w.num_q_heads, size=sample, replace=False)
        rows = np.stack([flat // w.num_q_heads, flat % w.num_q_heads], axis=1)
        ref = oracle_decode(c, rows)
        assert_close(out[rows[:, 0], rows[:, 1]], ref, name)


@pytest.mark.parametrize("batch,hkv", [(100, 128), (300, 64)])
def test_many_short_units_per_cta(pa, batch, hkv):
    """Thousands of one-stage units, more per CTA of the balanced schedule
    than one listing holds: exercises the repeated listings of a CTA's range
    (one pass per thread's sequence for up to 128 sequences, the sequential
    listing beyond)."""
    rng = np.random.default_rng(batch + hkv)
    lens = rng.integers(1, 17, size=batch)
    w = wl.custom(list(lens), hkv, hkv, 64, 16, seed=77 + batch)
    c = Case(w)
    write_new_tokens(pa, c)
    ref = oracle_decode(c)
    assert_close(run_decode(pa, c, 0), ref, f"B={batch} Hkv={hkv}")
    assert_close(run_decode(pa, c, 0, pa.PA_DECODE_EARLY_METADATA), ref, f"B={batch} Hkv={hkv} early")


# Balanced-schedule grid sizes: tiny grids (one CTA holds everything), sizes
# around one and two CTAs per SM of 148- and 152-SM parts, and grids larger
# than the number of resident CTAs.
GRID_SWEEP = [1, 2, 3, 5, 7, 13, 31, 64, 100, 147, 148, 151, 152, 153, 255, 296, 303, 304, 305, 607, 1000]


def _grid_workload(name):
    rng = np.random.default_rng(404)
    if name == "ragged":        # units of 1 .. 44 stages, many cut by range boundaries
        lens = list(rng.integers(1, 700, size=40))
        return wl.custom(lens, 64, 8, 128, 16, seed=405)
    if name == "one_stage":     # 128 sequences of one stage each (the beams' suffixes)
        return wl.custom(list(rng.integers(1, 17, size=128)), 64, 8, 128, 16, seed=406)
    # more sequences than one listing pass holds (stage prefix in the workspace), b = 4
    lens = list(rng.integers(0, 150, size=200))
    return wl.custom(lens, 4, 2, 64, 4, seed=407)


@pytest.mark.parametrize("name", ["ragged", "one_stage", "many_seqs_b4"])
def test_stream_k_grid_sweep(pa, name):
    """The balanced schedule at many grid sizes against the oracle.  The grid
    size moves every CTA range boundary, and with it which units are cut,
    which partial record each CTA writes and which records the merge kernel
    combines; the default grid follows the device's SM count, so these sizes
    cover what other SM counts would run."""
    w = _grid_workload(name)
    c = Case(w)
    write_new_tokens(pa, c)
    ref = oracle_decode(c)
    try:
        for ctas in GRID_SWEEP:
            pa.set_stream_k_ctas(ctas)
            assert_close(run_decode(pa, c, 0), ref, f"{name} ctas={ctas}")
            assert_close(run_decode(pa, c, 0, pa.PA_DECODE_EARLY_METADATA), ref, f"{name} ctas={ctas} early")
    finally:
        pa.set_stream_k_ctas(0)


def test_partitions_agree(pa):
    """P = 1 and many partitions both match the oracle on the same inputs."""
    w = wl.llama70b_decode(batch=16)
    c = Case(w)
    write_new_tokens(pa, c)
    ref = oracle_decode(c)
    outs = [run_decode(pa, c, part) for part in (16, 64, 256, 1024)]
    for part, o in zip((16, 64, 256, 1024), outs):
        assert_close(o, ref, f"part={part}")


def _move_blocks(c: Case, rng):
    """Same logical content under a new random placement (test-side)."""
    w = c.w
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    tables2 = np.where(w.tables >= 0, perm[np.maximum(w.tables, 0)], -1).astype(np.int32)
    pool2 = torch.zeros_like(c.pool)
    valid = w.tables >= 0
    src = torch.as_tensor(w.tables[valid].astype(np.int64), device=c.dev)
    dst = torch.as_tensor(tables2[valid].astype(np.int64), device=c.dev)
    pool2[dst] = c.pool[src]
    return tables2, pool2


def test_placement_invariance(pa):
    """Permuting physical placement leaves the output bit-identical."""
    w = wl.custom([5, 40, 333, 700, 1], 64, 8, 128, 16, num_blocks=512)
    c = Case(w)
    out1 = run_decode(pa, c, 64)
    tables2, pool2 = _move_blocks(c, np.random.default_rng(3))
    c.pool, c.tables = pool2, torch.as_tensor(tables2, device=c.dev)
    out2 = run_decode(pa, c, 64)
    assert torch.equal(out1, out2)


def test_shared_prefix_equals_private_copies(pa):
    w = wl.shared_prefix(batch=8)
    c = Case(w)
    out_shared = run_decode(pa, c)
    # give every sequence private copies of the shared prefix blocks
    shared = w.notes["shared_ids"]
    used = set(np.unique(w.tables[w.tables >= 0]).tolist())
    free = [i for i in range(w.num_blocks) if i not in used]
    tables = w.tables.copy()
    pool = c.pool.clone()
    k = 0
    for s in range(1, w.batch):
        fresh = np.asarray(free[k:k + len(shared)], np.int32)
        k += len(shared)
        pool[torch.as_tensor(fresh, device=c.dev).long()] = c.pool[torch.as_tensor(shared, device=c.dev).long()]
        tables[s, :len(shared)] = fresh
    c.pool, c.tables = pool, torch.as_tensor(tables, device=c.dev)
    out_private = run_decode(pa, c)
    assert torch.equal(out_shared, out_private)


def test_empty_sequences_and_junk_tails(pa):
    """seq_len 0 gives zeros; NaN junk in unused tail slots is never used."""
    w = wl.custom([0, 5, 0, 17, 33, 1], 8, 2, 128, 16, num_blocks=64)
    c = Case(w)
    nan = torch.full((w.head_dim,), float("nan"), dtype=torch.bfloat16, device=c.dev)
    for s, L in enumerate(w.seq_lens):
        if L % w.block_size:
            blk = int(w.tables[s, (L - 1) // w.block_size])
            c.pool[blk, :, :, L % w.block_size:, :] = nan
    for part in (0, 16):
        out = run_decode(pa, c, part)
        assert not torch.isnan(out).any()
        assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
        ref = oracle_decode(c)
        assert_close(out, ref, f"part={part}")


def test_layered_pool(pa):
    """The pages' layered pool shape [NB][2][L][Hkv][b][d], read one layer at a time."""
    w = wl.custom([20, 77, 130], 16, 4, 64, 16, num_blocks=40)
    layers = 3
    gen = torch.Generator(device="cpu").manual_seed(4)
    pool6 = wl.randn_bf16((w.num_blocks, 2, layers, w.num_kv_heads, w.block_size, w.head_dim), gen)
    q = wl.randn_bf16((w.batch, w.num_q_heads, w.head_dim), gen)
    dev = torch.device("cuda")
    pool6_d, q_d = pool6.to(dev), q.to(dev)
    tables, lens = torch.as_tensor(w.tables, device=dev), torch.as_tensor(w.seq_lens, device=dev)
    import oracle
    orc = oracle.load()
    geom = oracle.dense_geom(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, num_layers=layers)
    flat = bits(pool6).reshape(-1)
    slab = w.num_kv_heads * w.block_size * w.head_dim
    for layer in range(layers):
        out = torch.empty_like(q_d)
        nbytes = pa.decode_workspace_size(pool6_d, w.batch, w.num_q_heads, w.max_seq_len, 32, layer=layer)
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
        pa.decode(out, q_d, pool6_d, tables, lens, w.max_seq_len, w.scale, 32, ws, layer=layer)
        ref = orc.paged_decode(bits(q), flat[layer * slab:], geom, w.tables, w.seq_lens, w.num_q_heads, w.scale)
        assert_close(out, ref, f"layer {layer}")
    # copy-on-write copies through a layer view touch only that layer
    pairs = np.asarray([[int(w.tables[0, 0]), 39]], np.int32)
    before = bits(pool6_d).copy()
    pa.copy_blocks(pool6_d, torch.as_tensor(pairs, device=dev), layer=1)
    ref = before.reshape(-1).copy()
    orc.copy_blocks(ref[slab:], geom, pairs)
    assert np.array_equal(bits(pool6_d).reshape(-1), ref)


def test_copy_blocks_bit_exact(pa):
    w = wl.custom([100, 60], 8, 8, 128, 16, num_blocks=64)
    c = Case(w)
    pairs = np.asarray([[int(w.tables[0, 0]), 50], [int(w.tables[1, 3]), 51], [int(w.tables[0, 6]), 63]], np.int32)
    pa.copy_blocks(c.pool, torch.as_tensor(pairs, device=c.dev))
    c.orc.copy_blocks(c.pool_ref, c.geom, pairs)
    torch.cuda.synchronize()
    assert np.array_equal(bits(c.pool), c.pool_ref)
    assert pa.get_device_error() == 0


def test_device_errors_are_reported_not_faulted(pa):
    """Out-of-range table entries, slots, pairs and lengths set error bits and
    are never dereferenced; the context stays usable."""
    from paged_kv_cache_167_gb300 import binding as B
    w = wl.custom([40, 9], 8, 2, 64, 16, num_blocks=16)
    c = Case(w)
    pa.get_device_error(clear=True)
    bad_tables = c.tables.clone()
    bad_tables[0, 1] = w.num_blocks + 5
    c_tables = c.tables
    c.tables = bad_tables
    out = torch.empty_like(c.q)
    nbytes = pa.decode_workspace_size(c.pool, w.batch, w.num_q_heads, w.max_seq_len, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=c.dev)
    pa.decode(out, c.q, c.pool, c.tables, c.seq_lens, w.max_seq_len, w.scale, 0, ws)
    assert pa.get_device_error() & B.DEVERR_BLOCK_ID
    c.tables = c_tables
    slots = torch.as_tensor([w.num_blocks * w.block_size + 3, -1], device=c.dev, dtype=torch.int64)
    before = c.pool.clone()
    pa.reshape_and_cache(c.pool, c.new_k[:2], c.new_v[:2], slots)
    assert pa.get_device_error() & B.DEVERR_SLOT
    assert torch.equal(before, c.pool)
    pa.copy_blocks(c.pool, torch.as_tensor([[0, w.num_blocks]], device=c.dev, dtype=torch.int32))
    assert pa.get_device_error() & B.DEVERR_BLOCK_ID
    assert torch.equal(before, c.pool)
    long_lens = torch.as_tensor([w.max_blocks * w.block_size + 1, 9], device=c.dev, dtype=torch.int32)
    pa.decode(out, c.q, c.pool, c.tables, long_lens, w.max_seq_len, w.scale, 0, ws)
    assert pa.get_device_error() & B.DEVERR_SEQ_LEN
    # still healthy afterwards
    assert_close(run_decode(pa, c, 0), oracle_decode(c), "after errors")


def test_early_metadata_back_to_back(pa):
    """PA_DECODE_EARLY_METADATA in the bench's launch pattern: each call follows
    the slot writer that wrote its layer's new tokens (a kernel that writes the
    pool, not the lengths or the table), calls alternate between two layers'
    pools and queries, and nothing synchronises between them; every output
    equals the oracle's."""
    w = wl.CONFIGS["llama70b_decode"]()
    tensors = wl.make_tensors(w, "cpu")
    c = Case(w, tensors=tensors)
    gen = torch.Generator().manual_seed(99)
    q2 = torch.randn(c.q.shape, generator=gen).to(torch.bfloat16)
    pool2 = c.pool.clone()
    pool2_ref = c.pool_ref.copy()
    slots = pa.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size, w.num_blocks)
    slots_dev = torch.as_tensor(slots, device=c.dev)
    for pool, ref_pool in ((c.pool, c.pool_ref), (pool2, pool2_ref)):
        c.orc.reshape_and_cache(ref_pool, c.geom, bits(tensors["new_k"]), bits(tensors["new_v"]), slots)
    qs = [c.q, q2.to(c.dev)]
    pools = [c.pool, pool2]
    nbytes = pa.decode_workspace_size(c.pool, w.batch, w.num_q_heads, w.max_seq_len, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=c.dev)
    outs = [torch.empty_like(c.q) for _ in range(6)]
    for i in range(6):
        pa.reshape_and_cache(pools[i % 2], c.new_k, c.new_v, slots_dev)
        pa.decode(outs[i], qs[i % 2], pools[i % 2], c.tables, c.seq_lens, w.max_seq_len, w.scale, 0, ws,
                  flags=pa.PA_DECODE_EARLY_METADATA)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    refs = [c.orc.paged_decode(bits(tensors["q"]), c.pool_ref, c.geom, w.tables, w.seq_lens, w.num_q_heads, w.scale),
            c.orc.paged_decode(bits(q2), pool2_ref, c.geom, w.tables, w.seq_lens, w.num_q_heads, w.scale)]
    for i in range(6):
        assert_close(outs[i], refs[i % 2], f"call {i}")


def append_inputs(c: Case):
    """[B][Hkv][d] new K/V per sequence (rows of empty sequences are zero and
    ignored) and the oracle's pool after the same stores."""
    w = c.w
    nk = torch.zeros((w.batch, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16)
    nv = torch.zeros_like(nk)
    nk[torch.as_tensor(w.new_seq_idx.astype(np.int64))] = c.cpu["new_k"]
    nv[torch.as_tensor(w.new_seq_idx.astype(np.int64))] = c.cpu["new_v"]
    oslots = c.orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size)
    c.orc.reshape_and_cache(c.pool_ref, c.geom, bits(c.cpu["new_k"]), bits(c.cpu["new_v"]), oslots)
    return nk.to(c.dev), nv.to(c.dev)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bs", [4, 8, 16, 32, 64])
def test_decode_with_append(pa, d, bs):
    """pa_decode_ex with new_k / new_v: each sequence's last token is stored at
    its slot (bit-exact with the oracle's slot writer) and attended, with the
    automatic plan (stored inside the decode kernel) and with partitions (a
    separate store kernel first)."""
    for part in (0, 4 * bs):
        w = wl.custom(SWEEP_LENS + [0], 8, 2, d, bs, seed=2000 + d + bs)
        c = Case(w)
        nk, nv = append_inputs(c)
        out = run_decode_ex(pa, c, part, nk, nv, pa.PA_DECODE_EARLY_METADATA)
        assert np.array_equal(bits(c.pool), c.pool_ref), f"b={bs} part={part}: pool after the append"
        assert_close(out, oracle_decode(c), f"d={d} b={bs} part={part} append")


def run_decode_ex(pa, c: Case, part, nk, nv, flags):
    w = c.w
    out = torch.empty_like(c.q)
    nbytes = pa.decode_workspace_size(c.pool, w.batch, w.num_q_heads, w.max_seq_len, part)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=c.dev) if nbytes else None
    pa.decode(out, c.q, c.pool, c.tables, c.seq_lens, w.max_seq_len, w.scale, part, ws, flags=flags,
              new_k=nk, new_v=nv)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    return out


@pytest.mark.parametrize("name,sample", [("llama70b_decode", None), ("shared_prefix", 2048), ("beam_fork", 2048)])
def test_append_full_size(pa, name, sample):
    """The full-size workloads through the fused append + decode call, as the
    bench times it."""
    w = wl.CONFIGS[name]()
    c = Case(w)
    if w.copy_pairs is not None and len(w.copy_pairs):
        pa.copy_blocks(c.pool, torch.as_tensor(w.copy_pairs, device=c.dev))
        c.orc.copy_blocks(c.pool_ref, c.geom, w.copy_pairs)
    nk, nv = append_inputs(c)
    out = run_decode_ex(pa, c, 0, nk, nv, pa.PA_DECODE_EARLY_METADATA)
    assert np.array_equal(bits(c.pool), c.pool_ref), "pool after the append"
    if sample is None:
        assert_close(out, oracle_decode(c), name)
    else:
        rng = np.random.default_rng(6)
        flat = rng.choice(w.batch * w.num_q_heads, size=sample, replace=False)
        rows = np.stack([flat // w.num_q_heads, flat % w.num_q_heads], axis=1)
        assert_close(out[rows[:, 0], rows[:, 1]], oracle_decode(c, rows), name)


def test_append_errors_write_nothing(pa):
    """An out-of-range length or table entry stores nothing for that sequence
    (and raises its error bit); the other sequences are appended."""
    from paged_kv_cache_167_gb300 import binding as B
    w = wl.custom([40, 9, 17], 8, 2, 64, 16, num_blocks=16, seed=31)
    c = Case(w)
    nk, nv = append_inputs(c)
    before = bits(c.pool).copy()
    tables = c.tables.clone()
    tables[1, 0] = w.num_blocks + 3            # sequence 1's last block is out of range
    lens = c.seq_lens.clone()
    lens[2] = w.max_blocks * w.block_size + 5  # sequence 2's length is out of range
    out = torch.empty_like(c.q)
    nbytes = pa.decode_workspace_size(c.pool, w.batch, w.num_q_heads, w.max_seq_len, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=c.dev)
    pa.get_device_error(clear=True)
    pa.decode(out, c.q, c.pool, tables, lens, w.max_seq_len, w.scale, 0, ws, new_k=nk, new_v=nv)
    torch.cuda.synchronize()
    e = pa.get_device_error()
    assert e & B.DEVERR_BLOCK_ID and e & B.DEVERR_SEQ_LEN
    after = bits(c.pool)
    # only sequence 0's last slot changed
    slot0 = c.orc.slot_mapping(w.tables, np.asarray([0], np.int32), np.asarray([39]), w.block_size)[0]
    blk, off = divmod(int(slot0), w.block_size)
    mask = np.ones(after.shape, bool)
    mask[blk, :, :, off] = False
    assert np.array_equal(after[mask], before[mask])
    assert np.array_equal(after[blk, 0, :, off], bits(c.cpu["new_k"])[0])


@pytest.mark.parametrize("part", [0, 64])
def test_decode_from_host_buffers(pa, part):
    """pa_decode_host: q, tables, lengths and the new tokens from pinned host
    memory, the output back to host memory, one call; the pool bit-exact with
    the oracle's slot writer and the output within tolerance."""
    w = wl.custom([1, 17, 300, 64, 129, 850], 16, 2, 128, 16, seed=77)
    c = Case(w)
    q_h, k_h, v_h = (c.cpu[k].pin_memory() for k in ("q", "new_k", "new_v"))
    tables_h = torch.as_tensor(w.tables).pin_memory()
    lens_h = torch.as_tensor(w.seq_lens).pin_memory()
    out_h = torch.full_like(q_h, float("nan")).pin_memory()
    nb = pa.decode_host_staging_size(c.pool, w.batch, w.num_q_heads, w.tables.shape[1])
    staging = torch.empty(nb, dtype=torch.uint8, device=c.dev)
    wsb = pa.decode_workspace_size(c.pool, w.batch, w.num_q_heads, w.max_seq_len, part)
    ws = torch.empty(wsb, dtype=torch.uint8, device=c.dev) if wsb else None
    pa.decode_host(out_h, q_h, c.pool, tables_h, lens_h, w.max_seq_len, w.scale, staging, part, ws,
                   flags=pa.PA_DECODE_EARLY_METADATA, new_k_host=k_h, new_v_host=v_h)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    c.orc.reshape_and_cache(c.pool_ref, c.geom, bits(c.cpu["new_k"]), bits(c.cpu["new_v"]),
                            c.orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size))
    assert np.array_equal(bits(c.pool), c.pool_ref), "stored K/V differ from the slot writer's"
    assert_close(out_h, oracle_decode(c), f"host buffers part={part}")
