"""GPU parity of the cascade decode (pa_cascade_plan, pa_prefix_attention,
pa_decode_cascade) against the oracle, through the C ABI.

The cascade attends a prefix shared by a group of sequences once for the
whole group and each sequence's own blocks apart, then merges the two by
log-sum-exp; the result must be attention over the whole sequence, so the
reference is the oracle's plain decode over the full tables.  The prefix pass
alone is checked against the oracle's decode over the prefix tables (output)
and its log-sum-exp.  Log-sum-exp tolerance: the kernel sums fp32
probabilities of fp32 scores (accumulated from bf16 operands in fp32), so its
error is a few fp32 ulps of the running sum; 1e-3 absolute leaves a wide
margin while a dropped key (log(n) against log(n - 1), at least 1/n) or a
wrong scale fails it at these sizes."""
import numpy as np
import pytest
import torch

import pa_workloads as wl
from tests.parity import Case, assert_close

pytestmark = pytest.mark.gpu

bits = wl.bf16_bits
LSE_ATOL = 1e-3


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_167_gb300 as pa
    assert torch.cuda.is_available(), "a CUDA device is required"
    pa.get_device_error(clear=True)
    return pa


def write_new_tokens(pa, c: Case):
    """Store each sequence's last token through the slot writer (GPU) and the
    oracle's writer (host copy), as a decode step does before attending."""
    w = c.w
    slots = pa.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size, w.num_blocks)
    pa.reshape_and_cache(c.pool, c.new_k, c.new_v, torch.as_tensor(slots, device=c.dev))
    c.orc.reshape_and_cache(c.pool_ref, c.geom, bits(c.cpu["new_k"]), bits(c.cpu["new_v"]),
                            c.orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size))


def prefix_pass(pa, c: Case, plan, group_size, order="plan"):
    w, dev = c.w, c.dev
    o_part = torch.empty(c.q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty((w.batch, w.num_q_heads), dtype=torch.float32, device=dev)
    if isinstance(order, str):
        order = plan.get("group_order")
    pa.prefix_attention(o_part, lse, c.q, c.pool, torch.as_tensor(plan["prefix_tables"], device=dev),
                        torch.as_tensor(plan["prefix_lens"], device=dev), group_size,
                        int(plan["prefix_lens"].max()), w.scale,
                        group_order=None if order is None else torch.as_tensor(order, device=dev))
    return o_part, lse


def cascade(pa, c: Case, plan, group_size, partition_tokens=0, flags=0, new_kv=None):
    w, dev = c.w, c.dev
    o_part, lse = prefix_pass(pa, c, plan, group_size)
    max_s = max(1, int(plan["suffix_lens"].max()))
    out = torch.empty_like(c.q)
    nbytes = pa.decode_workspace_size(c.pool, w.batch, w.num_q_heads, max_s, partition_tokens)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
    nk, nv = new_kv if new_kv is not None else (None, None)
    pa.decode_cascade(out, c.q, c.pool, torch.as_tensor(plan["suffix_tables"], device=dev),
                      torch.as_tensor(plan["suffix_lens"], device=dev), max_s, w.scale, o_part, lse,
                      partition_tokens, ws, flags=flags, new_k=nk, new_v=nv)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    return out, o_part, lse


def oracle_full(c: Case, rows=None):
    return c.orc.paged_decode(bits(c.cpu["q"]), c.pool_ref, c.geom, c.w.tables, c.w.seq_lens,
                              c.w.num_q_heads, c.w.scale, rows=rows)


def oracle_prefix(c: Case, plan, group_size):
    per_seq = np.repeat(plan["prefix_tables"], group_size, axis=0)
    lens = np.repeat(plan["prefix_lens"], group_size).astype(np.int32)
    return c.orc.paged_decode_lse(bits(c.cpu["q"]), c.pool_ref, c.geom, per_seq, lens, c.w.num_q_heads,
                                  c.w.scale)


def check_lse(got: torch.Tensor, ref: np.ndarray, what: str):
    g = got.cpu().numpy().astype(np.float64)
    empty = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), empty), f"{what}: -inf pattern differs"
    err = np.abs(g[~empty] - ref[~empty])
    assert err.size == 0 or err.max() <= LSE_ATOL, f"{what}: lse max err {err.max()}"


def designed_plan(w, group_size):
    """The split the workload was built with (its groups' prefix lengths),
    written out without the planner."""
    b = w.block_size
    plens = np.asarray(w.notes["prefix_lens"], np.int32)
    W = w.tables.shape[1]
    pt = np.full((len(plens), W), -1, np.int32)
    st = np.full((w.batch, W), -1, np.int32)
    for gi, plen in enumerate(plens):
        pt[gi, :plen // b] = w.tables[gi * group_size, :plen // b]
    for s in range(w.batch):
        row = w.tables[s, plens[s // group_size] // b:]
        st[s, :len(row)] = row
    return {"prefix_tables": pt, "prefix_lens": plens, "suffix_tables": st,
            "suffix_lens": np.asarray(w.seq_lens, np.int32) - np.repeat(plens, group_size)}


def grouped_case(group, group_size, prefix_lens, seed, bs=16):
    rng = np.random.default_rng(seed)
    suffix = rng.integers(1, 300, size=len(prefix_lens) * group_size).tolist()
    w = wl.shared_groups(prefix_lens, suffix, group_size, 2 * group, 2, 128, bs, seed=seed)
    return Case(w)


# ---------------------------------------------------------------------------

@pytest.mark.parametrize("group", [1, 4, 8])
@pytest.mark.parametrize("group_size", [1, 3, 16, 37])
def test_prefix_pass_matches_oracle(pa, group, group_size):
    """Output and log-sum-exp of every query over its group's prefix: several
    128-key tiles, a ragged last tile, an empty prefix, groups that fill a
    fraction of an M-tile or several M-tiles."""
    c = grouped_case(group, group_size, [0, 16, 400, 1024, 144], seed=group * 100 + group_size)
    plan = designed_plan(c.w, group_size)
    if group_size > 1:   # the planner finds the same split (alone, a sequence shares all its full blocks)
        got = pa.cascade_plan(c.w.tables, c.w.seq_lens, group_size, c.w.block_size)
        for k in plan:
            assert np.array_equal(got[k], plan[k]), k
    o_part, lse = prefix_pass(pa, c, plan, group_size)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    ref_o, ref_lse = oracle_prefix(c, plan, group_size)
    assert_close(o_part, ref_o, f"prefix o G={group} n={group_size}")
    check_lse(lse, ref_lse, f"prefix lse G={group} n={group_size}")


def test_group_order_changes_nothing(pa):
    """The order the groups' CTAs start in is scheduling only: natural order,
    longest first and a random permutation give bit-identical results; an
    entry out of range raises PA_DEVERR_ORDER and nothing faults."""
    c = grouped_case(8, 3, [1024, 16, 400, 0, 144, 2048], seed=21)
    plan = pa.cascade_plan(c.w.tables, c.w.seq_lens, 3, c.w.block_size)
    assert plan["group_order"].tolist() == [5, 0, 2, 4, 1, 3]
    runs = []
    for order in (None, plan["group_order"], np.random.default_rng(1).permutation(6).astype(np.int32)):
        o, l = prefix_pass(pa, c, plan, 3, order)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        runs.append((o.cpu(), l.cpu()))
    for o, l in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1])
    prefix_pass(pa, c, plan, 3, np.asarray([0, 1, 2, 3, 4, 6], np.int32))
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0x10


@pytest.mark.parametrize("group", [2, 8])
@pytest.mark.parametrize("group_size", [1, 4, 9])
@pytest.mark.parametrize("part", [0, 64, 512])
def test_cascade_matches_full_decode(pa, group, group_size, part):
    """Prefix pass + suffix decode with the fold equals attention over the
    whole sequence, on the balanced schedule (part 0) and on split-context
    partitions (single and several partitions)."""
    c = grouped_case(group, group_size, [0, 32, 496, 1536], seed=7 + group * 10 + group_size)
    plan = pa.cascade_plan(c.w.tables, c.w.seq_lens, group_size, c.w.block_size)
    out, _, _ = cascade(pa, c, plan, group_size, part)
    assert_close(out, oracle_full(c), f"cascade G={group} n={group_size} part={part}")


@pytest.mark.parametrize("part", [0, 32, 256])
def test_empty_suffix_is_prefix_alone(pa, part):
    """Sequences with no tokens after the prefix (suffix length 0) get the
    prefix term alone; a group with no prefix gets plain decode; a sequence
    with neither gets zeros."""
    w = wl.shared_groups([64, 0, 208], [0, 5, 0, 130, 0, 0], 2, 8, 2, 128, 16, seed=31)
    c = Case(w)
    plan = designed_plan(w, 2)
    assert list(plan["suffix_lens"]) == [0, 5, 0, 130, 0, 0]
    out, _, _ = cascade(pa, c, plan, 2, part)
    ref = oracle_full(c)
    assert_close(out, ref, f"empty suffix part={part}")
    assert not out[2].float().abs().sum().item() and not ref[2].any()   # no prefix, no suffix


@pytest.mark.parametrize("part", [0, 128])
@pytest.mark.parametrize("flags", [0, 1])
def test_cascade_with_append(pa, part, flags):
    """The suffix decode stores each sequence's new token (positions counted in
    the suffix) before attending, as pa_decode_ex does."""
    c = grouped_case(8, 4, [256, 64, 0], seed=55)
    w = c.w
    plan = pa.cascade_plan(w.tables, w.seq_lens, 4, w.block_size)
    out, _, _ = cascade(pa, c, plan, 4, part, flags=flags, new_kv=(c.new_k, c.new_v))
    c.orc.reshape_and_cache(c.pool_ref, c.geom, bits(c.cpu["new_k"]), bits(c.cpu["new_v"]),
                            c.orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size))
    assert np.array_equal(bits(c.pool), c.pool_ref), "the appended K/V differ from the slot writer's"
    assert_close(out, oracle_full(c), f"cascade append part={part} flags={flags}")


@pytest.mark.parametrize("name,group_size", [("shared_prefix", 256), ("beam_fork", 4)])
def test_full_size_cascade(pa, name, group_size):
    """The shared-prompt batch (one group of 256 over a 2,000-token prompt) and
    the beam batch (32 groups of 4 beams after copy-on-write), as the bench
    runs them, on sampled rows."""
    w = wl.CONFIGS[name]()
    c = Case(w)
    if w.copy_pairs is not None and len(w.copy_pairs):
        pa.copy_blocks(c.pool, torch.as_tensor(w.copy_pairs, device=c.dev))
        c.orc.copy_blocks(c.pool_ref, c.geom, w.copy_pairs)
    write_new_tokens(pa, c)
    plan = pa.cascade_plan(w.tables, w.seq_lens, group_size, w.block_size)
    if name == "shared_prefix":
        assert list(plan["prefix_lens"]) == [2000]
    else:
        plen = w.notes["prompt_lens"]
        assert np.array_equal(plan["prefix_lens"], (plen // 16) * 16)
    out, _, _ = cascade(pa, c, plan, group_size, 0, flags=1)
    rng = np.random.default_rng(9)
    flat = rng.choice(w.batch * w.num_q_heads, size=2048, replace=False)
    rows = np.stack([flat // w.num_q_heads, flat % w.num_q_heads], axis=1)
    assert_close(out[rows[:, 0], rows[:, 1]], oracle_full(c, rows), name)


def _beam_case(pa):
    w = wl.beam_fork()
    c = Case(w)
    pa.copy_blocks(c.pool, torch.as_tensor(w.copy_pairs, device=c.dev))
    c.orc.copy_blocks(c.pool_ref, c.geom, w.copy_pairs)
    write_new_tokens(pa, c)
    return w, c, pa.cascade_plan(w.tables, w.seq_lens, 4, w.block_size)


def test_beam_cascade_repeatable_under_contention(pa):
    """The full-size beam cascade sixteen times, every other time while a
    second stream copies gigabytes (HBM contention makes K/V tiles land late
    and in other orders): every run is bit-identical to the first, and the
    first matches the oracle on every row.  The prefix pass is HBM-bound on
    this batch; a completion wait that passes early there leaves the last key
    tiles of one (group, kv-head) tile out of its output."""
    w, c, plan = _beam_case(pa)
    ref = oracle_full(c)
    ref_o, ref_lse = oracle_prefix(c, plan, 4)
    side = torch.cuda.Stream()
    src = torch.empty(1 << 30, dtype=torch.uint8, device=c.dev)
    dst = torch.empty_like(src)
    first = None
    for rep in range(16):
        if rep % 2:
            with torch.cuda.stream(side):
                for _ in range(3):
                    dst.copy_(src)
        out, o_part, lse = cascade(pa, c, plan, 4, 0, flags=1)
        torch.cuda.synchronize()
        if first is None:
            assert_close(o_part, ref_o, "beam prefix pass")
            check_lse(lse, ref_lse, "beam prefix lse")
            assert_close(out, ref, "beam cascade")
            first = (out.clone(), o_part.clone(), lse.clone())
        else:
            assert torch.equal(o_part, first[1]) and torch.equal(lse, first[2]), f"prefix pass differs at run {rep}"
            assert torch.equal(out, first[0]), f"cascade output differs at run {rep}"


@pytest.mark.parametrize("ctas", [1, 7, 64, 151, 152, 300, 304, 1000])
def test_beam_cascade_grid_sweep(pa, ctas):
    """The beam batch's suffix decode (one-stage units) with the prefix folded
    in, at several balanced-schedule grid sizes, against the oracle."""
    w, c, plan = _beam_case(pa)
    try:
        pa.set_stream_k_ctas(ctas)
        out, _, _ = cascade(pa, c, plan, 4, 0, flags=1)
    finally:
        pa.set_stream_k_ctas(0)
    assert_close(out, oracle_full(c), f"beam cascade ctas={ctas}")


def grouped_call(pa, c: Case, plan, group_size, max_suffix=None, new_kv=None, order="plan", flags=0):
    w, dev = c.w, c.dev
    out = torch.full_like(c.q, float("nan"))
    if isinstance(order, str):
        order = plan.get("group_order")
    ms = int(plan["suffix_lens"].max()) if max_suffix is None else max_suffix
    nk, nv = new_kv if new_kv is not None else (None, None)
    pa.decode_grouped(out, c.q, c.pool, torch.as_tensor(plan["prefix_tables"], device=dev),
                      torch.as_tensor(plan["prefix_lens"], device=dev),
                      torch.as_tensor(plan["suffix_tables"], device=dev),
                      torch.as_tensor(plan["suffix_lens"], device=dev), group_size,
                      int(plan["prefix_lens"].max()), ms, w.scale,
                      group_order=None if order is None else torch.as_tensor(order, device=dev), new_k=nk, new_v=nv,
                      flags=flags)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    return out


@pytest.mark.parametrize("group,group_size,bs,max_sfx", [(8, 4, 16, 32), (8, 8, 16, 16), (4, 3, 16, 32),
                                                         (1, 2, 16, 64), (2, 1, 16, 128), (8, 24, 8, 8)])
@pytest.mark.parametrize("append", [False, True])
def test_grouped_decode_matches_oracle(pa, group, group_size, bs, max_sfx, append):
    """pa_decode_grouped (prefix tiles, then one tile of every member's suffix
    blocks under a per-row block-diagonal mask) equals the oracle's attention
    over the whole tables: group sizes filling a fraction of an M-tile, one
    and several M-tiles per group (24 members of 8 heads), empty suffixes and
    empty prefixes; with `append`, each member's new token is stored by the
    call first, the pool bit-exact with the oracle's slot writer."""
    rng = np.random.default_rng(group * 1000 + group_size * 10 + bs + max_sfx)
    prefix = [0, 16 * bs // 16 * 1, 400 // bs * bs, 1024]
    suffix = rng.integers(0, max_sfx + 1, size=len(prefix) * group_size)
    suffix[0] = 0                # a member with neither prefix nor suffix (group 0 has no prefix)
    suffix[-1] = max_sfx         # a full suffix
    w = wl.shared_groups(prefix, list(suffix), group_size, 2 * group, 2, 128, bs, seed=int(rng.integers(1 << 30)))
    c = Case(w)
    plan = designed_plan(w, group_size)
    new_kv = None
    if append:   # each member with a suffix stores its last token; the oracle's writer does the same
        sel = np.asarray(plan["suffix_lens"])[w.new_seq_idx] > 0
        slots = c.orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size)
        c.orc.reshape_and_cache(c.pool_ref, c.geom, bits(c.cpu["new_k"]), bits(c.cpu["new_v"]),
                                np.where(sel, slots, -1))
        full_k = torch.zeros((w.batch, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16)
        full_v = torch.zeros_like(full_k)
        full_k[w.new_seq_idx] = c.cpu["new_k"]
        full_v[w.new_seq_idx] = c.cpu["new_v"]
        new_kv = (full_k.to(c.dev), full_v.to(c.dev))
    out = grouped_call(pa, c, plan, group_size, max_suffix=max_sfx, new_kv=new_kv)
    if append:
        assert np.array_equal(bits(c.pool), c.pool_ref), "the stored new tokens differ from the slot writer's"
    ref = oracle_full(c)
    assert_close(out, ref, f"grouped G={group} n={group_size} b={bs} append={append}")
    assert w.seq_lens[0] == 0 and not out[0].float().abs().sum().item()   # no keys at all: zeros


def test_grouped_full_size_beams_repeatable(pa):
    """The beam batch (32 groups of 4 after copy-on-write) through one
    pa_decode_grouped call that also stores every beam's new token: every
    row against the oracle, then eight more calls (every other one under a
    concurrent copy on a second stream, half of them reading the tables
    before the previous kernel has finished) bit-identical to the first."""
    w = wl.beam_fork()
    c = Case(w)
    pa.copy_blocks(c.pool, torch.as_tensor(w.copy_pairs, device=c.dev))
    c.orc.copy_blocks(c.pool_ref, c.geom, w.copy_pairs)
    plan = pa.cascade_plan(w.tables, w.seq_lens, 4, w.block_size)
    assert int(plan["suffix_lens"].max()) <= 16
    first = grouped_call(pa, c, plan, 4, new_kv=(c.new_k, c.new_v))
    c.orc.reshape_and_cache(c.pool_ref, c.geom, bits(c.cpu["new_k"]), bits(c.cpu["new_v"]),
                            c.orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size))
    assert np.array_equal(bits(c.pool), c.pool_ref), "the stored new tokens differ from the slot writer's"
    assert_close(first, oracle_full(c), "grouped beams")
    side = torch.cuda.Stream()
    src = torch.empty(1 << 30, dtype=torch.uint8, device=c.dev)
    dst = torch.empty_like(src)
    for rep in range(8):
        if rep % 2:
            with torch.cuda.stream(side):
                for _ in range(3):
                    dst.copy_(src)
        again = grouped_call(pa, c, plan, 4, new_kv=(c.new_k, c.new_v),
                             flags=pa.PA_DECODE_EARLY_METADATA if rep % 4 >= 2 else 0)
        assert torch.equal(again, first), f"grouped output differs at run {rep}"


def test_grouped_persistent_grid_sweep(pa):
    """Grouped decode (7 groups of 4 beams, 2 kv-heads: 14 units) with every
    grid size from one CTA (all units in one CTA, the pipeline handed from
    unit to unit, each unit's suffix tile zeroed and released in turn) to more
    CTAs than units: outputs bit for bit alike, the default grid's against
    the oracle.  The groups without a prefix make runs of one-tile units, in
    which the V warp can release two units' suffix tiles before the P.V lane
    waits for the first (with a single barrier for them, that wait saw the
    later phase and the CTA stalled)."""
    rng = np.random.default_rng(41)
    prefix = [0, 160, 0, 400, 1024, 48, 704]
    suffix = rng.integers(0, 33, size=len(prefix) * 4)
    w = wl.shared_groups(prefix, list(suffix), 4, 16, 2, 128, 16, seed=41)
    c = Case(w)
    plan = designed_plan(w, 4)
    base = grouped_call(pa, c, plan, 4)
    assert_close(base, oracle_full(c), "grouped sweep")
    try:
        for ctas in (1, 2, 3, 5, 13, 14, 15):
            pa.set_prefill_ctas(ctas)
            for flags in (0, pa.PA_DECODE_EARLY_METADATA):   # the tables read before or after the wait
                out = grouped_call(pa, c, plan, 4, flags=flags)
                assert torch.equal(out, base), f"{ctas} CTAs, flags {flags}: output differs from the default grid's"
    finally:
        pa.set_prefill_ctas(0)


def test_grouped_refuses_long_suffixes(pa):
    """Suffixes that do not fit one 128-key tile for the M-tile's members are
    refused on the host (the two-call cascade serves them)."""
    c = grouped_case(8, 4, [256, 64], seed=5)
    plan = pa.cascade_plan(c.w.tables, c.w.seq_lens, 4, c.w.block_size)
    with pytest.raises(pa.PagedAttentionError) as e:
        grouped_call(pa, c, plan, 4)
    assert e.value.status == 2
