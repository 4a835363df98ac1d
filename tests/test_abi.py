"""The C-ABI library loads, exports every function include/pa.h declares, and
rejects bad arguments on the host without launching anything (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_167_gb300 import binding
    return binding


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(B):
    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(B.LIBRARY)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows a signature for each of them
    assert set(names) <= set(B.SIGNATURES), set(names) - set(B.SIGNATURES)


def test_status_strings(B):
    for s in range(8):
        assert B.lib().pa_status_string(s)
    assert B.lib().pa_status_string(99) == b"unknown status"


def _pool(B, base=0x10000, nb=64, hkv=8, b=16, d=128, bstride=0, kvstride=0, dtype=0):
    return B.PaKvPool(base, nb, hkv, b, d, dtype, bstride, kvstride)


def test_host_validation(B):
    L = B.lib()
    P = ctypes.c_void_p
    good = _pool(B)
    ok_ptr = P(0x20000)
    args = lambda pool, out=ok_ptr, q=ok_ptr, hq=64, part=0, ws=P(0), wsb=0: (
        out, q, ctypes.byref(pool), ok_ptr, 8, ok_ptr, 4, hq, 100, 0.1, part, ws, wsb, P(0))
    assert L.pa_decode(*args(good, out=P(0))) == 1                     # null out
    assert L.pa_decode(*args(_pool(B, base=0x10001))) == 1              # misaligned pool
    assert L.pa_decode(*args(_pool(B, d=96))) == 2                      # head_dim not built
    assert L.pa_decode(*args(_pool(B, dtype=7))) == 2                   # dtype
    assert L.pa_decode(*args(good, hq=60)) == 1                         # Hq % Hkv
    assert L.pa_decode(*args(good, hq=8 * 16)) == 2                     # group 16 not built
    assert L.pa_decode(*args(good, part=24)) == 1                       # partition % b
    assert L.pa_decode(*args(good, part=16)) == 3                       # workspace missing
    assert L.pa_decode(*args(_pool(B, kvstride=100))) == 1              # overlapping halves
    ex = lambda flags, nk=P(0), nv=P(0), **kw: args(good, **kw)[:-1] + (nk, nv, flags, P(0))
    assert L.pa_decode_ex(*ex(0, nk=ok_ptr)) == 1                       # new_k without new_v
    assert L.pa_decode_ex(*ex(0, nk=ok_ptr, nv=P(0x20008))) == 1        # misaligned new_v
    assert L.pa_decode_ex(*ex(0x2)) == 1                                 # unknown flag bit
    assert L.pa_decode_ex(*ex(B.PA_DECODE_EARLY_METADATA, out=P(0))) == 1  # same checks as pa_decode
    assert L.pa_decode_ex(*ex(B.PA_DECODE_EARLY_METADATA, part=16)) == 3
    assert L.pa_reshape_and_cache(ctypes.byref(good), P(0), P(0), P(0), 0, P(0)) == 0  # nothing to do
    assert L.pa_reshape_and_cache(ctypes.byref(good), P(0x20008), ok_ptr, ok_ptr, 4, P(0)) == 1
    assert L.pa_copy_blocks(ctypes.byref(good), P(0), -1, P(0)) == 1
    assert L.pa_copy_blocks(ctypes.byref(good), P(0), 0, P(0)) == 0
    assert L.pa_prefill_chunk(ok_ptr, ok_ptr, ctypes.byref(_pool(B, d=64)), ok_ptr, 8, ok_ptr, 1, 4, 64, 10,
                              0.1, P(0)) == 2
    for bad_scale in (0.0, -0.1, float("nan")):                          # scale must be finite and > 0
        assert L.pa_prefill_chunk(ok_ptr, ok_ptr, ctypes.byref(good), ok_ptr, 8, ok_ptr, 1, 4, 64, 10,
                                  bad_scale, P(0)) == 1
    # cascade entry points: prefix terms are required, aligned; the prefix pass validates like prefill
    cas = lambda po, pl, **kw: args(good, **kw)[:-1] + (po, pl, P(0), P(0), 0, P(0))
    assert L.pa_decode_cascade(*cas(P(0), ok_ptr)) == 1                 # no prefix output
    assert L.pa_decode_cascade(*cas(ok_ptr, P(0))) == 1                 # no prefix lse
    assert L.pa_decode_cascade(*cas(P(0x20008), ok_ptr)) == 1           # misaligned prefix output
    assert L.pa_decode_cascade(*cas(ok_ptr, ok_ptr, part=16)) == 3      # workspace missing, as pa_decode
    pfx = lambda o, lse, scale=0.1, groups=1, gsz=4, maxlen=64: (o, lse, ok_ptr, ctypes.byref(good), ok_ptr, 8,
                                                                 ok_ptr, P(0), groups, gsz, 64, maxlen, scale, P(0))
    assert L.pa_prefix_attention(*pfx(ok_ptr, ok_ptr, groups=0)) == 0   # nothing to do
    assert L.pa_prefix_attention(*pfx(P(0x20008), ok_ptr)) == 1          # misaligned output
    assert L.pa_prefix_attention(*pfx(ok_ptr, P(0))) == 1                # no lse
    assert L.pa_prefix_attention(*pfx(ok_ptr, ok_ptr, scale=0.0)) == 1
    assert L.pa_prefix_attention(*pfx(ok_ptr, ok_ptr, maxlen=8 * 16 + 1)) == 1   # longer than the table
    assert L.pa_prefix_attention(*pfx(ok_ptr, ok_ptr, groups=70000)) == 1        # grid limit
    assert L.pa_prefix_attention(ok_ptr, ok_ptr, ok_ptr, ctypes.byref(_pool(B, d=64)), ok_ptr, 8, ok_ptr, P(0), 1, 4,
                                 64, 10, 0.1, P(0)) == 2
    # one step from host buffers: staging size and layout, host-side validation
    hs = L.pa_decode_host_staging_size(ctypes.byref(good), 4, 64, 8)
    assert hs == 2 * (4 * 64 * 128 * 2) + 2 * (4 * 8 * 128 * 2) + 256 + 256   # q, out, new K, new V, tables, lengths
    assert L.pa_decode_host_staging_size(ctypes.byref(good), 4, 64, 0) == 0
    host = lambda st=P(0x40000), stb=hs, nk=P(0), nv=P(0), q=ok_ptr: (
        ok_ptr, q, ctypes.byref(good), ok_ptr, 8, ok_ptr, 4, 64, 100, 0.1, 0, nk, nv, 0, st, stb, P(0), 0, P(0))
    assert L.pa_decode_host(*host(st=P(0))) == 3                       # no staging
    assert L.pa_decode_host(*host(stb=hs - 1)) == 3                    # staging too small
    assert L.pa_decode_host(*host(st=P(0x40010))) == 3                 # staging not 256-byte aligned
    assert L.pa_decode_host(*host(q=P(0))) == 1                        # no q
    assert L.pa_decode_host(*host(nk=ok_ptr)) == 1                     # new K without new V
    assert L.pa_check_wait_timeout(999, P(0)) == 1                    # limit below 1 us
    assert L.pa_check_wait_timeout(10**9 + 1, P(0)) == 1              # above 1 s
    err = ctypes.c_uint32()
    assert L.pa_get_device_error(None, 0, P(0)) == 1


def test_workspace_size(B):
    L = B.lib()
    pool = _pool(B, nb=16384)
    # 64 sequences, 64 q-heads, two 512-token partitions over 851 tokens
    n = L.pa_decode_workspace_size(ctypes.byref(pool), 64, 64, 851, 512)
    assert n == 64 * 64 * 2 * 128 * 4 + 64 * 64 * 2 * 2 * 4
    assert L.pa_decode_workspace_size(ctypes.byref(pool), 64, 64, 512, 512) == 0
    assert L.pa_decode_partition_tokens(ctypes.byref(pool), 64, 64, 851, 512) == 512
    # partition_tokens = 0 selects the balanced (stream-K) schedule: two
    # partial records of G heads per CTA
    assert L.pa_decode_partition_tokens(ctypes.byref(pool), 64, 64, 851, 0) == 0
    ws = L.pa_decode_workspace_size(ctypes.byref(pool), 64, 64, 851, 0)
    rup = lambda x: -(-x // 256) * 256
    ctas = ws and next(c for c in range(1, 4097)
                       if rup(2 * c * 8 * 128 * 4) + rup(2 * c * 8 * 2 * 4) == ws)
    assert ctas and ctas % 2 == 0


def test_block_layout_matches_oracle(B):
    orc = oracle.load()
    for b in (1, 4, 16, 32):
        for t in range(0, 300):
            assert B.block_layout(t, b) == orc.block_layout(t, b)
    for bad in ((-1, 4), (4, 0)):
        with pytest.raises(B.PagedAttentionError):
            B.block_layout(*bad)


def test_slot_mapping_matches_oracle(B):
    import pa_workloads as wl
    orc = oracle.load()
    for w in (wl.tiny(), wl.tiny_page_example(), wl.llama70b_decode(), wl.beam_fork()):
        got = B.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size, w.num_blocks)
        ref = orc.slot_mapping(w.tables, w.new_seq_idx, w.new_positions, w.block_size)
        assert np.array_equal(got, ref), w.name
    # every position of every sequence of the long-context batch
    w = wl.long_context()
    seq = np.repeat(np.arange(w.batch, dtype=np.int32), w.seq_lens)
    pos = np.concatenate([np.arange(L) for L in w.seq_lens]).astype(np.int64)
    assert np.array_equal(B.slot_mapping(w.tables, seq, pos, 16, w.num_blocks),
                          orc.slot_mapping(w.tables, seq, pos, 16))
    with pytest.raises(B.PagedAttentionError):
        B.slot_mapping(w.tables, [0], [w.max_blocks * 16], 16, w.num_blocks)   # past the table
    with pytest.raises(B.PagedAttentionError):
        B.slot_mapping(np.asarray([[5, 1, 7]]), [0], [9], 4, 7)                # block 7 outside an NB=7 pool


def test_product_does_not_touch_the_oracle():
    """The product package never imports or loads the oracle, and the oracle
    never imports the product."""
    pkg = os.path.join(ROOT, "paged_kv_cache_167_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, re.M), f
                assert "pa_oracle" not in text and "orc_" not in text, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert not re.search(r"^\s*(import|from)\s+paged_kv_cache_167_gb300", text, re.M), f
            assert "libpa.so" not in text and "pa_decode" not in text, f


def test_stream_k_grid_override_sizes_the_workspace(B):
    """pa_set_stream_k_ctas fixes the balanced grid: the workspace is then
    two fp32 records of G x (d + 2) per CTA, the outputs and the (m, l)
    pairs each rounded up to 256 bytes, with the grid capped at the batch's
    16-token stages; 0 restores the default and a negative count is refused."""
    L = B.lib()
    pool = _pool(B, nb=64, hkv=8, b=16, d=128)
    r256 = lambda x: (x + 255) // 256 * 256
    try:
        for ctas in (1, 7, 152, 304, 1000):
            assert L.pa_set_stream_k_ctas(ctas) == 0
            nseq, hq, maxlen = 33, 64, 500
            eff = min(ctas, nseq * 8 * ((maxlen + 15) // 16))
            want = r256(2 * eff * 8 * 128 * 4) + r256(2 * eff * 8 * 2 * 4)
            assert L.pa_decode_workspace_size(ctypes.byref(pool), nseq, hq, maxlen, 0) == want
        assert L.pa_set_stream_k_ctas(1000) == 0   # capped: 2 sequences x 8 heads x 1 stage
        assert L.pa_decode_workspace_size(ctypes.byref(pool), 2, 64, 16, 0) == \
            r256(2 * 16 * 8 * 128 * 4) + r256(2 * 16 * 8 * 2 * 4)
        assert L.pa_set_stream_k_ctas(-1) == 1
    finally:
        assert L.pa_set_stream_k_ctas(0) == 0


def test_grouped_decode_validation(B):
    """pa_decode_grouped checks shapes on the host and launches nothing on a
    refusal: the members of an M-tile must fit one 128-key suffix tile."""
    L = B.lib()
    P = ctypes.c_void_p
    good = _pool(B, nb=64, hkv=8, b=16, d=128)
    ok_ptr = P(0x20000)

    def call(out=ok_ptr, pool=good, gsz=4, groups=2, hq=64, max_pre=64, max_sfx=32, scale=0.1, nk=P(0), nv=P(0),
             flags=0):
        return L.pa_decode_grouped(out, ok_ptr, ctypes.byref(pool), ok_ptr, 8, ok_ptr, P(0), ok_ptr, 4, ok_ptr,
                                   groups, gsz, hq, max_pre, max_sfx, scale, nk, nv, flags, P(0))

    assert call(groups=0) == 0                         # nothing to do
    assert call(groups=0, flags=1) == 0                # PA_DECODE_EARLY_METADATA is accepted
    assert call(flags=2) == 1                          # an unknown flag bit
    assert call(max_sfx=33) == 2                       # 4 members x 3 blocks > 128 keys
    assert call(gsz=16, max_sfx=16) == 2               # 16 members (of G = 8) x 1 block > 128 keys
    assert call(pool=_pool(B, d=64)) == 2              # head_dim 64 not built for the tensor-core path
    assert call(out=P(0)) == 1
    assert call(out=P(0x20008)) == 1                   # misaligned
    assert call(nk=ok_ptr) == 1                        # new K without new V
    assert call(scale=0.0) == 1
    assert call(max_pre=8 * 16 + 1) == 1               # longer than the prefix table
    assert call(gsz=1, max_sfx=5 * 16) == 1           # fits the tile, but longer than the 4-block suffix table
