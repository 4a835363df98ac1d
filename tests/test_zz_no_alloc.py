"""pa_decode_noalloc -- decode for callers that cannot allocate device memory
(a plugin given only its input and output buffers, or a serving loop that
must not call cudaMalloc) -- matches the oracle and is bit-identical to
pa_decode with a caller workspace, call after call.

Both entry points run the same kernels with the same plan, so their outputs
must agree bit for bit; the array the allocation-free call uses keeps the
previous call's contents, so each case runs it twice in a row.  Kept in a
file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import pa_workloads as wl
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_167_gb300 as pa
    assert torch.cuda.is_available(), "a CUDA device is required"
    pa.get_device_error(clear=True)
    return pa


def _workload(name):
    if name == "many_seqs":   # more than 128 sequences: the stage prefix lives in the scratch array too
        rng = np.random.default_rng(29)
        return wl.custom(list(rng.integers(1, 400, size=200)), 64, 8, 128, 16, seed=29)
    return wl.CONFIGS[name]()


@pytest.mark.parametrize("name,part", [("llama70b_decode", 0), ("many_seqs", 0), ("llama70b_decode", 320),
                                       ("long_context", 512), ("tiny", 16)])
def test_noalloc_matches_oracle_and_workspace_decode(pa, name, part):
    import oracle
    w = _workload(name)
    dev = torch.device("cuda")
    t = wl.make_tensors(w, "cpu")
    q, pool = t["q"].to(dev), t["pool"].to(dev)
    tables, lens = torch.as_tensor(w.tables, device=dev), torch.as_tensor(w.seq_lens, device=dev)
    nbytes = pa.decode_workspace_size(pool, w.batch, w.num_q_heads, w.max_seq_len, part)
    assert 0 < nbytes <= SCRATCH_BYTES
    with_ws = torch.empty_like(q)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    pa.decode(with_ws, q, pool, tables, lens, w.max_seq_len, w.scale, part, ws)
    geom = oracle.dense_geom(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    ref = oracle.load().paged_decode(wl.bf16_bits(t["q"]), wl.bf16_bits(t["pool"]), geom, w.tables, w.seq_lens,
                                     w.num_q_heads, w.scale)
    for call in range(2):                     # the array keeps the previous call's contents
        out = torch.full_like(q, float("nan"))
        pa.decode_noalloc(out, q, pool, tables, lens, w.max_seq_len, w.scale, part)
        torch.cuda.synchronize()
        assert_close(out, ref, f"{name} part={part} call {call}")
        assert torch.equal(out, with_ws), f"{name} part={part} call {call}: differs from pa_decode"
    assert pa.get_device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(pa):
    w = wl.shared_prefix(batch=64)
    dev = torch.device("cuda")
    t = wl.make_tensors(w, "cpu")
    q, pool = t["q"].to(dev), t["pool"].to(dev)
    tables, lens = torch.as_tensor(w.tables, device=dev), torch.as_tensor(w.seq_lens, device=dev)
    part = 16
    assert pa.decode_workspace_size(pool, w.batch, w.num_q_heads, w.max_seq_len, part) > SCRATCH_BYTES
    out = torch.zeros_like(q)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.decode_noalloc(out, q, pool, tables, lens, w.max_seq_len, w.scale, part)
    assert e.value.status == 3          # PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0   # nothing was launched
