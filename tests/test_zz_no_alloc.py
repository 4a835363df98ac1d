"""pa_decode_noalloc -- decode for callers that cannot allocate device memory
(a plugin given only its input and output buffers, or a serving loop that
must not call cudaMalloc) -- matches pa_decode, call after call.

Kept in a file of its own that pytest collects last."""
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
    return pa


def _inputs(w, dev):
    t = wl.make_tensors(w, "cpu")
    return (t["q"].to(dev), t["pool"].to(dev), torch.as_tensor(w.tables, device=dev),
            torch.as_tensor(w.seq_lens, device=dev))


@pytest.mark.parametrize("name,part", [("llama70b_decode", 320), ("long_context", 512), ("tiny", 16)])
def test_noalloc_matches_workspace_decode(pa, name, part):
    w = wl.CONFIGS[name]()
    dev = torch.device("cuda")
    q, pool, tables, lens = _inputs(w, dev)
    nbytes = pa.decode_workspace_size(pool, w.batch, w.num_q_heads, w.max_seq_len, part)
    assert 0 < nbytes <= SCRATCH_BYTES
    ref = torch.empty_like(q)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    pa.decode(ref, q, pool, tables, lens, w.max_seq_len, w.scale, part, ws)
    ref_np = ref.float().cpu().numpy().astype(np.float64)
    for call in range(2):                     # the array keeps the previous call's contents
        out = torch.full_like(q, float("nan"))
        pa.decode_noalloc(out, q, pool, tables, lens, w.max_seq_len, w.scale, part)
        torch.cuda.synchronize()
        assert_close(out, ref_np, f"{name} call {call}")
    assert pa.get_device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(pa):
    w = wl.shared_prefix(batch=64)
    dev = torch.device("cuda")
    q, pool, tables, lens = _inputs(w, dev)
    part = 16
    assert pa.decode_workspace_size(pool, w.batch, w.num_q_heads, w.max_seq_len, part) > SCRATCH_BYTES
    out = torch.zeros_like(q)
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.decode_noalloc(out, q, pool, tables, lens, w.max_seq_len, w.scale, part)
    assert e.value.status == 3          # PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0   # nothing was launched
