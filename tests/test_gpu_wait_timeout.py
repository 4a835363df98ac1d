"""The bounded waits give up without a fault: a kernel whose barrier wait
nothing completes records PA_DEVERR_TIMEOUT after its limit and returns; the
host reads the word, and the context stays usable (a decode afterwards still
matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import pa_workloads as wl
from tests.parity import Case, assert_close

pytestmark = pytest.mark.gpu

PA_DEVERR_TIMEOUT = 0x8


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_167_gb300 as pa
    assert torch.cuda.is_available(), "a CUDA device is required"
    pa.get_device_error(clear=True)
    return pa


def test_wait_gives_up_and_context_survives(pa):
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pa.check_wait_timeout(20_000_000)          # 20 ms
    word = pa.get_device_error()               # synchronises, then clears
    elapsed = time.perf_counter() - t0
    assert word == PA_DEVERR_TIMEOUT
    assert elapsed >= 0.02
    assert pa.get_device_error() == 0
    w = wl.tiny()
    c = Case(w)
    out = torch.empty_like(c.q)
    nb = pa.decode_workspace_size(c.pool, w.batch, w.num_q_heads, w.max_seq_len, 0)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=c.dev)
    pa.decode(out, c.q, c.pool, c.tables, c.seq_lens, w.max_seq_len, w.scale, 0, ws)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    ref = c.orc.paged_decode(wl.bf16_bits(c.cpu["q"]), c.pool_ref, c.geom, w.tables, w.seq_lens, w.num_q_heads,
                             w.scale)
    assert_close(out, ref, "decode after a timed-out wait")
