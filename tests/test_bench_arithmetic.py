"""The bench's algorithmic byte and FLOP counts against closed forms of the
workloads (no GPU): the roofline's numerator must be the work the path has to
do, not what a kernel happened to move."""
import numpy as np

import bench
import pa_workloads as wl


def test_decode_bytes_llama():
    w = wl.llama70b_decode()
    L = w.seq_lens.astype(np.int64)
    kv = int(L.sum()) * 8 * 128 * 2 * 2                  # K and V rows of every attended token, bf16
    qo = 2 * 64 * 64 * 128 * 2                            # q and out once
    meta = 4 * int(((L + 15) // 16).sum()) + 4 * 64       # table entries used, lengths
    assert bench.decode_bytes(w) == kv + qo + meta
    assert bench.unique_decode_bytes(w) == bench.decode_bytes(w)   # no shared blocks
    assert 188e6 < bench.decode_bytes(w) < 191e6                  # the ~190 MB of the step


def test_unique_bytes_shared_prompt():
    """The 2,000-token prompt counts once: logical - unique = 255 x 2,000
    tokens of K and V for 8 heads."""
    w = wl.shared_prefix()
    diff = bench.decode_bytes(w) - bench.unique_decode_bytes(w)
    assert diff == 255 * 2000 * 8 * 128 * 2 * 2


def test_unique_bytes_beams():
    """Each prompt's full blocks count once for its four beams; every beam's
    last (own) block counts for itself."""
    w = wl.beam_fork()
    plen = w.notes["prompt_lens"].astype(np.int64)
    shared_tokens = (plen // 16) * 16
    diff = bench.decode_bytes(w) - bench.unique_decode_bytes(w)
    assert diff == int((3 * shared_tokens).sum()) * 8 * 128 * 2 * 2


def test_prefill_flops():
    w = wl.prefill_chunk()
    # 16 sequences; query j of the chunk sees 4096 + j + 1 keys; 4 d FLOPs a key and head
    visible = 16 * sum(4096 + j + 1 for j in range(512))
    assert bench.prefill_flops(w) == 4 * 128 * visible * 64 == 1168365322240


def test_cascade_groups():
    assert bench.cascade_group_size(wl.shared_prefix()) == 256
    assert bench.cascade_group_size(wl.beam_fork()) == 4
    assert bench.cascade_group_size(wl.llama70b_decode()) is None
