"""The bench's multi-rank path on the CPU (gloo, two processes): one process
per rank, each decoding its own batch, the job's time the slowest rank's, and
rank 0 alone printing the JSON line.  No GPU: the collective and the per-rank
workloads are what differs from one rank."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _reduce_worker(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each rank's timings differ; every rank must end with the maxima
    got = bench.reduce_max([1.0 + rank, 10.0 - rank, 5.0], world, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(got, f)


def test_reduce_max_over_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_reduce_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        with open(tmp_path / f"rank{rank}.json") as f:
            assert json.load(f) == [2.0, 10.0, 5.0]


def test_reduce_max_one_rank():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max([3.0, 1.5], 1, torch.device("cpu")) == [3.0, 1.5]


def test_each_rank_decodes_its_own_batch():
    sys.path.insert(0, ROOT)
    import bench
    w0, w1 = bench.rank_workload("llama70b_decode", 0), bench.rank_workload("llama70b_decode", 1)
    assert (w0.batch, w0.num_q_heads, w0.num_kv_heads, w0.head_dim, w0.block_size) == \
        (w1.batch, w1.num_q_heads, w1.num_kv_heads, w1.head_dim, w1.block_size)
    assert not np.array_equal(w0.seq_lens, w1.seq_lens) or not np.array_equal(w0.tables, w1.tables)
    assert bench.decode_bytes(w0) > 0 and bench.decode_bytes(w1) > 0
    t0, t1 = bench.rank_workload("tiny", 0), bench.rank_workload("tiny", 1)
    assert np.array_equal(t0.seq_lens, t1.seq_lens) and np.array_equal(t0.tables, t1.tables)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as the driver launches it for N = 2:
    rank 0 prints one JSON line, the other rank exits 0 without output."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--config", "tiny"]
    proc = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [ln for ln in proc.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, proc.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
