"""Multi-process host logic of bench.py (replicas only: no exchange step on the data path), run as
world-size-2 gloo ranks on the CPU: the timing barrier, the max-over-ranks of the elapsed time, and the
reference arm printing on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.distributed as dist
import torch.multiprocessing as mp

from tests.conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    got = bench.max_over_ranks(float(rank + 1) * 1.5, world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 3.0, 1: 3.0}


def test_reference_arm_only_rank0_prints(monkeypatch):
    import bench
    from qwen3_decoder_transformer_gb300 import configs
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus, workload = 1, 3, 2, "tiny"
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, configs.WORKLOADS["tiny"])
    assert buf.getvalue() == ""


def test_single_process_identity():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
