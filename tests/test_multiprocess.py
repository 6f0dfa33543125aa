"""The N > 1 path of bench.py on CPU: world_size-2 gloo process groups.

The layer's tokens are independent, so N GPUs run N replicas with no
collective on the data path; the only cross-rank steps are the barrier
around the timed region and the max over ranks of the step time, and the
reference arm runs on rank 0 alone. These run here with the gloo backend."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    from token_dispatch_grouped_moe_gb300.configs import CONFIGS
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        dist.barrier()
        got = bench.max_over_ranks(values[rank])
        # the reference arm: every rank but 0 returns without work
        args = type("A", (), {"ref_tokens": 1, "steps": 1, "warmup": 0})()
        ref = bench.bench_reference(args, CONFIGS["tiny"]) if rank != 0 else "skipped"
        q.put((rank, r, w, local, got, ref))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("values", [(3.5, 2.25), (1.0, 7.0)])
def test_max_over_ranks_gloo(values):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, values, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, r, w, local, got, ref in res:
        assert (r, w, local) == (rank, world, rank)
        assert got == max(values)
        if rank != 0:
            assert ref is None


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.5) == 4.5
