"""The bench's N>1 path on CPU: N independent replicas (the method's ranks are
buffers inside one GPU, so GPUs exchange nothing), a barrier around the timed
region and the max over ranks of the elapsed time -- world size 2 over gloo."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.dist_barrier(w)
    mx = bench.dist_max(10.0 * (rank + 1), w)

    args = bench.build_parser().parse_args(["--config", "1", "--steps", "1", "--warmup", "0"])
    ref = bench.reference_arm(args, r, w)
    q.put((rank, mx, ref is None))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_and_reference_arm_on_rank_zero_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    assert out[0][1] == out[1][1] == 20.0          # every rank sees the max
    assert out[0][2] is False and out[1][2] is True  # only rank 0 runs the reference arm


def test_single_process_needs_no_process_group():
    import bench
    assert bench.dist_max(3.5, 1) == 3.5
    bench.dist_barrier(1)
