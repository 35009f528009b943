"""bench.py's multi-GPU arithmetic on CPU: two gloo ranks (replicas only -- the
decode step has no cross-session collective, so each rank runs its own model
and sessions). The timed region's length is the slowest rank's, on every rank,
and the reported throughput is all ranks' tokens over that time."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, local_seconds, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest = bench.max_over_ranks(local_seconds[rank], world, "cpu")
        out.put((rank, slowest, bench.whole_job_tok_s(8, 10, world, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_all_tokens():
    world, local = 2, [0.25, 0.4]
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, local, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(out.get() for _ in range(world))
    for rank, slowest, tok_s in got:
        assert slowest == 0.4
        assert tok_s == pytest.approx(8 * 10 * world / 0.4)


def test_one_rank_is_its_own_maximum():
    import bench
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5
    assert bench.whole_job_tok_s(8, 256, 1, 0.5) == pytest.approx(4096.0)
