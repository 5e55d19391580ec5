"""The N > 1 path of bench.py on CPU: two gloo ranks, each an independent
replica; the only cross-rank operations are the timing barrier and the
max-over-ranks reduction of the step time (there is no data-path exchange)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        bench.barrier(world)
        t = 1.5 if rank == 0 else 2.5
        q.put((rank, bench.max_over_ranks(t, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == {0: 2.5, 1: 2.5}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_other_ranks_exit_without_work(capsys):
    import bench

    class A:
        steps, warmup = 1, 0

    assert bench.run_reference(A(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""


def test_counted_flops_conventions():
    import bench
    import workloads as W
    s = W.SPECS["gpt2"]
    f = bench.counted_flops(s, None)
    assert f["fwd"] == pytest.approx(0.5 * 4 * 1024 * 1024 * 64 * 8 * 12)
    assert f["step"] == pytest.approx(3.5 * f["fwd"])
    s2 = W.SPECS["bert"]
    f2 = bench.counted_flops(s2, [256] * 16)
    assert f2["fwd"] == pytest.approx(4 * 512 * 256 * 64 * 16 * 16)
    assert f2["nominal_step"] == pytest.approx(3.5 * 4 * 512 * 512 * 64 * 256)
