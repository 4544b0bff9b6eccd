"""The multi-rank path of bench.py on CPU: two gloo ranks (world size 2)
exercise the host logic a torchrun launch uses -- each rank's batch (same
workload shape, its own seed), the max over ranks of the timings, the sum of
the ranks' work, the aggregate throughput, and the reference arm running on
rank 0 alone.  The data path has no collective (weak scaling over
independent batches), so nothing else is exchanged."""
import contextlib
import io
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORLD = 2


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads

        p = workloads.make_workload("tiny_broadcast", seed=bench.rank_seed(0, rank), device="cpu")
        shapes = [None] * world
        dist.all_gather_object(shapes, (p.B, p.H, p.D, p.Lq, p.mode))
        lengths = [None] * world
        dist.all_gather_object(lengths, p.kv_lengths.tolist())

        times = bench.combine_over_ranks(dist, [10.0 + rank, 5.0 * rank, 7.0 - rank])
        fl = bench.flops(p, "fwd") + bench.flops(p, "bwd")
        job = bench.sum_over_ranks(dist, fl)
        fls = [None] * world
        dist.all_gather_object(fls, fl)

        class _Args:
            workload, seed, steps, warmup = "tiny_broadcast", 0, 1, 3
        printed = io.StringIO()
        with contextlib.redirect_stdout(printed):
            ref = bench.run_reference(_Args, rank, world) if rank != 0 else None
        out.put((rank, shapes, lengths, times, job, fls, ref, printed.getvalue()))
    finally:
        dist.destroy_process_group()


@pytest.fixture(scope="module")
def ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, WORLD, port, out)) for r in range(WORLD)]
    for pr in procs:
        pr.start()
    got = [out.get(timeout=120) for _ in range(WORLD)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    return sorted(got, key=lambda g: g[0])


def test_each_rank_has_its_own_batch_of_the_same_shape(ranks):
    (_, shapes0, lengths0, *_), (_, shapes1, lengths1, *_) = ranks
    assert shapes0 == shapes1 and shapes0[0] == shapes0[1]
    assert lengths0[0] != lengths0[1], "ranks must draw different batches"
    assert lengths0 == lengths1


def test_timings_take_the_slowest_rank(ranks):
    for _, _, _, times, *_ in ranks:
        assert times == [11.0, 5.0, 7.0]


def test_job_work_sums_the_ranks(ranks):
    import bench
    for _, _, _, _, job, fls, _, _ in ranks:
        assert job == pytest.approx(sum(fls))
        assert bench.aggregate_tflops(job, 2.0) == pytest.approx(sum(fls) / 2e-3 / 1e12)


def test_reference_arm_runs_on_rank_zero_only(ranks):
    rank1 = [r for r in ranks if r[0] == 1][0]
    assert rank1[6] is None and rank1[7] == ""
