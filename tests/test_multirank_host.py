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

import numpy as np
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


# ---------------------------------------------------------------------------
# One batch split across two ranks (bench.py --split-batch): each rank takes
# its share of the sequences, computes its shard (the fp64 oracle stands in
# for the device on the CPU), and broadcast mode's dQ is summed over the ranks
# with the same all-reduce the benchmark issues; rank 0 gathers every piece.
SPLIT_CASES = {
    "broadcast": lambda: __import__("workloads").make_problem(
        7, 2, 64, "broadcast", [5, 300, 1, 129, 700, 64, 200], Lq=70, seed=31),
    "self": lambda: __import__("workloads").make_problem(
        6, 2, 64, "self", [90, 0, 400, 33, 128, 260], q_lengths=[10, 7, 300, 0, 64, 129], seed=32),
}


def _split_main(rank: int, world: int, port: int, case: str, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle

        full = SPLIT_CASES[case]()
        ranges = bench.split_batch(full, world)
        p = bench.shard_problem(full, *ranges[rank])
        orc = oracle.default()
        O, L = orc.fwd(p.q, p.k, p.v, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq, p.D, p.scale)
        dq, dk, dv = orc.bwd(p.q, p.k, p.v, p.dout, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq, p.D,
                             p.scale)
        bench.reduce_dq(dist, p, dq)
        pieces = [None] * world
        dist.all_gather_object(pieces, (ranges[rank], O.numpy(), L.numpy(), dq.numpy(), dk.numpy(),
                                        dv.numpy()))
        out.put((rank, ranges, pieces))  # numpy arrays travel by value (tensors would by handle)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(SPLIT_CASES))
def test_split_batch_shards_recombine_to_the_whole_batch(case):
    import oracle
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_split_main, args=(r, WORLD, port, case, out)) for r in range(WORLD)]
    for pr in procs:
        pr.start()
    got = sorted([out.get(timeout=120) for _ in range(WORLD)], key=lambda g: g[0])
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    full = SPLIT_CASES[case]()
    ranges = got[0][1]
    assert ranges == got[1][1] and ranges[0][0] == 0 and ranges[-1][1] == full.B
    assert all(b0 < b1 for b0, b1 in ranges) and ranges[0][1] == ranges[1][0]
    orc = oracle.default()
    O, L = orc.fwd(full.q, full.k, full.v, full.kv_offsets, full.q_offsets, full.B, full.H, full.Lq,
                   full.D, full.scale)
    dq, dk, dv = orc.bwd(full.q, full.k, full.v, full.dout, full.kv_offsets, full.q_offsets, full.B,
                         full.H, full.Lq, full.D, full.scale)
    pieces = [tuple(torch.from_numpy(a) if isinstance(a, np.ndarray) else a for a in x)
              for x in got[0][2]]
    # each rank's O, LSE, dK, dV are the whole batch's rows of its sequences
    torch.testing.assert_close(torch.cat([x[1] for x in pieces]), O, rtol=0, atol=0)
    torch.testing.assert_close(torch.cat([x[2] for x in pieces], dim=1), L, rtol=0, atol=0)
    torch.testing.assert_close(torch.cat([x[4] for x in pieces]), dk, rtol=0, atol=0)
    torch.testing.assert_close(torch.cat([x[5] for x in pieces]), dv, rtol=0, atol=0)
    if full.mode == "broadcast":  # every rank holds the summed dQ
        for x in pieces:
            torch.testing.assert_close(x[3], dq, rtol=1e-12, atol=1e-12)
    else:
        torch.testing.assert_close(torch.cat([x[3] for x in pieces]), dq, rtol=0, atol=0)


def test_split_batch_balances_the_work():
    import bench
    import workloads
    p = workloads.make_workload("gem_broadcast", seed=0, batch=256)
    work = p.q_lengths * p.kv_lengths
    for world in (2, 4, 8):
        ranges = bench.split_batch(p, world)
        assert [r[0] for r in ranges[1:]] == [r[1] for r in ranges[:-1]]
        shares = np.array([work[b0:b1].sum() for b0, b1 in ranges]) / work.sum()
        # a range ends where the running work crosses its share: off by at most one sequence
        assert np.all(np.abs(shares - 1.0 / world) <= work.max() / work.sum() + 1e-12)
