"""Backward parity on the GPU: dQ, dK, dV from the CUDA path (which consumes
the CUDA forward's O and LSE) against the fp64 oracle, relative L2 <= 1e-2,
on the workloads at test size and on the edge cases."""
import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import jagged_attention_gb300 as jfa
    jfa.build()


def _run(p, num_ctas=0, flags=0):
    p = parity.to_cuda(p)
    plan = parity.make_plan(p, num_ctas, flags)
    out, lse, _ = parity.gpu_fwd(p, plan)
    dq, dk, dv = parity.gpu_bwd(p, out, lse, plan)
    rdq, rdk, rdv = parity.oracle_bwd(p)
    parity.check_grads(dq, dk, dv, rdq, rdk, rdv)
    return dq, dk, dv


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_broadcast_workload(seed):
    _run(workloads.make_workload("tiny_broadcast", seed=seed))


def test_jagged_self_workload():
    _run(workloads.make_workload("jagged_self", seed=0))


EDGE_LENGTHS = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 0, 700]


@pytest.mark.parametrize("D", [64, 128])
def test_self_edge_lengths(D):
    _run(workloads.make_problem(len(EDGE_LENGTHS), 2, D, "self", EDGE_LENGTHS, seed=3))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq", [1, 128, 200, 256, 300])
def test_broadcast_edge(D, Lq):
    _run(workloads.make_problem(6, 3, D, "broadcast", [5, 0, 128, 129, 1000, 300], Lq=Lq, seed=4))


def test_cross_lengths_with_queryless_sequences():
    # sequence 2 has keys but no queries: its dK / dV must come out zero
    dq, dk, dv = _run(workloads.make_problem(5, 2, 128, "self", [100, 300, 7, 0, 129],
                                             q_lengths=[130, 2, 0, 50, 256], seed=5))
    s, e = 400, 407
    assert dk[s:e].abs().max().item() == 0 and dv[s:e].abs().max().item() == 0


def test_long_sequences_and_few_ctas():
    _run(workloads.make_problem(3, 2, 128, "self", [3000, 1500, 129], seed=6), num_ctas=5)


def test_single_cta_broadcast():
    _run(workloads.make_problem(5, 2, 64, "broadcast", [300, 10, 0, 700, 128], Lq=130, seed=7),
         num_ctas=1)


def test_dk_dv_deterministic():
    p = parity.to_cuda(workloads.make_workload("tiny_broadcast", seed=1))
    plan = parity.make_plan(p)
    out, lse, _ = parity.gpu_fwd(p, plan)
    a = parity.gpu_bwd(p, out, lse, plan)
    b = parity.gpu_bwd(p, out, lse, plan)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dQ is reduce-added in arbitrary order: equal up to fp32 rounding
    assert (a[0] - b[0]).abs().max().item() <= 1e-5 * max(1.0, a[0].abs().max().item())


PACKED_LENGTHS = [60, 40, 30, 200, 64, 64, 1, 1, 0, 127, 1, 5, 0, 0, 33, 95]


@pytest.mark.parametrize("D", [64, 128])
def test_packed_short_sequences(D):
    import jagged_attention_gb300 as jfa
    _run(workloads.make_problem(len(PACKED_LENGTHS), 2, D, "self", PACKED_LENGTHS, seed=20),
         flags=jfa.PLAN_PACK_SHORT)


def test_packed_block_diagonal_segments():
    import jagged_attention_gb300 as jfa
    _run(workloads.make_problem(24, 2, 128, "self", [64] * 24, seed=21), flags=jfa.PLAN_PACK_SHORT)


# Mostly short sequences plus two long ones: the pre-pass clears only the long
# ones' dQ rows and the tiles of single-key-block sequences store theirs
# (dQ is NaN-prefilled, so a row neither cleared nor stored would show up).
OWNER_LENGTHS = [50, 128, 1, 300, 64, 64, 100, 90, 20, 129, 77]


@pytest.mark.parametrize("D", [64, 128])
def test_single_key_block_sequences_store_their_dq(D):
    _run(workloads.make_problem(len(OWNER_LENGTHS), 2, D, "self", OWNER_LENGTHS, seed=22))


def test_single_key_block_cross_attention():
    # queries with their own offsets: one key block but several query blocks
    _run(workloads.make_problem(4, 2, 128, "self", [100, 128, 700, 40],
                                q_lengths=[300, 0, 129, 257], seed=23))
