"""Dynamic tile assignment (JFA_PLAN_DYNAMIC) on the GPU: forward and backward
against the fp64 oracle, element by element, with the tiles claimed at run
time -- few CTAs (many claims each), edge lengths, broadcast, packed -- and
repeated launches of one plan (the claim counter is reset per launch)."""
import pytest
import torch

import jagged_attention_gb300 as jfa
import workloads
from tests import parity

pytestmark = pytest.mark.gpu

DYN = jfa.PLAN_DYNAMIC


@pytest.fixture(scope="module", autouse=True)
def _built():
    jfa.build()


def _run(p, num_ctas=0, flags=DYN):
    p = parity.to_cuda(p)
    plan = parity.make_plan(p, num_ctas, flags)
    out, lse, _ = parity.gpu_fwd(p, plan)
    O_ref, L_ref = parity.oracle_fwd(p)
    parity.check_fwd(out, lse, O_ref, L_ref)
    dq, dk, dv = parity.gpu_bwd(p, out, lse, plan)
    rdq, rdk, rdv = parity.oracle_bwd(p)
    parity.check_grads(dq, dk, dv, rdq, rdk, rdv)
    return plan


@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_broadcast(seed):
    _run(workloads.make_workload("tiny_broadcast", seed=seed))


@pytest.mark.parametrize("num_ctas", [0, 3])
def test_jagged_self(num_ctas):
    _run(workloads.make_workload("jagged_self", seed=0), num_ctas=num_ctas)


@pytest.mark.parametrize("D", [64, 128])
def test_self_edge_lengths(D):
    lengths = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 0, 700]
    _run(workloads.make_problem(len(lengths), 2, D, "self", lengths, seed=3), num_ctas=4)


@pytest.mark.parametrize("Lq", [200, 300])
def test_broadcast_edge(Lq):
    _run(workloads.make_problem(6, 3, 128, "broadcast", [5, 0, 128, 129, 1000, 300], Lq=Lq, seed=4),
         num_ctas=5)


def test_packed_dynamic():
    lengths = [60, 40, 30, 200, 64, 64, 1, 1, 0, 127, 1, 5, 0, 0, 33, 95]
    _run(workloads.make_problem(len(lengths), 2, 128, "self", lengths, seed=20), num_ctas=3,
         flags=DYN | jfa.PLAN_PACK_SHORT)


def test_repeated_launches_reset_the_counter():
    p = parity.to_cuda(workloads.make_workload("jagged_self", seed=1))
    plan = parity.make_plan(p, 7, DYN)
    o1, l1, _ = parity.gpu_fwd(p, plan)
    o2, l2, _ = parity.gpu_fwd(p, plan)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = parity.gpu_bwd(p, o1, l1, plan)
    g2 = parity.gpu_bwd(p, o1, l1, plan)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])


def test_default_claims_rule():
    # by default the backward claims its tiles in self mode and is dealt on
    # the host in broadcast mode; the forward is dealt on the host; the flags
    # force either way, and the default self-mode plan matches the oracle
    self_p = parity.to_cuda(workloads.make_workload("jagged_self", seed=2))
    bc = parity.to_cuda(workloads.make_workload("tiny_broadcast", seed=2))
    assert parity.make_plan(self_p).claims() == (False, True)
    assert parity.make_plan(bc).claims() == (False, False)
    assert parity.make_plan(self_p, 0, jfa.PLAN_STATIC).claims() == (False, False)
    assert parity.make_plan(bc, 0, DYN).claims() == (True, True)
    plan = _run(workloads.make_workload("jagged_self", seed=2), 5, 0)
    tiles, ptr = plan.tiles(1)
    assert ptr[0] == 0 and (ptr[1:] == tiles.shape[0]).all()  # one claim queue
    _run(workloads.make_workload("jagged_self", seed=2), 5, jfa.PLAN_STATIC)
