"""Forward as CTA pairs (JFA_PLAN_FWD_PAIRS, D = 128): two CTAs of a cluster
take the two query blocks of a pair tile and share each K/V block, one
thread issuing the pair's M = 256 tensor-core products.  Checked against the
fp64 oracle, and against the default one-CTA-per-block forward on the same
inputs, on broadcast and self-mode batches: empty sequences, ragged key
tails, a pair tile whose second query block is empty (odd block counts), few
pairs for many tiles, and when a plan runs the pair kernel."""
import pytest
import torch

import jagged_attention_gb300 as jfa
import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    jfa.build()


CASES = {
    # every sequence sees 256 queries: two query blocks, one pair tile each
    "broadcast_256": lambda: workloads.make_problem(6, 3, 128, "broadcast", [5, 0, 128, 129, 1000, 300],
                                                    Lq=256, seed=51),
    # ragged last query block (200 = 128 + 72 rows)
    "broadcast_200": lambda: workloads.make_problem(5, 2, 128, "broadcast", [64, 700, 1, 257, 128],
                                                    Lq=200, seed=52),
    # self mode: even block counts, one sequence with three blocks (its second
    # pair tile has an empty second block), empty and one-row sequences
    "self_mixed": lambda: workloads.make_problem(7, 2, 128, "self", [256, 255, 384, 0, 1024, 130, 512],
                                                 q_lengths=[256, 200, 300, 0, 1024, 256, 512], seed=53),
    "gem_slice": lambda: workloads.make_workload("gem_broadcast", seed=3, batch=64),
}


def _fwd(p, flags=0, num_ctas=0):
    plan = parity.make_plan(p, num_ctas, flags)
    out, lse, _ = parity.gpu_fwd(p, plan)
    return out, lse, plan


@pytest.mark.parametrize("num_ctas", [0, 2, 6])
@pytest.mark.parametrize("name", sorted(CASES))
def test_pair_forward_matches_oracle_and_single(name, num_ctas):
    p = parity.to_cuda(CASES[name]())
    out, lse, plan = _fwd(p, jfa.PLAN_FWD_PAIRS, num_ctas)
    assert plan.forward_pairs(), "the plan should run CTA pairs here"
    parity.check_fwd(out, lse, *parity.oracle_fwd(p))
    o1, l1, plan1 = _fwd(p, 0, num_ctas)
    assert not plan1.forward_pairs()
    # both kernels round the same fp32 arithmetic per row; they may differ
    # in the order of the PV accumulation only
    assert (out.float() - o1.float()).abs().max().item() <= 1e-2
    fin = torch.isfinite(l1)
    assert torch.equal(fin, torch.isfinite(lse))
    assert (lse[fin] - l1[fin]).abs().max().item() <= 1e-4


def test_backward_after_pair_forward():
    p = parity.to_cuda(CASES["broadcast_256"]())
    out, lse, plan = _fwd(p, jfa.PLAN_FWD_PAIRS)
    assert plan.forward_pairs()
    dq, dk, dv = parity.gpu_bwd(p, out, lse, plan)
    parity.check_grads(dq, dk, dv, *parity.oracle_bwd(p))


def test_plan_rule_for_pairs():
    PAIRS = jfa.PLAN_FWD_PAIRS
    even = parity.to_cuda(CASES["broadcast_256"]())
    # one CTA per block by default, with dynamic claiming, at D = 64, and
    # for packed tiles
    assert not parity.make_plan(even).forward_pairs()
    assert parity.make_plan(even, 0, PAIRS).forward_pairs()
    assert not parity.make_plan(even, 0, PAIRS | jfa.PLAN_DYNAMIC).forward_pairs()
    d64 = parity.to_cuda(workloads.make_problem(3, 2, 64, "broadcast", [300, 5, 128], Lq=256, seed=55))
    assert not parity.make_plan(d64, 0, PAIRS).forward_pairs()
    short = parity.to_cuda(workloads.make_problem(24, 2, 128, "self", [64] * 24, seed=56))
    assert not parity.make_plan(short, 0, PAIRS | jfa.PLAN_PACK_SHORT).forward_pairs()
    # one query block per sequence: every pair tile half empty, still pairs
    odd = parity.to_cuda(workloads.make_problem(6, 2, 128, "self", [100] * 6, seed=54))
    plan = parity.make_plan(odd, 0, PAIRS | jfa.PLAN_NO_PACK)
    assert plan.forward_pairs()
    out, lse, _ = parity.gpu_fwd(odd, plan)
    parity.check_fwd(out, lse, *parity.oracle_fwd(odd))
    # the pair schedule the plan launches is the host builder's
    tiles, ptr = parity.make_plan(even, 6, PAIRS).tiles(0)
    rt, rp = jfa.build_tiles(even.kv_offsets, None, H=even.H, Lq=even.Lq, num_ctas=3, direction=2)
    assert (tiles == rt).all() and (ptr == rp).all()
