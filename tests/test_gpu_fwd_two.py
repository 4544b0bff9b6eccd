"""Forward with two query tiles in flight per CTA (JFA_PLAN_FWD_TWO, D = 128):
each schedule tile covers two query blocks of one (sequence, head), which
share every K/V block, and the CTA alternates between them.  Checked against
the fp64 oracle, and against the one-tile forward on the same inputs, on
broadcast and self-mode batches: empty sequences, ragged key tails, a tile
whose second query block is empty or partial, few CTAs for many tiles (each
tile's O leaving through the K and V stages of its last key block while the
producer's next loads into those stages wait for it), the backward after it,
and when a plan runs it."""
import numpy as np
import pytest
import torch

import jagged_attention_gb300 as jfa
import workloads
from tests import parity

pytestmark = pytest.mark.gpu
TWO = jfa.PLAN_FWD_TWO


@pytest.fixture(scope="module", autouse=True)
def _built():
    jfa.build()


CASES = {
    "broadcast_256": lambda: workloads.make_problem(6, 3, 128, "broadcast", [5, 0, 128, 129, 1000, 300],
                                                    Lq=256, seed=61),
    "broadcast_200": lambda: workloads.make_problem(5, 2, 128, "broadcast", [64, 700, 1, 257, 128],
                                                    Lq=200, seed=62),
    "broadcast_600": lambda: workloads.make_problem(4, 2, 128, "broadcast", [900, 0, 130, 2000],
                                                    Lq=600, seed=63),
    "self_mixed": lambda: workloads.make_problem(7, 2, 128, "self", [256, 255, 384, 0, 1024, 130, 512],
                                                 q_lengths=[256, 200, 300, 0, 1024, 256, 512], seed=64),
    "gem_slice": lambda: workloads.make_workload("gem_broadcast", seed=4, batch=64),
}


def _fwd(p, flags=0, num_ctas=0):
    plan = parity.make_plan(p, num_ctas, flags)
    out, lse, _ = parity.gpu_fwd(p, plan)
    return out, lse, plan


@pytest.mark.parametrize("num_ctas", [0, 1, 3])
@pytest.mark.parametrize("name", sorted(CASES))
def test_two_tiles_match_oracle_and_one_tile(name, num_ctas):
    p = parity.to_cuda(CASES[name]())
    out, lse, plan = _fwd(p, TWO | jfa.PLAN_NO_PACK, num_ctas)
    assert plan.forward_form() == 2
    parity.check_fwd(out, lse, *parity.oracle_fwd(p))
    o1, l1, plan1 = _fwd(p, jfa.PLAN_FWD_ONE | jfa.PLAN_NO_PACK, num_ctas)
    assert plan1.forward_form() == 0
    # the same fp32 arithmetic per row, in the same order: equal bits
    assert torch.equal(out, o1)
    assert torch.equal(lse.nan_to_num(), l1.nan_to_num())


def test_backward_after_two_tile_forward():
    p = parity.to_cuda(CASES["broadcast_600"]())
    out, lse, plan = _fwd(p, TWO)
    dq, dk, dv = parity.gpu_bwd(p, out, lse, plan)
    parity.check_grads(dq, dk, dv, *parity.oracle_bwd(p))


def test_plan_rule_for_two_tiles():
    # by default: tiles of two query blocks holding >= 3 key blocks on average,
    # at most a quarter of them half empty, at least four of them per CTA
    even = parity.to_cuda(CASES["broadcast_256"]())          # 2.5 key blocks per tile
    assert parity.make_plan(even).forward_form() == 0
    assert parity.make_plan(even, 0, TWO).forward_form() == 2
    long_ = parity.to_cuda(CASES["broadcast_600"]())         # 2 of 3 tiles per sequence full
    assert parity.make_plan(long_).forward_form() == 0       # a third half empty
    gem = parity.to_cuda(CASES["gem_slice"]())               # 256 two-block tiles
    assert parity.make_plan(gem, 16).forward_form() == 2     # 16 per CTA
    assert parity.make_plan(gem, 152).forward_form() == 0    # under 4 per CTA
    assert parity.make_plan(gem, 16, jfa.PLAN_FWD_ONE).forward_form() == 0
    assert parity.make_plan(gem, 16, jfa.PLAN_FWD_PAIRS).forward_form() == 1
    assert parity.make_plan(even, 0, TWO | jfa.PLAN_DYNAMIC).forward_form() == 0
    d64 = parity.to_cuda(workloads.make_problem(3, 2, 64, "broadcast", [300, 5, 128], Lq=256, seed=65))
    assert parity.make_plan(d64, 0, TWO).forward_form() == 0
    # its schedule is the host builder's list of two-block tiles over num_ctas CTAs
    tiles, ptr = parity.make_plan(even, 5, TWO).tiles(0)
    rt, rp = jfa.build_tiles(even.kv_offsets, None, H=even.H, Lq=even.Lq, num_ctas=5, direction=2)
    assert np.array_equal(tiles, rt) and np.array_equal(ptr, rp)
