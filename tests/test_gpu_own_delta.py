"""Backward with Delta formed inside the kernel.  When every sequence with
queries has at most one key block, each backward tile meets all the keys of
its queries, and Delta_i = sum_d dO_id O_id equals sum_j P_ij dP_ij over that
tile's keys (O = P V, dP = dO V^T), so the kernel sums it itself and the
pre-pass that reads O and dO for it can be skipped (by default when the tiles
hold at least 96 key rows on average; JFA_PLAN_DELTA_IN_TILES whatever their
fill).  Checked here: parity with the fp64 oracle on the edge lengths of that
regime, agreement with the forced pre-pass (JFA_PLAN_DELTA_PREPASS), the
default rule, and which path ran -- an O filled with NaN reaches the gradients
only through the pre-pass."""
import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import jagged_attention_gb300 as jfa
    jfa.build()


SHORT = [1, 2, 63, 64, 65, 127, 128, 0, 100, 17, 128, 3]

CASES = {
    # self mode: one key block per sequence, ragged tails, an empty sequence
    "self": lambda D: workloads.make_problem(len(SHORT), 2, D, "self", SHORT, seed=30),
    # queries with their own offsets: up to three query blocks against one key
    # block, a sequence with queries but no keys, one with keys but no queries
    "cross": lambda D: workloads.make_problem(5, 2, D, "self", [128, 5, 0, 90, 64],
                                              q_lengths=[300, 1, 40, 0, 129], seed=31),
    # broadcast: every sequence sees the same 300 queries (three query blocks)
    "broadcast": lambda D: workloads.make_problem(6, 3, D, "broadcast", [5, 0, 128, 77, 1, 64],
                                                  Lq=300, seed=32),
}


def _grads(p, flags=0, poison_out=False):
    plan = parity.make_plan(p, 0, flags)
    out, lse, _ = parity.gpu_fwd(p, plan)
    if poison_out:
        out = torch.full_like(out, float("nan"))
    return parity.gpu_bwd(p, out, lse, plan)


def _in_tiles():
    import jagged_attention_gb300 as jfa
    return jfa.PLAN_DELTA_IN_TILES


@pytest.mark.parametrize("flags", [32, 1, 34])  # PLAN_NO_PACK, PLAN_PACK_SHORT, PLAN_DYNAMIC | PLAN_NO_PACK
@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("D", [64, 128])
def test_in_kernel_delta_matches_oracle(D, case, flags):
    p = parity.to_cuda(CASES[case](D))
    dq, dk, dv = _grads(p, flags | _in_tiles(), poison_out=True)
    parity.check_grads(dq, dk, dv, *parity.oracle_bwd(p))


@pytest.mark.parametrize("case", sorted(CASES))
def test_in_kernel_delta_agrees_with_the_prepass(case):
    import jagged_attention_gb300 as jfa
    p = parity.to_cuda(CASES[case](128))
    a = _grads(p, jfa.PLAN_DELTA_IN_TILES)
    b = _grads(p, jfa.PLAN_DELTA_PREPASS)
    parity.check_grads(*b, *parity.oracle_bwd(p))
    for x, y in zip(a, b):
        assert parity.rel_l2(x, y) <= parity.TOL_GRAD


@pytest.mark.parametrize("case", sorted(CASES))
def test_o_is_not_read_when_tiles_form_delta(case):
    import jagged_attention_gb300 as jfa
    p = parity.to_cuda(CASES[case](128))
    dq, dk, dv = _grads(p, jfa.PLAN_DELTA_IN_TILES, poison_out=True)
    parity.check_grads(dq, dk, dv, *parity.oracle_bwd(p))
    # the forced pre-pass does read O: its NaN reaches dK through Delta
    _, dk_pre, _ = _grads(p, jfa.PLAN_DELTA_PREPASS, poison_out=True)
    assert torch.isnan(dk_pre.float()).any()


def test_long_sequence_keeps_the_prepass():
    # one sequence of 129 keys: its tiles see only part of its keys, so the
    # plan must keep the pre-pass even when asked for tiles, and a NaN O must
    # show up in dK
    p = parity.to_cuda(workloads.make_problem(3, 2, 128, "self", [64, 129, 10], seed=33))
    _, dk, _ = _grads(p, _in_tiles(), poison_out=True)
    assert torch.isnan(dk.float()).any()
    parity.check_grads(*_grads(p, _in_tiles()), *parity.oracle_bwd(p))


def test_default_rule_full_tiles_form_delta():
    # 64-token segments packed two per tile: 128 key rows per tile
    import jagged_attention_gb300 as jfa
    p = parity.to_cuda(workloads.make_problem(24, 2, 128, "self", [64] * 24, seed=35))
    dq, dk, dv = _grads(p, jfa.PLAN_PACK_SHORT, poison_out=True)
    parity.check_grads(dq, dk, dv, *parity.oracle_bwd(p))


def test_default_rule_half_full_tiles_keep_the_prepass():
    # the same segments one per tile (packing turned off): 64 key rows per tile
    import jagged_attention_gb300 as jfa
    p = parity.to_cuda(workloads.make_problem(24, 2, 128, "self", [64] * 24, seed=35))
    _, dk, _ = _grads(p, jfa.PLAN_NO_PACK, poison_out=True)
    assert torch.isnan(dk.float()).any()
