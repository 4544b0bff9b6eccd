"""The plan-free entry points (jfa_fwd_simple / jfa_bwd_simple): tensors, host
offsets and sizes in one call, the library caching one plan per distinct
offsets.  Their results must equal the plan path's (bit for bit where that is
deterministic: O, LSE, dK, dV; dQ up to the order of its reduce-adds) and the
oracle's within the parity tolerances, also after the cache has released its
least recently used plan."""
import numpy as np
import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import jagged_attention_gb300 as jfa
    jfa.build()
    yield
    jfa.simple_release()


CASES = {
    "tiny_broadcast": lambda: workloads.make_workload("tiny_broadcast", seed=0),
    "jagged_self": lambda: workloads.make_workload("jagged_self", seed=0),
    "cross": lambda: workloads.make_problem(5, 2, 128, "self", [100, 300, 7, 0, 129],
                                            q_lengths=[130, 2, 0, 50, 256], seed=5),
}


def _simple(p):
    import jagged_attention_gb300 as jfa
    g = [parity.guarded((p.n_o_rows, p.H, p.D), torch.bfloat16),
         parity.guarded((p.H, p.n_o_rows), torch.float32),
         parity.guarded(p.q.shape, torch.float32),
         parity.guarded(p.k.shape, torch.bfloat16),
         parity.guarded(p.v.shape, torch.bfloat16)]
    out, lse, dq, dk, dv = (x.t for x in g)
    jfa.fwd_simple(p.q, p.k, p.v, p.kv_offsets, p.q_offsets, scale=p.scale, out=out, lse=lse)
    jfa.bwd_simple(p.q, p.k, p.v, out, p.dout, lse, p.kv_offsets, p.q_offsets, scale=p.scale,
                   dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert jfa.simple_device_status() == 0
    for x, n in zip(g, ("O", "LSE", "dQ", "dK", "dV")):
        x.check(n)
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("name", sorted(CASES))
def test_simple_equals_the_plan_path_and_the_oracle(name):
    p = parity.to_cuda(CASES[name]())
    out, lse, dq, dk, dv = _simple(p)
    plan = parity.make_plan(p)
    pout, plse, _ = parity.gpu_fwd(p, plan)
    pdq, pdk, pdv = parity.gpu_bwd(p, pout, plse, plan)
    assert torch.equal(out, pout) and torch.equal(lse.nan_to_num(), plse.nan_to_num())
    assert torch.equal(dk, pdk) and torch.equal(dv, pdv)
    assert (dq - pdq).abs().max().item() <= 1e-5 * max(1.0, pdq.abs().max().item())
    parity.check_fwd(out, lse, *parity.oracle_fwd(p))
    parity.check_grads(dq, dk, dv, *parity.oracle_bwd(p))


def test_simple_cache_releases_its_least_recent_plan():
    import jagged_attention_gb300 as jfa
    rng = np.random.default_rng(40)
    problems = [parity.to_cuda(workloads.make_problem(3, 2, 64, "self",
                                                      [int(x) for x in rng.integers(1, 300, 3)],
                                                      seed=41 + i)) for i in range(10)]
    first = _simple(problems[0])
    for p in problems[1:]:  # nine more distinct offsets: the cache holds eight
        out, lse, dq, dk, dv = _simple(p)
        parity.check_grads(dq, dk, dv, *parity.oracle_bwd(p))
    again = _simple(problems[0])  # rebuilt after its release
    assert torch.equal(first[0], again[0]) and torch.equal(first[3], again[3])
    jfa.simple_release()
    assert jfa.simple_device_status() == 0
