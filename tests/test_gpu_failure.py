"""Failure detection without a GPU fault: a kernel wait on a barrier nothing
arrives on runs out after its (shortened) limit, the timeout reaches the
host as JFA_ERR_DEVICE_TIMEOUT, the kernel returns normally, and the context
keeps working (a forward right after still matches the oracle)."""
import pytest

import jagged_attention_gb300 as jfa
import workloads
from tests import parity

JFA_ERR_INVALID_ARG = 1
JFA_ERR_DEVICE_TIMEOUT = 7


@pytest.fixture(scope="module", autouse=True)
def _built():
    jfa.build()


def test_selftest_rejects_bad_limits():
    # argument checks happen before any launch (runs without a GPU)
    assert jfa.selftest_wait_timeout(0)[0] == JFA_ERR_INVALID_ARG
    assert jfa.selftest_wait_timeout(3_000_000)[0] == JFA_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("limit_us", [2000, 20000])
def test_wait_timeout_is_reported_and_context_survives(limit_us):
    rc, waited = jfa.selftest_wait_timeout(limit_us)
    assert rc == JFA_ERR_DEVICE_TIMEOUT
    assert limit_us * 1000 <= waited < limit_us * 1000 + 50_000_000
    p = parity.to_cuda(workloads.make_workload("tiny_broadcast", seed=0))
    plan = parity.make_plan(p)
    out, lse, _ = parity.gpu_fwd(p, plan)
    O_ref, L_ref = parity.oracle_fwd(p)
    parity.check_fwd(out, lse, O_ref, L_ref)
    assert plan.device_status() == 0
