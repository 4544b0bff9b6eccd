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


def test_mma_selftest_rejects_bad_arguments():
    # argument checks happen before any launch (runs without a GPU)
    import ctypes
    L = jfa.lib()
    c = ctypes.c_ulonglong()
    assert L.jfa_selftest_mma_cycles(7, 16, 0, ctypes.byref(c), None, None) == JFA_ERR_INVALID_ARG
    assert L.jfa_selftest_mma_cycles(0, 0, 0, ctypes.byref(c), None, None) == JFA_ERR_INVALID_ARG
    assert L.jfa_selftest_mma_cycles(0, 12, 0, ctypes.byref(c), None, None) == JFA_ERR_INVALID_ARG
    assert L.jfa_selftest_mma_cycles(0, 16, 0, None, None, None) == JFA_ERR_INVALID_ARG
    assert L.jfa_selftest_mma_cycles(0, 16, 12, ctypes.byref(c), None, None) == JFA_ERR_INVALID_ARG
    assert L.jfa_selftest_mma_cycles(0, 24, 16, ctypes.byref(c), None, None) == JFA_ERR_INVALID_ARG


def test_plan_selftest_rejects_bad_arguments():
    # host-side checks only (no plan, bad codes and limits): runs without a GPU
    L = jfa.lib()
    assert L.jfa_plan_selftest(None, 1, 1000) == JFA_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("skip,flags", [(1, 0), (2, 0), (1, jfa.PLAN_FWD_PAIRS), (1, jfa.PLAN_FWD_TWO)])
def test_real_kernel_timeout_cascade(skip, flags):
    """One softmax warp of CTA 0 withholds one arrival (skip 1: the forward's
    first P block, 2: the backward's first dS^T), with every wait limited to
    20 ms: the MMA issuer's wait runs out, the abort reaches every role of the
    CTA (producer drain, MMA drain commit, TMEM release), the launch ends, the
    plan's status word reports JFA_ERR_DEVICE_TIMEOUT, and a normal forward
    and backward right after still match the oracle.  With CTA pairs the odd
    CTA's roles run out on their own waits (its loads' forwarder, its softmax
    warps) and both CTAs meet at the cluster barrier before releasing TMEM."""
    import torch
    if flags & (jfa.PLAN_FWD_PAIRS | jfa.PLAN_FWD_TWO):  # D = 128, two query blocks per sequence
        p = parity.to_cuda(workloads.make_problem(3, 2, 128, "broadcast", [300, 5, 128], Lq=256, seed=57))
    else:
        p = parity.to_cuda(workloads.make_workload("tiny_broadcast", seed=0))
    plan = parity.make_plan(p, 0, flags)
    assert plan.forward_form() == (1 if flags & jfa.PLAN_FWD_PAIRS else 2 if flags & jfa.PLAN_FWD_TWO else 0)
    out, lse, _ = parity.gpu_fwd(p, plan)
    plan.selftest(skip, 20000)
    if skip == 1:
        o2 = torch.empty_like(out)
        l2 = torch.empty_like(lse)
        jfa.fwd(plan, p.q, p.k, p.v, p.scale, out=o2, lse=l2)
    else:
        dq = torch.empty(p.q.shape, dtype=torch.float32, device="cuda")
        dk, dv = torch.empty_like(p.k), torch.empty_like(p.v)
        jfa.bwd(plan, p.q, p.k, p.v, out, p.dout, lse, p.scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    with pytest.raises(jfa.JfaError) as err:
        plan.device_status()
    assert err.value.code == JFA_ERR_DEVICE_TIMEOUT
    plan.selftest(0, 0)
    out, lse, _ = parity.gpu_fwd(p, plan)  # asserts a clean status word
    parity.check_fwd(out, lse, *parity.oracle_fwd(p))
    dq, dk, dv = parity.gpu_bwd(p, out, lse, plan)
    parity.check_grads(dq, dk, dv, *parity.oracle_bwd(p))
