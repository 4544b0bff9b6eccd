"""The backward entry point that allocates no device memory.

jfa_bwd_noalloc serves callers that cannot call cudaMalloc -- code inside a
framework whose pool allocator owns the device memory, or runtimes handed a
fixed set of pre-allocated buffers -- by keeping its schedule, offsets and
Delta row sums in a static device array instead of a plan and a workspace.
This file is collected last so that a run stopping at the first failure has
already run every other test.  Each case calls the entry point twice in a row
through the C ABI (the second call reuses the array the first one filled) and
compares dQ, dK and dV with jfa_bwd's, within the parity tests' relative-L2
tolerance.
"""
import ctypes

import pytest
import torch

import jagged_attention_gb300 as jfa
import workloads
from tests import parity

pytestmark = pytest.mark.gpu

_vp = ctypes.c_void_p


def _entry():
    L = jfa.lib()
    fn = L.jfa_bwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [jfa._i32p, jfa._i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp]
    return fn


def _outputs(p):
    """Guard-banded, NaN-prefilled dQ, dK, dV."""
    return (parity.guarded(p.q.shape, torch.float32), parity.guarded(p.k.shape, torch.bfloat16),
            parity.guarded(p.v.shape, torch.bfloat16))


def _launch(fn, p, out, lse, status, g):
    kv = jfa._offsets(p.kv_offsets)
    qo = jfa._offsets(p.q_offsets)
    dq, dk, dv = (x.t for x in g)
    return fn(jfa._i32ptr(kv), jfa._i32ptr(qo), p.B, p.H, p.Lq, p.D, p.q.data_ptr(), p.k.data_ptr(),
              p.v.data_ptr(), out.data_ptr(), p.dout.data_ptr(), lse.data_ptr(), p.scale,
              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), status.data_ptr(),
              torch.cuda.current_stream().cuda_stream)


def _call(fn, p, out, lse, status):
    g = _outputs(p)
    rc = _launch(fn, p, out, lse, status, g)
    assert rc == 0, jfa.STATUS_NAMES.get(rc, rc)
    torch.cuda.synchronize()
    for x, n in zip(g, ("dQ", "dK", "dV")):
        x.check(n)
    return tuple(x.t for x in g)


CASES = {
    "tiny_broadcast": lambda: workloads.make_workload("tiny_broadcast", seed=0),
    "jagged_self": lambda: workloads.make_workload("jagged_self", seed=1),
    "broadcast_edges": lambda: workloads.make_problem(6, 3, 128, "broadcast",
                                                      [5, 0, 128, 129, 1000, 300], Lq=200, seed=4),
    "cross_queryless": lambda: workloads.make_problem(5, 2, 64, "self", [100, 300, 7, 0, 129],
                                                      q_lengths=[130, 2, 0, 50, 256], seed=5),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_jfa_bwd_twice_in_a_row(name):
    jfa.build()
    fn = _entry()
    p = parity.to_cuda(CASES[name]())
    plan = parity.make_plan(p)
    out, lse, _ = parity.gpu_fwd(p, plan)
    ref = parity.gpu_bwd(p, out, lse, plan)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        got = _call(fn, p, out, lse, status)
        torch.cuda.synchronize()
        assert status.item() == 0
        for g, r in zip(got, ref):
            assert torch.isfinite(g.float()).all()
            assert parity.rel_l2(g, r) <= parity.TOL_GRAD


def test_noalloc_matches_the_oracle_and_allocates_nothing():
    jfa.build()
    fn = _entry()
    p = parity.to_cuda(workloads.make_problem(6, 3, 128, "broadcast", [5, 0, 128, 129, 1000, 300],
                                              Lq=200, seed=41))
    plan = parity.make_plan(p)
    out, lse, _ = parity.gpu_fwd(p, plan)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = _call(fn, p, out, lse, status)  # sets up the scratch address for this device
    assert status.item() == 0
    parity.check_grads(*first, *parity.oracle_bwd(p))
    # a second call, with its outputs already allocated, must leave the
    # device's free memory unchanged: nothing is allocated on its behalf
    g = _outputs(p)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    rc = _launch(fn, p, out, lse, status, g)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert rc == 0 and status.item() == 0
    assert free_after == free_before, (free_before, free_after)
    for x, n in zip(g, ("dQ", "dK", "dV")):
        x.check(n)
    parity.check_grads(*(x.t for x in g), *parity.oracle_bwd(p))


def test_noalloc_needs_no_delta_scratch_when_full_tiles_form_it():
    jfa.build()
    fn = _entry()
    # 2^19 rows x 16 heads of Delta would fill the whole 32 MiB array, but with
    # 128-token sequences every tile is full and forms its own Delta, so only
    # the schedule and offsets need room
    p = parity.to_cuda(workloads.make_problem(4096, 16, 64, "self", [128] * 4096, seed=34,
                                              device="cuda"))
    plan = parity.make_plan(p)
    out, lse, _ = parity.gpu_fwd(p, plan)
    ref = parity.gpu_bwd(p, out, lse, plan)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _call(fn, p, out, lse, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for g, r in zip(got, ref):  # compared on the device: 2^19 x 16 x 64 values each
        assert torch.isfinite(g).all()
        assert ((g.float() - r.float()).norm() / r.float().norm()).item() <= 1e-6
    del p, plan, out, lse, ref, got
    torch.cuda.empty_cache()


def test_noalloc_rejects_problems_beyond_its_scratch():
    jfa.build()
    fn = _entry()
    # 2^20 broadcast rows x 16 heads of Delta (64 MiB) cannot fit the 32 MiB
    # array: the call must refuse before launching anything.  The sequence has
    # 129 keys, two key blocks, so Delta needs the scratch (with one key block
    # the tiles would form it and the call would go ahead).  Every buffer has
    # the full size the arguments describe (about 10 GiB in all), so that the
    # call stays within bounds even if the check were ever to let it through.
    Lq, H, D, nk = 1 << 20, 16, 64, 129
    q = torch.zeros((Lq, H, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((nk, H, D), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    out = torch.zeros((Lq, H, D), dtype=torch.bfloat16, device="cuda")
    dout = torch.zeros_like(out)
    lse = torch.zeros((H, Lq), dtype=torch.float32, device="cuda")
    dq = torch.zeros((Lq, H, D), dtype=torch.float32, device="cuda")
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(k)
    kv = jfa._offsets([0, nk])
    rc = fn(jfa._i32ptr(kv), None, 1, H, Lq, D, q.data_ptr(), k.data_ptr(), v.data_ptr(),
            out.data_ptr(), dout.data_ptr(), lse.data_ptr(), 0.125, dq.data_ptr(), dk.data_ptr(),
            dv.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 5  # JFA_ERR_WORKSPACE
    del q, k, v, out, dout, lse, dq, dk, dv
    torch.cuda.empty_cache()
