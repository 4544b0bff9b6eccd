"""Full-size parity, element by element: the GEM-like broadcast, skewed
broadcast and block-diagonal workloads at their full sizes, run in the launch
configuration bench.py times (one persistent CTA per SM), against the fp64
oracle on every output element.

The oracle runs over the batch in chunks of whole sequences (a few hundred
thousand key rows at a time, so its fp64 copies stay a few GB); each chunk's
O, LSE, dK and dV are compared with the GPU's rows of the same sequences, and
in broadcast mode the chunks' dQ are summed into the one batch-wide dQ the
GPU reduces.  Each workload runs its plan variants (schedule flags) on the
GPU first, and the oracle pass checks all of them.

Bounds (bf16 inputs and outputs, fp32 accumulation):
* O: max-abs error <= 1e-2 over every element; LSE: max-abs <= 1e-3;
* dQ, dK, dV: relative L2 <= 1e-2 over the whole tensor;
* and, so that an error confined to a few tiles cannot hide in the whole
  tensor's norm, relative L2 <= 2e-2 for every (sequence, head) block of dK,
  dV (and of dQ in self mode), its denominator floored at 1e-3 of the
  blocks' RMS norm so that blocks whose exact gradient vanishes (a one-key
  sequence has dK = 0) are held to an absolute bound instead.
Every output is NaN-prefilled and guard-banded (tests/parity.py).
"""
import numpy as np
import pytest
import torch

import jagged_attention_gb300 as jfa
import oracle
import workloads
from tests import parity

pytestmark = pytest.mark.gpu

VARIANTS = {
    # the default (two query tiles per CTA), one tile per CTA, claimed tiles
    "gem_broadcast": [0, jfa.PLAN_FWD_ONE, jfa.PLAN_DYNAMIC],
    "skewed_broadcast": [0, jfa.PLAN_FWD_ONE],
    # unpacked, the default (packed, backward tiles claimed at run time), the
    # same with both passes dealt on the host, both passes claimed
    "block_diag": [jfa.PLAN_NO_PACK, 0, jfa.PLAN_STATIC, jfa.PLAN_DYNAMIC],
}
CHUNK_KV_ROWS = 1 << 17
LOCAL_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    jfa.build()


def _chunks(kvo: np.ndarray, max_rows: int):
    """Sequence ranges [b, e) holding at most max_rows key rows (at least one sequence)."""
    B = kvo.size - 1
    b = 0
    while b < B:
        e = b + 1
        while e < B and kvo[e + 1] - kvo[b] <= max_rows:
            e += 1
        yield b, e
        b = e


def _blocks(got: np.ndarray, ref: np.ndarray, offsets: np.ndarray):
    """Squared error and squared reference norm per (non-empty sequence, head)."""
    err2 = ((got - ref) ** 2).sum(axis=2)
    ref2 = (ref ** 2).sum(axis=2)
    starts = offsets[:-1][np.diff(offsets) > 0]
    if starts.size == 0:
        return np.zeros((0, got.shape[1])), np.zeros((0, got.shape[1]))
    return np.add.reduceat(err2, starts, axis=0), np.add.reduceat(ref2, starts, axis=0)


class _Tally:
    """Running whole-tensor and per-block error statistics of one gradient."""

    def __init__(self):
        self.err2 = 0.0
        self.ref2 = 0.0
        self.blocks_e, self.blocks_r = [], []

    def add(self, got, ref, offsets):
        g = got.astype(np.float64)
        self.err2 += float(((g - ref) ** 2).sum())
        self.ref2 += float((ref ** 2).sum())
        e, r = _blocks(g, ref, offsets)
        self.blocks_e.append(e)
        self.blocks_r.append(r)

    def check(self, name):
        rel = np.sqrt(self.err2 / self.ref2) if self.ref2 > 0 else np.sqrt(self.err2)
        assert rel <= parity.TOL_GRAD, f"{name}: whole-tensor relative L2 {rel:.3e}"
        e = np.concatenate(self.blocks_e)
        r = np.concatenate(self.blocks_r)
        if e.size:
            floor = 1e-3 * np.sqrt(r.mean())
            local = np.sqrt(e) / np.maximum(np.sqrt(r), floor)
            worst = np.unravel_index(np.argmax(local), local.shape)
            assert local.max() <= LOCAL_TOL, (
                f"{name}: (sequence, head) block {worst} relative L2 {local.max():.3e}")
        return rel


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_full_size_every_element(name):
    torch.cuda.empty_cache()
    orc = oracle.default()
    p = workloads.make_workload(name, seed=0, device="cuda")
    runs = {}
    for flags in VARIANTS[name]:
        plan = parity.make_plan(p, flags=flags)  # num_ctas = SM count, as bench.py runs it
        out, lse, _ = parity.gpu_fwd(p, plan)
        dq, dk, dv = parity.gpu_bwd(p, out, lse, plan)
        runs[flags] = (out, lse, dq, dk, dv)
        plan.close()

    kvo = p.kv_offsets.astype(np.int64)
    qo = None if p.q_offsets is None else p.q_offsets.astype(np.int64)
    H, D, Lq = p.H, p.D, p.Lq
    o_err = {f: 0.0 for f in runs}
    l_err = {f: 0.0 for f in runs}
    tallies = {f: {g: _Tally() for g in ("dK", "dV", "dQ")} for f in runs}
    dq_sum = np.zeros((Lq, H, D)) if p.mode == "broadcast" else None
    for b, e in _chunks(kvo, CHUNK_KV_ROWS):
        ks, ke = int(kvo[b]), int(kvo[e])
        kv_sub = kvo[b:e + 1] - kvo[b]
        k, v = p.k[ks:ke].cpu(), p.v[ks:ke].cpu()
        if p.mode == "broadcast":
            q, q_sub, qs, qe = p.q.cpu(), None, 0, Lq
            os_, oe = b * Lq, e * Lq
        else:
            qs, qe = int(qo[b]), int(qo[e])
            q_sub = qo[b:e + 1] - qo[b]
            q = p.q[qs:qe].cpu()
            os_, oe = qs, qe
        dout = p.dout[os_:oe].cpu()
        O_ref, L_ref = orc.fwd(q, k, v, kv_sub, q_sub, e - b, H, Lq, D, p.scale)
        dq_ref, dk_ref, dv_ref = orc.bwd(q, k, v, dout, kv_sub, q_sub, e - b, H, Lq, D, p.scale)
        O_ref, L_ref = O_ref.numpy(), L_ref.numpy()
        dq_ref, dk_ref, dv_ref = dq_ref.numpy(), dk_ref.numpy(), dv_ref.numpy()
        if dq_sum is not None:
            dq_sum += dq_ref
        fin = np.isfinite(L_ref)
        for f, (out, lse, dq, dk, dv) in runs.items():
            O = out[os_:oe].cpu().double().numpy()
            L = lse[:, os_:oe].cpu().double().numpy()
            assert np.isfinite(O).all(), f"flags {f}: O has unwritten or non-finite entries"
            assert np.array_equal(np.isfinite(L), fin), f"flags {f}: LSE finite pattern differs"
            if O.size:
                o_err[f] = max(o_err[f], float(np.abs(O - O_ref).max()))
            if fin.any():
                l_err[f] = max(l_err[f], float(np.abs(L[fin] - L_ref[fin]).max()))
            t = tallies[f]
            t["dK"].add(dk[ks:ke].cpu().double().numpy(), dk_ref, kv_sub)
            t["dV"].add(dv[ks:ke].cpu().double().numpy(), dv_ref, kv_sub)
            if p.mode == "self":
                t["dQ"].add(dq[qs:qe].cpu().double().numpy(), dq_ref, q_sub)
    for f, (out, lse, dq, dk, dv) in runs.items():
        assert o_err[f] <= parity.TOL_O, f"flags {f}: O max-abs error {o_err[f]:.3e}"
        assert l_err[f] <= parity.TOL_LSE, f"flags {f}: LSE max-abs error {l_err[f]:.3e}"
        if dq_sum is not None:  # the batch-summed dQ, and each head of it
            tallies[f]["dQ"].add(dq.cpu().double().numpy(), dq_sum, np.array([0, Lq]))
        for g in ("dK", "dV", "dQ"):
            tallies[f][g].check(f"flags {f} {g}")
    del runs, p
    torch.cuda.empty_cache()
