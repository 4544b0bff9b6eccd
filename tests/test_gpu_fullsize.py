"""Full-size parity: the GEM-like broadcast, skewed broadcast and
block-diagonal workloads at their full sizes, run in the launch configuration
bench.py times (one persistent CTA per SM), checked against the fp64 oracle
on sampled outputs it computes one by one:

* every output row written and finite (outputs are NaN-prefilled);
* O and LSE of sampled (sequence, head) pairs: the shortest, the longest and
  random sequences;
* dK and dV of the same pairs (the oracle's per-sequence backward);
* dQ: broadcast mode sums over every sequence, so sampled query rows are
  recomputed row by row over the whole batch of one head; self mode takes the
  sampled sequences' rows.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import jagged_attention_gb300 as jfa
    jfa.build()


def _sampled_sequences(p, rng, n_random=3):
    klen = p.kv_lengths
    nonempty = np.nonzero(klen > 0)[0]
    picks = {int(nonempty[np.argmin(klen[nonempty])]), int(np.argmax(klen))}
    picks.update(int(b) for b in rng.choice(nonempty, size=min(n_random, nonempty.size), replace=False))
    return sorted(picks)


@pytest.mark.parametrize("name,flags", [("gem_broadcast", 0), ("skewed_broadcast", 0),
                                        ("block_diag", 0), ("block_diag", 1),
                                        ("gem_broadcast", 2), ("block_diag", 3)])
def test_full_size_sampled_parity(name, flags):
    torch.cuda.empty_cache()
    orc = oracle.default()
    rng = np.random.default_rng(123)
    p = workloads.make_workload(name, seed=0, device="cuda")
    plan = parity.make_plan(p, flags=flags)  # num_ctas = SM count, as bench.py runs it
    out, lse, _ = parity.gpu_fwd(p, plan)
    dq, dk, dv = parity.gpu_bwd(p, out, lse, plan)

    assert torch.isfinite(out.float()).all(), "O has unwritten rows"
    assert not torch.isnan(lse).any(), "LSE has unwritten rows"
    for t, n in ((dq, "dQ"), (dk, "dK"), (dv, "dV")):
        assert torch.isfinite(t.float()).all(), f"{n} has unwritten or non-finite entries"

    kvo = p.kv_offsets.astype(np.int64)
    for b in _sampled_sequences(p, rng):
        h = int(rng.integers(p.H))
        ks, ke = int(kvo[b]), int(kvo[b + 1])
        if p.mode == "broadcast":
            qs, qe = 0, p.Lq
            os_, oe = b * p.Lq, (b + 1) * p.Lq
        else:
            qs, qe = int(p.q_offsets[b]), int(p.q_offsets[b + 1])
            os_, oe = qs, qe
        q = p.q[qs:qe, h].cpu()
        k = p.k[ks:ke, h].cpu()
        v = p.v[ks:ke, h].cpu()
        g = p.dout[os_:oe, h].cpu()
        O_ref, L_ref = orc.seq_fwd(q, k, v, p.scale)
        assert (out[os_:oe, h].cpu().double() - O_ref).abs().max().item() <= parity.TOL_O
        assert (lse[h, os_:oe].cpu().double() - L_ref).abs().max().item() <= parity.TOL_LSE
        dq_b, dk_ref, dv_ref = orc.seq_bwd(q, k, v, g, p.scale)
        assert parity.rel_l2(dk[ks:ke, h], dk_ref) <= parity.TOL_GRAD, ("dK", b, h)
        assert parity.rel_l2(dv[ks:ke, h], dv_ref) <= parity.TOL_GRAD, ("dV", b, h)
        if p.mode == "self":
            assert parity.rel_l2(dq[qs:qe, h], dq_b) <= parity.TOL_GRAD, ("dQ", b, h)

    if p.mode == "broadcast":
        # dQ rows summed over the whole batch for one head, recomputed row by row
        h = int(rng.integers(p.H))
        rows = np.array([0, 127, 128, p.Lq - 1] + list(rng.integers(0, p.Lq, size=2)))
        one = lambda t: t[:, h:h + 1].contiguous().cpu()
        ref = orc.dq_rows(one(p.q), one(p.k), one(p.v), one(p.dout), p.kv_offsets, None, p.B, 1,
                          p.Lq, p.D, p.scale, 0, rows)
        got = dq[torch.as_tensor(rows, device="cuda"), h]
        assert parity.rel_l2(got, ref) <= parity.TOL_GRAD, "dQ (batch-summed rows)"
    del out, lse, dq, dk, dv, p
    torch.cuda.empty_cache()
