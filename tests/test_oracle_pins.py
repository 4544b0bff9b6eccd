"""Pins for the fp64 oracle, checked against things other than itself.

* central finite differences of the oracle's own forward (pins the backward
  formulas to the forward definition);
* a padded-dense-with-mask recomputation with torch softmax / logsumexp and
  autograd (pins the forward and the gradients to library routines);
* torch's scaled_dot_product_attention on dense equal-length batches;
* closed forms: length-1 sequences give O = V and LSE = scale q.k; identical
  keys give O = mean(V) and LSE = scale q.k + ln L;
* invariants: rows of P sum to one, sum_j dV_j = sum_i dO_i, sum_j dK_j = 0,
  broadcast dQ equals the sum of per-sequence self-mode dQs, block-diagonal
  offsets equal independent per-block attention, and the row sum
  sum_d dO_id O_id equals sum_j P_ij dP_ij (O = P V, dP = dO V^T).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.torch_ref import padded_reference

ORC = oracle.default()


def _run(orc, p):
    O, L = orc.fwd(p.q, p.k, p.v, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq, p.D, p.scale)
    dq, dk, dv = orc.bwd(p.q, p.k, p.v, p.dout, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq, p.D,
                         p.scale)
    return O, L, dq, dk, dv


def _cases():
    return [
        workloads.make_problem(4, 2, 8, "self", [3, 0, 5, 1], seed=1),
        workloads.make_problem(3, 3, 16, "broadcast", [2, 7, 0], Lq=5, seed=2),
        workloads.make_problem(3, 2, 8, "self", [4, 3, 6], q_lengths=[2, 0, 5], seed=3),
        workloads.make_problem(2, 1, 64, "self", [33, 17], seed=4),
    ]


def torch_reference_errors(orc, p):
    O, L, dq, dk, dv = _run(orc, p)
    rO, rL, rdq, rdk, rdv = padded_reference(p.q, p.k, p.v, p.dout, p.kv_offsets, p.q_offsets,
                                             p.B, p.H, p.Lq, p.D, p.scale)
    fin = torch.isfinite(rL)
    assert torch.equal(fin, torch.isfinite(L)), "LSE -inf pattern differs"
    return {
        "O": (O - rO).abs().max().item(),
        "LSE": (L[fin] - rL[fin]).abs().max().item() if fin.any() else 0.0,
        "dQ": (dq - rdq).abs().max().item(),
        "dK": (dk - rdk).abs().max().item(),
        "dV": (dv - rdv).abs().max().item(),
    }


def finite_difference_errors(orc, p, eps=1e-6):
    """max |analytic - central FD| over every input element for loss = sum(O * dO)."""
    q, k, v, g = (t.double() for t in (p.q, p.k, p.v, p.dout))

    def loss(q_, k_, v_):
        O, _ = orc.fwd(q_, k_, v_, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq, p.D, p.scale)
        return float((O * g).sum())

    dq, dk, dv = orc.bwd(q, k, v, g, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq, p.D, p.scale)
    errs = {}
    for name, t, grad in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
        worst = 0.0
        flat = t.view(-1)
        for i in range(flat.numel()):
            old = flat[i].item()
            flat[i] = old + eps
            args = [q, k, v]
            lp = loss(*args)
            flat[i] = old - eps
            lm = loss(*args)
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            worst = max(worst, abs(fd - grad.view(-1)[i].item()))
        errs[name] = worst
    return errs


@pytest.mark.parametrize("case", range(4))
def test_matches_padded_masked_torch(case):
    p = _cases()[case]
    errs = torch_reference_errors(ORC, p)
    for k, e in errs.items():
        assert e < 1e-11, (k, e)


def test_finite_differences():
    p = workloads.make_problem(3, 2, 4, "self", [1, 4, 5], seed=5)
    errs = finite_difference_errors(ORC, p)
    for k, e in errs.items():
        assert e < 1e-7, (k, e)
    pb = workloads.make_problem(2, 1, 4, "broadcast", [3, 2], Lq=3, seed=6)
    errs = finite_difference_errors(ORC, pb)
    for k, e in errs.items():
        assert e < 1e-7, (k, e)


def test_dense_equals_sdpa():
    B, H, L, D = 3, 2, 9, 16
    p = workloads.make_problem(B, H, D, "self", [L] * B, seed=7)
    O, L_, dq, dk, dv = _run(ORC, p)
    q = p.q.double().view(B, L, H, D).permute(0, 2, 1, 3).clone().requires_grad_(True)
    k = p.k.double().view(B, L, H, D).permute(0, 2, 1, 3).clone().requires_grad_(True)
    v = p.v.double().view(B, L, H, D).permute(0, 2, 1, 3).clone().requires_grad_(True)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=p.scale)
    g = p.dout.double().view(B, L, H, D).permute(0, 2, 1, 3)
    (ref * g).sum().backward()
    back = lambda t: t.permute(0, 2, 1, 3).reshape(B * L, H, D)
    assert (back(ref.detach()) - O).abs().max() < 1e-12
    assert (back(q.grad) - dq).abs().max() < 1e-12
    assert (back(k.grad) - dk).abs().max() < 1e-12
    assert (back(v.grad) - dv).abs().max() < 1e-12


def test_length_one_sequences():
    p = workloads.make_problem(5, 2, 32, "self", [1] * 5, seed=8)
    O, L, dq, dk, dv = _run(ORC, p)
    q, k, v, g = (t.double() for t in (p.q, p.k, p.v, p.dout))
    assert torch.equal(O, v)                                       # O = V exactly
    lse_ref = p.scale * (q * k).sum(-1).T                           # [H, rows]
    assert (L - lse_ref).abs().max() < 1e-13
    assert dk.abs().max() == 0.0 and dq.abs().max() == 0.0         # dS = 0 exactly
    assert torch.equal(dv, g)                                      # dV = dO


def test_identical_keys():
    n = 7
    p = workloads.make_problem(2, 2, 16, "self", [n, 3], seed=9)
    k = p.k.clone()
    k[0:n] = k[0:1]            # every key of sequence 0 equals its first key
    p.k = k
    O, L, *_ = _run(ORC, p)
    v = p.v.double()
    q = p.q.double()
    mean_v = v[0:n].mean(0)                                          # [H, D]
    assert (O[0:n] - mean_v[None]).abs().max() < 1e-12
    lse_ref = p.scale * (q[0:n] * k.double()[0:1]).sum(-1).T + math.log(n)
    assert (L[:, 0:n] - lse_ref).abs().max() < 1e-12


def test_softmax_rows_sum_to_one():
    p = workloads.make_problem(3, 2, 16, "self", [6, 1, 9], seed=10)
    p.v = torch.ones_like(p.v)
    O, *_ = _run(ORC, p)
    assert (O - 1).abs().max() < 1e-13


def test_gradient_invariants():
    lens = [5, 9, 1, 12]
    p = workloads.make_problem(4, 3, 8, "self", lens, seed=11)
    _, _, dq, dk, dv = _run(ORC, p)
    off = p.kv_offsets
    g = p.dout.double()
    for b in range(4):
        s, e = int(off[b]), int(off[b + 1])
        assert (dv[s:e].sum(0) - g[s:e].sum(0)).abs().max() < 1e-12   # sum_j dV_j = sum_i dO_i
        assert dk[s:e].sum(0).abs().max() < 1e-12                    # sum_j dK_j = 0


def test_row_sum_equals_p_times_dp():
    # rowsum(dO * O) over the oracle's O equals sum_j P_ij (dO V^T)_ij with P
    # rebuilt from the oracle's LSE: the identity that lets a backward tile
    # holding every key of its queries form the row sum without reading O
    # (and a check that the oracle's O and LSE describe the same P)
    g = torch.Generator().manual_seed(12)
    for nq, nk, D in ((7, 5, 8), (1, 1, 4), (33, 70, 16), (4, 128, 64)):
        q, dout = (torch.randn(nq, D, generator=g, dtype=torch.float64) for _ in range(2))
        k, v = (torch.randn(nk, D, generator=g, dtype=torch.float64) for _ in range(2))
        scale = 1.0 / math.sqrt(D)
        O, L = ORC.seq_fwd(q, k, v, scale)
        P = torch.exp(scale * (q @ k.T) - L[:, None])
        lhs = (dout * O).sum(1)
        rhs = (P * (dout @ v.T)).sum(1)
        assert torch.allclose(lhs, rhs, rtol=1e-12, atol=1e-12), (nq, nk, D)


def test_broadcast_equals_sum_of_self_mode():
    B, H, D, Lq = 3, 2, 16, 6
    klens = [4, 9, 2]
    pb = workloads.make_problem(B, H, D, "broadcast", klens, Lq=Lq, seed=12)
    Ob, Lb, dqb, dkb, dvb = _run(ORC, pb)
    # the same problem in self mode with Q replicated once per sequence
    qrep = pb.q.repeat(B, 1, 1)
    ps = workloads.Problem(B, H, D, "self", 0, pb.kv_offsets,
                           workloads.offsets_from_lengths([Lq] * B), qrep, pb.k, pb.v, pb.dout,
                           pb.scale)
    Os, Ls, dqs, dks, dvs = _run(ORC, ps)
    assert (Ob - Os).abs().max() < 1e-13 and (Lb - Ls).abs().max() < 1e-13
    assert (dkb - dks).abs().max() < 1e-13 and (dvb - dvs).abs().max() < 1e-13
    dq_sum = dqs.view(B, Lq, H, D).sum(0)
    assert (dqb - dq_sum).abs().max() < 1e-12


def test_block_diagonal_equals_per_block_attention():
    nblk, blk, H, D = 6, 64, 2, 32
    p = workloads.make_problem(nblk, H, D, "self", [blk] * nblk, seed=13)
    O, L, dq, dk, dv = _run(ORC, p)
    for b in range(nblk):
        s = slice(b * blk, (b + 1) * blk)
        for h in range(H):
            q = p.q[s, h].double().clone().requires_grad_(True)
            k = p.k[s, h].double().clone().requires_grad_(True)
            v = p.v[s, h].double().clone().requires_grad_(True)
            ref = torch.softmax(p.scale * q @ k.T, -1) @ v
            (ref * p.dout[s, h].double()).sum().backward()
            assert (ref.detach() - O[s, h]).abs().max() < 1e-12
            assert (q.grad - dq[s, h]).abs().max() < 1e-12
            assert (k.grad - dk[s, h]).abs().max() < 1e-12


def test_dq_rows_and_seq_entry_points_agree_with_full():
    for p in _cases()[:3]:
        O, L, dq, dk, dv = _run(ORC, p)
        nrows = p.n_q_rows
        rows = np.arange(nrows)
        for h in range(p.H):
            got = ORC.dq_rows(p.q, p.k, p.v, p.dout, p.kv_offsets, p.q_offsets, p.B, p.H, p.Lq,
                              p.D, p.scale, h, rows)
            assert (got - dq[:, h]).abs().max() < 1e-12
        # per-(sequence, head) entry points on sequence 0, head 0
        b, h = 0, 0
        ko = p.kv_offsets
        ks = slice(int(ko[0]), int(ko[1]))
        if p.mode == "broadcast":
            qs, os_ = slice(0, p.Lq), slice(0, p.Lq)
        else:
            qs = os_ = slice(int(p.q_offsets[0]), int(p.q_offsets[1]))
        so, sl = ORC.seq_fwd(p.q[qs, h], p.k[ks, h], p.v[ks, h], p.scale)
        assert (so - O[os_, h]).abs().max() < 1e-13
        fin = torch.isfinite(sl)
        assert torch.equal(fin, torch.isfinite(L[h, os_]))
        sdq, sdk, sdv = ORC.seq_bwd(p.q[qs, h], p.k[ks, h], p.v[ks, h], p.dout[os_, h], p.scale)
        assert (sdk - dk[ks, h]).abs().max() < 1e-13
        assert (sdv - dv[ks, h]).abs().max() < 1e-13


def test_empty_sequences():
    p = workloads.make_problem(3, 2, 8, "self", [0, 4, 0], seed=14)
    O, L, dq, dk, dv = _run(ORC, p)
    assert O.shape[0] == 4 and L.shape == (2, 4)
    pb = workloads.make_problem(3, 2, 8, "broadcast", [0, 4, 0], Lq=3, seed=15)
    O, L, dq, dk, dv = _run(ORC, pb)
    assert O[0:3].abs().max() == 0 and O[6:9].abs().max() == 0
    assert torch.isinf(L[:, 0:3]).all() and (L[:, 0:3] < 0).all()
    assert torch.isfinite(L[:, 3:6]).all()


def test_rejects_bad_offsets():
    with pytest.raises(ValueError):
        ORC.fwd(torch.zeros(3, 1, 4), torch.zeros(3, 1, 4), torch.zeros(3, 1, 4),
                np.array([0, 2, 1, 3]), None, 3, 1, 1, 4, 0.5)
