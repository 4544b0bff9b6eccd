"""Independent fp64 checks used to pin the oracle (CPU only).

``padded_reference`` recomputes jagged attention the way a padded framework
would: pad every sequence to the longest one, mask the padded keys with -inf,
run torch's softmax / logsumexp on dense [B, H, Lq, Lk] scores and take the
gradients with autograd.  It shares nothing with ``oracle.c`` beyond the
definition both follow.
"""
from __future__ import annotations

import numpy as np
import torch


def padded_reference(q, k, v, dout, kv_offsets, q_offsets, B, H, Lq, D, scale):
    """Returns O [n_o,H,D], LSE [H,n_o], dQ, dK, dV (float64, packed layouts)."""
    kv_off = np.asarray(kv_offsets, dtype=np.int64)
    klen = np.diff(kv_off)
    if q_offsets is None:
        qlen = np.full(B, Lq, dtype=np.int64)
        q_off = None
    else:
        q_off = np.asarray(q_offsets, dtype=np.int64)
        qlen = np.diff(q_off)
    Lqm = max(1, int(qlen.max()) if B else 1)
    Lkm = max(1, int(klen.max()) if B else 1)

    q64 = q.detach().double().clone().requires_grad_(True)
    k64 = k.detach().double().clone().requires_grad_(True)
    v64 = v.detach().double().clone().requires_grad_(True)
    do64 = dout.detach().double()

    # index maps from padded positions to packed rows (-1 = padding)
    qidx = torch.full((B, Lqm), -1, dtype=torch.long)
    oidx = torch.full((B, Lqm), -1, dtype=torch.long)
    kidx = torch.full((B, Lkm), -1, dtype=torch.long)
    for b in range(B):
        nq, nk = int(qlen[b]), int(klen[b])
        q0 = 0 if q_off is None else int(q_off[b])
        o0 = b * Lq if q_off is None else int(q_off[b])
        qidx[b, :nq] = torch.arange(q0, q0 + nq)
        oidx[b, :nq] = torch.arange(o0, o0 + nq)
        kidx[b, :nk] = torch.arange(int(kv_off[b]), int(kv_off[b]) + nk)
    qmask = qidx >= 0
    kmask = kidx >= 0

    def gather(t, idx):  # packed [N,H,D] -> padded [B,H,L,D], zeros at padding
        g = t[idx.clamp(min=0)]                      # [B, L, H, D]
        g = g * (idx >= 0)[..., None, None].to(t.dtype)
        return g.permute(0, 2, 1, 3)

    Qp, Kp, Vp = gather(q64, qidx), gather(k64, kidx), gather(v64, kidx)
    S = scale * Qp @ Kp.transpose(-1, -2)            # [B,H,Lqm,Lkm]
    S = S.masked_fill(~kmask[:, None, None, :], float("-inf"))
    has_keys = torch.as_tensor(klen > 0)[:, None, None, None]
    S_safe = torch.where(has_keys, S, torch.zeros_like(S))
    P = torch.softmax(S_safe, dim=-1) * has_keys
    Op = P @ Vp                                      # [B,H,Lqm,D]
    lse_p = torch.where(has_keys[..., 0], torch.logsumexp(S_safe, dim=-1),
                        torch.full_like(S_safe[..., 0], float("-inf")))

    dOp = gather(do64, oidx)
    (Op * dOp).sum().backward()

    n_o = B * Lq if q_off is None else int(q_off[-1])
    O = torch.zeros(n_o, H, D, dtype=torch.float64)
    LSE = torch.zeros(H, n_o, dtype=torch.float64)
    Od = Op.detach().permute(0, 2, 1, 3)              # [B,Lqm,H,D]
    for b in range(B):
        nq = int(qlen[b])
        rows = oidx[b, :nq]
        O[rows] = Od[b, :nq]
        LSE[:, rows] = lse_p.detach()[b, :, :nq]
    return O, LSE, q64.grad, k64.grad, v64.grad
