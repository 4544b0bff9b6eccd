"""Reference tile schedules -- TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

A plain restatement of how the jagged FlashAttention pages hand work to
persistent CTAs, written independently of the C++ planner in the library:

* forward (alphasignal page, "Five changes unlocked the gains", item 1, and
  the yuxiaoba note, "Why both static and dynamic balancing help"): the host
  sorts (batch, head, query-block) tiles by their key/value workload and deals
  them to the SMs back and forth (boustrophedon / zigzag);
* backward (yuxiaoba note, same section; asivanadi0 blog, "Structural changes
  and layered opts", item 1): the host precomputes the valid (batch, head,
  key/value-block) tiles and assigns them round-robin.

Readings where the pages leave the details open:

* enumeration order is batch outer, then head, then block;
* a forward tile's cost is ceil(Lk_b / BN), the number of key/value blocks it
  visits; tiles of sequences with no keys (cost 0) are kept, because they must
  still write O = 0 and LSE = -inf;
* the sort is stable and by cost descending;
* with P = min(num_ctas, T), sorted tile i goes to round r = i // P at position
  k = i % P, and to CTA k when r is even, CTA P-1-k when r is odd;
* backward tiles exist only where the sequence has queries; tile i goes to CTA
  i % P; its cost field holds ceil(Lq_b / BM), the query blocks it visits;
* each CTA runs its tiles in round order.

Every tile is four int32: (b, h, blk, cost).  The result is CSR: ``tiles``
[T, 4] grouped by CTA and ``cta_ptr`` [P + 1].
"""
from __future__ import annotations

import numpy as np


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def fwd_tiles(q_lengths, kv_lengths, H: int, BM: int, BN: int, num_ctas: int):
    tiles = []
    for b in range(len(q_lengths)):
        cost = _ceil_div(int(kv_lengths[b]), BN)
        for h in range(H):
            for m in range(_ceil_div(int(q_lengths[b]), BM)):
                tiles.append((b, h, m, cost))
    order = sorted(range(len(tiles)), key=lambda i: -tiles[i][3])  # sorted() is stable
    T = len(tiles)
    P = min(num_ctas, T)
    per_cta = [[] for _ in range(P)]
    for i, t in enumerate(order):
        r, k = divmod(i, P)
        cta = k if r % 2 == 0 else P - 1 - k
        per_cta[cta].append(tiles[t])
    return _csr(per_cta, P)


def bwd_tiles(q_lengths, kv_lengths, H: int, BM: int, BN: int, num_ctas: int):
    tiles = []
    for b in range(len(q_lengths)):
        if int(q_lengths[b]) == 0:
            continue
        qblocks = _ceil_div(int(q_lengths[b]), BM)
        for h in range(H):
            for n in range(_ceil_div(int(kv_lengths[b]), BN)):
                tiles.append((b, h, n, qblocks))
    T = len(tiles)
    P = min(num_ctas, T)
    per_cta = [[] for _ in range(P)]
    for i, t in enumerate(tiles):
        per_cta[i % P].append(t)
    return _csr(per_cta, P)


def _csr(per_cta, P):
    ptr = np.zeros(P + 1, dtype=np.int32)
    for c in range(P):
        ptr[c + 1] = ptr[c] + len(per_cta[c])
    flat = [t for lst in per_cta for t in lst]
    tiles = np.asarray(flat, dtype=np.int32).reshape(-1, 4)
    return tiles, ptr
