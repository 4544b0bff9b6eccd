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

Optional packing of short sequences (the block-diagonal case of the TLX Block
Attention page, "One Constraint, Five Eliminations": a 64-token segment only
attends within itself), for self mode with one shared offsets array: scanning
b upward, a sequence of length 1..128 starts a run that greedily takes the
following sequences while the run's total stays within 128 rows; a run with
at least two non-empty sequences becomes one tile (b0, h, -nseq, 1) per head
and replaces those sequences' own tiles (forward cost 1, backward 1 query
block); other sequences keep their ordinary tiles.
"""
from __future__ import annotations

import numpy as np


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def short_packs(lengths, limit: int = 128):
    """pack[b]: run length for a run starting at b, 0 inside a run, 1 otherwise."""
    B = len(lengths)
    pack = [1] * B
    b = 0
    while b < B:
        L = int(lengths[b])
        if L == 0 or L > limit:
            b += 1
            continue
        total, e, nonempty = L, b + 1, 1
        while e < B and total + int(lengths[e]) <= limit:
            total += int(lengths[e])
            nonempty += int(lengths[e]) > 0
            e += 1
        if nonempty >= 2:
            pack[b] = e - b
            for i in range(b + 1, e):
                pack[i] = 0
            b = e
        else:
            b += 1
    return pack


def fwd_tiles(q_lengths, kv_lengths, H: int, BM: int, BN: int, num_ctas: int, pack=None, dynamic=False):
    tiles = []
    for b in range(len(q_lengths)):
        if pack is not None and pack[b] != 1:
            if pack[b] >= 2:
                tiles.extend((b, h, -pack[b], 1) for h in range(H))
            continue
        cost = _ceil_div(int(kv_lengths[b]), BN)
        for h in range(H):
            for m in range(_ceil_div(int(q_lengths[b]), BM)):
                tiles.append((b, h, m, cost))
    if dynamic:
        return claim_order(tiles, num_ctas)
    order = sorted(range(len(tiles)), key=lambda i: -tiles[i][3])  # sorted() is stable
    T = len(tiles)
    P = min(num_ctas, T)
    per_cta = [[] for _ in range(P)]
    for i, t in enumerate(order):
        r, k = divmod(i, P)
        cta = k if r % 2 == 0 else P - 1 - k
        per_cta[cta].append(tiles[t])
    return _csr(per_cta, P)


def claim_order(tiles, num_ctas: int):
    """Dynamic schedules: every tile once, stably sorted by its last field
    (cost) descending, one queue for all P = min(num_ctas, T) CTAs:
    cta_ptr = [0, T, ..., T]."""
    order = sorted(range(len(tiles)), key=lambda i: -tiles[i][3])  # sorted() is stable
    T = len(tiles)
    P = min(num_ctas, T)
    flat = np.asarray([tiles[i] for i in order], dtype=np.int32).reshape(-1, 4)
    ptr = np.full(P + 1, T, dtype=np.int32)
    ptr[0] = 0
    return flat, ptr


def bwd_tiles(q_lengths, kv_lengths, H: int, BM: int, BN: int, num_ctas: int, pack=None, dynamic=False):
    tiles = []
    for b in range(len(q_lengths)):
        if pack is not None and pack[b] != 1:
            if pack[b] >= 2:
                tiles.extend((b, h, -pack[b], 1) for h in range(H))
            continue
        if int(q_lengths[b]) == 0:
            continue
        qblocks = _ceil_div(int(q_lengths[b]), BM)
        for h in range(H):
            for n in range(_ceil_div(int(kv_lengths[b]), BN)):
                tiles.append((b, h, n, qblocks))
    if dynamic:
        return claim_order(tiles, num_ctas)
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
