"""The reference tile builder (oracle/tiles.py) against hand-worked schedules
and brute-force properties."""
import numpy as np
import pytest

from oracle import tiles
from tests.tiles_golden import load_cases

BM = BN = 128


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_reference_builder_matches_hand_worked(case):
    flags = case.get("flags", 0)
    pack = tiles.short_packs(case["kv_lengths"]) if flags & 1 else None
    dyn = bool(flags & 2)
    ft, fp = tiles.fwd_tiles(case["q_lengths"], case["kv_lengths"], case["H"], BM, BN, case["num_ctas"], pack, dyn)
    bt, bp = tiles.bwd_tiles(case["q_lengths"], case["kv_lengths"], case["H"], BM, BN, case["num_ctas"], pack, dyn)
    assert np.array_equal(fp, case["fwd_cta_ptr"]) and np.array_equal(ft, case["fwd"])
    assert np.array_equal(bp, case["bwd_cta_ptr"]) and np.array_equal(bt, case["bwd"])


def _cdiv(a, b):
    return -(-a // b)


@pytest.mark.parametrize("seed", range(6))
def test_schedule_properties(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    H = int(rng.integers(1, 5))
    klen = rng.integers(0, 700, size=B)
    klen[rng.random(B) < 0.2] = 0
    qlen = rng.integers(0, 400, size=B) if seed % 2 else klen.copy()
    P_req = int(rng.integers(1, 60))

    ft, fp = tiles.fwd_tiles(qlen, klen, H, BM, BN, P_req)
    want = {(b, h, m) for b in range(B) for h in range(H) for m in range(_cdiv(int(qlen[b]), BM))}
    got = [tuple(t[:3]) for t in ft]
    assert len(got) == len(set(got)) and set(got) == want          # every tile exactly once
    for t in ft:
        assert t[3] == _cdiv(int(klen[t[0]]), BN)
    P = len(fp) - 1
    assert P == min(P_req, len(want))
    if P:
        loads = [int(ft[fp[c]:fp[c + 1], 3].sum()) for c in range(P)]
        assert max(loads) - min(loads) <= int(ft[:, 3].max())         # balanced within one tile
        # within each CTA, costs never increase from round to round
        for c in range(P):
            cs = ft[fp[c]:fp[c + 1], 3]
            assert np.all(np.diff(cs) <= 0)

    bt, bp = tiles.bwd_tiles(qlen, klen, H, BM, BN, P_req)
    want = {(b, h, n) for b in range(B) if qlen[b] > 0 for h in range(H)
            for n in range(_cdiv(int(klen[b]), BN))}
    got = [tuple(t[:3]) for t in bt]
    assert len(got) == len(set(got)) and set(got) == want
    P = len(bp) - 1
    if P:
        counts = np.diff(bp)
        assert counts.max() - counts.min() <= 1                       # round-robin by count


def test_empty_problem():
    ft, fp = tiles.fwd_tiles([0, 0], [5, 0], 2, BM, BN, 8)
    assert ft.shape == (0, 4) and list(fp) == [0]


@pytest.mark.parametrize("seed", range(6))
def test_packed_schedule_properties(seed):
    rng = np.random.default_rng(50 + seed)
    B = int(rng.integers(1, 60))
    lens = rng.integers(0, 150, size=B)
    lens[rng.random(B) < 0.2] = 0
    pack = tiles.short_packs(lens)
    # packs cover consecutive sequences, fit one tile and hold >= 2 non-empty sequences
    covered = set()
    for b, n in enumerate(pack):
        if n >= 2:
            assert sum(int(x) for x in lens[b:b + n]) <= 128
            assert sum(int(x) > 0 for x in lens[b:b + n]) >= 2
            assert all(pack[i] == 0 for i in range(b + 1, b + n))
            covered.update(range(b, b + n))
        elif n == 0:
            assert b in covered
    ft, fp = tiles.fwd_tiles(lens, lens, 2, BM, BN, 7, pack)
    rows = {}
    for b, h, blk, cost in ft:
        if blk < 0:
            seqs = range(b, b - blk)
        else:
            seqs = [b]
        for s in seqs:
            rows.setdefault((s, h), 0)
            rows[(s, h)] += 1 if blk < 0 else 0
    # every non-empty sequence is either packed once per head or tiled normally
    for b in range(B):
        if lens[b] == 0:
            continue
        for h in range(2):
            if b in covered:
                assert rows[(b, h)] == 1
