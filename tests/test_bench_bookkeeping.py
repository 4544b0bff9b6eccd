"""The benchmark's bookkeeping (no GPU): the flop count it divides by, and its
host-side copies of the library's plan rules (which sequences are packed into
one tile, whether the backward tiles form Delta), checked against brute-force
counts and against the library's own host-only answers, so that a reported
TFLOP/s or byte figure cannot drift from what the kernels are given."""
import numpy as np
import pytest

import bench
import jagged_attention_gb300 as jfa
import workloads


@pytest.fixture(scope="module", autouse=True)
def _built():
    jfa.build()


def _problem(mode, kv_lengths, q_lengths=None, Lq=0, H=2, D=64):
    return workloads.make_problem(len(kv_lengths), H, D, mode, kv_lengths, Lq=Lq,
                                  q_lengths=q_lengths, seed=1)


def _pairs_by_counting(prob):
    # every (query row, key row) pair that meets, counted one at a time
    kv = prob.kv_offsets
    n = 0
    for b in range(prob.B):
        nq = prob.Lq if prob.q_offsets is None else int(prob.q_offsets[b + 1] - prob.q_offsets[b])
        for _ in range(nq):
            for _ in range(int(kv[b]), int(kv[b + 1])):
                n += 1
    return n


CASES = [
    ("broadcast", [5, 0, 130, 1, 64], None, 37),
    ("self", [3, 0, 129, 64, 1], None, 0),
    ("self", [10, 7, 0, 200], [0, 9, 4, 31], 0),   # cross: queries with their own lengths
]


@pytest.mark.parametrize("mode,kv,q,Lq", CASES)
def test_flops_count_every_query_key_pair(mode, kv, q, Lq):
    p = _problem(mode, kv, q, Lq)
    pairs = _pairs_by_counting(p)
    # forward: QK^T and PV, 2 D flops each per pair; backward: five products
    # of the same size (S^T, dP^T, dV, dK, dQ), S recomputed: 2.5 times that
    assert bench.pair_sum(p) == pairs
    assert bench.flops(p, "fwd") == 4.0 * p.D * p.H * pairs
    assert bench.flops(p, "bwd") == 10.0 * p.D * p.H * pairs


def _lengths(rng, B, hi, empty=0.1):
    x = rng.integers(1, hi + 1, size=B)
    x[rng.random(B) < empty] = 0
    return x.tolist()


def _runs_from_library(p, flags):
    # packed forward tiles are {b0, h, -nseq, 1}: the run [b0, b0 + nseq)
    tiles, _ = jfa.build_tiles(p.kv_offsets, p.q_offsets, H=1, Lq=p.Lq, num_ctas=4, direction=0,
                               flags=flags)
    return sorted((int(t[0]), int(t[0] - t[2])) for t in tiles if t[2] < 0)


@pytest.mark.parametrize("seed", range(8))
def test_packing_rule_matches_the_library(seed):
    rng = np.random.default_rng(seed)
    kv = _lengths(rng, 40, 100 if seed % 2 else 300)
    p = _problem("self", kv)
    for flags in (0, jfa.PLAN_PACK_SHORT, jfa.PLAN_NO_PACK):
        packed = jfa.plan_choices(p.kv_offsets, p.q_offsets, H=p.H, D=p.D, num_ctas=4,
                                  flags=flags)["packed"]
        runs = bench.packed_runs(p, packed)
        assert runs == _runs_from_library(p, flags), flags
        assert bool(runs) == bool(packed)


@pytest.mark.parametrize("seed", range(8))
def test_delta_rule_matches_the_library(seed):
    rng = np.random.default_rng(100 + seed)
    # mostly at most one key block per sequence (the rule's precondition), and
    # short enough that the tile fill crosses the 96-row threshold both ways
    kv = _lengths(rng, 30, [40, 80, 128, 140][seed % 4], empty=0.2)
    q = None if seed % 3 else _lengths(rng, 30, 60, empty=0.3)
    p = _problem("self", kv, q)
    for flags in (0, jfa.PLAN_PACK_SHORT, jfa.PLAN_NO_PACK, jfa.PLAN_DELTA_IN_TILES,
                  jfa.PLAN_DELTA_PREPASS, jfa.PLAN_PACK_SHORT | jfa.PLAN_DELTA_IN_TILES):
        packed = jfa.plan_choices(p.kv_offsets, p.q_offsets, H=p.H, D=p.D, num_ctas=4,
                                  flags=flags)["packed"]
        ours = bench.tiles_form_delta(p, packed, delta_prepass=bool(flags & jfa.PLAN_DELTA_PREPASS),
                                      delta_in_tiles=bool(flags & jfa.PLAN_DELTA_IN_TILES))
        assert ours == jfa.delta_in_tiles(p.kv_offsets, p.q_offsets, Lq=p.Lq, flags=flags), flags


def test_broadcast_plans_neither_pack_nor_form_delta_from_long_keys():
    p = _problem("broadcast", [300, 5, 129], Lq=64)
    assert bench.packed_runs(p, True) == []
    assert not bench.tiles_form_delta(p)
    assert not jfa.delta_in_tiles(p.kv_offsets, None, Lq=64)
