"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/jfa.h declares, its schedule builder matches the reference
builder bit for bit, and bad arguments are rejected before any launch."""
import ctypes

import numpy as np
import pytest

import jagged_attention_gb300 as jfa
import workloads
from oracle import tiles as ref_tiles
from tests.tiles_golden import load_cases


@pytest.fixture(scope="module", autouse=True)
def _built():
    jfa.build()


def test_exports_every_declared_function():
    names = jfa.header_functions()
    assert len(names) >= 9
    L = jfa.lib()
    for n in names:
        assert hasattr(L, n), n


def test_binding_constants_match_the_header():
    import re
    text = jfa.HEADER.read_text()
    flags = {m[0]: int(m[1]) for m in re.findall(r"#define JFA_PLAN_(\w+) (\d+)u", text)}
    assert flags == {"PACK_SHORT": jfa.PLAN_PACK_SHORT, "DYNAMIC": jfa.PLAN_DYNAMIC,
                     "DELTA_PREPASS": jfa.PLAN_DELTA_PREPASS, "DELTA_IN_TILES": jfa.PLAN_DELTA_IN_TILES,
                     "NO_PACK": jfa.PLAN_NO_PACK, "FWD_PAIRS": jfa.PLAN_FWD_PAIRS,
                     "STATIC": jfa.PLAN_STATIC, "FWD_TWO": jfa.PLAN_FWD_TWO,
                     "FWD_ONE": jfa.PLAN_FWD_ONE}
    codes = {int(m[1]): m[0] for m in re.findall(r"\b(JFA_(?:OK|ERR_\w+))\s*=\s*(\d+)", text)}
    assert codes == jfa.STATUS_NAMES


def _ref(qlen, klen, H, P, direction, pack=None, dynamic=False):
    fn = ref_tiles.fwd_tiles if direction == 0 else ref_tiles.bwd_tiles
    return fn(qlen, klen, H, 128, 128, P, pack, dynamic)


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_native_builder_matches_hand_worked(case):
    kv = workloads.offsets_from_lengths(case["kv_lengths"])
    ql = case["q_lengths"]
    bcast = len(set(ql.tolist())) == 1 and case["name"].startswith("broadcast")
    qo = None if bcast else workloads.offsets_from_lengths(ql)
    Lq = int(ql[0]) if bcast else 0
    # the hand-worked lists are host deals unless the case claims tiles
    flags = case.get("flags", 0)
    if not flags & jfa.PLAN_DYNAMIC:
        flags |= jfa.PLAN_STATIC
    for d, key in ((0, "fwd"), (1, "bwd")):
        t, p = jfa.build_tiles(kv, qo, H=case["H"], Lq=Lq, num_ctas=case["num_ctas"], direction=d,
                               flags=flags)
        assert np.array_equal(t, case[key]) and np.array_equal(p, case[f"{key}_cta_ptr"])


@pytest.mark.parametrize("seed", range(8))
def test_native_builder_matches_reference_random(seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 60))
    H = int(rng.integers(1, 6))
    klen = rng.integers(0, 1000, size=B)
    klen[rng.random(B) < 0.15] = 0
    P = int(rng.integers(1, 200))
    kv = workloads.offsets_from_lengths(klen)
    if seed % 2:
        Lq = int(rng.integers(0, 400))
        qlen, qo = np.full(B, Lq), None
    else:
        qlen = rng.integers(0, 700, size=B)
        Lq, qo = 0, workloads.offsets_from_lengths(qlen)
    for d in (0, 1):
        t, p = jfa.build_tiles(kv, qo, H=H, Lq=Lq, num_ctas=P, direction=d, flags=jfa.PLAN_STATIC)
        rt, rp = _ref(qlen, klen, H, P, d)
        assert np.array_equal(t, rt) and np.array_equal(p, rp)
        # by default the backward claims its tiles in self mode
        t, p = jfa.build_tiles(kv, qo, H=H, Lq=Lq, num_ctas=P, direction=d)
        rt, rp = _ref(qlen, klen, H, P, d, dynamic=(d == 1 and qo is not None))
        assert np.array_equal(t, rt) and np.array_equal(p, rp)
        t, p = jfa.build_tiles(kv, qo, H=H, Lq=Lq, num_ctas=P, direction=d, flags=jfa.PLAN_DYNAMIC)
        rt, rp = _ref(qlen, klen, H, P, d, dynamic=True)
        assert np.array_equal(t, rt) and np.array_equal(p, rp)


def test_dynamic_schedule_lists_every_tile_once_in_cost_order():
    lens = np.array([60, 40, 30, 200, 64, 64, 1000, 0, 129])
    kv = workloads.offsets_from_lengths(lens)
    for flags in (jfa.PLAN_DYNAMIC, jfa.PLAN_DYNAMIC | jfa.PLAN_PACK_SHORT):
        for d in (0, 1):
            t, p = jfa.build_tiles(kv, kv, H=3, num_ctas=5, direction=d, flags=flags)
            static, _ = jfa.build_tiles(kv, kv, H=3, num_ctas=5, direction=d, flags=flags & jfa.PLAN_PACK_SHORT)
            assert p[0] == 0 and (p[1:] == len(t)).all() and len(p) == min(5, len(t)) + 1
            assert (np.diff(t[:, 3]) <= 0).all()
            assert sorted(map(tuple, t)) == sorted(map(tuple, static))


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_native_builder_matches_reference_on_workloads(name):
    w = workloads.WORKLOADS[name]
    klen = workloads.draw_lengths(w.lengths, w.B, 0)
    kv = workloads.offsets_from_lengths(klen)
    if w.mode == "broadcast":
        qlen, qo, Lq = np.full(w.B, w.Lq), None, w.Lq
    else:
        qlen, qo, Lq = klen, kv, 0
    for d in (0, 1):
        t, p = jfa.build_tiles(kv, qo, H=w.H, Lq=Lq, num_ctas=152, direction=d,
                               flags=jfa.PLAN_NO_PACK | jfa.PLAN_STATIC)
        rt, rp = _ref(qlen, klen, w.H, 152, d)
        assert np.array_equal(t, rt) and np.array_equal(p, rp)
        # the default plan: packed where the default rule says so, the
        # backward's tiles claimed at run time in self mode
        t, p = jfa.build_tiles(kv, qo, H=w.H, Lq=Lq, num_ctas=152, direction=d)
        pack = ref_tiles.short_packs(klen) if qo is not None and _auto_packs(klen) else None
        rt, rp = _ref(qlen, klen, w.H, 152, d, pack, dynamic=(d == 1 and qo is not None))
        assert np.array_equal(t, rt) and np.array_equal(p, rp)


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_pair_schedule_matches_reference_on_workloads(name):
    # the forward over pair tiles (two query blocks per tile, the CTA-pair
    # kernel) is the forward schedule of the half-length query sequences
    w = workloads.WORKLOADS[name]
    klen = workloads.draw_lengths(w.lengths, w.B, 0)
    kv = workloads.offsets_from_lengths(klen)
    if w.mode == "broadcast":
        qlen, qo, Lq = np.full(w.B, w.Lq), None, w.Lq
    else:
        qlen, qo, Lq = klen, kv, 0
    t, p = jfa.build_tiles(kv, qo, H=w.H, Lq=Lq, num_ctas=76, direction=2)
    rt, rp = _ref((qlen + 1) // 2, klen, w.H, 76, 0)
    assert np.array_equal(t, rt) and np.array_equal(p, rp)
    # every query block of every (sequence, head) is in exactly one pair tile
    nblk = (qlen + 127) // 128
    assert t.shape[0] == w.H * int(((nblk + 1) // 2).sum())


@pytest.mark.parametrize("seed", range(4))
def test_pair_schedule_matches_reference_random(seed):
    rng = np.random.default_rng(500 + seed)
    B = int(rng.integers(1, 60))
    klen = rng.integers(0, 900, size=B)
    qlen = rng.integers(0, 900, size=B)
    kv, qo = workloads.offsets_from_lengths(klen), workloads.offsets_from_lengths(qlen)
    P = int(rng.integers(1, 80))
    t, p = jfa.build_tiles(kv, qo, H=2, num_ctas=P, direction=2)
    rt, rp = _ref((qlen + 1) // 2, klen, 2, P, 0)
    assert np.array_equal(t, rt) and np.array_equal(p, rp)


@pytest.mark.parametrize("seed", range(8))
def test_native_packed_builder_matches_reference_random(seed):
    rng = np.random.default_rng(300 + seed)
    B = int(rng.integers(1, 80))
    H = int(rng.integers(1, 4))
    lens = rng.integers(0, 140, size=B)
    lens[rng.random(B) < 0.2] = int(rng.integers(129, 600))
    lens[rng.random(B) < 0.1] = 0
    kv = workloads.offsets_from_lengths(lens)
    P = int(rng.integers(1, 100))
    pack = ref_tiles.short_packs(lens)
    for d in (0, 1):
        t, p = jfa.build_tiles(kv, kv, H=H, num_ctas=P, direction=d, flags=jfa.PLAN_PACK_SHORT | jfa.PLAN_STATIC)
        rt, rp = _ref(lens, lens, H, P, d, pack)
        assert np.array_equal(t, rt) and np.array_equal(p, rp)
        t, p = jfa.build_tiles(kv, kv, H=H, num_ctas=P, direction=d, flags=jfa.PLAN_PACK_SHORT)
        rt, rp = _ref(lens, lens, H, P, d, pack, dynamic=(d == 1))
        assert np.array_equal(t, rt) and np.array_equal(p, rp)
    # different query offsets or broadcast mode: the flag is ignored
    t, _ = jfa.build_tiles(kv, kv.copy() + 0, H=H, num_ctas=P, direction=0, flags=jfa.PLAN_PACK_SHORT)
    t0, _ = jfa.build_tiles(kv, None, H=H, Lq=64, num_ctas=P, direction=0, flags=jfa.PLAN_PACK_SHORT)
    assert np.array_equal(t0, _ref(np.full(B, 64), lens, H, P, 0)[0])


def test_packed_block_diagonal_workload_halves_the_tiles():
    w = workloads.WORKLOADS["block_diag"]
    kv = workloads.offsets_from_lengths(workloads.draw_lengths(w.lengths, w.B, 0))
    plain = jfa.build_tiles(kv, kv, H=w.H, num_ctas=152, direction=0, flags=jfa.PLAN_NO_PACK)[0]
    packed = jfa.build_tiles(kv, kv, H=w.H, num_ctas=152, direction=0, flags=jfa.PLAN_PACK_SHORT)[0]
    assert packed.shape[0] * 2 == plain.shape[0]
    assert (packed[:, 2] == -2).all() and (packed[:, 3] == 1).all()


def test_seed0_tile_counts():
    # tile totals of the five workloads at seed 0
    want = {"tiny_broadcast": (8, 8), "jagged_self": (624, 624), "gem_broadcast": (8192, 26028),
            "skewed_broadcast": (32768, 89248), "block_diag": (294912, 294912)}
    for name, (tf, tb) in want.items():
        w = workloads.WORKLOADS[name]
        kv = workloads.offsets_from_lengths(workloads.draw_lengths(w.lengths, w.B, 0))
        qo = None if w.mode == "broadcast" else kv
        nopack = jfa.PLAN_NO_PACK  # the unpacked schedule the quoted totals count
        assert jfa.build_tiles(kv, qo, H=w.H, Lq=w.Lq, num_ctas=152, direction=0, flags=nopack)[0].shape[0] == tf
        assert jfa.build_tiles(kv, qo, H=w.H, Lq=w.Lq, num_ctas=152, direction=1, flags=nopack)[0].shape[0] == tb


def _create(kv, qo, B, H, Lq, D, num_ctas=0, flags=0):
    L = jfa.lib()
    h = ctypes.c_void_p()
    kvp = None if kv is None else np.ascontiguousarray(kv, dtype=np.int32)
    qop = None if qo is None else np.ascontiguousarray(qo, dtype=np.int32)
    rc = L.jfa_plan_create_ex(None if kvp is None else kvp.ctypes.data_as(jfa._i32p),
                              None if qop is None else qop.ctypes.data_as(jfa._i32p),
                              B, H, Lq, D, num_ctas, flags, None, ctypes.byref(h))
    return rc


def test_rejects_bad_arguments_before_touching_the_device():
    ok = [0, 5, 9]
    assert _create(None, None, 2, 1, 4, 128) == 1                    # null offsets
    assert _create(ok, None, 2, 0, 4, 128) == 1                      # H < 1
    assert _create(ok, None, 2, 1, 4, 128, num_ctas=-1) == 1         # negative CTA count
    assert _create(ok, None, 2, 1, 4, 96) == 2                       # D not 64/128
    assert _create([1, 5, 9], None, 2, 1, 4, 128) == 3               # offsets[0] != 0
    assert _create([0, 5, 3], None, 2, 1, 4, 128) == 3               # decreasing
    assert _create(ok, [0, 2, 1], 2, 1, 0, 128) == 3                 # bad query offsets
    assert _create(ok, None, 2, 1, -1, 128) == 1                     # negative Lq
    assert _create(ok, None, 2, 1, 4, 128,                           # Delta both ways
                   flags=jfa.PLAN_DELTA_PREPASS | jfa.PLAN_DELTA_IN_TILES) == 1
    assert _create(ok, None, 2, 1, 4, 128,                           # claimed and dealt
                   flags=jfa.PLAN_DYNAMIC | jfa.PLAN_STATIC) == 1
    for both in (jfa.PLAN_FWD_PAIRS | jfa.PLAN_FWD_TWO, jfa.PLAN_FWD_TWO | jfa.PLAN_FWD_ONE,
                 jfa.PLAN_FWD_PAIRS | jfa.PLAN_FWD_ONE):                  # two forward forms
        assert _create(ok, None, 2, 1, 4, 128, flags=both) == 1
    L = jfa.lib()
    T, P = ctypes.c_int(), ctypes.c_int()
    kv = np.array([0, 4, 2], dtype=np.int32)
    assert L.jfa_build_tiles(kv.ctypes.data_as(jfa._i32p), None, 2, 1, 4, 8, 0, 0, None, None,
                             ctypes.byref(T), ctypes.byref(P)) == 3
    kv = np.array([0, 4, 6], dtype=np.int32)
    assert L.jfa_build_tiles(kv.ctypes.data_as(jfa._i32p), None, 2, 1, 4, 8, 3, 0, None, None,
                             ctypes.byref(T), ctypes.byref(P)) == 1  # bad direction (0, 1, 2 exist)
    assert L.jfa_plan_forward_pairs(None, None) == 1
    assert L.jfa_plan_claims(None, None, None) == 1
    assert L.jfa_plan_forward_form(None, None) == 1
    with pytest.raises(jfa.JfaError):
        jfa.build_tiles(kv, None, H=1, Lq=4, num_ctas=8, direction=1, flags=jfa.PLAN_DYNAMIC | jfa.PLAN_STATIC)
    assert L.jfa_fwd(None, None, None, None, 1.0, None, None, None) == 1
    assert L.jfa_bwd(None, None, None, None, None, None, None, 1.0, None, None, None, None, 0,
                     None) == 1
    assert L.jfa_status_string(7) == b"device wait timed out"
    # plan-free entry points: argument errors come back before any CUDA call
    kv = np.array([0, 5, 9], dtype=np.int32)
    bad = np.array([0, 5, 3], dtype=np.int32)
    kvp, badp = kv.ctypes.data_as(jfa._i32p), bad.ctypes.data_as(jfa._i32p)
    fwd_args = lambda off, B, H, D, scale: (None, None, None, off, None, B, H, 4, D, scale,
                                            None, None, None)
    assert L.jfa_fwd_simple(*fwd_args(None, 2, 1, 128, 0.1)) == 1   # null offsets
    assert L.jfa_fwd_simple(*fwd_args(kvp, 2, 0, 128, 0.1)) == 1    # H < 1
    assert L.jfa_fwd_simple(*fwd_args(kvp, 2, 1, 96, 0.1)) == 2     # D not 64/128
    assert L.jfa_fwd_simple(*fwd_args(badp, 2, 1, 128, 0.1)) == 3   # decreasing offsets
    assert L.jfa_fwd_simple(*fwd_args(kvp, 2, 1, 128, float("nan"))) == 1
    bwd_args = lambda off, D, scale: (None, None, None, off, None, 2, 1, 4, D, scale, None, None,
                                      None, None, None, None, None)
    assert L.jfa_bwd_simple(*bwd_args(badp, 128, 0.1)) == 3
    assert L.jfa_bwd_simple(*bwd_args(kvp, 64, float("inf"))) == 1
    assert L.jfa_simple_device_status(None, None) == 0               # nothing cached
    assert L.jfa_simple_release() == 0


def _auto_packs(klen):
    """The default packing rule restated: the reference packer's runs remove at
    least an eighth of the forward tiles (one tile per non-empty sequence of up
    to 128 rows, a run of n of them one tile)."""
    klen = np.asarray(klen, dtype=np.int64)
    runs = ref_tiles.short_packs(klen)
    saved = sum(int(np.count_nonzero(klen[b:b + n])) - 1 for b, n in enumerate(runs) if n > 1)
    return saved > 0 and 8 * saved >= int(((klen + 127) // 128).sum())


def _rule(klen, qlen, pack):
    """The documented rule, restated from the lengths alone: every sequence with
    queries has at most 128 keys, and the backward tiles (one per such
    sequence, or one per packed run) hold at least 96 key rows on average."""
    klen, qlen = np.asarray(klen), np.asarray(qlen)
    if not np.all((qlen == 0) | (klen <= 128)):
        return False
    runs = ref_tiles.short_packs(klen) if pack else None
    rows = tiles = 0
    b = 0
    while b < len(klen):
        n = runs[b] if runs is not None and runs[b] > 1 else 1
        if n > 1:
            rows, tiles, b = rows + int(klen[b:b + n].sum()), tiles + 1, b + n
            continue
        if qlen[b] > 0 and klen[b] > 0:
            rows, tiles = rows + int(klen[b]), tiles + 1
        b += 1
    return tiles > 0 and rows >= 96 * tiles


def test_noalloc_refuses_what_a_plan_refuses_before_touching_the_device():
    """jfa_bwd_noalloc checks its sizes as jfa_plan_create does, before any CUDA
    call: H * D * 2 bytes per row must stay below 2^31, and D must be 64 or 128."""
    import ctypes
    L = jfa.lib()
    fn = L.jfa_bwd_noalloc
    fn.restype = ctypes.c_int
    vp = ctypes.c_void_p
    fn.argtypes = [jfa._i32p, jfa._i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp]
    kv = jfa._offsets([0, 3])
    args = lambda H, D: (jfa._i32ptr(kv), None, 1, H, 2, D, None, None, None, None, None, None,
                         0.125, None, None, None, None, None)
    assert fn(*args(1 << 24, 64)) == 2   # 2^24 heads x 64 x 2 bytes = 2^31: JFA_ERR_UNSUPPORTED
    assert fn(*args(1, 96)) == 2         # D not in {64, 128}
    assert fn(*args(0, 64)) == 1         # no heads: JFA_ERR_INVALID_ARG


def test_packing_flags_are_exclusive():
    kv = np.array([0, 30, 60], dtype=np.int32)
    with pytest.raises(jfa.JfaError):
        jfa.build_tiles(kv, kv, H=1, num_ctas=2, direction=0,
                        flags=jfa.PLAN_PACK_SHORT | jfa.PLAN_NO_PACK)


@pytest.mark.parametrize("seed", range(6))
def test_delta_path_follows_the_documented_rule(seed):
    rng = np.random.default_rng(seed)
    for _ in range(40):
        B = int(rng.integers(1, 30))
        hi = int(rng.choice([64, 128, 129, 300]))
        klen = rng.integers(0, hi + 1, B)
        kv = np.concatenate([[0], np.cumsum(klen)]).astype(np.int32)
        for flags, pack in ((jfa.PLAN_NO_PACK, False), (jfa.PLAN_PACK_SHORT, True), (0, _auto_packs(klen))):
            want = _rule(klen, klen, pack)
            assert jfa.delta_in_tiles(kv, kv, flags=flags) == want
            assert jfa.delta_in_tiles(kv, kv, flags=flags | jfa.PLAN_DELTA_PREPASS) is False
            assert jfa.delta_in_tiles(kv, kv, flags=flags | jfa.PLAN_DELTA_IN_TILES) == bool(np.all(klen <= 128))
        # broadcast: every sequence has the Lq queries
        assert jfa.delta_in_tiles(kv, None, Lq=200) == _rule(klen, np.full(B, 200), False)


def test_delta_path_on_the_workloads():
    # the library, the benchmark's byte accounting and the expected answer
    # agree on every workload (lengths only: no tensors are drawn)
    import types
    import bench
    mode_flags = {"auto": 0, "force": jfa.PLAN_PACK_SHORT, "off": jfa.PLAN_NO_PACK}
    cases = {("tiny_broadcast", "auto"): False, ("jagged_self", "auto"): False,
             ("gem_broadcast", "auto"): False, ("block_diag", "off"): False,
             ("block_diag", "auto"): True, ("block_diag", "force"): True}
    for (name, mode), want in cases.items():
        w = workloads.WORKLOADS[name]
        klen = workloads.draw_lengths(w.lengths, w.B, 0)
        kv = workloads.offsets_from_lengths(klen)
        qlen = np.full(w.B, w.Lq) if w.mode == "broadcast" else klen
        qo = None if w.mode == "broadcast" else kv
        got = jfa.delta_in_tiles(kv, qo, Lq=w.Lq, flags=mode_flags[mode])
        prob = types.SimpleNamespace(kv_lengths=klen, q_lengths=qlen, mode=w.mode)
        pack = bench.packing_applies(prob, mode)
        assert got == want == bench.tiles_form_delta(prob, pack), (name, mode)
    with pytest.raises(jfa.JfaError):
        jfa.delta_in_tiles([0, 5], None, Lq=4, flags=jfa.PLAN_DELTA_PREPASS | jfa.PLAN_DELTA_IN_TILES)


@pytest.mark.parametrize("seed", range(4))
def test_bench_packing_matches_the_reference_packer(seed):
    # bench.py counts bytes with its own copy of the packing rule
    import types
    import bench
    rng = np.random.default_rng(100 + seed)
    for _ in range(50):
        klen = rng.integers(0, int(rng.choice([40, 80, 140])), int(rng.integers(1, 40)))
        prob = types.SimpleNamespace(kv_lengths=klen, q_lengths=klen, mode="self")
        pack = ref_tiles.short_packs(klen)
        want = [(b, b + n) for b, n in enumerate(pack) if n > 1]
        assert bench.packed_runs(prob, True) == want
        assert bench.packed_runs(prob, False) == []
        # the benchmark's copy of the default rule agrees with the library's plans
        kv = np.concatenate([[0], np.cumsum(klen)]).astype(np.int32)
        for mode, flags in (("auto", 0), ("force", jfa.PLAN_PACK_SHORT), ("off", jfa.PLAN_NO_PACK)):
            tiles = jfa.build_tiles(kv, kv, H=1, num_ctas=4, direction=0, flags=flags)[0]
            assert bench.packing_applies(prob, mode) == bool((tiles[:, 2] < 0).any()), (mode, klen)
        assert bench.packing_applies(prob, "auto") == _auto_packs(klen)


def test_bench_flushes_l2_only_for_small_workloads():
    # a step whose inputs would stay in the 129 MB L2 is timed after an L2 flush
    import types
    import bench
    p = workloads.make_workload("tiny_broadcast", seed=0)   # a real Problem (CPU tensors)
    assert bench.step_input_bytes(p) == sum(t.numel() * 2 for t in (p.q, p.k, p.v, p.dout))
    assert bench.needs_l2_flush(p)
    for name, flush in (("jagged_self", True), ("gem_broadcast", False), ("block_diag", False),
                        ("sparsity_0.9", False)):
        w = workloads.WORKLOADS[name]
        kv = workloads.offsets_from_lengths(workloads.draw_lengths(w.lengths, w.B, 0))
        rows_q = w.Lq if w.mode == "broadcast" else int(kv[-1])
        rows_o = w.B * w.Lq if w.mode == "broadcast" else int(kv[-1])
        prob = types.SimpleNamespace(H=w.H, D=w.D, n_q_rows=rows_q, n_o_rows=rows_o, kv_offsets=kv)
        assert bench.needs_l2_flush(prob) == flush, name


@pytest.mark.parametrize("lengths", [[5, 1_000_000, 300, 0, 129],      # wide cost range: comparison sort
                                     [64] * 300 + [129, 1, 1000]])      # narrow range: counting sort
def test_native_builder_cost_order_both_sort_paths(lengths):
    kl = np.array(lengths, dtype=np.int64)
    kv = workloads.offsets_from_lengths(kl)
    for d in (0, 1):
        for flags, dyn in ((0, False), (jfa.PLAN_DYNAMIC, True)):
            t, p = jfa.build_tiles(kv, None, H=3, Lq=1000, num_ctas=7, direction=d, flags=flags)
            rt, rp = ref_tiles.fwd_tiles(np.full(len(kl), 1000), kl, 3, 128, 128, 7, None, dyn) if d == 0 \
                else ref_tiles.bwd_tiles(np.full(len(kl), 1000), kl, 3, 128, 128, 7, None, dyn)
            assert np.array_equal(t, rt) and np.array_equal(p, rp)


def _choices(kv_lengths, q_lengths=None, *, H=4, D=128, Lq=0, num_ctas=16, flags=0):
    kv = np.concatenate([[0], np.cumsum(kv_lengths)]).astype(np.int32)
    qo = None if q_lengths is None else np.concatenate([[0], np.cumsum(q_lengths)]).astype(np.int32)
    return jfa.plan_choices(kv, qo, H=H, D=D, Lq=Lq, num_ctas=num_ctas, flags=flags)


def test_two_tile_forward_rule_at_its_thresholds():
    # two query tiles per CTA where the tiles of two query blocks hold >= 3 key
    # blocks on average, at most a quarter of them hold one query block, and
    # there are at least four of them per CTA (counted over heads)
    assert _choices([384] * 16, Lq=256)["forward_form"] == 2          # 3 key blocks, 64 tiles / 16 CTAs
    assert _choices([256] * 16, Lq=256)["forward_form"] == 0          # 2 key blocks
    assert _choices([384] * 16, Lq=256, num_ctas=17)["forward_form"] == 0   # under four per CTA
    assert _choices([384] * 16, Lq=384)["forward_form"] == 0          # half of the tiles half empty
    assert _choices([384] * 16, Lq=1152)["forward_form"] == 2         # one in five half empty
    assert _choices([384] * 16, Lq=640)["forward_form"] == 0          # one in three
    assert _choices([384] * 16, Lq=256, D=64)["forward_form"] == 0    # D = 128 only
    # the flags force either way, within what the kernels support
    assert _choices([256] * 16, Lq=256, flags=jfa.PLAN_FWD_TWO)["forward_form"] == 2
    assert _choices([384] * 16, Lq=256, flags=jfa.PLAN_FWD_ONE)["forward_form"] == 0
    assert _choices([384] * 16, Lq=256, flags=jfa.PLAN_FWD_PAIRS)["forward_form"] == 1
    assert _choices([384] * 16, Lq=256, flags=jfa.PLAN_FWD_TWO | jfa.PLAN_DYNAMIC)["forward_form"] == 0
    assert _choices([384] * 16, Lq=256, D=64, flags=jfa.PLAN_FWD_TWO)["forward_form"] == 0


def test_claim_and_packing_rules():
    # the backward claims its tiles at run time in self mode; both passes with
    # JFA_PLAN_DYNAMIC, neither with JFA_PLAN_STATIC
    assert _choices([300, 500], Lq=256)["claims"] == (False, False)
    assert _choices([300, 500], [300, 500])["claims"] == (False, True)
    assert _choices([300, 500], Lq=256, flags=jfa.PLAN_DYNAMIC)["claims"] == (True, True)
    assert _choices([300, 500], [300, 500], flags=jfa.PLAN_STATIC)["claims"] == (False, False)
    # short self-mode sequences are packed when that removes an eighth of the
    # forward tiles; never in broadcast mode or with JFA_PLAN_NO_PACK
    assert _choices([64] * 32, [64] * 32)["packed"]
    assert not _choices([64] * 32, [64] * 32, flags=jfa.PLAN_NO_PACK)["packed"]
    assert not _choices([64] * 32, Lq=64)["packed"]
    assert not _choices([1024] * 32, [1024] * 32)["packed"]


def test_plan_choices_rejects_bad_arguments():
    L = jfa.lib()
    kv = np.array([0, 4, 6], dtype=np.int32)
    out = ctypes.c_int()
    p = kv.ctypes.data_as(jfa._i32p)
    assert L.jfa_plan_choices(p, None, 2, 1, 4, 128, 0, 0, ctypes.byref(out), None, None, None) == 1
    assert L.jfa_plan_choices(None, None, 2, 1, 4, 128, 8, 0, None, None, None, None) == 1
    assert L.jfa_plan_choices(p, None, 2, 1, 4, 96, 8, 0, None, None, None, None) == 2   # D
    assert L.jfa_plan_choices(p, None, 2, 1, 4, 128, 8,
                              jfa.PLAN_FWD_TWO | jfa.PLAN_FWD_ONE, None, None, None, None) == 1
    bad = np.array([0, 6, 4], dtype=np.int32)
    assert L.jfa_plan_choices(bad.ctypes.data_as(jfa._i32p), None, 2, 1, 4, 128, 8, 0,
                              None, None, None, None) == 3
