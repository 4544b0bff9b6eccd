#!/usr/bin/env python
"""Benchmark of the jagged attention hot path on GB300.

One step = the whole path over one synthetic batch: forward (O, LSE), the
backward pre-pass (Delta, dQ cleared) and the key/value-stationary backward
(dQ reduced across the batch, dK, dV).  ``value`` is unpadded TFLOP/s
(forward 4*D*H*sum_b Lq_b*Lk_b, backward 2.5x that) with inputs resident in
HBM; ``e2e`` is the same metric through the public API with host buffers
(plan build from host offsets, H2D of q/k/v/dO, D2H of O/LSE/dQ/dK/dV).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference      # the fp64 oracle on the host cores

Under torchrun (N > 1) every rank runs an independent batch of the same
shape (weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import workloads  # noqa: E402

DEFAULT_WORKLOAD = "gem_broadcast"
METRIC = "jagged attn fwd/bwd TFLOP/s (unpadded FLOPs) and % of GB300 BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum of a
# 256-sequence capture of the same kernel, scaled by K/V tokens: x3.730),
# keyed by kernel and workload, valid only while the hash of the code the
# kernel compiles from (comments aside) matches.
NCU_TRAFFIC = {
    "jfa_bwd_kernel:gem_broadcast": {"bytes": 3.2421e+09, "src_hash": "ec96008415c21b59"},
    "jfa_fwd2_kernel:gem_broadcast": {"bytes": 1.7841e+09, "src_hash": "f7fdb3ba4f8766af"},
}


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def pair_sum(prob: workloads.Problem) -> int:
    """sum_b Lq_b * Lk_b (query-key pairs per head)."""
    return int(np.sum(prob.q_lengths.astype(np.int64) * prob.kv_lengths.astype(np.int64)))


def flops(prob, which: str) -> float:
    base = 4.0 * prob.D * prob.H * pair_sum(prob)
    return base if which == "fwd" else 2.5 * base


def packed_runs(prob, pack: bool) -> list:
    """Runs [b, e) of sequences the library packs into one tile: greedy runs of
    short sequences totalling <= 128 rows with >= 2 non-empty (self mode only)."""
    out = []
    if not pack or prob.mode == "broadcast":
        return out
    klen = prob.kv_lengths
    b = 0
    while b < len(klen):
        if klen[b] == 0 or klen[b] > 128:
            b += 1
            continue
        total, e, nonempty = klen[b], b + 1, 1
        while e < len(klen) and total + klen[e] <= 128:
            total += klen[e]
            nonempty += klen[e] > 0
            e += 1
        if nonempty >= 2:
            out.append((b, e))
            b = e
        else:
            b += 1
    return out


def packing_applies(prob, mode: str = "auto") -> bool:
    """Whether the library packs this batch's short sequences: mode "force"
    (JFA_PLAN_PACK_SHORT) whenever a run forms, "off" (JFA_PLAN_NO_PACK) never,
    "auto" (no flag) when the runs remove at least an eighth of the forward
    tiles (a run of n non-empty sequences replaces n one-block tiles by one)."""
    if mode == "off" or prob.mode == "broadcast":
        return False
    runs = packed_runs(prob, True)
    klen = np.asarray(prob.kv_lengths, dtype=np.int64)
    saved = sum(int(np.count_nonzero(klen[b:e])) - 1 for b, e in runs)
    tiles = int(((klen + 127) // 128).sum())
    return saved > 0 and (mode == "force" or 8 * saved >= tiles)


def plan_packs(plan) -> bool:
    """Whether a plan's forward schedule holds packed tiles (block field < 0)."""
    tiles, _ = plan.tiles(0)
    return bool((tiles[:, 2] < 0).any())


def dq_rows_cleared(prob, pack: bool) -> int:
    """Query rows whose fp32 dQ the backward pre-pass clears: the library clears
    the rows tiles reduce-add into or never write (all rows in broadcast mode;
    otherwise sequences with no key or more than one 128-key block, unless
    packed), and clears everything when that leaves more than four runs or
    more than half of the rows."""
    if prob.mode == "broadcast":
        return prob.n_q_rows
    klen, qlen = prob.kv_lengths, prob.q_lengths
    packed = np.zeros(len(klen), dtype=bool)
    for b, e in packed_runs(prob, pack):
        packed[b:e] = True
    runs, rows, prev_end, pos = 0, 0, -1, 0
    for b in range(len(qlen)):
        s, e = pos, pos + int(qlen[b])
        pos = e
        if e == s or packed[b] or 0 < klen[b] <= 128:
            continue
        runs += 0 if s == prev_end else 1
        rows += e - s
        prev_end = e
    return prob.n_q_rows if (runs > 4 or 2 * rows > prob.n_q_rows) else rows


L2_BYTES = 129 * 10**6         # GB300 L2
L2_FLUSH_BYTES = 256 * 2**20   # written between timed steps when the inputs would stay in L2


def step_input_bytes(prob) -> int:
    """Bytes one step reads from its inputs: Q, K, V, dO (bf16)."""
    row = prob.H * prob.D * 2
    return (prob.n_q_rows + 2 * int(prob.kv_offsets[-1]) + prob.n_o_rows) * row


def needs_l2_flush(prob) -> bool:
    """Inputs under twice the L2 would be served from L2 by the previous step:
    such workloads flush it between timed steps."""
    return step_input_bytes(prob) < 2 * L2_BYTES


def tiles_form_delta(prob, pack: bool = False, delta_prepass: bool = False,
                     delta_in_tiles: bool = False) -> bool:
    """Whether the backward forms Delta in its main pass, by the library's rule:
    every sequence with queries has at most one 128-key block, and the tiles
    hold at least 96 key rows on average (or the flags force one way)."""
    if delta_prepass:
        return False
    klen, qlen = np.asarray(prob.kv_lengths), np.asarray(prob.q_lengths)
    if not np.all((qlen == 0) | (klen <= 128)):
        return False
    if delta_in_tiles:
        return True
    runs = packed_runs(prob, pack)
    in_run = np.zeros(len(klen), dtype=bool)
    for b, e in runs:
        in_run[b:e] = True
    alone = ~in_run & (qlen > 0) & (klen > 0)
    tiles = len(runs) + int(alone.sum())
    rows = int(klen[in_run].sum()) + int(klen[alone].sum())
    return tiles > 0 and rows >= 96 * tiles


def alg_bytes(prob, which: str, pack: bool = False, own_delta: bool = False) -> float:
    """Algorithmic HBM bytes of one launch (each tensor read or written once);
    own_delta: Delta is formed in the main pass, so neither O nor Delta moves."""
    row = prob.H * prob.D
    q = prob.n_q_rows * row * 2
    kv = prob.k.shape[0] * row * 2
    o = prob.n_o_rows * row * 2
    lse = prob.n_o_rows * prob.H * 4
    if which == "fwd":
        return q + 2 * kv + o + lse
    if which == "pre":  # O and dO read, Delta written, the reduce-added dQ rows cleared
        return (0 if own_delta else 2 * o + lse) + dq_rows_cleared(prob, pack) * row * 4
    # main: Q, K, V, dO, LSE, Delta read; dQ (fp32), dK, dV written
    return q + 2 * kv + o + (1 if own_delta else 2) * lse + prob.n_q_rows * row * 4 + 2 * kv


_COMMENT_OR_STRING = re.compile(r'"(?:\\.|[^"\\\n])*"|//[^\n]*|/\*.*?\*/', re.S)


def code_text(text: str) -> str:
    """C/CUDA source with its comments removed and whitespace runs collapsed
    (string literals kept as written): what the compiler sees."""
    code = _COMMENT_OR_STRING.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return " ".join(code.split())


def src_hash(name: str) -> str:
    """Hash of the code (not the comments) of a kernel's source file and the
    local headers it includes, so that stored ncu traffic goes stale whenever
    any code the kernel compiles from changes."""
    csrc = ROOT / "jagged_attention_gb300" / "csrc"
    h = hashlib.sha256()
    for f in (name, "kernels.h", "sm103_ptx.cuh", "tiles.cuh"):
        h.update(code_text((csrc / f).read_text()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        lines = [l for l in Path(self.out.name).read_text().splitlines() if l.strip()]
        os.unlink(self.out.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s, p in zip(sm, power) if p > 0.25 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "samples": len(sm), "power_w_max": max(power), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
class OracleSample:
    """The fp64 oracle (forward + backward), as it stands, on the first S
    sequences of a batch; S is calibrated once so one run takes about
    target_s seconds on the host cores."""

    def __init__(self, prob, target_s: float):
        import oracle

        self.prob = prob
        self.orc = oracle.default()
        self.threads = self.orc.num_threads()
        S, (fl, dt) = 1, self.run(1)
        while dt < 0.5 * target_s and S < prob.B:
            S = min(prob.B, max(S + 1, int(S * target_s / max(dt, 1e-3))))
            fl, dt = self.run(S)
        self.S = S

    def run(self, S=None):
        p = self.prob
        S = self.S if S is None else S
        kvo = workloads.offsets_from_lengths(p.kv_lengths[:S])
        kv_rows = int(kvo[-1])
        k, v = p.k[:kv_rows].cpu(), p.v[:kv_rows].cpu()
        if p.mode == "broadcast":
            q, qo, Lq = p.q.cpu(), None, p.Lq
            dout = p.dout[:S * p.Lq].cpu()
        else:
            qo = workloads.offsets_from_lengths(p.q_lengths[:S])
            q, dout, Lq = p.q[:int(qo[-1])].cpu(), p.dout[:int(qo[-1])].cpu(), 0
        t0 = time.perf_counter()
        self.orc.fwd(q, k, v, kvo, qo, S, p.H, Lq, p.D, p.scale)
        self.orc.bwd(q, k, v, dout, kvo, qo, S, p.H, Lq, p.D, p.scale)
        dt = time.perf_counter() - t0
        fl = 3.5 * 4.0 * p.D * p.H * float(np.sum(p.q_lengths[:S] * p.kv_lengths[:S]))
        return fl, dt


# ---------------------------------------------------------------------------
# Multi-rank host logic (weak scaling: every rank runs an independent batch of
# the same shape; nothing is exchanged on the data path).
def rank_seed(seed: int, rank: int) -> int:
    """The seed of rank `rank`'s batch: same workload shape, its own data."""
    return seed + rank


def combine_over_ranks(dist, times, device="cpu"):
    """Max over ranks of each timing: the slowest rank sets the job's time."""
    t = torch.tensor(list(times), dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def sum_over_ranks(dist, x: float, device="cpu") -> float:
    """Sum over ranks (each rank's batch has its own lengths, so its own flops)."""
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t.item()


def aggregate_tflops(job_flops_per_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's work per step over the (max) step time."""
    return job_flops_per_step / (ms_per_step * 1e-3) / 1e12


# One batch split across ranks (--split-batch, strong scaling): each rank takes
# a contiguous run of sequences, the runs balanced by the work sum_b Lq_b*Lk_b;
# the sequences are independent, so only broadcast mode's dQ (every sequence
# adds into the one shared query block) is summed over the ranks.
def split_batch(prob, world: int) -> list:
    """Sequence ranges [b0, b1) of the ranks, cut where the running work crosses
    r/world of the total (each range non-empty while B >= world)."""
    work = np.asarray(prob.q_lengths, dtype=np.int64) * np.asarray(prob.kv_lengths, dtype=np.int64)
    cum = np.concatenate([[0], np.cumsum(work)])
    cuts = [0]
    for r in range(1, world):
        c = int(np.searchsorted(cum, cum[-1] * r / world, side="left"))
        cuts.append(min(max(c, cuts[-1] + 1), prob.B - (world - r)))
    cuts.append(prob.B)
    return [(cuts[r], cuts[r + 1]) for r in range(world)]


def shard_problem(prob, b0: int, b1: int):
    """The sub-problem of sequences [b0, b1): offsets rebased, tensors sliced
    (views); broadcast mode keeps the whole shared Q."""
    kvo = prob.kv_offsets.astype(np.int64)
    ks, ke = int(kvo[b0]), int(kvo[b1])
    kv_off = (kvo[b0:b1 + 1] - ks).astype(np.int32)
    if prob.mode == "broadcast":
        q_off, q = None, prob.q
        os_, oe = b0 * prob.Lq, b1 * prob.Lq
    else:
        qo = prob.q_offsets.astype(np.int64)
        qs, qe = int(qo[b0]), int(qo[b1])
        q_off, q = (qo[b0:b1 + 1] - qs).astype(np.int32), prob.q[qs:qe]
        os_, oe = qs, qe
    return workloads.Problem(b1 - b0, prob.H, prob.D, prob.mode, prob.Lq, kv_off, q_off, q,
                             prob.k[ks:ke], prob.v[ks:ke], prob.dout[os_:oe], prob.scale)


def reduce_dq(dist, prob, dq):
    """Broadcast mode: every rank's dQ holds its sequences' share of the one
    shared query block; the job's dQ is their sum.  Self mode: nothing."""
    if dist is not None and prob.mode == "broadcast":
        dist.all_reduce(dq, op=dist.ReduceOp.SUM)


# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    torch.manual_seed(0)
    w = workloads.WORKLOADS[args.workload]
    prob = workloads.make_workload(args.workload, seed=args.seed, device="cpu")
    budget = min(30.0, 150.0 / max(1, args.steps + args.warmup))
    sampler = OracleSample(prob, budget)
    tfs, secs = [], []
    for i in range(args.warmup + args.steps):
        fl, dt = sampler.run()
        if i >= args.warmup:
            tfs.append(fl / dt / 1e12)
            secs.append(dt)
    S, threads = sampler.S, sampler.threads
    value = statistics.median(tfs)
    sample = (f"first {S} of {w.B} sequences of the seed-{args.seed} {args.workload} batch, "
              f"fp64 forward + backward, {statistics.median(secs):.2f} s per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * statistics.median(secs), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B": w.B, "H": w.H, "D": w.D, "Lq": w.Lq,
                   "lengths": list(map(str, w.lengths)), "seed": args.seed},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------------------
def run_ours(args, rank, world, dist):
    import jagged_attention_gb300 as jfa

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        jfa.build()
    if dist is not None:
        dist.barrier()
    jfa.lib()
    w = workloads.WORKLOADS[args.workload]
    split = args.split_batch and dist is not None
    if split:  # every rank draws the same batch and keeps its share of the sequences
        full = workloads.make_workload(args.workload, seed=args.seed, device=dev, batch=args.batch)
        prob = shard_problem(full, *split_batch(full, world)[rank])
    else:
        prob = workloads.make_workload(args.workload, seed=rank_seed(args.seed, rank), device=dev,
                                       batch=args.batch)
    flags = plan_flags(args, jfa)
    pack = packing_applies(prob, pack_mode(args))
    own_delta = tiles_form_delta(prob, pack, args.delta_prepass, args.delta_in_tiles)
    plan = jfa.Plan(prob.kv_offsets, prob.q_offsets, H=prob.H, D=prob.D, Lq=prob.Lq, flags=flags)
    if plan_packs(plan) != pack:  # the byte accounting below follows the library's rule
        raise RuntimeError("bench.py's packing rule disagrees with the library's plan")
    out = torch.empty((prob.n_o_rows, prob.H, prob.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((prob.H, prob.n_o_rows), dtype=torch.float32, device=dev)
    dq = torch.empty(prob.q.shape, dtype=torch.float32, device=dev)
    dk = torch.empty_like(prob.k)
    dv = torch.empty_like(prob.v)
    ws = torch.empty(max(16, plan.workspace_bytes()), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        jfa.fwd(plan, prob.q, prob.k, prob.v, prob.scale, out=out, lse=lse, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        jfa.bwd_preprocess(plan, out, prob.dout, dq, dk, dv, ws, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        jfa.bwd_main(plan, prob.q, prob.k, prob.v, prob.dout, lse, prob.scale, dq, dk, dv, ws,
                     stream=stream)
        if split:
            reduce_dq(dist, prob, dq)  # NCCL, on the current stream
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    plan.device_status()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = needs_l2_flush(prob)
    scrub = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            if scrub is not None:
                scrub.fill_(i & 0xFF)  # evicts the previous step's inputs from L2
            step(evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    status = plan.device_status()
    total_ms = start.elapsed_time(stop)
    if flush:  # the L2 writes between steps are not part of a step
        total_ms = sum(e[0].elapsed_time(e[3]) for e in evs)
    k_fwd = sum(e[0].elapsed_time(e[1]) for e in evs)
    k_pre = sum(e[1].elapsed_time(e[2]) for e in evs)
    k_main = sum(e[2].elapsed_time(e[3]) for e in evs)
    total_ms, k_fwd, k_pre, k_main = combine_over_ranks(dist, [total_ms, k_fwd, k_pre, k_main], dev)
    ms_step = total_ms / args.steps

    fl_step = flops(prob, "fwd") + flops(prob, "bwd")
    fl_job = sum_over_ranks(dist, fl_step, dev)
    value = aggregate_tflops(fl_job, ms_step)

    # ---- end to end through the public API with host buffers ------------------
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, prob, dev, stream, jfa)
        e2e["ms_per_step"] = combine_over_ranks(dist, [e2e["ms_per_step"]], dev)[0]
        e2e["value"] = aggregate_tflops(fl_job, e2e["ms_per_step"])

    if rank != 0:
        return

    pk, pk_kind = peaks()
    # The timed region lasts well under the seconds-long loop the sustained
    # figure describes, so the kernels are held against the burst GEMM peak;
    # a region of several seconds would take the sustained one.
    timed_s = total_ms * 1e-3
    sustained = timed_s >= 3.0 and "bf16_tflops_sustained" in pk
    tf_peak = pk["bf16_tflops_sustained"] if sustained else pk["bf16_tflops"]
    bw_peak = pk["hbm_gbs"]
    # the two-tile forward is a kernel of its own; the pair forward is the
    # one-tile kernel instantiated for clusters
    fwd_form = plan.forward_form()
    fwd_name = "jfa_fwd2_kernel" if fwd_form == 2 else "jfa_fwd_kernel"
    bwd_name = "jfa_bwd_kernel"
    per_kernel = {
        fwd_name: {"ms": k_fwd / args.steps, "flops": flops(prob, "fwd"),
                   "bytes": alg_bytes(prob, "fwd"),
                   "src": "fwd2.cu" if fwd_form == 2 else "fwd.cu"},
        "bwd_preprocess": {"ms": k_pre / args.steps, "flops": 0.0,
                           "bytes": alg_bytes(prob, "pre", pack, own_delta), "src": "bwd.cu"},
        bwd_name: {"ms": k_main / args.steps, "flops": flops(prob, "bwd"),
                   "bytes": alg_bytes(prob, "main", own_delta=own_delta), "src": "bwd.cu"},
    }
    for name, d in per_kernel.items():
        s = d["ms"] * 1e-3
        d["tflops"] = d["flops"] / s / 1e12 if d["flops"] else 0.0
        d["gbs"] = d["bytes"] / s / 1e9 if s > 0 else 0.0
        d["tensor_frac"] = d["tflops"] / tf_peak
        d["hbm_frac"] = d["gbs"] / bw_peak
    dom_name = max((fwd_name, bwd_name), key=lambda n: per_kernel[n]["ms"])
    dom = per_kernel[dom_name]
    ridge = tf_peak * 1e12 / (bw_peak * 1e9)
    ai = dom["flops"] / dom["bytes"]
    # stored counters are per kernel form: the pair instantiation has its own
    form = ":pairs" if dom_name == "jfa_fwd_kernel" and fwd_form == 1 else ""
    key = f"{dom_name}:{args.workload}{form}"
    tr = NCU_TRAFFIC.get(key)
    traffic = tr["bytes"] if tr and tr.get("src_hash") == src_hash(dom["src"]) else None
    if ai >= ridge:
        roof = {"bound": "tensor", "achieved": dom["tflops"], "peak": tf_peak, "unit": "TFLOP/s",
                "frac": dom["tflops"] / tf_peak}
    else:
        roof = {"bound": "hbm", "achieved": dom["gbs"], "peak": bw_peak, "unit": "GB/s",
                "frac": dom["gbs"] / bw_peak}
    roof.update({"traffic": traffic, "kernel": dom_name, "peak_source": f"{pk_kind} "
                 f"({('bf16 sustained' if sustained else 'bf16 burst') if roof['bound'] == 'tensor' else 'hbm copy'}"
                 f", timed region {timed_s:.2f} s)",
                 "arith_intensity": ai, "ridge": ridge,
                 "tensor_frac": dom["tensor_frac"], "hbm_frac": dom["hbm_frac"]})

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sampler = OracleSample(prob, args.cpu_seconds)
        fl, secs = sampler.run()
        cpu = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": sampler.threads,
               "kind": "oracle",
               "sample": f"first {sampler.S} of {w.B} sequences of the same batch, fp64 forward "
                         f"+ backward, {secs:.1f} s"}

    kv_gb = 2 * prob.k.numel() * 2 / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "strong" if split else "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": full.B if split else prob.B, "H": w.H, "D": w.D,
                   "Lq": w.Lq,
                   "mode": w.mode, "lengths": list(map(str, w.lengths)), "seed": args.seed,
                   "sum_kv_tokens": int(prob.kv_offsets[-1]),
                   "l2": (f"inputs under twice L2 ({step_input_bytes(prob) / 1e6:.0f} MB per step): "
                          f"a {L2_FLUSH_BYTES >> 20} MiB write flushes L2 before every timed step, "
                          f"outside the step's timed interval") if flush else
                         f"inputs larger than L2 (K+V {kv_gb:.2f} GB per step), no flush",
                   "parallelism": (f"dp{world} (one batch split by sequence, broadcast dQ all-reduced)"
                                   if split else f"dp{world} (independent batches)"),
                   "plan": ("short sequences packed" if pack else "plain schedule")
                           + claims_note(plan)
                           + FORWARD_FORMS[plan.forward_form()],
                   "delta": "formed by the backward tiles" if own_delta else "pre-pass"},
        "fwd_tflops": per_kernel[fwd_name]["tflops"],
        "bwd_tflops": flops(prob, "bwd") / ((k_pre + k_main) / args.steps * 1e-3) / 1e12,
        "pct_bf16_peak": {"fwd": 100 * per_kernel[fwd_name]["tensor_frac"],
                          "bwd_main": 100 * per_kernel[bwd_name]["tensor_frac"],
                          "step": 100 * (value / world) / tf_peak},
        "kernels": per_kernel,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": None if e2e is None else {k: e2e[k] for k in
                                          ("value", "unit", "h2d_bytes_per_step",
                                           "d2h_bytes_per_step", "ms_per_step", "steps")},
        "gpu_launches": (2 if own_delta else 3) * args.steps,  # fwd, [Delta], bwd main
        "clocks": clk.summary(),
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def pack_mode(args) -> str:
    return "force" if args.pack else ("off" if args.no_pack else "auto")


FORWARD_FORMS = {0: "", 1: ", forward as CTA pairs", 2: ", forward with two query tiles per CTA"}


def claims_note(plan) -> str:
    fwd, bwd = plan.claims()
    if fwd and bwd:
        return ", tiles claimed at run time"
    if fwd or bwd:
        return ", " + ("forward" if fwd else "backward") + " tiles claimed at run time"
    return ""


def plan_flags(args, jfa) -> int:
    return ((jfa.PLAN_PACK_SHORT if args.pack else 0) | (jfa.PLAN_NO_PACK if args.no_pack else 0)
            | (jfa.PLAN_DYNAMIC if args.dynamic else 0) | (jfa.PLAN_STATIC if args.static else 0)
            | (jfa.PLAN_DELTA_PREPASS if args.delta_prepass else 0)
            | (jfa.PLAN_DELTA_IN_TILES if args.delta_in_tiles else 0)
            | (jfa.PLAN_FWD_PAIRS if args.fwd_pairs else 0) | (jfa.PLAN_FWD_TWO if args.fwd_two else 0)
            | (jfa.PLAN_FWD_ONE if args.fwd_one else 0))


def run_e2e(args, prob, dev, stream, jfa):
    """Public-API steps with host buffers, as a training loop would run them:
    each step builds a plan from the host offsets, copies its inputs from
    pinned host memory, runs forward + backward and copies every output back
    to pinned host memory.  Steps are pipelined over an upload, a compute and a
    download stream with two sets of device buffers -- step i's uploads overlap step i-1's kernels and
    step i-2's downloads -- so the copies of every step stay inside the timed
    region, overlapped rather than serialised."""
    pin = lambda t: t.cpu().pin_memory()
    hq, hk, hv, hdo = pin(prob.q), pin(prob.k), pin(prob.v), pin(prob.dout)
    ho = torch.empty((prob.n_o_rows, prob.H, prob.D), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((prob.H, prob.n_o_rows), dtype=torch.float32).pin_memory()
    hdq = torch.empty(prob.q.shape, dtype=torch.float32).pin_memory()
    hdk = torch.empty(prob.k.shape, dtype=torch.bfloat16).pin_memory()
    hdv = torch.empty(prob.v.shape, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo)) + 4 * (prob.B + 1) * (
        1 if prob.q_offsets is None else 2)
    d2h = sum(t.numel() * t.element_size() for t in (ho, hl, hdq, hdk, hdv))
    flags = plan_flags(args, jfa)
    s_in, s_cmp, s_out, s_plan = (torch.cuda.Stream(device=dev) for _ in range(4))

    def buffers():
        b = {"q": torch.empty_like(prob.q), "k": torch.empty_like(prob.k), "v": torch.empty_like(prob.v),
             "do": torch.empty_like(prob.dout),
             "o": torch.empty((prob.n_o_rows, prob.H, prob.D), dtype=torch.bfloat16, device=dev),
             "l": torch.empty((prob.H, prob.n_o_rows), dtype=torch.float32, device=dev),
             "dq": torch.empty(prob.q.shape, dtype=torch.float32, device=dev),
             "dk": torch.empty_like(prob.k), "dv": torch.empty_like(prob.v),
             "free": torch.cuda.Event(), "in": torch.cuda.Event(), "done": torch.cuda.Event()}
        b["free"].record(s_out)
        return b

    bufs = [buffers(), buffers()]
    probe = jfa.Plan(prob.kv_offsets, prob.q_offsets, H=prob.H, D=prob.D, Lq=prob.Lq, flags=flags)
    ws_bytes = max(16, probe.workspace_bytes())
    probe.close()
    for b in bufs:
        b["ws"] = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    plans = []  # kept until the end: releasing a plan frees device memory, which synchronises

    def step(i):
        b = bufs[i % 2]
        s_in.wait_event(b["free"])  # step i-2 has downloaded these buffers
        with torch.cuda.stream(s_in):
            for key, h in (("q", hq), ("k", hk), ("v", hv), ("do", hdo)):
                b[key].copy_(h, non_blocking=True)
            b["in"].record(s_in)
        # the plan uploads its schedule on its own stream (the call waits for that upload only)
        plan = jfa.Plan(prob.kv_offsets, prob.q_offsets, H=prob.H, D=prob.D, Lq=prob.Lq, flags=flags,
                        stream=s_plan)
        plans.append(plan)
        s_cmp.wait_event(b["in"])
        jfa.fwd(plan, b["q"], b["k"], b["v"], prob.scale, out=b["o"], lse=b["l"], stream=s_cmp)
        jfa.bwd(plan, b["q"], b["k"], b["v"], b["o"], b["do"], b["l"], prob.scale, dq=b["dq"], dk=b["dk"],
                dv=b["dv"], workspace=b["ws"], stream=s_cmp)
        b["done"].record(s_cmp)
        s_out.wait_event(b["done"])
        with torch.cuda.stream(s_out):
            for key, h in (("o", ho), ("l", hl), ("dq", hdq), ("dk", hdk), ("dv", hdv)):
                h.copy_(b[key], non_blocking=True)
            b["free"].record(s_out)

    n = max(3, min(args.steps, args.e2e_steps))
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(3, 3 + n):
        step(i)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1000 / n
    for pl in plans:
        pl.close()
    return {"unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": n,
            "pipelined": "uploads, kernels and downloads of consecutive steps overlap"}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(workloads.WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    sc = ap.add_mutually_exclusive_group()
    sc.add_argument("--dynamic", action="store_true",
                    help="claim both passes' tiles at run time (JFA_PLAN_DYNAMIC; by default the "
                         "library claims the backward's in self mode only)")
    sc.add_argument("--static", action="store_true",
                    help="deal both passes' tiles on the host (JFA_PLAN_STATIC)")
    ap.add_argument("--delta-prepass", action="store_true",
                    help="form Delta in the pre-pass even where the backward tiles could (A/B)")
    ap.add_argument("--delta-in-tiles", action="store_true",
                    help="let the backward tiles form Delta wherever they can, whatever their fill")
    pk = ap.add_mutually_exclusive_group()
    pk.add_argument("--pack", action="store_true",
                    help="pack short sequences into shared tiles wherever a run forms (by default "
                         "the library packs when that removes an eighth of the tiles)")
    pk.add_argument("--no-pack", action="store_true", help="never pack short sequences")
    fw = ap.add_mutually_exclusive_group()
    fw.add_argument("--fwd-pairs", action="store_true",
                    help="run the forward as CTA pairs where the plan allows (JFA_PLAN_FWD_PAIRS)")
    fw.add_argument("--fwd-two", action="store_true",
                    help="two query tiles per CTA wherever the plan allows (JFA_PLAN_FWD_TWO; by default "
                         "where tiles are long)")
    fw.add_argument("--fwd-one", action="store_true", help="one query tile per CTA (JFA_PLAN_FWD_ONE)")
    ap.add_argument("--batch", type=int, default=None,
                    help="keep only the first B sequences of the workload (profiling captures)")
    ap.add_argument("--split-batch", action="store_true",
                    help="under torchrun: split one batch across the ranks by sequence (strong "
                         "scaling; broadcast mode sums dQ over the ranks) instead of one batch per rank")
    ap.add_argument("--e2e-steps", type=int, default=10,
                    help="timed end-to-end steps (30 measured the same per-step time as 10)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} needs one process per GPU (torchrun --nproc-per-node "
                 f"{args.gpus}); this process sees WORLD_SIZE={world}")
    dist = None
    if world > 1:
        import torch.distributed as dist_
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist_.init_process_group(backend)
        dist = dist_
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
