"""Seeded synthetic workloads for jagged attention.

This module only draws lengths and tensors; it holds none of the attention
arithmetic, so both the fp64 oracle and the CUDA library can be fed from it.

Recipes (all seeded; seed 0 is the timing seed, seeds 0-2 the parity seeds):

* lengths come from ``numpy.random.default_rng(seed)``:
    - ``uniform(lo, hi)``  -> ``integers(lo, hi + 1, size=B)``
    - ``lognormal(median, sigma, lo, hi)`` -> ``rint(lognormal(ln median, sigma))``
      clipped to ``[lo, hi]``
    - ``skewed(frac, short, long)`` -> ``B - round(frac * B)`` short lengths drawn
      first, then ``round(frac * B)`` long lengths, concatenated and shuffled
    - ``fixed(L)`` -> every length equal to ``L``
    - ``sparsity(s, Lmax)`` -> lengths whose mean is ``(1 - s) * Lmax``, so that
      a fraction ``s`` of the padded [B, Lmax] grid is empty: uniform
      ``[round((1 - 2s) Lmax), Lmax]`` for ``s <= 0.5``, uniform
      ``[1, round(2 (1 - s) Lmax)]`` above
* tensors are N(0, 1) fp32 draws from a ``torch.Generator`` seeded with ``seed``
  on the device the tensor lives on, in the order q, k, v, dout, then rounded
  to bf16 (round to nearest even).  CPU and CUDA generators give different
  values for the same seed; every comparison feeds the same tensors to both
  sides.
* ``scale = 1 / sqrt(D)``.

The named workloads stand in for the production jagged shapes the JFA pages
benchmark (GEM jagged / broadcast-Q shapes, the skewed-length load balancing
case, the TLX Block Attention batch-1152, 4k-token, H=4, D=128
block-diagonal case, a broadcast-Q sweep over sparsity 0.1, 0.5 and 0.9,
and a dense case of 768 equal sequences with H=4, D=128); the pages publish
no dataset.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    mode: str                 # "self" (Q shares the K/V offsets) or "broadcast"
    lengths: tuple            # length recipe, see module docstring
    Lq: int = 0               # broadcast only: rows of the dense Q
    note: str = ""


WORKLOADS = {
    "tiny_broadcast": Workload(
        "tiny_broadcast", B=4, H=2, D=64, mode="broadcast", Lq=64,
        lengths=("uniform", 1, 128),
        note="tiny broadcast-Q: B=4 H=2 D=64 Lq=64, K/V lengths uniform [1,128]"),
    "jagged_self": Workload(
        "jagged_self", B=32, H=4, D=128, mode="self",
        lengths=("uniform", 64, 1024),
        note="jagged self-attention: B=32 H=4 D=128, lengths uniform [64,1024]"),
    "gem_broadcast": Workload(
        "gem_broadcast", B=1024, H=4, D=128, mode="broadcast", Lq=256,
        lengths=("lognormal", 512, 1.0, 16, 4096),
        note="GEM-like broadcast-Q: B=1024 H=4 D=128 Lq=256, K/V lengths "
             "lognormal(median 512, sigma 1) clipped to [16,4096]"),
    "skewed_broadcast": Workload(
        "skewed_broadcast", B=2048, H=8, D=128, mode="broadcast", Lq=256,
        lengths=("skewed", 0.1, (16, 256), (2048, 8192)),
        note="skewed broadcast-Q: B=2048 H=8 D=128 Lq=256, 90% of lengths "
             "uniform [16,256], 10% uniform [2048,8192], shuffled"),
    "block_diag": Workload(
        "block_diag", B=73728, H=4, D=128, mode="self",
        lengths=("fixed", 64),
        note="block-diagonal self-attention: 1152 rows x 4096 tokens cut "
             "into 73,728 segments of 64, H=4 D=128"),
    # jagged broadcast-Q sparsity sweep (measurement only)
    "sparsity_0.1": Workload(
        "sparsity_0.1", B=512, H=4, D=128, mode="broadcast", Lq=256,
        lengths=("sparsity", 0.1, 2048),
        note="broadcast-Q sweep point: B=512 H=4 D=128 Lq=256, 10% of a padded "
             "[512, 2048] grid empty (lengths uniform [1638, 2048])"),
    "sparsity_0.5": Workload(
        "sparsity_0.5", B=512, H=4, D=128, mode="broadcast", Lq=256,
        lengths=("sparsity", 0.5, 2048),
        note="broadcast-Q sweep point: 50% empty (lengths uniform [0, 2048])"),
    "sparsity_0.9": Workload(
        "sparsity_0.9", B=512, H=4, D=128, mode="broadcast", Lq=256,
        lengths=("sparsity", 0.9, 2048),
        note="broadcast-Q sweep point: 90% empty (lengths uniform [1, 410])"),
    "dense_768": Workload(
        "dense_768", B=768, H=4, D=128, mode="self",
        lengths=("fixed", 1024),
        note="dense equal-length self-attention: B=768 H=4 D=128, every "
             "sequence 1024 tokens (the pages give no length)"),
}


def draw_lengths(recipe: tuple, B: int, seed: int) -> np.ndarray:
    """Sequence lengths for one recipe (int64 numpy array of size B)."""
    rng = np.random.default_rng(seed)
    kind = recipe[0]
    if kind == "uniform":
        lo, hi = recipe[1], recipe[2]
        out = rng.integers(lo, hi + 1, size=B)
    elif kind == "lognormal":
        median, sigma, lo, hi = recipe[1:5]
        out = np.clip(np.rint(rng.lognormal(math.log(median), sigma, size=B)), lo, hi)
    elif kind == "skewed":
        frac, (slo, shi), (llo, lhi) = recipe[1], recipe[2], recipe[3]
        n_long = int(round(frac * B))
        short = rng.integers(slo, shi + 1, size=B - n_long)
        long_ = rng.integers(llo, lhi + 1, size=n_long)
        out = np.concatenate([short, long_])
        rng.shuffle(out)
    elif kind == "fixed":
        out = np.full(B, recipe[1])
    elif kind == "sparsity":
        s, lmax = recipe[1], recipe[2]
        if s <= 0.5:
            out = rng.integers(int(round((1 - 2 * s) * lmax)), lmax + 1, size=B)
        else:
            out = rng.integers(1, int(round(2 * (1 - s) * lmax)) + 1, size=B)
    elif kind == "explicit":
        out = np.asarray(recipe[1])
        assert out.size == B
    else:
        raise ValueError(f"unknown length recipe {recipe!r}")
    return np.asarray(out, dtype=np.int64)


def offsets_from_lengths(lengths) -> np.ndarray:
    """Exclusive prefix sum with a leading 0: int32 offsets of size B+1."""
    lengths = np.asarray(lengths, dtype=np.int64)
    off = np.zeros(lengths.size + 1, dtype=np.int64)
    np.cumsum(lengths, out=off[1:])
    if off[-1] >= 2**31:
        raise ValueError("total length does not fit int32 offsets")
    return off.astype(np.int32)


def randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) fp32 draw rounded to bf16 (round to nearest even)."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


@dataclass
class Problem:
    """One seeded problem instance: offsets on the host, tensors on ``device``."""
    B: int
    H: int
    D: int
    mode: str
    Lq: int
    kv_offsets: np.ndarray           # int32 [B+1]
    q_offsets: np.ndarray | None     # int32 [B+1] (self mode) or None (broadcast)
    q: torch.Tensor                  # bf16 [sum Lq or Lq, H, D]
    k: torch.Tensor                  # bf16 [sum Lk, H, D]
    v: torch.Tensor
    dout: torch.Tensor               # bf16 [rows of O, H, D]
    scale: float
    extra: dict = field(default_factory=dict)

    @property
    def n_q_rows(self) -> int:       # rows of Q
        return self.Lq if self.mode == "broadcast" else int(self.q_offsets[-1])

    @property
    def n_o_rows(self) -> int:       # rows of O / dO / LSE
        return self.B * self.Lq if self.mode == "broadcast" else int(self.q_offsets[-1])

    @property
    def q_lengths(self) -> np.ndarray:
        if self.mode == "broadcast":
            return np.full(self.B, self.Lq, dtype=np.int64)
        return np.diff(self.q_offsets.astype(np.int64))

    @property
    def kv_lengths(self) -> np.ndarray:
        return np.diff(self.kv_offsets.astype(np.int64))


def make_problem(B: int, H: int, D: int, mode: str, kv_lengths, *, Lq: int = 0,
                 q_lengths=None, seed: int = 0, device="cpu") -> Problem:
    """Build a problem from explicit lengths.

    In self mode ``q_lengths`` defaults to ``kv_lengths`` (Q, K and V share
    offsets); passing different ``q_lengths`` gives jagged cross-attention.
    """
    kv_off = offsets_from_lengths(kv_lengths)
    if mode == "broadcast":
        q_off = None
        n_q, n_o = Lq, B * Lq
    elif mode == "self":
        q_off = kv_off.copy() if q_lengths is None else offsets_from_lengths(q_lengths)
        n_q = n_o = int(q_off[-1])
    else:
        raise ValueError(mode)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = randn_bf16((n_q, H, D), g, device)
    k = randn_bf16((int(kv_off[-1]), H, D), g, device)
    v = randn_bf16((int(kv_off[-1]), H, D), g, device)
    dout = randn_bf16((n_o, H, D), g, device)
    return Problem(B, H, D, mode, Lq, kv_off, q_off, q, k, v, dout, 1.0 / math.sqrt(D))


def make_workload(name: str, seed: int = 0, device="cpu", batch: int | None = None) -> Problem:
    """A named workload; ``batch`` keeps only its first ``batch`` sequences
    (same length draw), for smaller captures of the same shape mix."""
    w = WORKLOADS[name]
    lengths = draw_lengths(w.lengths, w.B, seed)
    if batch is not None:
        lengths = lengths[:batch]
    return make_problem(lengths.size, w.H, w.D, w.mode, lengths, Lq=w.Lq, seed=seed, device=device)
