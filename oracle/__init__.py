"""fp64 CPU oracle for jagged attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package; the CUDA library never calls it.  It shares no
code with ``jagged_attention_gb300``.

``oracle.c`` holds the arithmetic (see its header for the definition and the
passages it restates); this module compiles it with gcc, loads it with ctypes
and converts torch tensors to the fp64 arrays it expects.  ``tiles.py`` holds
the independent restatement of the tile schedule.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np
import torch

HERE = Path(__file__).resolve().parent
SRC = HERE / "oracle.c"
LIB = HERE / "liboracle.so"

_c_dbl_p = ctypes.POINTER(ctypes.c_double)
_c_i64_p = ctypes.POINTER(ctypes.c_int64)


def build(src: Path = SRC, out: Path = LIB, force: bool = False) -> Path:
    """Compile the oracle with gcc (-O2, OpenMP, IEEE semantics: no fast-math)."""
    if not force and out.exists() and out.stat().st_mtime >= src.stat().st_mtime:
        return out
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                           str(src), "-o", str(tmp), "-lm"])
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: Path | None = None):
        path = build() if lib_path is None else Path(lib_path)
        self.path = path
        self.lib = ctypes.CDLL(str(path))
        L = self.lib
        L.oracle_fwd.restype = ctypes.c_int
        L.oracle_fwd.argtypes = [_c_dbl_p, _c_dbl_p, _c_dbl_p, _c_i64_p, _c_i64_p,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_double, _c_dbl_p, _c_dbl_p]
        L.oracle_bwd.restype = ctypes.c_int
        L.oracle_bwd.argtypes = [_c_dbl_p, _c_dbl_p, _c_dbl_p, _c_dbl_p, _c_i64_p, _c_i64_p,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_double, _c_dbl_p, _c_dbl_p, _c_dbl_p]
        L.oracle_dq_rows.restype = ctypes.c_int
        L.oracle_dq_rows.argtypes = [_c_dbl_p, _c_dbl_p, _c_dbl_p, _c_dbl_p, _c_i64_p, _c_i64_p,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_double, ctypes.c_int, _c_i64_p, ctypes.c_int,
                                     _c_dbl_p]
        L.oracle_seq_fwd.restype = None
        L.oracle_seq_fwd.argtypes = [_c_dbl_p, ctypes.c_int64, ctypes.c_int64,
                                     _c_dbl_p, _c_dbl_p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int, ctypes.c_double,
                                     _c_dbl_p, ctypes.c_int64, _c_dbl_p, ctypes.c_int64]
        L.oracle_seq_bwd.restype = None
        L.oracle_seq_bwd.argtypes = [_c_dbl_p, ctypes.c_int64, ctypes.c_int64,
                                     _c_dbl_p, _c_dbl_p, ctypes.c_int64, ctypes.c_int64,
                                     _c_dbl_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                     _c_dbl_p, ctypes.c_int64, _c_dbl_p, _c_dbl_p, ctypes.c_int64]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_num_threads.argtypes = []

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    # -- whole problem -----------------------------------------------------
    def fwd(self, q, k, v, kv_offsets, q_offsets, B, H, Lq, D, scale):
        """O [n_o, H, D] and LSE [H, n_o] in float64 (torch CPU tensors)."""
        qd, kd, vd = _f64(q), _f64(k), _f64(v)
        kvo = _i64(kv_offsets)
        qo = None if q_offsets is None else _i64(q_offsets)
        n_o = int(qo[-1]) if qo is not None else B * Lq
        o = np.zeros((n_o, H, D), dtype=np.float64)
        lse = np.zeros((H, n_o), dtype=np.float64)
        rc = self.lib.oracle_fwd(_p(qd), _p(kd), _p(vd), _pi(kvo), _pi(qo), B, H, Lq, D,
                                 float(scale), _p(o), _p(lse))
        if rc != 0:
            raise ValueError("oracle_fwd rejected the offsets")
        return torch.from_numpy(o), torch.from_numpy(lse)

    def bwd(self, q, k, v, dout, kv_offsets, q_offsets, B, H, Lq, D, scale):
        """dQ, dK, dV in float64 (the oracle recomputes its own O and LSE)."""
        qd, kd, vd, dod = _f64(q), _f64(k), _f64(v), _f64(dout)
        kvo = _i64(kv_offsets)
        qo = None if q_offsets is None else _i64(q_offsets)
        dq = np.zeros(qd.shape, dtype=np.float64)
        dk = np.zeros(kd.shape, dtype=np.float64)
        dv = np.zeros(vd.shape, dtype=np.float64)
        rc = self.lib.oracle_bwd(_p(qd), _p(kd), _p(vd), _p(dod), _pi(kvo), _pi(qo), B, H, Lq, D,
                                 float(scale), _p(dq), _p(dk), _p(dv))
        if rc != 0:
            raise ValueError("oracle_bwd rejected the offsets")
        return torch.from_numpy(dq), torch.from_numpy(dk), torch.from_numpy(dv)

    def dq_rows(self, q, k, v, dout, kv_offsets, q_offsets, B, H, Lq, D, scale, h, rows):
        """dQ[rows, h, :] (float64 [len(rows), D]) computed row by row."""
        qd, kd, vd, dod = _f64(q), _f64(k), _f64(v), _f64(dout)
        kvo = _i64(kv_offsets)
        qo = None if q_offsets is None else _i64(q_offsets)
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        out = np.zeros((r.size, D), dtype=np.float64)
        rc = self.lib.oracle_dq_rows(_p(qd), _p(kd), _p(vd), _p(dod), _pi(kvo), _pi(qo), B, H, Lq,
                                     D, float(scale), int(h), _pi(r), int(r.size), _p(out))
        if rc != 0:
            raise ValueError("oracle_dq_rows rejected the offsets")
        return torch.from_numpy(out)

    # -- one (sequence, head) ---------------------------------------------
    def seq_fwd(self, q, k, v, scale):
        """q [nq, D], k/v [nk, D] -> O [nq, D], LSE [nq] (float64)."""
        qd, kd, vd = _f64(q), _f64(k), _f64(v)
        nq, D = qd.shape
        nk = kd.shape[0]
        o = np.zeros((nq, D), dtype=np.float64)
        lse = np.zeros(nq, dtype=np.float64)
        self.lib.oracle_seq_fwd(_p(qd), D, nq, _p(kd), _p(vd), D, nk, D, float(scale),
                                _p(o), D, _p(lse), 1)
        return torch.from_numpy(o), torch.from_numpy(lse)

    def seq_bwd(self, q, k, v, dout, scale):
        """q, dout [nq, D], k/v [nk, D] -> dQ_b [nq, D], dK [nk, D], dV [nk, D]."""
        qd, kd, vd, dod = _f64(q), _f64(k), _f64(v), _f64(dout)
        nq, D = qd.shape
        nk = kd.shape[0]
        dq = np.zeros((nq, D), dtype=np.float64)
        dk = np.zeros((nk, D), dtype=np.float64)
        dv = np.zeros((nk, D), dtype=np.float64)
        self.lib.oracle_seq_bwd(_p(qd), D, nq, _p(kd), _p(vd), D, nk, _p(dod), D, D,
                                float(scale), _p(dq), D, _p(dk), _p(dv), D)
        return torch.from_numpy(dq), torch.from_numpy(dk), torch.from_numpy(dv)


def _f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _i64(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_c_dbl_p)


def _pi(a):
    return None if a is None else a.ctypes.data_as(_c_i64_p)


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
