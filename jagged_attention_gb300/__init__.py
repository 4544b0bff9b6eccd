"""Python binding of libjfa (jagged FlashAttention for GB300, sm_103a).

Argument marshalling only: every step of the forward and backward runs in the
CUDA kernels of ``libjfa.so`` behind the C ABI in ``include/jfa.h``.  torch is
used for device memory and streams.  There is no fallback: if the library
is missing or the device is not an sm_103 GPU, calls raise.

    plan = Plan(kv_offsets, q_offsets=None, H=4, Lq=256, D=128)   # broadcast-Q
    out, lse = fwd(plan, q, k, v, scale)
    dq, dk, dv = bwd(plan, q, k, v, out, dout, lse, scale)
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

import numpy as np
import torch

PKG = Path(__file__).resolve().parent
LIB_PATH = PKG / "libjfa.so"
HEADER = PKG.parent / "include" / "jfa.h"

JFA_OK = 0
STATUS_NAMES = {
    0: "JFA_OK", 1: "JFA_ERR_INVALID_ARG", 2: "JFA_ERR_UNSUPPORTED", 3: "JFA_ERR_BAD_OFFSETS",
    4: "JFA_ERR_ALIGNMENT", 5: "JFA_ERR_WORKSPACE", 6: "JFA_ERR_CUDA", 7: "JFA_ERR_DEVICE_TIMEOUT",
}
BLOCK_M = BLOCK_N = 128
PLAN_PACK_SHORT = 1  # JFA_PLAN_PACK_SHORT
PLAN_DYNAMIC = 2  # JFA_PLAN_DYNAMIC
PLAN_DELTA_PREPASS = 4  # JFA_PLAN_DELTA_PREPASS
PLAN_DELTA_IN_TILES = 8  # JFA_PLAN_DELTA_IN_TILES
PLAN_NO_PACK = 32  # JFA_PLAN_NO_PACK
PLAN_FWD_PAIRS = 64  # JFA_PLAN_FWD_PAIRS
PLAN_STATIC = 128  # JFA_PLAN_STATIC
PLAN_FWD_TWO = 256  # JFA_PLAN_FWD_TWO
PLAN_FWD_ONE = 512  # JFA_PLAN_FWD_ONE


class JfaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where} failed: {STATUS_NAMES.get(code, code)}")


_lib = None
_lib_lock = threading.Lock()
_vp = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> Path:
    """Compile libjfa.so in-tree (nvcc, sm_103a)."""
    from . import buildlib
    return buildlib.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not LIB_PATH.exists():
                raise RuntimeError(f"{LIB_PATH} is missing: build it with jagged_attention_gb300.build()")
            L = ctypes.CDLL(str(LIB_PATH))
            L.jfa_plan_create.argtypes = [_i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, _vp, ctypes.POINTER(_vp)]
            L.jfa_plan_destroy.argtypes = [_vp]
            L.jfa_plan_tiles.argtypes = [_vp, ctypes.c_int, _i32p, _i32p, _ip, _ip]
            L.jfa_build_tiles.argtypes = [_i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_uint, _i32p, _i32p,
                                          _ip, _ip]
            L.jfa_plan_create_ex.argtypes = [_i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_uint, _vp,
                                             ctypes.POINTER(_vp)]
            L.jfa_fwd.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp]
            L.jfa_bwd_workspace_bytes.argtypes = [_vp]
            L.jfa_bwd_workspace_bytes.restype = ctypes.c_size_t
            L.jfa_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp,
                                  _vp, ctypes.c_size_t, _vp]
            L.jfa_bwd_preprocess.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
            L.jfa_bwd_main.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp,
                                       _vp, ctypes.c_size_t, _vp]
            L.jfa_delta_in_tiles.argtypes = [_i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_uint, _ip]
            _ci = ctypes.c_int
            L.jfa_fwd_simple.argtypes = [_vp, _vp, _vp, _i32p, _i32p, _ci, _ci, _ci, _ci, ctypes.c_float,
                                         _vp, _vp, _vp]
            L.jfa_bwd_simple.argtypes = [_vp, _vp, _vp, _i32p, _i32p, _ci, _ci, _ci, _ci, ctypes.c_float,
                                         _vp, _vp, _vp, _vp, _vp, _vp, _vp]
            L.jfa_simple_device_status.argtypes = [_vp, _ip]
            L.jfa_simple_release.argtypes = []
            L.jfa_plan_device_status.argtypes = [_vp, _vp, _ip]
            L.jfa_plan_selftest.argtypes = [_vp, ctypes.c_int, ctypes.c_uint]
            L.jfa_plan_forward_pairs.argtypes = [_vp, _ip]
            L.jfa_plan_claims.argtypes = [_vp, _ip, _ip]
            L.jfa_plan_forward_form.argtypes = [_vp, _ip]
            L.jfa_status_string.argtypes = [ctypes.c_int]
            L.jfa_status_string.restype = ctypes.c_char_p
            for name in ("jfa_plan_create", "jfa_plan_create_ex", "jfa_plan_destroy", "jfa_plan_tiles", "jfa_build_tiles",
                         "jfa_fwd", "jfa_bwd", "jfa_bwd_preprocess", "jfa_bwd_main",
                         "jfa_plan_device_status", "jfa_delta_in_tiles", "jfa_fwd_simple",
                         "jfa_bwd_simple", "jfa_simple_device_status", "jfa_simple_release",
                         "jfa_plan_selftest", "jfa_plan_forward_pairs", "jfa_plan_claims",
                         "jfa_plan_forward_form"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def selftest_mma_cycles(form: int, count: int = 4096, group: int = 0, stream=None) -> tuple[float, float]:
    """(cycles per product to completion, cycles per product spent issuing) of
    one form (jfa_selftest_mma_cycles): 0 M128 N128, 1 M128 N256, 2 M128 N128
    with A in TMEM, 3 M128 N64, 4 form 0 with B MN-major, 5 form 0 with A and
    B MN-major, 6 form 2 with B MN-major; count a multiple of 8; group > 0
    waits for each group of that many products before issuing the next."""
    L = lib()
    fn = L.jfa_selftest_mma_cycles
    fn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_ulonglong),
                   ctypes.POINTER(ctypes.c_ulonglong), _vp]
    fn.restype = ctypes.c_int
    c, ci = ctypes.c_ulonglong(), ctypes.c_ulonglong()
    _check(fn(form, count, group, ctypes.byref(c), ctypes.byref(ci), _stream(stream)),
           "jfa_selftest_mma_cycles")
    return c.value / count, ci.value / count


def selftest_wait_timeout(limit_us: int = 20000, stream=None) -> tuple[int, int]:
    """Run the library's bounded-wait self-test (jfa_selftest_wait_timeout):
    returns (status code, measured wait in ns).  JFA_ERR_DEVICE_TIMEOUT (7) is
    the expected status."""
    L = lib()
    fn = L.jfa_selftest_wait_timeout
    fn.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_ulonglong), _vp]
    fn.restype = ctypes.c_int
    waited = ctypes.c_ulonglong()
    rc = fn(int(limit_us), ctypes.byref(waited), None if not torch.cuda.is_available() else _stream(stream))
    return rc, waited.value


def _check(rc: int, where: str):
    if rc != JFA_OK:
        raise JfaError(rc, where)


def _offsets(a) -> np.ndarray | None:
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i32ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(_i32p)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def build_tiles(kv_offsets, q_offsets=None, *, H: int, Lq: int = 0, num_ctas: int, direction: int,
                flags: int = 0):
    """Host-only schedule (no GPU): tiles int32 [T, 4] and cta_ptr int32 [P + 1]."""
    kv = _offsets(kv_offsets)
    qo = _offsets(q_offsets)
    B = kv.size - 1
    T, P = ctypes.c_int(), ctypes.c_int()
    L = lib()
    _check(L.jfa_build_tiles(_i32ptr(kv), _i32ptr(qo), B, H, Lq, num_ctas, direction, flags, None,
                             None, ctypes.byref(T), ctypes.byref(P)), "jfa_build_tiles")
    tiles = np.zeros((T.value, 4), dtype=np.int32)
    ptr = np.zeros(P.value + 1, dtype=np.int32)
    _check(L.jfa_build_tiles(_i32ptr(kv), _i32ptr(qo), B, H, Lq, num_ctas, direction, flags,
                             tiles.ctypes.data_as(_i32p), ptr.ctypes.data_as(_i32p),
                             ctypes.byref(T), ctypes.byref(P)), "jfa_build_tiles")
    return tiles, ptr


def delta_in_tiles(kv_offsets, q_offsets=None, *, Lq: int = 0, flags: int = 0) -> bool:
    """Host-only (no GPU): whether a plan with these offsets and flags has its
    backward tiles form Delta (then the backward does not read ``out``)."""
    kv = _offsets(kv_offsets)
    qo = _offsets(q_offsets)
    res = ctypes.c_int()
    _check(lib().jfa_delta_in_tiles(_i32ptr(kv), _i32ptr(qo), kv.size - 1, Lq, flags,
                                    ctypes.byref(res)), "jfa_delta_in_tiles")
    return bool(res.value)


def plan_choices(kv_offsets, q_offsets=None, *, H: int, D: int, Lq: int = 0, num_ctas: int,
                 flags: int = 0) -> dict:
    """Host-only (no GPU): the schedule choices a plan with these arguments makes
    on a device of ``num_ctas`` SMs (jfa_plan_choices): ``forward_form`` (0 one
    query tile per CTA, 1 CTA pairs, 2 two query tiles per CTA), whether the
    forward / backward claim their tiles at run time, and whether short
    sequences are packed."""
    kv = _offsets(kv_offsets)
    qo = _offsets(q_offsets)
    fn = lib().jfa_plan_choices
    fn.argtypes = [_i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_uint, _ip, _ip, _ip, _ip]
    fn.restype = ctypes.c_int
    form, fc, bc, pk = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(fn(_i32ptr(kv), _i32ptr(qo), kv.size - 1, H, Lq, D, num_ctas, flags, ctypes.byref(form),
              ctypes.byref(fc), ctypes.byref(bc), ctypes.byref(pk)), "jfa_plan_choices")
    return {"forward_form": form.value, "claims": (bool(fc.value), bool(bc.value)), "packed": bool(pk.value)}


class Plan:
    """A jfa_plan_t: offsets and tile schedules resident on the current device,
    which must be current again whenever the plan is used."""

    def __init__(self, kv_offsets, q_offsets=None, *, H: int, D: int, Lq: int = 0,
                 num_ctas: int = 0, flags: int = 0, stream=None):
        self.kv_offsets = _offsets(kv_offsets)
        self.q_offsets = _offsets(q_offsets)
        self.B = self.kv_offsets.size - 1
        self.H, self.D = H, D
        self.broadcast = q_offsets is None
        self.Lq = Lq if self.broadcast else 0
        self.n_kv = int(self.kv_offsets[-1])
        self.n_q = self.Lq if self.broadcast else int(self.q_offsets[-1])
        self.n_o = self.B * self.Lq if self.broadcast else self.n_q
        h = _vp()
        self.flags = flags
        _check(lib().jfa_plan_create_ex(_i32ptr(self.kv_offsets), _i32ptr(self.q_offsets), self.B,
                                        H, self.Lq, D, num_ctas, flags, _stream(stream),
                                        ctypes.byref(h)),
               "jfa_plan_create_ex")
        self._h = h

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("plan already destroyed")
        return self._h

    def tiles(self, direction: int):
        T, P = ctypes.c_int(), ctypes.c_int()
        L = lib()
        _check(L.jfa_plan_tiles(self.handle, direction, None, None, ctypes.byref(T), ctypes.byref(P)),
               "jfa_plan_tiles")
        tiles = np.zeros((T.value, 4), dtype=np.int32)
        ptr = np.zeros(P.value + 1, dtype=np.int32)
        _check(L.jfa_plan_tiles(self.handle, direction, tiles.ctypes.data_as(_i32p),
                                ptr.ctypes.data_as(_i32p), ctypes.byref(T), ctypes.byref(P)),
               "jfa_plan_tiles")
        return tiles, ptr

    def claims(self) -> tuple:
        """(forward, backward): whether each pass claims its tiles at run time."""
        f, b = ctypes.c_int(), ctypes.c_int()
        _check(lib().jfa_plan_claims(self.handle, ctypes.byref(f), ctypes.byref(b)), "jfa_plan_claims")
        return bool(f.value), bool(b.value)

    def forward_form(self) -> int:
        """0: one query tile per CTA, 1: CTA pairs, 2: two query tiles per CTA."""
        v = ctypes.c_int()
        _check(lib().jfa_plan_forward_form(self.handle, ctypes.byref(v)), "jfa_plan_forward_form")
        return v.value

    def forward_pairs(self) -> bool:
        """Whether the plan's forward runs as CTA pairs over pair tiles."""
        v = ctypes.c_int()
        _check(lib().jfa_plan_forward_pairs(self.handle, ctypes.byref(v)), "jfa_plan_forward_pairs")
        return bool(v.value)

    def workspace_bytes(self) -> int:
        return int(lib().jfa_bwd_workspace_bytes(self.handle))

    def device_status(self, stream=None) -> int:
        """Raise JfaError if a kernel recorded a timed-out wait; returns the raw word."""
        raw = ctypes.c_int()
        _check(lib().jfa_plan_device_status(self.handle, _stream(stream), ctypes.byref(raw)),
               "jfa_plan_device_status")
        return raw.value

    def selftest(self, skip: int, limit_us: int = 0):
        """Failure-path test only (jfa_plan_selftest): shorten every device wait of
        this plan's later launches to limit_us and withhold one arrival (skip 1:
        forward, 2: backward; 0: none)."""
        _check(lib().jfa_plan_selftest(self.handle, skip, limit_us), "jfa_plan_selftest")

    def close(self):
        if self._h is not None:
            _check(lib().jfa_plan_destroy(self._h), "jfa_plan_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _dev(t: torch.Tensor, name: str, dtype) -> int:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def fwd(plan: Plan, q, k, v, scale: float, out=None, lse=None, stream=None):
    """O (bf16 [n_o, H, D]) and LSE (fp32 [H, n_o]) through jfa_fwd."""
    dev = k.device if k.numel() else q.device
    if out is None:
        out = torch.empty((plan.n_o, plan.H, plan.D), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((plan.H, plan.n_o), dtype=torch.float32, device=dev)
    _check(lib().jfa_fwd(plan.handle, _dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
                         _dev(v, "v", torch.bfloat16), float(scale), _dev(out, "out", torch.bfloat16),
                         _dev(lse, "lse", torch.float32), _stream(stream)), "jfa_fwd")
    return out, lse


def bwd(plan: Plan, q, k, v, out, dout, lse, scale: float, dq=None, dk=None, dv=None,
        workspace=None, stream=None):
    """dQ (fp32, shape of q), dK and dV (bf16) through jfa_bwd."""
    if dq is None:
        dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    ws_bytes = plan.workspace_bytes()
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=k.device)
    _check(lib().jfa_bwd(plan.handle, _dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
                         _dev(v, "v", torch.bfloat16), _dev(out, "out", torch.bfloat16),
                         _dev(dout, "dout", torch.bfloat16), _dev(lse, "lse", torch.float32),
                         float(scale), _dev(dq, "dq", torch.float32), _dev(dk, "dk", torch.bfloat16),
                         _dev(dv, "dv", torch.bfloat16), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), _stream(stream)), "jfa_bwd")
    return dq, dk, dv


def _simple_sizes(q, k, kv_offsets, q_offsets):
    kv = _offsets(kv_offsets)
    qo = _offsets(q_offsets)
    B = kv.size - 1
    H, D = int(k.shape[1]), int(k.shape[2])
    Lq = int(q.shape[0]) if qo is None else 0
    n_o = B * Lq if qo is None else int(qo[-1])
    return kv, qo, B, H, Lq, D, n_o


def fwd_simple(q, k, v, kv_offsets, q_offsets=None, *, scale: float, out=None, lse=None,
               stream=None):
    """O and LSE through jfa_fwd_simple: no plan object (the library caches one per
    distinct offsets).  q_offsets None: broadcast mode, q holds the Lq shared rows."""
    kv, qo, B, H, Lq, D, n_o = _simple_sizes(q, k, kv_offsets, q_offsets)
    if out is None:
        out = torch.empty((n_o, H, D), dtype=torch.bfloat16, device=k.device)
    if lse is None:
        lse = torch.empty((H, n_o), dtype=torch.float32, device=k.device)
    _check(lib().jfa_fwd_simple(_dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
                                _dev(v, "v", torch.bfloat16), _i32ptr(kv), _i32ptr(qo), B, H, Lq, D,
                                float(scale), _dev(out, "out", torch.bfloat16),
                                _dev(lse, "lse", torch.float32), _stream(stream)), "jfa_fwd_simple")
    return out, lse


def bwd_simple(q, k, v, out, dout, lse, kv_offsets, q_offsets=None, *, scale: float, dq=None,
               dk=None, dv=None, stream=None):
    """dQ (fp32), dK, dV through jfa_bwd_simple (cached plan and workspace)."""
    kv, qo, B, H, Lq, D, _ = _simple_sizes(q, k, kv_offsets, q_offsets)
    if dq is None:
        dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    _check(lib().jfa_bwd_simple(_dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
                                _dev(v, "v", torch.bfloat16), _i32ptr(kv), _i32ptr(qo), B, H, Lq, D,
                                float(scale), _dev(out, "out", torch.bfloat16),
                                _dev(dout, "dout", torch.bfloat16), _dev(lse, "lse", torch.float32),
                                _dev(dq, "dq", torch.float32), _dev(dk, "dk", torch.bfloat16),
                                _dev(dv, "dv", torch.bfloat16), _stream(stream)), "jfa_bwd_simple")
    return dq, dk, dv


def simple_device_status(stream=None) -> int:
    """jfa_simple_device_status: status code (JFA_OK or JFA_ERR_DEVICE_TIMEOUT)."""
    raw = ctypes.c_int()
    return int(lib().jfa_simple_device_status(_stream(stream), ctypes.byref(raw)))


def simple_release():
    """Release the plans and workspaces the plan-free calls cached."""
    _check(lib().jfa_simple_release(), "jfa_simple_release")


def header_functions() -> list[str]:
    """Names of the functions include/jfa.h declares."""
    import re
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jfa_[a-z_0-9]+)\s*\(", text)))


def bwd_preprocess(plan: Plan, out, dout, dq, dk, dv, workspace, stream=None):
    """Delta into ``workspace`` (unless the plan's main pass forms it), dq cleared,
    dK/dV of query-less sequences zeroed."""
    _check(lib().jfa_bwd_preprocess(plan.handle, _dev(out, "out", torch.bfloat16),
                                    _dev(dout, "dout", torch.bfloat16), _dev(dq, "dq", torch.float32),
                                    _dev(dk, "dk", torch.bfloat16), _dev(dv, "dv", torch.bfloat16),
                                    workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "jfa_bwd_preprocess")


def bwd_main(plan: Plan, q, k, v, dout, lse, scale: float, dq, dk, dv, workspace, stream=None):
    """The key/value-stationary backward pass (after bwd_preprocess on the same stream)."""
    _check(lib().jfa_bwd_main(plan.handle, _dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
                              _dev(v, "v", torch.bfloat16), _dev(dout, "dout", torch.bfloat16),
                              _dev(lse, "lse", torch.float32), float(scale),
                              _dev(dq, "dq", torch.float32), _dev(dk, "dk", torch.bfloat16),
                              _dev(dv, "dv", torch.bfloat16), workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream(stream)),
           "jfa_bwd_main")
