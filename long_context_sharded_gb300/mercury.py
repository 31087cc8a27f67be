"""Thin ctypes binding of libmercury_attn.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
only turns torch tensors into pointers and sizes and status codes into
exceptions.  It loads the in-tree library built by ``build.py`` and raises
immediately if it is missing: there is no CPU fallback.

The functions keep the C names:
  mercury_plan_shift(R, shift)                      -> [R, R] int32 numpy table
  mercury_attn_sharded(q, k, v, R, shift, causal, out=None, lse=None, stream=None)
  mercury_attn_partial(q, k, v, R, shift, causal, o_part=None, lse_part=None, stream=None)
  mercury_lse_merge(o_part, lse_part, out=None, lse=None, stream=None)
  mercury_sync_status(stream=None)
  mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, budget_bytes, profile)
  mercury_choose_runs(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, n_sms, scratch_cap=-1) -> int
  mercury_attn_run_schedule(q, k, v, causal, plan, out=None, lse=None, stream=None)
  mercury_tune_schedule(q, k, v, R, shift, causal, budget_bytes, top_k, ...)
Tensors: q [B,Hq,Sq,d], k/v [B,Hkv,Skv,d] bf16 CUDA tensors, contiguous.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

MERCURY_OK = 0
MERCURY_EINVAL = -1
MERCURY_EALIGN = -2
MERCURY_ECUDA = -3
MERCURY_ETIMEOUT = -4
MERCURY_ENOMEM = -5
MERCURY_EBUDGET = -6
MERCURY_EBOUNDS = -7
MERCURY_MAX_R = 128

_STATUS_NAMES = {
    MERCURY_EINVAL: "EINVAL", MERCURY_EALIGN: "EALIGN", MERCURY_ECUDA: "ECUDA",
    MERCURY_ETIMEOUT: "ETIMEOUT", MERCURY_ENOMEM: "ENOMEM", MERCURY_EBUDGET: "EBUDGET",
    MERCURY_EBOUNDS: "EBOUNDS",
}

# Every symbol include/mercury_attn.h declares.
EXPORTED = ("mercury_plan_shift", "mercury_attn_sharded", "mercury_attn_partial",
            "mercury_lse_merge", "mercury_sync_status", "mercury_last_error",
            "mercury_work_decomposition", "mercury_work_item_rows", "mercury_attn_split_noalloc",
            "mercury_gemm_shifted", "mercury_attn_decode", "mercury_attn_sharded_bf16",
            "mercury_default_cost_profile", "mercury_measure_cost_profile",
            "mercury_plan_schedules", "mercury_attn_run_schedule", "mercury_tune_schedule",
            "mercury_tune_cache_clear", "mercury_choose_runs")


class CostProfile(ctypes.Structure):
    """mercury_cost_profile: kernel costs of one device (us, GB/s)."""
    _fields_ = [("tile_us", ctypes.c_double), ("tile1_us", ctypes.c_double),
                ("item_us", ctypes.c_double), ("launch_us", ctypes.c_double),
                ("merge_gbs", ctypes.c_double), ("hbm_gbs", ctypes.c_double),
                ("n_sms", ctypes.c_int), ("measured", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class Schedule(ctypes.Structure):
    """mercury_schedule: one candidate schedule (R, Rq, n_runs, shift) and its costs."""
    _fields_ = [("R", ctypes.c_int), ("Rq", ctypes.c_int), ("n_runs", ctypes.c_int),
                ("shift", ctypes.c_int), ("work_items", ctypes.c_longlong),
                ("scratch_bytes", ctypes.c_longlong), ("hbm_bytes", ctypes.c_longlong),
                ("predicted_us", ctypes.c_double), ("measured_us", ctypes.c_double),
                ("pareto", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class MercuryError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s (%d): %s" % (_STATUS_NAMES.get(status, "?"), status, message))
        self.status = status


# MERCURY_CHECKED_BUILD=1 loads the bounds-checked variant (build(check=True)).
CHECKED = os.environ.get("MERCURY_CHECKED_BUILD", "") == "1"


def _load() -> ctypes.CDLL:
    path = _build.CHECK_LIB_PATH if CHECKED else _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            "libmercury_attn.so is not built (%s); run long_context_sharded_gb300.build.build(%s) "
            "or __graft_entry__.build() first" % (path, "check=True" if CHECKED else ""))
    lib = ctypes.CDLL(path)
    i32, i64, p = ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p
    attn_args = [p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, i32, p, p, p]
    lib.mercury_plan_shift.argtypes = [i32, i32, p]
    lib.mercury_attn_sharded.argtypes = attn_args
    lib.mercury_attn_sharded_bf16.argtypes = attn_args
    lib.mercury_attn_partial.argtypes = attn_args
    lib.mercury_lse_merge.argtypes = [p, p, i32, i64, i32, p, p, p]
    lib.mercury_gemm_shifted.argtypes = [p, p, i32, i32, i32, i32, i32, p, p]
    lib.mercury_attn_decode.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, p, p, p]
    lib.mercury_attn_split_noalloc.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                               i32, p, p, p]
    lib.mercury_sync_status.argtypes = [p]
    lib.mercury_last_error.argtypes = []
    lib.mercury_last_error.restype = ctypes.c_char_p
    lib.mercury_work_decomposition.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, p]
    lib.mercury_work_item_rows.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                           i64, p, p, p]
    lib.mercury_default_cost_profile.argtypes = [i32, p]
    lib.mercury_measure_cost_profile.argtypes = [p, p]
    lib.mercury_plan_schedules.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i64, p, p,
                                           i32, p]
    lib.mercury_attn_run_schedule.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, i32, p, p, p, p]
    lib.mercury_tune_schedule.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, i32, i64,
                                          i32, p, p, p, p, p]
    lib.mercury_tune_cache_clear.argtypes = []
    lib.mercury_choose_runs.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i64, p]
    for name in EXPORTED:
        if name not in ("mercury_last_error", "mercury_tune_cache_clear"):
            getattr(lib, name).restype = i32
    lib.mercury_tune_cache_clear.restype = None
    return lib


lib = _load()


def _check(rc: int) -> None:
    if rc != MERCURY_OK:
        raise MercuryError(rc, lib.mercury_last_error().decode(errors="replace"))


def _stream_ptr(stream):
    """cudaStream_t of `stream`, or of the current stream of the current
    device.  The raw getter avoids building a torch Stream object, which costs
    more host time than the library's whole launch path on small calls; the
    public call is the fallback where the getter is absent."""
    if stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


_DTYPES = {}


def _dtype(name):
    """torch dtype object for "torch.bfloat16" / "torch.float32" (looked up once)."""
    dt = _DTYPES.get(name)
    if dt is None:
        import torch
        dt = _DTYPES[name] = getattr(torch, name.split(".", 1)[1])
    return dt


def _dev_ptr(t, dtype_name, what):
    """Device pointer of a contiguous CUDA tensor of the given dtype on the
    current device (the library runs on the current device, and a pointer
    into another device's memory would be read there).  Small calls are
    bound by this marshalling, so the checks use the cheapest tensor queries."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % what)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % what)
    if t.dtype is not _dtype(dtype_name):
        raise TypeError("%s must be %s (got %s)" % (what, dtype_name, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    cur = torch.cuda.current_device()
    if t.get_device() != cur:
        raise ValueError("%s is on %s but the current device is cuda:%d" % (what, t.device, cur))
    return t.data_ptr()


def _check_shape(t, shape, what):
    """A caller-provided output must have exactly the shape the call writes:
    the kernels write every element of that shape, so a smaller buffer would
    be overrun."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % what)
    if t.shape != shape:  # torch.Size is a tuple
        raise ValueError("%s must have shape %s (got %s)" % (what, tuple(int(x) for x in shape),
                                                            tuple(t.shape)))


def mercury_plan_shift(R: int, shift: int) -> np.ndarray:
    out = np.zeros((R * R if R > 0 else 1,), dtype=np.int32)
    _check(lib.mercury_plan_shift(R, shift, out.ctypes.data_as(ctypes.c_void_p)))
    return out.reshape(R, R)


def _shapes(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, S, d]")
    B, Hq, Sq, d = q.shape
    Bk, Hkv, Skv, dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or dk != d:
        raise ValueError("shape mismatch: q %s k %s v %s" % (tuple(q.shape), tuple(k.shape),
                                                             tuple(v.shape)))
    return B, Hq, Hkv, Sq, Skv, d


def mercury_attn_sharded(q, k, v, R: int, shift: int, causal: bool, out=None, lse=None,
                         stream=None):
    """Attention through the shifted schedule; returns (out fp32, lse fp32)."""
    import torch
    B, Hq, Hkv, Sq, Skv, d = _shapes(q, k, v)
    if out is None:
        out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check_shape(out, (B, Hq, Sq, d), "out")
    _check_shape(lse, (B, Hq, Sq), "lse")
    rc = lib.mercury_attn_sharded(
        _dev_ptr(q, "torch.bfloat16", "q"), _dev_ptr(k, "torch.bfloat16", "k"),
        _dev_ptr(v, "torch.bfloat16", "v"), B, Hq, Hkv, Sq, Skv, d, R, shift, int(bool(causal)),
        _dev_ptr(out, "torch.float32", "out"), _dev_ptr(lse, "torch.float32", "lse"),
        _stream_ptr(stream))
    _check(rc)
    return out, lse


def mercury_attn_sharded_bf16(q, k, v, R: int, shift: int, causal: bool, out=None, lse=None,
                              stream=None):
    """As mercury_attn_sharded, with O returned in bf16 (lse fp32)."""
    import torch
    B, Hq, Hkv, Sq, Skv, d = _shapes(q, k, v)
    if out is None:
        out = torch.empty((B, Hq, Sq, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check_shape(out, (B, Hq, Sq, d), "out")
    _check_shape(lse, (B, Hq, Sq), "lse")
    rc = lib.mercury_attn_sharded_bf16(
        _dev_ptr(q, "torch.bfloat16", "q"), _dev_ptr(k, "torch.bfloat16", "k"),
        _dev_ptr(v, "torch.bfloat16", "v"), B, Hq, Hkv, Sq, Skv, d, R, shift, int(bool(causal)),
        _dev_ptr(out, "torch.bfloat16", "out"), _dev_ptr(lse, "torch.float32", "lse"),
        _stream_ptr(stream))
    _check(rc)
    return out, lse


def mercury_attn_partial(q, k, v, R: int, shift: int, causal: bool, o_part=None, lse_part=None,
                         stream=None):
    """Per-step partials; returns (o_part [R,B,Hq,Sq,d], lse_part [R,B,Hq,Sq])."""
    import torch
    B, Hq, Hkv, Sq, Skv, d = _shapes(q, k, v)
    if o_part is None:
        o_part = torch.empty((R, B, Hq, Sq, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((R, B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check_shape(o_part, (R, B, Hq, Sq, d), "o_part")
    _check_shape(lse_part, (R, B, Hq, Sq), "lse_part")
    rc = lib.mercury_attn_partial(
        _dev_ptr(q, "torch.bfloat16", "q"), _dev_ptr(k, "torch.bfloat16", "k"),
        _dev_ptr(v, "torch.bfloat16", "v"), B, Hq, Hkv, Sq, Skv, d, R, shift, int(bool(causal)),
        _dev_ptr(o_part, "torch.float32", "o_part"), _dev_ptr(lse_part, "torch.float32", "lse_part"),
        _stream_ptr(stream))
    _check(rc)
    return o_part, lse_part


def mercury_lse_merge(o_part, lse_part, out=None, lse=None, stream=None):
    """Merge partials o_part [n, ..., d] / lse_part [n, ...] over the first axis."""
    import torch
    n_parts = o_part.shape[0]
    d = o_part.shape[-1]
    rows = o_part[0].numel() // d if n_parts else 0
    if lse_part.shape[0] != n_parts or lse_part[0].numel() != rows:
        raise ValueError("lse_part does not match o_part")
    if out is None:
        out = torch.empty(tuple(o_part.shape[1:]), dtype=torch.float32, device=o_part.device)
    if lse is None:
        lse = torch.empty(tuple(lse_part.shape[1:]), dtype=torch.float32, device=o_part.device)
    if out.numel() != rows * d or out.shape[-1] != d:
        raise ValueError("out must hold %d rows of %d (got shape %s)" % (rows, d, tuple(out.shape)))
    if lse.numel() != rows:
        raise ValueError("lse must hold %d rows (got shape %s)" % (rows, tuple(lse.shape)))
    rc = lib.mercury_lse_merge(
        _dev_ptr(o_part, "torch.float32", "o_part"), _dev_ptr(lse_part, "torch.float32", "lse_part"),
        n_parts, rows, d, _dev_ptr(out, "torch.float32", "out"),
        _dev_ptr(lse, "torch.float32", "lse"), _stream_ptr(stream))
    _check(rc)
    return out, lse


def mercury_attn_split_noalloc(q, k, v, R: int, shift: int, causal: bool, n_runs: int, out, lse,
                               stream=None):
    """Split-KV attention whose partials live in the library's fixed 64 MiB
    device array: no device memory is allocated (out and lse are the
    caller's).  Calls that may overlap on the GPU must not share a device."""
    B, Hq, Hkv, Sq, Skv, d = _shapes(q, k, v)
    _check_shape(out, (B, Hq, Sq, d), "out")
    _check_shape(lse, (B, Hq, Sq), "lse")
    rc = lib.mercury_attn_split_noalloc(
        _dev_ptr(q, "torch.bfloat16", "q"), _dev_ptr(k, "torch.bfloat16", "k"),
        _dev_ptr(v, "torch.bfloat16", "v"), B, Hq, Hkv, Sq, Skv, d, R, shift, int(bool(causal)),
        int(n_runs), _dev_ptr(out, "torch.float32", "out"), _dev_ptr(lse, "torch.float32", "lse"),
        _stream_ptr(stream))
    _check(rc)
    return out, lse


def mercury_attn_decode(q, k, v, n_splits: int = 0, causal: bool = False, out=None, lse=None, stream=None):
    """Short query side against a long KV, split over the KV and merged."""
    import torch
    B, Hq, Hkv, Sq, Skv, d = _shapes(q, k, v)
    if out is None:
        out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check_shape(out, (B, Hq, Sq, d), "out")
    _check_shape(lse, (B, Hq, Sq), "lse")
    rc = lib.mercury_attn_decode(
        _dev_ptr(q, "torch.bfloat16", "q"), _dev_ptr(k, "torch.bfloat16", "k"),
        _dev_ptr(v, "torch.bfloat16", "v"), B, Hq, Hkv, Sq, Skv, d, int(n_splits), int(bool(causal)),
        _dev_ptr(out, "torch.float32", "out"), _dev_ptr(lse, "torch.float32", "lse"), _stream_ptr(stream))
    _check(rc)
    return out, lse


def mercury_gemm_shifted(a, b, R: int, shift: int, c=None, stream=None):
    """C = A @ B through the shifted schedule: a [M,K], b [K,N] bf16 -> c [M,N] fp32."""
    import torch
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("a [M,K] and b [K,N] expected")
    M, K = a.shape
    N = b.shape[1]
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _check_shape(c, (M, N), "c")
    rc = lib.mercury_gemm_shifted(_dev_ptr(a, "torch.bfloat16", "a"), _dev_ptr(b, "torch.bfloat16", "b"),
                                  M, N, K, R, shift, _dev_ptr(c, "torch.float32", "c"), _stream_ptr(stream))
    _check(rc)
    return c


def mercury_sync_status(stream=None) -> None:
    _check(lib.mercury_sync_status(_stream_ptr(stream)))


def mercury_work_decomposition(B, Hq, Hkv, Sq, Skv, d, R, causal, mode):
    """mode: 0 fused, 1 per-step partials, g >= 2 split into g runs of steps."""
    info = (ctypes.c_longlong * 8)()
    _check(lib.mercury_work_decomposition(B, Hq, Hkv, Sq, Skv, d, R, int(bool(causal)),
                                          int(mode), info))
    keys = ("Mq", "Gp", "head_mode", "T_h", "T_r", "items_per_group", "n_items", "slots")
    return {k: int(info[i]) for i, k in enumerate(keys)}


def mercury_work_item_rows(B, Hq, Hkv, Sq, Skv, d, R, shift, causal, mode, item):
    rows = (ctypes.c_longlong * 256)()
    n = ctypes.c_int(0)
    step = ctypes.c_int(0)
    _check(lib.mercury_work_item_rows(B, Hq, Hkv, Sq, Skv, d, R, shift, int(bool(causal)),
                                      int(mode), item, rows, ctypes.byref(n),
                                      ctypes.byref(step)))
    return [rows[i] for i in range(n.value)], step.value


def mercury_default_cost_profile(n_sms: int) -> CostProfile:
    prof = CostProfile()
    _check(lib.mercury_default_cost_profile(int(n_sms), ctypes.byref(prof)))
    return prof


def mercury_measure_cost_profile(stream=None) -> CostProfile:
    """Time the kernels on the current device (allocates ~2 GB, synchronises)."""
    prof = CostProfile()
    _check(lib.mercury_measure_cost_profile(ctypes.byref(prof), _stream_ptr(stream)))
    return prof


def mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, budget_bytes, profile,
                           max_plans: int = 512):
    """Candidates within the budget, fastest predicted first: (list of Schedule, total count)."""
    plans = (Schedule * max(int(max_plans), 1))()
    n = ctypes.c_int(0)
    _check(lib.mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, int(bool(causal)), R, shift,
                                      int(budget_bytes), ctypes.byref(profile), plans,
                                      int(max_plans), ctypes.byref(n)))
    return [plans[i] for i in range(min(n.value, int(max_plans)))], n.value


def mercury_choose_runs(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, n_sms, scratch_cap=-1) -> int:
    """The run count mercury_attn_sharded uses for this shape on n_sms SMs (host only)."""
    n = ctypes.c_int(0)
    _check(lib.mercury_choose_runs(B, Hq, Hkv, Sq, Skv, d, int(bool(causal)), R, shift, int(n_sms),
                                   int(scratch_cap), ctypes.byref(n)))
    return n.value


def _schedule(plan):
    if isinstance(plan, Schedule):
        return plan
    s = Schedule()
    s.R, s.Rq, s.n_runs, s.shift = (int(x) for x in plan)
    s.measured_us = -1.0
    return s


def mercury_attn_run_schedule(q, k, v, causal: bool, plan, out=None, lse=None, stream=None):
    """Attention by the schedule `plan` (a Schedule or an (R, Rq, n_runs, shift) tuple)."""
    import torch
    B, Hq, Hkv, Sq, Skv, d = _shapes(q, k, v)
    if out is None:
        out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check_shape(out, (B, Hq, Sq, d), "out")
    _check_shape(lse, (B, Hq, Sq), "lse")
    plan = _schedule(plan)
    rc = lib.mercury_attn_run_schedule(
        _dev_ptr(q, "torch.bfloat16", "q"), _dev_ptr(k, "torch.bfloat16", "k"),
        _dev_ptr(v, "torch.bfloat16", "v"), B, Hq, Hkv, Sq, Skv, d, int(bool(causal)),
        ctypes.byref(plan), _dev_ptr(out, "torch.float32", "out"),
        _dev_ptr(lse, "torch.float32", "lse"), _stream_ptr(stream))
    _check(rc)
    return out, lse


def mercury_tune_schedule(q, k, v, R: int, shift: int, causal: bool, budget_bytes: int = 0,
                          top_k: int = 4, out=None, lse=None, stream=None):
    """Tune by measurement (cached per process); returns (out, lse, Schedule, cache_hit)."""
    import torch
    B, Hq, Hkv, Sq, Skv, d = _shapes(q, k, v)
    if out is None:
        out = torch.empty((B, Hq, Sq, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check_shape(out, (B, Hq, Sq, d), "out")
    _check_shape(lse, (B, Hq, Sq), "lse")
    best = Schedule()
    hit = ctypes.c_int(0)
    rc = lib.mercury_tune_schedule(
        _dev_ptr(q, "torch.bfloat16", "q"), _dev_ptr(k, "torch.bfloat16", "k"),
        _dev_ptr(v, "torch.bfloat16", "v"), B, Hq, Hkv, Sq, Skv, d, R, shift, int(bool(causal)),
        int(budget_bytes), int(top_k), _dev_ptr(out, "torch.float32", "out"),
        _dev_ptr(lse, "torch.float32", "lse"), _stream_ptr(stream), ctypes.byref(best),
        ctypes.byref(hit))
    _check(rc)
    return out, lse, best, bool(hit.value)


def mercury_tune_cache_clear() -> None:
    lib.mercury_tune_cache_clear()
