"""fp64 CPU oracle for shifted-schedule sharded attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``long_context_sharded_gb300``) never imports it and shares no code with it.

``oracle_attn.c`` holds the definitions (plain attention, per-step partials of
the shifted schedule, log-sum-exp merge, its own shift table); this module
compiles it with gcc and wraps it with ctypes.  ``brute.py`` holds an
independent numpy brute force used to pin the C oracle on tiny inputs.

Every function here is pinned by ``tests/test_oracle.py`` against closed forms,
invariants, hand-written shift tables and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_attn.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_attn.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle_attn.c into a shared library with gcc + OpenMP."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # MERCURY_ORACLE_LIB lets the mutant test load a deliberately broken
        # copy of this oracle to show that the pins catch it.
        override = os.environ.get("MERCURY_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        i32, i64, p = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        lib.oracle_shift_order.argtypes = [i32, i32, p]
        lib.oracle_shift_order.restype = i32
        lib.oracle_attn_rows.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, i32, i64, p, p, p]
        lib.oracle_attn_rows.restype = i32
        lib.oracle_attn_partial_rows.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32,
                                                 i32, i32, i32, i64, p, p, p]
        lib.oracle_attn_partial_rows.restype = i32
        lib.oracle_attn_sharded_rows.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32,
                                                 i32, i32, i32, i64, p, p, p]
        lib.oracle_attn_sharded_rows.restype = i32
        lib.oracle_lse_merge.argtypes = [p, p, i32, i64, i32, p, p]
        lib.oracle_lse_merge.restype = i32
        lib.oracle_unmasked_pairs.argtypes = [i32, i32, i32]
        lib.oracle_unmasked_pairs.restype = i64
        _lib = lib
        return lib


def _bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 array of bf16 bit patterns."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
        return np.ascontiguousarray(x)
    import torch  # local: the oracle itself needs only numpy
    if x.dtype != torch.bfloat16:
        raise TypeError("oracle inputs must be bf16")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows_array(rows, B, Hq, Sq):
    if rows is None:
        return np.arange(B * Hq * Sq, dtype=np.int64)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
    if r.size and (r.min() < 0 or r.max() >= B * Hq * Sq):
        raise ValueError("row index out of range")
    return r


def shift_order(R: int, shift: int) -> np.ndarray:
    """The oracle's own [R, R] shift table (rank i, step j) -> shard."""
    out = np.zeros((R, R), dtype=np.int32)
    if _load().oracle_shift_order(R, shift, _ptr(out)) != 0:
        raise ValueError("invalid (R, shift)")
    return out


def attn(q, k, v, causal: bool, rows=None):
    """Plain softmax attention in fp64.  q [B,Hq,Sq,d], k/v [B,Hkv,Skv,d] bf16.

    rows: optional flat row indices (b*Hq + h)*Sq + q.  Returns (out, lse):
    out [n_rows, d] (or [B,Hq,Sq,d] when rows is None), lse likewise."""
    B, Hq, Sq, d = q.shape
    _, Hkv, Skv, _ = k.shape
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    r = _rows_array(rows, B, Hq, Sq)
    out = np.zeros((r.size, d), dtype=np.float64)
    lse = np.zeros((r.size,), dtype=np.float64)
    rc = _load().oracle_attn_rows(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sq, Skv, d,
                                  int(bool(causal)), r.size, _ptr(r), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_rows failed (%d)" % rc)
    if rows is None:
        return out.reshape(B, Hq, Sq, d), lse.reshape(B, Hq, Sq)
    return out, lse


def attn_partial(q, k, v, R: int, shift: int, causal: bool, rows=None):
    """Per-step partials (O_j, LSE_j), slot j = step j.  Shapes [R, n_rows, d] and
    [R, n_rows] (or [R,B,Hq,Sq,d] / [R,B,Hq,Sq] when rows is None)."""
    B, Hq, Sq, d = q.shape
    _, Hkv, Skv, _ = k.shape
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    r = _rows_array(rows, B, Hq, Sq)
    op = np.zeros((R, r.size, d), dtype=np.float64)
    lp = np.zeros((R, r.size), dtype=np.float64)
    rc = _load().oracle_attn_partial_rows(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sq, Skv, d,
                                          R, shift, int(bool(causal)), r.size, _ptr(r),
                                          _ptr(op), _ptr(lp))
    if rc != 0:
        raise ValueError("oracle_attn_partial_rows failed (%d)" % rc)
    if rows is None:
        return op.reshape(R, B, Hq, Sq, d), lp.reshape(R, B, Hq, Sq)
    return op, lp


def attn_sharded(q, k, v, R: int, shift: int, causal: bool, rows=None):
    """Sharded schedule: per-step partials merged in step order."""
    B, Hq, Sq, d = q.shape
    _, Hkv, Skv, _ = k.shape
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    r = _rows_array(rows, B, Hq, Sq)
    out = np.zeros((r.size, d), dtype=np.float64)
    lse = np.zeros((r.size,), dtype=np.float64)
    rc = _load().oracle_attn_sharded_rows(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sq, Skv, d,
                                          R, shift, int(bool(causal)), r.size, _ptr(r),
                                          _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_sharded_rows failed (%d)" % rc)
    if rows is None:
        return out.reshape(B, Hq, Sq, d), lse.reshape(B, Hq, Sq)
    return out, lse


def lse_merge(o_part, lse_part):
    """Merge partials: o_part [n_parts, rows, d], lse_part [n_parts, rows] (fp64)."""
    op = np.ascontiguousarray(np.asarray(o_part, dtype=np.float64))
    lp = np.ascontiguousarray(np.asarray(lse_part, dtype=np.float64))
    n_parts, rows, d = op.shape
    if lp.shape != (n_parts, rows):
        raise ValueError("lse_part shape mismatch")
    out = np.zeros((rows, d), dtype=np.float64)
    lse = np.zeros((rows,), dtype=np.float64)
    rc = _load().oracle_lse_merge(_ptr(op), _ptr(lp), n_parts, rows, d, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_lse_merge failed (%d)" % rc)
    return out, lse


def unmasked_pairs(Sq: int, Skv: int, causal: bool) -> int:
    """Unmasked (query, key) pairs of one (b, h)."""
    return int(_load().oracle_unmasked_pairs(Sq, Skv, int(bool(causal))))
