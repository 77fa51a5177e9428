"""fp64 CPU oracle for block-sparse attention (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The library's product path never
does: the oracle shares no code with the CUDA kernels and neither side
imports the other.

The arithmetic lives in ``oracle.c`` (plain loops in double precision: the
full score row, elementwise score_mod / mask_mod, safe softmax).  This file
only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_handle = None

MASK_KINDS = {"full": 0, "causal": 1, "sliding_window": 2, "document": 3, "prefix_lm": 4, "table": 5}
SCORE_KINDS = {"none": 0, "softcap": 1, "alibi": 2, "rel_bias": 3, "alibi_softcap": 4}


class _Mask(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("window", ctypes.c_int), ("prefix_len", ctypes.c_int),
                ("seg", ctypes.c_void_p), ("seg_batch", ctypes.c_int), ("seg_len", ctypes.c_int),
                ("table", ctypes.c_void_p), ("table_batch", ctypes.c_int), ("table_q", ctypes.c_int),
                ("table_kv", ctypes.c_int)]


class _Score(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("softcap", ctypes.c_double),
                ("slopes", ctypes.c_void_p), ("rel_bias", ctypes.c_void_p), ("rel_max", ctypes.c_int)]


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP, no fast-math)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        os.makedirs(_LIBDIR, exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _lib():
    global _handle
    if _handle is None:
        build()
        h = ctypes.CDLL(_LIB)
        h.oracle_fwd_rows.restype = ctypes.c_int
        h.oracle_fwd_rows.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.POINTER(_Mask), ctypes.POINTER(_Score),
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        h.oracle_bwd.restype = ctypes.c_int
        h.oracle_bwd.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.POINTER(_Mask), ctypes.POINTER(_Score),
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        h.oracle_block_mask.restype = ctypes.c_int
        h.oracle_block_mask.argtypes = [
            ctypes.POINTER(_Mask), ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        _handle = h
    return _handle


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def _mask_struct(mask: str, window: int, prefix_len: int, seg: Optional[np.ndarray], keep: list,
                 table: Optional[np.ndarray] = None, q_len: int = 0, kv_len: int = 0):
    m = _Mask()
    m.kind = MASK_KINDS[mask]
    m.window = int(window)
    m.prefix_len = int(prefix_len)
    if mask == "document":
        s = np.ascontiguousarray(seg, dtype=np.int32)
        if s.ndim == 1:
            s = s[None, :]
        keep.append(s)
        m.seg = s.ctypes.data
        m.seg_batch = s.shape[0]
        m.seg_len = s.shape[1]
    if mask == "table":
        t = np.ascontiguousarray(table, dtype=bool).astype(np.uint8)
        if t.ndim == 2:
            t = t[None]
        if t.shape[1:] != (q_len, kv_len):
            raise ValueError(f"table must be [batch, {q_len}, {kv_len}], got {t.shape}")
        keep.append(t)
        m.table = t.ctypes.data
        m.table_batch, m.table_q, m.table_kv = t.shape
    return m


def fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, mask: str = "full", window: int = 0,
        prefix_len: int = 0, seg: Optional[np.ndarray] = None, score: str = "none",
        softcap: float = 0.0, slopes: Optional[np.ndarray] = None,
        rel_bias: Optional[np.ndarray] = None, rel_max: int = 0, scale: Optional[float] = None,
        rows: Optional[np.ndarray] = None, threads: Optional[int] = None, table: Optional[np.ndarray] = None):
    """Attention output and logsumexp in float64.

    mask "table": ``table`` is a bool array [batch (1 or B), Tq, Tkv] (or
    [Tq, Tkv]); query i of batch b attends to key j where it is true.

    q: [B, Hq, Tq, D], k / v: [B, Hkv, Tkv, D] (any float dtype; upcast).
    rows: optional flat row indices ``(b * Hq + h) * Tq + i``; when given the
    result is ``(o [len(rows), D], lse [len(rows)])``, otherwise
    ``(o [B, Hq, Tq, D], lse [B, Hq, Tq])``.
    """
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    B, Hq, Tq, D = q.shape
    Hkv, Tkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    keep: list = []
    m = _mask_struct(mask, window, prefix_len, seg, keep, table, Tq, Tkv)
    sc = _Score()
    sc.kind = SCORE_KINDS[score]
    sc.softcap = float(softcap)
    if score in ("alibi", "alibi_softcap"):
        sl = np.ascontiguousarray(slopes, dtype=np.float32)
        keep.append(sl)
        sc.slopes = sl.ctypes.data
    if score == "rel_bias":
        rb = np.ascontiguousarray(rel_bias, dtype=np.float32)
        keep.append(rb)
        sc.rel_bias = rb.ctypes.data
        sc.rel_max = int(rel_max)
    full = rows is None
    if full:
        rows = np.arange(B * Hq * Tq, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((rows.shape[0], D), dtype=np.float64)
    lse = np.empty((rows.shape[0],), dtype=np.float64)
    rc = _lib().oracle_fwd_rows(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, Hkv, Tq, Tkv, D, float(scale),
        ctypes.byref(m), ctypes.byref(sc), rows.ctypes.data, rows.shape[0],
        o.ctypes.data, lse.ctypes.data, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_fwd_rows rejected its arguments")
    if full:
        return o.reshape(B, Hq, Tq, D), lse.reshape(B, Hq, Tq)
    return o, lse


def bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray, *, mask: str = "full", window: int = 0,
        prefix_len: int = 0, seg: Optional[np.ndarray] = None, score: str = "none", softcap: float = 0.0,
        slopes: Optional[np.ndarray] = None, rel_bias: Optional[np.ndarray] = None, rel_max: int = 0,
        scale: Optional[float] = None, threads: Optional[int] = None, table: Optional[np.ndarray] = None):
    """Gradients (dq, dk, dv) in float64 of sum(O * dout) for the forward's
    arguments; dout has O's shape [B, Hq, Tq, D]."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    g = np.ascontiguousarray(dout, dtype=np.float32)
    B, Hq, Tq, D = q.shape
    Hkv, Tkv = k.shape[1], k.shape[2]
    if g.shape != q.shape:
        raise ValueError("dout must have q's shape")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    keep: list = []
    m = _mask_struct(mask, window, prefix_len, seg, keep, table, Tq, Tkv)
    sc = _Score()
    sc.kind = SCORE_KINDS[score]
    sc.softcap = float(softcap)
    if score in ("alibi", "alibi_softcap"):
        sl = np.ascontiguousarray(slopes, dtype=np.float32)
        keep.append(sl)
        sc.slopes = sl.ctypes.data
    if score == "rel_bias":
        rb = np.ascontiguousarray(rel_bias, dtype=np.float32)
        keep.append(rb)
        sc.rel_bias = rb.ctypes.data
        sc.rel_max = int(rel_max)
    dq = np.empty((B, Hq, Tq, D), dtype=np.float64)
    dk = np.empty((B, Hkv, Tkv, D), dtype=np.float64)
    dv = np.empty((B, Hkv, Tkv, D), dtype=np.float64)
    rc = _lib().oracle_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data, B, Hq, Hkv, Tq, Tkv, D,
                           float(scale), ctypes.byref(m), ctypes.byref(sc), dq.ctypes.data, dk.ctypes.data,
                           dv.ctypes.data, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_bwd rejected its arguments")
    return dq, dk, dv


def block_mask(*, mask: str, B: int, H: int, q_len: int, kv_len: int, window: int = 0,
               prefix_len: int = 0, seg: Optional[np.ndarray] = None, block: int = 128,
               threads: Optional[int] = None, table: Optional[np.ndarray] = None) -> dict:
    """Brute-force BlockMask (every in-range pair of every tile evaluated)."""
    keep: list = []
    m = _mask_struct(mask, window, prefix_len, seg, keep, table, q_len, kv_len)
    nq = (q_len + block - 1) // block
    nkv = (kv_len + block - 1) // block
    out = {
        "kv_num_blocks": np.empty((B, H, nq), dtype=np.int32),
        "kv_indices": np.empty((B, H, nq, nkv), dtype=np.int32),
        "full_kv_num_blocks": np.empty((B, H, nq), dtype=np.int32),
        "full_kv_indices": np.empty((B, H, nq, nkv), dtype=np.int32),
    }
    rc = _lib().oracle_block_mask(
        ctypes.byref(m), B, H, q_len, kv_len, block,
        out["kv_num_blocks"].ctypes.data, out["kv_indices"].ctypes.data,
        out["full_kv_num_blocks"].ctypes.data, out["full_kv_indices"].ctypes.data,
        threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_block_mask rejected its arguments")
    return out
