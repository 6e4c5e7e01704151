"""Python shim over the fp64 CPU oracle (``oracle/fa_oracle.c``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference arm may import this package.  It shares
no code with the CUDA library and never imports it.

All arrays are numpy float64 in the layouts the pages use:
Q ``[b, sq, hq, d]``, K/V ``[b, skv, hkv, d]``; outputs per requested row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MUT_NO_ALPHA_ON_O = 1
MUT_NO_SCALE = 2
MUT_STRICT_CAUSAL = 4
MUT_NO_ALPHA_ON_L = 8
MUT_BWD_NO_D = 16
MUT_BWD_NO_SCALE = 32
MUT_CAP_BEFORE_SCALE = 128
MUT_CAP_NO_DERIV = 256
MUT_BWD_DK_FROM_P = 64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_attention.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, i64, ctypes.c_int, i64,
                                         ctypes.c_double, ip, i64, dp, dp, ctypes.c_int]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention_window.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, i64, ctypes.c_int, i64, i64,
                                                i64, ctypes.c_double, ip, i64, dp, dp, ctypes.c_int]
        lib.oracle_attention_window.restype = ctypes.c_int
        lib.oracle_attention_ex.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, i64, ctypes.c_int, i64, i64,
                                            i64, ctypes.c_double, ctypes.c_double, ip, i64, dp, dp, ctypes.c_int]
        lib.oracle_attention_ex.restype = ctypes.c_int
        lib.oracle_attention_tiled.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, i64, ctypes.c_int, i64, i64, i64,
                                               ctypes.c_double, ctypes.c_double, ip, i64, i64, i64, dp, dp, dp, dp,
                                               ctypes.c_int]
        lib.oracle_attention_tiled.restype = ctypes.c_int
        lib.oracle_combine.argtypes = [dp, dp, i64, i64, i64, dp, dp]
        lib.oracle_combine.restype = None
        lib.oracle_visible.argtypes = [i64, i64, i64, ctypes.c_int, i64, ctypes.c_int]
        lib.oracle_visible.restype = ctypes.c_int
        lib.oracle_visible_window.argtypes = [i64, i64, i64, ctypes.c_int, i64, i64, i64, ctypes.c_int]
        lib.oracle_visible_window.restype = ctypes.c_int
        lib.oracle_attention_bwd.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64, i64, i64, ctypes.c_int, i64, i64,
                                             i64, ctypes.c_double, ctypes.c_double, dp, dp, dp, ctypes.c_int]
        lib.oracle_attention_bwd.restype = ctypes.c_int
        lib.oracle_split_efficiency.argtypes = [i64, i64, i64]
        lib.oracle_split_efficiency.restype = ctypes.c_double
        lib.oracle_num_splits.argtypes = [i64, i64, i64, i64]
        lib.oracle_num_splits.restype = i64
        _lib = lib
        return lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _as_f64(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return np.ascontiguousarray(a)


def all_rows(b: int, hq: int, sq: int) -> np.ndarray:
    """Every (batch, head, query) triple, ordered batch, head, query."""
    bi, hi, ii = np.meshgrid(np.arange(b), np.arange(hq), np.arange(sq), indexing="ij")
    return np.stack([bi.ravel(), hi.ravel(), ii.ravel()], axis=1).astype(np.int64)


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [b, s, h, d]")
    b, sq, hq, d = q.shape
    bk, skv, hkv, dk = k.shape
    if k.shape != v.shape or bk != b or dk != d or hq % hkv != 0:
        raise ValueError("inconsistent shapes")
    return b, sq, skv, hq, hkv, d


def default_offset(sq: int, skv: int) -> int:
    """Bottom-right causal alignment: row i sees keys j <= i + (skv - sq)."""
    return skv - sq


def attention(q, k, v, *, causal: bool = False, q_pos_offset: int | None = None, scale: float | None = None,
              rows=None, mutation: int = 0, window=(-1, -1), softcap: float = 0.0):
    """Direct definition.  Returns (O [nrows, d], LSE [nrows]) for the given rows
    (default: all rows, ordered batch, head, query).  window = (left, right) widths of
    the sliding window around key i + offset; -1 leaves a side unbounded.  softcap = c > 0
    caps every scaled score s to c * tanh(s / c) before the mask and the softmax."""
    lib = _load()
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    b, sq, skv, hq, hkv, d = _shapes(q, k, v)
    off = default_offset(sq, skv) if q_pos_offset is None else int(q_pos_offset)
    sc = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = all_rows(b, hq, sq) if rows is None else np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    n = rows.shape[0]
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    wl, wr = (int(window[0]), int(window[1]))
    rc = lib.oracle_attention_ex(_dp(q), _dp(k), _dp(v), b, sq, skv, hq, hkv, d, int(causal), off, wl, wr, sc,
                                 float(softcap), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, _dp(o),
                                 _dp(lse), int(mutation))
    if rc != 0:
        raise ValueError("oracle_attention: bad arguments")
    return o, lse


def attention_tiled(q, k, v, *, tile: int, num_splits: int = 1, causal: bool = False,
                    q_pos_offset: int | None = None, scale: float | None = None, rows=None, mutation: int = 0,
                    return_partials: bool = False, window=(-1, -1), softcap: float = 0.0):
    """Tile-by-tile online-softmax model (optionally split over the key axis and merged)."""
    lib = _load()
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    b, sq, skv, hq, hkv, d = _shapes(q, k, v)
    off = default_offset(sq, skv) if q_pos_offset is None else int(q_pos_offset)
    sc = 1.0 / np.sqrt(d) if scale is None else float(scale)
    rows = all_rows(b, hq, sq) if rows is None else np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    n = rows.shape[0]
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    op = np.zeros((num_splits, n, d), dtype=np.float64)
    lp = np.zeros((num_splits, n), dtype=np.float64)
    rc = lib.oracle_attention_tiled(_dp(q), _dp(k), _dp(v), b, sq, skv, hq, hkv, d, int(causal), off,
                                    int(window[0]), int(window[1]), sc, float(softcap),
                                    rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, int(tile),
                                    int(num_splits), _dp(o), _dp(lse), _dp(op), _dp(lp), int(mutation))
    if rc != 0:
        raise ValueError("oracle_attention_tiled: bad arguments")
    if return_partials:
        return o, lse, op, lp
    return o, lse


def attention_bwd(q, k, v, dout, *, causal: bool = False, q_pos_offset: int | None = None,
                  scale: float | None = None, window=(-1, -1), mutation: int = 0, softcap: float = 0.0):
    """Recompute-based backward pass.  Returns (dQ like q, dK like k, dV like v) for the
    upstream gradient dout (shaped like q)."""
    lib = _load()
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    b, sq, skv, hq, hkv, d = _shapes(q, k, v)
    if dout.shape != q.shape:
        raise ValueError("dout must be shaped like q")
    off = default_offset(sq, skv) if q_pos_offset is None else int(q_pos_offset)
    sc = 1.0 / np.sqrt(d) if scale is None else float(scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rc = lib.oracle_attention_bwd(_dp(q), _dp(k), _dp(v), _dp(dout), b, sq, skv, hq, hkv, d, int(causal), off,
                                  int(window[0]), int(window[1]), sc, float(softcap), _dp(dq), _dp(dk), _dp(dv),
                                  int(mutation))
    if rc != 0:
        raise ValueError("oracle_attention_bwd: bad arguments")
    return dq, dk, dv


def combine(o_part, lse_part):
    """Merge split partials: o_part [ns, nrows, d], lse_part [ns, nrows]."""
    lib = _load()
    op = _as_f64(o_part)
    lp = _as_f64(lse_part)
    ns, n, d = op.shape
    if lp.shape != (ns, n):
        raise ValueError("lse_part must be [ns, nrows]")
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    lib.oracle_combine(_dp(op), _dp(lp), ns, n, d, _dp(o), _dp(lse))
    return o, lse


def visible(i: int, j: int, skv: int, causal: bool, q_pos_offset: int, mutation: int = 0, window=(-1, -1)) -> bool:
    return bool(_load().oracle_visible_window(i, j, skv, int(causal), int(q_pos_offset), int(window[0]),
                                              int(window[1]), int(mutation)))


def split_efficiency(units: int, slots: int, s: int) -> float:
    return float(_load().oracle_split_efficiency(units, slots, s))


def num_splits(units: int, slots: int, nblk: int, max_splits: int = 128) -> int:
    return int(_load().oracle_num_splits(units, slots, nblk, max_splits))
