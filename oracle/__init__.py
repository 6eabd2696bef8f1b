"""CPU oracle for GQA decode and the K/V mean-pool conversion (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The CUDA library never links, loads or calls it, and
it imports nothing from the library.  The arithmetic lives in ``gqa_oracle.c``
(plain float64 loops, see its header for the passages it follows); this module
only compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off keeps every multiply and add separately rounded; no
# -ffast-math, so the compiler may not reassociate the sums.
CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile ``gqa_oracle.c`` into ``liboracle.so`` (gcc + OpenMP)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def load(path: Optional[str] = None):
    """Load the compiled oracle (building it first if needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    lib.oracle_gqa_decode_f64.restype = ctypes.c_int
    lib.oracle_gqa_decode_f64.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_float, P, ctypes.c_int64]
    lib.oracle_gqa_decode_window_f64.restype = ctypes.c_int
    lib.oracle_gqa_decode_window_f64.argtypes = [P, P, P, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, P,
                                                 ctypes.c_int64]
    lib.oracle_gather_pages.restype = ctypes.c_int
    lib.oracle_gather_pages.argtypes = [P, P, P, P] + [ctypes.c_int] * 7
    lib.oracle_append_row.restype = ctypes.c_int
    lib.oracle_append_row.argtypes = [P, P, P] + [ctypes.c_int] * 4
    lib.oracle_meanpool_f32.restype = ctypes.c_int
    lib.oracle_meanpool_f32.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int64]
    lib.oracle_meanpool_f64.restype = ctypes.c_int
    lib.oracle_meanpool_f64.argtypes = [P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int64]
    lib.oracle_group_of.restype = ctypes.c_int
    lib.oracle_group_of.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def gqa_decode_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, seq_lens: Optional[np.ndarray],
                   scale, rows: Optional[np.ndarray] = None, window: int = 0, lib=None) -> np.ndarray:
    """Float64 GQA decode.  q [B,H,d], k/v [B,G,Lmax,d] as uint16 bf16 bits.

    ``seq_lens=None``: every one of the Lmax positions is valid (cross-attention).
    ``window > 0``: only the last ``window`` valid positions are attended.
    Returns out [B, H, d] float64.  With ``rows`` (flat ids b*H+i), only those
    rows are computed; the others are NaN.
    """
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    B, H, d = q.shape
    Bk, G, L, dk = k.shape
    assert Bk == B and dk == d and v.shape == k.shape
    if seq_lens is not None:
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        assert sl.shape == (B,)
        slp = _ptr(sl)
    else:
        slp = None
    out = np.full((B, H, d), np.nan, dtype=np.float64)
    if rows is None:
        rp, nr = None, 0
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        rp, nr = _ptr(r), r.size
    rc = lib.oracle_gqa_decode_window_f64(_ptr(q), _ptr(k), _ptr(v), slp, int(window), _ptr(out),
                                          B, H, G, d, L, float(np.float32(scale)), rp, nr)
    if rc != 0:
        raise ValueError("oracle_gqa_decode_window_f64 rejected its arguments")
    return out


def gather_pages(pages: np.ndarray, table: np.ndarray, seq_lens: Optional[np.ndarray], Lmax: int,
                 fill: int = 0x7FC0, lib=None) -> np.ndarray:
    """Paged cache [num_pages, G, page_size, d] + block table [B, max_pages] -> [B, G, Lmax, d].

    Rows past each sequence's length hold ``fill`` (default: bf16 NaN bits).
    """
    lib = lib or load()
    pages = np.ascontiguousarray(pages, dtype=np.uint16)
    table = np.ascontiguousarray(table, dtype=np.int32)
    num_pages, G, page_size, d = pages.shape
    B, max_pages = table.shape
    out = np.full((B, G, Lmax, d), fill, dtype=np.uint16)
    sl = None if seq_lens is None else np.ascontiguousarray(seq_lens, dtype=np.int32)
    rc = lib.oracle_gather_pages(_ptr(pages), _ptr(table), None if sl is None else _ptr(sl), _ptr(out),
                                 B, G, d, page_size, max_pages, num_pages, Lmax)
    if rc != 0:
        raise ValueError("oracle_gather_pages rejected its arguments")
    return out


def append_row(cache: np.ndarray, row: np.ndarray, seq_lens: np.ndarray, lib=None) -> np.ndarray:
    """Copy of ``cache`` [B,G,Lmax,d] with ``row`` [B,G,d] written at position seq_lens[b] - 1."""
    lib = lib or load()
    out = np.array(cache, dtype=np.uint16, order="C", copy=True)
    row = np.ascontiguousarray(row, dtype=np.uint16)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, G, L, d = out.shape
    assert row.shape == (B, G, d) and sl.shape == (B,)
    if lib.oracle_append_row(_ptr(out), _ptr(row), _ptr(sl), B, G, d, L) != 0:
        raise ValueError("oracle_append_row rejected its arguments")
    return out


def meanpool_f32(w: np.ndarray, H: int, G: int, head_axis: int = 0, lib=None) -> np.ndarray:
    """fp32 mean-pool over heads.

    ``head_axis=0``: head-major ``[H, ...]`` -> ``[G, ...]``.
    ``head_axis=1``: ``[outer, H, inner]`` -> ``[outer, G, inner]``.
    """
    lib = lib or load()
    w = np.ascontiguousarray(w, dtype=np.float32)
    outer, inner, out_shape = _pool_shape(w, H, G, head_axis)
    out = np.empty(out_shape, dtype=np.float32)
    if lib.oracle_meanpool_f32(_ptr(w), _ptr(out), outer, H, G, inner) != 0:
        raise ValueError("oracle_meanpool_f32 rejected its arguments")
    return out


def meanpool_f64(w: np.ndarray, H: int, G: int, head_axis: int = 0, lib=None) -> np.ndarray:
    """float64 twin of :func:`meanpool_f32` (same order, double arithmetic)."""
    lib = lib or load()
    w = np.ascontiguousarray(w, dtype=np.float32)
    outer, inner, out_shape = _pool_shape(w, H, G, head_axis)
    out = np.empty(out_shape, dtype=np.float64)
    if lib.oracle_meanpool_f64(_ptr(w), _ptr(out), outer, H, G, inner) != 0:
        raise ValueError("oracle_meanpool_f64 rejected its arguments")
    return out


def _pool_shape(w: np.ndarray, H: int, G: int, head_axis: int):
    if head_axis == 0:                       # head-major [H, ...]
        assert w.shape[0] == H
        inner = int(np.prod(w.shape[1:], dtype=np.int64))
        return 1, inner, (G,) + w.shape[1:]
    assert head_axis == 1 and w.ndim == 3 and w.shape[1] == H   # [outer, H, inner]
    return w.shape[0], w.shape[2], (w.shape[0], G, w.shape[2])


def group_of(i: int, H: int, G: int, lib=None) -> int:
    return (lib or load()).oracle_group_of(i, H, G)


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()


def set_num_threads(n: int, lib=None) -> None:
    """OpenMP threads of later oracle calls (the CPU baseline times one thread and all cores)."""
    (lib or load()).oracle_set_num_threads(int(n))
