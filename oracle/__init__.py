"""CPU oracle for the dense GEMM / GEMV / expert-ID matmul path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are its only users.  It shares no code with the
CUDA library and never imports it.

``oracle.c`` holds the arithmetic (binary64 accumulation, the plain
definitions); this module only compiles it with gcc and marshals numpy
buffers.  Every function returns binary64 results together with
sum |a||b| per element, the scale of the parity tolerance.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (worked examples from the pages, closed forms,
library routines, brute force); none is unpinned.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DT_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            lib.oracle_decode.argtypes = [ctypes.c_int, vp, i64, dp]
            lib.oracle_decode.restype = None
            lib.oracle_gemm.argtypes = [ctypes.c_int, i64, i64, i64, i64, ctypes.c_int,
                                        ctypes.c_int, vp, i64, i64, vp, i64, i64, i64, vp,
                                        dp, dp, ctypes.c_int]
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_matmul_id.argtypes = [ctypes.c_int, i64, i64, i64, i64, i64, i64,
                                             ctypes.c_int, vp, vp, vp, i64, vp, dp, dp,
                                             ctypes.c_int]
            lib.oracle_matmul_id.restype = ctypes.c_int
            lib.oracle_map_distinct.argtypes = [i64, i64, i64, vp, vp, vp]
            lib.oracle_map_distinct.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def default_threads() -> int:
    return os.cpu_count() or 1


def decode(values: np.ndarray, dtype: str) -> np.ndarray:
    """binary64 value of every stored element (bf16 given as uint16 bits)."""
    src = np.ascontiguousarray(values)
    out = np.empty(src.size, dtype=np.float64)
    _load().oracle_decode(DT_CODE[dtype], _ptr(src), src.size, _ptr(out))
    return out.reshape(src.shape)


def gemm(dtype: str, batch: int, m: int, n: int, k: int, ta: bool, tb: bool,
         a: np.ndarray, lda: int, sa: int, b: np.ndarray, ldb: int, sb: int,
         idx: np.ndarray | None = None, nthreads: int | None = None):
    """C = op(A) op(B) per batch.

    ``a``/``b`` are flat element buffers (bf16 as uint16 bits) addressed with
    the leading dims and batch strides in elements.  Returns (c, c_abs): with
    ``idx`` None both are [batch, m, n]; otherwise 1-D, one entry per flat
    index b*m*n + i*n + j in ``idx``.
    """
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    if idx is None:
        count = batch * m * n
        idx_p = None
    else:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        count = idx.size
        idx_p = _ptr(idx)
    c = np.empty(count, dtype=np.float64)
    c_abs = np.empty(count, dtype=np.float64)
    rc = _load().oracle_gemm(DT_CODE[dtype], batch, m, n, k, int(ta), int(tb), _ptr(a), lda, sa,
                             _ptr(b), ldb, sb, count, idx_p, _ptr(c), _ptr(c_abs),
                             nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    if idx is None:
        return c.reshape(batch, m, n), c_abs.reshape(batch, m, n)
    return c, c_abs


def matmul_id(wdtype: str, m: int, n: int, k: int, top_k: int, n_experts: int,
              expert_stride_bytes: int, input_layout: int, w: np.ndarray, x: np.ndarray,
              ids: np.ndarray, idx: np.ndarray | None = None, nthreads: int | None = None):
    """Expert-ID matmul.  Returns (out, out_abs): [m, top_k, n] when ``idx`` is
    None, else 1-D over flat indices r*n + j (r = t*top_k + s)."""
    w = np.ascontiguousarray(w)
    x = np.ascontiguousarray(x, dtype=np.float32)
    ids = np.ascontiguousarray(ids, dtype=np.uint32)
    if idx is None:
        count = m * top_k * n
        idx_p = None
    else:
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        count = idx.size
        idx_p = _ptr(idx)
    out = np.empty(count, dtype=np.float64)
    out_abs = np.empty(count, dtype=np.float64)
    rc = _load().oracle_matmul_id(DT_CODE[wdtype], m, n, k, top_k, n_experts,
                                  expert_stride_bytes, input_layout, _ptr(w), _ptr(x), _ptr(ids),
                                  count, idx_p, _ptr(out), _ptr(out_abs),
                                  nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_matmul_id rejected its arguments")
    if idx is None:
        return out.reshape(m, top_k, n), out_abs.reshape(m, top_k, n)
    return out, out_abs


def map_distinct(m: int, top_k: int, n_experts: int, ids: np.ndarray):
    """Routing map: (counts u32 [n_experts], routed_rows u32 [n_experts, m]).
    Entries of routed_rows past counts[e] are zero here and carry no meaning."""
    ids = np.ascontiguousarray(ids, dtype=np.uint32)
    counts = np.zeros(n_experts, dtype=np.uint32)
    rows = np.zeros(n_experts * m, dtype=np.uint32)
    _load().oracle_map_distinct(m, top_k, n_experts, _ptr(ids), _ptr(counts), _ptr(rows))
    return counts, rows.reshape(n_experts, m)
