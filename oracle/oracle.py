"""ctypes front end of the plain-C oracle (test infrastructure only).

build() compiles oracle.c with gcc (OpenMP over slots; no other change to the
arithmetic).  The wrappers take numpy arrays in the same layout as the C-ABI
library's arguments and return numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=gnu11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # a prebuilt variant of the library (the pin-strength test loads copies of
        # oracle.c with one planted mistake each through this variable)
        lib = ctypes.CDLL(os.environ.get("IDXTOPK_ORACLE_LIB") or build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e2m1_value.argtypes = [ctypes.c_int]
        lib.oracle_ue8m0_value.restype = ctypes.c_double
        lib.oracle_ue8m0_value.argtypes = [ctypes.c_int]
        for fn in (lib.oracle_row_logits,):
            fn.restype = ctypes.c_longlong
            fn.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]
        lib.oracle_row_scores.restype = ctypes.c_longlong
        lib.oracle_row_scores.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]
        lib.oracle_select.restype = i64
        lib.oracle_select.argtypes = [P, i64, i64, i32, P]
        lib.oracle_prefill_rows.restype = ctypes.c_int
        lib.oracle_prefill_rows.argtypes = [P, P, P, P, P, P, i32, i32, i32, P, P, P, P, i32,
                                            i32, P, P, P, P]
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def threads() -> int:
    return int(_load().oracle_threads())


def e2m1_value(code: int) -> float:
    return float(_load().oracle_e2m1_value(int(code)))


def ue8m0_value(byte: int) -> float:
    return float(_load().oracle_ue8m0_value(int(byte)))


def _problem_arrays(p):
    return (_c(p.q_fp4, np.uint8), _c(p.q_scale, np.uint8), _c(p.k_cache_fp4, np.uint8),
            _c(p.k_scale, np.uint8), _c(p.weights, np.float32), _c(p.page_table, np.int32))


def row_logits(p, row: int, s_begin: int, s_end: int):
    """Exact per-head dots [(s_end - s_begin), 64] (float64) and the count of
    dots that are not exact in fp32."""
    q, qs, k, ks, _, pt = _problem_arrays(p)
    out = np.zeros((max(0, s_end - s_begin), 64), dtype=np.float64)
    n = _load().oracle_row_logits(_p(q), _p(qs), _p(k), _p(ks), _p(pt), pt.shape[1],
                                  k.shape[0], int(row), int(p.row_req[row]), int(s_begin),
                                  int(s_end), _p(out))
    if n < 0:
        raise OracleError("bad page entry")
    return out, int(n)


def row_scores(p, row: int, s_begin: int = None, s_end: int = None):
    """float64 scores of `row` over [s_begin, s_end) (default: its window)."""
    if s_begin is None:
        s_begin = int(p.row_start[row])
    if s_end is None:
        s_end = int(p.row_end[row])
    q, qs, k, ks, w, pt = _problem_arrays(p)
    out = np.zeros(max(0, s_end - s_begin), dtype=np.float64)
    n = _load().oracle_row_scores(_p(q), _p(qs), _p(k), _p(ks), _p(w), _p(pt), pt.shape[1],
                                  k.shape[0], int(row), int(p.row_req[row]), int(s_begin),
                                  int(s_end), _p(out))
    if n < 0:
        raise OracleError("bad page entry")
    return out, int(n)


def select(scores: np.ndarray, k: int, base: int = 0) -> np.ndarray:
    """Exact TopK indices (base + position) under the total order, -1 padded."""
    s = _c(scores, np.float64).ravel()
    out = np.empty(int(k), dtype=np.int32)
    _load().oracle_select(_p(s), s.size, int(base), int(k), _p(out))
    return out


def prefill_rows(p, rows=None, with_kth: bool = False):
    """Oracle outputs (phys, raw) [n_rows, topk] for the listed rows (default all)."""
    if rows is None:
        rows = np.arange(p.rows, dtype=np.int32)
    rows = _c(rows, np.int32)
    q, qs, k, ks, w, pt = _problem_arrays(p)
    rr, rs, re = _c(p.row_req, np.int32), _c(p.row_start, np.int32), _c(p.row_end, np.int32)
    K = int(p.topk)
    phys = np.empty((rows.size, K), dtype=np.int32)
    raw = np.empty((rows.size, K), dtype=np.int32)
    kth = np.empty(rows.size, dtype=np.float64)
    inexact = ctypes.c_longlong(0)
    st = _load().oracle_prefill_rows(_p(q), _p(qs), _p(k), _p(ks), _p(w), _p(pt), pt.shape[0],
                                     pt.shape[1], k.shape[0], _p(rr), _p(rs), _p(re), _p(rows),
                                     rows.size, K, _p(phys), _p(raw), _p(kth),
                                     ctypes.byref(inexact))
    if st == 1:
        raise OracleError("invalid row metadata")
    if st == 2:
        raise OracleError("invalid page entry")
    if with_kth:
        return phys, raw, kth, int(inexact.value)
    return phys, raw
