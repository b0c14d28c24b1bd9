"""ctypes wrapper around the fp64 C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg import this package.  It never touches the
CUDA library and the CUDA library never touches it.

The shared object is built with gcc into ``oracle/_build/liboracle.so`` on
first use (or by ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "liboracle.so")

ORC_OK = 0
ORC_BAD_VALUE = -1
ORC_BAD_SHAPE = -2
ORC_BAD_CODE = -3

_lib = None
_lock = threading.Lock()


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no vectorisation flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.orc_pack.argtypes = [p, i64, i64, p]
            lib.orc_unpack.argtypes = [p, i64, i64, p]
            lib.orc_stats.argtypes = [p, i64, i64, p, p]
            lib.orc_gemm.argtypes = [p, p, i64, i64, p, i64, p, i64, i64]
            lib.orc_swiglu.argtypes = [p, p, p, p, i64, i64, p, i64, p, i64, i64]
            lib.orc_silu.argtypes = [ctypes.c_double]
            lib.orc_silu.restype = ctypes.c_double
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_double.restype = ctypes.c_double
            lib.orc_rmsnorm.argtypes = [p, p, i64, i64, ctypes.c_double, p, p]
            lib.orc_rmsnorm_gemm.argtypes = [p, p, i64, i64, p, p, ctypes.c_double, i64, p, p, i64, i64]
            lib.orc_i8_gemm.argtypes = [p, p, i64, i64, p, i64, p, p, i64, i64]
            lib.orc_argmax.argtypes = [p, i64, i64, p]
            lib.orc_pack5.argtypes = [p, i64, i64, p]
            lib.orc_unpack5.argtypes = [p, i64, i64, p]
            lib.orc_gemm5.argtypes = [p, p, i64, i64, p, i64, p, i64, i64]
            for f in (lib.orc_pack, lib.orc_unpack, lib.orc_stats, lib.orc_gemm, lib.orc_swiglu, lib.orc_rmsnorm,
                      lib.orc_rmsnorm_gemm, lib.orc_i8_gemm, lib.orc_argmax, lib.orc_pack5, lib.orc_unpack5,
                      lib.orc_gemm5):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check(rc: int, what: str):
    if rc != ORC_OK:
        raise OracleError(f"{what}: oracle status {rc}")


def pack(t: np.ndarray) -> np.ndarray:
    """int8 [rows, k] -> uint32 [rows, k//16] in the project's 2-bit format."""
    t = np.ascontiguousarray(t, dtype=np.int8)
    rows, k = t.shape
    codes = np.zeros((rows, k // 16 if k % 64 == 0 else 0), dtype=np.uint32)
    _check(_load().orc_pack(_ptr(t), rows, k, _ptr(codes)), "pack")
    return codes


def unpack(codes: np.ndarray, k: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    rows = codes.shape[0]
    t = np.zeros((rows, k), dtype=np.int8)
    _check(_load().orc_unpack(_ptr(codes), rows, k, _ptr(t)), "unpack")
    return t


def stats(codes: np.ndarray, k: int):
    """Returns (rowsum int64 [rows], counts int64 [3] = zeros, plus, minus)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    rows = codes.shape[0]
    rowsum = np.zeros(rows, dtype=np.int64)
    counts = np.zeros(3, dtype=np.int64)
    _check(_load().orc_stats(_ptr(codes), rows, k, _ptr(rowsum), _ptr(counts)), "stats")
    return rowsum, counts


def _row_split(rows: int, threads: int):
    threads = max(1, min(threads, rows)) if rows > 0 else 1
    step = (rows + threads - 1) // threads if rows > 0 else 0
    return [(b, min(rows, b + step)) for b in range(0, rows, step)] if rows > 0 else []


def _run_rows(fn, rows: int, threads: int, rows_subset=None):
    """Run fn(row_begin, row_end) over row ranges on Python threads.

    ctypes releases the GIL during the C call, so the ranges run in parallel.
    ``rows_subset`` (sorted row indices) restricts the work to those rows.
    """
    if rows_subset is not None:
        ranges = [(int(r), int(r) + 1) for r in rows_subset]
    else:
        ranges = _row_split(rows, threads)
    errs = []

    def worker(chunk):
        for (b, e) in chunk:
            rc = fn(b, e)
            if rc != ORC_OK:
                errs.append(rc)
                return

    nthreads = max(1, min(threads, len(ranges)))
    chunks = [ranges[i::nthreads] for i in range(nthreads)]
    if nthreads == 1:
        worker(chunks[0] if chunks else [])
    else:
        ts = [threading.Thread(target=worker, args=(c,)) for c in chunks]
        for th in ts:
            th.start()
        for th in ts:
            th.join()
    if errs:
        raise OracleError(f"oracle status {errs[0]}")


def gemm(codes: np.ndarray, scale: np.ndarray, k: int, x_bits: np.ndarray,
         threads: int = 1, rows_subset=None) -> np.ndarray:
    """y [m, rows] float64 = scale * (T @ x), x given as bf16 bits [m, k]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    x_bits = np.ascontiguousarray(np.atleast_2d(x_bits), dtype=np.uint16)
    rows = codes.shape[0]
    m = x_bits.shape[0]
    assert x_bits.shape[1] == k
    y = np.zeros((m, rows), dtype=np.float64)
    lib = _load()
    _run_rows(lambda b, e: lib.orc_gemm(_ptr(codes), _ptr(scale), rows, k, _ptr(x_bits), m,
                                        _ptr(y), b, e), rows, threads, rows_subset)
    return y


def swiglu(g_codes, g_scale, u_codes, u_scale, k: int, x_bits: np.ndarray,
           threads: int = 1, rows_subset=None) -> np.ndarray:
    """h [m, rows] float64 = silu(g) * u."""
    g_codes = np.ascontiguousarray(g_codes, dtype=np.uint32)
    u_codes = np.ascontiguousarray(u_codes, dtype=np.uint32)
    g_scale = np.ascontiguousarray(g_scale, dtype=np.float32)
    u_scale = np.ascontiguousarray(u_scale, dtype=np.float32)
    x_bits = np.ascontiguousarray(np.atleast_2d(x_bits), dtype=np.uint16)
    rows = g_codes.shape[0]
    assert u_codes.shape == g_codes.shape
    m = x_bits.shape[0]
    h = np.zeros((m, rows), dtype=np.float64)
    lib = _load()
    _run_rows(lambda b, e: lib.orc_swiglu(_ptr(g_codes), _ptr(g_scale), _ptr(u_codes), _ptr(u_scale),
                                          rows, k, _ptr(x_bits), m, _ptr(h), b, e),
              rows, threads, rows_subset)
    return h


def silu(z: float) -> float:
    return _load().orc_silu(float(z))


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits))


def rmsnorm(x_bits: np.ndarray, g: np.ndarray, eps: float = 1e-6):
    """RMSNorm of each activation row, rounded to bf16 (see orc_rmsnorm).

    Returns (xn_bits uint16 [m, k], r float32 [m]) where r is each row's
    fp32 factor 1 / sqrt(mean x^2 + eps)."""
    x_bits = np.ascontiguousarray(np.atleast_2d(x_bits), dtype=np.uint16)
    g = np.ascontiguousarray(g, dtype=np.float32)
    m, k = x_bits.shape
    assert g.shape == (k,)
    xn = np.zeros((m, k), dtype=np.uint16)
    r = np.zeros(m, dtype=np.float32)
    _check(_load().orc_rmsnorm(_ptr(x_bits), _ptr(g), m, k, float(eps), _ptr(xn), _ptr(r)), "rmsnorm")
    return xn, r


def rmsnorm_gemm(codes, scale, k: int, x_bits: np.ndarray, g: np.ndarray, eps: float = 1e-6,
                 threads: int = 1, rows_subset=None) -> np.ndarray:
    """y [m, rows] float64 = scale * (T @ rmsnorm(x)): the projection that
    follows a norm (q/k/v after the attention norm)."""
    xn, _ = rmsnorm(x_bits, g, eps)
    return gemm(codes, scale, k, xn, threads=threads, rows_subset=rows_subset)


def rmsnorm_gemm_c(codes, scale, k: int, x_bits: np.ndarray, g: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """rmsnorm_gemm through the C composite orc_rmsnorm_gemm (one thread)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    x_bits = np.ascontiguousarray(np.atleast_2d(x_bits), dtype=np.uint16)
    g = np.ascontiguousarray(g, dtype=np.float32)
    rows = codes.shape[0]
    m = x_bits.shape[0]
    xn = np.zeros((m, k), dtype=np.uint16)
    y = np.zeros((m, rows), dtype=np.float64)
    _check(_load().orc_rmsnorm_gemm(_ptr(codes), _ptr(scale), rows, k, _ptr(x_bits), _ptr(g), float(eps), m,
                                    _ptr(xn), _ptr(y), 0, rows), "rmsnorm_gemm")
    return y


def rmsnorm_swiglu(g_codes, g_scale, u_codes, u_scale, k: int, x_bits: np.ndarray, g: np.ndarray,
                   eps: float = 1e-6, threads: int = 1, rows_subset=None) -> np.ndarray:
    """h = silu(gate) * up on rmsnorm(x): the feed-forward block's first step."""
    xn, _ = rmsnorm(x_bits, g, eps)
    return swiglu(g_codes, g_scale, u_codes, u_scale, k, xn, threads=threads, rows_subset=rows_subset)


def i8_gemm(w: np.ndarray, scale: np.ndarray, x_bits: np.ndarray, threads: int = 1, rows_subset=None,
            with_abs: bool = False):
    """int8 head logits [m, rows] float64 = scale * (W @ x); with_abs also
    returns scale * sum_k |w x| per logit (the fp32 error's yardstick)."""
    w = np.ascontiguousarray(w, dtype=np.int8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    x_bits = np.ascontiguousarray(np.atleast_2d(x_bits), dtype=np.uint16)
    rows, k = w.shape
    m = x_bits.shape[0]
    assert x_bits.shape[1] == k
    y = np.zeros((m, rows), dtype=np.float64)
    a = np.zeros((m, rows), dtype=np.float64)
    lib = _load()
    _run_rows(lambda b, e: lib.orc_i8_gemm(_ptr(w), _ptr(scale), rows, k, _ptr(x_bits), m, _ptr(y), _ptr(a), b, e),
              rows, threads, rows_subset)
    return (y, a) if with_abs else y


def argmax(y: np.ndarray) -> np.ndarray:
    """Per row of y [m, rows]: the index of the largest value, lowest on ties."""
    y = np.ascontiguousarray(np.atleast_2d(y), dtype=np.float64)
    m, rows = y.shape
    idx = np.zeros(m, dtype=np.int64)
    _check(_load().orc_argmax(_ptr(y), m, rows, _ptr(idx)), "argmax")
    return idx


def pack5(t: np.ndarray) -> np.ndarray:
    """int8 [rows, k] (k % 80 == 0) -> uint8 [rows, k//5] in the base-3 format."""
    t = np.ascontiguousarray(t, dtype=np.int8)
    rows, k = t.shape
    codes = np.zeros((rows, k // 5), dtype=np.uint8)
    _check(_load().orc_pack5(_ptr(t), rows, k, _ptr(codes)), "pack5")
    return codes


def unpack5(codes: np.ndarray, k: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    rows = codes.shape[0]
    t = np.zeros((rows, k), dtype=np.int8)
    _check(_load().orc_unpack5(_ptr(codes), rows, k, _ptr(t)), "unpack5")
    return t


def gemm5(codes: np.ndarray, scale: np.ndarray, k: int, x_bits: np.ndarray, threads: int = 1,
          rows_subset=None) -> np.ndarray:
    """y [m, rows] float64 = scale * (T @ x) from base-3 codes."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    x_bits = np.ascontiguousarray(np.atleast_2d(x_bits), dtype=np.uint16)
    rows = codes.shape[0]
    m = x_bits.shape[0]
    y = np.zeros((m, rows), dtype=np.float64)
    lib = _load()
    _run_rows(lambda b, e: lib.orc_gemm5(_ptr(codes), _ptr(scale), rows, k, _ptr(x_bits), m, _ptr(y), b, e),
              rows, threads, rows_subset)
    return y
